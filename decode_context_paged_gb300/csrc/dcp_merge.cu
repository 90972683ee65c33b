// dcp_merge.cu -- exact log-sum-exp merge of per-rank partial attention outputs.
//
// "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding", 5.2 (LSE_merged =
// log sum_d exp LSE_d) and 8 (ranks combined in a fixed order); "SGLang's path" (the
// partials recombine exactly).  One warp per output row: the lanes read the N_dcp LSE
// values, reduce max and weight sum with shuffles, then stream the N_dcp partial rows with
// 16-byte loads (each lane owns v_dim/32 contiguous-by-float4 columns) and write the merged
// row.  The kernel is HBM-bound: N*rows*(4*v_dim + 4) bytes read, rows*(4*v_dim + 4) written.
#include <cmath>

#include "dcp_internal.h"

namespace dcp {
namespace {

constexpr int kMergeWarps = 8;
constexpr int kPartBatch = 8;  // partial rows whose loads are in flight together

template <int VEC>  // float4 vectors per lane (v_dim = 128 * VEC)
__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_kernel(int n_parts, int64_t rows, const float *__restrict__ o_part,
                 const float *__restrict__ lse_part, float *__restrict__ o_out,
                 float *__restrict__ lse_out) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    constexpr int kVDimT = 128 * VEC;

    // max over parts (ascending d inside each lane, then a shuffle tree)
    float mx = -INFINITY;
    for (int d = lane; d < n_parts; d += 32) mx = fmaxf(mx, __ldg(lse_part + (int64_t)d * rows + row));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    float4 *dst = reinterpret_cast<float4 *>(o_out + row * kVDimT);
    if (mx == -INFINITY) {
#pragma unroll
        for (int k = 0; k < VEC; ++k) dst[lane + 32 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) lse_out[row] = -INFINITY;
        return;
    }

    float acc[VEC][4];
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
    float wsum = 0.f;
    for (int d0 = 0; d0 < n_parts; d0 += kPartBatch) {
        float4 buf[kPartBatch][VEC];
        float w[kPartBatch];
#pragma unroll
        for (int i = 0; i < kPartBatch; ++i) {
            const int d = d0 + i;
            w[i] = 0.f;
            if (d < n_parts) {
                const float l = __ldg(lse_part + (int64_t)d * rows + row);
                w[i] = (l == -INFINITY) ? 0.f : expf(l - mx);
                const float4 *src = reinterpret_cast<const float4 *>(o_part + ((int64_t)d * rows + row) * kVDimT);
#pragma unroll
                for (int k = 0; k < VEC; ++k) buf[i][k] = __ldg(src + lane + 32 * k);
            }
        }
#pragma unroll
        for (int i = 0; i < kPartBatch; ++i) {
            if (d0 + i < n_parts && w[i] != 0.f) {
                wsum += w[i];
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    acc[k][0] = fmaf(w[i], buf[i][k].x, acc[k][0]);
                    acc[k][1] = fmaf(w[i], buf[i][k].y, acc[k][1]);
                    acc[k][2] = fmaf(w[i], buf[i][k].z, acc[k][2]);
                    acc[k][3] = fmaf(w[i], buf[i][k].w, acc[k][3]);
                }
            }
        }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int k = 0; k < VEC; ++k)
        dst[lane + 32 * k] = make_float4(acc[k][0] * inv, acc[k][1] * inv, acc[k][2] * inv, acc[k][3] * inv);
    if (lane == 0) lse_out[row] = mx + logf(wsum);
}

template <int VEC>
cudaError_t launch_vec(int n_parts, int64_t rows, const float *o_part, const float *lse_part,
                       float *o_out, float *lse_out, cudaStream_t stream) {
    const int64_t blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    lse_merge_kernel<VEC><<<(unsigned)blocks, kMergeWarps * 32, 0, stream>>>(n_parts, rows, o_part,
                                                                            lse_part, o_out, lse_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(int n_parts, int64_t rows, int v_dim, const float *o_part,
                             const float *lse_part, float *o_out, float *lse_out,
                             cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    switch (v_dim / 128) {
        case 1: return launch_vec<1>(n_parts, rows, o_part, lse_part, o_out, lse_out, stream);
        case 2: return launch_vec<2>(n_parts, rows, o_part, lse_part, o_out, lse_out, stream);
        case 4: return launch_vec<4>(n_parts, rows, o_part, lse_part, o_out, lse_out, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dcp
