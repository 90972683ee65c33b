// dcp_merge.cu -- exact log-sum-exp merge of per-rank partial attention outputs.
//
// "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding", 5.2 (LSE_merged =
// log sum_d exp LSE_d) and 8 (ranks combined in a fixed order); "SGLang's path" (the
// partials recombine exactly).  One warp per 128-column slice of an output row: the lanes
// read the N_dcp LSE values, reduce the maximum with shuffles, then stream the N_dcp partial
// slices with 16-byte loads (one float4 per lane) and write the merged slice.  The kernel is HBM-bound: N*rows*(4*v_dim + 4) bytes read, rows*(4*v_dim + 4) written.
#include <algorithm>
#include <cmath>

#include "dcp_internal.h"
#include "dcp_ptx.cuh"

namespace dcp {
namespace {

constexpr int kMergeWarps = 8;
// Partial rows whose loads are in flight together: 4 (124 registers, two blocks per SM) beats 8
// (202 registers, one block per SM) by 10-15% on 2K-8K rows of 8 partials from HBM.
constexpr int kPartBatch = 4;

#ifndef DCP_MERGE_VEC
#define DCP_MERGE_VEC 4
#endif

// One warp per (row, slice of 128 * VEC columns): each lane owns VEC float4 of the slice.  The
// warp reads the N LSE values (a broadcast load each), reduces the maximum with shuffles, then
// streams the N partial slices with kPartBatch rows of 16-byte loads in flight per lane, summing
// the weighted rows in ascending rank order.
template <int VEC>
__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_kernel(int n_parts, int64_t rows, int slices, const float *__restrict__ o_part,
                 const float *__restrict__ lse_part, float *__restrict__ o_out, float *__restrict__ lse_out) {
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t task = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (task >= rows * slices) return;
    const int64_t row = task / slices;
    const int sl = (int)(task - row * slices);
    const int64_t vdim4 = 32 * VEC * (int64_t)slices;  // float4 per row
    const int64_t col4 = (int64_t)sl * 32 * VEC + lane;  // lane's first float4; then + 32 k

    float mx = -INFINITY;
    for (int d = lane; d < n_parts; d += 32) mx = fmaxf(mx, __ldg(lse_part + (int64_t)d * rows + row));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    float4 *dst = reinterpret_cast<float4 *>(o_out) + row * vdim4 + col4;
    if (mx == -INFINITY) {
#pragma unroll
        for (int k = 0; k < VEC; ++k) dst[32 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (sl == 0 && lane == 0) lse_out[row] = -INFINITY;
        return;
    }
    float4 acc[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
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
                const float4 *src = reinterpret_cast<const float4 *>(o_part) + ((int64_t)d * rows + row) * vdim4 + col4;
#pragma unroll
                for (int k = 0; k < VEC; ++k) buf[i][k] = __ldg(src + 32 * k);
            }
        }
#pragma unroll
        for (int i = 0; i < kPartBatch; ++i) {
            if (d0 + i < n_parts && w[i] != 0.f) {
                wsum += w[i];
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    acc[k].x = fmaf(w[i], buf[i][k].x, acc[k].x);
                    acc[k].y = fmaf(w[i], buf[i][k].y, acc[k].y);
                    acc[k].z = fmaf(w[i], buf[i][k].z, acc[k].z);
                    acc[k].w = fmaf(w[i], buf[i][k].w, acc[k].w);
                }
            }
        }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int k = 0; k < VEC; ++k) dst[32 * k] = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
    if (sl == 0 && lane == 0) lse_out[row] = mx + logf(wsum);
}

}  // namespace

cudaError_t launch_lse_merge(int n_parts, int64_t rows, int v_dim, const float *o_part,
                             const float *lse_part, float *o_out, float *lse_out,
                             cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    if (v_dim != 128 && v_dim != 256 && v_dim != 512) return cudaErrorInvalidValue;
    const int vec = std::min(DCP_MERGE_VEC, v_dim / 128);
    const int slices = v_dim / (128 * vec);
    const int64_t blocks = (rows * slices + kMergeWarps - 1) / kMergeWarps;
    switch (vec) {
        case 1: return launch_pdl(lse_merge_kernel<1>, dim3((unsigned)blocks), dim3(kMergeWarps * 32), 0, stream,
                                  n_parts, rows, slices, o_part, lse_part, o_out, lse_out);
        case 2: return launch_pdl(lse_merge_kernel<2>, dim3((unsigned)blocks), dim3(kMergeWarps * 32), 0, stream,
                                  n_parts, rows, slices, o_part, lse_part, o_out, lse_out);
        default: return launch_pdl(lse_merge_kernel<4>, dim3((unsigned)blocks), dim3(kMergeWarps * 32), 0, stream,
                                   n_parts, rows, slices, o_part, lse_part, o_out, lse_out);
    }
}

}  // namespace dcp
