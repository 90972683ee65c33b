// dcp_merge_row.cuh -- one warp merges n partial rows (O_i, LSE_i) of a 512-wide output.
//
// Exact log-sum-exp recombination ("Serving Macaron-V1 at Scale", 5.2; "SGLang's path"):
// M = max_i LSE_i, w_i = exp(LSE_i - M), LSE = M + ln sum w_i, O = sum w_i O_i / sum w_i,
// summed in ascending i; parts with LSE = -inf weigh zero; all -inf gives O = 0, LSE = -inf.
#pragma once

#include <cmath>
#include <cstdint>

namespace dcp {

// Partial i's row starts at o + i * o_stride (floats) and its LSE at lse[i * lse_stride].
// Lane owns float4 columns lane + 32k, k < 4.  `scale` multiplies the merged O.  kPar partial
// rows have their loads in flight together.
template <int kPar = 4>
__device__ __forceinline__ void warp_merge_row512(int n, const float *o, int64_t o_stride,
                                                  const float *lse, int64_t lse_stride,
                                                  float *o_out, float *lse_out, float scale) {
    const int lane = threadIdx.x & 31;
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) mx = fmaxf(mx, __ldcg(lse + i * lse_stride));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float4 *dst = reinterpret_cast<float4 *>(o_out);
    if (mx == -INFINITY) {
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[lane + 32 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    float acc[4][4] = {};
    float wsum = 0.f;
    for (int i0 = 0; i0 < n; i0 += kPar) {
        float4 x[kPar][4];
        float w[kPar];
#pragma unroll
        for (int j = 0; j < kPar; ++j) {
            const int i = i0 + j;
            w[j] = 0.f;
            if (i < n) {
                const float l = __ldcg(lse + i * lse_stride);
                w[j] = (l == -INFINITY) ? 0.f : expf(l - mx);
                const float4 *src = reinterpret_cast<const float4 *>(o + i * o_stride);
#pragma unroll
                for (int k = 0; k < 4; ++k) x[j][k] = __ldcg(src + lane + 32 * k);
            }
        }
#pragma unroll
        for (int j = 0; j < kPar; ++j) {
            if (w[j] == 0.f) continue;
            wsum += w[j];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[k][0] = fmaf(w[j], x[j][k].x, acc[k][0]);
                acc[k][1] = fmaf(w[j], x[j][k].y, acc[k][1]);
                acc[k][2] = fmaf(w[j], x[j][k].z, acc[k][2]);
                acc[k][3] = fmaf(w[j], x[j][k].w, acc[k][3]);
            }
        }
    }
    const float inv = scale / wsum;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        dst[lane + 32 * k] = make_float4(acc[k][0] * inv, acc[k][1] * inv, acc[k][2] * inv, acc[k][3] * inv);
    if (lane == 0) *lse_out = mx + logf(wsum);
}

}  // namespace dcp
