// dcp_attn.cu -- paged absorbed-MLA decode attention over DCP page shards (partial O + LSE).
//
// "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding", 5.1 (rank d owns the pages
// whose value is congruent to d mod N_dcp, at slot value div N_dcp), 5.2 (each rank attends
// over its own pages and returns a partial output plus its LSE), 5.3 (rows are 512 latent +
// 64 rope = 576 elements), 8 (multi-token verification under DCP); "SGLang's path" (the
// partial is a weighted sum plus a log-sum-exp that recombines exactly).
//
// Design (GB300 / sm_103a):
//  * A plan step on the device compacts each (rank, request) page list in page order and
//    cuts it into chunks of `tiles_per_chunk` 128-token tiles; a work unit is (rank,
//    request, chunk, query group), a query group being one new token and up to 64 heads.
//    Units are ordered by size (largest first) with the groups of one chunk adjacent, and
//    persistent CTAs (one per SM) take them from an atomic counter (CTA i starts with unit i).
//    When the queue's last round would leave SMs idle, the plan cuts that round's chunks into
//    balanced pieces (merged like chunks; deterministic, so results are reproducible).
//  * Tokens are the MMA's M dimension (128 = two pages), query rows its N.  Per tile
//    tcgen05 computes S^T[128 x n] = K_tile * Q^T into TMEM, the softmax warps turn it into
//    P^T in shared memory, and tcgen05 accumulates O^T[512 x 64] += V_tile^T * P^T in TMEM.
//    BF16 pools use kind::f16 (BF16 operands).  FP8-E4M3 pools use kind::f8f6f4 on the raw
//    page bytes: Q enters as two E4M3 terms (hi + lo, stacked as N = 128 rows, with a
//    power-of-two scale per query row) so the scores keep BF16-level accuracy, and P enters
//    as hi + lo terms accumulated into the same O^T.
//  * BF16: two TMA streams.  The K stream (all 576 dims of a tile, read from HBM with an L2
//    evict-last hint) feeds the score MMAs through a 4-slot ring; the V stream re-reads the
//    512 latent dims of the same pages (an L2 hit) into a 2-unit ring for P*V.
//    E4M3: one stream into a unified ring.  The four 128-dim latent blocks of a tile stay in
//    their slots from the score MMAs to the P*V MMAs, which read them as V; the ring holds two
//    tiles, plus a slot for the rope block.  Separate MMA-issuing threads for the two products
//    keep HBM loads in flight while the softmax of an earlier tile runs.
//  * Rows of a request's last page past its length may hold any bytes: the stream that feeds
//    P*V clears them in shared memory before the MMA reads them.
//  * Sixteen softmax warps (four warpgroups of 16 query columns each) own one token row per
//    thread (TMEM lane = row): scores are masked
//    (ragged last page, causal limit among the new tokens), column maxima are reduced with a
//    warp-shuffle reduce-scatter plus shared memory, exp2 weights go to shared memory, and
//    O^T is rescaled in TMEM only when a column's running max moved.
//  * Single-chunk segments write O_part / LSE_part directly; multi-chunk segments write
//    chunk partials to the workspace and a combine kernel merges them (exact LSE merge).
//  * Every mbarrier wait is bounded; on timeout the CTA stops, drains its in-flight copies
//    and MMAs, frees TMEM and reports DCP_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "dcp_internal.h"
#include "dcp_merge_row.cuh"
#include "dcp_ptx.cuh"

namespace dcp {
namespace {

constexpr uint32_t kKSlotBytes = 16384;  // K-stream ring slot
constexpr int kMaxVSlots = 8;            // V-stream ring slots (upper bound of the configurations)
constexpr int kMaxKSlots = 8;            // K-stream ring slots (upper bound of the configurations)
constexpr uint32_t kQBytes = 73728;      // 64 rows x 576 BF16, or 128 rows (hi, lo) x 576 E4M3
constexpr uint32_t kPBytes = 16384;      // one P^T buffer
constexpr int kGroupRows = 64;
constexpr int kThreads = 640;            // 0 K-TMA, 1 S-MMA, 2 V-TMA, 3 PV-MMA, 4-19 softmax
constexpr int kCols = 16;                // query columns per softmax warpgroup
constexpr int kSoftmaxWarps = 16;        // arrivals on the barriers the softmax warps release (one per warp)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;          // S buffers start at TMEM column 256 (O^T uses 0..255)
constexpr int kMaxTpc = 4096;

constexpr float kPScale = 4.f;           // FP8 P is stored as 4 * p (p <= 2^6 under the lazy max)

#ifndef DCP_ATTN_S_BUFS_BF16
#define DCP_ATTN_S_BUFS_BF16 3
#endif
#ifndef DCP_ATTN_S_BUFS_F8
#define DCP_ATTN_S_BUFS_F8 2
#endif
#ifndef DCP_ATTN_K_SLOTS_BF16
#define DCP_ATTN_K_SLOTS_BF16 4
#endif
#ifndef DCP_ATTN_P_BUFS_BF16
#define DCP_ATTN_P_BUFS_BF16 1
#endif
#ifndef DCP_ATTN_K_SLOTS_F8
#define DCP_ATTN_K_SLOTS_F8 4
#endif
#ifndef DCP_ATTN_P_BUFS_F8
#define DCP_ATTN_P_BUFS_F8 1
#endif
// V-stream ring: slots of DCP_ATTN_V_BLOCKS_* blocks, a block being one M-tile of the P*V
// product for the tile's 128 tokens (BF16: two 64-dim TMA boxes, 32 KB; E4M3: one 128-dim box,
// 16 KB).
#ifndef DCP_ATTN_V_SLOTS_BF16
#define DCP_ATTN_V_SLOTS_BF16 2
#endif
#ifndef DCP_ATTN_V_BLOCKS_BF16
#define DCP_ATTN_V_BLOCKS_BF16 1
#endif
#ifndef DCP_ATTN_V_SLOTS_F8
#define DCP_ATTN_V_SLOTS_F8 2
#endif
#ifndef DCP_ATTN_V_BLOCKS_F8
#define DCP_ATTN_V_BLOCKS_F8 2
#endif
// E4M3: one ring for both products.  A tile's four 128-dim blocks of K rows (16 KB each: 128
// latent dims x 2 pages) serve the score MMAs as K and stay resident until the P*V MMAs have
// used them as V, so V is never loaded a second time; the 64-dim rope block has a slot of its
// own and is freed by the score MMAs.  DCP_ATTN_D_SLOTS_F8 blocks = 2 tiles of lookahead.
#ifndef DCP_ATTN_UNIFIED_F8
#define DCP_ATTN_UNIFIED_F8 1
#endif
#ifndef DCP_ATTN_D_SLOTS_F8
#define DCP_ATTN_D_SLOTS_F8 8
#endif

template <bool F8>
struct Cfg {
    // BF16: four K slots and one P buffer (measured: trading a K slot for a second P buffer is
    // slower), a V ring of 2 x 32 KB.  E4M3: the unified ring (8 x 16 KB + the rope slot).
    static constexpr bool kUnified = F8 && DCP_ATTN_UNIFIED_F8;
    static constexpr int kKSlots = kUnified ? DCP_ATTN_D_SLOTS_F8 : F8 ? DCP_ATTN_K_SLOTS_F8 : DCP_ATTN_K_SLOTS_BF16;
    static constexpr int kPBufs = F8 ? DCP_ATTN_P_BUFS_F8 : DCP_ATTN_P_BUFS_BF16;
    static constexpr int kVSlots = kUnified ? 0 : F8 ? DCP_ATTN_V_SLOTS_F8 : DCP_ATTN_V_SLOTS_BF16;
    static constexpr int kVBlk = F8 ? DCP_ATTN_V_BLOCKS_F8 : DCP_ATTN_V_BLOCKS_BF16;  // M-tiles per V slot
    static constexpr uint32_t kVSlotBytes = kVBlk * 32768u / (F8 ? 2u : 1u);
    static constexpr int kVUnits = 4 / kVBlk;       // V-stream units per tile
    static constexpr uint32_t kOffRope = kKSlots * kKSlotBytes;             // unified ring: the rope slot
    static constexpr uint32_t kOffV = kOffRope + (kUnified ? 8192u : 0u);
    static constexpr uint32_t kOffQ = kOffV + kVSlots * kVSlotBytes;
    static constexpr uint32_t kOffP = kOffQ + kQBytes;
    static constexpr uint32_t kOffCtl = kOffP + kPBufs * kPBytes;
    static constexpr float kLazyTauV = F8 ? 6.f : 8.f;  // log2 margin of the lazy maximum
    static constexpr int kKBlocks = F8 ? 5 : 9;     // K-stream blocks per tile
    static constexpr int kSCols = F8 ? 128 : 64;    // TMEM columns per S buffer (hi, lo for FP8)
    static constexpr int kSBufs = F8 ? DCP_ATTN_S_BUFS_F8 : DCP_ATTN_S_BUFS_BF16;
    static constexpr uint32_t kIdescS = F8 ? idesc_e4m3_f32(128, 128, 0, 0) : idesc_bf16_f32(128, 64, 0, 0);
    static constexpr uint32_t kIdescPV = F8 ? idesc_e4m3_f32(128, 64, 1, 1) : idesc_bf16_f32(128, 64, 1, 1);
    // The swizzled buffers need 1024-byte alignment.  The dynamic shared memory of a CTA starts
    // 1024-aligned (after the 1 KB the system reserves); the unified ring's layout uses that and
    // reserves no alignment slack (the kernel checks the alignment before anything else).
    static constexpr uint32_t kPad = kUnified ? 0u : 1024u;
};

struct UnitInfo {
    int valid, d, b, g;
    int n_pages, out_index, limit, q_row0;
    int rows_valid;
    long long comp_base;
};

struct __align__(16) Ctl {
    float red[4][4][16];
    float m_run[64];             // per query column: the reference maximum of the lazy softmax
    float corr[64];
    float oscale[64];
    float qscale[64];            // per query column: softmax_scale * kappa * log2(e) (* 2^-qexp for FP8)
    uint64_t kfull[kMaxKSlots], kempty[kMaxKSlots];
    uint64_t rfull, rempty;      // unified ring: the rope slot
    uint64_t vfull[kMaxVSlots], vempty[kMaxVSlots];
    uint64_t vland;              // V units that need their tail rows cleared land here first
    uint64_t q_full, q_empty;
    uint64_t s_full[3], s_free[3];
    uint64_t p_full[2], o_done[2], o_free;  // p_full[t & 1]: P of global tile t written
    uint64_t unit_full[2], unit_empty[2];
    uint64_t drain_s, drain_pv;
    UnitInfo unit[2];
    uint32_t tmem_base;
    int abort_flag;
};
template <bool F8>
constexpr size_t smem_bytes() { return Cfg<F8>::kPad + Cfg<F8>::kOffCtl + sizeof(Ctl); }
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448, "shared memory budget");
static_assert(Cfg<false>::kVSlots <= kMaxVSlots && Cfg<true>::kVSlots <= kMaxVSlots, "V ring slots");
static_assert(Cfg<false>::kKSlots <= kMaxKSlots && Cfg<true>::kKSlots <= kMaxKSlots, "K ring slots");
static_assert(Cfg<true>::kVUnits > 0 && Cfg<false>::kVUnits > 0, "V units per tile");
static_assert(4 % Cfg<false>::kVBlk == 0 && 4 % Cfg<true>::kVBlk == 0, "V slot blocks divide the 4 M-tiles");

struct AttnMaps {
    CUtensorMap q[2];                  // BF16: [0] 64x64 boxes.  FP8 (hi|lo rows): [0] 128x64 SW128, [1] 64x64 SW64
    CUtensorMap kv[kMaxDcpAttn][2];    // same split per pool
};

struct KParams {
    const int32_t *seq_lens;
    const int64_t *req_page_ptr;
    const int32_t *comp_slot;  // [N][num_pages]: rank d's pages of request b start at d*num_pages + ptr[b]
    const int32_t *comp_page;  // page index j (within the request) of each compacted entry
    const int4 *units;         // {pair*G + g, page_begin, n_pages, out_index}
    const int *ctrl;           // [0] = number of units, [1] = work counter; [3..7] the plan's key
    unsigned long long plan_key;  // the key of this call's arguments (plan_key below)
    int *counter;
    const float *q_rscale;     // FP8: 2^-qexp per query row
    int B, T, H, HB, G, R;
    long long num_pages;
    int oob_row;               // a TMA row coordinate past the pool (zero fill)
    int tok_n;                 // 0: page-interleaved positions; N: token-interleaved with N ranks
    float sl2;                 // softmax_scale * kappa * log2(e)
    float out_scale;           // kappa (BF16) or kappa / 256 (FP8) applied to O
    float *o_part, *lse_part, *part_o, *part_lse;
    int32_t *dev_error;
    unsigned long long wait_limit_ns;
};

// ---------------------------------------------------------------------- warp reductions
// Reduce-scatter over the warp: on entry each lane holds the 32 column values of its token;
// on exit lane L holds the reduction over the warp's 32 tokens of column L (31 shuffles
// instead of 32 x 5 for a plain butterfly).
template <bool kMax>
__device__ __forceinline__ float rs_op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }

// Same for 16 columns: lanes 2c and 2c+1 both return column c's reduction (16 shuffles).
template <bool kMax>
__device__ __forceinline__ float reduce_scatter16(const float (&v)[16], int lane) {
    float r[8];
    {
        const bool upper = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float send = upper ? v[i] : v[i + 8];
            const float keep = upper ? v[i + 8] : v[i];
            r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
    }
#pragma unroll
    for (int half = 4, off = 8; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < half) {
                const float send = upper ? r[i] : r[i + half];
                const float keep = upper ? r[i + half] : r[i];
                r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, off));
            }
        }
    }
    return rs_op<kMax>(r[0], __shfl_xor_sync(0xffffffffu, r[0], 1));
}

template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(const float (&v)[32], int lane) {
    float r[16];
    {
        const bool upper = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float send = upper ? v[i] : v[i + 16];
            const float keep = upper ? v[i + 16] : v[i];
            r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
    }
#pragma unroll
    for (int half = 8, off = 8; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < half) {
                const float send = upper ? r[i] : r[i + half];
                const float keep = upper ? r[i + half] : r[i];
                r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, off));
            }
        }
    }
    return r[0];
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A plan stored in the workspace carries a key of the arguments it was made for (sizes, DCP
// size, dtype, pool slots, rank selection, layout) and the page table's last CSR offset.  A run
// whose own key or table differs, or a workspace that holds no plan, is refused on the device:
// DCP_DEVERR_PLAN_MISMATCH, and no unit is run.
constexpr int kPlanMagic = 0x44435031;  // "DCP1"

__device__ __forceinline__ bool plan_matches(const int *ctrl, unsigned long long key, const int64_t *req_page_ptr,
                                             int B) {
    const unsigned long long k = *reinterpret_cast<const unsigned long long *>(ctrl + 4);
    const long long last = *reinterpret_cast<const long long *>(ctrl + 6);
    return ctrl[3] == kPlanMagic && k == key && last == (long long)req_page_ptr[B];
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int32_t *err, uint64_t lim) {
    const bool ok = mbar_wait(bar, parity, abort, err, lim);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// E4M3 hi/lo split of 4 values (already scaled into range): hi = e4m3(x), lo = e4m3(x - hi).
__device__ __forceinline__ void split_e4m3x4(float a, float b, float c, float d, uint32_t &hi, uint32_t &lo) {
    const __nv_fp8x2_storage_t h01 = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t h23 = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw r01 = __nv_cvt_fp8x2_to_halfraw2(h01, __NV_E4M3);
    const __half2_raw r23 = __nv_cvt_fp8x2_to_halfraw2(h23, __NV_E4M3);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&r01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&r23));
    const __nv_fp8x2_storage_t l01 = __nv_cvt_float2_to_fp8x2(make_float2(a - f01.x, b - f01.y), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t l23 = __nv_cvt_float2_to_fp8x2(make_float2(c - f23.x, d - f23.y), __NV_SATFINITE, __NV_E4M3);
    hi = (uint32_t)h01 | ((uint32_t)h23 << 16);
    lo = (uint32_t)l01 | ((uint32_t)l23 << 16);
}

// FP8 path: Q (BF16) -> hi and lo E4M3 rows scaled by a power of two per row so that the
// row's largest magnitude lands in (224, 448]; q = (hi + lo) * 2^-qexp up to ~2^-8 relative.
// One warp per query row.  Output rows [0, R) = hi, [R, 2R) = lo; rscale[row] = 2^-qexp.
__device__ void q_split_row(int row, int R, const __nv_bfloat16 *__restrict__ q, uint8_t *__restrict__ qhl,
                            float *__restrict__ rscale) {
    const int lane = threadIdx.x & 31;
    const __nv_bfloat16 *src = q + (long long)row * kKDim;
    float v[18];
#pragma unroll
    for (int k = 0; k < 9; ++k) {  // lane covers columns 2*(lane + 32k), +1
        const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162 *>(src)[lane + 32 * k];
        v[2 * k] = __bfloat162float(x.x);
        v[2 * k + 1] = __bfloat162float(x.y);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 18; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;
    if (amax > 0.f) {
        e = (int)floorf(log2f(448.f / amax));
        e = max(-100, min(100, e));
    }
    const float sc = ldexpf(1.f, e);
    uint8_t *hi = qhl + (long long)row * kKDim;
    uint8_t *lo = qhl + ((long long)R + row) * kKDim;
#pragma unroll
    for (int k = 0; k < 9; ++k) {
        const int c = 2 * (lane + 32 * k);
        const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * k] * sc, v[2 * k + 1] * sc),
                                                                __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
        const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(
            make_float2(v[2 * k] * sc - hf.x, v[2 * k + 1] * sc - hf.y), __NV_SATFINITE, __NV_E4M3);
        *reinterpret_cast<__nv_fp8x2_storage_t *>(hi + c) = h;
        *reinterpret_cast<__nv_fp8x2_storage_t *>(lo + c) = l;
    }
    if (lane == 0) rscale[row] = ldexpf(1.f, -e);
}

template <bool F8>
__global__ void __launch_bounds__(kThreads, 1)
attn_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ KParams p) {
    using C = Cfg<F8>;
    constexpr float kLazyTau = C::kLazyTauV;
    extern __shared__ uint8_t smem_raw[];
    if (C::kPad == 0 && (smem_u32(smem_raw) & 1023u) != 0) {  // (uniform: every CTA returns)
        if (threadIdx.x == 0 && p.dev_error) atomicOr(p.dev_error, DCP_DEVERR_LAYOUT);
        return;
    }
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kring = base;
    uint8_t *vring = base + C::kOffV;
    uint8_t *sq = base + C::kOffQ;
    uint8_t *sp = base + C::kOffP;
    Ctl *ctl = reinterpret_cast<Ctl *>(base + C::kOffCtl);
    constexpr int kKSlots = C::kKSlots;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &ctl->abort_flag;
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKSlots; ++i) {
            mbar_init(&ctl->kfull[i], 1);
            mbar_init(&ctl->kempty[i], 1);
        }
        for (int i = 0; i < C::kVSlots; ++i) {
            mbar_init(&ctl->vfull[i], 1);
            mbar_init(&ctl->vempty[i], 1);
        }
        mbar_init(&ctl->vland, 1);
        mbar_init(&ctl->rfull, 1);
        mbar_init(&ctl->rempty, 1);
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(&ctl->s_full[i], 1);
            mbar_init(&ctl->s_free[i], kSoftmaxWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->unit_full[i], 1);
            mbar_init(&ctl->unit_empty[i], 7);
        }
        mbar_init(&ctl->p_full[0], kSoftmaxWarps);
        mbar_init(&ctl->p_full[1], kSoftmaxWarps);
        mbar_init(&ctl->o_done[0], 1);
        mbar_init(&ctl->o_done[1], 1);
        mbar_init(&ctl->o_free, kSoftmaxWarps);
        mbar_init(&ctl->drain_s, 1);
        mbar_init(&ctl->drain_pv, 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_wait();  // the plan (and the FP8 Q split) of this call
    grid_dep_launch();
    const uint32_t tmem = ctl->tmem_base;
    // CTA i's first unit is unit i (the queue's first round gives every CTA one unit): its record
    // is read while the plan is checked, and the atomic counter serves the later units only.
    int4 first_rec = make_int4(0, 0, 0, 0);
    if (warp == 0 && lane == 0) first_rec = p.units[blockIdx.x];  // in bounds: grid <= the unit capacity
    const bool plan_ok = plan_matches(p.ctrl, p.plan_key, p.req_page_ptr, p.B);
    if (!plan_ok && blockIdx.x == 0 && threadIdx.x == 0 && p.dev_error) atomicOr(p.dev_error, DCP_DEVERR_PLAN_MISMATCH);
    const int n_units = plan_ok ? p.ctrl[0] : 0;

    // Consumer side of the unit ring (S issuer, V producer, PV issuer): returns false at the
    // end of the work or on abort.
    auto next_unit = [&](uint32_t &k, UnitInfo &u) -> bool {
        const int e = k & 1;
        if (!mbar_wait(&ctl->unit_full[e], (k >> 1) & 1, abort_flag, p.dev_error, lim)) return false;
        u = ctl->unit[e];
        mbar_arrive(&ctl->unit_empty[e]);
        ++k;
        return u.valid != 0;
    };
    // Pool rows of a tile's two pages (a missing second page: a row past the pool, which the
    // TMA fills with zeros).  The producers load them a tile ahead, off their critical path.
    auto tile_rows = [&](const UnitInfo &u, int tile, int &r0, int &r1) {
        const int pg = 2 * tile;
        r0 = p.comp_slot[u.comp_base + pg] * 64;
        r1 = (pg + 1 < u.n_pages) ? p.comp_slot[u.comp_base + pg + 1] * 64 : p.oob_row;
    };
    auto tile_pages = [&](const UnitInfo &u, int tile, int &ja, int &jb) {
        const int pg = 2 * tile;
        ja = p.comp_page[u.comp_base + pg];
        jb = (pg + 1 < u.n_pages) ? p.comp_page[u.comp_base + pg + 1] : -1;
    };
    // Rows of the page with index j (within the request) that hold positions < seq.  Rows past
    // the request's length are not part of the sequence and may hold any bytes (NaN included):
    // P is zero there, but 0 x NaN would reach O, so the stream that feeds P*V clears them in
    // shared memory before releasing the block (it lands on vland first).
    auto valid_rows = [&](int j, int seq) -> int {
        long long nv;
        if (p.tok_n == 0) {
            nv = (long long)seq - 64LL * j;
        } else {
            const int c = j % p.tok_n;
            nv = seq > c ? ((long long)seq - c + p.tok_n - 1) / p.tok_n - 64LL * (j / p.tok_n) : 0;
        }
        return (int)(nv < 0 ? 0 : nv > 64 ? 64 : nv);
    };
    // Clear rows [nv, 64) of both pages of one 16 KB block ([page][64 rows][128 B]; a 128-byte row
    // of a block is contiguous whatever the swizzle).
    auto clear_tail = [&](uint8_t *blk, int nv0, int nv1) {
#pragma unroll 1
        for (int pg = 0; pg < 2; ++pg) {
            uint4 *row = reinterpret_cast<uint4 *>(blk + pg * 8192);
            for (int e = (pg ? nv1 : nv0) * 8; e < 64 * 8; ++e) row[e] = make_uint4(0, 0, 0, 0);
        }
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- K-stream TMA
        if (lane == 0) {
            prefetch_tmap(&maps.q[0]);
            // K rows are read again: from L2 by the V stream (separate V ring), or by the other
            // query groups of the same chunk (q_len > 1 or more than 64 heads).  Otherwise (the
            // unified ring, one query group) each row is read once.
            const uint64_t pol = (C::kUnified && p.G == 1) ? make_policy_evict_first() : make_policy_evict_last();
            uint32_t kpos = 0, q_cnt = 0, k = 0, rpos = 0, land_cnt = 0;
            uint32_t via_land = 0;  // unified ring: bit per slot, its latest block went through vland
            bool ok = true, land_pending = false;
            while (ok) {
                const int e = k & 1;
                if (!mbar_wait(&ctl->unit_empty[e], ((k >> 1) & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                // (no plan: no workspace write)
                const int idx = n_units <= 0 ? 0 : k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.counter, 1);
                UnitInfo u;
                u.valid = idx < n_units;
                if (u.valid) {
                    const int4 rec = k == 0 ? first_rec : p.units[idx];
                    const int pair = rec.x / p.G;
                    u.g = rec.x - pair * p.G;
                    u.d = pair / p.B;
                    u.b = pair - u.d * p.B;
                    const int t = u.g / p.HB, hb = u.g - (u.g / p.HB) * p.HB;
                    u.n_pages = rec.z;
                    u.out_index = rec.w;
                    u.limit = p.seq_lens[u.b] - p.T + t;
                    u.q_row0 = (u.b * p.T + t) * p.H + hb * kGroupRows;
                    u.rows_valid = min(kGroupRows, p.H - hb * kGroupRows);
                    u.comp_base = (long long)u.d * p.num_pages + p.req_page_ptr[u.b] + rec.y;
                }
                ctl->unit[e] = u;
                mbar_arrive(&ctl->unit_full[e]);
                ++k;
                if (!u.valid) break;
                const int nt = (u.n_pages + 1) >> 1;
                if (nt == 0) continue;
                if (!mbar_wait(&ctl->q_empty, (q_cnt & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                ++q_cnt;
                mbar_arrive_expect_tx(&ctl->q_full, kQBytes);
                if (F8) {
                    for (int b = 0; b < 4; ++b) {
                        tma_load_2d(sq + b * 16384, &maps.q[0], &ctl->q_full, b * 128, u.q_row0);
                        tma_load_2d(sq + b * 16384 + 8192, &maps.q[0], &ctl->q_full, b * 128, p.R + u.q_row0);
                    }
                    tma_load_2d(sq + 65536, &maps.q[1], &ctl->q_full, 512, u.q_row0);
                    tma_load_2d(sq + 65536 + 4096, &maps.q[1], &ctl->q_full, 512, p.R + u.q_row0);
                } else {
                    for (int kb = 0; kb < 9; ++kb)
                        tma_load_2d(sq + kb * 8192, &maps.q[0], &ctl->q_full, kb * 64, u.q_row0);
                }
                const CUtensorMap *km = maps.kv[u.d];
                int rn0, rn1, jn0 = 0, jn1 = -1;
                const int seq = p.seq_lens[u.b];
                tile_rows(u, 0, rn0, rn1);
                if (C::kUnified) tile_pages(u, 0, jn0, jn1);
                for (int i = 0; i < nt && ok; ++i) {
                    const int r0 = rn0, r1 = rn1;
                    int nv0 = 64, nv1 = 64;
                    if (C::kUnified) {
                        nv0 = valid_rows(jn0, seq);
                        nv1 = jn1 >= 0 ? valid_rows(jn1, seq) : 64;  // a missing page is zero-filled
                    }
                    if (i + 1 < nt) {  // the next tile's page metadata, a tile ahead
                        tile_rows(u, i + 1, rn0, rn1);
                        if (C::kUnified) tile_pages(u, i + 1, jn0, jn1);
                    }
                    const bool fix = nv0 < 64 || nv1 < 64;
                    for (int kb = 0; kb < C::kKBlocks; ++kb) {
                        if (C::kUnified && kb == 4) {  // rope: 64 dims, 64-byte swizzle, 4 KB per page
                            if (!mbar_wait(&ctl->rempty, (rpos & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                                ok = false;
                                break;
                            }
                            ++rpos;
                            uint8_t *dst = kring + C::kOffRope;
                            mbar_arrive_expect_tx(&ctl->rfull, 8192);
                            tma_load_2d_hint(dst, &km[1], &ctl->rfull, 512, r0, pol);
                            tma_load_2d_hint(dst + 4096, &km[1], &ctl->rfull, 512, r1, pol);
                            continue;
                        }
                        const uint32_t slot = kpos % kKSlots;
                        if (!mbar_wait(&ctl->kempty[slot], ((kpos / kKSlots) & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                            ok = false;
                            break;
                        }
                        ++kpos;
                        uint8_t *dst = kring + slot * kKSlotBytes;
                        if (F8 && kb == 4) {  // rope: 64 dims, 64-byte swizzle, 4 KB per page
                            mbar_arrive_expect_tx(&ctl->kfull[slot], 8192);
                            tma_load_2d_hint(dst, &km[1], &ctl->kfull[slot], 512, r0, pol);
                            tma_load_2d_hint(dst + 4096, &km[1], &ctl->kfull[slot], 512, r1, pol);
                        } else {
                            const int x = F8 ? kb * 128 : kb * 64;
                            // unified ring: a block with rows past the sequence serves P*V too
                            const bool via = C::kUnified && fix;
                            uint64_t *bar = via ? &ctl->vland : &ctl->kfull[slot];
                            if (C::kUnified) {
                                via_land = via ? (via_land | (1u << slot)) : (via_land & ~(1u << slot));
                                land_pending = via;
                            }
                            mbar_arrive_expect_tx(bar, kKSlotBytes);
                            tma_load_2d_hint(dst, &km[0], bar, x, r0, pol);
                            tma_load_2d_hint(dst + 8192, &km[0], bar, x, r1, pol);
                            if (via) {
                                if (!mbar_wait(&ctl->vland, land_cnt & 1, abort_flag, p.dev_error, lim)) {
                                    ok = false;
                                    break;
                                }
                                ++land_cnt;
                                land_pending = false;
                                clear_tail(dst, nv0, nv1);
                                fence_proxy_async_smem();
                                mbar_arrive(&ctl->kfull[slot]);
                            }
                        }
                    }
                }
            }
            if (!ok) {  // let issued TMA copies land before the CTA can exit (bounded waits)
                int never = 0;
                for (uint32_t q = kpos > (uint32_t)kKSlots ? kpos - kKSlots : 0; q < kpos; ++q)
                    if (!((via_land >> (q % kKSlots)) & 1u))
                        mbar_wait(&ctl->kfull[q % kKSlots], (q / kKSlots) & 1, &never, nullptr, lim);
                if (land_pending) mbar_wait(&ctl->vland, land_cnt & 1, &never, nullptr, lim);
                if (rpos > 0) mbar_wait(&ctl->rfull, (rpos - 1) & 1, &never, nullptr, lim);
                if (q_cnt > 0) mbar_wait(&ctl->q_full, (q_cnt - 1) & 1, &never, nullptr, lim);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- score MMAs
        if (lane == 0) {
            uint32_t kpos = 0, s_cnt = 0, q_cnt = 0, k = 0, rpos = 0;
            bool ok = true;
            const uint32_t kaddr = smem_u32(kring), q_addr = smem_u32(sq);
            UnitInfo u;
            while (ok && next_unit(k, u)) {
                const int nt = (u.n_pages + 1) >> 1;
                if (nt == 0) continue;
                if (!mbar_wait(&ctl->q_full, q_cnt & 1, abort_flag, p.dev_error, lim)) break;
                ++q_cnt;
                tc_fence_after();
                for (int i = 0; i < nt && ok; ++i) {
                    const uint32_t sb = s_cnt % C::kSBufs;
                    if (!mbar_wait(&ctl->s_free[sb], ((s_cnt / C::kSBufs) & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                        ok = false;
                        break;
                    }
                    ++s_cnt;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + kSCol + C::kSCols * sb;
                    for (int kb = 0; kb < C::kKBlocks; ++kb) {
                        const bool rope_slot = C::kUnified && kb == 4;
                        const uint32_t slot = kpos % kKSlots;
                        if (rope_slot ? !mbar_wait(&ctl->rfull, rpos & 1, abort_flag, p.dev_error, lim)
                                      : !mbar_wait(&ctl->kfull[slot], (kpos / kKSlots) & 1, abort_flag, p.dev_error, lim)) {
                            ok = false;
                            break;
                        }
                        if (rope_slot) ++rpos;
                        else ++kpos;
                        tc_fence_after();
                        const uint32_t a0 = rope_slot ? kaddr + C::kOffRope : kaddr + slot * kKSlotBytes;
                        if (F8) {
                            if (kb < 4) {
                                const uint32_t b0 = q_addr + kb * 16384;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_f8_ss(d_tmem, smem_desc(a0 + kk * 32, 16, 1024, kSwizzle128),
                                              smem_desc(b0 + kk * 32, 16, 1024, kSwizzle128), C::kIdescS,
                                              (kb | kk) != 0);
                            } else {
                                const uint32_t b0 = q_addr + 65536;
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    mma_f8_ss(d_tmem, smem_desc(a0 + kk * 32, 16, 512, kSwizzle64),
                                              smem_desc(b0 + kk * 32, 16, 512, kSwizzle64), C::kIdescS, 1);
                            }
                        } else {
                            const uint32_t b0 = q_addr + kb * 8192;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_f16_ss(d_tmem, smem_desc(a0 + kk * 32, 16, 1024, kSwizzle128),
                                           smem_desc(b0 + kk * 32, 16, 1024, kSwizzle128), C::kIdescS,
                                           (kb | kk) != 0);
                        }
                        // unified ring: the latent blocks stay until P*V has read them
                        if (rope_slot) mma_commit(&ctl->rempty);
                        else if (!C::kUnified) mma_commit(&ctl->kempty[slot]);
                    }
                    if (!ok) break;
                    mma_commit(&ctl->s_full[sb]);
                    if (i == nt - 1) mma_commit(&ctl->q_empty);
                }
            }
            mma_commit(&ctl->drain_s);
            int never = 0;
            mbar_wait(&ctl->drain_s, 0, &never, nullptr, 100000000ull);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- V-stream TMA
        // (unified ring: no V stream; the warp only follows the unit ring)
        if constexpr (C::kUnified) {
            if (lane == 0) {
                uint32_t k = 0;
                UnitInfo u;
                while (next_unit(k, u)) {
                }
            }
        } else if (lane == 0) {
            const uint64_t pol = make_policy_evict_first();
            uint32_t vpos = 0, k = 0, land_cnt = 0;
            bool ok = true, land_pending = false;
            uint32_t via_land = 0;  // bit per slot: its latest unit went through vland
            UnitInfo u;
            while (ok && next_unit(k, u)) {
                const int nt = (u.n_pages + 1) >> 1;
                const CUtensorMap *km = &maps.kv[u.d][0];
                if (nt == 0) continue;
                const int seq = p.seq_lens[u.b];
                int rn0, rn1, jn0, jn1;
                tile_rows(u, 0, rn0, rn1);
                tile_pages(u, 0, jn0, jn1);
                for (int i = 0; i < nt && ok; ++i) {
                    const int r0 = rn0, r1 = rn1;
                    const int nv0 = valid_rows(jn0, seq);
                    const int nv1 = jn1 >= 0 ? valid_rows(jn1, seq) : 64;  // a missing page is zero-filled
                    if (i + 1 < nt) {
                        tile_rows(u, i + 1, rn0, rn1);
                        tile_pages(u, i + 1, jn0, jn1);
                    }
                    const bool fix = nv0 < 64 || nv1 < 64;
                    for (int vu = 0; vu < C::kVUnits; ++vu) {
                        const uint32_t slot = vpos % C::kVSlots;
                        if (!mbar_wait(&ctl->vempty[slot], ((vpos / C::kVSlots) & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                            ok = false;
                            break;
                        }
                        ++vpos;
                        uint8_t *dst = vring + slot * C::kVSlotBytes;
                        uint64_t *bar = fix ? &ctl->vland : &ctl->vfull[slot];
                        via_land = fix ? (via_land | (1u << slot)) : (via_land & ~(1u << slot));
                        land_pending = fix;
                        mbar_arrive_expect_tx(bar, C::kVSlotBytes);
                        // the slot holds kBoxCols columns of 128-byte boxes (64 BF16 / 128 E4M3
                        // dims), each of both pages: [box column][page][64 rows][128 B]
                        constexpr int kBoxCols = (int)(C::kVSlotBytes / 16384);
                        const int w = F8 ? 128 : 64;
#pragma unroll
                        for (int h = 0; h < kBoxCols; ++h) {
                            const int x = (kBoxCols * vu + h) * w;
                            tma_load_2d_hint(dst + h * 16384, km, bar, x, r0, pol);
                            tma_load_2d_hint(dst + h * 16384 + 8192, km, bar, x, r1, pol);
                        }
                        if (fix) {
                            if (!mbar_wait(&ctl->vland, land_cnt & 1, abort_flag, p.dev_error, lim)) {
                                ok = false;
                                break;
                            }
                            ++land_cnt;
                            land_pending = false;
#pragma unroll 1
                            for (int h = 0; h < kBoxCols; ++h) clear_tail(dst + h * 16384, nv0, nv1);
                            fence_proxy_async_smem();
                            mbar_arrive(&ctl->vfull[slot]);
                        }
                    }
                }
            }
            if (!ok) {  // let issued TMA copies land before the CTA can exit (bounded waits)
                int never = 0;
                for (uint32_t q = vpos > (uint32_t)C::kVSlots ? vpos - C::kVSlots : 0; q < vpos; ++q)
                    if (!((via_land >> (q % C::kVSlots)) & 1u))
                        mbar_wait(&ctl->vfull[q % C::kVSlots], (q / C::kVSlots) & 1, &never, nullptr, lim);
                if (land_pending) mbar_wait(&ctl->vland, land_cnt & 1, &never, nullptr, lim);
            }
        }
    } else if (warp == 3) {
        // ---------------------------------------------------------------- P*V MMAs
        if (lane == 0) {
            uint32_t vpos = 0, p_cnt = 0, of_cnt = 0, k = 0;
            bool had_tiles = false, ok = true;
            const uint32_t vaddr = smem_u32(vring), p_addr = smem_u32(sp), kaddr = smem_u32(kring);
            UnitInfo u;
            while (ok && next_unit(k, u)) {
                const int nt = (u.n_pages + 1) >> 1;
                if (nt == 0) continue;
                for (int i = 0; i < nt && ok; ++i) {
                    if (!mbar_wait(&ctl->p_full[p_cnt & 1], (p_cnt >> 1) & 1, abort_flag, p.dev_error, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tile_g = p_cnt++;  // global tile index: P buffer, o_done parity
                    const uint32_t pb = p_addr + (tile_g % C::kPBufs) * kPBytes;
                    if (i == 0 && had_tiles) {
                        if (!mbar_wait(&ctl->o_free, of_cnt & 1, abort_flag, p.dev_error, lim)) {
                            ok = false;
                            break;
                        }
                        ++of_cnt;
                    }
                    tc_fence_after();
                    if constexpr (C::kUnified) {
                        // the tile's four latent blocks, still in the ring since its score MMAs
                        for (int m = 0; m < 4; ++m) {
                            const uint32_t slot = vpos % kKSlots;
                            if (!mbar_wait(&ctl->kfull[slot], (vpos / kKSlots) & 1, abort_flag, p.dev_error, lim)) {
                                ok = false;
                                break;
                            }
                            ++vpos;
                            tc_fence_after();
                            const uint32_t a0 = kaddr + slot * kKSlotBytes;
                            const uint32_t d_tmem = tmem + 64 * m;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t ad = smem_desc(a0 + kk * 4096, 16384, 1024, kSwizzle128);
                                mma_f8_ss(d_tmem, ad, smem_desc(pb + kk * 2048, 512, 512, kSwizzle64), C::kIdescPV,
                                          !(i == 0 && kk == 0));
                                mma_f8_ss(d_tmem, ad, smem_desc(pb + 8192 + kk * 2048, 512, 512, kSwizzle64),
                                          C::kIdescPV, 1);
                            }
                            mma_commit(&ctl->kempty[slot]);
                        }
                    } else {
                        for (int vu = 0; vu < C::kVUnits; ++vu) {
                            const uint32_t slot = vpos % C::kVSlots;
                            if (!mbar_wait(&ctl->vfull[slot], (vpos / C::kVSlots) & 1, abort_flag, p.dev_error, lim)) {
                                ok = false;
                                break;
                            }
                            ++vpos;
                            tc_fence_after();
                            const uint32_t a0 = vaddr + slot * C::kVSlotBytes;
#pragma unroll
                            for (int mt = 0; mt < C::kVBlk; ++mt) {  // M-tiles (128 V dims each) of the slot
                                const uint32_t d_tmem = tmem + 64 * (C::kVBlk * vu + mt);
                                if (F8) {
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk) {
                                        const uint64_t ad = smem_desc(a0 + mt * 16384 + kk * 4096, 16384, 1024, kSwizzle128);
                                        mma_f8_ss(d_tmem, ad, smem_desc(pb + kk * 2048, 512, 512, kSwizzle64),
                                                  C::kIdescPV, !(i == 0 && kk == 0));
                                        mma_f8_ss(d_tmem, ad, smem_desc(pb + 8192 + kk * 2048, 512, 512, kSwizzle64),
                                                  C::kIdescPV, 1);
                                    }
                                } else {
#pragma unroll
                                    for (int kk = 0; kk < 8; ++kk)
                                        mma_f16_ss(d_tmem, smem_desc(a0 + mt * 32768 + kk * 2048, 16384, 1024, kSwizzle128),
                                                   smem_desc(pb + kk * 2048, 1024, 1024, kSwizzle128), C::kIdescPV,
                                                   !(i == 0 && kk == 0));
                                }
                            }
                            mma_commit(&ctl->vempty[slot]);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&ctl->o_done[tile_g & 1]);
                }
                had_tiles = true;
            }
            mma_commit(&ctl->drain_pv);
            int never = 0;
            mbar_wait(&ctl->drain_pv, 0, &never, nullptr, 100000000ull);
        }
    } else {
        // ---------------------------------------------------------------- softmax warps
        // Four independent warpgroups; warpgroup g owns query columns [16g, 16g + 16) of every
        // tile.  Within a warpgroup each thread owns one token row (TMEM lane).
        const int wg = (warp - 4) >> 2;             // 0..3
        const int gtid = threadIdx.x - 128 - 128 * wg;  // 0..127 within the warpgroup
        const int quad = warp & 3;                  // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;           // token row of the tile = TMEM lane
        const int c0 = kCols * wg;                  // first query column of this warpgroup
        const int bar_a = 1 + 2 * wg, bar_b = 2 + 2 * wg;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint32_t s_cnt = 0, obs_all = 0, k = 0;
        // P*V of global tile t commits o_done[t & 1]; completions are observed strictly in tile
        // order, so a barrier can never complete twice between two observations.
        auto wait_pv = [&](uint32_t t) -> bool {
            while (obs_all <= t) {
                if (!warp_wait(&ctl->o_done[obs_all & 1], (obs_all >> 1) & 1, abort_flag, p.dev_error, lim))
                    return false;
                ++obs_all;
            }
            return true;
        };
        while (true) {
            const int e = k & 1;
            int fail = !warp_wait(&ctl->unit_full[e], (k >> 1) & 1, abort_flag, p.dev_error, lim);
            if (named_bar_or(bar_a, 128, fail)) break;
            const UnitInfo u = ctl->unit[e];
            // Per-column score scale and reference maximum, in shared memory (read back as
            // vectors each tile; registers stay free for the scores).  The reference trails the
            // true running maximum by at most kLazyTau (log2 units): a tile whose scores all
            // stay within that margin is exponentiated against the old reference (weights up to
            // 2^kLazyTau, exact after the final normalisation) and skips the cross-thread
            // maximum and the O rescale.
            if (u.valid && gtid < kCols) {
                float qs = p.sl2;
                if (F8) {
                    const int qr = u.q_row0 + c0 + gtid;
                    qs *= (qr < p.R) ? __ldg(p.q_rscale + qr) : 0.f;
                }
                ctl->qscale[c0 + gtid] = qs;
                ctl->m_run[c0 + gtid] = -INFINITY;
            }
            named_bar_sync(bar_b, 128);
            if (gtid == 0) mbar_arrive(&ctl->unit_empty[e]);
            ++k;
            if (!u.valid) break;
            const int nt = (u.n_pages + 1) >> 1;
            const bool direct = u.out_index < 0;
            const long long out_row0 = direct
                ? ((long long)u.d * p.B * p.T * p.H + (long long)u.q_row0)
                : (long long)u.out_index * kGroupRows;
            float *obase = direct ? p.o_part : p.part_o;
            float *lbase = direct ? p.lse_part : p.part_lse;
            if (nt == 0) {
                for (int idx = gtid; idx < kCols * (kVDim / 4); idx += 128) {
                    const int c = c0 + idx / (kVDim / 4), v4 = idx % (kVDim / 4);
                    if (c < u.rows_valid)
                        reinterpret_cast<float4 *>(obase + (out_row0 + c) * kVDim)[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (gtid < kCols && c0 + gtid < u.rows_valid) lbase[out_row0 + c0 + gtid] = -INFINITY;
                continue;
            }
            float lp[kCols];
#pragma unroll
            for (int c = 0; c < kCols; ++c) lp[c] = 0.f;
            const float4 *qs4 = reinterpret_cast<const float4 *>(&ctl->qscale[c0]);
            const float4 *mr4 = reinterpret_cast<const float4 *>(&ctl->m_run[c0]);
            // page index of this row's page in tile 0, then prefetched one tile ahead
            int j_cur = -1;
            {
                const int pl = row >> 6;
                if (pl < u.n_pages) j_cur = p.comp_page[u.comp_base + pl];
            }
            bool aborted = false;
            for (int i = 0; i < nt; ++i) {
                int j_next = -1;
                {
                    const int pl = 2 * (i + 1) + (row >> 6);
                    if (i + 1 < nt && pl < u.n_pages) j_next = p.comp_page[u.comp_base + pl];
                }
                const uint32_t g = s_cnt;  // global tile index
                const uint32_t sb = s_cnt % C::kSBufs;
                fail = !warp_wait(&ctl->s_full[sb], (s_cnt / C::kSBufs) & 1, abort_flag, p.dev_error, lim);
                ++s_cnt;
                float s[kCols];
                int over = 0;
                if (!fail) {
                    tc_fence_after();
                    const uint32_t ta = tmem + lane_base + kSCol + C::kSCols * sb + c0;
                    tmem_ld16(ta, s);
                    if (F8) {
                        float t[kCols];
                        tmem_ld16(ta + 64, t);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < kCols; ++c) s[c] += t[c];
                    } else {
                        tmem_wait_ld();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->s_free[sb]);  // one arrival per warp
                    // mask: ragged last page / missing second page / causal limit
                    // position of this row: 64 j + r (page layout), or (64 (j div N) + r) N + j mod N
                    // (token layout: entry j = jj N + d is rank d's local page jj)
                    const long long pos = p.tok_n == 0 ? (long long)j_cur * 64 + (row & 63)
                        : ((long long)(j_cur / p.tok_n) * 64 + (row & 63)) * p.tok_n + (j_cur % p.tok_n);
                    const bool valid = j_cur >= 0 && pos <= (long long)u.limit;
#pragma unroll
                    for (int q = 0; q < kCols / 4; ++q) {
                        const float4 a = qs4[q], m = mr4[q];
                        const float av[4] = {a.x, a.y, a.z, a.w}, mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int c = 4 * q + k;
                            s[c] = valid ? s[c] * av[k] : -INFINITY;
                            over |= s[c] > mv[k] + kLazyTau;
                        }
                    }
                }
                j_cur = j_next;
                if (named_bar_or(bar_a, 128, fail | over)) {
                    if (named_bar_or(bar_b, 128, fail)) {
                        aborted = true;
                        break;
                    }
                    // slow path: exact column maxima of this tile, new references, rescale
                    const float r = reduce_scatter16<true>(s, lane);
                    if ((lane & 1) == 0) ctl->red[wg][quad][lane >> 1] = r;
                    named_bar_sync(bar_a, 128);
                    if (gtid < kCols) {
                        const int c = c0 + gtid;
                        const float mt = fmaxf(fmaxf(ctl->red[wg][0][gtid], ctl->red[wg][1][gtid]),
                                               fmaxf(ctl->red[wg][2][gtid], ctl->red[wg][3][gtid]));
                        const float mo = ctl->m_run[c];
                        const float mn = fmaxf(mo, mt);
                        ctl->m_run[c] = mn;
                        ctl->corr[c] = (mn == mo) ? 1.f : fast_exp2(mo - mn);
                    }
                    named_bar_sync(bar_b, 128);
                    float cr[kCols];
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        cr[c] = ctl->corr[c0 + c];
                        lp[c] *= cr[c];
                    }
                    if (i > 0) {  // the rescale needs P*V of the previous tile complete
                        fail = !wait_pv(g - 1);
                        if (fail) continue;  // the next OR-barrier takes the warpgroup out
                        tc_fence_after();
#pragma unroll 1
                        for (int j = 0; j < 4; ++j) {
                            float o[kCols];
                            const uint32_t ta = tmem + lane_base + 64 * j + c0;
                            tmem_ld16(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < kCols; ++c) o[c] *= cr[c];
                            tmem_st16(ta, o);
                        }
                        tmem_wait_st();
                    }
                }
                // The weights, packed for the MMA in registers first: only the stores wait for
                // the P buffer's previous reader (P*V of tile g - kPBufs), which keeps the exp2 and
                // the conversions off the P*V -> P -> P*V chain.
#pragma unroll
                for (int q = 0; q < kCols / 4; ++q) {
                    const float4 m = mr4[q];
                    const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = 4 * q + k;
                        const float ms = mv[k] == -INFINITY ? 0.f : mv[k];
                        s[c] = fast_exp2(s[c] - ms);
                        lp[c] += s[c];
                    }
                }
                uint4 w0, w1;  // FP8: hi and lo E4M3 terms; BF16: columns 0-7 and 8-15
                if (F8) {
                    split_e4m3x4(s[0] * kPScale, s[1] * kPScale, s[2] * kPScale, s[3] * kPScale, w0.x, w1.x);
                    split_e4m3x4(s[4] * kPScale, s[5] * kPScale, s[6] * kPScale, s[7] * kPScale, w0.y, w1.y);
                    split_e4m3x4(s[8] * kPScale, s[9] * kPScale, s[10] * kPScale, s[11] * kPScale, w0.z, w1.z);
                    split_e4m3x4(s[12] * kPScale, s[13] * kPScale, s[14] * kPScale, s[15] * kPScale, w0.w, w1.w);
                } else {
                    w0 = make_uint4(pack_bf16(s[0], s[1]), pack_bf16(s[2], s[3]), pack_bf16(s[4], s[5]),
                                    pack_bf16(s[6], s[7]));
                    w1 = make_uint4(pack_bf16(s[8], s[9]), pack_bf16(s[10], s[11]), pack_bf16(s[12], s[13]),
                                    pack_bf16(s[14], s[15]));
                }
                if (g >= (uint32_t)C::kPBufs) {
                    fail = !wait_pv(g - C::kPBufs);
                    if (fail) continue;
                    tc_fence_after();
                }
                if (F8) {
                    // P^T row as hi and lo E4M3 rows of 64 bytes, MN-major, 64-byte swizzle;
                    // this warpgroup writes 16-byte chunk wg of each.
                    const uint32_t off = (row >> 3) * 512 + (row & 7) * 64;
                    const uint32_t sw = ((wg ^ ((row >> 1) & 3)) << 4);
                    uint8_t *pbuf = sp + (g % C::kPBufs) * kPBytes;
                    *reinterpret_cast<uint4 *>(pbuf + off + sw) = w0;
                    *reinterpret_cast<uint4 *>(pbuf + 8192 + off + sw) = w1;
                } else {
                    // P^T row: 64 BF16 values, MN-major with the 128-byte swizzle; this
                    // warpgroup writes 16-byte chunks 2wg and 2wg + 1.
                    uint8_t *prow = sp + (g % C::kPBufs) * kPBytes + (row >> 3) * 1024 + (row & 7) * 128;
                    *reinterpret_cast<uint4 *>(prow + (((2 * wg) ^ (row & 7)) << 4)) = w0;
                    *reinterpret_cast<uint4 *>(prow + (((2 * wg + 1) ^ (row & 7)) << 4)) = w1;
                }
                fence_proxy_async_smem();  // every writer's P stores, for the MMA's async proxy
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->p_full[g & 1]);
            }
            if (aborted) break;
            fail = !wait_pv(s_cnt - 1);
            tc_fence_after();
            {
                const float r = reduce_scatter16<false>(lp, lane);
                if ((lane & 1) == 0) ctl->red[wg][quad][lane >> 1] = r;
            }
            if (named_bar_or(bar_a, 128, fail)) break;
            if (gtid < kCols) {
                const int c = c0 + gtid;
                const float L = ctl->red[wg][0][gtid] + ctl->red[wg][1][gtid] + ctl->red[wg][2][gtid] +
                                ctl->red[wg][3][gtid];
                const float mr = ctl->m_run[c];
                const bool live = L > 0.f;
                ctl->oscale[c] = live ? p.out_scale / L : 0.f;
                if (c < u.rows_valid)
                    lbase[out_row0 + c] = live ? (mr + log2f(L)) * 0.69314718055994531f : -INFINITY;
            }
            named_bar_sync(bar_b, 128);
            float osc[kCols];
#pragma unroll
            for (int c = 0; c < kCols; ++c) osc[c] = ctl->oscale[c0 + c];
            // O^T from TMEM, one 128-dim block at a time; the next block's load is in flight
            // while this block's stores issue
            float oa[kCols], ob[kCols];
            tmem_ld16(tmem + lane_base + c0, oa);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float(&cur)[kCols] = (j & 1) ? ob : oa;
                float(&nxt)[kCols] = (j & 1) ? oa : ob;
                if (j + 1 < 4) tmem_ld16(tmem + lane_base + 64 * (j + 1) + c0, nxt);
                const int vcol = j * 128 + row;  // V dimension held by this lane
#pragma unroll
                for (int c = 0; c < kCols; ++c)
                    if (c0 + c < u.rows_valid)
                        obase[(out_row0 + c0 + c) * kVDim + vcol] = cur[c] * osc[c];
                if (j + 1 < 4) tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->o_free);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------ plan
// Per-rank compaction of every request's pages over tiles of 1024 pages of one request, in
// two launches:
//   plan_count_kernel  owner counts per tile (extra blocks: the FP8 Q split);
//   plan_build_kernel  one block per tile: each page to (pages of its owner in the request's
//                      earlier tiles) + (stable rank among same-owner pages of its tile); the
//                      last block: per (rank, request) totals, chunks, partial slots and the
//                      unit list.
// Rank d's pages of request b end up, in page order, at d * num_pages + req_page_ptr[b] + pos.
constexpr int kPlanTile = 1024;
constexpr int kPlanThreads = 512;

__device__ __forceinline__ int page_owner_slot(int v, int N, long long slots_per_rank, int &slot) {
    const int d = N <= 1 ? 0 : v % N;
    const long long s = N <= 1 ? (long long)v : (long long)(v / N);
    if (v < 0 || s >= slots_per_rank) return -1;
    slot = (int)s;
    return d;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_count_kernel(int N, long long slots_per_rank, int tiles_per_req, int tile_stride, int n_tile_blocks,
                  const int64_t *__restrict__ req_page_ptr, const int32_t *__restrict__ vpages,
                  int32_t *__restrict__ tile_cnt, int32_t *dev_error, int R, const __nv_bfloat16 *__restrict__ q,
                  uint8_t *__restrict__ qhl, float *__restrict__ rscale, const int *__restrict__ run_ctrl,
                  unsigned long long key, int B) {
    grid_dep_wait();
    grid_dep_launch();
    if ((int)blockIdx.x >= n_tile_blocks) {  // FP8 Q split: one warp per query row
        // a run of a stored plan (run_ctrl set) writes nothing when the workspace holds no plan for it
        if (run_ctrl && !plan_matches(run_ctrl, key, req_page_ptr, B)) return;
        const int row = ((int)blockIdx.x - n_tile_blocks) * (kPlanThreads / 32) + (int)(threadIdx.x >> 5);
        if (row < R) q_split_row(row, R, q, qhl, rscale);
        return;
    }
    __shared__ int cnt[kMaxDcpAttn];
    const int b = blockIdx.x / tile_stride, k0 = blockIdx.x % tile_stride;
    const long long r0 = req_page_ptr[b], r1 = req_page_ptr[b + 1];
    bool bad = false;
    for (int k = k0; r0 + (long long)k * kPlanTile < r1; k += tile_stride) {  // block-uniform
        const long long p0 = r0 + (long long)k * kPlanTile;
        if (threadIdx.x < kMaxDcpAttn) cnt[threadIdx.x] = 0;
        __syncthreads();
        for (int e = 0; e < kPlanTile / kPlanThreads; ++e) {
            const long long i = p0 + e * kPlanThreads + threadIdx.x;
            if (i < r1) {
                int slot;
                const int d = page_owner_slot(vpages[i], N, slots_per_rank, slot);
                if (d < 0) bad = true;
                else atomicAdd(&cnt[d], 1);
            }
        }
        __syncthreads();
        if (threadIdx.x < N) tile_cnt[((long long)b * tiles_per_req + k) * kMaxDcpAttn + threadIdx.x] = cnt[threadIdx.x];
    }
    if (bad && dev_error) atomicOr(dev_error, DCP_DEVERR_OUT_OF_RANGE);
}

// Exclusive scan of one value per thread over the block (blockDim.x a multiple of 32).
__device__ long long block_exclusive_scan(long long x, long long *scratch, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const long long t = lane < nw ? scratch[lane] : 0;
        long long s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) scratch[lane] = s - t;
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    const long long r = scratch[warp] + incl - x;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// One block per 1024-page tile of a request: stable scatter of its pages.
__device__ void plan_scatter_tile(int b, int k, int N, long long num_pages, long long slots_per_rank,
                                  int tiles_per_req, const int64_t *__restrict__ req_page_ptr,
                                  const int32_t *__restrict__ vpages, const int32_t *__restrict__ tile_cnt,
                                  int32_t *__restrict__ comp_slot, int32_t *__restrict__ comp_page) {
    __shared__ int wcnt[kPlanThreads / 32][kMaxDcpAttn];
    __shared__ int run[kMaxDcpAttn];
    const long long r0 = req_page_ptr[b];
    const long long p0 = r0 + (long long)k * kPlanTile, p1 = req_page_ptr[b + 1];
    if (p0 >= p1) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();  // the previous tile of this block is done with run[] and wcnt[]
    if (threadIdx.x < kMaxDcpAttn) {
        int base = 0;  // pages of this owner in the request's earlier tiles
        if (threadIdx.x < N)
            for (int kk = 0; kk < k; ++kk) base += tile_cnt[((long long)b * tiles_per_req + kk) * kMaxDcpAttn + threadIdx.x];
        run[threadIdx.x] = base;
    }
    for (int e = 0; e < kPlanTile / kPlanThreads; ++e) {
        const long long i = p0 + e * kPlanThreads + threadIdx.x;
        int d = -1, slot = 0;
        if (i < p1) d = page_owner_slot(vpages[i], N, slots_per_rank, slot);
        int my_rank_in_warp = 0;
        for (int dd = 0; dd < N; ++dd) {
            const unsigned m = __ballot_sync(0xffffffffu, d == dd);
            if (lane == 0) wcnt[warp][dd] = __popc(m);
            if (d == dd) my_rank_in_warp = __popc(m & ((1u << lane) - 1u));
        }
        __syncthreads();
        if (d >= 0) {
            int before = run[d];
            for (int w = 0; w < warp; ++w) before += wcnt[w][d];
            const long long pos = (long long)d * num_pages + r0 + before + my_rank_in_warp;
            comp_slot[pos] = slot;
            comp_page[pos] = (int)(i - r0);
        }
        __syncthreads();
        if (threadIdx.x < N) {
            int t = 0;
            for (int w = 0; w < kPlanThreads / 32; ++w) t += wcnt[w][threadIdx.x];
            run[threadIdx.x] += t;
        }
        __syncthreads();
    }
}

// The last block of plan_build_kernel: chunk each (rank, request) pair, emit units largest first
// with the G query groups of a chunk adjacent, cut the chunks of the queue's last, partly
// filled round into pieces (below), assign partial slots and list the multi-piece pairs.
//
// Tail cut.  Persistent CTAs take units from the queue in order, so with U units of similar
// size on P SMs the last U mod P of them run while the other SMs idle (48 requests x 8 ranks of
// 98 tiles on 152 SMs: 80 SMs run a third unit after the others are done).  The chunks from the
// first position of that round on -- the smallest, ties taken by the highest (request, rank,
// chunk), so that the cut pairs gather in few requests and the other requests' rows merge
// while the chunk partials combine -- are laid end to end in (size descending, request, rank,
// chunk) order and cut at the multiples of
// q = their work / P; each piece is a unit with a partial of its own (merged like chunks), and
// the pieces take the tail of the queue largest first.  Which chunks are cut, where, and the
// order of a pair's partials do not depend on thread timing, so results are reproducible.
// Only where the largest of those chunks is well above q (a cut costs a partial's round trip
// and a unit boundary, about three tiles) and the pieces fit the workspace.
constexpr int kMinPiece = 8;
constexpr int kMaxTailChunks = kPlanThreads;  // one thread per tail chunk in the sort and scans
__device__ void plan_build_units(int B, int N, int G, int only_rank, int tpc, int num_sms, long long max_units,
                                 long long max_partials, unsigned long long key,
                                 const int64_t *__restrict__ req_page_ptr,
                                 int tiles_per_req, const int32_t *__restrict__ tile_cnt, int32_t *__restrict__ counts,
                                 int32_t *__restrict__ pair_chunks, int32_t *__restrict__ pair_part,
                                 int32_t *__restrict__ multi_list, int4 *__restrict__ units, int *__restrict__ ctrl) {
    __shared__ int hist[kMaxTpc + 1];                    // chunks per size, then next queue position per size
    __shared__ unsigned long long tkey[kMaxTailChunks];  // tail chunk: (kMaxTpc - size) << 32 | b * N + d
    __shared__ int tchunk[kMaxTailChunks];               // tail chunk: chunk index within its pair
    __shared__ int tpieces[kMaxTailChunks];
    __shared__ long long scratch[33];
    __shared__ int n_multi, n_tail, n_extra, u_c, q_cut, tail_start, s_b, b_first;
    __shared__ unsigned long long part_before;
    const int n_pair = N * B;
    const int tid = threadIdx.x;
    auto active = [&](int pr) { return only_rank < 0 || pr / B == only_rank; };
    auto n_chunks = [&](int tiles) { return tiles == 0 ? 1 : (tiles + tpc - 1) / tpc; };
    auto chunk_size = [&](int tiles, int c) { return max(0, min(tpc, tiles - c * tpc)); };
    if (tid == 0) {
        n_multi = 0;
        n_tail = 0;
        n_extra = 0;
        part_before = 0;
    }
    for (int i = tid; i <= tpc; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int pr = tid; pr < n_pair; pr += blockDim.x) {  // per (rank, request): pages, chunks
        const int d = pr / B, b = pr % B;
        const long long np = req_page_ptr[b + 1] - req_page_ptr[b];
        const int nt = (int)((np + kPlanTile - 1) / kPlanTile);
        int acc = 0;
        for (int k = 0; k < nt; ++k) acc += tile_cnt[((long long)b * tiles_per_req + k) * kMaxDcpAttn + d];
        counts[pr] = acc;
        int chunks = 0;
        if (active(pr)) {
            const int tiles = (acc + 1) >> 1;
            chunks = n_chunks(tiles);
            for (int c = 0; c < chunks; ++c) atomicAdd(&hist[chunk_size(tiles, c)], 1);
            if (chunks > 1) atomicAdd(&part_before, (unsigned long long)chunks * G);
        }
        pair_chunks[pr] = chunks;  // grows by the pieces of cut chunks
    }
    __syncthreads();
    if (tid == 0) {
        // bucket starts, largest size first (positions in units of chunks)
        int acc = 0;
        for (int sz = tpc; sz >= 0; --sz) {
            const int h = hist[sz];
            hist[sz] = acc;
            acc += h;
        }
        u_c = acc;
        int q = 0, ts = acc, sb = 0, first = 0;
        const long long units_total = (long long)acc * G;
        const long long full = units_total / num_sms;
        if (full >= 1 && units_total % num_sms != 0) {
            ts = (int)((full * num_sms + G - 1) / G);
            long long s_tail = 0;
            int smax = -1;
            for (int sz = tpc; sz >= 0; --sz) {  // bucket sz holds positions [hist[sz], end)
                const int b0 = hist[sz], b1 = sz > 0 ? hist[sz - 1] : acc;
                if (b1 <= ts || b0 == b1) continue;
                if (smax < 0) {  // the boundary bucket: its chunks of rank >= first are in the tail
                    smax = sz;
                    sb = sz;
                    first = max(b0, ts) - b0;
                }
                s_tail += (long long)(b1 - max(b0, ts)) * sz;
            }
            const long long qq = (s_tail * G + num_sms - 1) / num_sms;
            const long long cuts = qq > 0 ? s_tail / qq : 0;
            const bool pays = qq >= kMinPiece && 4LL * smax > 5 * qq + 16;
            const bool fits = acc - ts <= kMaxTailChunks && units_total + cuts * G <= max_units &&
                              (long long)part_before + (cuts + (acc - ts)) * G <= max_partials;
            if (pays && fits) q = (int)qq;
        }
        q_cut = q;
        tail_start = q > 0 ? ts : acc;
        s_b = sb;
        b_first = first;
    }
    __syncthreads();
    const int q = q_cut, ts = tail_start, uc = u_c, sb = s_b;
    if (q == 0) {  // no cut: the partial slots first, then every unit with its final slot
        long long running = 0;
        for (int base = 0; base < n_pair; base += blockDim.x) {
            const int pr = base + tid;
            const int chunks = pr < n_pair ? pair_chunks[pr] : 0;
            long long tot;
            const long long off = block_exclusive_scan(chunks > 1 ? (long long)chunks * G : 0, scratch, &tot);
            if (pr < n_pair) {
                pair_part[pr] = chunks > 1 ? (int)(running + off) : -1;
                if (chunks > 1) multi_list[atomicAdd(&n_multi, 1)] = pr;
            }
            running += tot;
        }
        __syncthreads();
        for (int pr = tid; pr < n_pair; pr += blockDim.x) {
            if (!active(pr)) continue;
            const int cnt = counts[pr];
            const int tiles = (cnt + 1) >> 1;
            const int chunks = n_chunks(tiles);
            for (int c = 0; c < chunks; ++c) {
                const int pos = atomicAdd(&hist[chunk_size(tiles, c)], 1);
                const int page_begin = c * 2 * tpc;
                const int n_pages = max(0, min(2 * tpc, cnt - page_begin));
                for (int g = 0; g < G; ++g)
                    units[(long long)pos * G + g] =
                        make_int4(pr * G + g, page_begin, n_pages, chunks > 1 ? pair_part[pr] + c * G + g : -1);
            }
        }
        __syncthreads();
        if (tid == 0) {
            ctrl[0] = uc * G;
            ctrl[1] = 0;
            ctrl[2] = n_multi;
            ctrl[3] = kPlanMagic;
            *reinterpret_cast<unsigned long long *>(ctrl + 4) = key;
            *reinterpret_cast<long long *>(ctrl + 6) = (long long)req_page_ptr[B];
        }
        return;
    }
    // (request, rank, chunk) rank of each pair's first chunk of size sb among all chunks of that
    // size (kept in pair_part until the partial slots are assigned)
    {
        long long running = 0;
        for (int base = 0; base < n_pair; base += blockDim.x) {
            const int idx = base + tid;  // request-major
            const int pr = idx < n_pair ? (idx % N) * B + idx / N : n_pair;
            int x = 0;
            if (pr < n_pair && active(pr)) {
                const int tiles = (counts[pr] + 1) >> 1;
                if (tiles == 0) x = sb == 0;
                else x = (sb == tpc ? tiles / tpc : 0) + (tiles % tpc != 0 && tiles % tpc == sb);
            }
            long long tot;
            const long long off = block_exclusive_scan(x, scratch, &tot);
            if (pr < n_pair) pair_part[pr] = (int)(running + off);
            running += tot;
        }
    }
    __syncthreads();
    for (int pr = tid; pr < n_pair; pr += blockDim.x) {
        if (!active(pr)) continue;
        const int cnt = counts[pr];
        const int tiles = (cnt + 1) >> 1;
        const int chunks = n_chunks(tiles);
        for (int c = 0; c < chunks; ++c) {
            const int sz = chunk_size(tiles, c);
            const bool in_tail = q > 0 && (sz < sb || (sz == sb && pair_part[pr] + (sz == tpc ? c : 0) >= b_first));
            if (in_tail) {
                const int j = atomicAdd(&n_tail, 1);
                tkey[j] = ((unsigned long long)(kMaxTpc - sz) << 32) | (unsigned)((pr % B) * N + pr / B);
                tchunk[j] = c;
                continue;
            }
            const int pos = atomicAdd(&hist[sz], 1);
            const int page_begin = c * 2 * tpc;
            const int n_pages = max(0, min(2 * tpc, cnt - page_begin));
            for (int g = 0; g < G; ++g) units[(long long)pos * G + g] = make_int4(pr * G + g, page_begin, n_pages, c);
        }
    }
    __syncthreads();
    if (q > 0) {
        const int nt = n_tail;  // == uc - ts
        if (tid >= nt) {
            tkey[tid] = ~0ull;
            tchunk[tid] = 0x7fffffff;
        }
        __syncthreads();
        for (int k = 2; k <= kMaxTailChunks; k <<= 1) {  // bitonic sort by (key, chunk)
            for (int j = k >> 1; j > 0; j >>= 1) {
                const int l = tid ^ j;
                if (l > tid) {
                    const unsigned long long ka = tkey[tid], kb = tkey[l];
                    const int ca = tchunk[tid], cb = tchunk[l];
                    const bool gt = ka > kb || (ka == kb && ca > cb);
                    if (gt == ((tid & k) == 0)) {
                        tkey[tid] = kb;
                        tkey[l] = ka;
                        tchunk[tid] = cb;
                        tchunk[l] = ca;
                    }
                }
                __syncthreads();
            }
        }
        // end-to-end offsets, pieces: cuts at the multiples of q strictly inside [o, o + size)
        const bool mine = tid < nt;
        const int bn = mine ? (int)(tkey[tid] & 0xffffffffu) : 0;
        const int pr = (bn % N) * B + bn / N;
        const int sz = mine ? kMaxTpc - (int)(tkey[tid] >> 32) : 0;
        const int c = mine ? tchunk[tid] : 0;
        long long tot;
        const int o = (int)block_exclusive_scan(sz, scratch, &tot);
        const int m0 = o / q;
        const int k = (mine && sz > 0) ? (o + sz - 1) / q - m0 + 1 : 1;
        tpieces[tid] = k;
        for (int i = tid; i <= tpc; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        int first = 0;  // partial ordinal of this chunk's second piece: after the pair's chunks and
                        // the extra pieces of its tail chunks of lower index
        if (mine) {
            first = n_chunks((counts[pr] + 1) >> 1);
            for (int j = 0; j < nt; ++j)
                if ((int)(tkey[j] & 0xffffffffu) == bn && tchunk[j] < c) first += tpieces[j] - 1;
            if (k > 1) {
                atomicAdd(&pair_chunks[pr], k - 1);
                atomicAdd(&n_extra, k - 1);
            }
            for (int i = 0; i < k; ++i) {
                const int t0 = i == 0 ? 0 : (m0 + i) * q - o;
                const int t1 = i == k - 1 ? sz : (m0 + i + 1) * q - o;
                atomicAdd(&hist[t1 - t0], 1);
            }
        }
        __syncthreads();
        if (tid == 0) {  // the pieces fill the queue from position ts, largest first
            int acc = ts;
            for (int s2 = tpc; s2 >= 0; --s2) {
                const int h = hist[s2];
                hist[s2] = acc;
                acc += h;
            }
        }
        __syncthreads();
        if (mine) {
            const int cnt = counts[pr];
            const int page_begin = c * 2 * tpc;
            const int n_pages = max(0, min(2 * tpc, cnt - page_begin));
            for (int i = 0; i < k; ++i) {
                const int t0 = i == 0 ? 0 : (m0 + i) * q - o;
                const int t1 = i == k - 1 ? sz : (m0 + i + 1) * q - o;
                const int pb = page_begin + 2 * t0;
                const int np = max(0, min(page_begin + n_pages, page_begin + 2 * t1) - pb);
                const long long at = atomicAdd(&hist[t1 - t0], 1);
                const int ordinal = i == 0 ? c : first + i - 1;
                for (int g = 0; g < G; ++g) units[at * G + g] = make_int4(pr * G + g, pb, np, ordinal);
            }
        }
    }
    __syncthreads();
    // partial slots of the multi-piece pairs
    long long running = 0;
    for (int base = 0; base < n_pair; base += blockDim.x) {
        const int pr = base + tid;
        const int pieces = pr < n_pair ? pair_chunks[pr] : 0;
        long long tot;
        const long long need = pieces > 1 ? (long long)pieces * G : 0;
        const long long off = block_exclusive_scan(need, scratch, &tot);
        if (pr < n_pair) {
            pair_part[pr] = pieces > 1 ? (int)(running + off) : -1;
            if (pieces > 1) multi_list[atomicAdd(&n_multi, 1)] = pr;
        }
        running += tot;
    }
    __syncthreads();
    const long long n_units = (long long)(uc + n_extra) * G;
    for (long long i = tid; i < n_units; i += blockDim.x) {  // ordinal -> partial slot
        int4 r = units[i];
        const int pr = r.x / G, g = r.x - pr * G;
        r.w = pair_part[pr] >= 0 ? pair_part[pr] + r.w * G + g : -1;
        units[i] = r;
    }
    if (tid == 0) {
        ctrl[0] = (int)n_units;
        ctrl[1] = 0;
        ctrl[2] = n_multi;
        ctrl[3] = kPlanMagic;
        *reinterpret_cast<unsigned long long *>(ctrl + 4) = key;
        *reinterpret_cast<long long *>(ctrl + 6) = (long long)req_page_ptr[B];
    }
}

__global__ void __launch_bounds__(kPlanThreads)
plan_build_kernel(int B, int N, int G, int only_rank, int tpc, int num_sms, long long max_units, long long max_partials,
                  unsigned long long key, long long num_pages,
                  long long slots_per_rank,
                  int tiles_per_req, int tile_stride, const int64_t *__restrict__ req_page_ptr, const int32_t *__restrict__ vpages,
                  const int32_t *__restrict__ tile_cnt, int32_t *__restrict__ comp_slot, int32_t *__restrict__ comp_page,
                  int32_t *__restrict__ counts, int32_t *__restrict__ pair_chunks, int32_t *__restrict__ pair_part,
                  int32_t *__restrict__ multi_list, int4 *__restrict__ units, int *__restrict__ ctrl) {
    grid_dep_wait();
    grid_dep_launch();
    const int n_tile_blocks = B * tile_stride;
    if ((int)blockIdx.x < n_tile_blocks) {
        const int b = blockIdx.x / tile_stride;
        const long long np = req_page_ptr[b + 1] - req_page_ptr[b];
        for (int k = blockIdx.x % tile_stride; (long long)k * kPlanTile < np; k += tile_stride)
            plan_scatter_tile(b, k, N, num_pages, slots_per_rank, tiles_per_req, req_page_ptr, vpages, tile_cnt,
                              comp_slot, comp_page);
    } else
        plan_build_units(B, N, G, only_rank, tpc, num_sms, max_units, max_partials, key, req_page_ptr, tiles_per_req,
                         tile_cnt, counts, pair_chunks,
                         pair_part, multi_list, units, ctrl);
}

// Merge the chunk partials of the multi-chunk (rank, request) pairs listed by the plan into
// O_part / LSE_part; a grid-stride loop over (listed pair, query group, row), one warp each.
__global__ void combine_kernel(int B, int T, int H, int HB, int G, int *ctrl, unsigned long long key,
                               const int64_t *__restrict__ req_page_ptr,
                               const int32_t *__restrict__ multi_list, const int32_t *__restrict__ pair_chunks,
                               const int32_t *__restrict__ pair_part, const float *part_o, const float *part_lse,
                               float *o_part, float *lse_part) {
    grid_dep_wait();
    grid_dep_launch();
    if (!plan_matches(ctrl, key, req_page_ptr, B)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) ctrl[1] = 0;  // the work counter, ready for the next run of the plan
    const long long n_tasks = (long long)ctrl[2] * G * kGroupRows;
    const int wpb = blockDim.x >> 5;
    for (long long task = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); task < n_tasks;
         task += (long long)gridDim.x * wpb) {
        const int c = (int)(task % kGroupRows);
        const long long pg = task / kGroupRows;
        const int g = (int)(pg % G);
        const int pr = multi_list[pg / G];
        const int chunks = pair_chunks[pr];
        const int t = g / HB, hb = g % HB;
        const int rows_valid = min(kGroupRows, H - hb * kGroupRows);
        if (c >= rows_valid) continue;
        const int d = pr / B, b = pr % B;
        const long long first = (long long)pair_part[pr] + g;  // chunk k lives at first + k * G
        const long long out_row = (long long)d * B * T * H + ((long long)(b * T + t) * H) + hb * kGroupRows + c;
        warp_merge_row512(chunks, part_o + (first * kGroupRows + c) * kVDim, (long long)G * kGroupRows * kVDim,
                          part_lse + first * kGroupRows + c, (long long)G * kGroupRows,
                          o_part + out_row * kVDim, lse_part + out_row, 1.f);
    }
}

// Whether any rank's segment of request b was split into several pieces (warp-uniform: lane d
// reads rank d's piece count).
__device__ __forceinline__ bool request_split(int b, int B, int N, const int32_t *__restrict__ pair_chunks) {
    const int lane = threadIdx.x & 31;
    const bool split = lane < N && __ldg(pair_chunks + (long long)lane * B + b) > 1;
    return __any_sync(0xffffffffu, split);
}

// Fused merge, first launch after the attention kernel: one warp per task.  It combines the
// chunk partials of the multi-piece pairs (as combine_kernel does) and merges over the ranks,
// ascending rank order, the rows of the requests none of whose pairs was split; the rows of
// the other requests are merged by merge_after_combine_kernel.
__global__ void merge_combine_kernel(int B, int T, int H, int HB, int G, int N, int *ctrl, unsigned long long key,
                                     const int64_t *__restrict__ req_page_ptr,
                                     const int32_t *__restrict__ multi_list, const int32_t *__restrict__ pair_chunks,
                                     const int32_t *__restrict__ pair_part, const float *part_o,
                                     const float *part_lse, float *o_part, float *lse_part, float *o_out,
                                     float *lse_out) {
    grid_dep_wait();
    grid_dep_launch();
    if (!plan_matches(ctrl, key, req_page_ptr, B)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) ctrl[1] = 0;  // the work counter, ready for the next run of the plan
    const int n_multi = ctrl[2];
    const int wpb = blockDim.x >> 5;
    const long long n_comb = (long long)n_multi * G * kGroupRows;
    const long long rows = (long long)B * T * H;
    for (long long task = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); task < n_comb + rows;
         task += (long long)gridDim.x * wpb) {
        // one call site for both kinds of task (registers): n parts at o / lse with strides
        int n;
        const float *o, *lse;
        long long o_stride, lse_stride;
        float *dst, *dst_lse;
        if (task < n_comb) {
            const int c = (int)(task % kGroupRows);
            const long long pg = task / kGroupRows;
            const int g = (int)(pg % G);
            const int pr = multi_list[pg / G];
            const int t = g / HB, hb = g % HB;
            if (c >= min(kGroupRows, H - hb * kGroupRows)) continue;
            const int d = pr / B, b = pr % B;
            const long long first = (long long)pair_part[pr] + g;
            const long long out_row = (long long)d * B * T * H + ((long long)(b * T + t) * H) + hb * kGroupRows + c;
            n = pair_chunks[pr];
            o = part_o + (first * kGroupRows + c) * kVDim;
            o_stride = (long long)G * kGroupRows * kVDim;
            lse = part_lse + first * kGroupRows + c;
            lse_stride = (long long)G * kGroupRows;
            dst = o_part + out_row * kVDim;
            dst_lse = lse_part + out_row;
        } else {
            const long long row = task - n_comb;
            if (n_multi > 0 && request_split((int)row / (T * H), B, N, pair_chunks)) continue;  // rows < 2^31
            n = N;
            o = o_part + row * kVDim;
            o_stride = rows * kVDim;
            lse = lse_part + row;
            lse_stride = rows;
            dst = o_out + row * kVDim;
            dst_lse = lse_out + row;
        }
        warp_merge_row512(n, o, o_stride, lse, lse_stride, dst, dst_lse, 1.f);
    }
}

// Fused merge, second launch: the rank merge of the rows of the requests with a split pair,
// after merge_combine_kernel has combined their chunk partials; exits at once when there are
// none (ctrl[2] == 0).
__global__ void merge_after_combine_kernel(int N, long long rows, int TH, const int *__restrict__ ctrl,
                                           unsigned long long key, const int64_t *__restrict__ req_page_ptr, int B,
                                           const int32_t *__restrict__ pair_chunks, const float *o_part,
                                           const float *lse_part, float *o_out, float *lse_out) {
    grid_dep_wait();
    grid_dep_launch();
    if (!plan_matches(ctrl, key, req_page_ptr, B) || ctrl[2] == 0) return;
    const int wpb = blockDim.x >> 5;
    for (long long row = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * wpb) {
        if (!request_split((int)row / TH, B, N, pair_chunks)) continue;  // rows < 2^31
        warp_merge_row512(N, o_part + row * kVDim, rows * kVDim, lse_part + row, rows, o_out + row * kVDim,
                          lse_out + row, 1.f);
    }
}

// ------------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once (a function-local static: thread-safe initialisation).
EncodeTiledFn get_encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

// 2-D map over [rows][576] elements (BF16 or bytes) with a box of box_x elements by 64 rows.
bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, bool bf16, uint32_t box_x, bool swz128) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const uint32_t esz = bf16 ? 2 : 1;
    cuuint64_t dims[2] = {(cuuint64_t)kKDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kKDim * esz};
    cuuint32_t box[2] = {box_x, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Key of the arguments a plan depends on (splitmix64 steps over the fields).
unsigned long long plan_key(const AttnPlanShape &s, int dtype, int only_rank, int64_t slots_per_rank,
                            int token_layout) {
    const long long f[9] = {s.B, s.T, s.H, s.N, dtype, only_rank, (long long)slots_per_rank, (long long)s.num_pages,
                            token_layout};
    unsigned long long h = 0x9E3779B97F4A7C15ull;
    for (long long v : f) {
        h ^= (unsigned long long)v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h = (h ^ (h >> 30)) * 0xBF58476D1CE4E5B9ull;
        h = (h ^ (h >> 27)) * 0x94D049BB133111EBull;
        h ^= h >> 31;
    }
    return h;
}

}  // namespace

bool plan_attention(int B, int T, int H, int N, int64_t num_pages, int dtype, int num_sms,
                    AttnPlanShape *s) {
    if (B < 0 || T < 1 || H < 1 || N < 1 || N > kMaxDcpAttn || num_pages < 0 || num_sms < 1) return false;
    s->B = B;
    s->T = T;
    s->H = H;
    s->N = N;
    const int HB = (H + kGroupRows - 1) / kGroupRows;
    s->G = T * HB;
    s->heads_per_group = std::min(H, kGroupRows);
    s->num_pages = num_pages;
    // Chunk size: equal-segment cost model, makespan in tiles over num_sms persistent CTAs taking
    // units from a queue.  A chunk boundary costs the round trip of a partial (write + read of a
    // 64 x 512 fp32 chunk output, in tile-equivalents of KV bytes) plus about one tile of
    // epilogue and restart.  A last wave that keeps a fraction f of the SMs busy takes (1 + f) / 2
    // of a full wave: the kernel is bound by memory latency, which drops with the load (measured
    // on the 48 x 100K FP8 workload: unchunked units beat the 3-chunk split a whole-wave count
    // picks by 4%, while the 4 x 1M workload keeps its 7-chunk split).
    const long long pages_avg = B > 0 ? (num_pages + B - 1) / B : 0;
    const long long tiles_seg = std::max<long long>(1, ((pages_avg + N - 1) / N + 1) / 2);
    const long long n_seg = (long long)N * B * s->G;
    const double partial_cost = (2.0 * kGroupRows * kVDim * 4.0) / (128.0 * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1));
    const double chunk_cost = partial_cost + 1.0;
    double best = 1e300;
    long long tpc = tiles_seg;
    for (long long k = 1; k <= std::min<long long>(tiles_seg, 64); ++k) {
        const long long t = (tiles_seg + k - 1) / k;
        const long long chunks = (tiles_seg + t - 1) / t;
        const long long units = std::max<long long>(1, n_seg * chunks);
        const long long full = units / num_sms;
        const double f = (double)(units - full * num_sms) / num_sms;
        const double waves = (double)full + (f > 0.0 ? 0.5 + 0.5 * f : 0.0);
        const double cost = waves * ((double)t + (chunks > 1 ? chunk_cost : 0.0));
        if (cost < best - 1e-9) {
            best = cost;
            tpc = t;
        }
    }
    // With at least as many segments as SMs, segments of unequal length (the host sees only
    // their average) balance by themselves in the largest-first queue, so a chunk may grow to a
    // fair part of each SM's share of all tiles (measured on 64 requests of 2K to 500K tokens:
    // chunks from 0.55 to 1.0 of the share run within 2% of each other, 1.25 of it 12% slower,
    // the average-segment size 4% slower).
    if (n_seg >= num_sms) {
        const long long share = (long long)std::ceil(0.6 * (double)(n_seg * tiles_seg) / num_sms);
        tpc = std::max(tpc, share);
    }
    tpc = std::max<long long>(1, std::min<long long>(tpc, kMaxTpc));
    s->tiles_per_chunk = (int)tpc;
    s->max_partials = ((long long)s->G * (num_pages + (long long)N * B)) / tpc + s->G;
    s->max_units = n_seg + s->max_partials;
    s->n_seg = n_seg;
    size_t off = 0;
    s->off_counts = off;  off = align256(off + sizeof(int32_t) * (size_t)N * B);
    s->off_slots = off;   off = align256(off + sizeof(int32_t) * (size_t)N * num_pages);
    s->off_pages = off;   off = align256(off + sizeof(int32_t) * (size_t)N * num_pages);
    s->off_units = off;   off = align256(off + sizeof(int4) * (size_t)s->max_units);
    s->off_seg = off;     off = align256(off + sizeof(int32_t) * 2 * (size_t)N * B);
    s->off_multi = off;   off = align256(off + sizeof(int32_t) * (size_t)N * B);
    s->off_ctrl = off;    off = align256(off + sizeof(int32_t) * 8);
    s->tiles_per_req = (int)std::max<long long>(1, (num_pages + kPlanTile - 1) / kPlanTile);
    s->off_tiles = off;   off = align256(off + sizeof(int32_t) * (size_t)B * s->tiles_per_req * kMaxDcpAttn);
    s->off_part_o = off;  off = align256(off + sizeof(float) * (size_t)s->max_partials * kGroupRows * kVDim);
    s->off_part_lse = off; off = align256(off + sizeof(float) * (size_t)s->max_partials * kGroupRows);
    const size_t R = (size_t)B * T * H;
    s->off_qhl = off;     off = align256(off + (dtype == DCP_KV_FP8_E4M3 ? 2 * R * kKDim : 0));
    s->off_qscale = off;  off = align256(off + (dtype == DCP_KV_FP8_E4M3 ? sizeof(float) * R : 0));
    s->total_bytes = off;
    return true;
}

template <bool F8>
int launch_kernel(const AttnMaps &maps, const KParams &kp, int grid, cudaStream_t stream) {
    constexpr size_t smem = smem_bytes<F8>();
    if (cudaFuncSetAttribute(attn_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DCP_ERR_CUDA;
    return launch_pdl(attn_kernel<F8>, dim3(grid), dim3(kThreads), smem, stream, maps, kp) == cudaSuccess
               ? DCP_OK : DCP_ERR_CUDA;
}

int read_plan_info(const AttnPlanShape &s, const void *workspace, int32_t *info, cudaStream_t stream) {
    int ctrl[8];
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    if (cudaMemcpyAsync(ctrl, ws + s.off_ctrl, sizeof(ctrl), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return DCP_ERR_CUDA;
    const bool valid = ctrl[3] == kPlanMagic;
    info[0] = valid ? ctrl[0] : 0;
    info[1] = valid ? ctrl[2] : 0;
    info[2] = s.tiles_per_chunk;
    info[3] = valid ? 1 : 0;
    return DCP_OK;
}

int launch_attention(const AttnArgs &a, int num_sms, cudaStream_t stream) {
    const AttnPlanShape &s = a.shape;
    const bool f8 = a.dtype == DCP_KV_FP8_E4M3;
    if (s.B == 0) return DCP_OK;
    uint8_t *ws = a.workspace;
    int32_t *counts = reinterpret_cast<int32_t *>(ws + s.off_counts);
    int32_t *comp_slot = reinterpret_cast<int32_t *>(ws + s.off_slots);
    int32_t *comp_page = reinterpret_cast<int32_t *>(ws + s.off_pages);
    int4 *units = reinterpret_cast<int4 *>(ws + s.off_units);
    int32_t *pair_chunks = reinterpret_cast<int32_t *>(ws + s.off_seg);
    int32_t *pair_part = pair_chunks + (size_t)s.N * s.B;
    int *ctrl = reinterpret_cast<int *>(ws + s.off_ctrl);
    float *part_o = reinterpret_cast<float *>(ws + s.off_part_o);
    float *part_lse = reinterpret_cast<float *>(ws + s.off_part_lse);
    uint8_t *qhl = ws + s.off_qhl;
    float *qscale = reinterpret_cast<float *>(ws + s.off_qscale);
    const int R = s.B * s.T * s.H;

    int32_t *tile_cnt = reinterpret_cast<int32_t *>(ws + s.off_tiles);
    int32_t *multi_list = reinterpret_cast<int32_t *>(ws + s.off_multi);
    const unsigned long long key = plan_key(s, a.dtype, a.only_rank, a.slots_per_rank, a.token_layout);
    // blocks per request: about three blocks per SM in all, at most one per tile
    const int tile_stride = (int)std::max<long long>(
        1, std::min<long long>(s.tiles_per_req, (3LL * num_sms + s.B - 1) / s.B));
    // the plan (page-table work) unless running a stored plan; the FP8 Q split unless planning only
    const int n_tile_blocks = a.phase == 2 ? 0 : s.B * tile_stride;
    const int q_blocks = (f8 && a.phase != 1) ? (R + kPlanThreads / 32 - 1) / (kPlanThreads / 32) : 0;
    if (n_tile_blocks + q_blocks > 0 &&
        launch_pdl(plan_count_kernel, dim3(n_tile_blocks + q_blocks), dim3(kPlanThreads), 0, stream, s.N,
                   (long long)a.slots_per_rank, s.tiles_per_req, tile_stride, n_tile_blocks, a.req_page_ptr, a.dst_vpages, tile_cnt,
                   a.dev_error, R, reinterpret_cast<const __nv_bfloat16 *>(a.q), qhl, qscale,
                   a.phase == 2 ? (const int *)ctrl : nullptr, key, s.B) != cudaSuccess)
        return DCP_ERR_CUDA;
    if (a.phase != 2 &&
        launch_pdl(plan_build_kernel, dim3(n_tile_blocks + 1), dim3(kPlanThreads), 0, stream, s.B, s.N, s.G,
                   a.only_rank, s.tiles_per_chunk, num_sms, (long long)s.max_units, (long long)s.max_partials, key, (long long)s.num_pages, (long long)a.slots_per_rank, s.tiles_per_req,
                   tile_stride, a.req_page_ptr, a.dst_vpages, (const int32_t *)tile_cnt, comp_slot, comp_page, counts, pair_chunks,
                   pair_part, multi_list, units, ctrl) != cudaSuccess)
        return DCP_ERR_CUDA;
    if (a.phase == 1) return DCP_OK;

    AttnMaps maps;
    memset(&maps, 0, sizeof(maps));
    const uint64_t pool_rows = (uint64_t)a.slots_per_rank * kPage;
    if (f8) {
        if (!make_map(&maps.q[0], qhl, 2ull * R, false, 128, true) || !make_map(&maps.q[1], qhl, 2ull * R, false, 64, false))
            return DCP_ERR_CUDA;
        for (int d = 0; d < s.N; ++d)
            if (!make_map(&maps.kv[d][0], a.kv_pools[d], pool_rows, false, 128, true) ||
                !make_map(&maps.kv[d][1], a.kv_pools[d], pool_rows, false, 64, false))
                return DCP_ERR_CUDA;
    } else {
        if (!make_map(&maps.q[0], a.q, (uint64_t)R, true, 64, true)) return DCP_ERR_CUDA;
        for (int d = 0; d < s.N; ++d)
            if (!make_map(&maps.kv[d][0], a.kv_pools[d], pool_rows, true, 64, true)) return DCP_ERR_CUDA;
    }
    KParams kp;
    kp.seq_lens = a.seq_lens;
    kp.req_page_ptr = a.req_page_ptr;
    kp.comp_slot = comp_slot;
    kp.comp_page = comp_page;
    kp.units = units;
    kp.ctrl = ctrl;
    kp.plan_key = key;
    kp.counter = ctrl + 1;
    kp.q_rscale = qscale;
    kp.B = s.B;
    kp.T = s.T;
    kp.H = s.H;
    kp.HB = (s.H + kGroupRows - 1) / kGroupRows;
    kp.G = s.G;
    kp.R = R;
    kp.num_pages = s.num_pages;
    kp.oob_row = (int)std::min<int64_t>((int64_t)pool_rows, 0x7fffff00);
    kp.tok_n = a.token_layout ? std::max(s.N, 1) : 0;
    const float kappa = f8 ? a.kv_scale : 1.f;
    kp.sl2 = a.softmax_scale * kappa * 1.4426950408889634f;
    kp.out_scale = f8 ? kappa / kPScale : kappa;
    kp.o_part = a.o_part;
    kp.lse_part = a.lse_part;
    kp.part_o = part_o;
    kp.part_lse = part_lse;
    kp.dev_error = a.dev_error;
    kp.wait_limit_ns = a.wait_limit_ns;
    const int grid = (int)std::max<long long>(1, std::min<long long>(num_sms, s.max_units));
    const int st = f8 ? launch_kernel<true>(maps, kp, grid, stream) : launch_kernel<false>(maps, kp, grid, stream);
    if (st != DCP_OK) return st;
    if (a.o_out) {  // fused merge (see merge_combine_kernel)
        const long long rows = (long long)s.B * s.T * s.H;
        const long long tasks = rows + (long long)s.N * s.B * s.G * kGroupRows;  // rank merges + chunk combines
        const int blocks = (int)std::max<long long>(1, std::min<long long>((tasks + 7) / 8, 8LL * num_sms));
        if (launch_pdl(merge_combine_kernel, dim3(blocks), dim3(256), 0, stream, s.B, s.T, s.H, kp.HB, s.G, s.N,
                       ctrl, key, a.req_page_ptr, (const int32_t *)multi_list, (const int32_t *)pair_chunks,
                       (const int32_t *)pair_part, (const float *)part_o, (const float *)part_lse, a.o_part,
                       a.lse_part, a.o_out, a.lse_out) != cudaSuccess)
            return DCP_ERR_CUDA;
        const int mblocks = (int)std::max<long long>(1, std::min<long long>((rows + 7) / 8, 8LL * num_sms));
        if (launch_pdl(merge_after_combine_kernel, dim3(mblocks), dim3(256), 0, stream, s.N, rows, s.T * s.H,
                       (const int *)ctrl, key, a.req_page_ptr, s.B, (const int32_t *)pair_chunks,
                       (const float *)a.o_part, (const float *)a.lse_part, a.o_out, a.lse_out) != cudaSuccess)
            return DCP_ERR_CUDA;
        return DCP_OK;
    }
    // one warp per (listed pair, query group, row) when every pair has several chunks, capped
    const long long max_tasks = (long long)s.N * s.B * s.G * kGroupRows;
    const int combine_blocks = (int)std::max<long long>(1, std::min<long long>((max_tasks + 7) / 8, 8LL * num_sms));
    if (launch_pdl(combine_kernel, dim3(combine_blocks), dim3(256), 0, stream, s.B, s.T, s.H, kp.HB, s.G,
                   ctrl, key, a.req_page_ptr, (const int32_t *)multi_list, (const int32_t *)pair_chunks,
                   (const int32_t *)pair_part, (const float *)part_o, (const float *)part_lse, a.o_part,
                   a.lse_part) != cudaSuccess)
        return DCP_ERR_CUDA;
    return DCP_OK;
}

}  // namespace dcp
