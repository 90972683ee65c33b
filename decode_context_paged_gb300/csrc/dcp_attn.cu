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
//    persistent CTAs (one per SM) take them from an atomic counter.
//  * Per tile, tcgen05 computes S^T[128 tokens x 64 query rows] = K_tile * Q^T (K-major
//    BF16 operands, 128-byte swizzle, FP32 accumulator in TMEM, M = 128 tokens so the
//    whole tensor datapath is used), then O^T[512 x 64] += V_tile^T * P^T (V read MN-major
//    from the same page rows, P written by the softmax warps).  O^T (256 TMEM columns) and
//    two S buffers (64 columns each) fit in one 512-column allocation.
//  * TMA streams 64-row x 64-dim boxes of the page pool into an 8-slot ring of 16 KB blocks
//    (two pages per block): the nine 64-dim blocks of a tile for S, then the eight V blocks
//    again (they come back from L2) for P*V, so the ring never has to hold a whole tile.
//  * Four softmax warps own one token row each (TMEM lane = row): scores are masked
//    (ragged last page, causal limit among the new tokens), column maxima are reduced with
//    a warp-shuffle reduce-scatter plus shared memory, exp2 weights go to shared memory as
//    BF16 P^T, and O^T is rescaled in TMEM only when a column's running max moved.
//  * Single-chunk segments write O_part / LSE_part directly; multi-chunk segments write
//    chunk partials to the workspace and a combine kernel merges them (exact LSE merge).
//  * Every mbarrier wait is bounded; on timeout the CTA stops, drains its in-flight copies
//    and MMAs, frees TMEM and reports DCP_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dcp_internal.h"
#include "dcp_merge_row.cuh"
#include "dcp_ptx.cuh"

namespace dcp {
namespace {

constexpr int kRingSlots = 8;
constexpr uint32_t kBlockBytes = 16384;  // 128 token rows x 64 dims x 2 bytes
constexpr uint32_t kHalfBlock = 8192;    // one page (64 rows) x 64 dims
constexpr int kQBlocks = 9;              // 576 / 64
constexpr int kVBlocks = 8;              // 512 / 64
constexpr uint32_t kQBytes = kQBlocks * kHalfBlock;
constexpr uint32_t kPBytes = 16384;      // 128 tokens x 64 query rows x 2 bytes
constexpr int kGroupRows = 64;
constexpr uint32_t kOffQ = kRingSlots * kBlockBytes;
constexpr uint32_t kOffP = kOffQ + kQBytes;
constexpr uint32_t kOffCtl = kOffP + kPBytes;
constexpr int kThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;          // S buffers at TMEM columns 256 and 320
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, 1, 1);
constexpr int kMaxTpc = 4096;

struct UnitInfo {
    int valid, d, b, g;
    int n_pages, out_index, limit, q_row0;
    int rows_valid, pad0;
    long long comp_base;
};

struct __align__(16) Ctl {
    float red[4][64];
    float m_run[64];
    float corr[64];
    float oscale[64];
    uint64_t full[kRingSlots], empty[kRingSlots];
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_done, o_free;
    uint64_t unit_full[2], unit_empty[2];
    uint64_t drain;
    UnitInfo unit[2];
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kSmemBytes = 1024 + kOffCtl + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct AttnMaps {
    CUtensorMap q;
    CUtensorMap kv[kMaxDcpAttn];
};

struct KParams {
    const int32_t *seq_lens;
    const int64_t *req_page_ptr;
    const int32_t *comp_slot;  // [N][num_pages]: rank d's pages of request b start at d*num_pages + ptr[b]
    const int32_t *comp_page;  // page index j (within the request) of each compacted entry
    const int4 *units;         // {pair, page_begin, n_pages, out_index}, pair = d*B + b ... see plan
    const int *ctrl;           // [0] = number of units, [1] = work counter
    int *counter;
    int B, T, H, HB, G;
    long long num_pages;
    int oob_row;               // a TMA row coordinate past the pool (zero fill)
    float sl2;                 // softmax_scale * kappa * log2(e)
    float kv_scale;            // kappa applied to V
    float *o_part, *lse_part, *part_o, *part_lse;
    int32_t *dev_error;
    unsigned long long wait_limit_ns;
};

// ---------------------------------------------------------------------- warp reductions
// Reduce-scatter over the warp: on entry each lane holds the 64 column values of its token
// in v; on exit r[0], r[1] of lane L hold the reduction over the warp's 32 tokens of
// columns 2L and 2L+1.  62 shuffles instead of 64 x 5 for a plain butterfly.
template <bool kMax>
__device__ __forceinline__ float rs_op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }

template <bool kMax>
__device__ __forceinline__ void reduce_scatter64(const float (&v)[64], float (&r)[32], int lane) {
    {
        const bool upper = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float send = upper ? v[i] : v[i + 32];
            const float keep = upper ? v[i + 32] : v[i];
            r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
    }
#pragma unroll
    for (int half = 16, off = 8; half >= 2; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i < half) {
                const float send = upper ? r[i] : r[i + half];
                const float keep = upper ? r[i + half] : r[i];
                r[i] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, off));
            }
        }
    }
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

__global__ void __launch_bounds__(kThreads, 1)
attn_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = base;
    uint8_t *sq = base + kOffQ;
    uint8_t *sp = base + kOffP;
    Ctl *ctl = reinterpret_cast<Ctl *>(base + kOffCtl);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &ctl->abort_flag;
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRingSlots; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->s_full[i], 1);
            mbar_init(&ctl->s_free[i], 128);
            mbar_init(&ctl->unit_full[i], 1);
            mbar_init(&ctl->unit_empty[i], 2);
        }
        mbar_init(&ctl->p_full, 128);
        mbar_init(&ctl->o_done, 1);
        mbar_init(&ctl->o_free, 128);
        mbar_init(&ctl->drain, 1);
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
    const uint32_t tmem = ctl->tmem_base;
    const int n_units = p.ctrl[0];

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&maps.q);
            uint32_t ring_pos = 0, q_cnt = 0, k = 0;
            bool ok = true;
            auto load_block = [&](const CUtensorMap *km, int kb, int row0, int row1) -> bool {
                const uint32_t slot = ring_pos % kRingSlots;
                const uint32_t par = ((ring_pos / kRingSlots) & 1) ^ 1;
                ++ring_pos;
                if (!mbar_wait(&ctl->empty[slot], par, abort_flag, p.dev_error, lim)) return false;
                mbar_arrive_expect_tx(&ctl->full[slot], kBlockBytes);
                uint8_t *dst = ring + slot * kBlockBytes;
                tma_load_2d(dst, km, &ctl->full[slot], kb * 64, row0);
                tma_load_2d(dst + kHalfBlock, km, &ctl->full[slot], kb * 64, row1);
                return true;
            };
            auto pad_block = [&]() -> bool {
                const uint32_t slot = ring_pos % kRingSlots;
                const uint32_t par = ((ring_pos / kRingSlots) & 1) ^ 1;
                ++ring_pos;
                if (!mbar_wait(&ctl->empty[slot], par, abort_flag, p.dev_error, lim)) return false;
                mbar_arrive(&ctl->full[slot]);
                return true;
            };
            while (ok) {
                const int e = k & 1;
                if (!mbar_wait(&ctl->unit_empty[e], ((k >> 1) & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                const int idx = atomicAdd(p.counter, 1);
                UnitInfo u;
                u.valid = idx < n_units;
                if (u.valid) {
                    const int4 rec = p.units[idx];
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
                const CUtensorMap *km = &maps.kv[u.d];
                if (!mbar_wait(&ctl->q_empty, (q_cnt & 1) ^ 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                ++q_cnt;
                mbar_arrive_expect_tx(&ctl->q_full, kQBytes);
                for (int kb = 0; kb < kQBlocks; ++kb)
                    tma_load_2d(sq + kb * kHalfBlock, &maps.q, &ctl->q_full, kb * 64, u.q_row0);
                auto rows_of = [&](int tile, int &r0, int &r1) {
                    const int pg = 2 * tile;
                    r0 = p.comp_slot[u.comp_base + pg] * 64;
                    r1 = (pg + 1 < u.n_pages) ? p.comp_slot[u.comp_base + pg + 1] * 64 : p.oob_row;
                };
                auto load_S = [&](int tile) -> bool {
                    int r0, r1;
                    rows_of(tile, r0, r1);
                    for (int kb = 0; kb < kQBlocks; ++kb)
                        if (!load_block(km, kb, r0, r1)) return false;
                    return pad_block();
                };
                auto load_V = [&](int tile) -> bool {
                    int r0, r1;
                    rows_of(tile, r0, r1);
                    for (int kb = 0; kb < kVBlocks; ++kb)
                        if (!load_block(km, kb, r0, r1)) return false;
                    return true;
                };
                ok = load_S(0);
                for (int i = 1; i < nt && ok; ++i) ok = load_S(i) && load_V(i - 1);
                if (ok) ok = load_V(nt - 1);
            }
            if (!ok) {  // let issued TMA copies land before the CTA can exit
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t ring_pos = 0, s_cnt = 0, p_cnt = 0, q_cnt = 0, of_cnt = 0, k = 0;
            bool had_tiles = false, ok = true;
            const uint32_t ring_addr = smem_u32(ring), q_addr = smem_u32(sq), p_addr = smem_u32(sp);
            auto issue_S = [&]() -> bool {
                const uint32_t sb = s_cnt & 1;
                if (!mbar_wait(&ctl->s_free[sb], ((s_cnt >> 1) & 1) ^ 1, abort_flag, p.dev_error, lim)) return false;
                ++s_cnt;
                tc_fence_after();
                const uint32_t d_tmem = tmem + kSCol + 64 * sb;
                for (int kb = 0; kb < kQBlocks; ++kb) {
                    const uint32_t slot = ring_pos % kRingSlots;
                    if (!mbar_wait(&ctl->full[slot], (ring_pos / kRingSlots) & 1, abort_flag, p.dev_error, lim)) return false;
                    ++ring_pos;
                    tc_fence_after();
                    const uint32_t a0 = ring_addr + slot * kBlockBytes;
                    const uint32_t b0 = q_addr + kb * kHalfBlock;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_ss(d_tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024),
                                   smem_desc_sw128(b0 + kk * 32, 16, 1024), kIdescS, (kb | kk) != 0);
                    mma_commit(&ctl->empty[slot]);
                }
                {   // pad position of the ring
                    const uint32_t slot = ring_pos % kRingSlots;
                    if (!mbar_wait(&ctl->full[slot], (ring_pos / kRingSlots) & 1, abort_flag, p.dev_error, lim)) return false;
                    ++ring_pos;
                    mbar_arrive(&ctl->empty[slot]);
                }
                mma_commit(&ctl->s_full[sb]);
                return true;
            };
            auto issue_PV = [&](bool first) -> bool {
                if (!mbar_wait(&ctl->p_full, p_cnt & 1, abort_flag, p.dev_error, lim)) return false;
                ++p_cnt;
                if (first && had_tiles) {
                    if (!mbar_wait(&ctl->o_free, of_cnt & 1, abort_flag, p.dev_error, lim)) return false;
                    ++of_cnt;
                }
                tc_fence_after();
                for (int j = 0; j < kVBlocks / 2; ++j) {
                    const uint32_t sa = ring_pos % kRingSlots;
                    if (!mbar_wait(&ctl->full[sa], (ring_pos / kRingSlots) & 1, abort_flag, p.dev_error, lim)) return false;
                    ++ring_pos;
                    const uint32_t sb2 = ring_pos % kRingSlots;
                    if (!mbar_wait(&ctl->full[sb2], (ring_pos / kRingSlots) & 1, abort_flag, p.dev_error, lim)) return false;
                    ++ring_pos;
                    tc_fence_after();
                    const uint32_t a0 = ring_addr + sa * kBlockBytes;
                    const uint32_t d_tmem = tmem + 64 * j;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ss(d_tmem, smem_desc_sw128(a0 + kk * 2048, kBlockBytes, 1024),
                                   smem_desc_sw128(p_addr + kk * 2048, 1024, 1024), kIdescPV,
                                   !(first && kk == 0));
                    mma_commit(&ctl->empty[sa]);
                    mma_commit(&ctl->empty[sb2]);
                }
                mma_commit(&ctl->o_done);
                return true;
            };
            while (ok) {
                const int e = k & 1;
                if (!mbar_wait(&ctl->unit_full[e], (k >> 1) & 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                const UnitInfo u = ctl->unit[e];
                mbar_arrive(&ctl->unit_empty[e]);
                ++k;
                if (!u.valid) break;
                const int nt = (u.n_pages + 1) >> 1;
                if (nt == 0) continue;
                if (!mbar_wait(&ctl->q_full, q_cnt & 1, abort_flag, p.dev_error, lim)) {
                    ok = false;
                    break;
                }
                ++q_cnt;
                tc_fence_after();
                for (int i = 0; i < nt && ok; ++i) {
                    ok = issue_S();
                    if (ok && i == nt - 1) mma_commit(&ctl->q_empty);
                    if (ok && i > 0) ok = issue_PV(i - 1 == 0);
                }
                if (ok) ok = issue_PV(nt == 1);
                had_tiles = true;
            }
            // drain: every MMA issued so far has completed once `drain` flips
            mma_commit(&ctl->drain);
            int never = 0;
            mbar_wait(&ctl->drain, 0, &never, nullptr, 100000000ull);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int stid = threadIdx.x - 64;          // 0..127
        const int quad = warp & 3;                  // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;           // token row of the tile = TMEM lane
        const int wl = warp - 2;                    // 0..3 for the reduction scratch
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint32_t s_cnt = 0, od_cnt = 0, k = 0;
        while (true) {
            const int e = k & 1;
            int fail = !warp_wait(&ctl->unit_full[e], (k >> 1) & 1, abort_flag, p.dev_error, lim);
            if (named_bar_or(1, 128, fail)) break;
            const UnitInfo u = ctl->unit[e];
            named_bar_sync(2, 128);
            if (stid == 0) mbar_arrive(&ctl->unit_empty[e]);
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
                for (int idx = stid; idx < u.rows_valid * (kVDim / 4); idx += 128) {
                    const int c = idx / (kVDim / 4), v4 = idx - c * (kVDim / 4);
                    reinterpret_cast<float4 *>(obase + (out_row0 + c) * kVDim)[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (stid < u.rows_valid) lbase[out_row0 + stid] = -INFINITY;
                continue;
            }
            if (stid < 64) ctl->m_run[stid] = -INFINITY;
            float lp[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) lp[c] = 0.f;
            bool aborted = false;
            for (int i = 0; i < nt; ++i) {
                const uint32_t sb = s_cnt & 1;
                fail = !warp_wait(&ctl->s_full[sb], (s_cnt >> 1) & 1, abort_flag, p.dev_error, lim);
                ++s_cnt;
                float s[64];
                if (!fail) {
                    tc_fence_after();
                    {
                        float t32[32];
                        tmem_ld32(tmem + lane_base + kSCol + 64 * sb, t32);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) s[c] = t32[c];
                        tmem_ld32(tmem + lane_base + kSCol + 64 * sb + 32, t32);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) s[32 + c] = t32[c];
                    }
                    tc_fence_before();
                    mbar_arrive(&ctl->s_free[sb]);
                    // mask: ragged last page / missing second page / causal limit
                    const int pl = 2 * i + (row >> 6);
                    bool valid = pl < u.n_pages;
                    if (valid) {
                        const int j = p.comp_page[u.comp_base + pl];
                        valid = (long long)j * 64 + (row & 63) <= (long long)u.limit;
                    }
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = valid ? s[c] * p.sl2 : -INFINITY;
                    float r[32];
                    reduce_scatter64<true>(s, r, lane);
                    *reinterpret_cast<float2 *>(&ctl->red[wl][2 * lane]) = make_float2(r[0], r[1]);
                }
                if (named_bar_or(1, 128, fail)) {
                    aborted = true;
                    break;
                }
                int changed = 0;
                if (stid < 64) {
                    const float mt = fmaxf(fmaxf(ctl->red[0][stid], ctl->red[1][stid]),
                                           fmaxf(ctl->red[2][stid], ctl->red[3][stid]));
                    const float mo = ctl->m_run[stid];
                    const float mn = fmaxf(mo, mt);
                    const float cr = (mn == mo) ? 1.f : exp2f(mo - mn);
                    ctl->m_run[stid] = mn;
                    ctl->corr[stid] = cr;
                    changed = cr != 1.f;
                }
                const int any = named_bar_or(2, 128, changed);
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(&ctl->m_run[c]);
                    float4 c4 = make_float4(1.f, 1.f, 1.f, 1.f);
                    if (any) c4 = *reinterpret_cast<const float4 *>(&ctl->corr[c]);
                    const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
                    const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float ms = mm[q] == -INFINITY ? 0.f : mm[q];
                        s[c + q] = exp2f(s[c + q] - ms);
                        lp[c + q] = fmaf(lp[c + q], cc[q], s[c + q]);
                    }
                }
                if (i > 0) {
                    fail = !warp_wait(&ctl->o_done, od_cnt & 1, abort_flag, p.dev_error, lim);
                    ++od_cnt;
                    if (fail) continue;  // the next OR-barrier takes every thread out
                    tc_fence_after();
                    if (any) {
#pragma unroll 1
                        for (int j = 0; j < 8; ++j) {
                            float o32[32];
                            const uint32_t ta = tmem + lane_base + 32 * j;
                            tmem_ld32(ta, o32);
                            tmem_wait_ld();
                            const float *cr = &ctl->corr[(j & 1) * 32];
#pragma unroll
                            for (int c = 0; c < 32; ++c) o32[c] *= cr[c];
                            tmem_st32(ta, o32);
                        }
                        tmem_wait_st();
                    }
                }
                // P^T row `row`: 64 BF16 values, MN-major with the 128-byte swizzle
                uint8_t *prow = sp + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4 w;
                    w.x = pack_bf16(s[8 * cc + 0], s[8 * cc + 1]);
                    w.y = pack_bf16(s[8 * cc + 2], s[8 * cc + 3]);
                    w.z = pack_bf16(s[8 * cc + 4], s[8 * cc + 5]);
                    w.w = pack_bf16(s[8 * cc + 6], s[8 * cc + 7]);
                    *reinterpret_cast<uint4 *>(prow + ((cc ^ (row & 7)) << 4)) = w;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&ctl->p_full);
            }
            if (aborted) break;
            fail = !warp_wait(&ctl->o_done, od_cnt & 1, abort_flag, p.dev_error, lim);
            ++od_cnt;
            tc_fence_after();
            {
                float r[32];
                reduce_scatter64<false>(lp, r, lane);
                *reinterpret_cast<float2 *>(&ctl->red[wl][2 * lane]) = make_float2(r[0], r[1]);
            }
            if (named_bar_or(1, 128, fail)) break;
            if (stid < 64) {
                const float L = ctl->red[0][stid] + ctl->red[1][stid] + ctl->red[2][stid] + ctl->red[3][stid];
                const float mr = ctl->m_run[stid];
                const bool live = L > 0.f;
                ctl->oscale[stid] = live ? p.kv_scale / L : 0.f;
                if (stid < u.rows_valid)
                    lbase[out_row0 + stid] = live ? (mr + log2f(L)) * 0.69314718055994531f : -INFINITY;
            }
            named_bar_sync(2, 128);
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                float o32[32];
                tmem_ld32(tmem + lane_base + 32 * j, o32);
                tmem_wait_ld();
                const int vcol = (j >> 1) * 128 + row;  // V dimension held by this lane
                const int c0 = (j & 1) * 32;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c0 + c < u.rows_valid)
                        obase[(out_row0 + c0 + c) * kVDim + vcol] = o32[c] * ctl->oscale[c0 + c];
            }
            tc_fence_before();
            mbar_arrive(&ctl->o_free);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------ plan
// One warp per request: stable per-rank compaction of the request's pages.
__global__ void plan_pages_kernel(int B, int N, long long num_pages, long long slots_per_rank,
                                  const int64_t *__restrict__ req_page_ptr,
                                  const int32_t *__restrict__ vpages, int32_t *__restrict__ counts,
                                  int32_t *__restrict__ comp_slot, int32_t *__restrict__ comp_page,
                                  int32_t *dev_error) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    const long long p0 = req_page_ptr[b], p1 = req_page_ptr[b + 1];
    int cnt[kMaxDcpAttn];
#pragma unroll
    for (int d = 0; d < kMaxDcpAttn; ++d) cnt[d] = 0;
    bool bad = false;
    for (long long base = p0; base < p1; base += 32) {
        const long long i = base + lane;
        int d = -1;
        int slot = 0;
        if (i < p1) {
            const int v = vpages[i];
            const int dd = N <= 1 ? 0 : v % N;
            const long long s = N <= 1 ? (long long)v : (long long)(v / N);
            if (v < 0 || s >= slots_per_rank) {
                bad = true;
            } else {
                d = dd;
                slot = (int)s;
            }
        }
#pragma unroll
        for (int dd = 0; dd < kMaxDcpAttn; ++dd) {
            if (dd >= N) break;
            const unsigned m = __ballot_sync(0xffffffffu, d == dd);
            if (d == dd) {
                const long long pos = (long long)dd * num_pages + p0 + cnt[dd] + __popc(m & ((1u << lane) - 1u));
                comp_slot[pos] = slot;
                comp_page[pos] = (int)(i - p0);
            }
            cnt[dd] += __popc(m);
        }
    }
    if (bad && dev_error) atomicOr(dev_error, DCP_DEVERR_OUT_OF_RANGE);
    if (lane == 0)
        for (int d = 0; d < N; ++d) counts[d * B + b] = cnt[d];
}

// Single block: chunk each (rank, request) pair, assign partial slots, emit units largest
// first with the G query groups of one chunk adjacent.
constexpr int kPlanThreads = 1024;

__device__ long long block_exclusive_scan(long long x, long long *scratch, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const long long t = scratch[lane];
        long long s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        scratch[lane] = s - t;
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    const long long r = scratch[warp] + incl - x;
    *total = scratch[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_units_kernel(int B, int N, int G, int only_rank, int tpc, const int32_t *__restrict__ counts,
                  int32_t *__restrict__ pair_chunks, int32_t *__restrict__ pair_part,
                  int4 *__restrict__ units, int *__restrict__ ctrl) {
    __shared__ int hist[kMaxTpc + 1];
    __shared__ long long scratch[33];
    const int n_pair = N * B;
    for (int i = threadIdx.x; i <= tpc; i += kPlanThreads) hist[i] = 0;
    __syncthreads();
    long long running = 0;
    for (int base = 0; base < n_pair; base += kPlanThreads) {
        const int pr = base + threadIdx.x;
        int chunks = 0, tiles = 0;
        if (pr < n_pair) {
            const int d = pr / B;
            if (only_rank < 0 || d == only_rank) {
                tiles = (counts[pr] + 1) >> 1;
                chunks = tiles == 0 ? 1 : (tiles + tpc - 1) / tpc;
            }
            pair_chunks[pr] = chunks;
        }
        long long tot;
        const long long need = chunks > 1 ? (long long)chunks * G : 0;
        const long long off = block_exclusive_scan(need, scratch, &tot);
        if (pr < n_pair) pair_part[pr] = chunks > 1 ? (int)(running + off) : -1;
        running += tot;
        for (int c = 0; c < chunks; ++c) {
            const int sz = min(tpc, tiles - c * tpc);
            atomicAdd(&hist[sz < 0 ? 0 : sz], 1);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // bucket offsets, largest size first (in units of chunks)
        int acc = 0;
        for (int s = tpc; s >= 0; --s) {
            const int h = hist[s];
            hist[s] = acc;
            acc += h;
        }
        ctrl[0] = acc * G;
        ctrl[1] = 0;
    }
    __syncthreads();
    for (int pr = threadIdx.x; pr < n_pair; pr += kPlanThreads) {
        const int chunks = pair_chunks[pr];
        if (chunks == 0) continue;
        const int tiles = (counts[pr] + 1) >> 1;
        const int cnt = counts[pr];
        for (int c = 0; c < chunks; ++c) {
            const int sz = max(0, min(tpc, tiles - c * tpc));
            const int slot = atomicAdd(&hist[sz], 1);
            const int page_begin = c * 2 * tpc;
            const int n_pages = max(0, min(2 * tpc, cnt - page_begin));
            for (int g = 0; g < G; ++g) {
                const int out = chunks > 1 ? pair_part[pr] + c * G + g : -1;
                units[(long long)slot * G + g] = make_int4(pr * G + g, page_begin, n_pages, out);
            }
        }
    }
}

// Merge the chunk partials of multi-chunk (rank, request) pairs into O_part / LSE_part.
__global__ void combine_kernel(int B, int T, int H, int HB, int G, int N, const int32_t *pair_chunks,
                               const int32_t *pair_part, const float *part_o, const float *part_lse,
                               float *o_part, float *lse_part) {
    const long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long n_tasks = (long long)N * B * G * kGroupRows;
    if (task >= n_tasks) return;
    const int c = (int)(task % kGroupRows);
    const long long pg = task / kGroupRows;
    const int g = (int)(pg % G);
    const int pr = (int)(pg / G);
    const int chunks = pair_chunks[pr];
    if (chunks <= 1) return;
    const int t = g / HB, hb = g % HB;
    const int rows_valid = min(kGroupRows, H - hb * kGroupRows);
    if (c >= rows_valid) return;
    const int d = pr / B, b = pr % B;
    const long long first = (long long)pair_part[pr] + g;  // chunk k lives at first + k * G
    const long long out_row = (long long)d * B * T * H + ((long long)(b * T + t) * H) + hb * kGroupRows + c;
    warp_merge_row512(chunks, part_o + (first * kGroupRows + c) * kVDim, (long long)G * kGroupRows * kVDim,
                      part_lse + first * kGroupRows + c, (long long)G * kGroupRows,
                      o_part + out_row * kVDim, lse_part + out_row, 1.f);
}

// ------------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D BF16 map over [rows][576] with 64 x 64 boxes and the 128-byte swizzle.
bool make_map_bf16(CUtensorMap *m, const void *ptr, uint64_t rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kKDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kKDim * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

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
    // Chunk size: equal-segment cost model, makespan in tiles with a partial round trip
    // (write + read of a 64 x 512 fp32 chunk output, in tile-equivalents of KV bytes).
    const long long pages_avg = B > 0 ? (num_pages + B - 1) / B : 0;
    const long long tiles_seg = std::max<long long>(1, ((pages_avg + N - 1) / N + 1) / 2);
    const long long n_seg = (long long)N * B * s->G;
    const double partial_cost = (2.0 * kGroupRows * kVDim * 4.0) / (128.0 * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1));
    double best = 1e300;
    long long tpc = tiles_seg;
    for (long long k = 1; k <= std::min<long long>(tiles_seg, 64); ++k) {
        const long long t = (tiles_seg + k - 1) / k;
        const long long chunks = (tiles_seg + t - 1) / t;
        const long long units = std::max<long long>(1, n_seg * chunks);
        const long long waves = (units + num_sms - 1) / num_sms;
        const double cost = (double)waves * ((double)t + (chunks > 1 ? partial_cost : 0.0));
        if (cost < best - 1e-9) {
            best = cost;
            tpc = t;
        }
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
    s->off_ctrl = off;    off = align256(off + sizeof(int32_t) * 4);
    s->off_part_o = off;  off = align256(off + sizeof(float) * (size_t)s->max_partials * kGroupRows * kVDim);
    s->off_part_lse = off; off = align256(off + sizeof(float) * (size_t)s->max_partials * kGroupRows);
    s->total_bytes = off;
    return true;
}

int launch_attention(const AttnArgs &a, int num_sms, cudaStream_t stream) {
    const AttnPlanShape &s = a.shape;
    if (a.dtype != DCP_KV_BF16) return DCP_ERR_UNSUPPORTED;
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

    const int warps_per_block = 4;
    plan_pages_kernel<<<(s.B + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, stream>>>(
        s.B, s.N, s.num_pages, a.slots_per_rank, a.req_page_ptr, a.dst_vpages, counts, comp_slot, comp_page,
        a.dev_error);
    if (cudaGetLastError() != cudaSuccess) return DCP_ERR_CUDA;
    plan_units_kernel<<<1, kPlanThreads, 0, stream>>>(s.B, s.N, s.G, a.only_rank, s.tiles_per_chunk, counts,
                                                       pair_chunks, pair_part, units, ctrl);
    if (cudaGetLastError() != cudaSuccess) return DCP_ERR_CUDA;

    AttnMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!make_map_bf16(&maps.q, a.q, (uint64_t)s.B * s.T * s.H)) return DCP_ERR_CUDA;
    for (int d = 0; d < s.N; ++d)
        if (!make_map_bf16(&maps.kv[d], a.kv_pools[d], (uint64_t)a.slots_per_rank * kPage)) return DCP_ERR_CUDA;
    KParams kp;
    kp.seq_lens = a.seq_lens;
    kp.req_page_ptr = a.req_page_ptr;
    kp.comp_slot = comp_slot;
    kp.comp_page = comp_page;
    kp.units = units;
    kp.ctrl = ctrl;
    kp.counter = ctrl + 1;
    kp.B = s.B;
    kp.T = s.T;
    kp.H = s.H;
    kp.HB = (s.H + kGroupRows - 1) / kGroupRows;
    kp.G = s.G;
    kp.num_pages = s.num_pages;
    kp.oob_row = (int)std::min<int64_t>((int64_t)a.slots_per_rank * kPage, 0x7fffff00);
    const float kappa = a.dtype == DCP_KV_FP8_E4M3 ? a.kv_scale : 1.f;
    kp.sl2 = a.softmax_scale * kappa * 1.4426950408889634f;
    kp.kv_scale = kappa;
    kp.o_part = a.o_part;
    kp.lse_part = a.lse_part;
    kp.part_o = part_o;
    kp.part_lse = part_lse;
    kp.dev_error = a.dev_error;
    kp.wait_limit_ns = a.wait_limit_ns;
    if (cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
        return DCP_ERR_CUDA;
    const long long max_units = s.max_units;
    const int grid = (int)std::max<long long>(1, std::min<long long>(num_sms, max_units));
    attn_kernel<<<grid, kThreads, kSmemBytes, stream>>>(maps, kp);
    if (cudaGetLastError() != cudaSuccess) return DCP_ERR_CUDA;
    const long long n_tasks = (long long)s.N * s.B * s.G * kGroupRows;
    const int cw = 8;
    combine_kernel<<<(unsigned)((n_tasks + cw - 1) / cw), 32 * cw, 0, stream>>>(
        s.B, s.T, s.H, kp.HB, s.G, s.N, pair_chunks, pair_part, part_o, part_lse, a.o_part, a.lse_part);
    if (cudaGetLastError() != cudaSuccess) return DCP_ERR_CUDA;
    return DCP_OK;
}

}  // namespace dcp
