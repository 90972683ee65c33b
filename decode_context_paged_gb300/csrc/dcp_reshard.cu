// dcp_reshard.cu -- page-level 2D KV reshard (CP layer-split -> DCP page-interleaved) and the
// source-side page-index filter.
//
// "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding":
//   2 (2D reshard target: every path (r, d) moves L_r x P_d), 5.1 (owner = p mod N_dcp,
//   local slot = p div N_dcp), 6.2 (page index filter), 6.3 (mask on the decode-side page
//   value, source indices pass through), 6.4 (the copy unit is the physical 64-token page).
//
// The reshard is a pure HBM->HBM byte move: every (layer, page) item is one contiguous page
// read and one contiguous page written.  Each CTA runs a single issuing thread that streams
// 36 KB chunks through a 6-stage shared-memory ring with TMA bulk copies (cp.async.bulk
// global->shared completing on an mbarrier, then shared->global in bulk groups), 3 loads ahead
// of the stores (copy_ring in dcp_copy_ring.cuh).  The grid is one CTA per SM for short copies
// and one per pair of SMs for long ones (ring_ctas below).  Work is split as contiguous chunk
// ranges of the flattened (layer, page, chunk) space; all (r, d) paths share the launch.
#include <cuda_runtime.h>

#include <cstdlib>

#include "dcp_copy_ring.cuh"
#include "dcp_internal.h"
#include "dcp_ptx.cuh"

namespace dcp {
namespace {

__global__ void __launch_bounds__(32, 1) reshard_kernel(const __grid_constant__ ReshardArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x != 0) return;
    const int64_t cpp = a.page_bytes / kRingChunk;  // chunks per page
    const int64_t n_layers = a.layer_end - a.layer_begin;
    const int64_t total = n_layers * a.num_pages * cpp;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t c_begin = (int64_t)blockIdx.x * per;
    const int64_t c_end = c_begin + per < total ? c_begin + per : total;
    int r = 0;
    auto map = [&](int64_t c, const uint8_t *&src, uint8_t *&dst) -> bool {
        const int64_t item = c / cpp;
        const int64_t part = c - item * cpp;
        const int l = a.layer_begin + (int)(item / a.num_pages);
        const int64_t p = item - (int64_t)(l - a.layer_begin) * a.num_pages;
        while (r + 1 < a.n_cp && l >= a.layer_start[r + 1]) ++r;
        while (r > 0 && l < a.layer_start[r]) --r;
        const int32_t v = __ldg(a.dst_vpages + p);
        const int32_t src_idx = __ldg(a.src_pages + p);
        int d;
        int64_t slot;
        if (a.n_dcp <= 1) {
            d = 0;
            slot = v;
        } else {
            d = v % a.n_dcp;
            slot = v / a.n_dcp;
        }
        if (v < 0 || slot >= a.dst_slots || src_idx < 0 || src_idx >= a.src_pool_pages) {
            if (part == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
            return false;
        }
        if (a.only_dst >= 0 && d != a.only_dst) return false;
        src = a.src_pools[r] + ((int64_t)(l - a.layer_start[r]) * a.src_pool_pages + src_idx) * a.page_bytes +
              part * kRingChunk;
        dst = a.dst_pools[d] + ((int64_t)l * a.dst_slots + slot) * a.page_bytes + part * kRingChunk;
        return true;
    };
    copy_ring(c_begin, c_end, map, smem, a.dev_error, a.wait_limit_ns);
}

// Token-interleaved layout ("SGLang's path": rank d holds tokens d, d + N, d + 2N, ...): every
// destination local page (layer l, entry e = jj N + d of request b) gathers its 64 rows, row i
// being token t = (64 jj + i) N + d, from row t mod 64 of the request's source page t div 64 of
// the CP rank that owns layer l.  One block per destination page (grid-stride): the page's 64
// source row offsets go to shared memory first, then every thread keeps kTokUnroll 16-byte loads
// in flight before their stores.
constexpr int kTokThreads = 256;
constexpr int kTokUnroll = 8;

__global__ void __launch_bounds__(kTokThreads) token_reshard_kernel(const __grid_constant__ TokenReshardArgs a) {
    __shared__ int64_t row_src[64];  // byte offset of row i's source row in its layer, or -1
    grid_dep_wait();
    grid_dep_launch();
    const int n = a.n_dcp <= 1 ? 1 : a.n_dcp;
    const int vecs = (int)(a.row_bytes / 16);
    const int64_t page_bytes = a.row_bytes * 64;
    const int64_t items = (int64_t)a.num_layers * a.num_tok_entries;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int l = (int)(item / a.num_tok_entries);
        const int64_t eg = item - (int64_t)l * a.num_tok_entries;
        int lo = 0, hi = a.num_requests;  // request b with tok_page_ptr[b] <= eg < tok_page_ptr[b + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.tok_page_ptr + mid) <= eg) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        const int64_t e = eg - __ldg(a.tok_page_ptr + b);
        const int64_t jj = e / n;
        const int d = (int)(e - jj * n);
        const int32_t v = __ldg(a.tok_vpages + eg);
        const int64_t slot = a.n_dcp <= 1 ? (int64_t)v : (int64_t)(v / a.n_dcp);
        const int owner = a.n_dcp <= 1 ? 0 : (int)(v % a.n_dcp);
        if (v < 0 || owner != d || slot >= a.dst_slots) {  // uniform over the block
            if (threadIdx.x == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
            continue;
        }
        int r = 0;
        while (r + 1 < a.n_cp && l >= a.layer_start[r + 1]) ++r;
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            const int64_t t = (64 * jj + i) * n + d;
            int64_t off = -1;
            if (t < (int64_t)__ldg(a.seq_lens + b)) {
                const int32_t sp = __ldg(a.src_pages + __ldg(a.src_page_ptr + b) + t / 64);
                if (sp < 0 || sp >= a.src_pool_pages) {
                    if (a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
                } else {
                    off = (int64_t)sp * page_bytes + (t % 64) * a.row_bytes;
                }
            }
            row_src[i] = off;
        }
        __syncthreads();
        uint8_t *dst = a.dst_pools[d] + ((int64_t)l * a.dst_slots + slot) * page_bytes;
        const uint8_t *src_layer = a.src_pools[r] + (int64_t)(l - a.layer_start[r]) * a.src_pool_pages * page_bytes;
        const int total = 64 * vecs;
        for (int base = threadIdx.x; base < total; base += kTokUnroll * kTokThreads) {
            uint4 x[kTokUnroll];
            int dst_vec[kTokUnroll];  // vector index within the destination page, or -1
#pragma unroll
            for (int u = 0; u < kTokUnroll; ++u) {
                const int idx = base + u * kTokThreads;
                dst_vec[u] = -1;
                if (idx < total) {
                    const int i = idx / vecs, c = idx - i * vecs;
                    const int64_t off = row_src[i];
                    if (off >= 0) {
                        x[u] = __ldg(reinterpret_cast<const uint4 *>(src_layer + off) + c);
                        dst_vec[u] = idx;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kTokUnroll; ++u)
                if (dst_vec[u] >= 0) reinterpret_cast<uint4 *>(dst)[dst_vec[u]] = x[u];
        }
        __syncthreads();  // row_src is rewritten by the next item
    }
}

// The pages' initial design, kept as a bandwidth baseline ("Design Evolution", 6.1).
// Mode 0 (full transfer): every page entry of every layer to every DCP rank's receive buffer
// [layer][page entry] (N_dcp times the KV).  Mode 1 (in-place shard): each page entry of each
// layer from its owner's receive buffer to the owner's DCP slot.
__global__ void __launch_bounds__(32, 1) naive_kernel(const __grid_constant__ NaiveArgs na) {
    extern __shared__ __align__(128) uint8_t smem[];
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x != 0) return;
    const ReshardArgs &a = na.base;
    const int64_t cpp = a.page_bytes / kRingChunk;
    const int64_t lp = (int64_t)a.layer_end * a.num_pages;  // (layer, entry) items of one rank
    const int n_dst = a.n_dcp <= 1 ? 1 : a.n_dcp;
    const int64_t total = (na.mode == 0 ? n_dst : 1) * lp * cpp;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t c_begin = (int64_t)blockIdx.x * per;
    const int64_t c_end = c_begin + per < total ? c_begin + per : total;
    int r = 0;
    auto map = [&](int64_t c, const uint8_t *&src, uint8_t *&dst) -> bool {
        const int64_t item = c / cpp, part = c - item * cpp;
        const int64_t li = item % lp;  // layer * num_pages + entry
        const int l = (int)(li / a.num_pages);
        const int64_t i = li - (int64_t)l * a.num_pages;
        if (na.mode == 0) {
            const int d = (int)(item / lp);
            while (r + 1 < a.n_cp && l >= a.layer_start[r + 1]) ++r;
            while (r > 0 && l < a.layer_start[r]) --r;
            const int32_t s_idx = __ldg(a.src_pages + i);
            if (s_idx < 0 || s_idx >= a.src_pool_pages) {
                if (part == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
                return false;
            }
            src = a.src_pools[r] + ((int64_t)(l - a.layer_start[r]) * a.src_pool_pages + s_idx) * a.page_bytes +
                  part * kRingChunk;
            dst = na.recv[d] + li * a.page_bytes + part * kRingChunk;
            return true;
        }
        const int32_t v = __ldg(a.dst_vpages + i);
        const int d = a.n_dcp <= 1 ? 0 : v % a.n_dcp;
        const int64_t slot = a.n_dcp <= 1 ? (int64_t)v : (int64_t)(v / a.n_dcp);
        if (v < 0 || slot >= a.dst_slots) {
            if (part == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
            return false;
        }
        src = na.recv[d] + li * a.page_bytes + part * kRingChunk;
        dst = a.dst_pools[d] + ((int64_t)l * a.dst_slots + slot) * a.page_bytes + part * kRingChunk;
        return true;
    };
    copy_ring(c_begin, c_end, map, smem, a.dev_error, a.wait_limit_ns);
}

// Pack (to_staging) or unpack one path's items k in [item_begin, item_begin + n_items):
// layer j = k / n_idx, list entry i = k % n_idx; staging page k - item_begin.
__global__ void __launch_bounds__(32, 1) pack_kernel(const __grid_constant__ PackArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x != 0) return;
    const int64_t cpp = a.page_bytes / kRingChunk;
    const int64_t total = a.n_items * cpp;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t c_begin = (int64_t)blockIdx.x * per;
    const int64_t c_end = c_begin + per < total ? c_begin + per : total;
    auto map = [&](int64_t c, const uint8_t *&src, uint8_t *&dst) -> bool {
        const int64_t m = c / cpp, part = c - m * cpp;  // staging page m = item item_begin + m
        const int64_t k = a.item_begin + m;
        const int64_t j = k / a.n_idx, i = k - j * a.n_idx;
        const int32_t idx = __ldg(a.idx + i);
        uint8_t *stage = a.staging + m * a.page_bytes + part * kRingChunk;
        if (a.to_staging) {
            if (j >= a.n_layers || idx < 0 || idx >= a.pool_pages) {
                if (part == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
                return false;
            }
            src = a.pool + (j * a.pool_pages + idx) * a.page_bytes + part * kRingChunk;
            dst = stage;
        } else {
            const int64_t l = a.layer_offset + j;
            if (j >= a.n_layers || l < 0 || l >= a.pool_layers || idx < 0 || idx >= a.pool_pages) {
                if (part == 0 && a.dev_error) atomicOr(a.dev_error, DCP_DEVERR_OUT_OF_RANGE);
                return false;
            }
            src = stage;
            dst = a.pool + (l * a.pool_pages + idx) * a.page_bytes + part * kRingChunk;
        }
        return true;
    };
    copy_ring(c_begin, c_end, map, smem, a.dev_error, a.wait_limit_ns);
}

// Stable single-block compaction: keep entries whose decode-side page value belongs to rank d.
constexpr int kFilterThreads = 1024;
constexpr int kFilterItems = 8;

__global__ void __launch_bounds__(kFilterThreads)
filter_kernel(int64_t n, const int32_t *__restrict__ dst_vpages,
              const int32_t *__restrict__ transfer_idx, int n_dcp, int d,
              int32_t *__restrict__ out_slot, int32_t *__restrict__ out_src,
              int64_t *__restrict__ out_count) {
    __shared__ int warp_tot[kFilterThreads / 32];
    __shared__ int64_t running;
    grid_dep_wait();
    grid_dep_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) running = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += (int64_t)kFilterThreads * kFilterItems) {
        const int64_t i0 = base + (int64_t)tid * kFilterItems;
        int keep = 0;
        int32_t vals[kFilterItems];
#pragma unroll
        for (int k = 0; k < kFilterItems; ++k) {
            const int64_t i = i0 + k;
            vals[k] = i < n ? __ldg(dst_vpages + i) : -1;
            const bool kept = i < n && (n_dcp <= 1 || vals[k] % n_dcp == d);
            keep |= (int)kept << k;
        }
        const int cnt = __popc(keep);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
            int s = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_tot[lane] = s - t;  // exclusive prefix over warps
        }
        __syncthreads();
        int64_t pos = running + warp_tot[warp] + (incl - cnt);
#pragma unroll
        for (int k = 0; k < kFilterItems; ++k) {
            if (keep & (1 << k)) {
                out_slot[pos] = n_dcp <= 1 ? vals[k] : vals[k] / n_dcp;
                if (transfer_idx) out_src[pos] = __ldg(transfer_idx + i0 + k);
                ++pos;
            }
        }
        __syncthreads();
        if (tid == kFilterThreads - 1) running = pos;
        __syncthreads();
    }
    if (tid == 0) *out_count = running;
}

}  // namespace

// CTAs of the copy-ring kernels for a copy of `bytes` (read + write).  Long copies run one CTA per
// pair of SMs: measured on GB300 (152 SMs), 76 streaming CTAs beat 152 by 4-6% on copies of 5 to
// 53 GB (the reshard reaches 99-100% of the copy peak) and 60 to 114 CTAs land in between
// (plausibly the two SMs of a pair share their way to memory, so a second stream on a pair adds
// queueing rather than bandwidth).  Short copies keep one CTA per SM: on a 0.6 GB reshard inside
// a decode step, 152 CTAs are 1-2% faster (the shorter ramp counts more).  The switch sits at
// 16 MB per CTA of the half grid.
// DCP_RING_CTAS (environment, a positive count) overrides the choice; the tests use it to run
// the copy kernels on grids of other sizes.
inline int ring_ctas(int num_sms, int64_t bytes) {
    const char *e = std::getenv("DCP_RING_CTAS");
    if (e && *e) {
        const long v = std::strtol(e, nullptr, 10);
        if (v > 0) return (int)(v < 65535 ? v : 65535);
    }
    const int half = num_sms > 1 ? num_sms / 2 : 1;
    return bytes >= (int64_t)half * (16ll << 20) ? half : num_sms;
}

cudaError_t launch_reshard(const ReshardArgs &a, int num_sms, cudaStream_t stream) {
    if ((a.layer_end - a.layer_begin) <= 0 || a.num_pages <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(reshard_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRingSmem);
    if (e != cudaSuccess) return e;
    const int64_t bytes = 2 * a.num_pages * (int64_t)(a.layer_end - a.layer_begin) * a.page_bytes;
    return launch_pdl(reshard_kernel, dim3(ring_ctas(num_sms, bytes)), dim3(32), kRingSmem, stream, a);
}

cudaError_t launch_token_reshard(const TokenReshardArgs &a, int num_sms, cudaStream_t stream) {
    const int64_t items = (int64_t)a.num_layers * a.num_tok_entries;
    if (items <= 0) return cudaSuccess;
    // one resident wave, items taken grid-stride (measured on batch: 91.9% of the copy peak,
    // against 88.7% for two waves of 8 blocks per SM and 72.6% for 2 blocks per SM)
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, token_reshard_kernel, kTokThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const long long wave = (long long)per_sm * num_sms;
    const int grid = (int)(items < wave ? items : wave);
    return launch_pdl(token_reshard_kernel, dim3(grid), dim3(kTokThreads), 0, stream, a);
}

cudaError_t launch_naive(const NaiveArgs &a, int num_sms, cudaStream_t stream) {
    if (a.base.layer_end <= 0 || a.base.num_pages <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(naive_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingSmem);
    if (e != cudaSuccess) return e;
    const int n_dst = a.mode == 0 ? (a.base.n_dcp <= 1 ? 1 : a.base.n_dcp) : 1;
    const int64_t bytes = 2 * (int64_t)n_dst * a.base.layer_end * a.base.num_pages * a.base.page_bytes;
    return launch_pdl(naive_kernel, dim3(ring_ctas(num_sms, bytes)), dim3(32), kRingSmem, stream, a);
}

cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream) {
    if (a.n_items <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingSmem);
    if (e != cudaSuccess) return e;
    const int64_t chunks = a.n_items * (a.page_bytes / kRingChunk);
    const int ctas = ring_ctas(num_sms, 2 * a.n_items * a.page_bytes);
    const int grid = (int)(chunks < ctas ? chunks : ctas);
    return launch_pdl(pack_kernel, dim3(grid), dim3(32), kRingSmem, stream, a);
}

cudaError_t launch_filter(int64_t n, const int32_t *dst_vpages, const int32_t *transfer_idx,
                          int n_dcp, int d, int32_t *out_slot, int32_t *out_src,
                          int64_t *out_count, cudaStream_t stream) {
    return launch_pdl(filter_kernel, dim3(1), dim3(kFilterThreads), 0, stream, n, dst_vpages, transfer_idx, n_dcp, d,
                      out_slot, out_src, out_count);
}

}  // namespace dcp
