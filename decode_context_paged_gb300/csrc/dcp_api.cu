// dcp_api.cu -- the C ABI of libdcp.so: argument validation on the host, then launches.
//
// Every entry point checks shapes, pointers and alignment before anything runs and returns a
// dcp_status; nothing here allocates device memory or keeps state between calls.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "dcp_internal.h"

using namespace dcp;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int current_sm_count(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DCP_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DCP_ERR_CUDA;
    return DCP_OK;
}

// Wait limit for device pipeline waits; DCP_WAIT_LIMIT_NS overrides the default.
uint64_t wait_limit_ns() {
    const char *e = std::getenv("DCP_WAIT_LIMIT_NS");
    if (e && *e) {
        const unsigned long long v = std::strtoull(e, nullptr, 10);
        if (v > 0) return v;
    }
    return kWaitLimitNs;
}

// Layer assignment of "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding", 4.1 (restated
// here for the library; see dcp_layer_range).
void layer_range(int n_layers, int n_cp, int r, int *s, int *e) {
    const int base = n_layers / n_cp, extra = n_layers % n_cp;
    *s = r * base + (r < extra ? r : extra);
    *e = *s + base + (r < extra ? 1 : 0);
}

}  // namespace

extern "C" {

int dcp_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *dcp_status_string(int status) {
    switch (status) {
        case DCP_OK: return "ok";
        case DCP_ERR_INVALID_ARG: return "invalid argument";
        case DCP_ERR_OUT_OF_RANGE: return "page index outside its pool";
        case DCP_ERR_UNSUPPORTED: return "unsupported configuration";
        case DCP_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case DCP_ERR_CUDA: return "CUDA runtime error";
        case DCP_ERR_TIMEOUT: return "device pipeline wait timed out";
        default: return "unknown status";
    }
}

int dcp_device_error_status(int32_t word) {
    if (word & DCP_DEVERR_TIMEOUT) return DCP_ERR_TIMEOUT;
    if (word & DCP_DEVERR_OUT_OF_RANGE) return DCP_ERR_OUT_OF_RANGE;
    if (word & DCP_DEVERR_PLAN_MISMATCH) return DCP_ERR_WORKSPACE;
    if (word & DCP_DEVERR_LAYOUT) return DCP_ERR_UNSUPPORTED;
    return DCP_OK;
}

int dcp_layer_range(int n_layers, int n_cp, int r, int *start, int *end) {
    if (n_layers < 0 || n_cp < 1 || r < 0 || r >= n_cp || !start || !end) return DCP_ERR_INVALID_ARG;
    layer_range(n_layers, n_cp, r, start, end);
    return DCP_OK;
}

int dcp_filter_page_indices(int64_t n, const int32_t *dst_vpages, const int32_t *transfer_idx,
                            int n_dcp, int d, int32_t *out_slot, int32_t *out_src,
                            int64_t *out_count, dcp_stream_t stream) {
    if (n < 0 || n_dcp < 1 || d < 0 || d >= n_dcp || !out_count) return DCP_ERR_INVALID_ARG;
    if (n > 0 && (!dst_vpages || !out_slot)) return DCP_ERR_INVALID_ARG;
    if (transfer_idx && !out_src) return DCP_ERR_INVALID_ARG;
    if (launch_filter(n, dst_vpages, transfer_idx, n_dcp, d, out_slot, out_src, out_count,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DCP_ERR_CUDA;
    return DCP_OK;
}

int dcp_reshard_pages(int num_requests, const int64_t *req_page_ptr, int64_t num_pages,
                      const int32_t *src_pages, const int32_t *dst_vpages, int page_size,
                      int row_elems, int dtype, int num_layers, int n_cp,
                      const void *const *src_pools, int64_t src_pool_pages, int n_dcp,
                      void *const *dst_pools, int64_t dst_slots_per_rank, int only_src_rank,
                      int only_dst_rank, int32_t *dev_error, dcp_stream_t stream) {
    if (num_requests < 0 || num_pages < 0 || page_size != kPage || row_elems != kKDim) return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (num_layers < 0 || n_cp < 1 || n_cp > kMaxCp || n_dcp < 1 || n_dcp > kMaxDcpReshard) return DCP_ERR_INVALID_ARG;
    if (only_src_rank < -1 || only_src_rank >= n_cp || only_dst_rank < -1 || only_dst_rank >= n_dcp)
        return DCP_ERR_INVALID_ARG;
    if (src_pool_pages < 0 || dst_slots_per_rank < 0) return DCP_ERR_INVALID_ARG;
    if (num_requests == 0 || num_pages == 0 || num_layers == 0) return DCP_OK;
    if (!req_page_ptr || !src_pages || !dst_vpages || !src_pools || !dst_pools) return DCP_ERR_INVALID_ARG;
    ReshardArgs a{};
    a.req_page_ptr = req_page_ptr;
    a.src_pages = src_pages;
    a.dst_vpages = dst_vpages;
    a.num_requests = num_requests;
    a.num_pages = num_pages;
    a.page_bytes = (int64_t)kPage * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1);
    a.n_cp = n_cp;
    for (int r = 0; r < n_cp; ++r) {
        int s, e;
        layer_range(num_layers, n_cp, r, &s, &e);
        a.layer_start[r] = s;
        a.layer_start[r + 1] = e;
        a.src_pools[r] = static_cast<const uint8_t *>(src_pools[r]);
        if ((e > s) && (!src_pools[r] || !aligned(src_pools[r], 16))) return DCP_ERR_INVALID_ARG;
    }
    if (only_src_rank >= 0) {
        a.layer_begin = a.layer_start[only_src_rank];
        a.layer_end = a.layer_start[only_src_rank + 1];
    } else {
        a.layer_begin = 0;
        a.layer_end = num_layers;
    }
    a.src_pool_pages = src_pool_pages;
    a.n_dcp = n_dcp;
    for (int d = 0; d < n_dcp; ++d) {
        if (!dst_pools[d] || !aligned(dst_pools[d], 16)) return DCP_ERR_INVALID_ARG;
        a.dst_pools[d] = static_cast<uint8_t *>(dst_pools[d]);
    }
    a.dst_slots = dst_slots_per_rank;
    a.only_dst = only_dst_rank;
    a.dev_error = dev_error;
    a.wait_limit_ns = wait_limit_ns();
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    if (launch_reshard(a, sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DCP_ERR_CUDA;
    return DCP_OK;
}

int dcp_token_reshard(int num_requests, const int32_t *seq_lens, const int64_t *src_page_ptr,
                      const int32_t *src_pages, const int64_t *tok_page_ptr, int64_t num_tok_entries,
                      const int32_t *tok_vpages, int dtype, int num_layers, int n_cp, const void *const *src_pools,
                      int64_t src_pool_pages, int n_dcp, void *const *dst_pools, int64_t dst_slots_per_rank,
                      int32_t *dev_error, dcp_stream_t stream) {
    if (num_requests < 0 || num_tok_entries < 0 || num_layers < 0 || src_pool_pages < 0 || dst_slots_per_rank < 0)
        return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_cp < 1 || n_cp > kMaxCp || n_dcp < 1 || n_dcp > kMaxDcpReshard) return DCP_ERR_INVALID_ARG;
    if (num_requests == 0 || num_tok_entries == 0 || num_layers == 0) return DCP_OK;
    if (!seq_lens || !src_page_ptr || !src_pages || !tok_page_ptr || !tok_vpages || !src_pools || !dst_pools)
        return DCP_ERR_INVALID_ARG;
    TokenReshardArgs a{};
    a.seq_lens = seq_lens;
    a.src_page_ptr = src_page_ptr;
    a.src_pages = src_pages;
    a.tok_page_ptr = tok_page_ptr;
    a.tok_vpages = tok_vpages;
    a.num_requests = num_requests;
    a.num_tok_entries = num_tok_entries;
    a.row_bytes = (int64_t)kKDim * (dtype == DCP_KV_BF16 ? 2 : 1);
    a.num_layers = num_layers;
    a.n_cp = n_cp;
    for (int r = 0; r < n_cp; ++r) {
        int s0, e0;
        layer_range(num_layers, n_cp, r, &s0, &e0);
        a.layer_start[r] = s0;
        a.layer_start[r + 1] = e0;
        a.src_pools[r] = static_cast<const uint8_t *>(src_pools[r]);
        if ((e0 > s0) && (!src_pools[r] || !aligned(src_pools[r], 16))) return DCP_ERR_INVALID_ARG;
    }
    a.src_pool_pages = src_pool_pages;
    a.n_dcp = n_dcp;
    for (int d = 0; d < n_dcp; ++d) {
        if (!dst_pools[d] || !aligned(dst_pools[d], 16)) return DCP_ERR_INVALID_ARG;
        a.dst_pools[d] = static_cast<uint8_t *>(dst_pools[d]);
    }
    a.dst_slots = dst_slots_per_rank;
    a.dev_error = dev_error;
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    return launch_token_reshard(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

int dcp_naive_full_transfer(int64_t num_pages, const int32_t *src_pages, int dtype, int num_layers, int n_cp,
                            const void *const *src_pools, int64_t src_pool_pages, int n_dcp, void *const *recv_bufs,
                            int32_t *dev_error, dcp_stream_t stream) {
    if (num_pages < 0 || num_layers < 0 || src_pool_pages < 0) return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_cp < 1 || n_cp > kMaxCp || n_dcp < 1 || n_dcp > kMaxDcpReshard) return DCP_ERR_INVALID_ARG;
    if (num_pages == 0 || num_layers == 0) return DCP_OK;
    if (!src_pages || !src_pools || !recv_bufs) return DCP_ERR_INVALID_ARG;
    NaiveArgs na{};
    ReshardArgs &a = na.base;
    a.src_pages = src_pages;
    a.num_pages = num_pages;
    a.page_bytes = (int64_t)kPage * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1);
    a.n_cp = n_cp;
    for (int r = 0; r < n_cp; ++r) {
        int s0, e0;
        layer_range(num_layers, n_cp, r, &s0, &e0);
        a.layer_start[r] = s0;
        a.layer_start[r + 1] = e0;
        a.src_pools[r] = static_cast<const uint8_t *>(src_pools[r]);
        if ((e0 > s0) && (!src_pools[r] || !aligned(src_pools[r], 16))) return DCP_ERR_INVALID_ARG;
    }
    a.layer_begin = 0;
    a.layer_end = num_layers;
    a.src_pool_pages = src_pool_pages;
    a.n_dcp = n_dcp;
    for (int d = 0; d < n_dcp; ++d) {
        if (!recv_bufs[d] || !aligned(recv_bufs[d], 16)) return DCP_ERR_INVALID_ARG;
        na.recv[d] = static_cast<uint8_t *>(recv_bufs[d]);
    }
    a.dev_error = dev_error;
    a.wait_limit_ns = wait_limit_ns();
    na.mode = 0;
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    return launch_naive(na, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

int dcp_naive_inplace_shard(int64_t num_pages, const int32_t *dst_vpages, int dtype, int num_layers, int n_dcp,
                            const void *const *recv_bufs, void *const *dst_pools, int64_t dst_slots_per_rank,
                            int32_t *dev_error, dcp_stream_t stream) {
    if (num_pages < 0 || num_layers < 0 || dst_slots_per_rank < 0) return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_dcp < 1 || n_dcp > kMaxDcpReshard) return DCP_ERR_INVALID_ARG;
    if (num_pages == 0 || num_layers == 0) return DCP_OK;
    if (!dst_vpages || !recv_bufs || !dst_pools) return DCP_ERR_INVALID_ARG;
    NaiveArgs na{};
    ReshardArgs &a = na.base;
    a.dst_vpages = dst_vpages;
    a.num_pages = num_pages;
    a.page_bytes = (int64_t)kPage * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1);
    a.n_cp = 1;
    a.layer_begin = 0;
    a.layer_end = num_layers;
    a.n_dcp = n_dcp;
    for (int d = 0; d < n_dcp; ++d) {
        if (!recv_bufs[d] || !aligned(recv_bufs[d], 16) || !dst_pools[d] || !aligned(dst_pools[d], 16))
            return DCP_ERR_INVALID_ARG;
        na.recv[d] = static_cast<uint8_t *>(const_cast<void *>(recv_bufs[d]));
        a.dst_pools[d] = static_cast<uint8_t *>(dst_pools[d]);
    }
    a.dst_slots = dst_slots_per_rank;
    a.dev_error = dev_error;
    a.wait_limit_ns = wait_limit_ns();
    na.mode = 1;
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    return launch_naive(na, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

static int pack_impl(int64_t n_idx, const int32_t *idx, int n_layers, int layer_offset, int64_t item_begin,
                     int64_t n_items, int dtype, const void *pool, int64_t pool_pages, int pool_layers,
                     const void *staging, size_t staging_bytes, int to_staging, int32_t *dev_error,
                     dcp_stream_t stream) {
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_idx < 0 || n_layers < 0 || item_begin < 0 || n_items < 0 || pool_pages < 0 || pool_layers < 0)
        return DCP_ERR_INVALID_ARG;
    if (n_items == 0) return DCP_OK;
    if (n_idx == 0 || item_begin + n_items > n_idx * (int64_t)n_layers) return DCP_ERR_INVALID_ARG;
    const int64_t page_bytes = (int64_t)kPage * kKDim * (dtype == DCP_KV_BF16 ? 2 : 1);
    if (!idx || !pool || !staging || !aligned(pool, 16) || !aligned(staging, 16)) return DCP_ERR_INVALID_ARG;
    if ((int64_t)staging_bytes < n_items * page_bytes) return DCP_ERR_INVALID_ARG;
    PackArgs a{};
    a.idx = idx;
    a.n_idx = n_idx;
    a.n_layers = n_layers;
    a.layer_offset = layer_offset;
    a.item_begin = item_begin;
    a.n_items = n_items;
    a.page_bytes = page_bytes;
    a.pool = static_cast<uint8_t *>(const_cast<void *>(pool));
    a.pool_pages = pool_pages;
    a.pool_layers = pool_layers;
    a.staging = static_cast<uint8_t *>(const_cast<void *>(staging));
    a.to_staging = to_staging;
    a.dev_error = dev_error;
    a.wait_limit_ns = wait_limit_ns();
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    return launch_pack(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

int dcp_pack_pages(int64_t n_idx, const int32_t *src_idx, int n_layers, int64_t item_begin, int64_t n_items,
                   int dtype, const void *src_pool, int64_t src_pool_pages, void *staging, size_t staging_bytes,
                   int32_t *dev_error, dcp_stream_t stream) {
    return pack_impl(n_idx, src_idx, n_layers, 0, item_begin, n_items, dtype, src_pool, src_pool_pages, n_layers,
                     staging, staging_bytes, 1, dev_error, stream);
}

int dcp_unpack_pages(int64_t n_idx, const int32_t *dst_slot, int n_layers, int layer_offset, int64_t item_begin,
                     int64_t n_items, int dtype, const void *staging, size_t staging_bytes, void *dst_pool,
                     int num_layers, int64_t dst_slots, int32_t *dev_error, dcp_stream_t stream) {
    return pack_impl(n_idx, dst_slot, n_layers, layer_offset, item_begin, n_items, dtype, dst_pool, dst_slots,
                     num_layers, staging, staging_bytes, 0, dev_error, stream);
}

size_t dcp_partial_decode_attn_workspace_size(int num_requests, int q_len, int num_heads, int n_dcp,
                                              int64_t num_pages) {
    int sms = 0;
    if (current_sm_count(&sms) != DCP_OK) return 0;
    AttnPlanShape s;
    if (!plan_attention(num_requests, q_len, num_heads, n_dcp, num_pages, DCP_KV_BF16, sms, &s)) return 0;
    AttnPlanShape s8;
    plan_attention(num_requests, q_len, num_heads, n_dcp, num_pages, DCP_KV_FP8_E4M3, sms, &s8);
    return s.total_bytes > s8.total_bytes ? s.total_bytes : s8.total_bytes;
}

static int partial_attn_impl(int num_requests, int q_len, int num_heads, const void *q,
                            const int32_t *seq_lens, const int64_t *req_page_ptr,
                            int64_t num_pages, const int32_t *dst_vpages, int page_size,
                            int dtype, float kv_scale, float softmax_scale, int n_dcp,
                            const void *const *kv_pools, int64_t slots_per_rank, int only_rank,
                            float *o_part, float *lse_part, float *o_out, float *lse_out, void *workspace,
                            size_t workspace_bytes, int32_t *dev_error, dcp_stream_t stream,
                            int token_layout = 0, int phase = 0) {
    if (num_requests < 0 || q_len < 1 || num_heads < 1 || num_pages < 0 || page_size != kPage)
        return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_dcp < 1 || n_dcp > kMaxDcpAttn || only_rank < -1 || only_rank >= n_dcp) return DCP_ERR_INVALID_ARG;
    if (slots_per_rank < 1 || slots_per_rank * kPage > 0x7fffff00LL) return DCP_ERR_INVALID_ARG;
    if ((int64_t)num_requests * q_len * num_heads > 0x7fffff00LL) return DCP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || (dtype == DCP_KV_FP8_E4M3 && !(kv_scale > 0.f))) return DCP_ERR_INVALID_ARG;
    if (num_requests == 0) return DCP_OK;
    if (!q || !seq_lens || !req_page_ptr || !o_part || !lse_part || !kv_pools) return DCP_ERR_INVALID_ARG;
    if (num_pages > 0 && !dst_vpages) return DCP_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(o_part, 16)) return DCP_ERR_INVALID_ARG;
    for (int d = 0; d < n_dcp; ++d)
        if (!kv_pools[d] || !aligned(kv_pools[d], 16)) return DCP_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    AttnArgs a{};
    if (!plan_attention(num_requests, q_len, num_heads, n_dcp, num_pages, dtype, sms, &a.shape))
        return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < a.shape.total_bytes || !aligned(workspace, 256)) return DCP_ERR_WORKSPACE;
    a.q = q;
    a.seq_lens = seq_lens;
    a.req_page_ptr = req_page_ptr;
    a.dst_vpages = dst_vpages;
    a.dtype = dtype;
    a.kv_scale = kv_scale;
    a.softmax_scale = softmax_scale;
    for (int d = 0; d < n_dcp; ++d) a.kv_pools[d] = kv_pools[d];
    a.slots_per_rank = slots_per_rank;
    a.only_rank = only_rank;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.o_out = o_out;
    a.lse_out = lse_out;
    a.token_layout = token_layout;
    a.phase = phase;
    a.workspace = static_cast<uint8_t *>(workspace);
    a.dev_error = dev_error;
    a.wait_limit_ns = wait_limit_ns();
    return launch_attention(a, sms, reinterpret_cast<cudaStream_t>(stream));
}

int dcp_partial_decode_attn(int num_requests, int q_len, int num_heads, const void *q,
                            const int32_t *seq_lens, const int64_t *req_page_ptr,
                            int64_t num_pages, const int32_t *dst_vpages, int page_size,
                            int dtype, float kv_scale, float softmax_scale, int n_dcp,
                            const void *const *kv_pools, int64_t slots_per_rank, int only_rank,
                            float *o_part, float *lse_part, void *workspace,
                            size_t workspace_bytes, int32_t *dev_error, dcp_stream_t stream) {
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, only_rank,
                             o_part, lse_part, nullptr, nullptr, workspace, workspace_bytes, dev_error, stream);
}

int dcp_partial_decode_attn_tokens(int num_requests, int q_len, int num_heads, const void *q,
                                   const int32_t *seq_lens, const int64_t *req_page_ptr, int64_t num_pages,
                                   const int32_t *dst_vpages, int page_size, int dtype, float kv_scale,
                                   float softmax_scale, int n_dcp, const void *const *kv_pools,
                                   int64_t slots_per_rank, int only_rank, float *o_part, float *lse_part,
                                   void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                   dcp_stream_t stream) {
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, only_rank,
                             o_part, lse_part, nullptr, nullptr, workspace, workspace_bytes, dev_error, stream, 1);
}

int dcp_attn_plan(int num_requests, int q_len, int num_heads, const int64_t *req_page_ptr, int64_t num_pages,
                  const int32_t *dst_vpages, int dtype, int n_dcp, int64_t slots_per_rank, int only_rank,
                  void *workspace, size_t workspace_bytes, int32_t *dev_error, dcp_stream_t stream) {
    // The plan reads neither Q nor the pools: placeholders that pass the argument checks.
    static const uint8_t dummy[16] __attribute__((aligned(16))) = {};
    const void *pools[kMaxDcpAttn];
    for (int d = 0; d < kMaxDcpAttn; ++d) pools[d] = dummy;
    if (num_requests > 0 && !req_page_ptr) return DCP_ERR_INVALID_ARG;
    return partial_attn_impl(num_requests, q_len, num_heads, dummy, reinterpret_cast<const int32_t *>(dummy),
                             req_page_ptr, num_pages, dst_vpages, kPage, dtype, 1.f, 1.f, n_dcp, pools, slots_per_rank,
                             only_rank, reinterpret_cast<float *>(const_cast<uint8_t *>(dummy)),
                             reinterpret_cast<float *>(const_cast<uint8_t *>(dummy)), nullptr, nullptr, workspace,
                             workspace_bytes, dev_error, stream, 0, 1);
}

int dcp_attn_plan_info(int num_requests, int q_len, int num_heads, int64_t num_pages, int dtype, int n_dcp,
                       const void *workspace, size_t workspace_bytes, int32_t *info, dcp_stream_t stream) {
    if (num_requests < 0 || q_len < 1 || num_heads < 1 || num_pages < 0 || !info) return DCP_ERR_INVALID_ARG;
    if (dtype != DCP_KV_BF16 && dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
    if (n_dcp < 1 || n_dcp > kMaxDcpAttn) return DCP_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = current_sm_count(&sms)) return st;
    AttnPlanShape s;
    if (!plan_attention(num_requests, q_len, num_heads, n_dcp, num_pages, dtype, sms, &s)) return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < s.total_bytes || !aligned(workspace, 256)) return DCP_ERR_WORKSPACE;
    return read_plan_info(s, workspace, info, reinterpret_cast<cudaStream_t>(stream));
}

int dcp_partial_decode_attn_run(int num_requests, int q_len, int num_heads, const void *q, const int32_t *seq_lens,
                                const int64_t *req_page_ptr, int64_t num_pages, const int32_t *dst_vpages,
                                int page_size, int dtype, float kv_scale, float softmax_scale, int n_dcp,
                                const void *const *kv_pools, int64_t slots_per_rank, int only_rank, float *o_part,
                                float *lse_part, void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                dcp_stream_t stream) {
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, only_rank,
                             o_part, lse_part, nullptr, nullptr, workspace, workspace_bytes, dev_error, stream, 0, 2);
}

int dcp_decode_attn_merged_run(int num_requests, int q_len, int num_heads, const void *q, const int32_t *seq_lens,
                               const int64_t *req_page_ptr, int64_t num_pages, const int32_t *dst_vpages,
                               int page_size, int dtype, float kv_scale, float softmax_scale, int n_dcp,
                               const void *const *kv_pools, int64_t slots_per_rank, float *o_part, float *lse_part,
                               float *o_out, float *lse_out, void *workspace, size_t workspace_bytes,
                               int32_t *dev_error, dcp_stream_t stream) {
    if (num_requests > 0 && (!o_out || !lse_out || !aligned(o_out, 16))) return DCP_ERR_INVALID_ARG;
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, -1, o_part,
                             lse_part, o_out, lse_out, workspace, workspace_bytes, dev_error, stream, 0, 2);
}

int dcp_decode_attn_merged_tokens(int num_requests, int q_len, int num_heads, const void *q,
                                  const int32_t *seq_lens, const int64_t *req_page_ptr, int64_t num_pages,
                                  const int32_t *dst_vpages, int page_size, int dtype, float kv_scale,
                                  float softmax_scale, int n_dcp, const void *const *kv_pools,
                                  int64_t slots_per_rank, float *o_part, float *lse_part, float *o_out,
                                  float *lse_out, void *workspace, size_t workspace_bytes,
                                  int32_t *dev_error, dcp_stream_t stream) {
    if (num_requests > 0 && (!o_out || !lse_out || !aligned(o_out, 16))) return DCP_ERR_INVALID_ARG;
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, -1, o_part,
                             lse_part, o_out, lse_out, workspace, workspace_bytes, dev_error, stream, 1);
}

int dcp_decode_attn_merged(int num_requests, int q_len, int num_heads, const void *q,
                           const int32_t *seq_lens, const int64_t *req_page_ptr, int64_t num_pages,
                           const int32_t *dst_vpages, int page_size, int dtype, float kv_scale,
                           float softmax_scale, int n_dcp, const void *const *kv_pools,
                           int64_t slots_per_rank, float *o_part, float *lse_part, float *o_out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           int32_t *dev_error, dcp_stream_t stream) {
    if (num_requests > 0 && (!o_out || !lse_out || !aligned(o_out, 16))) return DCP_ERR_INVALID_ARG;
    return partial_attn_impl(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages, dst_vpages,
                             page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools, slots_per_rank, -1, o_part,
                             lse_part, o_out, lse_out, workspace, workspace_bytes, dev_error, stream);
}

int dcp_lse_merge(int n_parts, int64_t rows, int v_dim, const float *o_part, const float *lse_part,
                  float *o_out, float *lse_out, dcp_stream_t stream) {
    if (n_parts < 1 || n_parts > 64 || rows < 0) return DCP_ERR_INVALID_ARG;
    if (v_dim != 128 && v_dim != 256 && v_dim != 512) return DCP_ERR_INVALID_ARG;
    if (rows == 0) return DCP_OK;
    if (!o_part || !lse_part || !o_out || !lse_out) return DCP_ERR_INVALID_ARG;
    if (!aligned(o_part, 16) || !aligned(o_out, 16)) return DCP_ERR_INVALID_ARG;
    if (launch_lse_merge(n_parts, rows, v_dim, o_part, lse_part, o_out, lse_out,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DCP_ERR_CUDA;
    return DCP_OK;
}

}  // extern "C"
