// dcp_internal.h -- declarations shared between the library's translation units (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/dcp.h"

namespace dcp {

constexpr int kPage = DCP_PAGE_TOKENS;
constexpr int kKDim = DCP_K_DIM;
constexpr int kVDim = DCP_V_DIM;
constexpr int kMaxCp = 64;
constexpr int kMaxDcpReshard = 64;
constexpr int kMaxDcpAttn = DCP_MAX_RANKS;

// Default limit for one device-side pipeline wait (nanoseconds of wall time).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Launch `kernel` on `stream` with programmatic stream serialization (the kernel calls
// grid_dep_wait() before touching global memory, so this is safe after any predecessor).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- reshard (dcp_reshard.cu)
struct ReshardArgs {
    const int64_t *req_page_ptr;
    const int32_t *src_pages;
    const int32_t *dst_vpages;
    int num_requests;
    int64_t num_pages;
    int64_t page_bytes;
    int layer_begin;                 // layers [layer_begin, layer_end) are moved
    int layer_end;
    int n_cp;
    int layer_start[kMaxCp + 1];     // source rank r owns [layer_start[r], layer_start[r+1])
    const uint8_t *src_pools[kMaxCp];
    int64_t src_pool_pages;
    int n_dcp;
    uint8_t *dst_pools[kMaxDcpReshard];
    int64_t dst_slots;
    int only_dst;
    int32_t *dev_error;
    uint64_t wait_limit_ns;
};
cudaError_t launch_reshard(const ReshardArgs &a, int num_sms, cudaStream_t stream);

// ---- token-interleaved reshard: a row gather into the token-interleaved layout (dcp_reshard.cu)
struct TokenReshardArgs {
    const int32_t *seq_lens;
    const int64_t *src_page_ptr;   // prefill-side CSR: request b's source pages
    const int32_t *src_pages;
    const int64_t *tok_page_ptr;   // destination CSR: entry jj N + d = rank d's local page jj
    const int32_t *tok_vpages;
    int num_requests;
    int64_t num_tok_entries;
    int64_t row_bytes;
    int num_layers, n_cp;
    int layer_start[kMaxCp + 1];
    const uint8_t *src_pools[kMaxCp];
    int64_t src_pool_pages;
    int n_dcp;
    uint8_t *dst_pools[kMaxDcpReshard];
    int64_t dst_slots;
    int32_t *dev_error;
};
cudaError_t launch_token_reshard(const TokenReshardArgs &a, int num_sms, cudaStream_t stream);

// ---- the naive baseline: full transfer to every DCP rank, then an in-place shard (dcp_reshard.cu)
struct NaiveArgs {
    ReshardArgs base;                     // page table, layer split, source and destination pools
    uint8_t *recv[kMaxDcpReshard];        // per DCP rank: [num_layers][num_pages] receive buffer
    int mode;                             // 0 = full transfer, 1 = in-place shard
};
cudaError_t launch_naive(const NaiveArgs &a, int num_sms, cudaStream_t stream);

// ---- pack / unpack of one path's pages through a staging buffer (dcp_reshard.cu)
struct PackArgs {
    const int32_t *idx;      // [n_idx]: source page indices (pack) or destination slots (unpack)
    int64_t n_idx;
    int n_layers;            // layers of the sending rank
    int layer_offset;        // unpack: destination layer of source layer 0
    int64_t item_begin, n_items;
    int64_t page_bytes;
    uint8_t *pool;           // pack: source pool [n_layers][pool_pages]; unpack: [pool_layers][pool_pages]
    int64_t pool_pages;
    int pool_layers;
    uint8_t *staging;
    int to_staging;          // 1 = pack, 0 = unpack
    int32_t *dev_error;
    uint64_t wait_limit_ns;
};
cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream);

cudaError_t launch_filter(int64_t n, const int32_t *dst_vpages, const int32_t *transfer_idx,
                          int n_dcp, int d, int32_t *out_slot, int32_t *out_src,
                          int64_t *out_count, cudaStream_t stream);

// ---- merge (dcp_merge.cu)
cudaError_t launch_lse_merge(int n_parts, int64_t rows, int v_dim, const float *o_part,
                             const float *lse_part, float *o_out, float *lse_out,
                             cudaStream_t stream);

// ---- attention (dcp_attn.cu)
struct AttnPlanShape {
    int B, T, H, N, G, heads_per_group;
    int64_t num_pages;
    int tiles_per_chunk;
    int64_t max_units;
    int64_t max_partials;
    int64_t n_seg;
    size_t off_counts, off_slots, off_pages, off_units, off_seg, off_ctrl, off_part_o,
        off_part_lse, off_qhl, off_qscale, off_tiles, off_multi;
    int tiles_per_req;
    size_t total_bytes;
};
bool plan_attention(int B, int T, int H, int N, int64_t num_pages, int dtype, int num_sms,
                    AttnPlanShape *out);

struct AttnArgs {
    AttnPlanShape shape;
    const void *q;
    const int32_t *seq_lens;
    const int64_t *req_page_ptr;
    const int32_t *dst_vpages;
    int dtype;
    float kv_scale;
    float softmax_scale;
    const void *kv_pools[kMaxDcpAttn];
    int64_t slots_per_rank;
    int only_rank;
    float *o_part;
    float *lse_part;
    float *o_out;    // non-null: also merge the ranks' partials (exact LSE merge) into o_out / lse_out
    float *lse_out;
    int token_layout;  // 1: the page table is token-interleaved (entry jj N + d = rank d's local page jj)
    int phase;         // 0: plan and run; 1: plan only (page-table work into the workspace); 2: run a plan
    uint8_t *workspace;
    int32_t *dev_error;
    uint64_t wait_limit_ns;
};
int launch_attention(const AttnArgs &a, int num_sms, cudaStream_t stream);
// Reads the plan header of a workspace laid out as `s` (synchronous on `stream`): info[0] units
// in the queue, info[1] pairs with several pieces, info[2] tiles per chunk, info[3] 1 if the
// workspace holds a plan.
int read_plan_info(const AttnPlanShape &s, const void *workspace, int32_t *info, cudaStream_t stream);

}  // namespace dcp
