// dcp_attn_static.cu -- dcp_partial_decode_attn_static: the partial-attention entry point for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a host that has handed the whole device memory
// to its own pool allocator and exposes only tensor pointers to plug-ins, or a decode loop in
// which an allocation (which may synchronise the device) is not allowed.  They cannot supply
// the caller-owned workspace dcp_partial_decode_attn needs.  This variant uses a scratch
// buffer that lives in the library itself: a file-scope device array of fixed size, created
// when the module is loaded and held by every GPU that loads the library until the process
// exits.  It allocates nothing per call.
//
// The caller still passes every input and output.  The scratch holds the per-(rank, request)
// page lists, the unit list and the chunk partials of one call; the plan kernels rewrite all
// of it (including the work counter, which they reset to zero) before the attention kernel
// reads it, so nothing has to be cleared between calls.  Every call shares the one array:
// calls that overlap on the GPU (different streams, or different host threads, without
// ordering between them) race on it and must not be issued.
#include <cuda_runtime.h>

#include <mutex>

#include "dcp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = DCP_STATIC_ATTN_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's host-side name is
// only a stand-in, so the address is looked up once per device, with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DCP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return DCP_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return DCP_OK;
}

}  // namespace

extern "C" int dcp_partial_decode_attn_static(int num_requests, int q_len, int num_heads, const void *q,
                                              const int32_t *seq_lens, const int64_t *req_page_ptr,
                                              int64_t num_pages, const int32_t *dst_vpages, int page_size,
                                              int dtype, float kv_scale, float softmax_scale, int n_dcp,
                                              const void *const *kv_pools, int64_t slots_per_rank,
                                              int only_rank, float *o_part, float *lse_part,
                                              int32_t *dev_error, dcp_stream_t stream) {
    // The size check needs the same plan the call will use; it is done before the scratch
    // address is looked up so that oversized requests fail without touching the device.
    if (num_requests < 0 || q_len < 1 || num_heads < 1 || num_pages < 0 || n_dcp < 1 ||
        n_dcp > DCP_MAX_RANKS)
        return DCP_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DCP_ERR_CUDA;
    dcp::AttnPlanShape shape;
    if (!dcp::plan_attention(num_requests, q_len, num_heads, n_dcp, num_pages, dtype, sms, &shape))
        return DCP_ERR_INVALID_ARG;
    if (shape.total_bytes > kStaticScratchBytes) return DCP_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    return dcp_partial_decode_attn(num_requests, q_len, num_heads, q, seq_lens, req_page_ptr, num_pages,
                                   dst_vpages, page_size, dtype, kv_scale, softmax_scale, n_dcp, kv_pools,
                                   slots_per_rank, only_rank, o_part, lse_part, scratch, kStaticScratchBytes,
                                   dev_error, stream);
}
