// dcp_copy_ring.cuh -- a single issuing thread streams fixed-size chunks HBM -> shared memory ->
// HBM through a ring with TMA bulk copies (cp.async.bulk global->shared completing on an
// mbarrier, then shared->global in bulk groups), keeping ~kLag loads in flight.  The caller
// maps a chunk index to its source and destination; used by the page reshard and by the
// pack / unpack of one path's pages.
#pragma once

#include "dcp_ptx.cuh"

namespace dcp {

#ifndef DCP_RING_STAGES
#define DCP_RING_STAGES 6
#endif
#ifndef DCP_RING_LAG
#define DCP_RING_LAG 3
#endif
#ifndef DCP_RING_CHUNK
#define DCP_RING_CHUNK 36864
#endif
// The largest chunk that divides both page sizes (73,728 and 36,864 bytes): fewer, larger bulk
// copies move more bytes per issue (measured: 36 KB x 6 stages beats 18 KB x 11 by 4-7%, 9 KB
// x 23 is 30% slower).
constexpr uint32_t kRingChunk = DCP_RING_CHUNK;
constexpr int kRingStages = DCP_RING_STAGES;
constexpr int kRingLag = DCP_RING_LAG;  // loads kept ahead of stores
static_assert(kRingStages - kRingLag - 1 >= 0, "ring too small for the lag");
constexpr size_t kRingSmem = (size_t)kRingStages * kRingChunk + kRingStages * sizeof(uint64_t);

// Copies the chunks c in [c_begin, c_end) for which map(c, src, dst) returns true (map sets
// the chunk's source and destination addresses).  Call from one thread; `smem` holds
// kRingSmem bytes.  Returns false when a wait gave up (after letting issued copies land).
template <class Map>
__device__ bool copy_ring(int64_t c_begin, int64_t c_end, Map map, uint8_t *smem, int32_t *dev_error,
                          uint64_t wait_limit_ns) {
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kRingStages * kRingChunk);
    __shared__ int abort_flag;
    abort_flag = 0;
    for (int s = 0; s < kRingStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    fence_proxy_async_smem();

    uint8_t *store_dst[kRingStages] = {};
    int64_t issued = 0, stored = 0;
    bool ok = true;
    auto store_one = [&]() -> bool {
        const int stage = (int)(stored % kRingStages);
        const uint32_t parity = (uint32_t)((stored / kRingStages) & 1);
        if (!mbar_wait(&bars[stage], parity, &abort_flag, dev_error, wait_limit_ns)) return false;
        bulk_s2g(store_dst[stage], smem + (size_t)stage * kRingChunk, kRingChunk);
        bulk_commit();
        ++stored;
        return true;
    };
    for (int64_t c = c_begin; c < c_end && ok; ++c) {
        const uint8_t *src;
        uint8_t *dst;
        if (!map(c, src, dst)) continue;
        const int stage = (int)(issued % kRingStages);
        if (issued >= kRingStages) bulk_wait_read<kRingStages - kRingLag - 1>();  // stage's old store has read smem
        mbar_arrive_expect_tx(&bars[stage], kRingChunk);
        bulk_g2s(smem + (size_t)stage * kRingChunk, src, kRingChunk, &bars[stage]);
        store_dst[stage] = dst;
        ++issued;
        while (issued - stored > kRingLag && ok) ok = store_one();
    }
    while (ok && stored < issued) ok = store_one();
    bulk_wait<0>();
    if (!ok) {
        // A load wait gave up: let the loads already issued (chunks stored..issued-1) land before
        // the CTA exits, each with a bounded wait of its own.
        int never = 0;
        for (int64_t c = stored; c < issued; ++c)
            mbar_wait(&bars[c % kRingStages], (uint32_t)((c / kRingStages) & 1), &never, nullptr, wait_limit_ns);
    }
    return ok;
}

}  // namespace dcp
