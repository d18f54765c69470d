// lookback.cuh -- decoupled look-back for the exclusive prefix of per-tile
// escape counts across CTAs (Merrill & Garland, "Single-pass Parallel Prefix
// Scan with Decoupled Look-back", 2016), on 64-bit state words that carry an
// epoch tag (see common.cuh).  Used by the single-launch encode pipeline and
// by the tile-prefix kernel of the multi-kernel encode.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace splitzip {

// ------------------------------------------------------ decoupled look-back
//
// Run by all 32 lanes of the look-back warp.  Walks back over earlier tiles' state words until it meets an inclusive
// prefix, publishes this tile's inclusive prefix and returns the exclusive
// one.  Each poll issues kLookK rows of 32 contiguous state words (row m,
// lane l: predecessor 32m + l, nearest first) and consumes the rows in order,
// because with every CTA working at once a tile's nearest few hundred
// predecessors are often all in flight and carry only aggregates.  A poll
// that finds a word not yet written backs off before the next one; every
// wait is bounded by a.spin_limit polls.
constexpr int kLookK = 4;

// The tile's own word is published by the compute warps the moment its escape
// count is known (publish_count below), so that later tiles' look-backs find
// it as early as possible; this function only adds the inclusive prefix.
__device__ __forceinline__ void publish_count(uint64_t* states, uint32_t tile, uint32_t epoch,
                                              uint32_t aggregate, bool stall_first) {
    if (tile == 0) {
        if (!stall_first)
            st_relaxed_gpu(states, make_state(kFlagPrefix, aggregate, epoch));
    } else {
        st_relaxed_gpu(states + tile, make_state(kFlagAggregate, aggregate, epoch));
    }
}

__device__ __forceinline__ uint32_t look_back(uint64_t* states, uint32_t* status, uint32_t tile,
                                              uint32_t epoch, uint32_t aggregate,
                                              uint32_t spin_limit) {
    const int lane = threadIdx.x & 31;
    if (tile == 0) return 0;
    uint32_t excl = 0, polls = 0, backoff = 256;
    bool timed_out = false;
    int64_t pred = (int64_t)tile - 1;  // nearest predecessor not yet summed
    while (true) {
        uint64_t w[kLookK];
#pragma unroll
        for (int m = 0; m < kLookK; m++) {
            const int64_t idx = pred - (m * 32 + lane);
            w[m] = idx >= 0 ? ld_relaxed_gpu(states + idx) : make_state(kFlagPrefix, 0u, epoch);
        }
        bool found = false, wait = false;
        uint32_t rows = 0;
#pragma unroll
        for (int m = 0; m < kLookK; m++) {
            if (found || wait) continue;  // warp-uniform
            const uint32_t f = state_flag(w[m], epoch);
            const uint32_t pm = __ballot_sync(0xFFFFFFFFu, f == kFlagPrefix);
            const uint32_t bad = __ballot_sync(0xFFFFFFFFu, f == 0u);
            // Lanes up to and including the nearest inclusive prefix (all 32 if none).
            const uint32_t need = pm ? (((pm & (0u - pm)) << 1) - 1u) : 0xFFFFFFFFu;
            if (bad & need) {
                wait = true;
                continue;
            }
            excl += __reduce_add_sync(0xFFFFFFFFu, ((need >> lane) & 1u) ? (uint32_t)w[m] : 0u);
            rows++;
            found = pm != 0;
        }
        if (found) break;
        pred -= 32 * (int64_t)rows;
        if (wait) {
            if (++polls > spin_limit) {
                timed_out = true;
                break;
            }
            __nanosleep(backoff);
            backoff = backoff < 2048 ? backoff * 2 : 2048;
        }
    }
    if (lane == 0) {
        if (timed_out) atomicOr(status, kStatusTimeout);
        // Published even after a time-out so that later tiles are not held up.
        st_relaxed_gpu(states + tile, make_state(kFlagPrefix, excl + aggregate, epoch));
    }
    return excl;
}

}  // namespace splitzip
