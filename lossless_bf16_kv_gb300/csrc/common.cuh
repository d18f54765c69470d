// common.cuh -- device helpers shared by the SplitZip kernels (sm_103a).
//
// Nothing here is arithmetic of the codec itself: it is the workspace layout,
// the tile-state word of the cross-tile escape prefix, PTX wrappers and a
// multiply-shift division by the chunk size.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace splitzip {

constexpr int kThreads = 256;  // every kernel runs 256-thread CTAs (8 warps)
constexpr int kWarps = kThreads / 32;

// ----------------------------------------------------------- workspace
//
// [0, 4096)      header (below)
// then           the encode's block and superblock escape counters (fixed size)
// then           one 64-bit tile-state word per encode tile
// The dense pass hands its tiles out from up to kDenseStripes counters: with
// S stripes, stripe s holds tiles s, s + S, s + 2 S, ...
constexpr uint32_t kDenseStripes = 4;

struct WsHeader {
    uint32_t ticket;        // encode: next tile id handed to a starting CTA
    uint32_t done;          // encode: CTAs finished in the running launch
    uint32_t epoch;         // encode: launch counter, tags tile-state words
    uint32_t status;        // encode: status bits raised by the running launch
    uint32_t last_status;   // encode: status bits of the last finished launch
    uint32_t cal_done;      // calibrate: CTAs finished in the running launch
    uint64_t last_escapes;  // encode: E of the last finished launch
    uint64_t cal_covered;   // calibrate: covered count (synchronous API readback)
    uint8_t cal_cb[16];     // calibrate: codebook (synchronous API readback)
    uint32_t dense_next;    // encode: the dense pass's tile counter (one stripe)
    uint32_t dense_done;    // encode: tiles the dense pass has processed
    uint64_t reserved[23];
    unsigned long long hist[256];  // calibrate: global exponent histogram, zero between launches
    // encode: the dense pass's tile counters when it uses several stripes of
    // tiles, each in a 128-byte line of its own (element [s][0]); zero
    // between launches.
    alignas(128) uint32_t dense_stripe[kDenseStripes][32];
};
static_assert(sizeof(WsHeader) <= 4096, "header must fit its slot");
constexpr size_t kWsHeaderBytes = 4096;
// Right after the header, at an offset and of a size that do not depend on
// the element count (so a workspace reused for other sizes keeps them where
// the previous call re-armed them): the encode's escape counters per block of
// 64 tiles and per superblock of 4096 tiles, for up to 2^32 elements.
constexpr size_t kWsSumsBytes = 4 * ((1ull << 32) / 8192 / 64 + (1ull << 32) / 8192 / 4096);
static_assert(kWsSumsBytes % 256 == 0, "keeps the regions after it 256-byte aligned");
// The single-launch pipeline's look-back state words follow.
constexpr size_t kWsStatesOffset = kWsHeaderBytes + kWsSumsBytes;

constexpr uint32_t kStatusOverflow = 1u;
constexpr uint32_t kStatusTimeout = 2u;

// Tile-state word of the decoupled look-back:
//   bits  0..31  value (aggregate or inclusive prefix of escape counts)
//   bits 32..33  flag: 0 not ready, 1 aggregate, 2 inclusive prefix
//   bits 34..63  epoch tag (launch counter mod 2^30); a word with another tag
//                is left over from an earlier launch and reads as not ready.
constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagPrefix = 2u;

__host__ __device__ __forceinline__ uint64_t make_state(uint32_t flag, uint32_t value,
                                                        uint32_t epoch) {
    return (uint64_t)value | ((uint64_t)flag << 32) | ((uint64_t)(epoch & 0x3FFFFFFFu) << 34);
}
__device__ __forceinline__ uint32_t state_flag(uint64_t w, uint32_t epoch) {
    if ((uint32_t)(w >> 34) != (epoch & 0x3FFFFFFFu)) return 0;
    return (uint32_t)(w >> 32) & 3u;
}

// ------------------------------------------------------------- PTX bits

// prmt.b32 in its default mode: selector nibble bit 3 replicates the sign bit
// of the selected byte (used by the decode's 16-entry codebook lookup).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Streaming loads (read once: evict-first).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.cs.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
    uint32_t v;
    asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
// Streaming stores (written once, never read back by the writing thread).
// No "memory" clobber: the compiler may move this thread's other loads across
// them (the streams are not re-read), while the asm volatile statements that
// publish to other threads (mbarrier arrives, state-word stores) keep their
// order relative to these stores.
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y));
}
__device__ __forceinline__ void st_stream4(void* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v));
}

// ------------------------------------------------------------- codebook
//
// The 16 codebook bytes as four little-endian words: from the launch
// parameters, or from device memory (4-byte aligned) when dcb is not null --
// a codebook that an earlier kernel on the stream (device-side calibration)
// wrote, read without a round trip through the host.
__device__ __forceinline__ void codebook_words(const uint8_t* dcb, const uint32_t (&param)[4],
                                               uint32_t (&w)[4]) {
    if (dcb) {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(dcb);
#pragma unroll
        for (int q = 0; q < 4; q++) w[q] = __ldg(p + q);
    } else {
#pragma unroll
        for (int q = 0; q < 4; q++) w[q] = param[q];
    }
}

// Whether the codebook words hold 16 distinct exponents, each at most
// max_exp (255 for BF16, 31 for E5M2).
__device__ __forceinline__ bool codebook_valid(const uint32_t (&w)[4], uint32_t max_exp) {
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 16; k++) {
        const uint32_t e = (w[k >> 2] >> (8 * (k & 3))) & 0xFFu;
        ok = ok && e <= max_exp;
#pragma unroll
        for (int j = 0; j < k; j++) ok = ok && ((w[j >> 2] >> (8 * (j & 3))) & 0xFFu) != e;
    }
    return ok;
}

// ------------------------------------------------------------- division
//
// q = floor(x / d) as (x * m) >> 33 with m = ceil(2^33 / d), exact for
// x < 2^17 and 1 <= d <= 2^16 (Granlund & Montgomery, "Division by Invariant
// Integers using Multiplication", 1994): with m*d = 2^33 + e, 0 <= e < d, the
// error term x*e / (d * 2^33) stays below 1/d because x*e < 2^17 * 2^16.
//
// For any 32-bit x, q = floor(x / d) is the high 64 bits of x * M with
// M = ceil(2^64 / d) (Lemire, Kaser and Kurz, "Faster Remainder by Direct
// Computation", 2019: exact for every 32-bit numerator and divisor d >= 2).
struct ChunkDiv {
    uint32_t d;    // chunk size
    uint32_t m;    // ceil(2^33 / d)
    uint64_t m64;  // ceil(2^64 / d)
};
__host__ __device__ __forceinline__ ChunkDiv make_chunk_div(uint32_t d) {
    ChunkDiv c;
    c.d = d;
    c.m = (uint32_t)(((1ull << 33) + d - 1) / d);
    c.m64 = d > 1 ? ~0ull / d + 1 : 0;
    return c;
}
__device__ __forceinline__ uint32_t chunk_quot(ChunkDiv c, uint32_t x) {
    return (uint32_t)(((uint64_t)x * c.m) >> 33);
}
// floor(x / d) for any 32-bit x (d >= 2).
__device__ __forceinline__ uint32_t chunk_quot32(ChunkDiv c, uint32_t x) {
    return (uint32_t)__umul64hi(c.m64, (uint64_t)x);
}

}  // namespace splitzip

namespace splitzip {

// ------------------------------------------------ mbarrier and bulk copies

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    [[maybe_unused]] uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];"
                 : "=l"(state)
                 : "r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx_bytes) {
    [[maybe_unused]] uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state)
                 : "r"(smem_addr(bar)), "r"(tx_bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase of `bar` with the given parity; gives up after `limit`
// polls (each try_wait may itself suspend for a short, hardware-bounded
// time) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// One-dimensional bulk copy global -> shared, completing on `bar` (the
// destination and source 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// Per-thread asynchronous copies global -> shared (cp.async).  A thread that
// waits for its own groups sees its own copies; no other thread's.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
// An L2 policy that marks lines evict-first (for data read exactly once).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// An L2 policy that marks lines evict-last (for small data that a following
// kernel reads back while large streams pass through L2).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Stores under an L2 cache policy.
__device__ __forceinline__ void st_policy2(void* p, uint16_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"(v), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_policy8(void* p, uint2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "l"(pol)
                 : "memory");
}
// Programmatic dependent launch: a grid lets the launch that depends on it
// start early, and that launch waits until this grid has completed and its
// memory operations are visible before it goes past wait_prerequisite_grid.
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Loads of data read for the last time (evict-first in L2).
__device__ __forceinline__ uint16_t ld_last2(const void* p) {
    uint16_t v;
    asm volatile("ld.global.lu.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_last8(const void* p) {
    uint2 v;
    asm volatile("ld.global.lu.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_last16(const void* p) {
    uint4 v;
    asm volatile("ld.global.lu.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// cp_async16 with an L2 cache policy for the global read.
__device__ __forceinline__ void cp_async16_hint(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)),
                 "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Named barrier over the first `threads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------- launch waves
//
// How many CTAs of kernel K fit on the current device at once: its SM count
// times the CTAs of `threads` threads with `smem` bytes of dynamic shared
// memory that one SM holds (K's dynamic shared-memory limit raised to smem
// first).  Computed once per kernel and device, then taken from a cache, so
// a call does not pay the attribute and occupancy queries each time.
struct Wave {
    int sms = 0;
    int per_sm = 0;
    uint64_t ctas() const { return (uint64_t)(sms > 0 ? sms : 1) * (uint64_t)(per_sm > 0 ? per_sm : 1); }
};

template <auto K>
cudaError_t launch_wave(int threads, size_t smem, Wave& out) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static Wave cache[kMaxDevices];
    static bool known[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    std::unique_lock<std::mutex> lock(mu, std::defer_lock);
    if (cached) {
        lock.lock();
        if (known[dev]) {
            out = cache[dev];
            return cudaSuccess;
        }
    }
    Wave w;
    e = cudaDeviceGetAttribute(&w.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&w.per_sm, K, threads, smem);
    if (e != cudaSuccess) return e;
    if (cached) {
        cache[dev] = w;
        known[dev] = true;
    }
    out = w;
    return cudaSuccess;
}

}  // namespace splitzip
