// encode.cu -- SplitZip encode kernels for sm_103a (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README section Abstract; arXiv abstract on the paper index page):
// split each value into its exponent and its exact sign+mantissa bits, map the
// exponent through the 16-entry codebook to a 4-bit code, and send exponents
// outside the codebook to a chunk-local escape stream of (position, value).
//
// One launch, one pass over the input, persistent CTAs (two per SM), each a
// warp-specialised pipeline over 8192-element tiles claimed by atomic ticket:
//   producer warp   claims tiles and streams each tile's input into a
//                   three-stage shared-memory ring with bulk copies
//                   (cp.async.bulk + mbarrier);
//   8 compute warps split the fields (byte permutes), look the exponents up in
//                   a 256-entry shared table, pack the nibbles and store the
//                   dense code and sign+mantissa streams (fixed offsets); they
//                   count escapes, rank them with a block scan and drop them,
//                   with the rank of every chunk boundary, into one of two
//                   shared-memory escape slots, then go straight on to the
//                   next tile;
//   look-back warp  takes a filled slot, publishes the tile's escape count and
//                   runs a decoupled look-back (Merrill & Garland, "Single-pass
//                   Parallel Prefix Scan with Decoupled Look-back", 2016) over
//                   earlier tiles' state words for the tile's global escape
//                   offset, then writes the slot's escapes and chunk offsets.
// Only the look-back warp ever waits on other CTAs, and it runs one tile
// behind the compute warps.  Escapes come out in element order, which is
// chunk order then position order within a chunk, for any chunk size.  Every
// wait is bounded: a wait that runs out records SPLITZIP_ERR_TIMEOUT, lets the
// pipeline drain with every access in bounds, and returns.
#include <cstdint>

#include "common.cuh"
#include "fields.cuh"
#include "lookback.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

// ------------------------------------------------------------ pipeline

constexpr uint32_t kInvalidTile = 0xFFFFFFFFu;
constexpr int kTile = 8192;                      // elements per tile, both formats
constexpr int kStages = 3;                       // input ring depth
constexpr int kSlots = 8;                        // escape slots (compute -> look-back)
constexpr int kLookbackWarps = 4;                // look-back warp w serves slots w, w + 4
constexpr int kListCap = 1024;                   // escapes a slot holds; more: direct path
constexpr int kComputeWarps = kThreads / 32;     // 8
constexpr int kComputeThreads = kThreads;
constexpr int kProducerWarp = kComputeWarps;     // warp 8
constexpr int kEncodeThreads = kComputeThreads + 32 + 32 * kLookbackWarps;  // 416
constexpr int kMaxBoundaries = kTile / 8 + 1;    // chunk starts one tile can hold
constexpr uint64_t kWaitNs = 2000000000ull;      // an mbarrier wait gives up after 2 s

template <int kElemBytes>
struct EncodeSmem {
    alignas(128) uint8_t stage[kStages][kTile * kElemBytes];  // input ring (bulk-copy target)
    uint16_t list_pos[kSlots][kListCap];  // escapes by rank in tile: position in chunk
    uint8_t list_val[kSlots][kListCap];   //                          raw exponent
    uint16_t bnd[kSlots][kMaxBoundaries];  // rank in tile at each chunk start, by chunk
    uint8_t table[256];                   // exponent -> code (kMissEntry: escape)
    uint32_t warp_tot[2][kWarps][2];
    uint32_t stage_tile[kStages], stage_q0[kStages], stage_r0[kStages];
    uint32_t slot_tile[kSlots], slot_agg[kSlots], slot_q0[kSlots], slot_r0[kSlots];
    uint32_t slot_excl[kSlots];           // direct path: the tile's global escape offset
    uint32_t cur_tile, cur_excl;
    uint32_t err;
    alignas(8) uint64_t full[kStages];    // producer -> compute: stage filled (tx bytes)
    uint64_t empty[kStages];              // compute -> producer: stage consumed
    uint64_t slot_full[kSlots];           // compute -> look-back: slot filled (8 warps)
    uint64_t slot_empty[kSlots];          // look-back -> compute: slot written out
    uint64_t slot_prefix[kSlots];         // look-back -> compute: offset of a direct tile
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase (time-based, so the bound does not depend
// on how long a single try_wait suspends).  Waits off the critical path pass
// sleep_ns > 0 so that their polling does not take issue slots from the
// compute warps.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 16; i++) {
            if (sleep_ns) __nanosleep(sleep_ns);
            if (mbar_try_wait(bar, parity)) return true;
        }
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

template <int kElemBytes>
__device__ __forceinline__ void record_timeout(const EncodeArgs& a, EncodeSmem<kElemBytes>& sm) {
    atomicOr(&reinterpret_cast<WsHeader*>(a.ws)->status, kStatusTimeout);
    *reinterpret_cast<volatile uint32_t*>(&sm.err) = 1u;
}

// Block scan over the 256 compute threads (named barrier 1).  Each thread
// holds counts c[k] (k < G <= 4) for its groups; group (k, t) precedes
// (k', t') in element order iff k < k' or (k == k' and t < t').  Returns the
// tile total and each group's exclusive rank in the tile.
template <int G>
__device__ __forceinline__ uint32_t block_ranks(const uint32_t (&c)[G], uint32_t (&rank)[G],
                                                uint32_t (*wt)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t p01 = c[0] | (G > 1 ? c[1] << 16 : 0u);
    uint32_t p23 = (G > 2 ? c[2] : 0u) | (G > 3 ? c[3] << 16 : 0u);
    const uint32_t own01 = p01, own23 = p23;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, p01, d);
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, p23, d);
        if (lane >= d) {
            p01 += u;
            p23 += v;
        }
    }
    if (lane == 31) {
        wt[warp][0] = p01;
        wt[warp][1] = p23;
    }
    named_sync(1, kComputeThreads);
    uint32_t pre01 = 0, pre23 = 0, tot01 = 0, tot23 = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
        const uint32_t x = wt[w][0], y = wt[w][1];
        if (w < warp) {
            pre01 += x;
            pre23 += y;
        }
        tot01 += x;
        tot23 += y;
    }
    const uint32_t ex01 = p01 - own01 + pre01, ex23 = p23 - own23 + pre23;
    const uint32_t tot[4] = {tot01 & 0xFFFFu, tot01 >> 16, tot23 & 0xFFFFu, tot23 >> 16};
    const uint32_t exk[4] = {ex01 & 0xFFFFu, ex01 >> 16, ex23 & 0xFFFFu, ex23 >> 16};
    uint32_t base = 0;
#pragma unroll
    for (int k = 0; k < G; k++) {
        rank[k] = base + exk[k];
        base += tot[k];
    }
    return base;
}

// Where a tile's escapes go once ranked: into the slot's list (the look-back
// warp copies them out), or straight to the escape stream at excl + rank.
struct EscapeSink {
    uint16_t* lpos;
    uint8_t* lval;
    uint16_t* gpos;
    uint8_t* gval;
    uint64_t cap;    // direct: escape capacity
    uint32_t excl;   // direct: the tile's global offset
    bool direct;
    __device__ __forceinline__ void put(uint32_t rank, uint32_t pos, uint32_t e) const {
        if (direct) {
            const uint32_t g = excl + rank;
            if ((uint64_t)g < cap) {
                gpos[g] = (uint16_t)pos;
                gval[g] = (uint8_t)e;
            }
        } else if (rank < (uint32_t)kListCap) {
            lpos[rank] = (uint16_t)pos;
            lval[rank] = (uint8_t)e;
        }
    }
};

// ------------------------------------------------------ per-format tiles
//
// BF16: thread t's groups of 8 sit at tile offsets k*2048 + 8t (k < 4), so a
// warp reads 512 contiguous bytes of the stage per group (no bank conflicts)
// and writes 128 contiguous code bytes and 256 sign+mantissa bytes.
struct Bf16Tile {
    static constexpr int kElemBytes = 2;
    static constexpr int kGroups = 4;
    struct Keep {
        uint32_t ex[kGroups][2], ent[kGroups][2], cnt[kGroups];
    };
    static __device__ __forceinline__ uint32_t loff(int k) {
        return k * (kThreads * 8) + threadIdx.x * 8;
    }

    static __device__ __forceinline__ void process(const EncodeArgs& a, const uint8_t* stage,
                                                   const uint8_t* table, uint32_t t0, Keep& kp) {
        const bool full = (uint64_t)t0 + kTile <= a.n;
        if (full) {
            // Whole tile: every group's stage reads and table lookups first,
            // then the stores, so that the lookups of all groups overlap.
            uint32_t sm[kGroups][2];
#pragma unroll
            for (int k = 0; k < kGroups; k++) {
                const uint4 v = *reinterpret_cast<const uint4*>(stage + 2 * loff(k));
                split_bf16(v.x, v.y, sm[k][0], kp.ex[k][0]);
                split_bf16(v.z, v.w, sm[k][1], kp.ex[k][1]);
            }
#pragma unroll
            for (int k = 0; k < kGroups; k++) {
                kp.ent[k][0] = lookup4(table, kp.ex[k][0]);
                kp.ent[k][1] = lookup4(table, kp.ex[k][1]);
            }
#pragma unroll
            for (int k = 0; k < kGroups; k++) {
                const uint32_t i = t0 + loff(k);
                kp.cnt[k] = miss_count(kp.ent[k][0], kp.ent[k][1]);
                st_stream4(a.codes + i / 2, pack_nibbles(kp.ent[k][0], kp.ent[k][1]));
                st_stream8(a.signman + i, make_uint2(sm[k][0], sm[k][1]));
            }
            return;
        }
        const uint32_t pad = (a.cbw[0] & 0xFFu) << 7;  // exponent cb[0], sign 0, mantissa 0: code 0
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t l = loff(k), i = t0 + l;
            kp.cnt[k] = 0;
            kp.ent[k][0] = kp.ent[k][1] = 0;
            if (i >= a.n) continue;
            uint4 v;
            const bool whole = a.n - i >= 8;  // i < n here
            if (whole) {
                v = *reinterpret_cast<const uint4*>(stage + 2 * l);
            } else {
                const uint16_t* h = reinterpret_cast<const uint16_t*>(stage) + l;
                const uint32_t rem = a.n - i;
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; m++)
                    w[m] = (2 * m < (int)rem ? h[2 * m] : pad) |
                           ((2 * m + 1 < (int)rem ? (uint32_t)h[2 * m + 1] : pad) << 16);
                v = make_uint4(w[0], w[1], w[2], w[3]);
            }
            uint32_t sm0, sm1;
            split_bf16(v.x, v.y, sm0, kp.ex[k][0]);
            split_bf16(v.z, v.w, sm1, kp.ex[k][1]);
            kp.ent[k][0] = lookup4(table, kp.ex[k][0]);
            kp.ent[k][1] = lookup4(table, kp.ex[k][1]);
            const uint32_t codes = pack_nibbles(kp.ent[k][0], kp.ent[k][1]);
            kp.cnt[k] = miss_count(kp.ent[k][0], kp.ent[k][1]);
            if (whole) {
                st_stream4(a.codes + i / 2, codes);
                st_stream8(a.signman + i, make_uint2(sm0, sm1));
            } else {
                const uint32_t rem = a.n - i;
                for (uint32_t j = 0; j < (rem + 1) / 2; j++) a.codes[i / 2 + j] = (uint8_t)(codes >> (8 * j));
                for (uint32_t j = 0; j < rem; j++)
                    a.signman[i + j] = (uint8_t)((j < 4 ? sm0 : sm1) >> (8 * (j & 3)));
            }
        }
    }

    // Rank in tile at every chunk start this thread's groups hold.
    static __device__ __forceinline__ void emit_bnd(const EncodeArgs& a, const Keep& kp,
                                                    const uint32_t (&rank)[kGroups], uint32_t t0,
                                                    uint32_t r0, uint16_t* bnd) {
        const bool full = (uint64_t)t0 + kTile <= a.n;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t l = loff(k);
            if (!full && t0 + l >= a.n) continue;
            const uint32_t x = r0 + l;
            const uint32_t q = chunk_quot(a.cdiv, x);
            if (x == q * a.cdiv.d) bnd[q] = (uint16_t)rank[k];
        }
    }

    // Escapes by rank; a group of 8 lies inside one chunk (chunk % 8 == 0).
    static __device__ __forceinline__ void emit_escapes(const EncodeArgs& a, const Keep& kp,
                                                        const uint32_t (&rank)[kGroups],
                                                        uint32_t t0, uint32_t r0,
                                                        const EscapeSink& sink) {
        const bool full = (uint64_t)t0 + kTile <= a.n;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            if (!kp.cnt[k]) continue;
            const uint32_t l = loff(k);
            if (!full && t0 + l >= a.n) continue;
            const uint32_t x = r0 + l;
            const uint32_t r = x - chunk_quot(a.cdiv, x) * a.cdiv.d;
            uint32_t g = rank[k];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((kp.ent[k][j >> 2] >> (8 * (j & 3))) & kMissEntry) {
                    sink.put(g, r + j, (kp.ex[k][j >> 2] >> (8 * (j & 3))) & 0xFFu);
                    g++;
                }
            }
        }
    }
};

// E5M2: thread t's group is the 32 elements at tile offset 32t (two 16-byte
// stage reads): 16 code bytes and 12 bytes of packed 3-bit fields.
struct E5m2Tile {
    static constexpr int kElemBytes = 1;
    static constexpr int kGroups = 1;
    struct Keep {
        uint32_t ex[8], ent[8], cnt[kGroups];
    };
    static __device__ __forceinline__ uint32_t loff() { return threadIdx.x * 32; }

    static __device__ __forceinline__ void process(const EncodeArgs& a, const uint8_t* stage,
                                                   const uint8_t* table, uint32_t t0, Keep& kp) {
        const bool full = (uint64_t)t0 + kTile <= a.n;
        const uint32_t l = loff(), i = t0 + l;
        kp.cnt[0] = 0;
#pragma unroll
        for (int m = 0; m < 8; m++) kp.ent[m] = 0;
        if (!full && i >= a.n) return;
        const bool whole = full || a.n - i >= 32;  // i < n when not full
        uint32_t w[8];
        if (whole) {
            const uint4 v0 = *reinterpret_cast<const uint4*>(stage + l);
            const uint4 v1 = *reinterpret_cast<const uint4*>(stage + l + 16);
            w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
            w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
        } else {
            const uint32_t pad = (a.cbw[0] & 0x1Fu) << 2;  // exponent cb[0], sign 0, mantissa 0
            const uint32_t rem = a.n - i;
#pragma unroll
            for (int m = 0; m < 8; m++) {
                uint32_t acc = 0;
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    const uint32_t j = m * 4 + b;
                    acc |= (j < rem ? (uint32_t)stage[l + j] : pad) << (8 * b);
                }
                w[m] = acc;
            }
        }
        uint32_t f12[8];
#pragma unroll
        for (int m = 0; m < 8; m++) {
            split_e5m2(w[m], kp.ex[m], f12[m]);
            kp.ent[m] = lookup4(table, kp.ex[m]);
        }
        uint4 codes;
        codes.x = pack_nibbles(kp.ent[0], kp.ent[1]);
        codes.y = pack_nibbles(kp.ent[2], kp.ent[3]);
        codes.z = pack_nibbles(kp.ent[4], kp.ent[5]);
        codes.w = pack_nibbles(kp.ent[6], kp.ent[7]);
#pragma unroll
        for (int m = 0; m < 8; m += 2) kp.cnt[0] += miss_count(kp.ent[m], kp.ent[m + 1]);
        // 8 x 12 bits -> 96 bits, little-endian.
        const uint32_t s0 = f12[0] | (f12[1] << 12) | (f12[2] << 24);
        const uint32_t s1 = (f12[2] >> 8) | (f12[3] << 4) | (f12[4] << 16) | (f12[5] << 28);
        const uint32_t s2 = (f12[5] >> 4) | (f12[6] << 8) | (f12[7] << 20);
        uint8_t* smp = a.signman + (uint64_t)(i / 32) * 12;
        if (whole) {
            st_stream16(a.codes + i / 2, codes);
            st_stream4(smp, s0);
            st_stream4(smp + 4, s1);
            st_stream4(smp + 8, s2);
        } else {
            const uint32_t rem = a.n - i;
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
            for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                a.codes[i / 2 + j] = (uint8_t)(cw[j >> 2] >> (8 * (j & 3)));
            const uint32_t sw[3] = {s0, s1, s2};
            for (uint32_t j = 0; j < (3 * rem + 7) / 8; j++)
                smp[j] = (uint8_t)(sw[j >> 2] >> (8 * (j & 3)));
        }
    }

    // Four runs of 8 elements per group; each run lies inside one chunk.
    static __device__ __forceinline__ void emit_bnd(const EncodeArgs& a, const Keep& kp,
                                                    const uint32_t (&rank)[kGroups], uint32_t t0,
                                                    uint32_t r0, uint16_t* bnd) {
        const bool full = (uint64_t)t0 + kTile <= a.n;
        const uint32_t l = loff();
        uint32_t g = rank[0];
#pragma unroll
        for (int s = 0; s < 4; s++) {
            if (!full && t0 + l + 8 * s >= a.n) break;
            const uint32_t x = r0 + l + 8 * s;
            const uint32_t q = chunk_quot(a.cdiv, x);
            if (x == q * a.cdiv.d) bnd[q] = (uint16_t)g;
            g += miss_count(kp.ent[2 * s], kp.ent[2 * s + 1]);
        }
    }

    static __device__ __forceinline__ void emit_escapes(const EncodeArgs& a, const Keep& kp,
                                                        const uint32_t (&rank)[kGroups],
                                                        uint32_t t0, uint32_t r0,
                                                        const EscapeSink& sink) {
        if (!kp.cnt[0]) return;
        const bool full = (uint64_t)t0 + kTile <= a.n;
        const uint32_t l = loff();
        uint32_t g = rank[0];
#pragma unroll
        for (int s = 0; s < 4; s++) {
            if (!full && t0 + l + 8 * s >= a.n) break;
            const uint32_t e_lo = kp.ent[2 * s], e_hi = kp.ent[2 * s + 1];
            if (!miss_count(e_lo, e_hi)) continue;
            const uint32_t x = r0 + l + 8 * s;
            const uint32_t r = x - chunk_quot(a.cdiv, x) * a.cdiv.d;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (((j < 4 ? e_lo : e_hi) >> (8 * (j & 3))) & kMissEntry) {
                    sink.put(g, r + j, (kp.ex[2 * s + (j >> 2)] >> (8 * (j & 3))) & 0xFFu);
                    g++;
                }
            }
        }
    }
};

// ------------------------------------------------------------------ roles

// Lane 0 of the producer warp: claim tiles and fill the input ring.
template <class F>
__device__ void producer_role(const EncodeArgs& a, EncodeSmem<F::kElemBytes>& sm) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    uint32_t pending = 0, parity = 0;  // stages whose last arrival is a bulk copy, and its parity
    for (uint32_t j = 0;; j++) {
        const uint32_t s = j % kStages, use = j / kStages;
        bool ok = wait_phase(&sm.empty[s], (use & 1) ^ 1, 128);
        if (!ok) record_timeout(a, sm);
        const bool stop = !ok || *reinterpret_cast<volatile uint32_t*>(&sm.err);
        const uint32_t tile = stop ? kInvalidTile : atomicAdd(&hdr->ticket, 1u);
        if (tile >= a.num_tiles) {
            sm.stage_tile[s] = kInvalidTile;
            mbar_arrive(&sm.full[s]);
            pending &= ~(1u << s);
            break;
        }
        const uint32_t t0 = tile * (uint32_t)kTile;  // tile < num_tiles: t0 < n < 2^32
        const uint32_t q0 = t0 / a.cdiv.d;
        sm.stage_tile[s] = tile;
        sm.stage_q0[s] = q0;
        sm.stage_r0[s] = t0 - q0 * a.cdiv.d;
        const uint32_t len = a.n - t0 < (uint32_t)kTile ? a.n - t0 : (uint32_t)kTile;
        const uint32_t bytes = len * F::kElemBytes, b16 = bytes & ~15u;
        const uint8_t* src = a.x + (uint64_t)t0 * F::kElemBytes;
        for (uint32_t b = b16; b < bytes; b++) sm.stage[s][b] = src[b];  // < 16 tail bytes
        if (b16) {
            mbar_arrive_expect_tx(&sm.full[s], b16);
            bulk_load(sm.stage[s], src, b16, &sm.full[s]);
            pending |= 1u << s;
            parity = (parity & ~(1u << s)) | ((use & 1) << s);
        } else {
            mbar_arrive(&sm.full[s]);
            pending &= ~(1u << s);
        }
    }
    // No bulk copy may still be writing this CTA's shared memory when it exits
    // (on the normal path the compute warps have consumed every stage already).
    for (uint32_t s = 0; s < kStages; s++)
        if ((pending >> s) & 1u) wait_phase(&sm.full[s], (parity >> s) & 1u);
}

// The 8 compute warps.
template <class F>
__device__ void compute_role(const EncodeArgs& a, EncodeSmem<F::kElemBytes>& sm, uint32_t epoch) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix_par = 0;  // bit k: parity of the next slot_prefix[k] phase
    uint32_t j = 0;
    for (;; j++) {
        const uint32_t s = j % kStages, par = (j / kStages) & 1;
        const uint32_t k = j % kSlots, spar = ((j / kSlots) & 1) ^ 1;
        if (tid == 0) {
            uint32_t t = kInvalidTile;
            if (wait_phase(&sm.full[s], par)) t = sm.stage_tile[s];
            else record_timeout(a, sm);
            // The slot is needed either way: for this tile or for an end marker.
            if (!wait_phase(&sm.slot_empty[k], spar)) record_timeout(a, sm);
            sm.cur_tile = t;
        }
        named_sync(1, kComputeThreads);
        const uint32_t tile = sm.cur_tile;
        if (tile == kInvalidTile) break;
        mbar_try_wait(&sm.full[s], par);        // acquire the stage data in this thread
        mbar_try_wait(&sm.slot_empty[k], spar);  // and the slot's release by its look-back warp
        const uint32_t t0 = tile * (uint32_t)kTile;
        const uint32_t r0 = sm.stage_r0[s], q0 = sm.stage_q0[s];

        typename F::Keep kp;
        F::process(a, sm.stage[s], sm.table, t0, kp);
        uint32_t rank[F::kGroups];
        const uint32_t aggregate = block_ranks<F::kGroups>(kp.cnt, rank, sm.warp_tot[j & 1]);
        const bool direct = aggregate > (uint32_t)kListCap;  // uniform
        // Past the scan's barrier every compute thread is done with stage s.
        if (tid == 0) {
            publish_count(reinterpret_cast<uint64_t*>(a.ws + kWsStatesOffset), tile, epoch, aggregate,
                          (a.test_flags & kTestStallFirstTile) != 0);
            mbar_arrive(&sm.empty[s]);
            sm.slot_tile[k] = tile;
            sm.slot_agg[k] = aggregate;
            sm.slot_q0[k] = q0;
            sm.slot_r0[k] = r0;
        }
        F::emit_bnd(a, kp, rank, t0, r0, sm.bnd[k]);
        EscapeSink sink{sm.list_pos[k], sm.list_val[k], a.esc_pos, a.esc_val, a.esc_capacity, 0u,
                        direct};
        if (!direct) F::emit_escapes(a, kp, rank, t0, r0, sink);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.slot_full[k]);
        if (direct) {
            // Too many escapes for a slot: wait for this tile's offset and write
            // them from registers.
            if (tid == 0) {
                if (!wait_phase(&sm.slot_prefix[k], (prefix_par >> k) & 1u)) record_timeout(a, sm);
                sm.cur_excl = sm.slot_excl[k];
            }
            prefix_par ^= 1u << k;
            named_sync(1, kComputeThreads);
            sink.excl = sm.cur_excl;
            F::emit_escapes(a, kp, rank, t0, r0, sink);
        }
    }
    // End markers, one for each look-back warp (slot j was already waited for).
    for (uint32_t m = 0; m < (uint32_t)kLookbackWarps; m++) {
        const uint32_t jj = j + m, k = jj % kSlots, spar = ((jj / kSlots) & 1) ^ 1;
        if (tid == 0) {
            if (m > 0 && !wait_phase(&sm.slot_empty[k], spar)) record_timeout(a, sm);
            sm.slot_tile[k] = kInvalidTile;
        }
        if (lane == 0) mbar_arrive(&sm.slot_full[k]);
    }
}

// Look-back warp lw: the tiles j = lw, lw + 4, ... of this CTA (slots lw and
// lw + 4): global escape offset, escapes (unless direct) and chunk offsets.
template <class F>
__device__ void lookback_role(const EncodeArgs& a, EncodeSmem<F::kElemBytes>& sm,
                              uint32_t epoch, uint32_t lw) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    const int lane = threadIdx.x & 31;
    for (uint32_t j = lw;; j += kLookbackWarps) {
        const uint32_t k = j % kSlots, par = (j / kSlots) & 1;
        bool ok = lane == 0 ? wait_phase(&sm.slot_full[k], par, 256) : false;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) {
            if (lane == 0) record_timeout(a, sm);
            break;
        }
        mbar_try_wait(&sm.slot_full[k], par);
        const uint32_t tile = sm.slot_tile[k];
        if (tile == kInvalidTile) break;
        const uint32_t agg = min(sm.slot_agg[k], (uint32_t)kTile);
        const uint32_t q0 = sm.slot_q0[k], r0 = sm.slot_r0[k];
        const bool direct = agg > (uint32_t)kListCap;
        const uint32_t excl = look_back(reinterpret_cast<uint64_t*>(a.ws + kWsStatesOffset),
                                        &reinterpret_cast<WsHeader*>(a.ws)->status, tile, epoch, agg,
                                        a.spin_limit);
        if (direct) {
            if (lane == 0) {
                sm.slot_excl[k] = excl;
                mbar_arrive(&sm.slot_prefix[k]);
            }
        } else {
            const uint16_t* lpos = sm.list_pos[k];
            const uint8_t* lval = sm.list_val[k];
            for (uint32_t r = lane; r < agg; r += 32) {
                const uint32_t g = excl + r;
                if ((uint64_t)g < a.esc_capacity) {
                    a.esc_pos[g] = lpos[r];
                    a.esc_val[g] = lval[r];
                }
            }
        }
        const uint32_t t0 = tile * (uint32_t)kTile;
        const uint32_t len = a.n - t0 < (uint32_t)kTile ? a.n - t0 : (uint32_t)kTile;
        const uint32_t qa = r0 ? 1u : 0u, qb = chunk_quot(a.cdiv, r0 + len - 1);
        for (uint32_t q = qa + lane; q <= qb && q < (uint32_t)kMaxBoundaries; q += 32)
            a.chunk_off[q0 + q] = excl + sm.bnd[k][q];
        if (tile == a.num_tiles - 1 && lane == 0) {
            const uint32_t total = excl + agg;
            a.chunk_off[a.nchunks] = total;
            hdr->last_escapes = total;
            if ((uint64_t)total > a.esc_capacity) atomicOr(&hdr->status, kStatusOverflow);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.slot_empty[k]);
    }
}

// Last CTA of the launch: move the status bits out and re-arm the header.  A
// clean launch hands out exactly num_tiles + gridDim.x tickets (each producer
// draws one past the end); anything else means the header did not start zeroed.
__device__ void cta_finished(const EncodeArgs& a, uint32_t epoch, bool failed) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    __threadfence();
    const uint32_t prev = atomicAdd(&hdr->done, 1u);
    if (prev == gridDim.x - 1) {
        __threadfence();
        const uint32_t tickets = atomicAdd(&hdr->ticket, 0u);
        const bool timed_out = (atomicAdd(&hdr->status, 0u) & kStatusTimeout) != 0;
        if (!failed && !timed_out && tickets != a.num_tiles + gridDim.x)
            atomicOr(&hdr->status, kStatusBadWorkspace);
        hdr->last_status = atomicExch(&hdr->status, 0u);
        hdr->ticket = 0;
        hdr->done = 0;
        hdr->epoch = epoch + 1u;
        __threadfence();
    }
}

template <class F>
__global__ void __launch_bounds__(kEncodeThreads, 2) encode_kernel(const EncodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    auto& sm = *reinterpret_cast<EncodeSmem<F::kElemBytes>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    __shared__ uint32_t s_epoch;
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int k = 0; k < kSlots; k++) {
            mbar_init(&sm.slot_full[k], kComputeWarps);
            mbar_init(&sm.slot_empty[k], 1);
            mbar_init(&sm.slot_prefix[k], 1);
        }
        sm.err = 0;
        s_epoch = *reinterpret_cast<volatile uint32_t*>(&reinterpret_cast<WsHeader*>(a.ws)->epoch);
        fence_mbar_init();
    }
    if (tid < 256) sm.table[tid] = (uint8_t)kMissEntry;
    __syncthreads();
    if (tid < 16) sm.table[(a.cbw[tid >> 2] >> (8 * (tid & 3))) & 0xFFu] = (uint8_t)tid;
    __syncthreads();
    const uint32_t epoch = s_epoch;
    if (warp < kComputeWarps) {
        compute_role<F>(a, sm, epoch);
    } else if (warp == kProducerWarp) {
        if ((tid & 31) == 0) producer_role<F>(a, sm);
    } else {
        lookback_role<F>(a, sm, epoch, (uint32_t)(warp - kProducerWarp - 1));
    }
    __syncthreads();
    if (tid == 0) cta_finished(a, epoch, *reinterpret_cast<volatile uint32_t*>(&sm.err) != 0);
}

template <class F>
cudaError_t launch_pipeline(const EncodeArgs& a, cudaStream_t s) {
    constexpr size_t smem = sizeof(EncodeSmem<F::kElemBytes>);
    Wave wv;
    const cudaError_t e = launch_wave<encode_kernel<F>>(kEncodeThreads, smem, wv);
    if (e != cudaSuccess) return e;
    if (wv.per_sm < 1) return cudaErrorInvalidConfiguration;
    const uint32_t grid = min(a.num_tiles, (uint32_t)(wv.sms * wv.per_sm));
    encode_kernel<F><<<grid, kEncodeThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int encode_tile_elems(bool e5m2) { return (void)e5m2, kTile; }

cudaError_t launch_encode(const EncodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.num_tiles == 0) return cudaSuccess;
    return e5m2 ? launch_pipeline<E5m2Tile>(a, s) : launch_pipeline<Bf16Tile>(a, s);
}

}  // namespace splitzip
