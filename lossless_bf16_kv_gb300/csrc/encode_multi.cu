// encode_multi.cu -- SplitZip encode in three launches (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README section Abstract; arXiv abstract on the paper index page):
// split each value into exponent and exact sign+mantissa bits, code frequent
// exponents with the 16-entry codebook, send the rest to a chunk-local escape
// stream of (position, value).
//
// The only cross-tile dependency of the format is the escape stream's order
// (chunk, then position) and its offsets.  Here it is taken out of the
// streaming pass:
//   dense   one resident wave of CTAs drawing 8192-element tiles from one
//           counter (four for large BF16 tensors): input staged through a
//           per-thread cp.async ring, field split, code lookup in shared-
//           memory word tables, dense code and sign+mantissa stores.  Each
//           warp ranks the escapes of its segments (ballots when no group
//           holds two escapes, else one shuffle scan) and stores the
//           segments' counts and its first 32 escapes, as one list in element
//           order within each segment, in the workspace; the tile's count
//           goes to the tile's and its block's counters, a completed block's
//           to its superblock's.
//   place   four tiles per warp and round, a lane per warp list (BF16: eight
//           lists of four segments per tile) or per segment (E5M2: eight per
//           tile): the tile offsets from the block and superblock counters
//           (no scan pass, no waits), segment offsets by shuffle scans,
//           escapes copied to their final places, chunk offsets at chunk
//           starts.  A segment whose escapes do not all fit in its warp's
//           list is rebuilt from the input by the whole warp.
//   finish  one CTA: E, chunk_off[C], the call's status and checks; re-arms
//           the counters.
// Segments: BF16 -- the 256 consecutive elements warp w covers with its group
// k (element order 8k + w, count slot 4w + k); warp w's list holds its four
// segments' escapes in order k = 0..3.  E5M2 -- the 1024 elements of warp w,
// the whole list.  Entries hold the position in the segment and the raw
// exponent.
#include <cstdint>

#include "common.cuh"
#include "fields.cuh"
#include "kernels.h"
#include "lookback.cuh"

namespace splitzip {
namespace {

constexpr int kTileElems = 8192;     // elements per tile (dense pass: a CTA per tile at a time)
constexpr int kSegsMax = 32;         // segment slots per tile in the workspace
constexpr int kEntries = 256;        // escape entries per tile in the workspace
constexpr int kWarpCap = kEntries / kWarps;  // 32: entries of one warp's escape list
// Superblocks of the largest tensor (2^32 - 1 elements).
constexpr uint32_t kMaxSupers = (uint32_t)(((1ull << 32) / kTileElems) / kSuperTiles);  // 128
static_assert(kMaxSupers % 32 == 0, "whole superblock counts per lane");

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct MultiPtrs {
    uint64_t* states;
    uint32_t* tile_tot;  // escapes per tile
    uint16_t* seg_cnt;
    uint16_t* seg_ent;
    uint32_t* blk;       // per block of kBlockTiles tiles: escapes | tiles done << kBlkCountShift
    uint32_t* sup;       // escapes per superblock of kSuperTiles tiles
    uint32_t nblocks, nsupers;
    bool striped;  // the dense pass draws its tiles from F::kStripes counters
};

// Stores of segment counts and escape list entries: under the L2 policy pol
// (evict-last) for a format whose lists stay in L2 until placement, plain
// otherwise.
template <bool kKeep>
__device__ __forceinline__ void st_list2(uint16_t* p, uint32_t v, uint64_t pol) {
    if constexpr (kKeep) st_policy2(p, (uint16_t)v, pol);
    else *p = (uint16_t)v;
}
template <bool kKeep>
__device__ __forceinline__ void st_list8(uint16_t* p, uint2 v, uint64_t pol) {
    if constexpr (kKeep) st_policy8(p, v, pol);
    else *reinterpret_cast<uint2*>(p) = v;
}

// Warp-wide exclusive scan of one word per lane, excl = sum of p over the
// lower lanes.  Also returns lane 31's exclusive prefix and word, from which
// the caller forms the warp totals (the formats pack several small counts in
// p, each field wide enough for its exclusive prefix but not necessarily for
// the total).
__device__ __forceinline__ void warp_scan_excl(uint32_t p, uint32_t& excl, uint32_t& e31,
                                               uint32_t& p31) {
    const uint32_t lane = threadIdx.x & 31;
    uint32_t x = __shfl_up_sync(0xFFFFFFFFu, p, 1);
    x = lane ? x : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, d);
        if (lane >= (uint32_t)d) x += y;
    }
    excl = x;
    e31 = __shfl_sync(0xFFFFFFFFu, x, 31);
    p31 = __shfl_sync(0xFFFFFFFFu, p, 31);
}

// Codebook entry 0 (the exponent of code 0), from wherever the codebook is.
__device__ __forceinline__ uint32_t codebook_entry0(const EncodeArgs& a) {
    return a.dcb ? (uint32_t)__ldg(a.dcb) : (a.cbw[0] & 0xFFu);
}

// ------------------------------------------------------------------- BF16
//
// Thread t's groups of 8 at tile offsets k*2048 + 8t (k < 4): each warp load
// covers 512 contiguous input bytes and each warp store 128 code bytes and
// 256 sign+mantissa bytes.
//
// The exponent -> code map is four 256-entry word tables in shared memory,
// one per element position j within a half group of four:
//   T_j[e] = code(e) << 4j          for e in the codebook,
//   T_j[e] = 1 << (16 + j)          for an escape (code 0, flag bit).
// The four entries of elements 4h..4h+3 occupy disjoint bits, so their sum is
// the half group's four code nibbles (bits 0..15) and escape flags (bits
// 16..19).
struct Bf16Dense {
    static constexpr int kGroups = 4;
    static constexpr int kSegs = 32;
    static constexpr int kSegLen = 256;
    static constexpr int kOffBits = 8;
    static constexpr int kPlaceRounds = 2;  // placement: rounds of four tiles per warp
    static constexpr bool kListPlace = true;  // placement with a lane per warp list
    // Counts and lists stored evict-last, so that placement finds them in L2
    // (with its 8- and 16-byte loads of them: 1.151 -> 1.144 ms per encode at
    // 2^31 elements; with a lane per segment it had made the dense pass 3%
    // slower).
    static constexpr bool kKeepLists = true;
    static constexpr uint32_t kExpMask = 0xFFu;
    // Four tile counters, each hit by a quarter of the CTAs' draws (one
    // counter: 1.164 against 1.158 ms at 2^31 elements).
    static constexpr uint32_t kStripes = 4;
    struct Tables {
        uint32_t t[4][256];
    };
    static constexpr int kElemBytes = 2;
    static constexpr int kMinBlocks = 6;  // resident CTAs per SM (shared memory allows 6)
    struct Keep {
        uint32_t miss[kGroups]; // escape flags: bits 0..3 elements 0..3, bits 16..19 elements 4..7
        uint32_t cnt;           // escapes of group k in byte k (at most 8 each)
    };
    static __device__ __forceinline__ uint32_t loff(int k) {
        return k * (kThreads * 8) + threadIdx.x * 8;
    }
    // Segment 8k + w (element order: group k of warp w) is kept at workspace
    // slot 4w + k, so that a warp's four counts are one 8-byte store.
    static __device__ __forceinline__ uint32_t slot(int k) { return (threadIdx.x >> 5) * 4 + k; }
    static __device__ __forceinline__ void build_tables(Tables& tb, const uint32_t (&cbw)[4]) {
        const uint32_t tid = threadIdx.x;
#pragma unroll
        for (int j = 0; j < 4; j++) tb.t[j][tid] = 1u << (16 + j);
        __syncthreads();
        if (tid < 16) {
            const uint32_t q = tid >> 2;
            const uint32_t w = q == 0 ? cbw[0] : q == 1 ? cbw[1] : q == 2 ? cbw[2] : cbw[3];
            const uint32_t e = (w >> (8 * (tid & 3))) & 0xFFu;
#pragma unroll
            for (int j = 0; j < 4; j++) tb.t[j][e] = tid << (4 * j);
        }
        __syncthreads();
    }

    // Table entry of table j for the exponent at bits 7..14 (lo) or 23..30 (hi)
    // of word w.
    static __device__ __forceinline__ uint32_t ent_lo(const Tables& tb, int j, uint32_t w) {
        return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(tb.t[j]) +
                                                  ((w >> 5) & 0x3FCu));
    }
    static __device__ __forceinline__ uint32_t ent_hi(const Tables& tb, int j, uint32_t w) {
        return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(tb.t[j]) +
                                                  ((w >> 21) & 0x3FCu));
    }
    // Codes, sign+mantissa bytes and escape flags of the 8 values in v.
    static __device__ __forceinline__ void group(const Tables& tb, const uint4& v, uint32_t& codes,
                                                 uint2& sm, uint32_t& miss) {
        // Low and high bytes of four values each; sign from the high byte, mantissa
        // from the low byte.
        const uint32_t lo0 = __byte_perm(v.x, v.y, 0x6420), hi0 = __byte_perm(v.x, v.y, 0x7531);
        const uint32_t lo1 = __byte_perm(v.z, v.w, 0x6420), hi1 = __byte_perm(v.z, v.w, 0x7531);
        sm = make_uint2((hi0 & 0x80808080u) | (lo0 & 0x7F7F7F7Fu),
                        (hi1 & 0x80808080u) | (lo1 & 0x7F7F7F7Fu));
        const uint32_t A = ent_lo(tb, 0, v.x) + ent_hi(tb, 1, v.x) + ent_lo(tb, 2, v.y) + ent_hi(tb, 3, v.y);
        const uint32_t B = ent_lo(tb, 0, v.z) + ent_hi(tb, 1, v.z) + ent_lo(tb, 2, v.w) + ent_hi(tb, 3, v.w);
        codes = __byte_perm(A, B, 0x5410);
        miss = __byte_perm(A, B, 0x7632);
    }

    // Input words of a full tile: load k of thread t is the 16 bytes of its
    // group k, staged at ring slot [k][t].
    static constexpr int kLoads = kGroups;
    static constexpr bool kSharedStage = false;  // each thread reads back only its own copies
    static __device__ __forceinline__ const uint8_t* load_src(const EncodeArgs& a, uint32_t t0,
                                                             int k) {
        // One 64-bit base per tile and constant group offsets (a 32-bit element
        // index per group would cost an add and a widening add per access).
        return a.x + 2ull * (t0 + threadIdx.x * 8) + (uint32_t)(k * kThreads * 16);
    }
    static __device__ __forceinline__ uint32_t load_slot(int k) { return k * kThreads + threadIdx.x; }
    static __device__ __forceinline__ void compute_full(const EncodeArgs& a, const Tables& tb,
                                                        uint32_t t0, const uint4* stage, Keep& kp) {
        uint4 v[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; k++) v[k] = stage[load_slot(k)];
        const uint32_t i0 = t0 + threadIdx.x * 8;  // group 0's first element
        uint8_t* cbase = a.codes + i0 / 2;
        uint8_t* sbase = a.signman + i0;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            uint32_t codes, miss;
            uint2 sm;
            group(tb, v[k], codes, sm, miss);
            kp.miss[k] = miss;
            st_stream4(cbase + k * (kThreads * 4), codes);
            st_stream8(sbase + k * (kThreads * 8), sm);
        }
        kp.cnt = __popc(kp.miss[0]) | (__popc(kp.miss[1]) << 8) | (__popc(kp.miss[2]) << 16) |
                 (__popc(kp.miss[3]) << 24);
    }

    // The last, partial tile (element by element at its end).
    static __device__ __forceinline__ void process_partial(const EncodeArgs& a, const Tables& tb,
                                                           uint32_t t0, Keep& kp) {
        const uint32_t pad = codebook_entry0(a) << 7;  // exponent cb[0], sign 0, mantissa 0: code 0
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(a.x);
        kp.cnt = 0;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = t0 + loff(k);
            kp.miss[k] = 0;
            if (i >= a.n) continue;
            const uint32_t rem = a.n - i;
            const bool whole = rem >= 8;
            uint4 v;
            if (whole) {
                v = ld_stream16(a.x + 2ull * i);
            } else {
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; m++)
                    w[m] = (2u * m < rem ? xs[i + 2 * m] : pad) |
                           ((2u * m + 1 < rem ? (uint32_t)xs[i + 2 * m + 1] : pad) << 16);
                v = make_uint4(w[0], w[1], w[2], w[3]);
            }
            uint32_t codes, miss;
            uint2 sm;
            group(tb, v, codes, sm, miss);
            kp.miss[k] = miss;
            kp.cnt |= (uint32_t)__popc(miss) << (8 * k);
            if (whole) {
                st_stream4(a.codes + i / 2, codes);
                st_stream8(a.signman + i, sm);
            } else {
                for (uint32_t j = 0; j < (rem + 1) / 2; j++) a.codes[i / 2 + j] = (uint8_t)(codes >> (8 * j));
                for (uint32_t j = 0; j < rem; j++)
                    a.signman[i + j] = (uint8_t)((j < 4 ? sm.x : sm.y) >> (8 * (j & 3)));
            }
        }
    }

    // True when one of this lane's groups holds two or more escapes.
    static __device__ __forceinline__ bool multi(const Keep& kp) {
        return (kp.cnt & 0xFEFEFEFEu) != 0;
    }
    // Escape entries go to the warp's list of kWarpCap entries, ordered by
    // group k, then lane, then element (so a tile's escapes fill a few
    // sectors): an escape's rank is its group's base (the escapes of the
    // warp's lower groups) plus its rank within the group.
    //
    // Counts and escapes when no group of the warp holds more than one escape
    // (almost every tile at KV-cache escape rates): a group's rank is the
    // number of lower lanes whose same group has an escape, a segment's total
    // the population of that ballot.
    // Both return the warp's escape count (the same in every lane).
    static __device__ __forceinline__ uint32_t bookkeep_single(const Keep& kp, uint16_t* row,
                                                               uint16_t* ent, const uint8_t* in,
                                                               uint64_t pol) {
        const uint32_t lane = threadIdx.x & 31, lt = (1u << lane) - 1u;
        uint32_t has[kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; k++) has[k] = __ballot_sync(0xFFFFFFFFu, kp.miss[k] != 0);
        const uint32_t c0 = __popc(has[0]), c1 = __popc(has[1]), c2 = __popc(has[2]);
        const uint32_t c3 = __popc(has[3]);
        if (lane == 0)
            st_list8<kKeepLists>(row + slot(0), make_uint2(c0 | (c1 << 16), c2 | (c3 << 16)), pol);
        if (kp.cnt) {
            uint32_t excl = 0;
#pragma unroll
            for (int k = 0; k < kGroups; k++) excl |= (uint32_t)__popc(has[k] & lt) << (8 * k);
            const uint32_t base[kGroups] = {0u, c0, c0 + c1, c0 + c1 + c2};
            emit(kp, excl, base, ent, in, pol);
        }
        return c0 + c1 + c2 + c3;
    }
    // Counts and escapes in general: one packed warp scan of the four groups'
    // counts.
    static __device__ __forceinline__ uint32_t bookkeep_multi(const Keep& kp, uint16_t* row,
                                                              uint16_t* ent, const uint8_t* in,
                                                              uint64_t pol) {
        uint32_t excl, e31, p31;
        warp_scan_excl(kp.cnt, excl, e31, p31);
        const uint32_t t02 = (e31 & 0x00FF00FFu) + (p31 & 0x00FF00FFu);  // totals of groups 0, 2
        const uint32_t t13 = ((e31 >> 8) & 0x00FF00FFu) + ((p31 >> 8) & 0x00FF00FFu);  // 1, 3
        if ((threadIdx.x & 31) == 0)
            st_list8<kKeepLists>(
                row + slot(0),
                make_uint2(__byte_perm(t02, t13, 0x5410), __byte_perm(t02, t13, 0x7632)), pol);
        if (kp.cnt) {
            const uint32_t c0 = t02 & 0xFFFFu, c1 = t13 & 0xFFFFu, c2 = t02 >> 16;
            const uint32_t base[kGroups] = {0u, c0, c0 + c1, c0 + c1 + c2};
            emit(kp, excl, base, ent, in, pol);
        }
        return (t02 & 0xFFFFu) + (t02 >> 16) + (t13 & 0xFFFFu) + (t13 >> 16);
    }

    // The warp's first kWarpCap escapes into its list.  excl: the exclusive
    // escape ranks of this lane's groups, one per byte; base: the groups'
    // bases; in: the tile's input (group k of this thread at element loff(k)).
    static __device__ __forceinline__ void emit(const Keep& kp, uint32_t excl,
                                                const uint32_t (&base)[kGroups], uint16_t* ent,
                                                const uint8_t* in, uint64_t pol) {
        const uint32_t lane = threadIdx.x & 31;
        uint16_t* e = ent + (threadIdx.x >> 5) * kWarpCap;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            uint32_t m = kp.miss[k];
            if (!m) continue;
            uint32_t g = base[k] + ((excl >> (8 * k)) & 0xFFu);
            const uint16_t* x = reinterpret_cast<const uint16_t*>(in) + loff(k);
            while (m && g < (uint32_t)kWarpCap) {
                const uint32_t b = __ffs(m) - 1;  // bit b: element (b & 3) + 4 * (b >> 4)
                m &= m - 1;
                const uint32_t j = (b & 3u) + ((b >> 4) << 2);
                const uint32_t ex = ((uint32_t)x[j] >> 7) & kExpMask;
                st_list2<kKeepLists>(e + g++, (8 * lane + j) | (ex << kOffBits), pol);
            }
        }
    }

    // Exponent of element i of the input (placement's chunk ranks).
    static __device__ __forceinline__ uint32_t exponent_at(const EncodeArgs& a, uint32_t i) {
        return (reinterpret_cast<const uint16_t*>(a.x)[i] >> 7) & 0xFFu;
    }
};

// ------------------------------------------------------------------- E5M2
//
// Thread t's group is the 32 elements at tile offset 32t: 16 code bytes and
// 12 bytes of packed 3-bit fields (three 4-byte stores).
struct E5m2Dense {
    static constexpr int kSegs = kWarps;              // 8
    static constexpr int kSegLen = 1024;
    static constexpr int kOffBits = 10;
    static constexpr int kPlaceRounds = 2;  // placement: rounds of four tiles per warp
    static constexpr int kPreload = 8;      // placement: entries per segment loaded ahead
    static constexpr bool kListPlace = false;  // a lane per segment (the segment is the warp's)
    // Counts and lists stored evict-last, so that placement finds them in L2.
    static constexpr bool kKeepLists = true;
    static constexpr uint32_t kExpMask = 0x1Fu;
    // Eight code tables, one per element position q = 0..7 within a pair of
    // input words, indexed by exponent.  Entry t[q][e] holds e's code shifted
    // to nibble q & 3 (bits 0..15: the codes of one word's four elements) and,
    // for an exponent outside the codebook, code 0 with a flag at bit 16 + q.
    // OR-ing a word's four entries gives its 16 code bits; OR-ing a pair's two
    // results gives the pair's 8 escape flags in byte 2.  A byte masked with
    // 0x7C is 4e, the entry's byte offset within its table: lanes reading one
    // table with different exponents always hit different banks.
    struct Tables {
        uint32_t t[8][32];
    };
    static constexpr int kElemBytes = 1;
    static constexpr int kMinBlocks = 6;  // resident CTAs per SM (registers cap it at 40 each)
    // One tile counter: the whole GPU then works on one window of consecutive
    // tiles (four stripes: 0.719 -> 0.736 ms at 2^31 elements).
    static constexpr uint32_t kStripes = 1;
    struct Keep {
        uint32_t mm;   // escape flags of the lane's 32 elements, bit j for element j
        uint32_t cnt;  // popcount of mm
    };
    static __device__ __forceinline__ void build_tables(Tables& tb, const uint32_t (&cbw)[4]) {
        static_assert(kThreads == 256, "one table entry per thread");
        const uint32_t q = threadIdx.x >> 5, e = threadIdx.x & 31;
        uint32_t ent = 1u << (16 + q);
#pragma unroll
        for (int k = 0; k < 16; k++)  // codebook entries are distinct
            if (((cbw[k >> 2] >> (8 * (k & 3))) & 0xFFu) == e) ent = (uint32_t)k << (4 * (q & 3));
        tb.t[q][e] = ent;
        __syncthreads();
    }
    // Table entries of the four bytes of w, OR-ed: table q0 + b for byte b.
    template <int q0>
    static __device__ __forceinline__ uint32_t lookup_word(const Tables& tb, uint32_t w) {
        const uint32_t m = w & 0x7C7C7C7Cu;  // 4 x exponent in each byte
        const char* t = reinterpret_cast<const char*>(&tb.t[q0][0]);
        auto at = [&](int b, uint32_t off) {
            return *reinterpret_cast<const uint32_t*>(t + 128 * b + off);
        };
        return at(0, __byte_perm(m, 0u, 0x4440)) | at(1, __byte_perm(m, 0u, 0x4441)) |
               at(2, __byte_perm(m, 0u, 0x4442)) | at(3, __byte_perm(m, 0u, 0x4443));
    }
    static __device__ __forceinline__ uint32_t slot(int) { return threadIdx.x >> 5; }
    static __device__ __forceinline__ uint32_t storage(uint32_t s) { return s; }

    // Input words of a full tile.  Warp w's 1 KiB (elements 1024w..1024w+1023)
    // arrives as 64 pieces of 16 bytes, lane l copying pieces l and 32 + l of
    // it (coalesced), into stage slots [64w + piece]; thread t then reads its
    // own 32 bytes (pieces 2l and 2l + 1) after a __syncwarp.
    static constexpr int kLoads = 2;
    static constexpr bool kSharedStage = true;  // lanes read pieces other lanes copied
    static __device__ __forceinline__ const uint8_t* load_src(const EncodeArgs& a, uint32_t t0,
                                                             int k) {
        return a.x + t0 + 1024 * (threadIdx.x >> 5) + 512 * k + 16 * (threadIdx.x & 31);
    }
    static __device__ __forceinline__ uint32_t load_slot(int k) {
        return 64 * (threadIdx.x >> 5) + 32 * k + (threadIdx.x & 31);
    }
    static __device__ __forceinline__ void compute_full(const EncodeArgs& a, const Tables& tb,
                                                        uint32_t t0, const uint4* stage, Keep& kp) {
        const uint32_t base = 64 * (threadIdx.x >> 5) + 2 * (threadIdx.x & 31);
        const uint4 v0 = stage[base], v1 = stage[base + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        finish(a, tb, t0 + threadIdx.x * 32, w, true, kp);
    }
    static __device__ __forceinline__ void process_partial(const EncodeArgs& a, const Tables& tb,
                                                           uint32_t t0, Keep& kp) {
        const uint32_t i = t0 + threadIdx.x * 32;
        kp.cnt = 0;
        kp.mm = 0;
        if (i >= a.n) return;
        const bool whole = a.n - i >= 32;  // i < n here
        uint32_t w[8];
        if (whole) {
            const uint4 v0 = ld_stream16(a.x + i);
            const uint4 v1 = ld_stream16(a.x + i + 16);
            w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
            w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
        } else {
            const uint32_t pad = (codebook_entry0(a) & 0x1Fu) << 2;  // exponent cb[0], sign 0, mantissa 0
            const uint32_t rem = a.n - i;
#pragma unroll
            for (int m = 0; m < 8; m++) {
                uint32_t acc = 0;
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    const uint32_t j = m * 4 + b;
                    acc |= (j < rem ? (uint32_t)a.x[i + j] : pad) << (8 * b);
                }
                w[m] = acc;
            }
        }
        finish(a, tb, i, w, whole, kp);
    }

    // Fields, codes and stores of the 32 elements at i (input words w).
    static __device__ __forceinline__ void finish(const EncodeArgs& a, const Tables& tb,
                                                  uint32_t i, const uint32_t (&w)[8], bool whole,
                                                  Keep& kp) {
        uint32_t f12[8], r[8];
#pragma unroll
        for (int m = 0; m < 8; m++) f12[m] = fields12_e5m2(w[m]);
#pragma unroll
        for (int m = 0; m < 8; m += 2) {
            r[m] = lookup_word<0>(tb, w[m]);
            r[m + 1] = lookup_word<4>(tb, w[m + 1]);
        }
        uint4 codes;  // word p: the codes of words 2p (low half) and 2p + 1
        codes.x = __byte_perm(r[0], r[1], 0x5410);
        codes.y = __byte_perm(r[2], r[3], 0x5410);
        codes.z = __byte_perm(r[4], r[5], 0x5410);
        codes.w = __byte_perm(r[6], r[7], 0x5410);
        // Byte 2 of r[2p] | r[2p + 1]: the flags of elements 8p..8p+7, in order.
        const uint32_t o0 = r[0] | r[1], o1 = r[2] | r[3], o2 = r[4] | r[5], o3 = r[6] | r[7];
        kp.mm = __byte_perm(__byte_perm(o0, o1, 0x0062), __byte_perm(o2, o3, 0x0062), 0x5410);
        kp.cnt = __popc(kp.mm);
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

    static __device__ __forceinline__ bool multi(const Keep& kp) { return kp.cnt >= 2; }
    // Counts and escapes when no lane of the warp holds more than one escape.
    static __device__ __forceinline__ uint32_t bookkeep_single(const Keep& kp, uint16_t* row,
                                                               uint16_t* ent, const uint8_t* in,
                                                               uint64_t pol) {
        const uint32_t lane = threadIdx.x & 31;
        const uint32_t has = __ballot_sync(0xFFFFFFFFu, kp.cnt != 0);
        if (lane == 0) st_list2<kKeepLists>(row + slot(0), __popc(has), pol);
        if (kp.cnt) emit(kp, __popc(has & ((1u << lane) - 1u)), ent, in, pol);
        return __popc(has);
    }

    static __device__ __forceinline__ uint32_t bookkeep_multi(const Keep& kp, uint16_t* row,
                                                              uint16_t* ent, const uint8_t* in,
                                                              uint64_t pol) {
        uint32_t excl, e31, p31;
        warp_scan_excl(kp.cnt, excl, e31, p31);
        if ((threadIdx.x & 31) == 0) st_list2<kKeepLists>(row + slot(0), e31 + p31, pol);
        if (kp.cnt) emit(kp, excl, ent, in, pol);
        return e31 + p31;
    }
    // One segment per warp: segment s's entries are warp s's whole list.
    static __device__ __forceinline__ uint32_t seg_list(uint32_t s) { return s; }
    static __device__ __forceinline__ uint32_t seg_base(uint32_t, uint32_t, uint32_t) { return 0u; }

    // The lane's first escapes, from rank excl on, into the segment's entries;
    // in: the tile's input (this lane's 32 elements at byte 32 t).
    static __device__ __forceinline__ void emit(const Keep& kp, uint32_t excl, uint16_t* ent,
                                                const uint8_t* in, uint64_t pol) {
        const uint32_t lane = threadIdx.x & 31;
        const uint8_t* x = in + 32 * threadIdx.x;
        uint16_t* e = ent + slot(0) * kWarpCap;
        uint32_t g = excl;
        for (uint32_t m = kp.mm; m && g < (uint32_t)kWarpCap; m &= m - 1) {
            const uint32_t j = __ffs(m) - 1;
            st_list2<kKeepLists>(
                e + g++, (32 * lane + j) | ((((uint32_t)x[j] >> 2) & kExpMask) << kOffBits), pol);
        }
    }

    static __device__ __forceinline__ uint32_t exponent_at(const EncodeArgs& a, uint32_t i) {
        return (a.x[i] >> 2) & 0x1Fu;
    }
};

// ------------------------------------------------------------ dense pass

// One resident wave of CTAs; the code table is built once per CTA.  Tiles
// are handed out one at a time from counters in the workspace header, so CTAs
// that run faster take more tiles: with a static split, CTAs of equal work
// finished up to three times apart.  There are F::kStripes counters, each in
// its own L2 line, stripe s handing out tiles s, s + kStripes, ... in
// increasing order; a CTA draws from its home stripe and moves on to the next
// when one runs dry.  Thread 0 draws the id of the tile two iterations ahead
// while the CTA works on the current one; one CTA barrier per tile publishes
// it.  The input of
// full tiles comes through a per-thread ring of kDenseStages shared-memory
// slots filled by cp.async: while a thread works on one tile, its copies of
// the next kDenseStages - 1 tiles are in flight, with no registers held for
// them.  A slot is refilled only after the values read from it have been used
// by the tile's stores.
constexpr int kDenseStages = 2;
constexpr uint32_t kNoTile = 0xFFFFFFFFu;  // drawn once every stripe is dry

template <class F>
constexpr size_t dense_smem_bytes() {
    return (size_t)kDenseStages * F::kLoads * kThreads * sizeof(uint4);
}

template <class F>
__global__ void __launch_bounds__(kThreads, F::kMinBlocks) dense_kernel(const EncodeArgs a,
                                                                       const MultiPtrs p) {
    constexpr int L = F::kLoads, S = kDenseStages;
    static_assert(kDenseStages == 2, "two tile ids ahead");
    extern __shared__ uint4 ring[];  // [S][L][kThreads]
    __shared__ typename F::Tables tables;
    __shared__ uint32_t s_grab[4];   // tile ids drawn by thread 0: [0..1] alternate, [2..3] the first two
    __shared__ uint32_t s_tot[2];    // the tile's escape count, summed over the warps (alternate)
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    launch_dependents();  // placement CTAs may take SM slots as this pass's CTAs finish
    // Thread 0's draws with several stripes: from its home stripe, then from
    // the next ones as they run dry; kNoTile once every stripe is dry (so no
    // tile follows it).  With one (or p.striped false), the counter hands out
    // tiles in order and the first draw takes two.
    uint32_t tries = 0;
    constexpr uint32_t NS = F::kStripes;
    static_assert(NS >= 1 && NS <= kDenseStripes, "stripe counters in the header");
    auto draw = [&]() -> uint32_t {
        while (tries < NS) {
            const uint32_t st = (blockIdx.x + tries) % NS;
            const uint32_t t = st + NS * atomicAdd(&hdr->dense_stripe[st][0], 1u);
            if (t < a.num_tiles) return t;
            tries++;
        }
        return kNoTile;
    };
    if (threadIdx.x == 0) {
        if (NS == 1 || !p.striped) {
            s_grab[2] = atomicAdd(&hdr->dense_next, 2u);
            s_grab[3] = s_grab[2] + 1;
        } else {
            s_grab[2] = draw();
            s_grab[3] = draw();
        }
        s_tot[0] = s_tot[1] = 0;
    }
    {
        uint32_t cbw[4];
        codebook_words(a.dcb, a.cbw, cbw);
        F::build_tables(tables, cbw);  // ends with a CTA barrier: s_grab[2..3] are visible
    }
    // With F::kKeepLists, counts and list entries stay in L2 for the prefix and
    // placement passes while the tensor streams through.
    const uint64_t keep = F::kKeepLists ? l2_evict_last_policy() : 0u;
    const uint32_t full_tiles = a.n / (uint32_t)kTileElems;
    auto fill = [&](uint32_t tile, int slot) {
        if (tile < full_tiles) {
#pragma unroll
            for (int k = 0; k < L; k++)
                cp_async16(&ring[slot * L * kThreads + F::load_slot(k)],
                           F::load_src(a, tile * (uint32_t)kTileElems, k));
        }
        cp_async_commit();  // one group per tile, empty for a tile not staged
    };
    uint32_t tile = s_grab[2], next = s_grab[3];
    fill(tile, 0);
    fill(next, 1);
    int slot = 0;
    uint32_t it = 0;
    for (; tile < a.num_tiles; it++) {
        if (threadIdx.x == 0) {  // two ahead
            if (NS == 1 || !p.striped) s_grab[it & 1] = atomicAdd(&hdr->dense_next, 1u);
            else s_grab[it & 1] = draw();
        }
        const uint32_t t0 = tile * (uint32_t)kTileElems;
        typename F::Keep kp;
        const uint8_t* in;  // the tile's input, from which the escapes are read
        if (tile < full_tiles) {
            cp_async_wait<S - 1>();  // this tile's group (the oldest pending) has landed
            if (F::kSharedStage) __syncwarp();  // the warp's copies, visible to all its lanes
            F::compute_full(a, tables, t0, ring + slot * L * kThreads, kp);
            in = reinterpret_cast<const uint8_t*>(ring + slot * L * kThreads);
        } else {
            F::process_partial(a, tables, t0, kp);
            in = a.x + (size_t)t0 * F::kElemBytes;
        }
        // The bookkeeping reads escapes from the stage: refill after it.
        uint16_t* row = p.seg_cnt + (size_t)tile * kSegsMax;
        uint16_t* ent = p.seg_ent + (size_t)tile * kEntries;
        const uint32_t wt = !__any_sync(0xFFFFFFFFu, F::multi(kp))
                                ? F::bookkeep_single(kp, row, ent, in, keep)
                                : F::bookkeep_multi(kp, row, ent, in, keep);
        if ((threadIdx.x & 31) == 0 && wt) atomicAdd(&s_tot[it & 1], wt);
        __syncthreads();  // the drawn id and the tile's count are in; every lane has read the stage
        if (threadIdx.x == 0) {
            // The tile's escape count, and its block's, for placement.  The
            // tile that completes its block adds the block's count to the
            // superblock's: tiles in flight lie in a window of consecutive
            // tiles, so a per-tile add there would make one hot address.
            const uint32_t tot = s_tot[it & 1];
            s_tot[it & 1] = 0;  // written again two tiles on, after the next barrier
            p.tile_tot[tile] = tot;
            const uint32_t bk = tile / kBlockTiles, left = a.num_tiles - bk * kBlockTiles;
            const uint32_t in_block = left < kBlockTiles ? left : kBlockTiles;
            const uint32_t old = atomicAdd(p.blk + bk, tot + (1u << kBlkCountShift));
            if ((old >> kBlkCountShift) == in_block - 1u) {
                const uint32_t btot = (old & kBlkEscMask) + tot;
                if (btot) atomicAdd(p.sup + tile / kSuperTiles, btot);
            }
        }
        const uint32_t ahead = s_grab[it & 1];
        fill(ahead, slot);
        slot = slot + 1 == S ? 0 : slot + 1;
        tile = next;
        next = ahead;
    }
    cp_async_wait<0>();
    if (threadIdx.x == 0 && it) atomicAdd(&hdr->dense_done, it);  // tiles this CTA processed
}

// ------------------------------------------------------ escape offsets
//
// The dense pass adds each tile's escape count to its block's (kBlockTiles
// tiles) counter, and each block's to its superblock's (kSuperTiles tiles).  The exclusive
// escape offset of tile t is then the sum over the superblocks before t's,
// the blocks of t's superblock before t's block, and the tiles of t's block
// before t: a warp finds the offsets of a whole block with one round of
// loads (at most 4 + 2 + 2 per lane) and warp scans, with no pass of its own
// and no waits.

// For the block holding tile `first`: before = the escapes of all tiles before
// the block; ex_lo / ex_hi = the exclusive offset, inside the block, of the
// block's tile `lane` / `32 + lane`.  All lanes call it.
__device__ __forceinline__ void block_offsets(const MultiPtrs& p, uint32_t first,
                                              uint32_t num_tiles, uint32_t& before,
                                              uint32_t& ex_lo, uint32_t& ex_hi) {
    static_assert(kBlockTiles == 64 && kSuperTiles % (32 * kBlockTiles) == 0, "two tiles per lane");
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t sp = first / kSuperTiles, bk = first / kBlockTiles, t0 = bk * kBlockTiles;
    // Every load is issued before any is used (one memory round trip): at
    // most kMaxSupers / 32 superblock and kSuperTiles / kBlockTiles / 32 block
    // counts per lane.
    constexpr uint32_t kSupPerLane = kMaxSupers / 32, kBlkPerLane = kSuperTiles / kBlockTiles / 32;
    const uint32_t v_lo = t0 + lane < num_tiles ? __ldcg(p.tile_tot + t0 + lane) : 0u;
    const uint32_t v_hi = t0 + 32 + lane < num_tiles ? __ldcg(p.tile_tot + t0 + 32 + lane) : 0u;
    uint32_t vs[kSupPerLane], vb[kBlkPerLane];
#pragma unroll
    for (uint32_t k = 0; k < kSupPerLane; k++) {
        const uint32_t i = lane + 32 * k;
        vs[k] = i < sp ? __ldcg(p.sup + i) : 0u;
    }
#pragma unroll
    for (uint32_t k = 0; k < kBlkPerLane; k++) {
        const uint32_t i = sp * (kSuperTiles / kBlockTiles) + lane + 32 * k;
        vb[k] = i < bk ? __ldcg(p.blk + i) & kBlkEscMask : 0u;
    }
    uint32_t acc = 0;
#pragma unroll
    for (uint32_t k = 0; k < kSupPerLane; k++) acc += vs[k];
#pragma unroll
    for (uint32_t k = 0; k < kBlkPerLane; k++) acc += vb[k];
#pragma unroll
    for (int d = 16; d; d >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, d);
    uint32_t lo = v_lo, hi = v_hi;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, lo, d), w = __shfl_up_sync(0xFFFFFFFFu, hi, d);
        if (lane >= (uint32_t)d) {
            lo += u;
            hi += w;
        }
    }
    before = acc;
    ex_lo = lo - v_lo;
    ex_hi = hi - v_hi + __shfl_sync(0xFFFFFFFFu, lo, 31);
}

// Offset of the block's tile j (0 <= j < 64) from block_offsets' results; all
// lanes call it, each with its own j.
__device__ __forceinline__ uint32_t offset_in_block(uint32_t before, uint32_t ex_lo,
                                                    uint32_t ex_hi, uint32_t j) {
    const uint32_t a = __shfl_sync(0xFFFFFFFFu, ex_lo, j & 31u);
    const uint32_t b = __shfl_sync(0xFFFFFFFFu, ex_hi, j & 31u);
    return before + (j < 32 ? a : b);
}

// One CTA after placement: E is the sum of the superblock counters;
// chunk_off[C], the status bits and the checks of the call; the counters are
// zeroed for the next encode.  Every tile processed exactly once and blocks
// adding up to the superblocks show a workspace that started consistent.  (A
// launch of its own: electing the last placement CTA cost every CTA a fence
// and a returning atomic while it held its SM slot.)
constexpr int kFinishThreads = 1024;
constexpr int kFinishWarps = kFinishThreads / 32;
constexpr uint32_t kMaxBlocks = kMaxSupers * (kSuperTiles / kBlockTiles);  // 8192

template <class F>
__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const EncodeArgs a, const MultiPtrs p) {
    static_assert(kMaxBlocks % kFinishThreads == 0 && kMaxSupers <= kFinishThreads, "whole rounds");
    constexpr int kPer = kMaxBlocks / kFinishThreads;
    __shared__ uint32_t s_part[3][kFinishWarps];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Every count is loaded before any is used or zeroed, and thread 0's
    // header words and device codebook with them (one memory round trip).
    uint32_t dense_done = 0, status = 0, cbw[4] = {0, 0, 0, 0};
    if (threadIdx.x == 0) {
        dense_done = __ldcg(&hdr->dense_done);
        status = __ldcg(&hdr->status);
        if (a.dcb) codebook_words(a.dcb, a.cbw, cbw);
    }
    uint32_t vb[kPer];
#pragma unroll
    for (int k = 0; k < kPer; k++) {
        const uint32_t i = threadIdx.x + k * kFinishThreads;
        vb[k] = i < p.nblocks ? __ldcg(p.blk + i) : 0u;
    }
    uint32_t e_sup = threadIdx.x < p.nsupers ? __ldcg(p.sup + threadIdx.x) : 0u, e_blk = 0, t_blk = 0;
#pragma unroll
    for (int k = 0; k < kPer; k++) {
        e_blk += vb[k] & kBlkEscMask;
        t_blk += vb[k] >> kBlkCountShift;
    }
    // Placement reads the counters: zero them (and write the call's results)
    // only once it has finished.  The loads above read what the dense pass
    // wrote, complete before placement started.
    wait_prerequisite_grid();
#pragma unroll
    for (int k = 0; k < kPer; k++) {
        const uint32_t i = threadIdx.x + k * kFinishThreads;
        if (i < p.nblocks) p.blk[i] = 0;
    }
    if (threadIdx.x < p.nsupers) p.sup[threadIdx.x] = 0;
#pragma unroll
    for (int d = 16; d; d >>= 1) {
        e_sup += __shfl_xor_sync(0xFFFFFFFFu, e_sup, d);
        e_blk += __shfl_xor_sync(0xFFFFFFFFu, e_blk, d);
        t_blk += __shfl_xor_sync(0xFFFFFFFFu, t_blk, d);
    }
    if (lane == 0) {
        s_part[0][warp] = e_sup;
        s_part[1][warp] = e_blk;
        s_part[2][warp] = t_blk;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t total = 0, blocks = 0, counted = 0;
#pragma unroll
        for (int w = 0; w < kFinishWarps; w++) {
            total += s_part[0][w];
            blocks += s_part[1][w];
            counted += s_part[2][w];
        }
        a.chunk_off[a.nchunks] = total;
        hdr->last_escapes = total;
        if ((uint64_t)total > a.esc_capacity) status |= kStatusOverflow;
        // A codebook from device memory is checked here, once per encode.
        if (a.dcb && !codebook_valid(cbw, F::kExpMask)) status |= kStatusBadCodebook;
        if (dense_done != a.num_tiles || counted != a.num_tiles || blocks != total)
            status |= kStatusBadWorkspace;
        hdr->last_status = status;
        hdr->status = 0;
        hdr->done = 0;
#pragma unroll
        for (uint32_t st = 0; st < kDenseStripes; st++) hdr->dense_stripe[st][0] = 0;
        hdr->dense_next = 0;
        hdr->dense_done = 0;
        __threadfence();
    }
}

// ------------------------------------------------------------- placement

__device__ __forceinline__ void put_escape(const EncodeArgs& a, uint32_t g, uint32_t pos,
                                           uint32_t e) {
    if ((uint64_t)g < a.esc_capacity) {
        a.esc_pos[g] = (uint16_t)pos;
        a.esc_val[g] = (uint8_t)e;
    }
}

// Whether exponent e (< 256) is one of the 16 codebook entries, four per word:
// some byte of cbw[q] ^ (e in every byte) is zero.
__device__ __forceinline__ bool in_codebook(const uint32_t (&cbw)[4], uint32_t e) {
    const uint32_t rep = e * 0x01010101u;
    uint32_t z = 0;
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t t = cbw[q] ^ rep;
        z |= (t - 0x01010101u) & ~t & 0x80808080u;  // nonzero iff t has a zero byte
    }
    return z != 0;
}

// The escapes of segment sg (element order) of tile `tile`, rebuilt from the
// input by the whole warp: a segment whose escapes did not all fit in its
// warp's list (escape-heavy data).  Lane j takes the segment's elements
// j * PER .. j * PER + PER - 1 (one or two 16-byte loads), flags its escapes
// through the shared-memory table isesc (1 for an exponent outside the
// codebook), and stores them from g0 + (the escapes of the lower lanes) on, in
// element order.  All lanes call it.
template <class F>
__device__ __forceinline__ void rebuild_segment(const EncodeArgs& a, uint32_t tile, uint32_t sg,
                                                uint32_t g0, const uint8_t* isesc) {
    constexpr uint32_t PER = F::kSegLen / 32;  // 8 BF16 or 32 E5M2 elements per lane
    constexpr uint32_t W = PER * F::kElemBytes / 4;  // input words per lane: 4 or 8
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t t0 = tile * (uint32_t)kTileElems;
    const uint32_t len = a.n - t0 < (uint32_t)kTileElems ? a.n - t0 : (uint32_t)kTileElems;
    const uint32_t l0 = sg * F::kSegLen + lane * PER;  // the lane's first element, tile-local
    const uint8_t* src = a.x + (size_t)(t0 + l0) * F::kElemBytes;
    uint32_t w[W];
    if (l0 + PER <= len) {
#pragma unroll
        for (uint32_t q = 0; q < W; q += 4) {
            const uint4 v = ld_stream16(src + 4 * q);
            w[q] = v.x; w[q + 1] = v.y; w[q + 2] = v.z; w[q + 3] = v.w;
        }
    } else {  // the segment ends inside this lane's elements (or before them)
#pragma unroll
        for (uint32_t q = 0; q < W; q++) {
            uint32_t acc = 0;
#pragma unroll
            for (uint32_t b = 0; b < 4; b++)
                if (l0 * F::kElemBytes + 4 * q + b < len * F::kElemBytes)
                    acc |= (uint32_t)src[4 * q + b] << (8 * b);
            w[q] = acc;
        }
    }
    // Exponent of the lane's element k (k < PER).
    auto exponent = [&](uint32_t k) {
        if constexpr (PER == 8) {
            uint32_t v = w[0];
#pragma unroll
            for (uint32_t q = 1; q < W; q++) v = (k >> 1) == q ? w[q] : v;
            return ((v >> (16 * (k & 1u) + 7)) & 0xFFu);
        } else {
            uint32_t v = w[0];
#pragma unroll
            for (uint32_t q = 1; q < W; q++) v = (k >> 2) == q ? w[q] : v;
            return ((v >> (8 * (k & 3u) + 2)) & 0x1Fu);
        }
    };
    uint32_t mask = 0;
#pragma unroll
    for (uint32_t k = 0; k < PER; k++)
        if (l0 + k < len && isesc[exponent(k)]) mask |= 1u << k;
    uint32_t excl, e31, p31;
    warp_scan_excl(__popc(mask), excl, e31, p31);
    uint32_t g = g0 + excl;
    const uint32_t r0 = t0 - chunk_quot32(a.cdiv, t0) * a.cdiv.d;  // the tile's start in its chunk
    for (uint32_t m = mask; m; m &= m - 1) {
        const uint32_t k = __ffs(m) - 1;
        const uint32_t x = r0 + l0 + k;  // < d + kTileElems, in chunk_quot's exact range
        put_escape(a, g++, x - chunk_quot(a.cdiv, x) * a.cdiv.d, exponent(k));
    }
}

// Placement with a lane per segment (E5M2, whose segment is a warp's whole
// list).  A warp places the escapes of F::kPlaceRounds x 32 / kSegs
// consecutive tiles (2 x 4): in round r lane l takes segment l mod kSegs
// (element order) of tile tile0 + r * 32 / kSegs + l / kSegs.  Every round's
// tile offset and counts are loaded before any is used, and every round's
// first F::kPreload entries before any escape is stored (loads cannot pass
// the stores, which the compiler must assume may alias them), so a warp waits
// for two memory round trips in all rather than two per tile.
template <class F, int R>
__global__ void __launch_bounds__(kThreads, 4) place_kernel(const EncodeArgs a, const MultiPtrs p,
                                                            uint32_t num_tiles) {
    constexpr uint32_t kOffMask = (1u << F::kOffBits) - 1u;
    constexpr uint32_t SEGS = F::kSegs, TPW = 32 / F::kSegs;
    constexpr int K = F::kPreload;
    static_assert(kBlockTiles % (TPW * R) == 0, "a warp's tiles lie in one block");
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ uint8_t isesc_all[kWarps][256];  // per warp: 1 for an exponent outside the codebook
    uint8_t* isesc = isesc_all[warp];
    const uint32_t tile0 = (blockIdx.x * kWarps + warp) * TPW * R;
    wait_prerequisite_grid();        // the dense pass has completed, its writes visible
    launch_dependents();             // the finishing launch may start (it waits for this grid)
    if (tile0 >= num_tiles) return;  // warp-uniform
    const uint32_t sub = lane / SEGS, sgl = lane % SEGS;  // this lane's tile and segment
    const uint32_t lbase = lane & ~(SEGS - 1);
    const uint32_t s0 = sgl * F::kSegLen;  // the segment's tile-local start
    auto tile_of = [&](int r) { return tile0 + (uint32_t)r * TPW + sub; };

    uint32_t excl[R], cnt[R], off[R], sbase[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        const uint32_t tile = tile_of(r);
        cnt[r] = tile < num_tiles ? ld_last2(p.seg_cnt + (size_t)tile * kSegsMax + F::storage(sgl)) : 0u;
    }
    {
        uint32_t before, ex_lo, ex_hi;
        block_offsets(p, tile0, num_tiles, before, ex_lo, ex_hi);
        const uint32_t b0 = tile0 / kBlockTiles * kBlockTiles;
#pragma unroll
        for (int r = 0; r < R; r++) {
            const uint32_t tile = tile_of(r);
            const uint32_t o = offset_in_block(before, ex_lo, ex_hi, tile - b0);
            excl[r] = tile < num_tiles ? o : 0u;
        }
    }
#pragma unroll
    for (int r = 0; r < R; r++) {
        // Exclusive scan of the counts within each tile's group of SEGS lanes.
        uint32_t incl = cnt[r];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += u;
        }
        const uint32_t first = __shfl_sync(0xFFFFFFFFu, incl - cnt[r], lbase);
        off[r] = incl - cnt[r] - first;
        // Where this lane's segment's entries start in its warp list.
        sbase[r] = F::seg_base(sgl, cnt[r], lbase);
    }
    auto entries = [&](int r) {
        return p.seg_ent + (size_t)tile_of(r) * kEntries + F::seg_list(sgl) * kWarpCap + sbase[r];
    };
    // Every segment is a whole warp list, starting on a 16-byte boundary: its
    // first eight entries are one 16-byte load.
    static_assert(K == 8 && SEGS == kWarps, "a list per segment, eight entries preloaded");
    uint32_t ev[R][K];
#pragma unroll
    for (int r = 0; r < R; r++) {
        const bool listed = sbase[r] + cnt[r] <= (uint32_t)kWarpCap;
        const uint4 v = listed && cnt[r] ? ld_last16(entries(r)) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < K; k++) ev[r][k] = (vw[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
    }

    // Escapes of segment sgl of each round's tile, in element order.  When the
    // chunk size is a multiple of the segment length the segment lies in one
    // chunk, and an escape's position in it is the segment's offset in that
    // chunk plus the entry's offset.
    const bool seg_in_chunk = a.cdiv.d % (uint32_t)F::kSegLen == 0;
#pragma unroll
    for (int r = 0; r < R; r++) {
        if (!cnt[r]) continue;
        const uint32_t t0 = tile_of(r) * (uint32_t)kTileElems;
        const uint32_t r0 = t0 - chunk_quot32(a.cdiv, t0) * a.cdiv.d;
        const uint32_t g0 = excl[r] + off[r];
        if (sbase[r] + cnt[r] <= (uint32_t)kWarpCap) {
            const uint16_t* es = entries(r);
            if (seg_in_chunk && (uint64_t)g0 + cnt[r] <= a.esc_capacity) {
                const uint32_t xs = r0 + s0, base = xs - chunk_quot(a.cdiv, xs) * a.cdiv.d;
                auto put = [&](uint32_t g, uint32_t e) {
                    a.esc_pos[g] = (uint16_t)(base + (e & kOffMask));
                    a.esc_val[g] = (uint8_t)(e >> F::kOffBits);
                };
#pragma unroll
                for (int k = 0; k < K; k++)
                    if ((uint32_t)k < cnt[r]) put(g0 + k, ev[r][k]);
                for (uint32_t q = K; q < cnt[r]; q++) put(g0 + q, es[q]);
            } else {
                auto put = [&](uint32_t g, uint32_t e) {
                    const uint32_t x = r0 + s0 + (e & kOffMask);
                    put_escape(a, g, x - chunk_quot(a.cdiv, x) * a.cdiv.d, e >> F::kOffBits);
                };
#pragma unroll
                for (int k = 0; k < K; k++)
                    if ((uint32_t)k < cnt[r]) put(g0 + k, ev[r][k]);
                for (uint32_t q = K; q < cnt[r]; q++) put(g0 + q, es[q]);
            }
        }  // else: more escapes than the segment's list entries, rebuilt below
    }
    // Segments whose escapes overflowed their lists, rebuilt by the whole warp
    // one at a time (the warp first builds its escape table).
    bool table = false;
#pragma unroll
    for (int r = 0; r < R; r++) {
        for (uint32_t ov = __ballot_sync(0xFFFFFFFFu, cnt[r] && sbase[r] + cnt[r] > (uint32_t)kWarpCap);
             ov; ov &= ov - 1) {
            const uint32_t l = __ffs(ov) - 1;
            const uint32_t g0 = __shfl_sync(0xFFFFFFFFu, excl[r] + off[r], l);
            if (!table) {  // warp-uniform
                uint32_t cbw[4];
                codebook_words(a.dcb, a.cbw, cbw);
#pragma unroll
                for (uint32_t e = lane; e < 256; e += 32) isesc[e] = !in_codebook(cbw, e);
                __syncwarp();
                table = true;
            }
            rebuild_segment<F>(a, tile0 + (uint32_t)r * TPW + l / SEGS, l % SEGS, g0, isesc);
        }
    }


    // chunk_off at every chunk start of each of the warp's tiles: the exclusive
    // escape rank of the chunk's first element.  When the chunk size is a
    // multiple of the segment length every chunk start inside a tile is a
    // segment start (tiles and segments start at multiples of it), and the
    // lane of that segment writes it from its own offset.
    if (seg_in_chunk) {
#pragma unroll
        for (int r = 0; r < R; r++) {
            const uint32_t tile = tile_of(r);
            if (tile >= num_tiles) continue;
            const uint32_t t0 = tile * (uint32_t)kTileElems;
            const uint32_t len = a.n - t0 < (uint32_t)kTileElems ? a.n - t0 : (uint32_t)kTileElems;
            const uint32_t q0 = chunk_quot32(a.cdiv, t0), x = t0 - q0 * a.cdiv.d + s0;
            const uint32_t qx = chunk_quot(a.cdiv, x);  // x < d + kTileElems
            if (s0 < len && x == qx * a.cdiv.d) a.chunk_off[q0 + qx] = excl[r] + off[r];
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < R; r++) {
        for (uint32_t t = 0; t < TPW; t++) {
            const uint32_t tl = tile0 + (uint32_t)r * TPW + t;
            if (tl >= num_tiles) break;  // warp-uniform
            const uint32_t u0 = tl * (uint32_t)kTileElems;
            const uint32_t ulen = a.n - u0 < (uint32_t)kTileElems ? a.n - u0 : (uint32_t)kTileElems;
            const uint32_t uq0 = chunk_quot32(a.cdiv, u0), ur0 = u0 - uq0 * a.cdiv.d;
            const uint32_t uexcl = __shfl_sync(0xFFFFFFFFu, excl[r], t * SEGS);
            const uint16_t* uent = p.seg_ent + (size_t)tl * kEntries;
            const uint32_t qa = ur0 ? 1u : 0u, qb = chunk_quot(a.cdiv, ur0 + ulen - 1);
            for (uint32_t b0 = qa; b0 <= qb; b0 += 32) {
                const uint32_t q = b0 + lane;
                const bool valid = q <= qb;
                const uint32_t bl = valid ? q * a.cdiv.d - ur0 : 0u;  // tile-local chunk start
                const uint32_t sg = bl / F::kSegLen;
                const uint32_t o = __shfl_sync(0xFFFFFFFFu, off[r], t * SEGS + sg);
                const uint32_t c = __shfl_sync(0xFFFFFFFFu, cnt[r], t * SEGS + sg);
                const uint32_t bb = __shfl_sync(0xFFFFFFFFu, sbase[r], t * SEGS + sg);
                if (valid) {
                    const uint32_t lim = bl - sg * F::kSegLen;
                    uint32_t rank = 0;
                    if (lim == 0) {
                    } else if (bb + c <= (uint32_t)kWarpCap) {
                        const uint16_t* es = uent + F::seg_list(sg) * kWarpCap + bb;
                        for (uint32_t q2 = 0; q2 < c; q2++) rank += (es[q2] & kOffMask) < lim;
                    } else {
                        uint32_t cbw[4];
                        codebook_words(a.dcb, a.cbw, cbw);
                        for (uint32_t l = sg * F::kSegLen; l < bl; l++)
                            rank += !in_codebook(cbw, F::exponent_at(a, u0 + l));
                    }
                    a.chunk_off[uq0 + q] = uexcl + o + rank;
                }
            }
        }
    }
}

// BF16 placement with a lane per warp list: in round r, lanes 8t..8t+7 take
// tile tile0 + TPW r + t and lane 8t + w the list the dense pass's warp w wrote,
// which holds its four segments (w + 8k, elements 2048k + 256w .. + 255 of
// the tile, k = 0..3) in order k.  The lane's four counts are one 8-byte
// load; a scan of the counts packed two to a word (16-bit fields: a tile's
// total per k is at most 8 x 256) over the tile's eight lanes gives each
// segment's offset in the tile, the element order being k-major.  The lane
// then walks its list's entries (the first eight from one 16-byte load).
// Per tile this issues a fraction of the instructions of a lane per segment
// (32 segments, each with its own scans and loads).
__device__ __forceinline__ uint32_t pick4(uint32_t k, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3) {
    return k == 0 ? a0 : k == 1 ? a1 : k == 2 ? a2 : a3;
}

// TPW tiles per warp and round: four, or two for smaller tensors (lanes
// 16..31 idle).  With four, a tensor of 2^26 elements leaves 13 warps per SM,
// and with 60% escapes each rebuilt up to 128 overflowed segments one after
// another (encode 0.37 ms against 0.245 with two and 0.225 with one); a tile
// per warp made the KV layer 3 us slower (54 against 51 us).
template <int R, uint32_t TPW>
__global__ void __launch_bounds__(kThreads, 4) place_lists_kernel(const EncodeArgs a,
                                                                  const MultiPtrs p,
                                                                  uint32_t num_tiles) {
    using F = Bf16Dense;
    constexpr uint32_t G = 8;  // lanes (lists) per tile
    static_assert(TPW == 1 || TPW == 2 || TPW == 4, "one, two or four tiles per warp and round");
    constexpr uint32_t kOffMask = (1u << F::kOffBits) - 1u;
    static_assert(G == kWarps && F::kSegLen * kWarps * 4 == kTileElems, "four segments per list");
    static_assert(kBlockTiles % (TPW * R) == 0, "a warp's tiles lie in one block");
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ uint8_t isesc_all[kWarps][256];  // per warp: 1 for an exponent outside the codebook
    uint8_t* isesc = isesc_all[warp];
    const uint32_t tile0 = (blockIdx.x * kWarps + warp) * TPW * R;
    wait_prerequisite_grid();        // the dense pass has completed, its writes visible
    launch_dependents();             // the finishing launch may start (it waits for this grid)
    if (tile0 >= num_tiles) return;  // warp-uniform
    const uint32_t sub = lane / G, w = lane % G;
    // The lane's tile; num_tiles (no tile) for an idle lane.
    auto tile_of = [&](int r) { return sub < TPW ? tile0 + (uint32_t)r * TPW + sub : num_tiles; };
    auto list_of = [&](int r) {
        return p.seg_ent + (size_t)tile_of(r) * kEntries + w * (uint32_t)kWarpCap;
    };

    // Round trip 1: every round's counts and the block's offsets.
    uint2 c4[R];
    uint32_t toff[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        const uint32_t tile = tile_of(r);
        c4[r] = tile < num_tiles ? ld_last8(p.seg_cnt + (size_t)tile * kSegsMax + 4 * w)
                                 : make_uint2(0u, 0u);
    }
    {
        uint32_t before, ex_lo, ex_hi;
        block_offsets(p, tile0, num_tiles, before, ex_lo, ex_hi);
        const uint32_t b0 = tile0 / kBlockTiles * kBlockTiles;
#pragma unroll
        for (int r = 0; r < R; r++) toff[r] = offset_in_block(before, ex_lo, ex_hi, tile_of(r) - b0);
    }
    // Round trip 2: the first eight entries of every non-empty list.
    uint4 pre[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        const bool any = (c4[r].x | c4[r].y) != 0u;
        pre[r] = any ? ld_last16(list_of(r)) : make_uint4(0u, 0u, 0u, 0u);
    }

    const bool seg_in_chunk = a.cdiv.d % (uint32_t)F::kSegLen == 0;
    bool table = false;
#pragma unroll
    for (int r = 0; r < R; r++) {
        const uint32_t tile = tile_of(r);
        const bool valid = tile < num_tiles;
        // Segment offsets in the tile: exclusive over the lower lists for the
        // same k, plus the tile's totals of the lower k.
        uint32_t i0 = c4[r].x, i1 = c4[r].y;
#pragma unroll
        for (uint32_t d = 1; d < G; d <<= 1) {
            const uint32_t u0 = __shfl_up_sync(0xFFFFFFFFu, i0, d, G);
            const uint32_t u1 = __shfl_up_sync(0xFFFFFFFFu, i1, d, G);
            if (w >= d) {
                i0 += u0;
                i1 += u1;
            }
        }
        const uint32_t T0 = __shfl_sync(0xFFFFFFFFu, i0, G - 1, G);
        const uint32_t T1 = __shfl_sync(0xFFFFFFFFu, i1, G - 1, G);
        const uint32_t e0 = i0 - c4[r].x, e1 = i1 - c4[r].y;
        const uint32_t t0 = T0 & 0xFFFFu, t01 = t0 + (T0 >> 16), t012 = t01 + (T1 & 0xFFFFu);
        const uint32_t off0 = e0 & 0xFFFFu, off1 = t0 + (e0 >> 16);
        const uint32_t off2 = t01 + (e1 & 0xFFFFu), off3 = t012 + (e1 >> 16);
        const uint32_t c0 = c4[r].x & 0xFFFFu, c1 = c4[r].x >> 16;
        const uint32_t c2 = c4[r].y & 0xFFFFu, c3 = c4[r].y >> 16;
        const uint32_t S1 = c0, S2 = c0 + c1, S3 = S2 + c2, tot = S3 + c3;
        // Segments whose entries did not all fit in the list (rebuilt below).
        const uint32_t ovf = (S1 > (uint32_t)kWarpCap ? 1u : 0u) | (S2 > (uint32_t)kWarpCap ? 2u : 0u) |
                             (S3 > (uint32_t)kWarpCap ? 4u : 0u) | (tot > (uint32_t)kWarpCap ? 8u : 0u);
        const uint32_t ovk = ovf & ((c0 ? 1u : 0u) | (c1 ? 2u : 0u) | (c2 ? 4u : 0u) | (c3 ? 8u : 0u));
        const uint32_t t0e = tile * (uint32_t)kTileElems;
        const uint32_t r0 = valid ? t0e - chunk_quot32(a.cdiv, t0e) * a.cdiv.d : 0u;
        // The listed segments are a prefix of the four (the ends S1, S2, S3,
        // tot grow): walk the entries up to the end of the last one.
        const uint32_t cap = (uint32_t)kWarpCap;
        const uint32_t nl = !valid ? 0u : tot <= cap ? tot : S3 <= cap ? S3 : S2 <= cap ? S2 : S1 <= cap ? S1 : 0u;
        const uint16_t* es = list_of(r);
        for (uint32_t q = 0; q < nl; q++) {
            const uint32_t k = (q >= S1 ? 1u : 0u) + (q >= S2 ? 1u : 0u) + (q >= S3 ? 1u : 0u);
            uint32_t e;
            if (q < 8) {
                const uint32_t v = pick4(q >> 1, pre[r].x, pre[r].y, pre[r].z, pre[r].w);
                e = (v >> (16 * (q & 1u))) & 0xFFFFu;
            } else {
                e = ld_last2(es + q);
            }
            const uint32_t g = toff[r] + pick4(k, off0, off1, off2, off3) + q - pick4(k, 0u, S1, S2, S3);
            const uint32_t x = r0 + 2048u * k + (uint32_t)F::kSegLen * w + (e & kOffMask);
            put_escape(a, g, x - chunk_quot(a.cdiv, x) * a.cdiv.d, e >> F::kOffBits);
        }
        // Overflowed segments, rebuilt by the whole warp one at a time.
        for (uint32_t ov = __ballot_sync(0xFFFFFFFFu, ovk != 0); ov; ov &= ov - 1) {
            const uint32_t l = __ffs(ov) - 1;
            const uint32_t lk = __shfl_sync(0xFFFFFFFFu, ovk, l);
            const uint32_t lo0 = __shfl_sync(0xFFFFFFFFu, toff[r] + off0, l);
            const uint32_t lo1 = __shfl_sync(0xFFFFFFFFu, toff[r] + off1, l);
            const uint32_t lo2 = __shfl_sync(0xFFFFFFFFu, toff[r] + off2, l);
            const uint32_t lo3 = __shfl_sync(0xFFFFFFFFu, toff[r] + off3, l);
            if (!table) {  // warp-uniform
                uint32_t cbw[4];
                codebook_words(a.dcb, a.cbw, cbw);
#pragma unroll
                for (uint32_t ee = lane; ee < 256; ee += 32) isesc[ee] = !in_codebook(cbw, ee);
                __syncwarp();
                table = true;
            }
            for (uint32_t m = lk; m; m &= m - 1) {
                const uint32_t k = __ffs(m) - 1;
                rebuild_segment<F>(a, tile0 + (uint32_t)r * TPW + l / G, (l % G) + 8 * k,
                                   pick4(k, lo0, lo1, lo2, lo3), isesc);
            }
        }
        // chunk_off at the chunk starts of the tile.  When the chunk size is a
        // multiple of the segment length every chunk start is a segment start
        // (tiles and segments start at multiples of it), written by the lane
        // of that segment's list.
        if (seg_in_chunk) {
            if (!valid) continue;
            const uint32_t len = a.n - t0e < (uint32_t)kTileElems ? a.n - t0e : (uint32_t)kTileElems;
            const uint32_t q0 = chunk_quot32(a.cdiv, t0e);
#pragma unroll
            for (uint32_t k = 0; k < 4; k++) {
                const uint32_t ps = 2048u * k + (uint32_t)F::kSegLen * w;  // the segment's start
                const uint32_t x = r0 + ps, qx = chunk_quot(a.cdiv, x);  // x < d + kTileElems
                if (ps < len && x == qx * a.cdiv.d)
                    a.chunk_off[q0 + qx] = toff[r] + pick4(k, off0, off1, off2, off3);
            }
            continue;
        }
        // Other chunk sizes: the rank of each chunk start from the offset of
        // the segment holding it and that segment's entries before it.
        for (uint32_t t = 0; t < TPW; t++) {
            const uint32_t tl = tile0 + (uint32_t)r * TPW + t;
            if (tl >= num_tiles) break;  // warp-uniform
            const uint32_t u0 = tl * (uint32_t)kTileElems;
            const uint32_t ulen = a.n - u0 < (uint32_t)kTileElems ? a.n - u0 : (uint32_t)kTileElems;
            const uint32_t uq0 = chunk_quot32(a.cdiv, u0), ur0 = u0 - uq0 * a.cdiv.d;
            const uint16_t* uent = p.seg_ent + (size_t)tl * kEntries;
            const uint32_t qa = ur0 ? 1u : 0u, qb = chunk_quot(a.cdiv, ur0 + ulen - 1);
            for (uint32_t b0 = qa; b0 <= qb; b0 += 32) {
                const uint32_t q = b0 + lane;
                const bool ok = q <= qb;
                const uint32_t bl = ok ? q * a.cdiv.d - ur0 : 0u;  // tile-local chunk start
                const uint32_t sg = bl / (uint32_t)F::kSegLen, sw = sg & 7u, sk = sg >> 3;
                const uint32_t src = t * G + sw;  // the lane holding that segment's list
                const uint32_t so0 = __shfl_sync(0xFFFFFFFFu, toff[r] + off0, src);
                const uint32_t so1 = __shfl_sync(0xFFFFFFFFu, toff[r] + off1, src);
                const uint32_t so2 = __shfl_sync(0xFFFFFFFFu, toff[r] + off2, src);
                const uint32_t so3 = __shfl_sync(0xFFFFFFFFu, toff[r] + off3, src);
                const uint32_t sS1 = __shfl_sync(0xFFFFFFFFu, S1, src);
                const uint32_t sS2 = __shfl_sync(0xFFFFFFFFu, S2, src);
                const uint32_t sS3 = __shfl_sync(0xFFFFFFFFu, S3, src);
                const uint32_t stot = __shfl_sync(0xFFFFFFFFu, tot, src);
                if (ok) {
                    const uint32_t base = pick4(sk, 0u, sS1, sS2, sS3);
                    const uint32_t end = pick4(sk, sS1, sS2, sS3, stot);
                    const uint32_t lim = bl - sg * (uint32_t)F::kSegLen;
                    uint32_t rank = 0;
                    if (lim == 0) {
                    } else if (end <= (uint32_t)kWarpCap) {
                        const uint16_t* e = uent + sw * (uint32_t)kWarpCap;
                        for (uint32_t q2 = base; q2 < end; q2++) rank += (e[q2] & kOffMask) < lim;
                    } else {
                        uint32_t cbw[4];
                        codebook_words(a.dcb, a.cbw, cbw);
                        for (uint32_t l2 = sg * (uint32_t)F::kSegLen; l2 < bl; l2++)
                            rank += !in_codebook(cbw, F::exponent_at(a, u0 + l2));
                    }
                    a.chunk_off[uq0 + q] = pick4(sk, so0, so1, so2, so3) + rank;
                }
            }
        }
    }
}

template <class F>
cudaError_t launch_passes(const EncodeArgs& a, cudaStream_t s) {
    const MultiLayout L = multi_layout(a.n);
    MultiPtrs p;
    p.states = reinterpret_cast<uint64_t*>(a.ws + L.states);
    p.tile_tot = reinterpret_cast<uint32_t*>(a.ws + L.tile_tot);
    p.seg_cnt = reinterpret_cast<uint16_t*>(a.ws + L.seg_cnt);
    p.seg_ent = reinterpret_cast<uint16_t*>(a.ws + L.seg_ent);
    p.blk = reinterpret_cast<uint32_t*>(a.ws + L.sums);
    p.sup = p.blk + (kWsSumsBytes / 4 - kMaxSupers);  // fixed place
    p.nblocks = (uint32_t)L.nblocks;
    p.nsupers = (uint32_t)L.nsupers;
    const uint32_t tiles = a.num_tiles;
    constexpr size_t smem = dense_smem_bytes<F>();
    Wave wv;
    cudaError_t e = launch_wave<dense_kernel<F>>(kThreads, smem, wv);
    if (e != cudaSuccess) return e;
    const uint64_t wave = wv.ctas();
    // Stripes pay off once every CTA takes many tiles; with few, the draws
    // that find stripes dry at the end cost more than they save.
    p.striped = F::kStripes > 1 && tiles >= 64 * wave;
    dense_kernel<F><<<(uint32_t)(tiles < wave ? tiles : wave), kThreads, smem, s>>>(a, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // Placement takes F::kPlaceRounds rounds of tiles per warp, or one round
    // when that would leave fewer than two waves of CTAs (smaller tensors:
    // more, shorter warps; escape-heavy segments are rebuilt warp by warp).
    constexpr uint32_t kTilesPerRound = kWarps * (32 / F::kSegs);  // per CTA
    const uint64_t two_waves = 2ull * (uint64_t)(wv.sms > 0 ? wv.sms : 1) * 4;  // 4 CTAs per SM
    const uint32_t wide = kTilesPerRound * F::kPlaceRounds;
    // Programmatic dependent launches: placement CTAs start on the SMs the
    // dense pass frees at its end and wait there for it to complete (one KV
    // layer 51.9 -> 50.1 us, E5M2 at 2^31 elements 0.719 -> 0.717 ms).  Not
    // after a striped BF16 pass, which ended 2 us later with them waiting.
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    const bool early = !p.striped;
    auto launch = [&](auto kernel, uint32_t grid, uint32_t threads) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.stream = s;
        cfg.attrs = &attr;
        cfg.numAttrs = early ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kernel, a, p, tiles);
    };
    if constexpr (F::kListPlace) {  // a lane per warp list
        // Four tiles per warp in kPlaceRounds rounds, or two tiles per warp
        // when that would leave fewer than two waves of CTAs.
        const uint32_t wide2 = kWarps * 4 * F::kPlaceRounds;  // tiles per CTA
        e = (tiles + wide2 - 1) / wide2 >= two_waves
                ? launch(place_lists_kernel<F::kPlaceRounds, 4>, (tiles + wide2 - 1) / wide2, kThreads)
                : launch(place_lists_kernel<1, 2>, (tiles + 2 * kWarps - 1) / (2 * kWarps), kThreads);
    } else {
        e = (tiles + wide - 1) / wide >= two_waves
                ? launch(place_kernel<F, F::kPlaceRounds>, (tiles + wide - 1) / wide, kThreads)
                : launch(place_kernel<F, 1>, (tiles + kTilesPerRound - 1) / kTilesPerRound, kThreads);
    }
    if (e != cudaSuccess) return e;
    // The finishing CTA loads and sums the counters while placement runs and
    // waits for it only to write.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kFinishThreads);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, finish_kernel<F>, a, p);
}

}  // namespace

MultiLayout multi_layout(uint64_t n) {
    const uint64_t tiles = n ? (n + kTileElems - 1) / kTileElems : 1;
    MultiLayout L;
    L.sums = kWsHeaderBytes;  // fixed offset and size, whatever n is
    size_t off = kWsStatesOffset;
    L.states = off;
    off += align256(8 * tiles);
    L.tile_tot = off;
    off += align256(4 * tiles);
    L.seg_cnt = off;
    off += align256(2 * kSegsMax * tiles);
    L.seg_ent = off;
    off += align256(2 * kEntries * tiles);
    L.nblocks = (tiles + kBlockTiles - 1) / kBlockTiles;
    L.nsupers = (tiles + kSuperTiles - 1) / kSuperTiles;
    L.bytes = off;
    return L;
}

cudaError_t launch_encode_multi(const EncodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.num_tiles == 0) return cudaSuccess;
    return e5m2 ? launch_passes<E5m2Dense>(a, s) : launch_passes<Bf16Dense>(a, s);
}

}  // namespace splitzip
