// decode.cu -- SplitZip decode kernels for sm_103a (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README sections Codec API and FAQ; arXiv abstract on the paper
// index page): unpack the 4-bit codes, look each up in the 16-entry codebook,
// reassemble sign, exponent and mantissa, and put the raw exponent of every
// escape back at its position; the result is bitwise identical to the input.
//
// One launch, no communication between CTAs; the only CTA barrier follows the
// BF16 table build at the start.  Warps walk contiguous segments (1024 BF16
// or 2048 E5M2 elements) grid-stride:
//   - the dense streams (codes, sign+mantissa) of the next segment are loaded
//     into registers (BF16), or reach shared memory through a per-warp ring of
//     kDecodeStages slots filled by cp.async (E5M2: 16 bytes per lane per
//     copy, fully coalesced, kDecodeStages - 1 segments ahead);
//   - the segment's slice [lo, hi) of the escape stream is found two segments
//     ahead (chunk_off at a chunk start, else a warp-wide search of the
//     ascending positions inside the chunk) and its first 32 escapes are
//     loaded one segment ahead;
//   - each lane decodes its exponents in registers: BF16 two codes at a time
//     from a 256-entry shared-memory table of code bytes (built per CTA from
//     the codebook), E5M2 a code word (eight codes) at a time by byte permutes
//     of the 16 entries held in four registers;
//   - a segment with escapes parks its exponent words in shared memory, each
//     lane holding an escape overwrites that element's exponent byte, and the
//     words are read back (escapes beyond the first 32 of a segment are read
//     in further batches);
//   - SWAR reassembly and 16-byte stores.
// All escape metadata is clamped, so malformed streams cannot make the kernel
// read or write out of bounds.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

// Exponents of the eight codes of a code word (code k in nibble k of cw)
// from the codebook held in four words (cb0 = entries 0..3, ..., cb3 =
// entries 12..15): codes 0..3 into lo, codes 4..7 into hi.  Entries 0..7 and
// 8..15 are each one byte permute; a third permute in sign-replicate mode
// turns bit 3 of each code into a 0x00/0xFF byte mask that picks between the
// two.  The masks are formed once for all eight codes (a permute reads only
// the low 16 bits of its selector).
__device__ __forceinline__ void cb_lookup8(const uint32_t (&cb)[4], uint32_t cw, uint32_t& lo,
                                           uint32_t& hi) {
    const uint32_t sel = cw & 0x77777777u;
    const uint32_t t = cw & 0x88888888u;
    const uint32_t u = t | (t >> 3);  // nibble 9 where bit 3 is set, else 0
    const uint32_t sh = sel >> 16, uh = u >> 16;
    const uint32_t m0 = prmt(0x00008000u, 0u, u), m1 = prmt(0x00008000u, 0u, uh);
    lo = (prmt(cb[2], cb[3], sel) & m0) | (prmt(cb[0], cb[1], sel) & ~m0);
    hi = (prmt(cb[2], cb[3], sh) & m1) | (prmt(cb[0], cb[1], sh) & ~m1);
}

// Exponents of all 256 code bytes, two per entry (code byte c holds one
// element in its low nibble, the next in its high nibble): entry c is
// F::exp_byte(cb[c & 15]) | F::exp_byte(cb[c >> 4]) << 8.  One entry per
// thread of the CTA; all threads call it before any returns.
template <class F>
__device__ __forceinline__ void build_pairs(uint16_t* t, const uint32_t (&cbw)[4]) {
    static_assert(kThreads == 256, "one pair-table entry per thread");
    const uint32_t c = threadIdx.x;
    auto cb = [&](uint32_t k) {  // static word selects keep the parameters out of local memory
        const uint32_t q = k >> 2;
        const uint32_t w = q == 0 ? cbw[0] : q == 1 ? cbw[1] : q == 2 ? cbw[2] : cbw[3];
        return F::exp_byte((w >> (8 * (k & 3u))) & 0xFFu);
    };
    t[c] = (uint16_t)(cb(c & 15u) | (cb(c >> 4) << 8));
    __syncthreads();
}

// The codebook as each format's decode reads it: BF16 through the pair table
// in shared memory, E5M2 from four registers holding F::exp_byte of each entry
// (its segments already stream through shared memory, and more shared-memory
// loads measured slower there).
struct Luts {
    const uint16_t* pairs;
    uint32_t cb[4];
};

// Four exponent bytes of the four codes in c16 (two code bytes).
__device__ __forceinline__ uint32_t pair_lookup4(const uint16_t* t, uint32_t c16) {
    return __byte_perm(t[c16 & 0xFFu], t[(c16 >> 8) & 0xFFu], 0x5410);
}

// Four BF16 values from four sign+mantissa bytes and four exponent bytes.
__device__ __forceinline__ uint2 assemble_bf16(uint32_t sm, uint32_t ex) {
    const uint32_t lo = (sm & 0x7F7F7F7Fu) | ((ex << 7) & 0x80808080u);
    const uint32_t hi = (sm & 0x80808080u) | ((ex >> 1) & 0x7F7F7F7Fu);
    return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

// Four E5M2 values from four 3-bit fields (12 bits, field k at bits 3k) and
// four exponents already in place (bits 2..6 of each byte).
__device__ __forceinline__ uint32_t assemble_e5m2(uint32_t f12, uint32_t ex2) {
    const uint32_t t = (f12 & 0x3Fu) | ((f12 & 0xFC0u) << 10);
    const uint32_t f = (t & 0x00070007u) | ((t & 0x00380038u) << 5);
    return ((f << 5) & 0x80808080u) | ex2 | (f & 0x03030303u);
}

// First index j in [b, e) with pos[j] >= r, for positions in ascending order
// (any result in [b, e] otherwise).  All 32 lanes of a warp call it.
__device__ uint32_t lower_bound_warp(const uint16_t* pos, uint32_t b, uint32_t e, uint32_t r) {
    const uint32_t lane = threadIdx.x & 31;
    // b <= e throughout; probe indices are formed in 64 bits so that e near
    // 2^32 cannot wrap them.
    while (e - b > 32) {
        const uint32_t step = (e - b + 31) / 32;
        const uint64_t j = (uint64_t)b + (uint64_t)lane * step;
        const bool lt = j < e && pos[j] < r;
        const uint32_t k = __popc(__ballot_sync(0xFFFFFFFFu, lt));
        if (k == 0) return b;
        const uint32_t nb = b + (k - 1) * step + 1;  // <= e: lane k - 1 probed below e
        const uint64_t ne = (uint64_t)b + (uint64_t)k * step;
        b = nb;
        e = ne < e ? (uint32_t)ne : e;
    }
    const bool lt = lane < e - b && pos[b + lane] < r;
    return b + __popc(__ballot_sync(0xFFFFFFFFu, lt));
}

__device__ __forceinline__ uint32_t clamp_off(const DecodeArgs& a, uint32_t c) {
    const uint64_t v = a.chunk_off[c];
    return (uint32_t)(v < a.esc_count ? v : a.esc_count);
}

// Index of the first escape of element x or later (x <= n).  All lanes call it.
__device__ uint32_t escape_bound(const DecodeArgs& a, uint32_t x) {
    if (x >= a.n) return clamp_off(a, a.nchunks);
    const uint32_t c = chunk_quot32(a.cdiv, x);
    const uint32_t r = x - c * a.cdiv.d;
    const uint32_t b = clamp_off(a, c);
    if (r == 0) return b;
    const uint32_t e = max(b, clamp_off(a, c + 1));
    return lower_bound_warp(a.esc_pos, b, e, r);
}

// Chunk of escape entry j: the largest c in [ca, cb] with chunk_off[c] <= j
// (entries of empty chunks share offsets; the largest such c owns j).
__device__ __forceinline__ uint32_t chunk_of_entry(const DecodeArgs& a, uint32_t j, uint32_t ca,
                                                   uint32_t cb) {
    uint32_t lo = ca, hi = cb;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (clamp_off(a, mid) <= j) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// A batch of up to 32 escapes of one segment, one per lane: entry j, its
// position in chunk and raw exponent (j = 0xFFFFFFFF: no entry).
struct EscBatch {
    uint32_t j, pos, val;
};

__device__ __forceinline__ EscBatch load_batch(const DecodeArgs& a, uint32_t b, uint32_t hi) {
    const uint32_t lane = threadIdx.x & 31, j = b + lane;
    EscBatch e{0xFFFFFFFFu, 0u, 0u};
    if (b < hi && lane < hi - b) {  // not j < hi: b + lane may wrap
        e.j = j;
        e.pos = a.esc_pos[j];
        e.val = a.esc_val[j];
    }
    return e;
}

// Element index (relative to the segment start s0) of batch entry e, or
// 0xFFFFFFFF when the entry is absent or its metadata points outside the
// segment [s0, s1); chunks ca..cb overlap the segment.
__device__ __forceinline__ uint32_t batch_local(const DecodeArgs& a, const EscBatch& e,
                                                uint32_t s0, uint32_t s1, uint32_t ca,
                                                uint32_t cb) {
    if (e.j == 0xFFFFFFFFu) return 0xFFFFFFFFu;
    const uint32_t c = ca == cb ? ca : chunk_of_entry(a, e.j, ca, cb);
    const uint32_t x = c * a.cdiv.d + e.pos;
    return (e.pos < a.cdiv.d && x >= s0 && x < s1) ? x - s0 : 0xFFFFFFFFu;
}

// Puts the raw exponents of escapes [lo, hi) of segment [s0, s1) into the
// lane's exponent words: the words are parked in the warp's patch area, each
// lane holding an escape (the first 32 in eb, then further batches) overwrites
// its element's exponent byte, and the words are read back.  All lanes call it.
template <class F>
__device__ __forceinline__ void patch_escapes(const DecodeArgs& a, const EscBatch& eb, uint32_t lo,
                                              uint32_t hi, uint32_t s0, uint32_t s1, uint32_t* pex,
                                              typename F::Ex& ex) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t ca = chunk_quot32(a.cdiv, s0), cbk = chunk_quot32(a.cdiv, s1 - 1);
#pragma unroll
    for (int q = 0; q < F::kExWords; q++) pex[q * 32 + lane] = ex.e[q];
    __syncwarp();
    auto put = [&](const EscBatch& e) {
        const uint32_t local = batch_local(a, e, s0, s1, ca, cbk);
        if (local != 0xFFFFFFFFu) {
            uint32_t q, l, byte;
            F::locate(local, q, l, byte);
            reinterpret_cast<uint8_t*>(pex)[(q * 32 + l) * 4 + byte] = (uint8_t)F::exp_byte(e.val);
        }
    };
    put(eb);
    for (uint32_t b = lo; hi - b > 32;) {  // lo <= b < hi; no sum that could wrap
        b += 32;
        put(load_batch(a, b, hi));
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < F::kExWords; q++) ex.e[q] = pex[q * 32 + lane];
    __syncwarp();  // the next segment's patch area writes come after these reads
}

constexpr int kDecodeStages = 2;

// Shared memory of a decode CTA: the patch area ([warp][exponent word][lane])
// and, for a format decoded through the ring, the ring ([stage][warp][stage
// bytes]) in front of it.
template <class F>
constexpr size_t decode_smem_bytes() {
    return (F::kRing ? (size_t)kDecodeStages * kWarps * F::kStageBytes : 0) +
           (size_t)kWarps * F::kExWords * 32 * 4;
}

// Segment loop shared by both formats.  F provides:
//   kSeg, kStageBytes, kExWords   elements per segment, dense bytes per
//                                 segment (codes first, then sign+mantissa),
//                                 exponent words per lane
//   sm_offset(s0)                 byte offset of the segment's sign+mantissa
//   struct Dense / struct Ex      the lane's dense words / exponent words e[]
//   read(stage, lane)             -> Dense, from a staged full segment
//   load(a, s0, lane)             -> Dense, straight from global memory
//   decode(cb, d, ex)             exponents of the lane's elements
//   locate(local, q, l, byte)     exponent word q of lane l, byte, of element
//                                 `local` of the segment
//   store(a, s0, s1, lane, d, ex)
template <class F>
__device__ __forceinline__ void decode_segments(const DecodeArgs& a, uint8_t* smem,
                                                const Luts& lut) {
    constexpr int S = kDecodeStages;
    constexpr uint32_t kPieces = F::kStageBytes / 16;
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t warps = gridDim.x * kWarps;
    const uint32_t nseg = (uint32_t)(((uint64_t)a.n + F::kSeg - 1) / F::kSeg);  // n may be 2^32 - 1
    const uint32_t full_segs = a.n / (uint32_t)F::kSeg;
    uint8_t* ring = smem + (size_t)warp * F::kStageBytes;  // stage s at ring + s * kWarps * kStageBytes
    uint32_t* pex = reinterpret_cast<uint32_t*>(smem + (size_t)S * kWarps * F::kStageBytes) +
                    (size_t)warp * F::kExWords * 32;
    uint32_t seg = blockIdx.x * kWarps + warp;
    if (seg >= nseg) return;  // warp-uniform
    const uint64_t pol = l2_evict_first_policy();  // the streams are read once

    // Lanes copy the segment's dense bytes 16 at a time; a lane may read bytes
    // another lane copied, so every read of a stage follows this lane's wait
    // and a __syncwarp, and every refill follows a __syncwarp after the reads.
    auto fill = [&](uint32_t sg, int stage) {
        if (sg < full_segs) {
            const uint32_t s0 = sg * (uint32_t)F::kSeg;
            uint8_t* dst = ring + (size_t)stage * kWarps * F::kStageBytes;
#pragma unroll
            for (uint32_t q = 0; q < (kPieces + 31) / 32; q++) {
                const uint32_t piece = q * 32 + lane;
                if (piece < kPieces) {
                    const uint32_t off = piece * 16;
                    const uint8_t* src = off < (uint32_t)F::kCodeBytes
                                             ? a.codes + s0 / 2 + off
                                             : a.signman + F::sm_offset(s0) + (off - F::kCodeBytes);
                    cp_async16_hint(dst + off, src, pol);
                }
            }
        }
        cp_async_commit();  // one group per segment, empty when not staged
    };
    auto bounds = [&](uint32_t sg, uint32_t& lo, uint32_t& hi) {
        lo = hi = 0;
        if (sg >= nseg) return;  // warp-uniform
        const uint32_t s0 = sg * (uint32_t)F::kSeg;
        const uint32_t s1 = a.n - s0 < (uint32_t)F::kSeg ? a.n : s0 + F::kSeg;
        lo = escape_bound(a, s0);
        hi = max(lo, escape_bound(a, s1));
    };

#pragma unroll
    for (int st = 0; st < S; st++) fill(seg + st * warps, st);
    uint32_t lo, hi, lo1, hi1;
    bounds(seg, lo, hi);
    bounds(seg + warps, lo1, hi1);
    EscBatch eb = load_batch(a, lo, hi);
    int stage = 0;
    while (true) {
        const uint32_t s0 = seg * (uint32_t)F::kSeg;
        const uint32_t s1 = a.n - s0 < (uint32_t)F::kSeg ? a.n : s0 + F::kSeg;
        const uint32_t next = seg + warps;
        const bool more = next < nseg;
        uint32_t lo2, hi2;
        bounds(next + warps, lo2, hi2);  // two segments ahead
        typename F::Dense d;
        if (seg < full_segs) {
            cp_async_wait<S - 1>();  // this segment's group (the oldest pending) has landed
            __syncwarp();
            d = F::read(ring + (size_t)stage * kWarps * F::kStageBytes, lane);
        } else {
            d = F::load(a, s0, lane);
        }
        typename F::Ex ex;
        F::decode(lut, d, ex);
        if (lo < hi) patch_escapes<F>(a, eb, lo, hi, s0, s1, pex, ex);  // warp-uniform
        if (more) eb = load_batch(a, lo1, hi1);
        F::store(a, s0, s1, lane, d, ex);
        __syncwarp();  // every lane has read the stage before it is refilled
        fill(seg + S * warps, stage);
        stage = stage + 1 == S ? 0 : stage + 1;
        if (!more) break;
        seg = next;
        lo = lo1;
        hi = hi1;
        lo1 = lo2;
        hi1 = hi2;
    }
    cp_async_wait<0>();
}

// The same segment loop with the next segment's dense words prefetched into
// registers instead of a shared-memory ring (one segment ahead).
template <class F>
__device__ __forceinline__ void decode_segments_regs(const DecodeArgs& a, uint8_t* smem,
                                                     const Luts& lut) {
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t warps = gridDim.x * kWarps;
    const uint32_t nseg = (uint32_t)(((uint64_t)a.n + F::kSeg - 1) / F::kSeg);  // n may be 2^32 - 1
    uint32_t* pex = reinterpret_cast<uint32_t*>(smem) + (size_t)warp * F::kExWords * 32;
    uint32_t seg = blockIdx.x * kWarps + warp;
    if (seg >= nseg) return;  // warp-uniform
    auto bounds = [&](uint32_t sg, uint32_t& lo, uint32_t& hi) {
        const uint32_t s0 = sg * (uint32_t)F::kSeg;
        const uint32_t s1 = a.n - s0 < (uint32_t)F::kSeg ? a.n : s0 + F::kSeg;
        lo = escape_bound(a, s0);
        hi = max(lo, escape_bound(a, s1));
    };
    uint32_t lo, hi;
    bounds(seg, lo, hi);
    typename F::Dense d = F::load(a, seg * (uint32_t)F::kSeg, lane);
    EscBatch eb = load_batch(a, lo, hi);
    while (true) {
        const uint32_t s0 = seg * (uint32_t)F::kSeg;
        const uint32_t s1 = a.n - s0 < (uint32_t)F::kSeg ? a.n : s0 + F::kSeg;
        const uint32_t next = seg + warps;
        const bool more = next < nseg;
        typename F::Dense dn;
        uint32_t lo_n = 0, hi_n = 0;
        if (more) {
            dn = F::load(a, next * (uint32_t)F::kSeg, lane);
            bounds(next, lo_n, hi_n);
        }
        typename F::Ex ex;
        F::decode(lut, d, ex);
        if (lo < hi) patch_escapes<F>(a, eb, lo, hi, s0, s1, pex, ex);  // warp-uniform
        if (more) eb = load_batch(a, lo_n, hi_n);
        F::store(a, s0, s1, lane, d, ex);
        if (!more) break;
        seg = next;
        lo = lo_n;
        hi = hi_n;
        d = dn;
    }
}

// ------------------------------------------------------------------- BF16
//
// Segment [s0, s0 + 1024); lane l holds the groups of 8 at s0 + 256 k + 8 l
// (k < 4): the warp's reads cover 128 code bytes and 256 sign+mantissa bytes
// per group, each store 512 output bytes.  (kStageBytes sizes the ring a
// format decoded through one would need; BF16 prefetches into registers.)
struct Bf16Seg {
    // Dense words prefetched into registers one segment ahead: at 2^31
    // elements this measured 1.22 ms against 1.40 ms through the ring.
    static constexpr bool kRing = false;
    static constexpr int kSeg = 1024;
    static constexpr int kGroups = 4;
    static constexpr int kCodeBytes = kSeg / 2;
    static constexpr int kStageBytes = kCodeBytes + kSeg;
    static constexpr int kExWords = 2 * kGroups;
    struct Dense {
        uint32_t code[kGroups];
        uint2 sm[kGroups];
    };
    struct Ex {
        uint32_t e[kExWords];  // word 2k + h: elements 4h..4h+3 of group k
    };
    static __device__ __forceinline__ Dense load(const DecodeArgs& a, uint32_t s0, uint32_t lane) {
        Dense d;
        const uint32_t s1 = a.n - s0 < (uint32_t)kSeg ? a.n : s0 + kSeg;
        const bool full = s1 - s0 == (uint32_t)kSeg;
        // (Per-segment 64-bit bases with constant group offsets cut this kernel's
        // instructions by 15% but ran 3% slower at 2^31 elements; kept as is.)
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = s0 + 256 * k + 8 * lane;
            if (full || (uint64_t)i + 8 <= s1) {
                d.code[k] = ld_stream4(a.codes + i / 2);
                d.sm[k] = ld_stream8(a.signman + i);
            } else {
                d.code[k] = 0;
                d.sm[k] = make_uint2(0, 0);
                if (i < s1) {
                    const uint32_t rem = s1 - i;
                    for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                        d.code[k] |= (uint32_t)a.codes[i / 2 + j] << (8 * j);
                    for (uint32_t j = 0; j < rem; j++) {
                        const uint32_t b = (uint32_t)a.signman[i + j] << (8 * (j & 3));
                        if (j < 4) d.sm[k].x |= b; else d.sm[k].y |= b;
                    }
                }
            }
        }
        return d;
    }
    static constexpr bool kPairs = true;  // exponents from the pair table
    static constexpr int kMinBlocks = 4;  // resident CTAs per SM: 64 registers
    static __device__ __forceinline__ uint32_t exp_byte(uint32_t e) { return e; }
    static __device__ __forceinline__ void decode(const Luts& lut, const Dense& d, Ex& ex) {
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            ex.e[2 * k] = pair_lookup4(lut.pairs, d.code[k] & 0xFFFFu);
            ex.e[2 * k + 1] = pair_lookup4(lut.pairs, d.code[k] >> 16);
        }
    }
    static __device__ __forceinline__ void locate(uint32_t local, uint32_t& q, uint32_t& l,
                                                  uint32_t& byte) {
        q = 2 * (local >> 8) + ((local >> 2) & 1u);
        l = (local >> 3) & 31u;
        byte = local & 3u;
    }
    static __device__ __forceinline__ void store(const DecodeArgs& a, uint32_t s0, uint32_t s1,
                                                 uint32_t lane, const Dense& d, const Ex& ex) {
        const bool full = s1 - s0 == (uint32_t)kSeg;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = s0 + 256 * k + 8 * lane;
            if (!full && i >= s1) continue;
            const uint2 o0 = assemble_bf16(d.sm[k].x, ex.e[2 * k]);
            const uint2 o1 = assemble_bf16(d.sm[k].y, ex.e[2 * k + 1]);
            if (full || s1 - i >= 8) {  // i < s1 here
                st_stream16(a.y + 2ull * i, make_uint4(o0.x, o0.y, o1.x, o1.y));
            } else {
                const uint32_t w[4] = {o0.x, o0.y, o1.x, o1.y};
                uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + i;
                for (uint32_t j = 0; j < s1 - i; j++) yp[j] = (uint16_t)(w[j >> 1] >> (16 * (j & 1)));
            }
        }
    }
};

// ------------------------------------------------------------------- E5M2
//
// Segment [s0, s0 + 2048); lane l holds the groups of 32 at s0 + 1024 k + 32 l
// (k < 2): 16 code bytes and 12 bytes of packed 3-bit fields in, 32 output
// bytes out per group.  Stage layout: the segment's 1024 code bytes, then its
// 768 bytes of 3-bit fields.
struct E5m2Seg {
    // Dense words through the two-stage ring: at 2^31 elements this measured
    // 0.94 ms against 0.96 ms with register prefetch.
    static constexpr bool kRing = true;
    static constexpr int kSeg = 2048;
    static constexpr int kGroups = 2;
    static constexpr int kCodeBytes = kSeg / 2;
    static constexpr int kStageBytes = kCodeBytes + kSeg * 3 / 8;
    static constexpr int kExWords = 8 * kGroups;
    struct Dense {
        uint4 code[kGroups];
        uint32_t smw[kGroups][3];
    };
    struct Ex {
        uint32_t e[kExWords];  // word 8k + m: elements 4m..4m+3 of group k
    };
    static __device__ __forceinline__ uint32_t sm_offset(uint32_t s0) { return s0 / 8 * 3; }
    static __device__ __forceinline__ Dense read(const uint8_t* stage, uint32_t lane) {
        Dense d;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            d.code[k] = *reinterpret_cast<const uint4*>(stage + 512 * k + 16 * lane);
            const uint32_t* w =
                reinterpret_cast<const uint32_t*>(stage + kCodeBytes + 384 * k + 12 * lane);
            d.smw[k][0] = w[0];
            d.smw[k][1] = w[1];
            d.smw[k][2] = w[2];
        }
        return d;
    }
    static __device__ __forceinline__ Dense load(const DecodeArgs& a, uint32_t s0, uint32_t lane) {
        Dense d;
        const uint32_t s1 = a.n - s0 < (uint32_t)kSeg ? a.n : s0 + kSeg;
        const bool full = s1 - s0 == (uint32_t)kSeg;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = s0 + 1024 * k + 32 * lane;
            const uint8_t* smp = a.signman + (uint64_t)(i / 32) * 12;
            if (full || (uint64_t)i + 32 <= s1) {
                d.code[k] = ld_stream16(a.codes + i / 2);
                d.smw[k][0] = ld_stream4(smp);
                d.smw[k][1] = ld_stream4(smp + 4);
                d.smw[k][2] = ld_stream4(smp + 8);
            } else {
                uint32_t cw[4] = {0, 0, 0, 0};
                d.smw[k][0] = d.smw[k][1] = d.smw[k][2] = 0;
                if (i < s1) {
                    const uint32_t rem = s1 - i;
                    for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                        cw[j >> 2] |= (uint32_t)a.codes[i / 2 + j] << (8 * (j & 3));
                    for (uint32_t j = 0; j < (3 * rem + 7) / 8; j++)
                        d.smw[k][j >> 2] |= (uint32_t)smp[j] << (8 * (j & 3));
                }
                d.code[k] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            }
        }
        return d;
    }
    // Exponents enter the words already shifted to bits 2..6 of the byte.
    static constexpr bool kPairs = false;  // exponents from the codebook registers
    static constexpr int kMinBlocks = 5;  // resident CTAs per SM: 48 registers, 1.4% faster than 4
    static __device__ __forceinline__ uint32_t exp_byte(uint32_t e) { return (e << 2) & 0x7Cu; }
    static __device__ __forceinline__ void decode(const Luts& lut, const Dense& d, Ex& ex) {
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t cw[4] = {d.code[k].x, d.code[k].y, d.code[k].z, d.code[k].w};
#pragma unroll
            for (int i = 0; i < 4; i++) cb_lookup8(lut.cb, cw[i], ex.e[8 * k + 2 * i], ex.e[8 * k + 2 * i + 1]);
        }
    }
    static __device__ __forceinline__ void locate(uint32_t local, uint32_t& q, uint32_t& l,
                                                  uint32_t& byte) {
        q = 8 * (local >> 10) + ((local >> 2) & 7u);
        l = (local >> 5) & 31u;
        byte = local & 3u;
    }
    static __device__ __forceinline__ void store(const DecodeArgs& a, uint32_t s0, uint32_t s1,
                                                 uint32_t lane, const Dense& d, const Ex& ex) {
        const bool full = s1 - s0 == (uint32_t)kSeg;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = s0 + 1024 * k + 32 * lane;
            if (!full && i >= s1) continue;
            const uint32_t w0 = d.smw[k][0], w1 = d.smw[k][1], w2 = d.smw[k][2];
            const uint32_t f12[8] = {
                w0 & 0xFFFu, (w0 >> 12) & 0xFFFu, __funnelshift_r(w0, w1, 24) & 0xFFFu,
                (w1 >> 4) & 0xFFFu, (w1 >> 16) & 0xFFFu, __funnelshift_r(w1, w2, 28) & 0xFFFu,
                (w2 >> 8) & 0xFFFu, w2 >> 20};
            uint32_t out[8];
#pragma unroll
            for (int m = 0; m < 8; m++) out[m] = assemble_e5m2(f12[m], ex.e[8 * k + m]);
            if (full) {
                uint8_t* yb = a.y + (s0 + 32 * lane) + 1024 * k;
                st_stream16(yb, make_uint4(out[0], out[1], out[2], out[3]));
                st_stream16(yb + 16, make_uint4(out[4], out[5], out[6], out[7]));
            } else if (s1 - i >= 32) {  // i < s1 here
                st_stream16(a.y + i, make_uint4(out[0], out[1], out[2], out[3]));
                st_stream16(a.y + i + 16, make_uint4(out[4], out[5], out[6], out[7]));
            } else {
                for (uint32_t j = 0; j < s1 - i; j++) a.y[i + j] = (uint8_t)(out[j >> 2] >> (8 * (j & 3)));
            }
        }
    }
};

template <class F>
__global__ void __launch_bounds__(kThreads, F::kMinBlocks) decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint16_t pairs[256];
    Luts lut;
    lut.pairs = pairs;
    uint32_t cbw[4];
    codebook_words(a.dcb, a.cbw, cbw);
    if constexpr (F::kPairs) build_pairs<F>(pairs, cbw);
#pragma unroll
    for (int q = 0; q < 4; q++) {  // F::exp_byte of each byte of the codebook words
        const uint32_t w = cbw[q];
        lut.cb[q] = F::exp_byte(w & 0xFFu) | (F::exp_byte((w >> 8) & 0xFFu) << 8) |
                    (F::exp_byte((w >> 16) & 0xFFu) << 16) | (F::exp_byte(w >> 24) << 24);
    }
    if constexpr (F::kRing) decode_segments<F>(a, smem, lut);
    else decode_segments_regs<F>(a, smem, lut);
}

template <class F>
cudaError_t launch_segments(const DecodeArgs& a, cudaStream_t s) {
    constexpr size_t smem = decode_smem_bytes<F>();
    Wave wv;
    const cudaError_t e = launch_wave<decode_kernel<F>>(kThreads, smem, wv);
    if (e != cudaSuccess) return e;
    const uint64_t nseg = ((uint64_t)a.n + F::kSeg - 1) / F::kSeg;
    const uint64_t ctas = (nseg + kWarps - 1) / kWarps;
    const uint64_t wave = wv.ctas();
    decode_kernel<F><<<(uint32_t)(ctas < wave ? ctas : wave), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int decode_tile_elems(bool e5m2) { return (e5m2 ? E5m2Seg::kSeg : Bf16Seg::kSeg) * kWarps; }

cudaError_t launch_decode(const DecodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    return e5m2 ? launch_segments<E5m2Seg>(a, s) : launch_segments<Bf16Seg>(a, s);
}

}  // namespace splitzip
