// decode.cu -- SplitZip decode kernels for sm_103a (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README sections Codec API and FAQ; arXiv abstract on the paper
// index page): unpack the 4-bit codes, look each up in the 16-entry codebook,
// reassemble sign, exponent and mantissa, and put the raw exponent of every
// escape back at its position; the result is bitwise identical to the input.
//
// One launch, no communication between CTAs.  Warps walk contiguous segments
// (1024 BF16 or 2048 E5M2 elements) grid-stride:
//   - the dense streams (codes, sign+mantissa) of the next segment are loaded
//     into registers (BF16), or reach shared memory through a per-warp ring
//     filled by cp.async (E5M2: 16 bytes per lane per copy, coalesced);
//   - the segment's slice [lo, hi) of the escape stream is found ahead of the
//     segment (chunk_off at a chunk start, else a warp-wide search of the
//     ascending positions inside the chunk) and its first 32 escapes are
//     loaded one segment ahead;
//   - BF16: each lane decodes its exponents two codes at a time from a
//     256-entry shared-memory table of code bytes (built per CTA from the
//     codebook); a segment with escapes parks its exponent words in shared
//     memory, each lane holding an escape overwrites that element's exponent
//     byte, and the words are read back; SWAR reassembly and 16-byte stores;
//   - E5M2: a code word (eight codes) at a time by byte permutes of the 16
//     entries held in four registers, fields spread by shifts and selects,
//     16-byte stores; each escape is then written over its output byte.
// All escape metadata is clamped, so malformed streams cannot make the kernel
// read or write out of bounds.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

// Exponents of the eight codes of a code word (code k in nibble k of cw)
// from the codebook held in four words (cb[0] = entries 0..3, ..., cb[3] =
// entries 12..15), every entry already shifted into the E5M2 exponent field
// (bits 2..6, so bit 7 of each entry is 0).  One byte permute reads entries
// 0..7 with the codes as selectors: a code of 8 or more has selector bit 3
// set, which makes the permute replicate bit 7 of the chosen entry -- 0.  A
// second permute reads entries 8..15 with selector bit 3 flipped, so codes
// below 8 give 0 there.  The exponent bytes of codes 0..3 are lo_a | lo_b,
// of codes 4..7 hi_a | hi_b (a permute reads the low 16 bits of its
// selector).
__device__ __forceinline__ void cb_lookup8(const uint32_t (&cb)[4], uint32_t cw, uint32_t& lo_a,
                                           uint32_t& lo_b, uint32_t& hi_a, uint32_t& hi_b) {
    const uint32_t cx = cw ^ 0x88888888u;
    lo_a = prmt(cb[0], cb[1], cw);
    lo_b = prmt(cb[2], cb[3], cx);
    hi_a = prmt(cb[0], cb[1], cw >> 16);
    hi_b = prmt(cb[2], cb[3], cx >> 16);
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

// The codebook as the BF16 decode reads it: through the pair table in shared
// memory.
struct Luts {
    const uint16_t* pairs;
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

// Shared memory of a BF16 decode CTA: the patch area ([warp][exponent
// word][lane]).
template <class F>
constexpr size_t decode_smem_bytes() {
    return (size_t)kWarps * F::kExWords * 32 * 4;
}

// Segment loop of the BF16 decode.  F provides:
//   kSeg, kExWords                elements per segment, exponent words per lane
//   struct Dense / struct Ex      the lane's dense words / exponent words e[]
//   load(a, s0, lane)             -> Dense, straight from global memory
//   decode(lut, d, ex)            exponents of the lane's elements
//   locate(local, q, l, byte)     exponent word q of lane l, byte, of element
//                                 `local` of the segment
//   store(a, s0, s1, lane, d, ex)
// The next segment's dense words are prefetched into registers (one segment
// ahead), its escape slice found and its first 32 escapes loaded one ahead.
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
    static constexpr uint32_t kSegsPerWarp = 27;  // segments a warp walks (sets the grid)
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
// Segment [s0, s0 + 2048) per warp; lane l holds the groups of 32 elements at
// s0 + 1024 k + 32 l (k < 2): 16 code bytes and 12 bytes of packed 3-bit
// fields in, 32 output bytes out per group.  The dense bytes of a segment
// (its 1024 code bytes, then its 768 field bytes) reach shared memory through
// a per-warp ring of kE5Stages slots filled by cp.async, 16 bytes per lane
// per copy (coalesced, evict-first in L2), kE5Stages - 1 segments ahead.
// Each output word is assembled in registers and stored; the escapes of the
// segment are then written over their elements as single bytes (sign and
// mantissa from the staged fields, the raw exponent from the escape stream),
// ordered after the word stores by a __syncwarp.
namespace e5 {

constexpr int kSeg = 2048;
constexpr int kCodeBytes = kSeg / 2;
constexpr int kFieldBytes = kSeg * 3 / 8;
constexpr int kStageBytes = kCodeBytes + kFieldBytes;  // 1792
constexpr int kPieces = kStageBytes / 16;              // 112 copies of 16 bytes
constexpr int kStages = 2;
constexpr int kMinBlocks = 6;      // resident CTAs per SM
constexpr uint32_t kSegsPerWarp = 4;  // segments a warp walks (sets the grid)

// a where m is set, b elsewhere (one LOP3).
__device__ __forceinline__ uint32_t sel(uint32_t a, uint32_t b, uint32_t m) {
    return (a & m) | (b & ~m);
}

// The eight output words of a group: codes c (16 bytes), fields w0..w2
// (12 bytes, field j at bits 3j..3j+2 of the 96-bit little-endian stream).
// Fields are spread eight at a time: a 24-bit run of eight fields is split
// into two 12-bit halves 16 bits apart, each half into two 6-bit pairs 8 bits
// apart; the even and odd fields of the pairs are masked out and interleaved
// byte by byte with permutes.  Multiplying a byte holding sign << 2 | mantissa
// by 33 adds a copy 5 bits up, which puts the sign at bit 7 (no carry between
// bytes: 7 * 33 < 256); masking keeps bits 7, 1 and 0, and the exponents
// (bits 2..6) are OR-ed in.
__device__ __forceinline__ void group(const uint32_t (&cb)[4], const uint4& c, uint32_t w0,
                                      uint32_t w1, uint32_t w2, uint32_t (&out)[8]) {
    uint32_t a[8], b[8];
    cb_lookup8(cb, c.x, a[0], b[0], a[1], b[1]);
    cb_lookup8(cb, c.y, a[2], b[2], a[3], b[3]);
    cb_lookup8(cb, c.z, a[4], b[4], a[5], b[5]);
    cb_lookup8(cb, c.w, a[6], b[6], a[7], b[7]);
    const uint32_t v[4] = {w0, __funnelshift_r(w0, w1, 24), __funnelshift_r(w1, w2, 16), w2 >> 8};
#pragma unroll
    for (int p = 0; p < 4; p++) {  // fields 8p..8p+7 (bits above the 24th are ignored)
        const uint32_t h = sel(v[p] << 4, v[p], 0xFFFF0000u);  // fields 4..7 at bits 16..27
        const uint32_t q = sel(h << 2, h, 0xFF00FF00u);        // pair k at bits 8k..8k+5
        const uint32_t ev = q & 0x07070707u, od = (q >> 3) & 0x07070707u;
        const uint32_t x0 = __byte_perm(ev, od, 0x5140), x1 = __byte_perm(ev, od, 0x7362);
        out[2 * p] = ((x0 * 33u) & 0x83838383u) | a[2 * p] | b[2 * p];
        out[2 * p + 1] = ((x1 * 33u) & 0x83838383u) | a[2 * p + 1] | b[2 * p + 1];
    }
}

// The 3-bit field of element j of a field stream f of `bytes` bytes.
__device__ __forceinline__ uint32_t field_at(const uint8_t* f, uint64_t j) {
    const uint64_t bit = 3 * j;
    const uint32_t sh = (uint32_t)(bit & 7);
    uint32_t v = f[bit >> 3];
    if (sh > 5) v |= (uint32_t)f[(bit >> 3) + 1] << 8;  // the field runs into the next byte
    return (v >> sh) & 7u;
}

// Escape slice [lo, hi) of a segment.  When both ends of the segment are
// chunk starts the two chunk_off loads are returned unclamped, to be clamped
// (finish) an iteration later, when their values have arrived; otherwise the
// slice is searched (and clamped) at once.
struct Slice {
    uint32_t lo, hi;
};
__device__ __forceinline__ Slice slice_issue(const DecodeArgs& a, uint32_t sg, uint32_t nseg) {
    Slice b{0u, 0u};
    if (sg >= nseg) return b;  // warp-uniform
    const uint32_t s0 = sg * (uint32_t)kSeg;
    const uint32_t s1 = a.n - s0 < (uint32_t)kSeg ? a.n : s0 + kSeg;
    const uint32_t c0 = chunk_quot32(a.cdiv, s0);
    const uint32_t c1 = s1 >= a.n ? a.nchunks : chunk_quot32(a.cdiv, s1);
    if (s0 == c0 * a.cdiv.d && (s1 >= a.n || s1 == c1 * a.cdiv.d)) {
        b.lo = a.chunk_off[c0];
        b.hi = a.chunk_off[c1];
    } else {
        b.lo = escape_bound(a, s0);
        b.hi = max(b.lo, escape_bound(a, s1));
    }
    return b;
}
__device__ __forceinline__ Slice slice_finish(const DecodeArgs& a, Slice b) {
    const uint32_t lo = (uint64_t)b.lo < a.esc_count ? b.lo : (uint32_t)a.esc_count;
    const uint32_t hi = (uint64_t)b.hi < a.esc_count ? b.hi : (uint32_t)a.esc_count;
    return Slice{lo, max(lo, hi)};
}

// Up to 32 escapes of a segment, one per lane, as loaded one segment ahead:
// pv = position in chunk | raw exponent << 16 (0xFFFFFFFF: no entry), and the
// escape offset of the chunk that starts inside the segment (for a segment
// that overlaps two chunks; the entries from there on belong to the second).
struct Batch {
    uint32_t pv, mid;
};
__device__ __forceinline__ Batch batch_issue(const DecodeArgs& a, uint32_t b, uint32_t hi,
                                             uint32_t s0, uint32_t s1) {
    const uint32_t lane = threadIdx.x & 31;
    Batch e{0xFFFFFFFFu, 0u};
    if (b < hi && lane < hi - b) {  // not b + lane < hi: the sum may wrap
        e.pv = (uint32_t)a.esc_pos[b + lane] | ((uint32_t)a.esc_val[b + lane] << 16);
        const uint32_t ca = chunk_quot32(a.cdiv, s0), cbk = chunk_quot32(a.cdiv, s1 - 1);
        if (cbk == ca + 1) e.mid = a.chunk_off[cbk];
    }
    return e;
}

// Segment-relative index of batch entry j = b + lane (its values in e), or
// 0xFFFFFFFF when absent or when its metadata points outside [s0, s1).
__device__ __forceinline__ uint32_t batch_index(const DecodeArgs& a, const Batch& e, uint32_t j,
                                                uint32_t s0, uint32_t s1) {
    if (e.pv == 0xFFFFFFFFu) return 0xFFFFFFFFu;
    const uint32_t ca = chunk_quot32(a.cdiv, s0), cbk = chunk_quot32(a.cdiv, s1 - 1);
    const uint32_t c = ca == cbk ? ca
                       : cbk == ca + 1 ? (j >= e.mid ? cbk : ca)
                                       : chunk_of_entry(a, j, ca, cbk);
    const uint32_t pos = e.pv & 0xFFFFu;
    const uint32_t x = c * a.cdiv.d + pos;
    return (pos < a.cdiv.d && x >= s0 && x < s1) ? x - s0 : 0xFFFFFFFFu;
}

// Writes the escapes [lo, hi) of segment [s0, s1) over their output bytes
// (the first 32 in eb, then further batches).  fields: the segment's staged
// field bytes, or null to read them from the field stream.
__device__ __forceinline__ void patch(const DecodeArgs& a, const Batch& eb, uint32_t lo,
                                      uint32_t hi, uint32_t s0, uint32_t s1, const uint8_t* fields) {
    const uint32_t lane = threadIdx.x & 31;
    auto put = [&](const Batch& e, uint32_t b) {
        const uint32_t local = batch_index(a, e, b + lane, s0, s1);
        if (local != 0xFFFFFFFFu) {
            const uint32_t f = fields ? field_at(fields, local) : field_at(a.signman, (uint64_t)s0 + local);
            a.y[s0 + local] = (uint8_t)(((f & 4u) << 5) | (((e.pv >> 16) << 2) & 0x7Cu) | (f & 3u));
        }
    };
    put(eb, lo);
    for (uint32_t b = lo; hi - b > 32;) {  // lo <= b < hi; no sum that could wrap
        b += 32;
        put(batch_issue(a, b, hi, s0, s1), b);
    }
}

// The dense words of group k of a segment not staged (the last, partial one),
// straight from global memory; bytes past s1 read as 0.
__device__ __forceinline__ void load_partial(const DecodeArgs& a, uint32_t s0, uint32_t s1,
                                             uint32_t i, uint4& c, uint32_t (&w)[3]) {
    (void)s0;
    uint32_t cw[4] = {0, 0, 0, 0};
    w[0] = w[1] = w[2] = 0;
    const uint8_t* smp = a.signman + (uint64_t)(i / 32) * 12;
    if (i < s1) {
        const uint32_t rem = s1 - i < 32 ? s1 - i : 32;
        const uint32_t nc = (rem + 1) / 2, ns = (3 * rem + 7) / 8;
#pragma unroll
        for (int j = 0; j < 16; j++)
            if ((uint32_t)j < nc) cw[j >> 2] |= (uint32_t)a.codes[i / 2 + j] << (8 * (j & 3));
#pragma unroll
        for (int j = 0; j < 12; j++)
            if ((uint32_t)j < ns) w[j >> 2] |= (uint32_t)smp[j] << (8 * (j & 3));
    }
    c = make_uint4(cw[0], cw[1], cw[2], cw[3]);
}

}  // namespace e5

__global__ void __launch_bounds__(kThreads, e5::kMinBlocks) decode_e5m2_kernel(const DecodeArgs a) {
    using namespace e5;
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t cb[4];  // the codebook, each entry shifted into the exponent field
    {
        uint32_t cbw[4];
        codebook_words(a.dcb, a.cbw, cbw);
#pragma unroll
        for (int q = 0; q < 4; q++) cb[q] = (cbw[q] << 2) & 0x7C7C7C7Cu;
    }
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t warps = gridDim.x * kWarps;
    const uint32_t nseg = (uint32_t)(((uint64_t)a.n + kSeg - 1) / kSeg);  // n may be 2^32 - 1
    const uint32_t full_segs = a.n / (uint32_t)kSeg;
    uint8_t* ring = smem + (size_t)warp * kStageBytes;  // stage st at ring + st * kWarps * kStageBytes
    uint32_t seg = blockIdx.x * kWarps + warp;
    if (seg >= nseg) return;  // warp-uniform
    const uint64_t pol = l2_evict_first_policy();  // the streams are read once

    // Lanes copy the segment's dense bytes 16 at a time; a lane reads bytes
    // other lanes copied, so every read of a stage follows this lane's wait
    // and a __syncwarp, and every refill follows a __syncwarp after the reads.
    auto fill = [&](uint32_t sg, int st) {
        if (sg < full_segs) {
            const uint32_t s0 = sg * (uint32_t)kSeg;
            uint8_t* dst = ring + (size_t)st * kWarps * kStageBytes;
#pragma unroll
            for (uint32_t q = 0; q < (kPieces + 31) / 32; q++) {
                const uint32_t piece = q * 32 + lane;
                if (piece < (uint32_t)kPieces) {
                    const uint32_t off = piece * 16;
                    const uint8_t* src = off < (uint32_t)kCodeBytes
                                             ? a.codes + s0 / 2 + off
                                             : a.signman + (uint64_t)(s0 / 8) * 3 + (off - kCodeBytes);
                    cp_async16_hint(dst + off, src, pol);
                }
            }
        }
        cp_async_commit();  // one group per segment, empty when not staged
    };

#pragma unroll
    for (int st = 0; st < kStages; st++) fill(seg + st * warps, st);
    Slice cur = slice_finish(a, slice_issue(a, seg, nseg));
    Slice nxt = slice_issue(a, seg + warps, nseg);  // finished an iteration later
    Batch eb = batch_issue(a, cur.lo, cur.hi, seg * (uint32_t)kSeg,
                           a.n - seg * (uint32_t)kSeg < (uint32_t)kSeg ? a.n : seg * (uint32_t)kSeg + kSeg);
    int stage = 0;
    while (true) {
        const uint32_t s0 = seg * (uint32_t)kSeg;
        const uint32_t s1 = a.n - s0 < (uint32_t)kSeg ? a.n : s0 + kSeg;
        const uint32_t next = seg + warps;
        const bool more = next < nseg;
        const Slice nxt2 = slice_issue(a, next + warps, nseg);  // two segments ahead
        nxt = slice_finish(a, nxt);
        Batch ebn{0xFFFFFFFFu, 0u};
        if (more) {
            const uint32_t n0 = next * (uint32_t)kSeg;
            ebn = batch_issue(a, nxt.lo, nxt.hi, n0, a.n - n0 < (uint32_t)kSeg ? a.n : n0 + kSeg);
        }
        const uint8_t* st_base = ring + (size_t)stage * kWarps * kStageBytes;
        const bool staged = seg < full_segs;  // warp-uniform
        if (staged) {
            cp_async_wait<kStages - 1>();  // this segment's group (the oldest pending) has landed
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const uint4 c = *reinterpret_cast<const uint4*>(st_base + 512 * k + 16 * lane);
                const uint32_t* w =
                    reinterpret_cast<const uint32_t*>(st_base + kCodeBytes + 384 * k + 12 * lane);
                uint32_t out[8];
                group(cb, c, w[0], w[1], w[2], out);
                uint8_t* yb = a.y + (s0 + 32 * lane) + 1024 * k;
                st_stream16(yb, make_uint4(out[0], out[1], out[2], out[3]));
                st_stream16(yb + 16, make_uint4(out[4], out[5], out[6], out[7]));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const uint32_t i = s0 + 1024 * k + 32 * lane;
                uint4 c;
                uint32_t w[3];
                load_partial(a, s0, s1, i, c, w);
                uint32_t out[8];
                group(cb, c, w[0], w[1], w[2], out);
                if (i < s1) {
                    if (s1 - i >= 32) {
                        st_stream16(a.y + i, make_uint4(out[0], out[1], out[2], out[3]));
                        st_stream16(a.y + i + 16, make_uint4(out[4], out[5], out[6], out[7]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            if ((uint32_t)j < s1 - i) a.y[i + j] = (uint8_t)(out[j >> 2] >> (8 * (j & 3)));
                    }
                }
            }
        }
        if (cur.lo < cur.hi) {  // warp-uniform
            __syncwarp();  // the word stores of every lane come before the escape bytes
            patch(a, eb, cur.lo, cur.hi, s0, s1, staged ? st_base + kCodeBytes : nullptr);
        }
        __syncwarp();  // every lane has read the stage before it is refilled
        fill(seg + kStages * warps, stage);
        stage = stage + 1 == kStages ? 0 : stage + 1;
        if (!more) break;
        seg = next;
        cur = nxt;
        nxt = nxt2;
        eb = ebn;
    }
    cp_async_wait<0>();
}

template <class F>
__global__ void __launch_bounds__(kThreads, F::kMinBlocks) decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint16_t pairs[256];
    Luts lut;
    lut.pairs = pairs;
    uint32_t cbw[4];
    codebook_words(a.dcb, a.cbw, cbw);
    build_pairs<F>(pairs, cbw);
    decode_segments_regs<F>(a, smem, lut);
}

// Grid of kernel K over the segments: enough CTAs that each warp walks about
// segs_per_warp segments grid-stride (at least four resident waves, at most one
// CTA per kWarps segments).  With a single resident wave, CTAs of equal shares
// finish far apart and the SMs of the early ones idle at the end; with several
// waves of shorter shares the hardware starts the later CTAs on whichever SMs
// free up first.  Measured at 2^31 elements: BF16 1.217 ms with one wave,
// 1.138 ms at 27 segments per warp; E5M2 0.764 ms against 0.643 ms at 4 (2 was
// slower: 0.725 ms; one CTA per 8 segments slower still).  Smaller tensors
// still get four waves (2^27 elements: BF16 79.9 -> 77.8 us, E5M2 49.2 ->
// 47.1 us against one wave).
template <auto K>
cudaError_t launch_segment_wave(const DecodeArgs& a, uint32_t seg_elems, size_t smem,
                                uint32_t segs_per_warp, cudaStream_t s) {
    Wave wv;
    const cudaError_t e = launch_wave<K>(kThreads, smem, wv);
    if (e != cudaSuccess) return e;
    const uint64_t nseg = ((uint64_t)a.n + seg_elems - 1) / seg_elems;
    const uint64_t ctas = (nseg + kWarps - 1) / kWarps;
    uint64_t grid = (nseg + (uint64_t)kWarps * segs_per_warp - 1) / ((uint64_t)kWarps * segs_per_warp);
    if (grid < 4 * wv.ctas()) grid = 4 * wv.ctas();  // at least four waves
    if (grid > ctas) grid = ctas;
    K<<<(uint32_t)grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int decode_tile_elems(bool e5m2) { return (e5m2 ? e5::kSeg : Bf16Seg::kSeg) * kWarps; }

cudaError_t launch_decode(const DecodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    if (e5m2)
        return launch_segment_wave<decode_e5m2_kernel>(
            a, e5::kSeg, (size_t)e5::kStages * kWarps * e5::kStageBytes, e5::kSegsPerWarp, s);
    return launch_segment_wave<decode_kernel<Bf16Seg>>(a, Bf16Seg::kSeg, decode_smem_bytes<Bf16Seg>(),
                                                       Bf16Seg::kSegsPerWarp, s);
}

}  // namespace splitzip
