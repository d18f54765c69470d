// decode.cu -- SplitZip decode kernels for sm_103a (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README sections Codec API and FAQ; arXiv abstract on the paper
// index page): unpack the 4-bit codes, look each up in the 16-entry codebook,
// reassemble sign, exponent and mantissa, and put the raw exponent of every
// escape back at its position; the result is bitwise identical to the input.
//
// One launch, no communication between CTAs.  Each CTA decodes a fixed tile of
// elements (8192 BF16, 16384 E5M2):
//   1. it issues the loads of its dense streams (codes, sign+mantissa) first;
//   2. while they are in flight it finds the tile's slice [lo, hi) of the
//      escape stream (chunk_off at a chunk start, else a warp-wide search of
//      the ascending positions inside the chunk), clears a per-element escape
//      bitmap in shared memory and scatters the slice's raw exponents into a
//      shared-memory byte array;
//   3. each thread decodes its groups in registers: codebook lookup by byte
//      permutes (the 16 entries live in four registers), SWAR reassembly,
//      exponent patch where the bitmap says so, 16-byte stores.
// All escape metadata is clamped, so malformed streams cannot make the kernel
// read or write out of bounds.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

// Exponents of four codes (code k in nibble k of c16) from the codebook held
// in four words (cb0 = entries 0..3, ..., cb3 = entries 12..15).  Entries
// 0..7 and 8..15 are each one byte permute; a third permute in sign-replicate
// mode turns bit 3 of each code into a 0x00/0xFF byte mask that picks between
// the two.
__device__ __forceinline__ uint32_t cb_lookup4(const uint32_t (&cb)[4], uint32_t c16) {
    const uint32_t sel = c16 & 0x7777u;
    const uint32_t lo = prmt(cb[0], cb[1], sel);
    const uint32_t hi = prmt(cb[2], cb[3], sel);
    const uint32_t t = c16 & 0x8888u;
    const uint32_t m = prmt(0x00008000u, 0u, t | (t >> 3));  // nibble 9 -> 0xFF, 0 -> 0x00
    return (hi & m) | (lo & ~m);
}

// 4-bit mask -> byte mask (bit k set -> byte k = 0xFF).
__device__ __forceinline__ uint32_t expand_nibble(uint32_t b) {
    return ((b * 0x00204081u) & 0x01010101u) * 0xFFu;
}

// Four BF16 values from four sign+mantissa bytes and four exponent bytes.
__device__ __forceinline__ uint2 assemble_bf16(uint32_t sm, uint32_t ex) {
    const uint32_t lo = (sm & 0x7F7F7F7Fu) | ((ex << 7) & 0x80808080u);
    const uint32_t hi = (sm & 0x80808080u) | ((ex >> 1) & 0x7F7F7F7Fu);
    return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

// Four E5M2 values from four 3-bit fields (12 bits, field k at bits 3k) and
// four exponent bytes.
__device__ __forceinline__ uint32_t assemble_e5m2(uint32_t f12, uint32_t ex) {
    const uint32_t t = (f12 & 0x3Fu) | ((f12 & 0xFC0u) << 10);
    const uint32_t f = (t & 0x00070007u) | ((t & 0x00380038u) << 5);
    return ((f << 5) & 0x80808080u) | ((ex << 2) & 0x7C7C7C7Cu) | (f & 0x03030303u);
}

// First index j in [b, e) with pos[j] >= r, for positions in ascending order
// (any result in [b, e] otherwise).  All 32 lanes of a warp call it.
__device__ uint32_t lower_bound_warp(const uint16_t* pos, uint32_t b, uint32_t e, uint32_t r) {
    const uint32_t lane = threadIdx.x & 31;
    while (e - b > 32) {
        const uint32_t step = (e - b + 31) / 32;
        const uint32_t j = b + lane * step;
        const bool lt = j < e && pos[j] < r;
        const uint32_t k = __popc(__ballot_sync(0xFFFFFFFFu, lt));
        if (k == 0) return b;
        const uint32_t nb = b + (k - 1) * step + 1;
        const uint32_t ne = min(e, b + k * step);
        b = nb;
        e = ne;
    }
    const bool lt = b + lane < e && pos[b + lane] < r;
    return b + __popc(__ballot_sync(0xFFFFFFFFu, lt));
}

__device__ __forceinline__ uint32_t clamp_off(const DecodeArgs& a, uint32_t c) {
    const uint64_t v = a.chunk_off[c];
    return (uint32_t)(v < a.esc_count ? v : a.esc_count);
}

// Index of the first escape of element x or later (x <= n).  All lanes call it.
__device__ uint32_t escape_bound(const DecodeArgs& a, uint32_t x) {
    if (x >= a.n) return clamp_off(a, a.nchunks);
    const uint32_t c = x / a.cdiv.d;
    const uint32_t r = x - c * a.cdiv.d;
    const uint32_t b = clamp_off(a, c);
    if (r == 0) return b;
    const uint32_t e = max(b, clamp_off(a, c + 1));
    return lower_bound_warp(a.esc_pos, b, e, r);
}

// Steps 2 of the kernel: slice bounds, bitmap clear, scatter.  `exps` holds
// kTile bytes, `mask` kTile/32 words.
template <int kTile>
__device__ __forceinline__ void scatter_escapes(const DecodeArgs& a, uint32_t t0,
                                                uint8_t* exps, uint32_t* mask,
                                                uint32_t* s_bounds) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t t1 = (uint64_t)t0 + kTile < a.n ? t0 + kTile : a.n;
    if (warp == 0) {
        const uint32_t lo = escape_bound(a, t0);
        if (lane == 0) s_bounds[0] = lo;
    } else if (warp == 1) {
        const uint32_t hi = escape_bound(a, t1);
        if (lane == 0) s_bounds[1] = hi;
    }
    for (int w = tid; w < kTile / 32; w += kThreads) mask[w] = 0;
    __syncthreads();
    const uint32_t lo = s_bounds[0], hi = max(s_bounds[0], s_bounds[1]);
    if (lo == hi) return;
    const uint32_t ca = t0 / a.cdiv.d, cb = (t1 - 1) / a.cdiv.d;
    const uint32_t nc = cb - ca + 1;
    auto scatter_chunk = [&](uint32_t c, uint32_t first, uint32_t step) {
        const uint32_t b = max(clamp_off(a, c), lo);
        const uint32_t e = min(clamp_off(a, c + 1), hi);
        const uint32_t cbase = c * a.cdiv.d;
        for (uint32_t j = b + first; j < e; j += step) {
            const uint32_t p = a.esc_pos[j];
            const uint32_t l = cbase + p - t0;  // wraps to a large value if below t0
            if (p < a.cdiv.d && l < (uint32_t)kTile && cbase + p < t1) {
                exps[l] = a.esc_val[j];
                atomicOr(&mask[l >> 5], 1u << (l & 31));
            }
        }
    };
    if (nc >= (uint32_t)kWarps) {
        for (uint32_t c = ca + warp; c <= cb; c += kWarps) scatter_chunk(c, lane, 32);
    } else {
        for (uint32_t c = ca; c <= cb; c++) scatter_chunk(c, tid, kThreads);
    }
}

// ------------------------------------------------------------------- BF16

constexpr int kBf16Groups = 4;                          // groups of 8 per thread
constexpr int kBf16Tile = kThreads * kBf16Groups * 8;  // 8192 elements
constexpr uint32_t kBf16Stride = kThreads * 8;

__global__ void __launch_bounds__(kThreads) decode_bf16_kernel(const DecodeArgs a) {
    __shared__ __align__(16) uint8_t exps[kBf16Tile];
    __shared__ uint32_t mask[kBf16Tile / 32];
    __shared__ uint32_t s_bounds[2];

    const int tid = threadIdx.x;
    const uint32_t t0 = blockIdx.x * (uint32_t)kBf16Tile;
    const bool full = (uint64_t)t0 + kBf16Tile <= a.n;
    const uint32_t cb[4] = {a.cbw[0], a.cbw[1], a.cbw[2], a.cbw[3]};

    uint32_t code[kBf16Groups];
    uint2 sm[kBf16Groups];
#pragma unroll
    for (int k = 0; k < kBf16Groups; k++) {
        const uint32_t i = t0 + k * kBf16Stride + tid * 8;
        if (full || i + 8 <= a.n) {
            code[k] = ld_stream4(a.codes + i / 2);
            sm[k] = ld_stream8(a.signman + i);
        } else {
            code[k] = 0;
            sm[k] = make_uint2(0, 0);
            if (i < a.n) {
                const uint32_t rem = a.n - i;
                for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                    code[k] |= (uint32_t)a.codes[i / 2 + j] << (8 * j);
                for (uint32_t j = 0; j < rem; j++) {
                    const uint32_t b = (uint32_t)a.signman[i + j] << (8 * (j & 3));
                    if (j < 4) sm[k].x |= b; else sm[k].y |= b;
                }
            }
        }
    }

    scatter_escapes<kBf16Tile>(a, t0, exps, mask, s_bounds);
    __syncthreads();

#pragma unroll
    for (int k = 0; k < kBf16Groups; k++) {
        const uint32_t loff = k * kBf16Stride + tid * 8;
        const uint32_t i = t0 + loff;
        if (!full && i >= a.n) continue;
        uint32_t ex0 = cb_lookup4(cb, code[k] & 0xFFFFu);
        uint32_t ex1 = cb_lookup4(cb, code[k] >> 16);
        const uint32_t mb = reinterpret_cast<const uint8_t*>(mask)[loff >> 3];
        if (mb) {
            const uint2 xv = *reinterpret_cast<const uint2*>(exps + loff);
            const uint32_t m0 = expand_nibble(mb & 0xFu), m1 = expand_nibble(mb >> 4);
            ex0 = (xv.x & m0) | (ex0 & ~m0);
            ex1 = (xv.y & m1) | (ex1 & ~m1);
        }
        const uint2 o0 = assemble_bf16(sm[k].x, ex0);
        const uint2 o1 = assemble_bf16(sm[k].y, ex1);
        if (full || i + 8 <= a.n) {
            st_stream16(a.y + 2ull * i, make_uint4(o0.x, o0.y, o1.x, o1.y));
        } else {
            const uint32_t w[4] = {o0.x, o0.y, o1.x, o1.y};
            uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + i;
            for (uint32_t j = 0; j < a.n - i; j++) yp[j] = (uint16_t)(w[j >> 1] >> (16 * (j & 1)));
        }
    }
}

// ------------------------------------------------------------------- E5M2

constexpr int kE5m2Groups = 2;                          // groups of 32 per thread
constexpr int kE5m2Tile = kThreads * kE5m2Groups * 32; // 16384 elements
constexpr uint32_t kE5m2Stride = kThreads * 32;

__global__ void __launch_bounds__(kThreads) decode_e5m2_kernel(const DecodeArgs a) {
    __shared__ __align__(16) uint8_t exps[kE5m2Tile];
    __shared__ uint32_t mask[kE5m2Tile / 32];
    __shared__ uint32_t s_bounds[2];

    const int tid = threadIdx.x;
    const uint32_t t0 = blockIdx.x * (uint32_t)kE5m2Tile;
    const bool full = (uint64_t)t0 + kE5m2Tile <= a.n;
    const uint32_t cb[4] = {a.cbw[0], a.cbw[1], a.cbw[2], a.cbw[3]};

    uint4 code[kE5m2Groups];
    uint32_t smw[kE5m2Groups][3];
#pragma unroll
    for (int k = 0; k < kE5m2Groups; k++) {
        const uint32_t i = t0 + k * kE5m2Stride + tid * 32;
        const uint8_t* smp = a.signman + (uint64_t)(i / 32) * 12;
        if (full || i + 32 <= a.n) {
            code[k] = ld_stream16(a.codes + i / 2);
            smw[k][0] = ld_stream4(smp);
            smw[k][1] = ld_stream4(smp + 4);
            smw[k][2] = ld_stream4(smp + 8);
        } else {
            uint32_t cw[4] = {0, 0, 0, 0};
            smw[k][0] = smw[k][1] = smw[k][2] = 0;
            if (i < a.n) {
                const uint32_t rem = a.n - i;
                for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                    cw[j >> 2] |= (uint32_t)a.codes[i / 2 + j] << (8 * (j & 3));
                for (uint32_t j = 0; j < (3 * rem + 7) / 8; j++)
                    smw[k][j >> 2] |= (uint32_t)smp[j] << (8 * (j & 3));
            }
            code[k] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        }
    }

    scatter_escapes<kE5m2Tile>(a, t0, exps, mask, s_bounds);
    __syncthreads();

#pragma unroll
    for (int k = 0; k < kE5m2Groups; k++) {
        const uint32_t loff = k * kE5m2Stride + tid * 32;
        const uint32_t i = t0 + loff;
        if (!full && i >= a.n) continue;
        const uint32_t s0 = smw[k][0], s1 = smw[k][1], s2 = smw[k][2];
        const uint32_t f12[8] = {
            s0 & 0xFFFu, (s0 >> 12) & 0xFFFu, __funnelshift_r(s0, s1, 24) & 0xFFFu,
            (s1 >> 4) & 0xFFFu, (s1 >> 16) & 0xFFFu, __funnelshift_r(s1, s2, 28) & 0xFFFu,
            (s2 >> 8) & 0xFFFu, s2 >> 20};
        const uint32_t cw[4] = {code[k].x, code[k].y, code[k].z, code[k].w};
        const uint32_t mword = mask[loff >> 5];
        uint32_t out[8];
#pragma unroll
        for (int m = 0; m < 8; m++) {
            uint32_t ex = cb_lookup4(cb, (cw[m >> 1] >> (16 * (m & 1))) & 0xFFFFu);
            const uint32_t mb = (mword >> (4 * m)) & 0xFu;
            if (mb) {
                const uint32_t xv = *reinterpret_cast<const uint32_t*>(exps + loff + 4 * m);
                const uint32_t mm = expand_nibble(mb);
                ex = (xv & mm) | (ex & ~mm);
            }
            out[m] = assemble_e5m2(f12[m], ex);
        }
        if (full || i + 32 <= a.n) {
            st_stream16(a.y + i, make_uint4(out[0], out[1], out[2], out[3]));
            st_stream16(a.y + i + 16, make_uint4(out[4], out[5], out[6], out[7]));
        } else {
            for (uint32_t j = 0; j < a.n - i; j++) a.y[i + j] = (uint8_t)(out[j >> 2] >> (8 * (j & 3)));
        }
    }
}

}  // namespace

int decode_tile_elems(bool e5m2) { return e5m2 ? kE5m2Tile : kBf16Tile; }

cudaError_t launch_decode(const DecodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.num_tiles == 0) return cudaSuccess;
    if (e5m2)
        decode_e5m2_kernel<<<a.num_tiles, kThreads, 0, s>>>(a);
    else
        decode_bf16_kernel<<<a.num_tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace splitzip
