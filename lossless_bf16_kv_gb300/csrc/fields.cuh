// fields.cuh -- per-element SplitZip encode arithmetic shared by the encode
// kernels: BF16 / E5M2 field split, exponent -> code table lookup, nibble
// packing and escape counting ("SplitZip: Ultra-Fast Lossless KV Compression
// for Disaggregated LLM Serving", README section Abstract: sign and mantissa
// kept exact, frequent exponents as fixed 4-bit codes, rare ones escaped).
#pragma once

#include <cstdint>

namespace splitzip {

constexpr uint32_t kMissEntry = 0x10u;  // table entry of an exponent outside the codebook

// Four table entries for the four exponent bytes of `ex`, one per byte.
__device__ __forceinline__ uint32_t lookup4(const uint8_t* table, uint32_t ex) {
    const uint32_t e0 = table[ex & 0xFFu];
    const uint32_t e1 = table[(ex >> 8) & 0xFFu];
    const uint32_t e2 = table[(ex >> 16) & 0xFFu];
    const uint32_t e3 = table[ex >> 24];
    return __byte_perm(__byte_perm(e0, e1, 0x0040), __byte_perm(e2, e3, 0x0040), 0x5410);
}

// Packs the codes of two entry words (elements 0..3 and 4..7) into 8 nibbles:
// byte j holds elements 2j (low nibble) and 2j+1 (high nibble).
__device__ __forceinline__ uint32_t pack_nibbles(uint32_t w_lo, uint32_t w_hi) {
    const uint32_t p_lo = (w_lo & 0x0F0F0F0Fu) | ((w_lo >> 4) & 0xF0F0F0F0u);
    const uint32_t p_hi = (w_hi & 0x0F0F0F0Fu) | ((w_hi >> 4) & 0xF0F0F0F0u);
    return __byte_perm(p_lo, p_hi, 0x6420);
}

__device__ __forceinline__ uint32_t miss_count(uint32_t w_lo, uint32_t w_hi) {
    return __popc((w_lo & 0x10101010u) | ((w_hi & 0x10101010u) >> 1));
}

// ------------------------------------------------------------------- BF16
//
// Field split of 8 BF16 values (4 words, 2 values each): the low bytes of
// elements 0..3 gather into one word and the high bytes into another, so the
// sign+mantissa byte (sign from the high byte's bit 7, mantissa from the low
// byte's bits 0..6) and the exponent byte (high byte bits 0..6 above low byte
// bit 7) come out four at a time.
__device__ __forceinline__ void split_bf16(uint32_t a, uint32_t b, uint32_t& sm, uint32_t& ex) {
    const uint32_t lo = __byte_perm(a, b, 0x6420);
    const uint32_t hi = __byte_perm(a, b, 0x7531);
    sm = (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
    ex = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
}

// The four three-bit fields (sign << 2 | mantissa) of 4 E5M2 bytes packed in
// 12 bits, field of byte k at bits 3k..3k+2.  With field k in byte k of f,
// f >> 15 = 512 f3 + 2 f2 (f0 and f1 shift out), and a byte dot product with
// (1, 8, 62, 0) added to it gives f0 + 8 f1 + 64 f2 + 512 f3 (fields are below
// 8, so no sum carries into the next field).
__device__ __forceinline__ uint32_t fields12_e5m2(uint32_t w) {
    const uint32_t f = ((w >> 5) & 0x04040404u) | (w & 0x03030303u);  // field k in byte k
    return __dp4a(f, 0x003E0801u, f >> 15);
}

// 4 E5M2 bytes -> 4 exponent bytes and the 12 bits of their fields.
__device__ __forceinline__ void split_e5m2(uint32_t w, uint32_t& ex, uint32_t& f12) {
    ex = (w >> 2) & 0x1F1F1F1Fu;
    f12 = fields12_e5m2(w);
}

}  // namespace splitzip
