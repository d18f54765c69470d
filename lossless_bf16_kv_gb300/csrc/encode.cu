// encode.cu -- SplitZip encode kernels for sm_103a (BF16 and FP8 E5M2).
//
// Method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
// Serving", README section Abstract; arXiv abstract on the paper index page):
// split each value into its exponent and its exact sign+mantissa bits, map the
// exponent through the 16-entry codebook to a 4-bit code, and send exponents
// outside the codebook to a chunk-local escape stream of (position, value).
//
// One launch, one pass over the input.  Each CTA takes a tile (8192 BF16 or
// 16384 E5M2 elements) by atomic ticket, so every tile a CTA can wait on
// belongs to a CTA that has already started.  Per tile:
//   1. 16-byte loads of the input; SWAR field split; exponent -> code lookup
//      in a 256-entry shared-memory table (entry 0x10 marks an escape);
//      nibble packing; the dense code and sign+mantissa streams are stored
//      right away (fixed offsets, no dependence on other tiles).
//   2. Escape counts per thread group; a block-wide scan gives each group's
//      rank inside the tile; warp 0 publishes the tile's count and runs a
//      decoupled look-back (Merrill & Garland, "Single-pass Parallel Prefix
//      Scan with Decoupled Look-back", 2016) over earlier tiles' state words
//      to get the tile's exclusive escape prefix.
//   3. Escapes are written compacted at their global ranks, and chunk_off is
//      written at every chunk boundary inside the tile.
// Escapes are therefore in element order, which is chunk order then position
// order within a chunk, for any chunk size.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

constexpr uint32_t kMissEntry = 0x10u;  // table entry of an exponent outside the codebook

// ------------------------------------------------------------------ setup

struct TileInfo {
    uint32_t tile;   // tile id (ticket)
    uint32_t epoch;  // launch epoch
    uint32_t t0;     // first element of the tile
    uint32_t q0;     // t0 / chunk
    uint32_t r0;     // t0 % chunk
};

// Takes the ticket, reads the epoch and builds the exponent -> entry table.
template <int kTile>
__device__ __forceinline__ TileInfo tile_setup(const EncodeArgs& a, uint8_t* table,
                                               uint32_t* s_info) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    const int tid = threadIdx.x;
    if (tid == 0) {
        const uint32_t tile = atomicAdd(&hdr->ticket, 1u);
        const uint32_t epoch = *reinterpret_cast<volatile uint32_t*>(&hdr->epoch);
        const uint32_t t0 = tile * (uint32_t)kTile;  // tile < num_tiles keeps t0 < n < 2^32
        const uint32_t q0 = t0 / a.cdiv.d;
        s_info[0] = tile;
        s_info[1] = epoch;
        s_info[2] = t0;
        s_info[3] = q0;
        s_info[4] = t0 - q0 * a.cdiv.d;
    }
    table[tid] = (uint8_t)kMissEntry;
    __syncthreads();
    if (tid < 16) table[(a.cbw[tid >> 2] >> (8 * (tid & 3))) & 0xFFu] = (uint8_t)tid;
    __syncthreads();
    TileInfo t;
    t.tile = s_info[0];
    t.epoch = s_info[1];
    t.t0 = s_info[2];
    t.q0 = s_info[3];
    t.r0 = s_info[4];
    return t;
}

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

// ------------------------------------------------------- block-wide scan
//
// Each thread holds counts c[k] (k < G <= 4) for its groups; group (k, t) comes
// before (k', t') in element order iff k < k' or (k == k' and t < t').  Returns
// the exclusive rank of each group inside the tile and the tile total.
template <int G>
__device__ __forceinline__ uint32_t block_ranks(const uint32_t (&c)[G], uint32_t (&rank)[G],
                                                uint32_t (*s_warp)[2]) {
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
        s_warp[warp][0] = p01;
        s_warp[warp][1] = p23;
    }
    __syncthreads();
    uint32_t pre01 = 0, pre23 = 0, tot01 = 0, tot23 = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
        const uint32_t x = s_warp[w][0], y = s_warp[w][1];
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

// ------------------------------------------------------ decoupled look-back
//
// Run by all 32 lanes of warp 0.  Publishes the tile's aggregate, walks back
// over earlier tiles' state words 32 at a time until it meets an inclusive
// prefix, publishes this tile's inclusive prefix and returns the exclusive one.
// Every wait is bounded by a.spin_limit polls.
__device__ __forceinline__ uint32_t look_back(const EncodeArgs& a, const TileInfo& t,
                                              uint32_t aggregate) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    uint64_t* states = reinterpret_cast<uint64_t*>(a.ws + kWsHeaderBytes);
    const int lane = threadIdx.x & 31;
    if (t.tile == 0) {
        if (lane == 0 && !(a.test_flags & kTestStallFirstTile))
            st_relaxed_gpu(states, make_state(kFlagPrefix, aggregate, t.epoch));
        return 0;
    }
    if (lane == 0) st_relaxed_gpu(states + t.tile, make_state(kFlagAggregate, aggregate, t.epoch));
    uint32_t excl = 0, polls = 0;
    bool timed_out = false;
    int64_t pred = (int64_t)t.tile - 1;
    while (true) {
        const int64_t idx = pred - lane;
        const uint64_t w = idx >= 0 ? ld_relaxed_gpu(states + idx)
                                    : make_state(kFlagPrefix, 0u, t.epoch);
        const uint32_t f = state_flag(w, t.epoch);
        const uint32_t pm = __ballot_sync(0xFFFFFFFFu, f == kFlagPrefix);
        const uint32_t bad = __ballot_sync(0xFFFFFFFFu, f == 0u);
        // Lanes up to and including the nearest inclusive prefix (all 32 if none).
        const uint32_t need = pm ? (((pm & (0u - pm)) << 1) - 1u) : 0xFFFFFFFFu;
        if (bad & need) {
            if (++polls > a.spin_limit) {
                timed_out = true;
                break;
            }
            __nanosleep(100);
            continue;
        }
        excl += __reduce_add_sync(0xFFFFFFFFu, ((need >> lane) & 1u) ? (uint32_t)w : 0u);
        if (pm) break;
        pred -= 32;
    }
    if (lane == 0) {
        if (timed_out) atomicOr(&hdr->status, kStatusTimeout);
        // Published even after a time-out so that later tiles are not held up.
        st_relaxed_gpu(states + t.tile, make_state(kFlagPrefix, excl + aggregate, t.epoch));
    }
    return excl;
}

// CTA exit bookkeeping (thread 0): the last CTA to finish moves the status
// bits out and re-arms the header for the next launch.
__device__ __forceinline__ void count_finished(const EncodeArgs& a, uint32_t epoch) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    __threadfence();
    const uint32_t prev = atomicAdd(&hdr->done, 1u);
    if (prev == a.num_tiles - 1) {
        __threadfence();
        hdr->last_status = atomicExch(&hdr->status, 0u);
        hdr->ticket = 0;
        hdr->done = 0;
        hdr->epoch = epoch + 1u;
        __threadfence();
    }
}

// End of a tile: the tile holding the last element records E and the
// overflow bit, then the CTA counts itself finished.
__device__ __forceinline__ void tile_finish(const EncodeArgs& a, const TileInfo& t,
                                            uint32_t total) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    if (threadIdx.x != 0) return;
    if (t.tile == a.num_tiles - 1) {
        a.chunk_off[a.nchunks] = total;
        hdr->last_escapes = total;
        if ((uint64_t)total > a.esc_capacity) atomicOr(&hdr->status, kStatusOverflow);
    }
    count_finished(a, t.epoch);
}

// A ticket at or past the grid size means the header did not start zeroed:
// touch nothing but the header, and report it.
__device__ __forceinline__ bool stray_tile(const EncodeArgs& a, const TileInfo& t) {
    if (t.tile < a.num_tiles) return false;
    if (threadIdx.x == 0) {
        atomicOr(&reinterpret_cast<WsHeader*>(a.ws)->status, kStatusBadWorkspace);
        count_finished(a, t.epoch);
    }
    return true;
}

__device__ __forceinline__ void put_escape(const EncodeArgs& a, uint32_t rank, uint32_t pos,
                                           uint32_t e) {
    if ((uint64_t)rank < a.esc_capacity) {
        a.esc_pos[rank] = (uint16_t)pos;
        a.esc_val[rank] = (uint8_t)e;
    }
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

constexpr int kBf16Groups = 4;                              // groups of 8 per thread
constexpr int kBf16Tile = kThreads * kBf16Groups * 8;      // 8192 elements
constexpr uint32_t kBf16Stride = kThreads * 8;             // elements between a thread's groups

__global__ void __launch_bounds__(kThreads) encode_bf16_kernel(const EncodeArgs a) {
    __shared__ uint8_t table[256];
    __shared__ uint32_t s_info[5];
    __shared__ uint32_t s_warp[kWarps][2];
    __shared__ uint32_t s_excl;

    const TileInfo t = tile_setup<kBf16Tile>(a, table, s_info);
    if (stray_tile(a, t)) return;
    const int tid = threadIdx.x;
    const uint32_t pad = (a.cbw[0] & 0xFFu) << 7;  // exponent cb[0], sign 0, mantissa 0: code 0
    const bool full = (uint64_t)t.t0 + kBf16Tile <= a.n;

    uint32_t ex[kBf16Groups][2], ent[kBf16Groups][2], cnt[kBf16Groups];
#pragma unroll
    for (int k = 0; k < kBf16Groups; k++) {
        const uint32_t i = t.t0 + k * kBf16Stride + tid * 8;
        uint4 v;
        if (full || i + 8 <= a.n) {
            v = ld_stream16(a.x + 2ull * i);
        } else {
            uint16_t h[8];
#pragma unroll
            for (int j = 0; j < 8; j++)
                h[j] = (i < a.n && j < (int)(a.n - i))
                           ? reinterpret_cast<const uint16_t*>(a.x)[i + j]
                           : (uint16_t)pad;
            v.x = h[0] | ((uint32_t)h[1] << 16);
            v.y = h[2] | ((uint32_t)h[3] << 16);
            v.z = h[4] | ((uint32_t)h[5] << 16);
            v.w = h[6] | ((uint32_t)h[7] << 16);
        }
        uint32_t sm0, sm1;
        split_bf16(v.x, v.y, sm0, ex[k][0]);
        split_bf16(v.z, v.w, sm1, ex[k][1]);
        ent[k][0] = lookup4(table, ex[k][0]);
        ent[k][1] = lookup4(table, ex[k][1]);
        const uint32_t codes = pack_nibbles(ent[k][0], ent[k][1]);
        cnt[k] = miss_count(ent[k][0], ent[k][1]);
        if (full || i + 8 <= a.n) {
            st_stream4(a.codes + i / 2, codes);
            st_stream8(a.signman + i, make_uint2(sm0, sm1));
        } else if (i < a.n) {
            const uint32_t rem = a.n - i;
            for (uint32_t j = 0; j < (rem + 1) / 2; j++) a.codes[i / 2 + j] = (uint8_t)(codes >> (8 * j));
            for (uint32_t j = 0; j < rem; j++)
                a.signman[i + j] = (uint8_t)((j < 4 ? sm0 : sm1) >> (8 * (j & 3)));
        }
    }

    uint32_t rank[kBf16Groups];
    const uint32_t aggregate = block_ranks<kBf16Groups>(cnt, rank, s_warp);
    if (tid < 32) {
        const uint32_t excl = look_back(a, t, aggregate);
        if (tid == 0) s_excl = excl;
    }
    __syncthreads();
    const uint32_t excl = s_excl;

#pragma unroll
    for (int k = 0; k < kBf16Groups; k++) {
        const uint32_t loff = k * kBf16Stride + tid * 8;
        const uint32_t i = t.t0 + loff;
        if (!full && i >= a.n) continue;
        // A group of 8 lies inside one chunk (chunk % 8 == 0, group 8-aligned).
        const uint32_t x = t.r0 + loff;
        const uint32_t q = chunk_quot(a.cdiv, x);
        const uint32_t r = x - q * a.cdiv.d;
        uint32_t g = excl + rank[k];
        if (r == 0) a.chunk_off[t.q0 + q] = g;
        if (cnt[k]) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const uint32_t e = ent[k][j >> 2] >> (8 * (j & 3));
                if (e & kMissEntry) {
                    put_escape(a, g, r + j, (ex[k][j >> 2] >> (8 * (j & 3))) & 0xFFu);
                    g++;
                }
            }
        }
    }
    tile_finish(a, t, excl + aggregate);
}

// ------------------------------------------------------------------- E5M2
//
// A thread group is 32 consecutive elements (two 16-byte loads): 16 code
// bytes and 12 sign+mantissa bytes (32 three-bit fields) per group.

// 4 E5M2 bytes -> 4 exponent bytes and 4 three-bit fields packed in 12 bits
// (field of byte k at bits 3k..3k+2).
__device__ __forceinline__ void split_e5m2(uint32_t w, uint32_t& ex, uint32_t& f12) {
    ex = (w >> 2) & 0x1F1F1F1Fu;
    const uint32_t f = ((w >> 5) & 0x04040404u) | (w & 0x03030303u);  // sign<<2 | mantissa
    const uint32_t t = f | (f >> 5);
    f12 = (t & 0x3Fu) | ((t >> 10) & 0xFC0u);
}

constexpr int kE5m2Groups = 2;                              // groups of 32 per thread
constexpr int kE5m2Tile = kThreads * kE5m2Groups * 32;     // 16384 elements
constexpr uint32_t kE5m2Stride = kThreads * 32;

__global__ void __launch_bounds__(kThreads) encode_e5m2_kernel(const EncodeArgs a) {
    __shared__ uint8_t table[256];
    __shared__ uint32_t s_info[5];
    __shared__ uint32_t s_warp[kWarps][2];
    __shared__ uint32_t s_excl;

    const TileInfo t = tile_setup<kE5m2Tile>(a, table, s_info);
    if (stray_tile(a, t)) return;
    const int tid = threadIdx.x;
    const uint32_t pad = (a.cbw[0] & 0x1Fu) << 2;  // exponent cb[0], sign 0, mantissa 0
    const bool full = (uint64_t)t.t0 + kE5m2Tile <= a.n;

    uint32_t ex[kE5m2Groups][8], ent[kE5m2Groups][8], cnt[kE5m2Groups];
#pragma unroll
    for (int k = 0; k < kE5m2Groups; k++) {
        const uint32_t i = t.t0 + k * kE5m2Stride + tid * 32;
        uint32_t w[8];
        if (full || i + 32 <= a.n) {
            const uint4 v0 = ld_stream16(a.x + i);
            const uint4 v1 = ld_stream16(a.x + i + 16);
            w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
            w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
        } else {
#pragma unroll
            for (int m = 0; m < 8; m++) {
                uint32_t acc = 0;
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    const uint32_t j = m * 4 + b;
                    const uint32_t byte = (i < a.n && j < a.n - i) ? a.x[i + j] : pad;
                    acc |= byte << (8 * b);
                }
                w[m] = acc;
            }
        }
        uint32_t f12[8];
        cnt[k] = 0;
#pragma unroll
        for (int m = 0; m < 8; m++) {
            split_e5m2(w[m], ex[k][m], f12[m]);
            ent[k][m] = lookup4(table, ex[k][m]);
        }
        uint4 codes;
        codes.x = pack_nibbles(ent[k][0], ent[k][1]);
        codes.y = pack_nibbles(ent[k][2], ent[k][3]);
        codes.z = pack_nibbles(ent[k][4], ent[k][5]);
        codes.w = pack_nibbles(ent[k][6], ent[k][7]);
#pragma unroll
        for (int m = 0; m < 8; m += 2) cnt[k] += miss_count(ent[k][m], ent[k][m + 1]);
        // 8 x 12 bits -> 96 bits, little-endian.
        const uint32_t s0 = f12[0] | (f12[1] << 12) | (f12[2] << 24);
        const uint32_t s1 = (f12[2] >> 8) | (f12[3] << 4) | (f12[4] << 16) | (f12[5] << 28);
        const uint32_t s2 = (f12[5] >> 4) | (f12[6] << 8) | (f12[7] << 20);
        uint8_t* smp = a.signman + (uint64_t)(i / 32) * 12;
        if (full || i + 32 <= a.n) {
            st_stream16(a.codes + i / 2, codes);
            st_stream4(smp, s0);
            st_stream4(smp + 4, s1);
            st_stream4(smp + 8, s2);
        } else if (i < a.n) {
            const uint32_t rem = a.n - i;
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
            for (uint32_t j = 0; j < (rem + 1) / 2; j++)
                a.codes[i / 2 + j] = (uint8_t)(cw[j >> 2] >> (8 * (j & 3)));
            const uint32_t sw[3] = {s0, s1, s2};
            for (uint32_t j = 0; j < (3 * rem + 7) / 8; j++)
                smp[j] = (uint8_t)(sw[j >> 2] >> (8 * (j & 3)));
        }
    }

    uint32_t rank[kE5m2Groups];
    const uint32_t aggregate = block_ranks<kE5m2Groups>(cnt, rank, s_warp);
    if (tid < 32) {
        const uint32_t excl = look_back(a, t, aggregate);
        if (tid == 0) s_excl = excl;
    }
    __syncthreads();
    const uint32_t excl = s_excl;

#pragma unroll
    for (int k = 0; k < kE5m2Groups; k++) {
        const uint32_t loff = k * kE5m2Stride + tid * 32;
        const uint32_t i = t.t0 + loff;
        if (!full && i >= a.n) continue;
        uint32_t g = excl + rank[k];
        // Four runs of 8 elements; each lies inside one chunk.
#pragma unroll
        for (int s = 0; s < 4; s++) {
            if (!full && i + 8 * s >= a.n) break;
            const uint32_t x = t.r0 + loff + 8 * s;
            const uint32_t q = chunk_quot(a.cdiv, x);
            const uint32_t r = x - q * a.cdiv.d;
            if (r == 0) a.chunk_off[t.q0 + q] = g;
            const uint32_t e_lo = ent[k][2 * s], e_hi = ent[k][2 * s + 1];
            if (miss_count(e_lo, e_hi)) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const uint32_t e = (j < 4 ? e_lo : e_hi) >> (8 * (j & 3));
                    if (e & kMissEntry) {
                        put_escape(a, g, r + j, (ex[k][2 * s + (j >> 2)] >> (8 * (j & 3))) & 0xFFu);
                        g++;
                    }
                }
            }
        }
    }
    tile_finish(a, t, excl + aggregate);
}

}  // namespace

int encode_tile_elems(bool e5m2) { return e5m2 ? kE5m2Tile : kBf16Tile; }

cudaError_t launch_encode(const EncodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.num_tiles == 0) return cudaSuccess;
    if (e5m2)
        encode_e5m2_kernel<<<a.num_tiles, kThreads, 0, s>>>(a);
    else
        encode_bf16_kernel<<<a.num_tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace splitzip
