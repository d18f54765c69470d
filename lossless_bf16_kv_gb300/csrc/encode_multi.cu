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
//   K1 dense     one CTA per 8192-element tile, no inter-CTA communication:
//                16-byte loads, field split, table lookup, nibble packing,
//                dense code and sign+mantissa stores.  Each warp ranks the
//                escapes of its segments with shuffles and stores the count
//                and the first few escapes of every segment in the
//                workspace.
//   K2 prefix    exclusive prefix of the per-tile escape counts (sums of the
//                segment counts; 2048 tiles per CTA,
//                decoupled look-back across CTAs, bounded waits); E.
//   K3 place     a warp per tile: segment offsets by shuffle scan, escapes
//                copied to their final places, chunk offsets at chunk starts.
//                A segment with more escapes than its workspace share is
//                rebuilt from the input in element order.
// Segments: BF16 -- the 256 consecutive elements warp w covers with its group
// k (k-major: segment 8k + w), 8 workspace entries each; E5M2 -- the 1024
// elements of warp w, 32 entries each.  Entries hold the position in the
// segment and the raw exponent.
#include <cstdint>

#include "common.cuh"
#include "fields.cuh"
#include "kernels.h"
#include "lookback.cuh"

namespace splitzip {
namespace {

constexpr int kTileElems = 8192;     // elements per tile (K1 CTA / K3 warp)
constexpr int kSegsMax = 32;         // segment slots per tile in the workspace
constexpr int kEntries = 256;        // escape entries per tile in the workspace
constexpr int kScanTiles = 2048;     // tiles per K2 CTA (8 per thread)

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct MultiPtrs {
    uint64_t* states;
    uint32_t* tile_excl;
    uint16_t* seg_cnt;
    uint16_t* seg_ent;
};

__device__ __forceinline__ void build_table(uint8_t* table, const uint32_t (&cbw)[4]) {
    const int tid = threadIdx.x;
    table[tid] = (uint8_t)kMissEntry;
    __syncthreads();
    if (tid < 16) table[(cbw[tid >> 2] >> (8 * (tid & 3))) & 0xFFu] = (uint8_t)tid;
    __syncthreads();
}

// Warp-wide exclusive scan of up to four small counts per lane (packed two
// to a word): rel[k] = sum of c[k] over lower lanes, tot[k] = warp sum.
template <int G>
__device__ __forceinline__ void warp_scan(const uint32_t (&c)[G], uint32_t (&rel)[G],
                                          uint32_t (&tot)[G]) {
    const int lane = threadIdx.x & 31;
    uint32_t p01 = c[0] | (G > 1 ? c[1] << 16 : 0u);
    uint32_t p23 = (G > 2 ? c[2] : 0u) | (G > 3 ? c[3] << 16 : 0u);
    const uint32_t own01 = p01, own23 = p23;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, p01, d);
        if (lane >= d) p01 += u;
        if (G > 2) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, p23, d);
            if (lane >= d) p23 += v;
        }
    }
    const uint32_t t01 = __shfl_sync(0xFFFFFFFFu, p01, 31);
    const uint32_t t23 = G > 2 ? __shfl_sync(0xFFFFFFFFu, p23, 31) : 0u;
    const uint32_t e01 = p01 - own01, e23 = p23 - own23;
    const uint32_t ex[4] = {e01 & 0xFFFFu, e01 >> 16, e23 & 0xFFFFu, e23 >> 16};
    const uint32_t tt[4] = {t01 & 0xFFFFu, t01 >> 16, t23 & 0xFFFFu, t23 >> 16};
#pragma unroll
    for (int k = 0; k < G; k++) {
        rel[k] = ex[k];
        tot[k] = tt[k];
    }
}

// ------------------------------------------------------------------- BF16
//
// Thread t's groups of 8 at tile offsets k*2048 + 8t (k < 4): each warp load
// covers 512 contiguous input bytes and each warp store 128 code bytes and
// 256 sign+mantissa bytes.
struct Bf16Dense {
    static constexpr int kGroups = 4;
    static constexpr int kSegs = 32;
    static constexpr int kSegLen = 256;
    static constexpr int kSegCap = kEntries / kSegs;  // 8
    static constexpr int kOffBits = 8;
    static constexpr uint32_t kExpMask = 0xFFu;
    struct Keep {
        uint32_t ex[kGroups][2], ent[kGroups][2], cnt[kGroups];
    };
    static __device__ __forceinline__ uint32_t loff(int k) {
        return k * (kThreads * 8) + threadIdx.x * 8;
    }
    static __device__ __forceinline__ uint32_t seg(int k) { return k * kWarps + (threadIdx.x >> 5); }

    static __device__ __forceinline__ void process(const EncodeArgs& a, const uint8_t* table,
                                                   uint32_t t0, Keep& kp) {
        const bool full = (uint64_t)t0 + kTileElems <= a.n;
        if (full) {
            uint4 v[kGroups];
#pragma unroll
            for (int k = 0; k < kGroups; k++) v[k] = ld_stream16(a.x + 2ull * (t0 + loff(k)));
            uint32_t sm[kGroups][2];
#pragma unroll
            for (int k = 0; k < kGroups; k++) {
                split_bf16(v[k].x, v[k].y, sm[k][0], kp.ex[k][0]);
                split_bf16(v[k].z, v[k].w, sm[k][1], kp.ex[k][1]);
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
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(a.x);
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            const uint32_t i = t0 + loff(k);
            kp.cnt[k] = 0;
            kp.ent[k][0] = kp.ent[k][1] = 0;
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
                for (uint32_t j = 0; j < (rem + 1) / 2; j++) a.codes[i / 2 + j] = (uint8_t)(codes >> (8 * j));
                for (uint32_t j = 0; j < rem; j++)
                    a.signman[i + j] = (uint8_t)((j < 4 ? sm0 : sm1) >> (8 * (j & 3)));
            }
        }
    }

    // The first kSegCap escapes of each segment into its workspace entries.
    static __device__ __forceinline__ void emit(const Keep& kp, const uint32_t (&rel)[kGroups],
                                                uint16_t* ent) {
        const uint32_t lane = threadIdx.x & 31;
#pragma unroll
        for (int k = 0; k < kGroups; k++) {
            if (!kp.cnt[k]) continue;
            uint32_t g = rel[k];
            uint16_t* e = ent + seg(k) * kSegCap;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((kp.ent[k][j >> 2] >> (8 * (j & 3))) & kMissEntry) {
                    if (g < (uint32_t)kSegCap)
                        e[g] = (uint16_t)((8 * lane + j) | (((kp.ex[k][j >> 2] >> (8 * (j & 3))) & kExpMask) << kOffBits));
                    g++;
                }
            }
        }
    }

    // Exponent of element i of the input (K3's rebuild of a full segment).
    static __device__ __forceinline__ uint32_t exponent_at(const EncodeArgs& a, uint32_t i) {
        return (reinterpret_cast<const uint16_t*>(a.x)[i] >> 7) & 0xFFu;
    }
};

// ------------------------------------------------------------------- E5M2
//
// Thread t's group is the 32 elements at tile offset 32t: 16 code bytes and
// 12 bytes of packed 3-bit fields (three 4-byte stores).
struct E5m2Dense {
    static constexpr int kGroups = 1;
    static constexpr int kSegs = kWarps;              // 8
    static constexpr int kSegLen = 1024;
    static constexpr int kSegCap = kEntries / kSegs;  // 32
    static constexpr int kOffBits = 10;
    static constexpr uint32_t kExpMask = 0x1Fu;
    struct Keep {
        uint32_t ex[8], ent[8], cnt[kGroups];
    };
    static __device__ __forceinline__ uint32_t seg(int) { return threadIdx.x >> 5; }

    static __device__ __forceinline__ void process(const EncodeArgs& a, const uint8_t* table,
                                                   uint32_t t0, Keep& kp) {
        const bool full = (uint64_t)t0 + kTileElems <= a.n;
        const uint32_t i = t0 + threadIdx.x * 32;
        kp.cnt[0] = 0;
#pragma unroll
        for (int m = 0; m < 8; m++) kp.ent[m] = 0;
        if (!full && i >= a.n) return;
        const bool whole = full || i + 32 <= a.n;
        uint32_t w[8];
        if (whole) {
            const uint4 v0 = ld_stream16(a.x + i);
            const uint4 v1 = ld_stream16(a.x + i + 16);
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
                    acc |= (j < rem ? (uint32_t)a.x[i + j] : pad) << (8 * b);
                }
                w[m] = acc;
            }
        }
        uint32_t f12[8];
#pragma unroll
        for (int m = 0; m < 8; m++) split_e5m2(w[m], kp.ex[m], f12[m]);
#pragma unroll
        for (int m = 0; m < 8; m++) kp.ent[m] = lookup4(table, kp.ex[m]);
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

    static __device__ __forceinline__ void emit(const Keep& kp, const uint32_t (&rel)[kGroups],
                                                uint16_t* ent) {
        if (!kp.cnt[0]) return;
        const uint32_t lane = threadIdx.x & 31;
        uint32_t g = rel[0];
        uint16_t* e = ent + seg(0) * kSegCap;
#pragma unroll
        for (int m = 0; m < 8; m++) {
            if (!(kp.ent[m] & 0x10101010u)) continue;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                if ((kp.ent[m] >> (8 * b)) & kMissEntry) {
                    if (g < (uint32_t)kSegCap)
                        e[g] = (uint16_t)((32 * lane + 4 * m + b) | (((kp.ex[m] >> (8 * b)) & kExpMask) << kOffBits));
                    g++;
                }
            }
        }
    }

    static __device__ __forceinline__ uint32_t exponent_at(const EncodeArgs& a, uint32_t i) {
        return (a.x[i] >> 2) & 0x1Fu;
    }
};

// --------------------------------------------------------------- K1 dense

// Grid-stride over tiles (one resident wave): the code table is built once
// per CTA and the tile loop has no barrier at all.
template <class F>
__global__ void __launch_bounds__(kThreads) dense_kernel(const EncodeArgs a, const MultiPtrs p) {
    constexpr int G = F::kGroups;
    __shared__ uint8_t table[256];
    build_table(table, a.cbw);
    const uint32_t lane = threadIdx.x & 31;
    for (uint32_t tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x) {
        const uint32_t t0 = tile * (uint32_t)kTileElems;
        typename F::Keep kp;
        F::process(a, table, t0, kp);
        uint32_t rel[G], tot[G];
        warp_scan<G>(kp.cnt, rel, tot);
#pragma unroll
        for (int g = 0; g < G; g++)
            if (lane == (uint32_t)g) p.seg_cnt[(size_t)tile * kSegsMax + F::seg(g)] = (uint16_t)tot[g];
        F::emit(kp, rel, p.seg_ent + (size_t)tile * kEntries);
    }
}

// -------------------------------------------------------------- K2 prefix

// Last CTA of a prefix launch: move the status bits out and re-arm the
// header.  Each CTA draws exactly one ticket, so a clean launch leaves
// gridDim.x tickets; anything else means the header did not start zeroed.
__device__ void prefix_finished(const EncodeArgs& a, uint32_t epoch) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    __threadfence();
    const uint32_t prev = atomicAdd(&hdr->done, 1u);
    if (prev == gridDim.x - 1) {
        __threadfence();
        const uint32_t tickets = atomicAdd(&hdr->ticket, 0u);
        const bool timed_out = (atomicAdd(&hdr->status, 0u) & kStatusTimeout) != 0;
        if (!timed_out && tickets != gridDim.x) atomicOr(&hdr->status, kStatusBadWorkspace);
        hdr->last_status = atomicExch(&hdr->status, 0u);
        hdr->ticket = 0;
        hdr->done = 0;
        hdr->epoch = epoch + 1u;
        __threadfence();
    }
}

__global__ void __launch_bounds__(kThreads) prefix_kernel(const EncodeArgs a, const MultiPtrs p,
                                                          uint32_t num_tiles, uint32_t num_blocks,
                                                          uint32_t segs) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    __shared__ uint32_t s_blk, s_epoch, s_excl;
    __shared__ uint32_t s_warp[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_blk = atomicAdd(&hdr->ticket, 1u);  // blocks in start order: predecessors are running
        s_epoch = *reinterpret_cast<volatile uint32_t*>(&hdr->epoch);
    }
    __syncthreads();
    const uint32_t blk = s_blk, epoch = s_epoch;
    if (blk >= num_blocks) {  // the header did not start zeroed: touch nothing else
        if (tid == 0) {
            atomicOr(&hdr->status, kStatusBadWorkspace);
            prefix_finished(a, epoch);
        }
        return;
    }
    // Tile totals: the sum of each tile's segment counts (16-bit, 32 per tile,
    // the first `segs` in use).
    const uint32_t base = blk * (uint32_t)kScanTiles + tid * 8;
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        v[i] = 0;
        if (base + i >= num_tiles) continue;
        const uint4* row = reinterpret_cast<const uint4*>(p.seg_cnt + (size_t)(base + i) * kSegsMax);
#pragma unroll
        for (int q = 0; q < kSegsMax / 8; q++) {
            if ((uint32_t)q * 8 >= segs) break;
            const uint4 c = row[q];
            const uint32_t w = (c.x & 0xFFFFu) + (c.x >> 16) + (c.y & 0xFFFFu) + (c.y >> 16) +
                               (c.z & 0xFFFFu) + (c.z >> 16) + (c.w & 0xFFFFu) + (c.w >> 16);
            v[i] += w;
        }
    }
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) sum += v[i];
    uint32_t incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t pre = 0, agg = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
        pre += w < warp ? s_warp[w] : 0u;
        agg += s_warp[w];
    }
    if (warp == 0) {
        uint64_t* states = p.states;
        if (lane == 0)
            publish_count(states, blk, epoch, agg, (a.test_flags & kTestStallFirstTile) != 0);
        const uint32_t excl = look_back(states, &hdr->status, blk, epoch, agg, a.spin_limit);
        if (lane == 0) s_excl = excl;
    }
    __syncthreads();
    uint32_t running = s_excl + pre + incl - sum;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        if (base + i < num_tiles) p.tile_excl[base + i] = running;
        running += v[i];
    }
    if (blk == num_blocks - 1 && tid == 0) {
        const uint32_t total = s_excl + agg;
        a.chunk_off[a.nchunks] = total;
        hdr->last_escapes = total;
        if ((uint64_t)total > a.esc_capacity) atomicOr(&hdr->status, kStatusOverflow);
    }
    __syncthreads();
    if (tid == 0) prefix_finished(a, epoch);
}

// --------------------------------------------------------------- K3 place

__device__ __forceinline__ void put_escape(const EncodeArgs& a, uint32_t g, uint32_t pos,
                                           uint32_t e) {
    if ((uint64_t)g < a.esc_capacity) {
        a.esc_pos[g] = (uint16_t)pos;
        a.esc_val[g] = (uint8_t)e;
    }
}

template <class F>
__global__ void __launch_bounds__(kThreads) place_kernel(const EncodeArgs a, const MultiPtrs p,
                                                         uint32_t num_tiles) {
    constexpr uint32_t kOffMask = (1u << F::kOffBits) - 1u;
    __shared__ uint8_t table[256];
    build_table(table, a.cbw);
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t tile = blockIdx.x * kWarps + warp;
    if (tile >= num_tiles) return;  // warp-uniform
    const uint32_t t0 = tile * (uint32_t)kTileElems;
    const uint32_t len = a.n - t0 < (uint32_t)kTileElems ? a.n - t0 : (uint32_t)kTileElems;
    const uint32_t q0 = t0 / a.cdiv.d, r0 = t0 - q0 * a.cdiv.d;
    const uint32_t excl = p.tile_excl[tile];
    const uint32_t cnt = lane < (uint32_t)F::kSegs ? p.seg_cnt[(size_t)tile * kSegsMax + lane] : 0u;
    uint32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    const uint32_t off = incl - cnt;
    const uint16_t* ent = p.seg_ent + (size_t)tile * kEntries;

    // Escapes of segment `lane`, in element order.
    if (cnt) {
        const uint32_t s0 = lane * F::kSegLen;
        const uint32_t g0 = excl + off;
        if (cnt <= (uint32_t)F::kSegCap) {
            for (uint32_t r = 0; r < cnt; r++) {
                const uint32_t e = ent[lane * F::kSegCap + r];
                const uint32_t x = r0 + s0 + (e & kOffMask);
                put_escape(a, g0 + r, x - chunk_quot(a.cdiv, x) * a.cdiv.d, e >> F::kOffBits);
            }
        } else {
            // More escapes than the segment's entries: rebuild from the input.
            const uint32_t end = s0 + F::kSegLen < len ? s0 + F::kSegLen : len;
            uint32_t g = g0;
            for (uint32_t l = s0; l < end; l++) {
                const uint32_t e = F::exponent_at(a, t0 + l);
                if (table[e] & kMissEntry) {
                    const uint32_t x = r0 + l;
                    put_escape(a, g++, x - chunk_quot(a.cdiv, x) * a.cdiv.d, e);
                }
            }
        }
    }

    // chunk_off at every chunk start in the tile: the exclusive escape rank of
    // the chunk's first element.
    const uint32_t qa = r0 ? 1u : 0u, qb = chunk_quot(a.cdiv, r0 + len - 1);
    for (uint32_t b0 = qa; b0 <= qb; b0 += 32) {
        const uint32_t q = b0 + lane;
        const bool valid = q <= qb;
        const uint32_t bl = valid ? q * a.cdiv.d - r0 : 0u;  // tile-local index of the chunk start
        const uint32_t sg = bl / F::kSegLen;
        const uint32_t o = __shfl_sync(0xFFFFFFFFu, off, sg);
        const uint32_t c = __shfl_sync(0xFFFFFFFFu, cnt, sg);
        if (valid) {
            const uint32_t lim = bl - sg * F::kSegLen;
            uint32_t rank = 0;
            if (c <= (uint32_t)F::kSegCap) {
                for (uint32_t r = 0; r < c; r++) rank += (ent[sg * F::kSegCap + r] & kOffMask) < lim;
            } else {
                for (uint32_t l = sg * F::kSegLen; l < bl; l++)
                    rank += (table[F::exponent_at(a, t0 + l)] & kMissEntry) != 0;
            }
            a.chunk_off[q0 + q] = excl + o + rank;
        }
    }
}

template <class F>
cudaError_t launch_three(const EncodeArgs& a, cudaStream_t s) {
    const MultiLayout L = multi_layout(a.n);
    MultiPtrs p;
    p.states = reinterpret_cast<uint64_t*>(a.ws + L.states);
    p.tile_excl = reinterpret_cast<uint32_t*>(a.ws + L.tile_excl);
    p.seg_cnt = reinterpret_cast<uint16_t*>(a.ws + L.seg_cnt);
    p.seg_ent = reinterpret_cast<uint16_t*>(a.ws + L.seg_ent);
    const uint32_t tiles = a.num_tiles;
    const uint32_t blocks = (tiles + kScanTiles - 1) / kScanTiles;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dense_kernel<F>, kThreads, 0);
    if (e != cudaSuccess) return e;
    const uint64_t wave = (uint64_t)(sms > 0 ? sms : 1) * (uint64_t)(per_sm > 0 ? per_sm : 1);
    dense_kernel<F><<<(uint32_t)(tiles < wave ? tiles : wave), kThreads, 0, s>>>(a, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prefix_kernel<<<blocks, kThreads, 0, s>>>(a, p, tiles, blocks, F::kSegs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    place_kernel<F><<<(tiles + kWarps - 1) / kWarps, kThreads, 0, s>>>(a, p, tiles);
    return cudaGetLastError();
}

}  // namespace

MultiLayout multi_layout(uint64_t n) {
    const uint64_t tiles = n ? (n + kTileElems - 1) / kTileElems : 1;
    MultiLayout L;
    size_t off = kWsHeaderBytes;
    L.states = off;
    off += align256(8 * tiles);
    L.tile_excl = off;
    off += align256(4 * tiles);
    L.seg_cnt = off;
    off += align256(2 * kSegsMax * tiles);
    L.seg_ent = off;
    off += align256(2 * kEntries * tiles);
    L.bytes = off;
    return L;
}

cudaError_t launch_encode_multi(const EncodeArgs& a, bool e5m2, cudaStream_t s) {
    if (a.num_tiles == 0) return cudaSuccess;
    return e5m2 ? launch_three<E5m2Dense>(a, s) : launch_three<Bf16Dense>(a, s);
}

}  // namespace splitzip
