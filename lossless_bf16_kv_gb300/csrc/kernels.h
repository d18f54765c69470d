// kernels.h -- launch arguments and launchers of the SplitZip kernels
// (internal to the library; the public interface is include/splitzip.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace splitzip {

constexpr uint32_t kTestStallFirstTile = 1u;    // tile 0 never publishes (test hook)
constexpr uint32_t kTestPipelined = 2u;         // test hook: run the single-launch pipeline
constexpr uint32_t kStatusBadWorkspace = 4u;    // a CTA drew a ticket past the grid
constexpr uint32_t kStatusBadCodebook = 8u;     // a device-resident codebook was not valid
constexpr uint32_t kDefaultSpinLimit = 1u << 21;  // look-back polls (load + 32 ns sleep): ~1 s

struct EncodeArgs {
    const uint8_t* x;  // input bit patterns, 16-byte aligned
    uint32_t n;        // elements
    ChunkDiv cdiv;     // chunk size and its division multiplier
    uint32_t nchunks;  // ceil(n / chunk)
    uint8_t* codes;
    uint8_t* signman;
    uint16_t* esc_pos;
    uint8_t* esc_val;
    uint32_t* chunk_off;
    uint64_t esc_capacity;
    uint8_t* ws;         // workspace: header + tile states
    uint32_t num_tiles;  // grid size
    uint32_t spin_limit;
    uint32_t test_flags;
    uint32_t cbw[4];     // codebook bytes, 4 per word, little-endian
    const uint8_t* dcb = nullptr;  // or, when not null, the 16 codebook bytes in device memory
};

struct DecodeArgs {
    const uint8_t* codes;
    const uint8_t* signman;
    const uint16_t* esc_pos;
    const uint8_t* esc_val;
    const uint32_t* chunk_off;
    uint64_t esc_count;  // escape entries present
    uint32_t n;
    ChunkDiv cdiv;
    uint32_t nchunks;
    uint8_t* y;          // output bit patterns, 16-byte aligned
    uint32_t num_tiles;
    uint32_t cbw[4];
    const uint8_t* dcb = nullptr;  // when not null: the codebook in device memory instead of cbw
};

struct CalibArgs {
    const uint8_t* x;
    uint32_t n;
    uint32_t grid;
    uint8_t* ws;
    uint8_t* cb_out;        // 16 bytes, device
    uint64_t* covered_out;  // device
    uint64_t* hist_out;     // device, 256 (BF16) / 32 (E5M2) counts, or null
};

// Workspace layout of the multi-kernel encode, all offsets from the workspace
// start (256-byte aligned):
//   [0, 4096)            header (WsHeader)
//   states               8 bytes per tile: look-back state words (the single-
//                        launch pipeline)
//   tile_tot             4 bytes per tile: the tile's escape count
//   seg_cnt              32 x uint16 per tile: escapes per segment
//   seg_ent              256 x uint16 per tile: per warp, a list of its first
//                        32 escapes (position in segment | exponent << offset bits)
//   sums                 (right after the header, fixed size) uint32 words of
//                        blocks of kBlockTiles tiles (escape count in the low
//                        kBlkCountShift bits, tiles counted above them), then
//                        escape counts of superblocks of kSuperTiles tiles
//                        (zero between encodes)
constexpr uint32_t kBlockTiles = 64;
constexpr uint32_t kSuperTiles = 4096;
constexpr uint32_t kBlkCountShift = 24;  // a block holds at most 64 x 8192 = 2^19 escapes
constexpr uint32_t kBlkEscMask = (1u << kBlkCountShift) - 1u;
struct MultiLayout {
    size_t states, tile_tot, seg_cnt, seg_ent, sums, bytes;
    uint64_t nblocks, nsupers;
};
MultiLayout multi_layout(uint64_t n);

int encode_tile_elems(bool e5m2);
int decode_tile_elems(bool e5m2);
cudaError_t launch_encode(const EncodeArgs& a, bool e5m2, cudaStream_t s);        // one launch
cudaError_t launch_encode_multi(const EncodeArgs& a, bool e5m2, cudaStream_t s);  // three launches
cudaError_t launch_decode(const DecodeArgs& a, bool e5m2, cudaStream_t s);
cudaError_t launch_calibrate(const CalibArgs& a, bool e5m2, cudaStream_t s);
uint32_t calibrate_grid(uint32_t n, int num_sms);

}  // namespace splitzip
