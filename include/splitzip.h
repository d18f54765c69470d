/*
 * splitzip.h -- C ABI of the GB300 (sm_103a) SplitZip lossless KV-cache codec.
 *
 * The method ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated
 * LLM Serving", project README, sections Abstract, Highlights and FAQ; the
 * arXiv abstract on the paper index page): every BF16 value is split into an
 * exact sign+mantissa byte and an 8-bit exponent; the exponent is mapped
 * through an offline-calibrated top-16 codebook to a fixed 4-bit code; an
 * exponent outside the codebook goes to a chunk-local sparse escape stream of
 * (position, raw exponent); decode unpacks the codes, looks them up, patches
 * the escapes and gives back the bitwise-identical tensor.  The FP8 E5M2
 * variant codes the 5-bit exponent the same way and keeps sign and the 2
 * mantissa bits exact in a packed 3-bit field.
 *
 * Stream format (one encoded tensor of n elements, chunk size `chunk`,
 * C = ceil(n / chunk) chunks, E escapes):
 *   codes      uint8[ceil(n/2)]  4-bit code of element i in byte i/2, low nibble
 *                                for even i; an escaped element stores code 0;
 *                                an odd n leaves the last high nibble 0.
 *   signman    BF16: uint8[n], byte i = sign<<7 | mantissa(7 bits).
 *              E5M2: uint8[ceil(3n/8)], 3-bit field sign<<2 | mantissa(2 bits)
 *                    of element i at bits 3i..3i+2 of a little-endian bit
 *                    stream; padding bits are 0.
 *   esc_pos    uint16[E]  position of the escaped element within its chunk.
 *   esc_val    uint8[E]   its raw exponent.
 *              Escapes are ordered by chunk, then by position (= element order).
 *   chunk_off  uint32[C+1] exclusive prefix of per-chunk escape counts;
 *              chunk_off[C] = E.
 *   codebook   16 distinct exponents; code k stands for exponent exp[k].
 *   compressed size = ceil(n/2) + |signman| + 3E + 4(C+1) bytes (the codebook
 *   is shared codec state, not counted).
 *
 * Ownership and threading: the library allocates nothing.  Every device
 * pointer is caller-owned device memory on the current CUDA device; every
 * call enqueues on the caller's stream (NULL = legacy default stream).  Calls
 * that share a workspace must be ordered on one stream (or otherwise
 * serialised); independent workspaces may run concurrently.
 *
 * Errors: a host-side check that fails returns SPLITZIP_ERR_INVALID_ARG and
 * enqueues nothing.  A CUDA launch or runtime failure returns
 * SPLITZIP_ERR_CUDA.  Conditions found on the device (escape overflow, a
 * bounded wait that gave up) are recorded in the workspace and returned by
 * splitzip_encode_status().  No call ever writes outside the buffers and
 * sizes it is given, whatever the data.
 */
#ifndef SPLITZIP_H
#define SPLITZIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st *splitzip_stream_t;

typedef enum splitzip_status {
    SPLITZIP_OK = 0,
    SPLITZIP_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or codebook */
    SPLITZIP_ERR_ESCAPE_OVERFLOW = 2, /* E > esc_capacity: escapes past capacity dropped */
    SPLITZIP_ERR_TIMEOUT = 3,         /* a bounded device wait gave up: streams invalid */
    SPLITZIP_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed */
    SPLITZIP_ERR_WORKSPACE = 5,       /* workspace not zero-initialised (or overwritten) */
    SPLITZIP_ERR_TOO_LARGE = 6        /* n above SPLITZIP_NOALLOC_MAX_ELEMENTS (no-allocation encode) */
} splitzip_status;

/* Largest chunk size: positions are uint16 within a chunk. */
#define SPLITZIP_MAX_CHUNK 65536u
/* Largest element count: chunk_off entries are uint32. */
#define SPLITZIP_MAX_ELEMENTS 0xFFFFFFFFull

/* The calibrated top-16 codebook: code k stands for raw exponent exp[k].
 * Entries must be distinct (and < 32 for E5M2). */
typedef struct splitzip_codebook {
    uint8_t exp[16];
} splitzip_codebook;

/* One encoded tensor's streams, all caller-owned device memory.
 * codes and signman must be 16-byte aligned, chunk_off 4-byte aligned.
 * esc_pos / esc_val hold esc_capacity entries (may be NULL when 0). */
typedef struct splitzip_streams {
    uint8_t *codes;       /* ceil(n/2) bytes */
    uint8_t *signman;     /* n bytes (BF16) or ceil(3n/8) bytes (E5M2) */
    uint16_t *esc_pos;    /* esc_capacity entries */
    uint8_t *esc_val;     /* esc_capacity entries */
    uint32_t *chunk_off;  /* ceil(n/chunk) + 1 entries */
    uint64_t esc_capacity;
} splitzip_streams;

/* ---------------------------------------------------------------- sizes */

/* Bytes of device workspace needed by calibrate/encode for n elements, about
 * 0.07 bytes per element (per 8192-element tile: a look-back word, an escape
 * count, 32 segment counts and 256 escape entries; escape counts per block of
 * 64 tiles and per superblock of 4096 tiles; independent of the chunk size
 * today -- the argument is kept for later formats).  The workspace must be
 * zero-filled once after allocation (splitzip_workspace_init); the library
 * keeps it consistent afterwards. */
size_t splitzip_workspace_bytes(uint64_t n, uint32_t chunk_size);

/* Zero-fill `bytes` of workspace on stream s (one cudaMemsetAsync). */
splitzip_status splitzip_workspace_init(void *d_workspace, size_t bytes,
                                        splitzip_stream_t s);

/* Stream lengths in bytes (pure host functions). */
uint64_t splitzip_codes_bytes(uint64_t n);
uint64_t splitzip_signman_bytes(uint64_t n);       /* BF16: n */
uint64_t splitzip_signman_bytes_e5m2(uint64_t n);  /* E5M2: ceil(3n/8) */
uint64_t splitzip_num_chunks(uint64_t n, uint32_t chunk_size);

/* Compressed size of an encoded tensor ("compressed_bytes" of the encoded
 * object, README section Codec API): ceil(n/2) + S + 3E + 4(C+1), S = n for
 * BF16 and ceil(3n/8) for E5M2.  Pure host closed form; returns 0 for
 * chunk_size 0. */
uint64_t splitzip_compressed_bytes(uint64_t n, uint32_t chunk_size, uint64_t n_escapes);
uint64_t splitzip_compressed_bytes_e5m2(uint64_t n, uint32_t chunk_size, uint64_t n_escapes);

/* ---------------------------------------------------------- calibration */

/* Offline calibration (the codebook of the 16 most frequent exponents,
 * calibrated ahead of time: arXiv abstract; README sections Highlights and
 * Codec API, where calibrate(x) returns the coverage): histogram the exponents of the n elements at d_x (16-byte
 * aligned bit patterns), pick the 16 most frequent (ties to the smaller
 * exponent; zero-count exponents fill up if fewer than 16 occur), and return
 * the codebook and coverage = (elements whose exponent is in the codebook) / n
 * to HOST memory.  Synchronises stream s.  1 <= n <= SPLITZIP_MAX_ELEMENTS. */
splitzip_status splitzip_calibrate(const void *d_x, uint64_t n,
                                   splitzip_codebook *cb_out, double *coverage_out,
                                   void *d_workspace, splitzip_stream_t s);
splitzip_status splitzip_calibrate_e5m2(const void *d_x, uint64_t n,
                                        splitzip_codebook *cb_out, double *coverage_out,
                                        void *d_workspace, splitzip_stream_t s);

/* Asynchronous calibration into DEVICE memory: d_cb_out receives the 16
 * codebook bytes, d_covered_out (8-byte aligned) the covered element count.
 * Nothing is synchronised. */
splitzip_status splitzip_calibrate_async(const void *d_x, uint64_t n, uint8_t *d_cb_out,
                                         uint64_t *d_covered_out, void *d_workspace,
                                         splitzip_stream_t s);
splitzip_status splitzip_calibrate_async_e5m2(const void *d_x, uint64_t n, uint8_t *d_cb_out,
                                              uint64_t *d_covered_out, void *d_workspace,
                                              splitzip_stream_t s);

/* The exponent histogram of the n elements at d_x (16-byte aligned) into
 * DEVICE memory: d_hist_out (8-byte aligned) receives 256 (BF16) or 32 (E5M2)
 * uint64 counts, bin e = elements whose exponent is e.  The same kernel as
 * calibration (the pages' calibration step starts from this histogram; it
 * also feeds exponent-entropy and top-k coverage reports).  Asynchronous on
 * s; uses the workspace like splitzip_calibrate_async.
 * 1 <= n <= SPLITZIP_MAX_ELEMENTS. */
splitzip_status splitzip_histogram(const void* d_x, uint64_t n, uint64_t* d_hist_out,
                                   void* d_workspace, splitzip_stream_t s);
splitzip_status splitzip_histogram_e5m2(const void* d_x, uint64_t n, uint64_t* d_hist_out,
                                        void* d_workspace, splitzip_stream_t s);

/* --------------------------------------------------------------- encode */

/* Encode n elements at d_x (16-byte aligned; BF16 or E5M2 bit patterns) with
 * codebook *cb (host memory, copied into the launch) into out's streams
 * (README section Abstract; arXiv abstract).  Three kernel launches, enqueued
 * on s; returns without synchronising.  chunk_size: a multiple of 8 in
 * [8, SPLITZIP_MAX_CHUNK].  1 <= n <= SPLITZIP_MAX_ELEMENTS.
 * If E > esc_capacity, the dense streams and chunk_off are still complete and
 * chunk_off[C] = E, the first esc_capacity escapes are stored, and
 * splitzip_encode_status reports SPLITZIP_ERR_ESCAPE_OVERFLOW. */
splitzip_status splitzip_encode(const void *d_x, uint64_t n, uint32_t chunk_size,
                                const splitzip_codebook *cb, const splitzip_streams *out,
                                void *d_workspace, splitzip_stream_t s);
splitzip_status splitzip_encode_e5m2(const void *d_x, uint64_t n, uint32_t chunk_size,
                                     const splitzip_codebook *cb, const splitzip_streams *out,
                                     void *d_workspace, splitzip_stream_t s);

/* splitzip_encode with the codebook in DEVICE memory: d_codebook points to
 * the 16 codebook bytes (4-byte aligned), for example as written by
 * splitzip_calibrate_async on the same stream.  The pages calibrate the
 * codebook ahead of time and keep it as codec state (README sections
 * Highlights and Codec API; arXiv abstract); reading it on the device lets a
 * caller calibrate per tensor or per KV-cache layer and encode right after,
 * with no host round trip.  The bytes are read when the kernels run (the
 * codebook may still be being written by earlier work on s).  Since the host
 * cannot check them, the encode checks them itself: a codebook whose 16
 * entries are not distinct (or, for E5M2, not all below 32) makes
 * splitzip_encode_status report SPLITZIP_ERR_INVALID_ARG, the streams then
 * being invalid (every write still stays inside the given buffers).  Other
 * arguments, results and errors as for splitzip_encode[_e5m2]. */
splitzip_status splitzip_encode_devcb(const void *d_x, uint64_t n, uint32_t chunk_size,
                                      const uint8_t *d_codebook, const splitzip_streams *out,
                                      void *d_workspace, splitzip_stream_t s);
splitzip_status splitzip_encode_devcb_e5m2(const void *d_x, uint64_t n, uint32_t chunk_size,
                                           const uint8_t *d_codebook,
                                           const splitzip_streams *out, void *d_workspace,
                                           splitzip_stream_t s);

/* Synchronise s and report the most recent finished encode on d_workspace:
 * SPLITZIP_OK, SPLITZIP_ERR_ESCAPE_OVERFLOW, SPLITZIP_ERR_INVALID_ARG (a
 * device codebook given to splitzip_encode_devcb[_e5m2] was not valid),
 * SPLITZIP_ERR_TIMEOUT or SPLITZIP_ERR_WORKSPACE (the later codes win; all but
 * the first two mean the streams are invalid).  *n_escapes_out (may be NULL)
 * receives E, the escapes needed. */
splitzip_status splitzip_encode_status(const void *d_workspace, splitzip_stream_t s,
                                       uint64_t *n_escapes_out);

/* --------------------------------------------------------------- decode */

/* Decode in's streams (n elements, chunk_size, codebook *cb) into d_y
 * (16-byte aligned; n BF16 / E5M2 values) -- README sections Codec API and
 * FAQ: the result is bitwise identical to the encoded input.  Needs no
 * workspace; one kernel launch on s, not synchronised.  in->esc_capacity is
 * the number of escape entries present (at least chunk_off[C]).  Escape
 * metadata is bounds-checked: malformed chunk_off / esc_pos entries never
 * cause an out-of-bounds access (the affected values are then unspecified). */
splitzip_status splitzip_decode(const splitzip_streams *in, uint64_t n, uint32_t chunk_size,
                                const splitzip_codebook *cb, void *d_y, splitzip_stream_t s);
splitzip_status splitzip_decode_e5m2(const splitzip_streams *in, uint64_t n,
                                     uint32_t chunk_size, const splitzip_codebook *cb,
                                     void *d_y, splitzip_stream_t s);

/* splitzip_decode with the codebook in DEVICE memory (16 bytes, 4-byte
 * aligned), read when the kernel runs -- the decode side of
 * splitzip_encode_devcb.  The bytes are not checked: with a codebook other
 * than the one the streams were encoded with the values are unspecified, but
 * every access stays inside the given buffers. */
splitzip_status splitzip_decode_devcb(const splitzip_streams *in, uint64_t n, uint32_t chunk_size,
                                      const uint8_t *d_codebook, void *d_y, splitzip_stream_t s);
splitzip_status splitzip_decode_devcb_e5m2(const splitzip_streams *in, uint64_t n,
                                           uint32_t chunk_size, const uint8_t *d_codebook,
                                           void *d_y, splitzip_stream_t s);

/* ------------------------------------------------ encode without workspace */

/* Largest n accepted by splitzip_encode_noalloc (2^31 BF16 elements, 4 GiB). */
#define SPLITZIP_NOALLOC_MAX_ELEMENTS (1ull << 31)

/* BF16 encode for callers that cannot allocate device memory when they encode
 * -- for example a serving engine's KV-transfer hook running while the
 * engine's own memory pool owns the device (a cudaMalloc there may fail or
 * stall every stream), or a plugin that is handed only its input and output
 * buffers.  The method's pages have no counterpart of this entry point.
 *
 * Same streams, arguments and results as splitzip_encode, but no workspace:
 * the scratch lives in a fixed array inside the library (about 2 MiB, held by
 * every GPU that loads the library until the process exits), so n may not
 * exceed SPLITZIP_NOALLOC_MAX_ELEMENTS (SPLITZIP_ERR_TOO_LARGE otherwise).
 * Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current, and once more after the device's context
 * has been reset, e.g. by cudaDeviceReset, since the array may then sit
 * elsewhere); make that first call before any stream capture.  Every call
 * shares the one array, which keeps the last call's contents; each call clears
 * what must start at zero, but calls that overlap on the GPU (different
 * streams or threads) race and must not be issued.
 * d_status_out (4-byte aligned device memory, may be NULL) receives the
 * device-side status bits of this encode once it finishes: 0 = success,
 * bit 0 (1) = escape overflow (E > esc_capacity), bit 1 (2) = a bounded wait
 * gave up (streams invalid), bit 2 (4) = the encode found its scratch state
 * inconsistent (streams invalid; the next call starts clean again).  E is
 * chunk_off[C], as for splitzip_encode. */
splitzip_status splitzip_encode_noalloc(const void *d_x, uint64_t n, uint32_t chunk_size,
                                        const splitzip_codebook *cb,
                                        const splitzip_streams *out, uint32_t *d_status_out,
                                        splitzip_stream_t s);

/* Library version: major*10000 + minor*100 + patch. */
int splitzip_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLITZIP_H */
