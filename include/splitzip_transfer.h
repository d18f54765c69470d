/*
 * splitzip_transfer.h -- portable SplitZip payloads and pipelined transfers
 * between device tensors and host payloads (GB300, sm_103a).
 *
 * The pages describe SplitZip as the codec on the KV-cache transfer path of
 * prefill/decode disaggregated serving ("SplitZip: Ultra-Fast Lossless KV
 * Compression for Disaggregated LLM Serving", README sections Highlights and
 * FAQ; arXiv abstract: compressed KV is transferred instead of raw KV), and
 * list integration-facing codebook and payload metadata on their roadmap
 * (README section Roadmap).  This header gives both:
 *
 *   - a self-describing payload: everything a receiver needs to decode (format,
 *     sizes, codebooks, escape counts, stream offsets) in one host buffer, so
 *     decode needs no live codec state;
 *   - splitzip_encode_to_host / splitzip_decode_from_host, which move a tensor
 *     slice by slice (for a KV cache: layer by layer) between device memory and
 *     a host payload, overlapping the codec kernels with the copies in both
 *     directions.
 *
 * Payload format, version 1 (all integers little-endian; every region starts
 * at a multiple of 16 bytes from the payload start):
 *
 *   offset 0     header, 64 bytes:
 *                  char     magic[8]      "SPLITZIP"
 *                  uint32   version       1
 *                  uint32   format        SPLITZIP_FORMAT_BF16 or _E5M2
 *                  uint64   n             elements of the whole tensor
 *                  uint64   slice_elems   elements per slice (the last may be shorter)
 *                  uint32   num_slices    ceil(n / slice_elems)
 *                  uint32   chunk_size
 *                  uint64   n_escapes     sum of the slices' escape counts
 *                  uint64   total_bytes   bytes of the whole payload
 *   offset 64    slice table, num_slices entries of 48 bytes (splitzip_slice_entry):
 *                  uint64   n             elements of the slice
 *                  uint64   n_escapes     E of the slice
 *                  uint64   off_dense     offset of the slice's dense region
 *                  uint64   off_escapes   offset of the slice's escape region
 *                  uint8    codebook[16]  the slice's codebook
 *   dense regions, slice by slice: codes (ceil(n/2) bytes), signman (n or
 *                ceil(3n/8) bytes), chunk_off ((C+1) x uint32), each region
 *                starting 16-byte aligned, zero padding between them;
 *   escape regions, slice by slice: esc_pos (E x uint16) then esc_val
 *                (E x uint8), the region 16-byte aligned, zero padding after.
 *
 * Each slice is an independently encoded SplitZip tensor in the stream format
 * of splitzip.h (its own chunk_off, escapes in chunk then position order).
 * The dense regions' sizes depend only on n, slice_elems and chunk_size, so a
 * sender can write them as soon as a slice is encoded; the escape regions
 * follow in slice order.
 *
 * Threading and memory: the library allocates no memory.  The transfer calls
 * take caller-owned device scratch (splitzip_transfer_scratch_bytes) and three
 * caller streams; they create and destroy a few CUDA events per call.  Host
 * buffers given to them should be pinned (cudaHostAlloc / cudaHostRegister)
 * for the copies to run asynchronously at full link speed.
 */
#ifndef SPLITZIP_TRANSFER_H
#define SPLITZIP_TRANSFER_H

#include "splitzip.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SPLITZIP_FORMAT_BF16 0u
#define SPLITZIP_FORMAT_E5M2 1u
#define SPLITZIP_PAYLOAD_VERSION 1u
#define SPLITZIP_PAYLOAD_HEADER_BYTES 64u
#define SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES 48u

/* One entry of the slice table, as stored in the payload. */
typedef struct splitzip_slice_entry {
    uint64_t n;
    uint64_t n_escapes;
    uint64_t off_dense;
    uint64_t off_escapes;
    splitzip_codebook cb;
} splitzip_slice_entry;

/* The header fields of a payload, as returned by splitzip_payload_parse. */
typedef struct splitzip_payload_info {
    uint32_t version;
    uint32_t format;
    uint64_t n;
    uint64_t slice_elems;
    uint32_t num_slices;
    uint32_t chunk_size;
    uint64_t n_escapes;
    uint64_t total_bytes;
} splitzip_payload_info;

/* ------------------------------------------------------ payload sizes */

/* Bytes of a payload holding n elements in slices of slice_elems elements
 * with n_escapes escapes in total: header, slice table, dense regions and
 * escape regions (each escape region padded to 16 bytes, so this is an upper
 * bound when the escapes are spread over several slices; exact for one
 * slice).  Returns 0 for invalid arguments. */
uint64_t splitzip_payload_bytes_bound(uint32_t format, uint64_t n, uint32_t chunk_size,
                                      uint64_t slice_elems, uint64_t n_escapes);

/* Parse and validate the header and slice table of a host payload of `bytes`
 * bytes: magic, version, format, chunk size, slice count and sizes, and that
 * every region lies inside the buffer in the layout above.  Fills *info (and,
 * when `entries` is not NULL, up to max_entries slice entries).  Returns
 * SPLITZIP_ERR_INVALID_ARG for anything malformed.  Pure host function. */
splitzip_status splitzip_payload_parse(const void* h_payload, uint64_t bytes,
                                       splitzip_payload_info* info,
                                       splitzip_slice_entry* entries, uint32_t max_entries);

/* ------------------------------------------------- pipelined transfers */

/* Device scratch the transfer calls need for slices of slice_elems elements:
 * three buffer sets, each a raw slice, its streams (escape capacity one per
 * element, so no slice can overflow) and an encode workspace. */
size_t splitzip_transfer_scratch_bytes(uint32_t format, uint64_t slice_elems,
                                       uint32_t chunk_size);

/* Encode the n elements at x slice by slice into the host payload h_payload
 * (capacity payload_capacity bytes; host memory, else SPLITZIP_ERR_INVALID_ARG),
 * writing the whole payload including its header; *payload_bytes receives its
 * size.
 *
 * x: device memory, or host memory (pinned for speed), 16-byte aligned; the
 *    call finds out which with cudaPointerGetAttributes and, for host input,
 *    copies each slice to the device first.
 * cbs: num_cbs codebooks in host memory: 1 (shared by all slices) or one per
 *    slice (for example a codebook calibrated per KV-cache layer); or cbs NULL
 *    and num_cbs 0: every slice is calibrated on the device, right before it
 *    is encoded, on its own elements (splitzip_calibrate_async, then
 *    splitzip_encode_devcb), and the slice table carries the codebook each
 *    slice got.  This is the pages' calibration step (a top-16 codebook fixed
 *    ahead of the encode: README sections Highlights and Codec API) taken per
 *    layer, so that a codebook follows the KV statistics of its own layer
 *    with no host round trip.
 * slice_elems: a multiple of chunk_size and of 16 (so every slice starts on a
 *    chunk and on a 16-byte boundary), at least chunk_size.
 * d_scratch: splitzip_transfer_scratch_bytes(format, slice_elems, chunk_size)
 *    bytes of device memory, 256-byte aligned; its contents on entry do not
 *    matter.
 * s_compute, s_h2d, s_d2h: three distinct streams for the kernels, the
 *    host-to-device copies and the device-to-host copies.
 * The call is synchronous: it returns when the payload is complete.  The host
 * thread waits for each slice's escape count before it places the slice's
 * escapes, while later slices keep the device busy.
 * Errors: SPLITZIP_ERR_INVALID_ARG (arguments), SPLITZIP_ERR_ESCAPE_OVERFLOW
 * (the payload would exceed payload_capacity; *payload_bytes then receives
 * the size needed), SPLITZIP_ERR_TIMEOUT / SPLITZIP_ERR_WORKSPACE (a slice's
 * encode reported it), SPLITZIP_ERR_CUDA. */
splitzip_status splitzip_encode_to_host(const void* x, uint64_t n, uint32_t format,
                                        uint32_t chunk_size, const splitzip_codebook* cbs,
                                        uint32_t num_cbs, uint64_t slice_elems,
                                        void* h_payload, uint64_t payload_capacity,
                                        uint64_t* payload_bytes, void* d_scratch,
                                        size_t scratch_bytes, splitzip_stream_t s_compute,
                                        splitzip_stream_t s_h2d, splitzip_stream_t s_d2h);

/* A CUDA event (a cudaEvent_t). */
typedef struct CUevent_st *splitzip_event_t;

/* splitzip_encode_to_host for a tensor still being written slice by slice (a
 * KV cache produced layer by layer, the pages' producer side of the transfer
 * path): before the call reads slice i -- its host-to-device copy or its
 * encode -- the call's streams wait on slice_ready[i], an event the producer
 * records once slice i is written.  Slices whose events have completed are
 * encoded and copied out while later slices are still being produced.
 * num_events: 0 (slice_ready may then be NULL; the call is exactly
 * splitzip_encode_to_host) or the number of slices, ceil(n / slice_elems).
 * The events are only waited on, never recorded or destroyed.  Each must
 * already be recorded when the call is made (its record enqueued on the
 * producing stream, the work itself may still be pending): as with
 * cudaStreamWaitEvent, the call waits for the work of the event's most recent
 * record at that moment, and a record made later is not seen.  Like
 * splitzip_encode_to_host the call returns once the whole payload is in host
 * memory, so it blocks until every slice's producer work has completed.
 * Other arguments, errors and the payload as for splitzip_encode_to_host. */
splitzip_status splitzip_encode_to_host_events(const void* x, uint64_t n, uint32_t format,
                                               uint32_t chunk_size, const splitzip_codebook* cbs,
                                               uint32_t num_cbs, uint64_t slice_elems,
                                               void* h_payload, uint64_t payload_capacity,
                                               uint64_t* payload_bytes, void* d_scratch,
                                               size_t scratch_bytes, splitzip_stream_t s_compute,
                                               splitzip_stream_t s_h2d, splitzip_stream_t s_d2h,
                                               const splitzip_event_t* slice_ready,
                                               uint32_t num_events);

/* Decode a host payload (as written by splitzip_encode_to_host, `bytes` long,
 * in host memory, else SPLITZIP_ERR_INVALID_ARG) into y: n elements of the payload's format, in device memory or in host
 * memory (pinned for speed), 16-byte aligned.  The payload is validated with
 * splitzip_payload_parse first; n must equal its element count.  Slices are
 * copied to the device, decoded and (for host output) copied back, the three
 * overlapping across slices.  d_scratch as for splitzip_encode_to_host with
 * the payload's slice size.  Synchronous.  The output is bitwise identical to
 * the encoded input. */
splitzip_status splitzip_decode_from_host(const void* h_payload, uint64_t bytes, void* y,
                                          uint64_t n, void* d_scratch, size_t scratch_bytes,
                                          splitzip_stream_t s_compute, splitzip_stream_t s_h2d,
                                          splitzip_stream_t s_d2h);

#ifdef __cplusplus
}
#endif

#endif /* SPLITZIP_TRANSFER_H */
