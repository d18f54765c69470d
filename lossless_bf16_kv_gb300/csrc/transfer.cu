// transfer.cu -- portable SplitZip payloads and pipelined device <-> host
// transfers (include/splitzip_transfer.h).
//
// The codec's place in disaggregated serving is the KV-cache transfer between
// the prefill and the decode side ("SplitZip: Ultra-Fast Lossless KV
// Compression for Disaggregated LLM Serving", README sections Highlights and
// FAQ; arXiv abstract).  These calls cut a tensor into slices (a KV cache:
// layer by layer), encode each slice with the codec kernels and move its
// streams into a self-describing host payload while the next slices are being
// encoded -- and the reverse for decode.  All arithmetic of the codec stays in
// the kernels behind splitzip_encode / splitzip_decode; this file is the host
// orchestration: payload layout, copies, events and checks.
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/splitzip.h"
#include "../../include/splitzip_transfer.h"
#include "common.cuh"
#include "trace.h"

namespace {

constexpr char kMagic[8] = {'S', 'P', 'L', 'I', 'T', 'Z', 'I', 'P'};
constexpr int kBuffers = 3;  // buffer sets in the device scratch (three slices in flight)

inline uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
inline uint64_t align16(uint64_t v) { return (v + 15) & ~(uint64_t)15; }
inline uint64_t align256(uint64_t v) { return (v + 255) & ~(uint64_t)255; }

bool format_ok(uint32_t f) { return f == SPLITZIP_FORMAT_BF16 || f == SPLITZIP_FORMAT_E5M2; }
bool chunk_ok(uint32_t c) { return c >= 8 && c <= SPLITZIP_MAX_CHUNK && c % 8 == 0; }
uint64_t elem_bytes(uint32_t f) { return f == SPLITZIP_FORMAT_BF16 ? 2 : 1; }
uint64_t signman_bytes(uint32_t f, uint64_t n) {
    return f == SPLITZIP_FORMAT_BF16 ? n : ceil_div(3 * n, 8);
}

// Offsets of one slice's dense region, relative to the region start.
struct DenseLayout {
    uint64_t codes, signman, chunk_off, bytes;
};
DenseLayout dense_layout(uint32_t f, uint64_t n, uint32_t chunk) {
    DenseLayout d;
    d.codes = 0;
    d.signman = align16(ceil_div(n, 2));
    d.chunk_off = align16(d.signman + signman_bytes(f, n));
    d.bytes = align16(d.chunk_off + 4 * (ceil_div(n, chunk) + 1));
    return d;
}

// The fixed part of a payload: header, slice table and every dense region.
struct PayloadLayout {
    uint32_t slices;
    uint64_t dense_start;   // offset of slice 0's dense region
    uint64_t escape_start;  // offset of slice 0's escape region
};
PayloadLayout payload_layout(uint32_t f, uint64_t n, uint32_t chunk, uint64_t se) {
    PayloadLayout p;
    p.slices = (uint32_t)ceil_div(n, se);
    p.dense_start = align16(SPLITZIP_PAYLOAD_HEADER_BYTES +
                            (uint64_t)p.slices * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES);
    const uint64_t full = n / se, rest = n - full * se;
    p.escape_start = p.dense_start + full * dense_layout(f, se, chunk).bytes +
                     (rest ? dense_layout(f, rest, chunk).bytes : 0);
    return p;
}
uint64_t slice_len(uint64_t n, uint64_t se, uint32_t i) {
    const uint64_t s0 = (uint64_t)i * se;
    return n - s0 < se ? n - s0 : se;
}
uint64_t slice_dense_offset(const PayloadLayout& p, uint32_t f, uint64_t se, uint32_t chunk,
                            uint32_t i) {
    return p.dense_start + (uint64_t)i * dense_layout(f, se, chunk).bytes;  // slices before i are full
}

bool codebook_ok(const splitzip_codebook& cb, uint32_t f) {
    bool seen[256] = {false};
    for (int k = 0; k < 16; k++) {
        const uint8_t e = cb.exp[k];
        if (seen[e] || (f == SPLITZIP_FORMAT_E5M2 && e >= 32)) return false;
        seen[e] = true;
    }
    return true;
}

void put_u32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
void put_u64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get_u32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
uint64_t get_u64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

void write_header(uint8_t* h, uint32_t f, uint64_t n, uint64_t se, uint32_t slices,
                  uint32_t chunk, uint64_t esc, uint64_t total) {
    std::memcpy(h, kMagic, 8);
    put_u32(h + 8, SPLITZIP_PAYLOAD_VERSION);
    put_u32(h + 12, f);
    put_u64(h + 16, n);
    put_u64(h + 24, se);
    put_u32(h + 32, slices);
    put_u32(h + 36, chunk);
    put_u64(h + 40, esc);
    put_u64(h + 48, total);
    put_u64(h + 56, 0);
}
void write_entry(uint8_t* e, const splitzip_slice_entry& s) {
    put_u64(e, s.n);
    put_u64(e + 8, s.n_escapes);
    put_u64(e + 16, s.off_dense);
    put_u64(e + 24, s.off_escapes);
    std::memcpy(e + 32, s.cb.exp, 16);
}

}  // namespace

extern "C" {

uint64_t splitzip_payload_bytes_bound(uint32_t format, uint64_t n, uint32_t chunk_size,
                                      uint64_t slice_elems, uint64_t n_escapes) {
    if (!format_ok(format) || !chunk_ok(chunk_size) || n == 0 || slice_elems == 0) return 0;
    const PayloadLayout p = payload_layout(format, n, chunk_size, slice_elems);
    return p.escape_start + align16(3 * n_escapes) + 16ull * (p.slices - 1);
}

splitzip_status splitzip_payload_parse(const void* h_payload, uint64_t bytes,
                                       splitzip_payload_info* info,
                                       splitzip_slice_entry* entries, uint32_t max_entries) {
    if (!h_payload || !info || bytes < SPLITZIP_PAYLOAD_HEADER_BYTES) return SPLITZIP_ERR_INVALID_ARG;
    const uint8_t* h = static_cast<const uint8_t*>(h_payload);
    if (std::memcmp(h, kMagic, 8) != 0) return SPLITZIP_ERR_INVALID_ARG;
    splitzip_payload_info in;
    in.version = get_u32(h + 8);
    in.format = get_u32(h + 12);
    in.n = get_u64(h + 16);
    in.slice_elems = get_u64(h + 24);
    in.num_slices = get_u32(h + 32);
    in.chunk_size = get_u32(h + 36);
    in.n_escapes = get_u64(h + 40);
    in.total_bytes = get_u64(h + 48);
    if (in.version != SPLITZIP_PAYLOAD_VERSION || !format_ok(in.format) || !chunk_ok(in.chunk_size))
        return SPLITZIP_ERR_INVALID_ARG;
    if (in.n == 0 || in.n > SPLITZIP_MAX_ELEMENTS || in.slice_elems == 0 ||
        in.slice_elems % in.chunk_size != 0 || in.slice_elems % 16 != 0)
        return SPLITZIP_ERR_INVALID_ARG;
    if ((uint64_t)in.num_slices != ceil_div(in.n, in.slice_elems)) return SPLITZIP_ERR_INVALID_ARG;
    if (in.total_bytes > bytes) return SPLITZIP_ERR_INVALID_ARG;
    const PayloadLayout p = payload_layout(in.format, in.n, in.chunk_size, in.slice_elems);
    if (p.escape_start > in.total_bytes) return SPLITZIP_ERR_INVALID_ARG;
    uint64_t esc_off = p.escape_start, esc_sum = 0;
    for (uint32_t i = 0; i < in.num_slices; i++) {
        const uint8_t* e = h + SPLITZIP_PAYLOAD_HEADER_BYTES + (uint64_t)i * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES;
        splitzip_slice_entry s;
        s.n = get_u64(e);
        s.n_escapes = get_u64(e + 8);
        s.off_dense = get_u64(e + 16);
        s.off_escapes = get_u64(e + 24);
        std::memcpy(s.cb.exp, e + 32, 16);
        if (s.n != slice_len(in.n, in.slice_elems, i) || s.n_escapes > s.n) return SPLITZIP_ERR_INVALID_ARG;
        if (s.off_dense != slice_dense_offset(p, in.format, in.slice_elems, in.chunk_size, i))
            return SPLITZIP_ERR_INVALID_ARG;
        if (s.off_escapes != esc_off || !codebook_ok(s.cb, in.format)) return SPLITZIP_ERR_INVALID_ARG;
        esc_off += align16(3 * s.n_escapes);
        esc_sum += s.n_escapes;
        if (esc_off > in.total_bytes) return SPLITZIP_ERR_INVALID_ARG;
        if (entries && i < max_entries) entries[i] = s;
    }
    if (esc_sum != in.n_escapes || esc_off != in.total_bytes) return SPLITZIP_ERR_INVALID_ARG;
    *info = in;
    return SPLITZIP_OK;
}

}  // extern "C"

namespace {

// One buffer set of the device scratch.  Its dense region is laid out like a
// payload slice's dense region (codes, signman, chunk_off at the same
// offsets), so a slice's dense streams cross the link in one copy.
struct BufferSet {
    uint8_t* raw;    // a raw slice (host input / host output staging)
    uint8_t* dense;  // codes, signman, chunk_off as in the payload
    uint8_t* esc;    // encode: esc_pos[se] then esc_val[se]; decode: the payload's escape region
    uint8_t* ws;     // encode workspace
    size_t ws_bytes;
};

struct ScratchLayout {
    size_t raw, dense, esc, ws, ws_bytes, set_bytes;
};
ScratchLayout scratch_layout(uint32_t f, uint64_t se, uint32_t chunk) {
    ScratchLayout L;
    size_t off = 0;
    L.raw = off;    off += align256(se * elem_bytes(f));
    L.dense = off;  off += align256(dense_layout(f, se, chunk).bytes);
    L.esc = off;    off += align256(3 * se);
    L.ws = off;
    L.ws_bytes = splitzip_workspace_bytes(se, chunk);
    off += align256(L.ws_bytes);
    L.set_bytes = off;
    return L;
}
BufferSet buffer_set(uint8_t* base, const ScratchLayout& L, int b) {
    uint8_t* s = base + (size_t)b * L.set_bytes;
    BufferSet B;
    B.raw = s + L.raw;
    B.dense = s + L.dense;
    B.esc = s + L.esc;
    B.ws = s + L.ws;
    B.ws_bytes = L.ws_bytes;
    return B;
}

// True when p is host memory (registered, mapped or plain pageable memory).
bool is_host_pointer(const void* p, bool* ok) {
    cudaPointerAttributes attr;
    const cudaError_t e = cudaPointerGetAttributes(&attr, p);
    *ok = e == cudaSuccess;
    if (!*ok) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeUnregistered;
}

// Events of one call, destroyed on every exit path.
struct Events {
    cudaEvent_t ev[4][kBuffers];
    int made = 0;
    bool create() {
        for (int k = 0; k < 4; k++)
            for (int b = 0; b < kBuffers; b++) {
                if (cudaEventCreateWithFlags(&ev[k][b], cudaEventDisableTiming) != cudaSuccess)
                    return false;
                made++;
            }
        return true;
    }
    ~Events() {
        int m = 0;
        for (int k = 0; k < 4; k++)
            for (int b = 0; b < kBuffers; b++)
                if (m++ < made) cudaEventDestroy(ev[k][b]);
    }
};

splitzip_status finish(cudaStream_t a, cudaStream_t b, cudaStream_t c, splitzip_status st) {
    const cudaError_t e1 = cudaStreamSynchronize(a), e2 = cudaStreamSynchronize(b),
                      e3 = cudaStreamSynchronize(c);
    if (st == SPLITZIP_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess))
        return SPLITZIP_ERR_CUDA;
    return st;
}

}  // namespace

extern "C" {

size_t splitzip_transfer_scratch_bytes(uint32_t format, uint64_t slice_elems, uint32_t chunk_size) {
    if (!format_ok(format) || !chunk_ok(chunk_size) || slice_elems == 0) return 0;
    return (size_t)kBuffers * scratch_layout(format, slice_elems, chunk_size).set_bytes;
}

splitzip_status splitzip_encode_to_host(const void* x, uint64_t n, uint32_t format,
                                        uint32_t chunk_size, const splitzip_codebook* cbs,
                                        uint32_t num_cbs, uint64_t slice_elems,
                                        void* h_payload, uint64_t payload_capacity,
                                        uint64_t* payload_bytes, void* d_scratch,
                                        size_t scratch_bytes, splitzip_stream_t s_compute,
                                        splitzip_stream_t s_h2d, splitzip_stream_t s_d2h) {
    return splitzip_encode_to_host_events(x, n, format, chunk_size, cbs, num_cbs, slice_elems,
                                          h_payload, payload_capacity, payload_bytes, d_scratch,
                                          scratch_bytes, s_compute, s_h2d, s_d2h, nullptr, 0);
}

splitzip_status splitzip_encode_to_host_events(const void* x, uint64_t n, uint32_t format,
                                               uint32_t chunk_size, const splitzip_codebook* cbs,
                                               uint32_t num_cbs, uint64_t slice_elems,
                                               void* h_payload, uint64_t payload_capacity,
                                               uint64_t* payload_bytes, void* d_scratch,
                                               size_t scratch_bytes, splitzip_stream_t s_compute,
                                               splitzip_stream_t s_h2d, splitzip_stream_t s_d2h,
                                               const splitzip_event_t* slice_ready,
                                               uint32_t num_events) {
    splitzip::TraceRange trace("splitzip_encode_to_host");
    if (!x || !h_payload || !payload_bytes || !d_scratch) return SPLITZIP_ERR_INVALID_ARG;
    // No codebooks: every slice is calibrated on the device right before its encode.
    const bool calibrate_slices = cbs == nullptr && num_cbs == 0;
    if (!cbs && !calibrate_slices) return SPLITZIP_ERR_INVALID_ARG;
    if (!format_ok(format) || !chunk_ok(chunk_size) || n == 0 || n > SPLITZIP_MAX_ELEMENTS)
        return SPLITZIP_ERR_INVALID_ARG;
    if (slice_elems < chunk_size || slice_elems % chunk_size || slice_elems % 16)
        return SPLITZIP_ERR_INVALID_ARG;
    const uint32_t S = (uint32_t)ceil_div(n, slice_elems);
    if (!calibrate_slices && num_cbs != 1 && num_cbs != S) return SPLITZIP_ERR_INVALID_ARG;
    if (num_events != 0 && (num_events != S || !slice_ready)) return SPLITZIP_ERR_INVALID_ARG;
    for (uint32_t i = 0; i < num_cbs; i++)
        if (!codebook_ok(cbs[i], format)) return SPLITZIP_ERR_INVALID_ARG;
    if (((uintptr_t)x & 15) || ((uintptr_t)d_scratch & 255)) return SPLITZIP_ERR_INVALID_ARG;
    if (s_compute == s_h2d || s_compute == s_d2h || s_h2d == s_d2h) return SPLITZIP_ERR_INVALID_ARG;
    if (scratch_bytes < splitzip_transfer_scratch_bytes(format, slice_elems, chunk_size))
        return SPLITZIP_ERR_INVALID_ARG;
    bool ok = false;
    const bool host_in = is_host_pointer(x, &ok);
    if (!ok) return SPLITZIP_ERR_INVALID_ARG;
    // The host writes the payload's header, table and padding itself.
    if (!is_host_pointer(h_payload, &ok) || !ok) return SPLITZIP_ERR_INVALID_ARG;

    const cudaStream_t sc = (cudaStream_t)s_compute, sh = (cudaStream_t)s_h2d,
                       sd = (cudaStream_t)s_d2h;
    const uint64_t eb = elem_bytes(format);
    const ScratchLayout SL = scratch_layout(format, slice_elems, chunk_size);
    const PayloadLayout PL = payload_layout(format, n, chunk_size, slice_elems);
    uint8_t* out = static_cast<uint8_t*>(h_payload);
    const bool dense_fits = PL.escape_start <= payload_capacity;
    if (!dense_fits) {
        *payload_bytes = splitzip_payload_bytes_bound(format, n, chunk_size, slice_elems, n);
        return SPLITZIP_ERR_ESCAPE_OVERFLOW;
    }
    Events E;
    if (!E.create()) return SPLITZIP_ERR_CUDA;
    cudaEvent_t* h2d_done = E.ev[0];   // raw slice on the device (host input)
    cudaEvent_t* enc_done = E.ev[1];   // slice encoded
    cudaEvent_t* dense_done = E.ev[2]; // dense streams and status word copied out
    cudaEvent_t* d2h_done = E.ev[3];   // every copy out of the buffer set issued and done

    std::vector<splitzip_slice_entry> table(S);
    // Slice i's device status word is copied into the first bytes of its own
    // slice-table entry (host memory the caller pinned; rewritten at the end),
    // and a codebook calibrated on the device into the entry's codebook field.
    auto status_slot = [&](uint32_t i) {
        return out + SPLITZIP_PAYLOAD_HEADER_BYTES + (uint64_t)i * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES;
    };
    uint64_t esc_off = PL.escape_start, esc_total = 0;
    bool overflow = false;
    splitzip_status st = SPLITZIP_OK;
    uint8_t* scratch = static_cast<uint8_t*>(d_scratch);
    for (int b = 0; b < kBuffers && st == SPLITZIP_OK; b++) {
        const BufferSet B = buffer_set(scratch, SL, b);
        if (splitzip_workspace_init(B.ws, B.ws_bytes, s_compute) != SPLITZIP_OK) st = SPLITZIP_ERR_CUDA;
    }

    // Escapes of slice j: wait for its dense copies (which carry chunk_off, so
    // E = chunk_off[C]), then copy its escape streams to the next free spot.
    auto place_escapes = [&](uint32_t j) -> splitzip_status {
        const int b = (int)(j % kBuffers);
        const BufferSet B = buffer_set(scratch, SL, b);
        if (cudaEventSynchronize(dense_done[b]) != cudaSuccess) return SPLITZIP_ERR_CUDA;
        const uint64_t nj = slice_len(n, slice_elems, j);
        const DenseLayout DL = dense_layout(format, nj, chunk_size);
        const uint64_t dense_off = slice_dense_offset(PL, format, slice_elems, chunk_size, j);
        const uint64_t C = ceil_div(nj, chunk_size);
        // The dense copy carried the device region's padding bytes: zero them.
        uint8_t* dst = out + dense_off;
        const uint64_t cbb = ceil_div(nj, 2), smb = signman_bytes(format, nj), cob = 4 * (C + 1);
        std::memset(dst + cbb, 0, DL.signman - cbb);
        std::memset(dst + DL.signman + smb, 0, DL.chunk_off - DL.signman - smb);
        std::memset(dst + DL.chunk_off + cob, 0, DL.bytes - DL.chunk_off - cob);
        uint32_t ej32;
        std::memcpy(&ej32, out + dense_off + DL.chunk_off + 4 * C, 4);
        uint32_t stj;
        std::memcpy(&stj, status_slot(j), 4);
        if (stj & 2u) return SPLITZIP_ERR_TIMEOUT;
        if (stj & 4u) return SPLITZIP_ERR_WORKSPACE;
        if (stj & 8u) return SPLITZIP_ERR_CUDA;  // cannot happen: calibration yields a valid codebook
        const uint64_t ej = ej32;
        if (ej > nj) return SPLITZIP_ERR_CUDA;  // cannot happen for a finished encode
        table[j].n = nj;
        table[j].n_escapes = ej;
        table[j].off_dense = dense_off;
        table[j].off_escapes = esc_off;
        if (calibrate_slices) std::memcpy(table[j].cb.exp, status_slot(j) + 32, 16);
        else table[j].cb = cbs[num_cbs == 1 ? 0 : j];
        const uint64_t region = align16(3 * ej);
        if (!overflow && esc_off + region <= payload_capacity) {
            if (ej) {
                if (cudaMemcpyAsync(out + esc_off, B.esc, 2 * ej, cudaMemcpyDeviceToHost, sd) != cudaSuccess ||
                    cudaMemcpyAsync(out + esc_off + 2 * ej, B.esc + 2 * slice_elems, ej,
                                    cudaMemcpyDeviceToHost, sd) != cudaSuccess)
                    return SPLITZIP_ERR_CUDA;
            }
            std::memset(out + esc_off + 3 * ej, 0, region - 3 * ej);
        } else {
            overflow = true;
        }
        esc_off += region;
        esc_total += ej;
        if (cudaEventRecord(d2h_done[b], sd) != cudaSuccess) return SPLITZIP_ERR_CUDA;
        return SPLITZIP_OK;
    };

    for (uint32_t i = 0; i < S && st == SPLITZIP_OK; i++) {
        const int b = (int)(i % kBuffers);
        const BufferSet B = buffer_set(scratch, SL, b);
        const uint64_t ni = slice_len(n, slice_elems, i);
        const uint8_t* src = static_cast<const uint8_t*>(x) + (uint64_t)i * slice_elems * eb;
        cudaError_t e = cudaSuccess;
        if (i >= (uint32_t)kBuffers) e = cudaStreamWaitEvent(sc, d2h_done[b], 0);  // streams of b free
        if (e == cudaSuccess && num_events) {  // slice i has been written by its producer
            e = cudaStreamWaitEvent(sc, (cudaEvent_t)slice_ready[i], 0);
            if (e == cudaSuccess && host_in) e = cudaStreamWaitEvent(sh, (cudaEvent_t)slice_ready[i], 0);
        }
        if (host_in) {
            if (e == cudaSuccess && i >= (uint32_t)kBuffers) e = cudaStreamWaitEvent(sh, enc_done[b], 0);
            if (e == cudaSuccess) e = cudaMemcpyAsync(B.raw, src, ni * eb, cudaMemcpyHostToDevice, sh);
            if (e == cudaSuccess) e = cudaEventRecord(h2d_done[b], sh);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, h2d_done[b], 0);
            src = B.raw;
        }
        if (e != cudaSuccess) { st = SPLITZIP_ERR_CUDA; break; }
        const DenseLayout DL = dense_layout(format, ni, chunk_size);
        splitzip_streams ss;
        ss.codes = B.dense + DL.codes;
        ss.signman = B.dense + DL.signman;
        ss.chunk_off = reinterpret_cast<uint32_t*>(B.dense + DL.chunk_off);
        ss.esc_pos = reinterpret_cast<uint16_t*>(B.esc);
        ss.esc_val = B.esc + 2 * slice_elems;
        ss.esc_capacity = ni;
        splitzip::WsHeader* hdr = reinterpret_cast<splitzip::WsHeader*>(B.ws);
        if (calibrate_slices) {
            // The slice's own top-16, left in its workspace header for the encode.
            st = format == SPLITZIP_FORMAT_BF16
                     ? splitzip_calibrate_async(src, ni, hdr->cal_cb, &hdr->cal_covered, B.ws, s_compute)
                     : splitzip_calibrate_async_e5m2(src, ni, hdr->cal_cb, &hdr->cal_covered, B.ws,
                                                     s_compute);
            if (st != SPLITZIP_OK) break;
            st = format == SPLITZIP_FORMAT_BF16
                     ? splitzip_encode_devcb(src, ni, chunk_size, hdr->cal_cb, &ss, B.ws, s_compute)
                     : splitzip_encode_devcb_e5m2(src, ni, chunk_size, hdr->cal_cb, &ss, B.ws, s_compute);
        } else {
            const splitzip_codebook& cb = cbs[num_cbs == 1 ? 0 : i];
            st = format == SPLITZIP_FORMAT_BF16
                     ? splitzip_encode(src, ni, chunk_size, &cb, &ss, B.ws, s_compute)
                     : splitzip_encode_e5m2(src, ni, chunk_size, &cb, &ss, B.ws, s_compute);
        }
        if (st != SPLITZIP_OK) break;
        uint8_t* dst = out + slice_dense_offset(PL, format, slice_elems, chunk_size, i);
        e = cudaEventRecord(enc_done[b], sc);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, enc_done[b], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, B.dense, DL.bytes, cudaMemcpyDeviceToHost, sd);
        if (e == cudaSuccess) e = cudaMemcpyAsync(status_slot(i), &hdr->last_status, 4, cudaMemcpyDeviceToHost, sd);
        if (e == cudaSuccess && calibrate_slices)
            e = cudaMemcpyAsync(status_slot(i) + 32, hdr->cal_cb, 16, cudaMemcpyDeviceToHost, sd);
        if (e == cudaSuccess) e = cudaEventRecord(dense_done[b], sd);
        if (e != cudaSuccess) { st = SPLITZIP_ERR_CUDA; break; }
        if (i >= 1) st = place_escapes(i - 1);
    }
    if (st == SPLITZIP_OK) st = place_escapes(S - 1);
    st = finish(sc, sh, sd, st);
    if (st != SPLITZIP_OK) return st;
    *payload_bytes = esc_off;
    if (overflow) return SPLITZIP_ERR_ESCAPE_OVERFLOW;
    write_header(out, format, n, slice_elems, S, chunk_size, esc_total, esc_off);
    for (uint32_t j = 0; j < S; j++)
        write_entry(out + SPLITZIP_PAYLOAD_HEADER_BYTES + (uint64_t)j * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES, table[j]);
    std::memset(out + SPLITZIP_PAYLOAD_HEADER_BYTES + (uint64_t)S * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES, 0,
                PL.dense_start - SPLITZIP_PAYLOAD_HEADER_BYTES - (uint64_t)S * SPLITZIP_PAYLOAD_SLICE_ENTRY_BYTES);
    return SPLITZIP_OK;
}

}  // extern "C"

extern "C" {

splitzip_status splitzip_decode_from_host(const void* h_payload, uint64_t bytes, void* y,
                                          uint64_t n, void* d_scratch, size_t scratch_bytes,
                                          splitzip_stream_t s_compute, splitzip_stream_t s_h2d,
                                          splitzip_stream_t s_d2h) {
    splitzip::TraceRange trace("splitzip_decode_from_host");
    if (!h_payload || !y || !d_scratch) return SPLITZIP_ERR_INVALID_ARG;
    bool queried = false;  // the host parses the payload: it must be host memory
    if (!is_host_pointer(h_payload, &queried) || !queried) return SPLITZIP_ERR_INVALID_ARG;
    splitzip_payload_info info;
    if (splitzip_payload_parse(h_payload, bytes, &info, nullptr, 0) != SPLITZIP_OK)
        return SPLITZIP_ERR_INVALID_ARG;
    if (info.n != n) return SPLITZIP_ERR_INVALID_ARG;
    std::vector<splitzip_slice_entry> table(info.num_slices);
    if (splitzip_payload_parse(h_payload, bytes, &info, table.data(), info.num_slices) != SPLITZIP_OK)
        return SPLITZIP_ERR_INVALID_ARG;
    const uint32_t f = info.format, chunk = info.chunk_size;
    const uint64_t se = info.slice_elems;
    if (((uintptr_t)y & 15) || ((uintptr_t)d_scratch & 255)) return SPLITZIP_ERR_INVALID_ARG;
    if (s_compute == s_h2d || s_compute == s_d2h || s_h2d == s_d2h) return SPLITZIP_ERR_INVALID_ARG;
    if (scratch_bytes < splitzip_transfer_scratch_bytes(f, se, chunk)) return SPLITZIP_ERR_INVALID_ARG;
    bool ok = false;
    const bool host_out = is_host_pointer(y, &ok);
    if (!ok) return SPLITZIP_ERR_INVALID_ARG;

    const cudaStream_t sc = (cudaStream_t)s_compute, sh = (cudaStream_t)s_h2d,
                       sd = (cudaStream_t)s_d2h;
    const uint64_t eb = elem_bytes(f);
    const ScratchLayout SL = scratch_layout(f, se, chunk);
    const uint8_t* in = static_cast<const uint8_t*>(h_payload);
    uint8_t* scratch = static_cast<uint8_t*>(d_scratch);
    Events E;
    if (!E.create()) return SPLITZIP_ERR_CUDA;
    cudaEvent_t* h2d_done = E.ev[0];  // the slice's streams are on the device
    cudaEvent_t* dec_done = E.ev[1];  // the slice is decoded (its streams are free)
    cudaEvent_t* d2h_done = E.ev[3];  // the decoded slice left the staging buffer

    splitzip_status st = SPLITZIP_OK;
    for (uint32_t i = 0; i < info.num_slices && st == SPLITZIP_OK; i++) {
        const int b = (int)(i % kBuffers);
        const BufferSet B = buffer_set(scratch, SL, b);
        const splitzip_slice_entry& t = table[i];
        const DenseLayout DL = dense_layout(f, t.n, chunk);
        const uint8_t* dense = in + t.off_dense;
        cudaError_t e = cudaSuccess;
        if (i >= (uint32_t)kBuffers) e = cudaStreamWaitEvent(sh, dec_done[b], 0);  // streams of b free
        if (e == cudaSuccess) e = cudaMemcpyAsync(B.dense, dense, DL.bytes, cudaMemcpyHostToDevice, sh);
        if (e == cudaSuccess && t.n_escapes)
            e = cudaMemcpyAsync(B.esc, in + t.off_escapes, 3 * t.n_escapes, cudaMemcpyHostToDevice, sh);
        if (e == cudaSuccess) e = cudaEventRecord(h2d_done[b], sh);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, h2d_done[b], 0);
        if (e == cudaSuccess && host_out && i >= (uint32_t)kBuffers) e = cudaStreamWaitEvent(sc, d2h_done[b], 0);
        if (e != cudaSuccess) { st = SPLITZIP_ERR_CUDA; break; }
        splitzip_streams ss;
        ss.codes = B.dense + DL.codes;
        ss.signman = B.dense + DL.signman;
        ss.chunk_off = reinterpret_cast<uint32_t*>(B.dense + DL.chunk_off);
        ss.esc_pos = reinterpret_cast<uint16_t*>(B.esc);
        ss.esc_val = B.esc + 2 * t.n_escapes;
        ss.esc_capacity = t.n_escapes;
        uint8_t* dst = host_out ? B.raw : static_cast<uint8_t*>(y) + (uint64_t)i * se * eb;
        st = f == SPLITZIP_FORMAT_BF16 ? splitzip_decode(&ss, t.n, chunk, &t.cb, dst, s_compute)
                                       : splitzip_decode_e5m2(&ss, t.n, chunk, &t.cb, dst, s_compute);
        if (st != SPLITZIP_OK) break;
        e = cudaEventRecord(dec_done[b], sc);
        if (e == cudaSuccess && host_out) {
            e = cudaStreamWaitEvent(sd, dec_done[b], 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(static_cast<uint8_t*>(y) + (uint64_t)i * se * eb, B.raw, t.n * eb,
                                    cudaMemcpyDeviceToHost, sd);
            if (e == cudaSuccess) e = cudaEventRecord(d2h_done[b], sd);
        }
        if (e != cudaSuccess) st = SPLITZIP_ERR_CUDA;
    }
    return finish(sc, sh, sd, st);
}

}  // extern "C"
