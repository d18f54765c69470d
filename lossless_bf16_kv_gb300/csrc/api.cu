// api.cu -- the extern "C" entry points of include/splitzip.h: host-side
// argument checks, launch configuration and status mapping.  Every step of
// the codec runs in the kernels of encode.cu, decode.cu and calibrate.cu.
#include <cstdint>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "../../include/splitzip.h"
#include "../../include/splitzip_testing.h"
#include "kernels.h"
#include "trace.h"

using namespace splitzip;

namespace {

int num_sms_current() {
    static std::mutex mu;
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 128) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v;
    }
    std::lock_guard<std::mutex> g(mu);
    if (!cache[dev]) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return cache[dev];
}

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

bool codebook_ok(const splitzip_codebook* cb, bool e5m2) {
    bool seen[256] = {false};
    for (int k = 0; k < 16; k++) {
        const uint8_t e = cb->exp[k];
        if (seen[e] || (e5m2 && e >= 32)) return false;
        seen[e] = true;
    }
    return true;
}

void pack_codebook(const splitzip_codebook* cb, uint32_t (&w)[4]) {
    for (int k = 0; k < 4; k++)
        w[k] = (uint32_t)cb->exp[4 * k] | ((uint32_t)cb->exp[4 * k + 1] << 8) |
               ((uint32_t)cb->exp[4 * k + 2] << 16) | ((uint32_t)cb->exp[4 * k + 3] << 24);
}

bool chunk_ok(uint32_t chunk) {
    return chunk >= 8 && chunk <= SPLITZIP_MAX_CHUNK && chunk % 8 == 0;
}

bool count_ok(uint64_t n) { return n >= 1 && n <= SPLITZIP_MAX_ELEMENTS; }

inline splitzip_status from_cuda(cudaError_t e) {
    return e == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
}

// Exactly one of cb (host memory, checked here) and dcb (device memory, 4-byte
// aligned, checked by the encode itself) gives the codebook.
splitzip_status encode_impl(const void* d_x, uint64_t n, uint32_t chunk,
                            const splitzip_codebook* cb, const uint8_t* dcb,
                            const splitzip_streams* out, void* ws, cudaStream_t s, bool e5m2,
                            uint32_t spin_limit, uint32_t flags) {
    if (!d_x || (!cb == !dcb) || !out || !ws) return SPLITZIP_ERR_INVALID_ARG;
    if (dcb && (!aligned(dcb, 4) || (flags & kTestPipelined))) return SPLITZIP_ERR_INVALID_ARG;
    if (!count_ok(n) || !chunk_ok(chunk)) return SPLITZIP_ERR_INVALID_ARG;
    if (!out->codes || !out->signman || !out->chunk_off) return SPLITZIP_ERR_INVALID_ARG;
    if (out->esc_capacity && (!out->esc_pos || !out->esc_val)) return SPLITZIP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(out->codes, 16) || !aligned(out->signman, 16) ||
        !aligned(out->chunk_off, 4) || !aligned(out->esc_pos, 2) || !aligned(ws, 16))
        return SPLITZIP_ERR_INVALID_ARG;
    if (cb && !codebook_ok(cb, e5m2)) return SPLITZIP_ERR_INVALID_ARG;
    EncodeArgs a;
    a.x = static_cast<const uint8_t*>(d_x);
    a.n = (uint32_t)n;
    a.cdiv = make_chunk_div(chunk);
    a.nchunks = (uint32_t)ceil_div(n, chunk);
    a.codes = out->codes;
    a.signman = out->signman;
    a.esc_pos = out->esc_pos;
    a.esc_val = out->esc_val;
    a.chunk_off = out->chunk_off;
    a.esc_capacity = out->esc_capacity;
    a.ws = static_cast<uint8_t*>(ws);
    a.num_tiles = (uint32_t)ceil_div(n, (uint64_t)encode_tile_elems(e5m2));
    a.spin_limit = spin_limit ? spin_limit : kDefaultSpinLimit;
    a.test_flags = flags;
    if (cb) pack_codebook(cb, a.cbw);
    else a.cbw[0] = a.cbw[1] = a.cbw[2] = a.cbw[3] = 0;
    a.dcb = dcb;
    return from_cuda((flags & kTestPipelined) ? launch_encode(a, e5m2, s)
                                              : launch_encode_multi(a, e5m2, s));
}

// Exactly one of cb (host memory, checked here) and dcb (device memory,
// 4-byte aligned, not checked) gives the codebook.
splitzip_status decode_impl(const splitzip_streams* in, uint64_t n, uint32_t chunk,
                            const splitzip_codebook* cb, const uint8_t* dcb, void* d_y,
                            cudaStream_t s, bool e5m2) {
    if (!in || (!cb == !dcb) || !d_y) return SPLITZIP_ERR_INVALID_ARG;
    if (dcb && !aligned(dcb, 4)) return SPLITZIP_ERR_INVALID_ARG;
    if (!count_ok(n) || !chunk_ok(chunk)) return SPLITZIP_ERR_INVALID_ARG;
    if (!in->codes || !in->signman || !in->chunk_off) return SPLITZIP_ERR_INVALID_ARG;
    if (in->esc_capacity && (!in->esc_pos || !in->esc_val)) return SPLITZIP_ERR_INVALID_ARG;
    if (!aligned(d_y, 16) || !aligned(in->codes, 16) || !aligned(in->signman, 16) ||
        !aligned(in->chunk_off, 4) || !aligned(in->esc_pos, 2))
        return SPLITZIP_ERR_INVALID_ARG;
    if (cb && !codebook_ok(cb, e5m2)) return SPLITZIP_ERR_INVALID_ARG;
    DecodeArgs a;
    a.codes = in->codes;
    a.signman = in->signman;
    a.esc_pos = in->esc_pos;
    a.esc_val = in->esc_val;
    a.chunk_off = in->chunk_off;
    a.esc_count = in->esc_capacity;
    a.n = (uint32_t)n;
    a.cdiv = make_chunk_div(chunk);
    a.nchunks = (uint32_t)ceil_div(n, chunk);
    a.y = static_cast<uint8_t*>(d_y);
    a.num_tiles = (uint32_t)ceil_div(n, (uint64_t)decode_tile_elems(e5m2));
    if (cb) pack_codebook(cb, a.cbw);
    else a.cbw[0] = a.cbw[1] = a.cbw[2] = a.cbw[3] = 0;
    a.dcb = dcb;
    return from_cuda(launch_decode(a, e5m2, s));
}

splitzip_status calibrate_async_impl(const void* d_x, uint64_t n, uint8_t* d_cb,
                                     uint64_t* d_covered, void* ws, cudaStream_t s, bool e5m2) {
    if (!d_x || !d_cb || !d_covered || !ws) return SPLITZIP_ERR_INVALID_ARG;
    if (!count_ok(n)) return SPLITZIP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_covered, 8) || !aligned(ws, 16))
        return SPLITZIP_ERR_INVALID_ARG;
    CalibArgs a;
    a.x = static_cast<const uint8_t*>(d_x);
    a.n = (uint32_t)n;
    a.grid = calibrate_grid((uint32_t)n, num_sms_current());
    a.ws = static_cast<uint8_t*>(ws);
    a.cb_out = d_cb;
    a.covered_out = d_covered;
    a.hist_out = nullptr;
    return from_cuda(launch_calibrate(a, e5m2, s));
}

splitzip_status histogram_impl(const void* d_x, uint64_t n, uint64_t* d_hist, void* ws,
                               cudaStream_t s, bool e5m2) {
    if (!d_x || !d_hist || !ws) return SPLITZIP_ERR_INVALID_ARG;
    if (!count_ok(n)) return SPLITZIP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_hist, 8) || !aligned(ws, 16)) return SPLITZIP_ERR_INVALID_ARG;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    CalibArgs a;
    a.x = static_cast<const uint8_t*>(d_x);
    a.n = (uint32_t)n;
    a.grid = calibrate_grid((uint32_t)n, num_sms_current());
    a.ws = static_cast<uint8_t*>(ws);
    a.cb_out = hdr->cal_cb;  // the codebook and coverage land in the workspace, unused
    a.covered_out = &hdr->cal_covered;
    a.hist_out = d_hist;
    return from_cuda(launch_calibrate(a, e5m2, s));
}

splitzip_status calibrate_sync_impl(const void* d_x, uint64_t n, splitzip_codebook* cb_out,
                                    double* coverage_out, void* ws, cudaStream_t s, bool e5m2) {
    if (!cb_out || !coverage_out || !ws) return SPLITZIP_ERR_INVALID_ARG;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    splitzip_status st = calibrate_async_impl(d_x, n, hdr->cal_cb, &hdr->cal_covered, ws, s, e5m2);
    if (st != SPLITZIP_OK) return st;
    struct {
        uint64_t covered;
        uint8_t cb[16];
    } host;
    static_assert(offsetof(WsHeader, cal_cb) == offsetof(WsHeader, cal_covered) + 8,
                  "readback layout");
    cudaError_t e = cudaMemcpyAsync(&host, &hdr->cal_covered, sizeof(host),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return SPLITZIP_ERR_CUDA;
    std::memcpy(cb_out->exp, host.cb, 16);
    *coverage_out = (double)host.covered / (double)n;
    return SPLITZIP_OK;
}

}  // namespace

extern "C" {

size_t splitzip_workspace_bytes(uint64_t n, uint32_t chunk_size) {
    (void)chunk_size;
    return multi_layout(n).bytes;
}

splitzip_status splitzip_workspace_init(void* d_workspace, size_t bytes, splitzip_stream_t s) {
    if (!d_workspace || bytes < kWsHeaderBytes) return SPLITZIP_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(d_workspace, 0, bytes, (cudaStream_t)s));
}

uint64_t splitzip_codes_bytes(uint64_t n) { return ceil_div(n, 2); }
uint64_t splitzip_signman_bytes(uint64_t n) { return n; }
uint64_t splitzip_signman_bytes_e5m2(uint64_t n) { return ceil_div(3 * n, 8); }
uint64_t splitzip_num_chunks(uint64_t n, uint32_t chunk_size) {
    return chunk_size ? ceil_div(n, chunk_size) : 0;
}

uint64_t splitzip_compressed_bytes(uint64_t n, uint32_t chunk_size, uint64_t n_escapes) {
    if (!chunk_size) return 0;
    return ceil_div(n, 2) + n + 3 * n_escapes + 4 * (ceil_div(n, chunk_size) + 1);
}

uint64_t splitzip_compressed_bytes_e5m2(uint64_t n, uint32_t chunk_size, uint64_t n_escapes) {
    if (!chunk_size) return 0;
    return ceil_div(n, 2) + ceil_div(3 * n, 8) + 3 * n_escapes + 4 * (ceil_div(n, chunk_size) + 1);
}

splitzip_status splitzip_calibrate(const void* d_x, uint64_t n, splitzip_codebook* cb_out,
                                   double* coverage_out, void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_calibrate");
    return calibrate_sync_impl(d_x, n, cb_out, coverage_out, d_workspace, (cudaStream_t)s, false);
}

splitzip_status splitzip_calibrate_e5m2(const void* d_x, uint64_t n, splitzip_codebook* cb_out,
                                        double* coverage_out, void* d_workspace,
                                        splitzip_stream_t s) {
    TraceRange trace("splitzip_calibrate_e5m2");
    return calibrate_sync_impl(d_x, n, cb_out, coverage_out, d_workspace, (cudaStream_t)s, true);
}

splitzip_status splitzip_calibrate_async(const void* d_x, uint64_t n, uint8_t* d_cb_out,
                                         uint64_t* d_covered_out, void* d_workspace,
                                         splitzip_stream_t s) {
    TraceRange trace("splitzip_calibrate_async");
    return calibrate_async_impl(d_x, n, d_cb_out, d_covered_out, d_workspace, (cudaStream_t)s,
                                false);
}

splitzip_status splitzip_calibrate_async_e5m2(const void* d_x, uint64_t n, uint8_t* d_cb_out,
                                              uint64_t* d_covered_out, void* d_workspace,
                                              splitzip_stream_t s) {
    TraceRange trace("splitzip_calibrate_async_e5m2");
    return calibrate_async_impl(d_x, n, d_cb_out, d_covered_out, d_workspace, (cudaStream_t)s,
                                true);
}

splitzip_status splitzip_histogram(const void* d_x, uint64_t n, uint64_t* d_hist_out,
                                   void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_histogram");
    return histogram_impl(d_x, n, d_hist_out, d_workspace, (cudaStream_t)s, false);
}

splitzip_status splitzip_histogram_e5m2(const void* d_x, uint64_t n, uint64_t* d_hist_out,
                                        void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_histogram_e5m2");
    return histogram_impl(d_x, n, d_hist_out, d_workspace, (cudaStream_t)s, true);
}

splitzip_status splitzip_encode(const void* d_x, uint64_t n, uint32_t chunk_size,
                                const splitzip_codebook* cb, const splitzip_streams* out,
                                void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_encode");
    return encode_impl(d_x, n, chunk_size, cb, nullptr, out, d_workspace, (cudaStream_t)s, false,
                       0, 0);
}

splitzip_status splitzip_encode_e5m2(const void* d_x, uint64_t n, uint32_t chunk_size,
                                     const splitzip_codebook* cb, const splitzip_streams* out,
                                     void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_encode_e5m2");
    return encode_impl(d_x, n, chunk_size, cb, nullptr, out, d_workspace, (cudaStream_t)s, true,
                       0, 0);
}

splitzip_status splitzip_encode_test(const void* d_x, uint64_t n, uint32_t chunk_size,
                                     const splitzip_codebook* cb, const splitzip_streams* out,
                                     void* d_workspace, splitzip_stream_t s, int is_e5m2,
                                     const splitzip_encode_test_opts* opts) {
    const uint32_t limit = opts ? opts->spin_limit : 0;
    const uint32_t flags =
        opts ? (opts->flags & (SPLITZIP_TEST_STALL_FIRST_TILE | SPLITZIP_TEST_PIPELINED)) : 0;
    return encode_impl(d_x, n, chunk_size, cb, nullptr, out, d_workspace, (cudaStream_t)s,
                       is_e5m2 != 0, limit, flags);
}

splitzip_status splitzip_encode_status(const void* d_workspace, splitzip_stream_t s,
                                       uint64_t* n_escapes_out) {
    TraceRange trace("splitzip_encode_status");
    if (!d_workspace || !aligned(d_workspace, 16)) return SPLITZIP_ERR_INVALID_ARG;
    const WsHeader* hdr = static_cast<const WsHeader*>(d_workspace);
    struct {
        uint32_t last_status;
        uint32_t cal_done;
        uint64_t last_escapes;
    } host;
    static_assert(offsetof(WsHeader, last_escapes) == offsetof(WsHeader, last_status) + 8,
                  "readback layout");
    cudaError_t e = cudaMemcpyAsync(&host, &hdr->last_status, sizeof(host),
                                    cudaMemcpyDeviceToHost, (cudaStream_t)s);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)s);
    if (e != cudaSuccess) return SPLITZIP_ERR_CUDA;
    if (n_escapes_out) *n_escapes_out = host.last_escapes;
    if (host.last_status & kStatusBadWorkspace) return SPLITZIP_ERR_WORKSPACE;
    if (host.last_status & kStatusTimeout) return SPLITZIP_ERR_TIMEOUT;
    if (host.last_status & kStatusBadCodebook) return SPLITZIP_ERR_INVALID_ARG;
    if (host.last_status & kStatusOverflow) return SPLITZIP_ERR_ESCAPE_OVERFLOW;
    return SPLITZIP_OK;
}

splitzip_status splitzip_decode(const splitzip_streams* in, uint64_t n, uint32_t chunk_size,
                                const splitzip_codebook* cb, void* d_y, splitzip_stream_t s) {
    TraceRange trace("splitzip_decode");
    return decode_impl(in, n, chunk_size, cb, nullptr, d_y, (cudaStream_t)s, false);
}

splitzip_status splitzip_decode_e5m2(const splitzip_streams* in, uint64_t n,
                                     uint32_t chunk_size, const splitzip_codebook* cb, void* d_y,
                                     splitzip_stream_t s) {
    TraceRange trace("splitzip_decode_e5m2");
    return decode_impl(in, n, chunk_size, cb, nullptr, d_y, (cudaStream_t)s, true);
}

splitzip_status splitzip_encode_devcb(const void* d_x, uint64_t n, uint32_t chunk_size,
                                      const uint8_t* d_codebook, const splitzip_streams* out,
                                      void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_encode_devcb");
    return encode_impl(d_x, n, chunk_size, nullptr, d_codebook, out, d_workspace,
                       (cudaStream_t)s, false, 0, 0);
}

splitzip_status splitzip_encode_devcb_e5m2(const void* d_x, uint64_t n, uint32_t chunk_size,
                                           const uint8_t* d_codebook, const splitzip_streams* out,
                                           void* d_workspace, splitzip_stream_t s) {
    TraceRange trace("splitzip_encode_devcb_e5m2");
    return encode_impl(d_x, n, chunk_size, nullptr, d_codebook, out, d_workspace,
                       (cudaStream_t)s, true, 0, 0);
}

splitzip_status splitzip_decode_devcb(const splitzip_streams* in, uint64_t n, uint32_t chunk_size,
                                      const uint8_t* d_codebook, void* d_y, splitzip_stream_t s) {
    TraceRange trace("splitzip_decode_devcb");
    return decode_impl(in, n, chunk_size, nullptr, d_codebook, d_y, (cudaStream_t)s, false);
}

splitzip_status splitzip_decode_devcb_e5m2(const splitzip_streams* in, uint64_t n,
                                           uint32_t chunk_size, const uint8_t* d_codebook,
                                           void* d_y, splitzip_stream_t s) {
    TraceRange trace("splitzip_decode_devcb_e5m2");
    return decode_impl(in, n, chunk_size, nullptr, d_codebook, d_y, (cudaStream_t)s, true);
}

int splitzip_version(void) { return 110; }

}  // extern "C"
