// encode_noalloc.cu -- BF16 encode that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they encode: a
// serving engine's KV-transfer hook that runs while the engine's own pool
// owns all of device memory (a cudaMalloc there may fail, or synchronise the
// whole device and stall the decode streams), or a plugin whose host
// framework hands it only the input and output buffers.  For them this entry
// point keeps the encode's scratch (the look-back header and the per-tile
// state words) in a fixed array inside the library instead of in a caller
// workspace.  It runs the same encode kernel as splitzip_encode.
//
// The array is zero at load time and every launch leaves it ready for the
// next one; each call still clears the ticket, done and status words before
// it launches.  All calls share the one array: calls whose work overlaps on
// the GPU (other streams, other host threads) race and must not be issued.
#include <cstdint>
#include <mutex>

#include <cuda.h>  // driver types only: the two driver calls are reached through the runtime

#include "../../include/splitzip.h"
#include "kernels.h"

using namespace splitzip;

namespace {

constexpr uint64_t kNoAllocMaxElements = SPLITZIP_NOALLOC_MAX_ELEMENTS;
constexpr uint64_t kNoAllocTiles = kNoAllocMaxElements / 8192;  // BF16 encode tile
constexpr size_t kNoAllocScratchBytes = kWsStatesOffset + 8 * kNoAllocTiles;

// Every GPU that loads the library holds this array (about 2 MiB) until exit.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Id of the context current on this thread (0 if none is, or if the driver
// does not offer the calls).  The array's device address belongs to one
// context: a device reset makes a new one, in which the array may sit
// elsewhere, so the cached address is keyed on the context's id.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is fetched once
// per device (and again after a device reset), with that device current, and
// cached.
cudaError_t scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_setup_mutex);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // binds the device's context
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" splitzip_status splitzip_encode_noalloc(const void* d_x, uint64_t n,
                                                   uint32_t chunk_size,
                                                   const splitzip_codebook* cb,
                                                   const splitzip_streams* out,
                                                   uint32_t* d_status_out, splitzip_stream_t s) {
    if (n > kNoAllocMaxElements) return SPLITZIP_ERR_TOO_LARGE;
    if (!d_x || !cb || !out || n == 0) return SPLITZIP_ERR_INVALID_ARG;
    if (chunk_size < 8 || chunk_size > SPLITZIP_MAX_CHUNK || chunk_size % 8) return SPLITZIP_ERR_INVALID_ARG;
    if (!out->codes || !out->signman || !out->chunk_off) return SPLITZIP_ERR_INVALID_ARG;
    if (out->esc_capacity && (!out->esc_pos || !out->esc_val)) return SPLITZIP_ERR_INVALID_ARG;
    if (((uintptr_t)d_x & 15) || ((uintptr_t)out->codes & 15) || ((uintptr_t)out->signman & 15) ||
        ((uintptr_t)out->chunk_off & 3) || ((uintptr_t)out->esc_pos & 1) ||
        ((uintptr_t)d_status_out & 3))
        return SPLITZIP_ERR_INVALID_ARG;
    bool seen[256] = {false};
    for (int k = 0; k < 16; k++) {
        if (seen[cb->exp[k]]) return SPLITZIP_ERR_INVALID_ARG;
        seen[cb->exp[k]] = true;
    }

    void* scratch = nullptr;
    cudaStream_t st = (cudaStream_t)s;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return SPLITZIP_ERR_CUDA;
    WsHeader* hdr = static_cast<WsHeader*>(scratch);
    // ticket and done (adjacent), then status; the epoch is left as it is so
    // that state words of earlier calls keep reading as stale.
    if (cudaMemsetAsync(&hdr->ticket, 0, 2 * sizeof(uint32_t), st) != cudaSuccess ||
        cudaMemsetAsync(&hdr->status, 0, sizeof(uint32_t), st) != cudaSuccess)
        return SPLITZIP_ERR_CUDA;

    EncodeArgs a;
    a.x = static_cast<const uint8_t*>(d_x);
    a.n = (uint32_t)n;
    a.cdiv = make_chunk_div(chunk_size);
    a.nchunks = (uint32_t)((n + chunk_size - 1) / chunk_size);
    a.codes = out->codes;
    a.signman = out->signman;
    a.esc_pos = out->esc_pos;
    a.esc_val = out->esc_val;
    a.chunk_off = out->chunk_off;
    a.esc_capacity = out->esc_capacity;
    a.ws = static_cast<uint8_t*>(scratch);
    a.num_tiles = (uint32_t)((n + encode_tile_elems(false) - 1) / encode_tile_elems(false));
    a.spin_limit = kDefaultSpinLimit;
    a.test_flags = 0;
    for (int k = 0; k < 4; k++)
        a.cbw[k] = (uint32_t)cb->exp[4 * k] | ((uint32_t)cb->exp[4 * k + 1] << 8) |
                   ((uint32_t)cb->exp[4 * k + 2] << 16) | ((uint32_t)cb->exp[4 * k + 3] << 24);
    if (launch_encode(a, false, st) != cudaSuccess) return SPLITZIP_ERR_CUDA;
    if (d_status_out &&
        cudaMemcpyAsync(d_status_out, &hdr->last_status, sizeof(uint32_t),
                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return SPLITZIP_ERR_CUDA;
    return SPLITZIP_OK;
}
