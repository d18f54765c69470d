// calibrate.cu -- SplitZip codebook calibration for sm_103a (BF16 and E5M2).
//
// Method: "A calibrated top-16 exponent codebook eliminates online
// histogramming" (arXiv abstract on the paper index page); the codec's
// calibrate(x) returns the coverage ("SplitZip: Ultra-Fast Lossless KV
// Compression for Disaggregated LLM Serving", README section Codec API).
//
// One launch.  Each CTA histograms its grid-stride share of the input into
// per-warp shared-memory bins (one set of 256 counters per warp, so warps do
// not contend), folds them and adds them into the workspace's global
// histogram.  The last CTA to finish (an atomic counter) ranks the bins by
// (count descending, exponent ascending), writes the first 16 as the
// codebook together with the covered count (and, when asked, the whole
// histogram), and zeroes the global histogram for the next launch.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace splitzip {
namespace {

template <bool kE5m2>
__device__ __forceinline__ void count_word(uint32_t* hw, uint32_t w) {
    if (kE5m2) {
#pragma unroll
        for (int b = 0; b < 4; b++) atomicAdd(&hw[(w >> (8 * b + 2)) & 0x1Fu], 1u);
    } else {
        atomicAdd(&hw[(w >> 7) & 0xFFu], 1u);
        atomicAdd(&hw[(w >> 23) & 0xFFu], 1u);
    }
}

template <bool kE5m2>
__global__ void __launch_bounds__(kThreads) calibrate_kernel(const CalibArgs a) {
    __shared__ uint32_t h[kWarps][256];
    __shared__ unsigned long long s_cnt[256];
    __shared__ uint8_t s_cb[16];
    __shared__ uint32_t s_last;

    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    const int tid = threadIdx.x, warp = tid >> 5;
    constexpr uint32_t kPerVec = kE5m2 ? 16u : 8u;  // elements per 16-byte vector
    constexpr int kBins = kE5m2 ? 32 : 256;

    for (int i = tid; i < kWarps * 256; i += kThreads) (&h[0][0])[i] = 0;
    __syncthreads();

    uint32_t* hw = h[warp];
    const uint32_t nvec = a.n / kPerVec;
    const uint32_t stride = a.grid * kThreads;
    uint32_t v = blockIdx.x * kThreads + tid;
    for (; v + stride < nvec; v += 2 * stride) {  // two vectors in flight per thread
        const uint4 p = ld_stream16(a.x + 16ull * v);
        const uint4 q = ld_stream16(a.x + 16ull * (v + stride));
        count_word<kE5m2>(hw, p.x); count_word<kE5m2>(hw, p.y);
        count_word<kE5m2>(hw, p.z); count_word<kE5m2>(hw, p.w);
        count_word<kE5m2>(hw, q.x); count_word<kE5m2>(hw, q.y);
        count_word<kE5m2>(hw, q.z); count_word<kE5m2>(hw, q.w);
    }
    if (v < nvec) {
        const uint4 p = ld_stream16(a.x + 16ull * v);
        count_word<kE5m2>(hw, p.x); count_word<kE5m2>(hw, p.y);
        count_word<kE5m2>(hw, p.z); count_word<kE5m2>(hw, p.w);
    }
    // Elements after the last whole vector (fewer than kPerVec).
    if (blockIdx.x == 0) {
        const uint32_t i = nvec * kPerVec + tid;
        if (tid < (int)kPerVec && i < a.n) {
            const uint32_t e = kE5m2 ? (a.x[i] >> 2) & 0x1Fu
                                     : (reinterpret_cast<const uint16_t*>(a.x)[i] >> 7) & 0xFFu;
            atomicAdd(&hw[e], 1u);
        }
    }
    __syncthreads();

    {
        uint32_t sum = 0;
#pragma unroll
        for (int w = 0; w < kWarps; w++) sum += h[w][tid];
        if (sum) atomicAdd(&hdr->hist[tid], (unsigned long long)sum);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&hdr->cal_done, 1u) == a.grid - 1;
    __syncthreads();
    if (!s_last) return;

    // Last CTA: every other CTA's additions are in the global histogram.
    __threadfence();
    s_cnt[tid] = tid < kBins ? ld_relaxed_gpu(reinterpret_cast<const uint64_t*>(&hdr->hist[tid]))
                             : 0ull;
    __syncthreads();
    if (tid < kBins) {
        const unsigned long long c = s_cnt[tid];
        uint32_t rank = 0;
        for (int b = 0; b < kBins; b++) {
            const unsigned long long o = s_cnt[b];
            rank += (o > c) || (o == c && b < tid);
        }
        if (rank < 16) s_cb[rank] = (uint8_t)tid;
    }
    __syncthreads();
    if (tid < 16) a.cb_out[tid] = s_cb[tid];
    if (a.hist_out && tid < kBins) a.hist_out[tid] = s_cnt[tid];
    if (tid == 0) {
        unsigned long long covered = 0;
        for (int k = 0; k < 16; k++) covered += s_cnt[s_cb[k]];
        *a.covered_out = covered;
    }
    hdr->hist[tid] = 0ull;
    if (tid == 0) hdr->cal_done = 0;
    __threadfence();
}

}  // namespace

uint32_t calibrate_grid(uint32_t n, int num_sms) {
    const uint64_t vecs = (uint64_t)n / 8 + 1;
    const uint64_t want = (vecs + 2 * kThreads - 1) / (2 * kThreads);
    const uint64_t cap = (uint64_t)(num_sms > 0 ? num_sms : 1) * 8;
    return (uint32_t)(want < 1 ? 1 : (want < cap ? want : cap));
}

cudaError_t launch_calibrate(const CalibArgs& a, bool e5m2, cudaStream_t s) {
    if (e5m2)
        calibrate_kernel<true><<<a.grid, kThreads, 0, s>>>(a);
    else
        calibrate_kernel<false><<<a.grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace splitzip
