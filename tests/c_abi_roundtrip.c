/* c_abi_roundtrip.c -- one calibrate / encode / decode round trip through the
 * C ABI of include/splitzip.h alone: plain C99 and the CUDA runtime, no Python
 * between the caller and the library.
 *
 *   c_abi_roundtrip bf16|e5m2 input.bin calib.bin chunk out_prefix
 *
 * input.bin, calib.bin: raw element bits (2 bytes per BF16 value, 1 per E5M2).
 * The codebook is calibrated on calib.bin, input.bin is encoded with it and
 * decoded again.  Writes out_prefix.{cb,codes,signman,esc_pos,esc_val,chunk_off}
 * (the codebook and the streams, escapes cut to E entries) and prints
 * "E=<escapes> bytes=<compressed bytes> coverage=<c> exact=<0|1>".
 * Exit status 0 when every call succeeded and the decode is bit-exact. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "splitzip.h"

#define CK(x)                                                                   \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
            return 2;                                                           \
        }                                                                       \
    } while (0)
#define SZ(x)                                                                   \
    do {                                                                        \
        splitzip_status s_ = (x);                                               \
        if (s_ != SPLITZIP_OK) {                                                \
            fprintf(stderr, "%s: status %d\n", #x, (int)s_);                    \
            return 3;                                                           \
        }                                                                       \
    } while (0)

static void *read_file(const char *path, size_t *len) {
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    fseek(f, 0, SEEK_END);
    long sz = ftell(f);
    fseek(f, 0, SEEK_SET);
    void *p = sz > 0 ? malloc((size_t)sz) : NULL;
    if (p && fread(p, 1, (size_t)sz, f) != (size_t)sz) {
        free(p);
        p = NULL;
    }
    fclose(f);
    *len = p ? (size_t)sz : 0;
    return p;
}

/* Copies `len` bytes from the device and writes them to prefix.name. */
static int dump(const char *prefix, const char *name, const void *d_src, size_t len) {
    char path[4096];
    snprintf(path, sizeof path, "%s.%s", prefix, name);
    void *h = malloc(len ? len : 1);
    if (!h) return 1;
    if (len && cudaMemcpy(h, d_src, len, cudaMemcpyDeviceToHost) != cudaSuccess) {
        free(h);
        return 1;
    }
    FILE *f = fopen(path, "wb");
    int bad = !f || fwrite(h, 1, len, f) != len;
    if (f) fclose(f);
    free(h);
    return bad;
}

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s bf16|e5m2 input.bin calib.bin chunk out_prefix\n", argv[0]);
        return 1;
    }
    const int e5m2 = strcmp(argv[1], "e5m2") == 0;
    const size_t eb = e5m2 ? 1 : 2;
    size_t xbytes = 0, cbytes = 0;
    void *hx = read_file(argv[2], &xbytes), *hc = read_file(argv[3], &cbytes);
    if (!hx || !hc || xbytes % eb || cbytes % eb) {
        fprintf(stderr, "cannot read the inputs\n");
        return 1;
    }
    const uint64_t n = xbytes / eb, nc = cbytes / eb;
    const uint32_t chunk = (uint32_t)strtoul(argv[4], NULL, 10);
    const char *prefix = argv[5];

    cudaStream_t s;
    CK(cudaStreamCreate(&s));
    const size_t wsb = splitzip_workspace_bytes(n > nc ? n : nc, chunk);
    void *dx, *dc, *dy, *ws;
    CK(cudaMalloc(&dx, xbytes));
    CK(cudaMalloc(&dc, cbytes));
    CK(cudaMalloc(&dy, xbytes));
    CK(cudaMalloc(&ws, wsb));
    CK(cudaMemcpy(dx, hx, xbytes, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dc, hc, cbytes, cudaMemcpyHostToDevice));
    SZ(splitzip_workspace_init(ws, wsb, s));

    splitzip_codebook cb;
    double coverage = 0.0;
    if (e5m2) SZ(splitzip_calibrate_e5m2(dc, nc, &cb, &coverage, ws, s));
    else SZ(splitzip_calibrate(dc, nc, &cb, &coverage, ws, s));

    const uint64_t codes_b = splitzip_codes_bytes(n);
    const uint64_t sm_b = e5m2 ? splitzip_signman_bytes_e5m2(n) : splitzip_signman_bytes(n);
    const uint64_t C = splitzip_num_chunks(n, chunk);
    splitzip_streams st;
    st.esc_capacity = n;  /* every element could escape */
    CK(cudaMalloc((void **)&st.codes, codes_b));
    CK(cudaMalloc((void **)&st.signman, sm_b));
    CK(cudaMalloc((void **)&st.esc_pos, 2 * n));
    CK(cudaMalloc((void **)&st.esc_val, n));
    CK(cudaMalloc((void **)&st.chunk_off, 4 * (C + 1)));
    if (e5m2) SZ(splitzip_encode_e5m2(dx, n, chunk, &cb, &st, ws, s));
    else SZ(splitzip_encode(dx, n, chunk, &cb, &st, ws, s));
    uint64_t E = 0;
    SZ(splitzip_encode_status(ws, s, &E));
    if (e5m2) SZ(splitzip_decode_e5m2(&st, n, chunk, &cb, dy, s));
    else SZ(splitzip_decode(&st, n, chunk, &cb, dy, s));
    CK(cudaStreamSynchronize(s));

    void *hy = malloc(xbytes);
    if (!hy) return 1;
    CK(cudaMemcpy(hy, dy, xbytes, cudaMemcpyDeviceToHost));
    const int exact = memcmp(hx, hy, xbytes) == 0;

    char path[4096];
    snprintf(path, sizeof path, "%s.cb", prefix);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(cb.exp, 1, 16, f) != 16) return 1;
    fclose(f);
    if (dump(prefix, "codes", st.codes, codes_b) || dump(prefix, "signman", st.signman, sm_b) ||
        dump(prefix, "esc_pos", st.esc_pos, 2 * E) || dump(prefix, "esc_val", st.esc_val, E) ||
        dump(prefix, "chunk_off", st.chunk_off, 4 * (C + 1)))
        return 1;

    const uint64_t bytes = e5m2 ? splitzip_compressed_bytes_e5m2(n, chunk, E)
                                : splitzip_compressed_bytes(n, chunk, E);
    printf("E=%llu bytes=%llu coverage=%.17g exact=%d\n", (unsigned long long)E,
           (unsigned long long)bytes, coverage, exact);

    cudaFree(st.codes);
    cudaFree(st.signman);
    cudaFree(st.esc_pos);
    cudaFree(st.esc_val);
    cudaFree(st.chunk_off);
    cudaFree(dx);
    cudaFree(dc);
    cudaFree(dy);
    cudaFree(ws);
    cudaStreamDestroy(s);
    free(hx);
    free(hc);
    free(hy);
    return exact ? 0 : 4;
}
