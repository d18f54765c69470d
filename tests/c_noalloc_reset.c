/* c_noalloc_reset.c -- the no-allocation BF16 encode across a device reset,
 * through the C ABI of include/splitzip.h from plain C99.
 *
 *   c_noalloc_reset input.bin codebook.bin chunk out_prefix
 *
 * input.bin: raw BF16 bits; codebook.bin: the 16 codebook bytes.  Encodes the
 * input with splitzip_encode_noalloc, resets the device (cudaDeviceReset ends
 * this process's context, so the library's fixed scratch array is created
 * anew, possibly at another address), and encodes it again.  Writes
 * out_prefix.<round>.{codes,signman,esc_pos,esc_val,chunk_off} for rounds 0
 * and 1 (escapes cut to E entries) and prints "status0=<s> status1=<s>
 * E0=<e> E1=<e>".  Exit status 0 when every call succeeded. */
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

static int dump(const char *prefix, int round, const char *name, const void *d_src, size_t len) {
    char path[4096];
    snprintf(path, sizeof path, "%s.%d.%s", prefix, round, name);
    void *h = malloc(len ? len : 1);
    if (!h) return 1;
    if (len && cudaMemcpy(h, d_src, len, cudaMemcpyDeviceToHost) != cudaSuccess) {
        free(h);
        return 1;
    }
    FILE *f = fopen(path, "wb");
    int bad = !f || (len && fwrite(h, 1, len, f) != len);
    if (f) fclose(f);
    free(h);
    return bad;
}

/* One encode on freshly allocated buffers; fills *status and *E. */
static int one_round(const uint16_t *hx, uint64_t n, uint32_t chunk, const splitzip_codebook *cb,
                     const char *prefix, int round, uint32_t *status, uint32_t *E) {
    const uint64_t C = (n + chunk - 1) / chunk;
    void *dx = NULL, *dcodes = NULL, *dsm = NULL, *dpos = NULL, *dval = NULL, *doff = NULL,
         *dstatus = NULL;
    CK(cudaMalloc(&dx, 2 * n));
    CK(cudaMalloc(&dcodes, (n + 1) / 2));
    CK(cudaMalloc(&dsm, n));
    CK(cudaMalloc(&dpos, 2 * n));
    CK(cudaMalloc(&dval, n));
    CK(cudaMalloc(&doff, 4 * (C + 1)));
    CK(cudaMalloc(&dstatus, 4));
    CK(cudaMemcpy(dx, hx, 2 * n, cudaMemcpyHostToDevice));
    CK(cudaMemset(dstatus, 0xFF, 4));
    splitzip_streams s;
    s.codes = (uint8_t *)dcodes;
    s.signman = (uint8_t *)dsm;
    s.esc_pos = (uint16_t *)dpos;
    s.esc_val = (uint8_t *)dval;
    s.chunk_off = (uint32_t *)doff;
    s.esc_capacity = n;
    splitzip_status st = splitzip_encode_noalloc(dx, n, chunk, cb, &s, (uint32_t *)dstatus, NULL);
    if (st != SPLITZIP_OK) {
        fprintf(stderr, "round %d: splitzip_encode_noalloc returned %d\n", round, (int)st);
        return 3;
    }
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(status, dstatus, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(E, (uint32_t *)doff + C, 4, cudaMemcpyDeviceToHost));
    const uint64_t e = *E < n ? *E : n;
    if (dump(prefix, round, "codes", dcodes, (n + 1) / 2) || dump(prefix, round, "signman", dsm, n) ||
        dump(prefix, round, "esc_pos", dpos, 2 * e) || dump(prefix, round, "esc_val", dval, e) ||
        dump(prefix, round, "chunk_off", doff, 4 * (C + 1)))
        return 4;
    cudaFree(dx);
    cudaFree(dcodes);
    cudaFree(dsm);
    cudaFree(dpos);
    cudaFree(dval);
    cudaFree(doff);
    cudaFree(dstatus);
    return 0;
}

int main(int argc, char **argv) {
    if (argc != 5) {
        fprintf(stderr, "usage: %s input.bin codebook.bin chunk out_prefix\n", argv[0]);
        return 1;
    }
    size_t xlen = 0, cblen = 0;
    uint16_t *hx = (uint16_t *)read_file(argv[1], &xlen);
    uint8_t *hcb = (uint8_t *)read_file(argv[2], &cblen);
    if (!hx || !hcb || cblen != 16 || xlen < 2) {
        fprintf(stderr, "bad input files\n");
        return 1;
    }
    splitzip_codebook cb;
    memcpy(cb.exp, hcb, 16);
    const uint64_t n = xlen / 2;
    const uint32_t chunk = (uint32_t)strtoul(argv[3], NULL, 10);
    uint32_t status[2] = {0, 0}, E[2] = {0, 0};
    int rc = one_round(hx, n, chunk, &cb, argv[4], 0, &status[0], &E[0]);
    if (rc) return rc;
    CK(cudaDeviceReset());
    rc = one_round(hx, n, chunk, &cb, argv[4], 1, &status[1], &E[1]);
    if (rc) return rc;
    printf("status0=%u status1=%u E0=%u E1=%u\n", status[0], status[1], E[0], E[1]);
    free(hx);
    free(hcb);
    return 0;
}
