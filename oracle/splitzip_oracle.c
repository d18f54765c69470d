/*
 * splitzip_oracle.c -- plain, slow, single-threaded CPU oracle of the SplitZip
 * lossless KV-cache codec (BF16 and FP8 E5M2).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline / reference arm load this file's library.
 * It shares no code, header, table or constant with the CUDA library: every
 * step is restated here from the method's description, one element at a time,
 * so that a reader can check it against the pages by eye.
 *
 * Sources (page title, section):
 *  [A]  "SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
 *       Serving" (project README), section Abstract: frequent exponent values
 *       get fixed 4-bit codes, sign and mantissa bits are kept exact, rare
 *       exponent values go to a sparse escape stream.
 *  [H]  same page, section Highlights: offline-calibrated top-16 exponent
 *       codebooks with chunk-local sparse escape metadata.
 *  [API] same page, section Codec API: chunk_size=1024, calibrate(x) returns
 *       coverage, encode/decode round trip is bitwise (int16 views equal),
 *       encoded objects expose compressed_bytes.
 *  [FAQ] same page, section FAQ: sign and mantissa stored unchanged; FP8 E5M2
 *       gives up to 1.14x additional compression.
 *  [ARX] "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
 *       Serving" (paper index page), section Abstract (arXiv): fixed-length
 *       codes for frequent exponents, sparse escape stream of (position,
 *       value), calibrated top-16 exponent codebook, FP8 extension.
 *  [ZS] "ZipServ Guide: Lossless BF16 Compression for Fast LLMs", section
 *       "The Hidden Accuracy Collapse of Quantized Models": BF16 is 1 sign,
 *       8 exponent and 7 mantissa bits (a standard fact, used only for the
 *       field layout).
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of the repository):
 *  R1  code k maps to the k-th most frequent calibration exponent; ties go to
 *      the smaller exponent; all 16 codes name exponents (no in-band escape
 *      code); zero-count exponents fill the codebook if fewer than 16 occur.
 *  R2  an escaped element stores code 0 in the dense code stream.
 *  R3  nibble i of the code stream is byte i/2; even i is the low nibble; an
 *      odd element count leaves the last high nibble 0.
 *  R4  BF16 sign+mantissa byte = sign<<7 | mantissa (7 bits).
 *  R5  E5M2 sign+mantissa field = sign<<2 | mantissa (2 bits), 3 bits per
 *      element, element i at bits 3i..3i+2 of a little-endian bit stream
 *      (8 elements per 3 bytes); the stream is ceil(3n/8) bytes, zero-padded.
 *  R6  the escape stream is two arrays: position within the chunk (uint16)
 *      and raw exponent (uint8); chunks are concatenated in order and each
 *      chunk's escapes are in ascending position order.
 *  R7  chunk metadata is uint32 chunk_off[C+1], C = ceil(n/chunk): the
 *      exclusive prefix of per-chunk escape counts, chunk_off[C] = E.  The
 *      last chunk may be shorter than chunk.
 *  R8  compressed_bytes = ceil(n/2) + S + 3E + 4(C+1), S = n (BF16) or
 *      ceil(3n/8) (E5M2); the 16-entry codebook is shared state, not counted.
 *  R9  special values (zeros, subnormals, infinities, NaNs) are plain bit
 *      patterns; their exponents are ordinary symbols.
 */
#include <stdint.h>
#include <stddef.h>

/* ---------------------------------------------------------------- fields */

/* BF16 bit layout [ZS]: bit 15 sign, bits 14..7 exponent, bits 6..0 mantissa. */
static unsigned bf16_sign(uint16_t u)     { return (u >> 15) & 0x1u; }
static unsigned bf16_exponent(uint16_t u) { return (u >> 7) & 0xFFu; }
static unsigned bf16_mantissa(uint16_t u) { return u & 0x7Fu; }

static uint16_t bf16_assemble(unsigned sign, unsigned exponent, unsigned mantissa)
{
    return (uint16_t)((sign << 15) | (exponent << 7) | mantissa);
}

/* FP8 E5M2 bit layout: bit 7 sign, bits 6..2 exponent, bits 1..0 mantissa. */
static unsigned e5m2_sign(uint8_t u)     { return (u >> 7) & 0x1u; }
static unsigned e5m2_exponent(uint8_t u) { return (u >> 2) & 0x1Fu; }
static unsigned e5m2_mantissa(uint8_t u) { return u & 0x3u; }

static uint8_t e5m2_assemble(unsigned sign, unsigned exponent, unsigned mantissa)
{
    return (uint8_t)((sign << 7) | (exponent << 2) | mantissa);
}

/* ----------------------------------------------------------- small helpers */

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

/* Code of exponent e: the index k with cb[k] == e, or -1 when e is not one of
 * the 16 codebook exponents (an escape).  A plain linear search [A], [ARX]. */
static int codebook_lookup(const uint8_t cb[16], unsigned e)
{
    for (int k = 0; k < 16; k++)
        if (cb[k] == e)
            return k;
    return -1;
}

/* R3: element i's 4-bit code lives in byte i/2, low nibble for even i. */
static void put_nibble(uint8_t *codes, uint64_t i, unsigned code)
{
    if (i % 2 == 0)
        codes[i / 2] = (uint8_t)((codes[i / 2] & 0xF0u) | code);
    else
        codes[i / 2] = (uint8_t)((codes[i / 2] & 0x0Fu) | (code << 4));
}

static unsigned get_nibble(const uint8_t *codes, uint64_t i)
{
    if (i % 2 == 0)
        return codes[i / 2] & 0x0Fu;
    return (codes[i / 2] >> 4) & 0x0Fu;
}

/* R5: element i's 3-bit field occupies bits 3i, 3i+1, 3i+2 of a little-endian
 * bit stream (bit b of the stream is bit b%8 of byte b/8). */
static void put_field3(uint8_t *stream, uint64_t i, unsigned v)
{
    for (unsigned b = 0; b < 3; b++) {
        uint64_t bit = 3 * i + b;
        if ((v >> b) & 1u)
            stream[bit / 8] = (uint8_t)(stream[bit / 8] | (1u << (bit % 8)));
        else
            stream[bit / 8] = (uint8_t)(stream[bit / 8] & ~(1u << (bit % 8)));
    }
}

static unsigned get_field3(const uint8_t *stream, uint64_t i)
{
    unsigned v = 0;
    for (unsigned b = 0; b < 3; b++) {
        uint64_t bit = 3 * i + b;
        v |= ((stream[bit / 8] >> (bit % 8)) & 1u) << b;
    }
    return v;
}

/* ------------------------------------------------------------ calibration */

/* Exponent histogram of a BF16 tensor: hist[b] = #{i : exponent(x_i) = b}. */
void oracle_histogram_bf16(const uint16_t *x, uint64_t n, uint64_t hist[256])
{
    for (int b = 0; b < 256; b++)
        hist[b] = 0;
    for (uint64_t i = 0; i < n; i++)
        hist[bf16_exponent(x[i])]++;
}

/* Exponent histogram of an E5M2 tensor (32 bins). */
void oracle_histogram_e5m2(const uint8_t *x, uint64_t n, uint64_t hist[32])
{
    for (int b = 0; b < 32; b++)
        hist[b] = 0;
    for (uint64_t i = 0; i < n; i++)
        hist[e5m2_exponent(x[i])]++;
}

/* Top-16 codebook from a histogram of nbins bins ([H], [ARX], reading R1):
 * sixteen rounds of "take the unchosen bin with the largest count; on equal
 * counts the smaller exponent".  Returns -1 if nbins < 16. */
int oracle_top16(const uint64_t *hist, int nbins, uint8_t cb[16])
{
    unsigned char chosen[256];
    if (nbins < 16 || nbins > 256)
        return -1;
    for (int b = 0; b < nbins; b++)
        chosen[b] = 0;
    for (int k = 0; k < 16; k++) {
        int best = -1;
        for (int b = 0; b < nbins; b++) {
            if (chosen[b])
                continue;
            if (best < 0 || hist[b] > hist[best])
                best = b; /* strict '>' keeps the smaller exponent on a tie */
        }
        chosen[best] = 1;
        cb[k] = (uint8_t)best;
    }
    return 0;
}

/* Coverage [API]: the fraction of calibration elements whose exponent is in
 * the codebook. */
static double coverage_of(const uint64_t *hist, const uint8_t cb[16], uint64_t n)
{
    uint64_t covered = 0;
    for (int k = 0; k < 16; k++)
        covered += hist[cb[k]];
    return n ? (double)covered / (double)n : 0.0;
}

double oracle_calibrate_bf16(const uint16_t *x, uint64_t n, uint8_t cb[16])
{
    uint64_t hist[256];
    oracle_histogram_bf16(x, n, hist);
    oracle_top16(hist, 256, cb);
    return coverage_of(hist, cb, n);
}

double oracle_calibrate_e5m2(const uint8_t *x, uint64_t n, uint8_t cb[16])
{
    uint64_t hist[32];
    oracle_histogram_e5m2(x, n, hist);
    oracle_top16(hist, 32, cb);
    return coverage_of(hist, cb, n);
}

/* ------------------------------------------------------------------ encode */

/* BF16 encode ([A], [H], [ARX], readings R2-R7).  Walks the chunks in order;
 * within a chunk, element by element: split the fields, write the exact
 * sign+mantissa byte, look the exponent up in the codebook, write the 4-bit
 * code (0 for an escape) and append (position in chunk, raw exponent) to the
 * escape stream for a miss.  Escapes beyond esc_capacity are counted but not
 * stored.  Returns E, the number of escapes the input needs. */
uint64_t oracle_encode_bf16(const uint16_t *x, uint64_t n, uint32_t chunk,
                            const uint8_t cb[16], uint8_t *codes,
                            uint8_t *signman, uint16_t *esc_pos,
                            uint8_t *esc_val, uint64_t esc_capacity,
                            uint32_t *chunk_off)
{
    uint64_t nchunks = ceil_div(n, chunk);
    uint64_t E = 0;
    for (uint64_t b = 0; b < ceil_div(n, 2); b++)
        codes[b] = 0;
    for (uint64_t c = 0; c < nchunks; c++) {
        uint64_t start = c * chunk;
        uint64_t len = (n - start < chunk) ? n - start : chunk;
        chunk_off[c] = (uint32_t)E;
        for (uint64_t p = 0; p < len; p++) {
            uint64_t i = start + p;
            uint16_t u = x[i];
            unsigned e = bf16_exponent(u);
            int code = codebook_lookup(cb, e);
            signman[i] = (uint8_t)((bf16_sign(u) << 7) | bf16_mantissa(u));
            if (code < 0) {
                if (E < esc_capacity) {
                    esc_pos[E] = (uint16_t)p;
                    esc_val[E] = (uint8_t)e;
                }
                E++;
                code = 0;
            }
            put_nibble(codes, i, (unsigned)code);
        }
    }
    chunk_off[nchunks] = (uint32_t)E;
    return E;
}

/* E5M2 encode: the same steps on the 5-bit exponent, with the 3-bit
 * sign+mantissa field packed per reading R5. */
uint64_t oracle_encode_e5m2(const uint8_t *x, uint64_t n, uint32_t chunk,
                            const uint8_t cb[16], uint8_t *codes,
                            uint8_t *signman, uint16_t *esc_pos,
                            uint8_t *esc_val, uint64_t esc_capacity,
                            uint32_t *chunk_off)
{
    uint64_t nchunks = ceil_div(n, chunk);
    uint64_t E = 0;
    for (uint64_t b = 0; b < ceil_div(n, 2); b++)
        codes[b] = 0;
    for (uint64_t b = 0; b < ceil_div(3 * n, 8); b++)
        signman[b] = 0;
    for (uint64_t c = 0; c < nchunks; c++) {
        uint64_t start = c * chunk;
        uint64_t len = (n - start < chunk) ? n - start : chunk;
        chunk_off[c] = (uint32_t)E;
        for (uint64_t p = 0; p < len; p++) {
            uint64_t i = start + p;
            uint8_t u = x[i];
            unsigned e = e5m2_exponent(u);
            int code = codebook_lookup(cb, e);
            put_field3(signman, i, (e5m2_sign(u) << 2) | e5m2_mantissa(u));
            if (code < 0) {
                if (E < esc_capacity) {
                    esc_pos[E] = (uint16_t)p;
                    esc_val[E] = (uint8_t)e;
                }
                E++;
                code = 0;
            }
            put_nibble(codes, i, (unsigned)code);
        }
    }
    chunk_off[nchunks] = (uint32_t)E;
    return E;
}

/* ------------------------------------------------------------------ decode */

/* BF16 decode ([API], [FAQ], [ARX]): per chunk, unpack each code, look up its
 * exponent in the codebook, reassemble sign, exponent and mantissa; then put
 * the raw exponent of every escape of that chunk back at its position.
 * Returns 0, or -1 if the escape metadata points outside the chunk or the
 * escape arrays (the streams are then malformed). */
int oracle_decode_bf16(const uint8_t *codes, const uint8_t *signman,
                       const uint16_t *esc_pos, const uint8_t *esc_val,
                       const uint32_t *chunk_off, uint64_t n, uint32_t chunk,
                       const uint8_t cb[16], uint64_t esc_count, uint16_t *y)
{
    uint64_t nchunks = ceil_div(n, chunk);
    for (uint64_t c = 0; c < nchunks; c++) {
        uint64_t start = c * chunk;
        uint64_t len = (n - start < chunk) ? n - start : chunk;
        for (uint64_t p = 0; p < len; p++) {
            uint64_t i = start + p;
            unsigned e = cb[get_nibble(codes, i)];
            unsigned sm = signman[i];
            y[i] = bf16_assemble((sm >> 7) & 1u, e, sm & 0x7Fu);
        }
        if (chunk_off[c] > chunk_off[c + 1] || chunk_off[c + 1] > esc_count)
            return -1;
        for (uint64_t j = chunk_off[c]; j < chunk_off[c + 1]; j++) {
            uint64_t p = esc_pos[j];
            if (p >= len)
                return -1;
            uint16_t u = y[start + p];
            y[start + p] = bf16_assemble(bf16_sign(u), esc_val[j], bf16_mantissa(u));
        }
    }
    return 0;
}

/* E5M2 decode: as above with the 5-bit exponent and the 3-bit field. */
int oracle_decode_e5m2(const uint8_t *codes, const uint8_t *signman,
                       const uint16_t *esc_pos, const uint8_t *esc_val,
                       const uint32_t *chunk_off, uint64_t n, uint32_t chunk,
                       const uint8_t cb[16], uint64_t esc_count, uint8_t *y)
{
    uint64_t nchunks = ceil_div(n, chunk);
    for (uint64_t c = 0; c < nchunks; c++) {
        uint64_t start = c * chunk;
        uint64_t len = (n - start < chunk) ? n - start : chunk;
        for (uint64_t p = 0; p < len; p++) {
            uint64_t i = start + p;
            unsigned e = cb[get_nibble(codes, i)];
            unsigned f = get_field3(signman, i);
            y[i] = e5m2_assemble((f >> 2) & 1u, e, f & 0x3u);
        }
        if (chunk_off[c] > chunk_off[c + 1] || chunk_off[c + 1] > esc_count)
            return -1;
        for (uint64_t j = chunk_off[c]; j < chunk_off[c + 1]; j++) {
            uint64_t p = esc_pos[j];
            if (p >= len || esc_val[j] > 31)
                return -1;
            uint8_t u = y[start + p];
            y[start + p] = e5m2_assemble(e5m2_sign(u), esc_val[j], e5m2_mantissa(u));
        }
    }
    return 0;
}

/* -------------------------------------------------------- size accounting */

/* Reading R8 of the encoded object's compressed_bytes [API]. */
uint64_t oracle_compressed_bytes_bf16(uint64_t n, uint32_t chunk, uint64_t E)
{
    return ceil_div(n, 2) + n + 3 * E + 4 * (ceil_div(n, chunk) + 1);
}

uint64_t oracle_compressed_bytes_e5m2(uint64_t n, uint32_t chunk, uint64_t E)
{
    return ceil_div(n, 2) + ceil_div(3 * n, 8) + 3 * E + 4 * (ceil_div(n, chunk) + 1);
}
