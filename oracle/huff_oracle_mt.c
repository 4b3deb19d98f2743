/*
 * huff_oracle_mt.c -- the CPU oracle's steps run over several host threads.
 *
 * TEST AND BASELINE INFRASTRUCTURE ONLY, like huff_oracle.c: the GPU
 * library never calls it.  It exists to time the oracle on all of a host's
 * cores beside the pages' own CPU figures ("Lossless Compression for LLM
 * Tensor Incremental Snapshots", English abstract and experiment highlights:
 * byte-grouping plus Huffman on a 16-core CPU), and its payload must be
 * byte-identical to the sequential ref_encode's (the tests check that).
 *
 * The work is split the way that page's key design 3 splits it, into tasks
 * that run in parallel; here a task is a contiguous range of chunks:
 *   encode  1. each chunk's bit count, sum of len[in[i]] (parallel);
 *           2. the exclusive prefix sum of the counts gives off[] (sequential);
 *           3. each chunk appends its codes one bit at a time from off[c],
 *              most significant bit first, as ref_encode does (parallel); a
 *              byte shared with a neighbouring chunk is updated with an
 *              atomic OR, every other byte belongs to one chunk only.
 *   decode  each chunk read one bit at a time from off[c] with the canonical
 *           first_code / first_index test, as ref_decode does (parallel).
 *   histogram, delta and byte planes: element ranges (parallel), per-thread
 *           histograms summed at the end.
 * Code lengths and canonical codes come from huff_oracle.c unchanged.
 *
 * Threads are plain POSIX threads; threads = 1 runs everything on the
 * calling thread.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MT_OK 0
#define MT_ERR_INVALID_ARG (-1)
#define MT_ERR_BUFFER_TOO_SMALL (-2)
#define MT_ERR_SYMBOL_NOT_IN_CODEBOOK (-3)
#define MT_ERR_CORRUPT_STREAM (-4)
#define MT_MAX_THREADS 256

typedef void (*mt_body)(void *ctx, uint64_t lo, uint64_t hi, int t);

typedef struct {
    mt_body fn;
    void *ctx;
    uint64_t lo, hi;
    int t;
} mt_task;

static void *mt_run(void *p)
{
    mt_task *k = (mt_task *)p;
    k->fn(k->ctx, k->lo, k->hi, k->t);
    return NULL;
}

/* fn(ctx, lo, hi, t) over [0, count) cut into `threads` contiguous ranges. */
static int mt_for(uint64_t count, int threads, mt_body fn, void *ctx)
{
    if (threads < 1) threads = 1;
    if (threads > MT_MAX_THREADS) threads = MT_MAX_THREADS;
    if ((uint64_t)threads > count) threads = count ? (int)count : 1;
    mt_task task[MT_MAX_THREADS];
    pthread_t tid[MT_MAX_THREADS];
    for (int t = 0; t < threads; ++t) {
        task[t].fn = fn;
        task[t].ctx = ctx;
        task[t].lo = count * (uint64_t)t / (uint64_t)threads;
        task[t].hi = count * (uint64_t)(t + 1) / (uint64_t)threads;
        task[t].t = t;
    }
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, mt_run, &task[t]) != 0) break;
        started = t;
    }
    mt_run(&task[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    for (int t = started + 1; t < threads; ++t) mt_run(&task[t]); /* threads that could not start */
    return threads;
}

/* ---------------------------------------------------------------- histogram */
typedef struct {
    const uint8_t *in;
    uint64_t (*part)[256];
} hist_ctx;

static void hist_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    hist_ctx *c = (hist_ctx *)p;
    uint64_t *h = c->part[t];
    for (int b = 0; b < 256; ++b) h[b] = 0;
    for (uint64_t i = lo; i < hi; ++i) h[c->in[i]] += 1;
}

int mt_histogram(const uint8_t *in, uint64_t n, uint64_t *hist, int threads)
{
    uint64_t (*part)[256] = calloc(MT_MAX_THREADS, sizeof *part);
    if (!part) return MT_ERR_INVALID_ARG;
    hist_ctx c = {in, part};
    int used = mt_for(n, threads, hist_body, &c);
    for (int b = 0; b < 256; ++b) hist[b] = 0;
    for (int t = 0; t < used; ++t)
        for (int b = 0; b < 256; ++b) hist[b] += part[t][b];
    free(part);
    return MT_OK;
}

/* ---------------------------------------------------------------- delta + byte planes */
typedef struct {
    const uint16_t *a, *b;
    uint8_t *hi, *lo;
    uint16_t *w;
} plane_ctx;

static void split_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    plane_ctx *c = (plane_ctx *)p;
    (void)t;
    for (uint64_t i = lo; i < hi; ++i) {
        uint16_t v = c->b ? (uint16_t)(c->a[i] ^ c->b[i]) : c->a[i];
        c->hi[i] = (uint8_t)(v >> 8);
        c->lo[i] = (uint8_t)(v & 0xffu);
    }
}

/* hi/lo planes of a (XOR b when b is not NULL). */
void mt_delta_split(const uint16_t *a, const uint16_t *b, uint64_t n, uint8_t *hi, uint8_t *lo, int threads)
{
    plane_ctx c = {a, b, hi, lo, NULL};
    mt_for(n, threads, split_body, &c);
}

static void merge_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    plane_ctx *c = (plane_ctx *)p;
    (void)t;
    for (uint64_t i = lo; i < hi; ++i) {
        uint16_t v = (uint16_t)(((uint16_t)c->hi[i] << 8) | c->lo[i]);
        c->w[i] = c->b ? (uint16_t)(v ^ c->b[i]) : v;
    }
}

/* w = (hi << 8 | lo) (XOR b when b is not NULL). */
void mt_merge_xor(const uint8_t *hi, const uint8_t *lo, const uint16_t *b, uint64_t n, uint16_t *w, int threads)
{
    plane_ctx c = {NULL, b, (uint8_t *)hi, (uint8_t *)lo, w};
    mt_for(n, threads, merge_body, &c);
}

/* ---------------------------------------------------------------- encode */
typedef struct {
    const uint8_t *in;
    uint64_t n, chunk, n_chunks;
    const uint8_t *len;
    const uint32_t *code;
    uint64_t *off;
    uint8_t *payload;
    int missing;
} enc_ctx;

static void count_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    enc_ctx *c = (enc_ctx *)p;
    (void)t;
    for (uint64_t ch = lo; ch < hi; ++ch) {
        uint64_t first = ch * c->chunk;
        uint64_t last = first + c->chunk < c->n ? first + c->chunk : c->n;
        uint64_t bits = 0;
        for (uint64_t i = first; i < last; ++i) {
            if (c->len[c->in[i]] == 0) __atomic_store_n(&c->missing, 1, __ATOMIC_RELAXED);
            bits += c->len[c->in[i]];
        }
        c->off[ch] = bits;
    }
}

static void pack_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    enc_ctx *c = (enc_ctx *)p;
    (void)t;
    for (uint64_t ch = lo; ch < hi; ++ch) {
        uint64_t first = ch * c->chunk;
        uint64_t last = first + c->chunk < c->n ? first + c->chunk : c->n;
        uint64_t pos = c->off[ch];
        uint64_t b_first = c->off[ch] / 8, b_last = (c->off[ch + 1] + 7) / 8 - 1;
        for (uint64_t i = first; i < last; ++i) {
            int L = c->len[c->in[i]];
            for (int b = L - 1; b >= 0; --b) {
                if ((c->code[c->in[i]] >> b) & 1u) {
                    uint8_t bit = (uint8_t)(0x80u >> (pos % 8));
                    uint64_t byte = pos / 8;
                    if (byte == b_first || byte == b_last)
                        __atomic_fetch_or(&c->payload[byte], bit, __ATOMIC_RELAXED);
                    else
                        c->payload[byte] |= bit;
                }
                ++pos;
            }
        }
    }
}

/* Same contract as ref_encode; payload byte-identical to it. */
int mt_encode(const uint8_t *in, uint64_t n, const uint8_t *len, const uint32_t *code, uint64_t chunk_bytes,
              uint8_t *payload, uint64_t cap, uint64_t *off, int threads)
{
    if (chunk_bytes == 0) return MT_ERR_INVALID_ARG;
    uint64_t n_chunks = (n + chunk_bytes - 1) / chunk_bytes;
    enc_ctx c = {in, n, chunk_bytes, n_chunks, len, code, off, payload, 0};
    mt_for(n_chunks, threads, count_body, &c);
    if (c.missing) return MT_ERR_SYMBOL_NOT_IN_CODEBOOK;
    uint64_t pos = 0;
    for (uint64_t ch = 0; ch < n_chunks; ++ch) {
        uint64_t bits = off[ch];
        off[ch] = pos;
        pos += bits;
    }
    off[n_chunks] = pos;
    if ((pos + 7) / 8 > cap) return MT_ERR_BUFFER_TOO_SMALL;
    memset(payload, 0, (size_t)cap);
    mt_for(n_chunks, threads, pack_body, &c);
    return MT_OK;
}

/* ---------------------------------------------------------------- decode */
typedef struct {
    const uint8_t *payload;
    uint64_t total_bits;
    const uint64_t *off;
    uint64_t n, chunk;
    uint64_t bl[64], first_code[64], first_index[64];
    uint8_t sorted[256];
    int max_len;
    uint8_t *out;
    int bad;
} dec_ctx;

static void dec_body(void *p, uint64_t lo, uint64_t hi, int t)
{
    dec_ctx *c = (dec_ctx *)p;
    (void)t;
    for (uint64_t ch = lo; ch < hi; ++ch) {
        uint64_t pos = c->off[ch];
        uint64_t first = ch * c->chunk;
        uint64_t count = c->n - first < c->chunk ? c->n - first : c->chunk;
        for (uint64_t i = 0; i < count; ++i) {
            uint64_t cw = 0;
            int L = 0;
            for (;;) {
                if (pos >= c->total_bits || L >= c->max_len) {
                    __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
                    return;
                }
                cw = (cw << 1) | ((c->payload[pos / 8] >> (7 - pos % 8)) & 1u);
                ++pos;
                ++L;
                if (c->bl[L] > 0 && cw >= c->first_code[L] && cw - c->first_code[L] < c->bl[L]) {
                    c->out[first + i] = c->sorted[c->first_index[L] + (cw - c->first_code[L])];
                    break;
                }
            }
        }
        if (pos != c->off[ch + 1]) __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
    }
}

/* Same contract as ref_decode. */
int mt_decode(const uint8_t *payload, uint64_t payload_bytes, const uint64_t *off, uint64_t n, uint64_t chunk_bytes,
              const uint8_t *len, uint8_t *out, int threads)
{
    if (chunk_bytes == 0) return MT_ERR_INVALID_ARG;
    dec_ctx *c = calloc(1, sizeof *c);
    if (!c) return MT_ERR_INVALID_ARG;
    c->payload = payload;
    c->total_bits = payload_bytes * 8;
    c->off = off;
    c->n = n;
    c->chunk = chunk_bytes;
    c->out = out;
    for (int s = 0; s < 256; ++s) {
        c->bl[len[s]] += 1;
        if (len[s] > c->max_len) c->max_len = len[s];
    }
    c->bl[0] = 0;
    uint64_t code = 0, idx = 0;
    for (int L = 1; L < 64; ++L) {
        code = (code + c->bl[L - 1]) << 1;
        c->first_code[L] = code;
        c->first_index[L] = idx;
        idx += c->bl[L];
    }
    int k = 0;
    for (int L = 1; L <= c->max_len; ++L)
        for (int s = 0; s < 256; ++s)
            if (len[s] == L) c->sorted[k++] = (uint8_t)s;
    mt_for((n + chunk_bytes - 1) / chunk_bytes, threads, dec_body, c);
    int st = c->bad ? MT_ERR_CORRUPT_STREAM : MT_OK;
    free(c);
    return st;
}
