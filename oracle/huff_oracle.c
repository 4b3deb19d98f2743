/*
 * huff_oracle.c -- plain, slow, sequential CPU oracle for canonical Huffman
 * coding of ML tensor bytes.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent yardstick that the
 * GPU library is compared against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it follows (sources, by page title and section):
 *   [P1] "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
 *        Methodology steps 1-4: count 8-bit symbol frequencies over warm-up
 *        batches, average them, build one Huffman codebook once, then encode
 *        every later tensor with that codebook alone.
 *   [P2] "Lossless Compression for LLM Tensor Incremental Snapshots"
 *        (arXiv 2505.09810), Method details / technical framework and the
 *        English abstract: byte-grouping of bf16 tensors, frequency statistics
 *        per byte group, Huffman tree and encode per group, and the reverse
 *        for decompression; incremental delta between snapshots.
 *   [RFC1951] DEFLATE specification section 3.2.2: canonical code assignment
 *        from code lengths (the pages do not say how codes are assigned; the
 *        canonical form is the plainest reading that lets a codebook travel
 *        as its 256 lengths only, which is the point of P1's fixed codebook).
 *   [T81] ITU-T T.81 (JPEG) Annex K.3, procedure Adjust_BITS, without its
 *        reserved-code step: the stated rule used to limit lengths to max_len.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - tie-break: nodes are compared by (count, id); leaves have id = symbol,
 *     internal nodes get ids 256, 257, ... in creation order;
 *   - HUFF_COVER_ALL raises zero counts to one before the tree is built;
 *   - bits are appended most-significant-bit first: stream bit k is bit
 *     7 - (k mod 8) of byte k / 8; pad bits are zero; chunks are not padded;
 *   - the delta operator is XOR of the 16-bit patterns; the byte groups of a
 *     little-endian bf16 word are hi = w >> 8 and lo = w & 0xff.
 *
 * Every routine is written as the textbook definition, step by step, with
 * bit-at-a-time loops; nothing is blocked, fused or reordered for speed.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#define REF_OK 0
#define REF_ERR_INVALID_ARG (-1)
#define REF_ERR_BUFFER_TOO_SMALL (-2)
#define REF_ERR_SYMBOL_NOT_IN_CODEBOOK (-3)
#define REF_ERR_CORRUPT_STREAM (-4)

#define REF_COVER_ALL 1u
#define REF_MAX_DEPTH 512

/* ------------------------------------------------------------------------ */
/* C1  Histogram [P1 Methodology step 1; P2 framework stage 2].             */
/* hist[b] = number of i < n with in[i * stride] == b.  int8 data is read   */
/* as its two's-complement byte.                                            */
/* ------------------------------------------------------------------------ */
void ref_histogram(const uint8_t *in, uint64_t n, uint64_t stride, uint64_t *hist)
{
    for (int b = 0; b < 256; ++b) hist[b] = 0;
    for (uint64_t i = 0; i < n; ++i) hist[in[i * stride]] += 1;
}

/* ------------------------------------------------------------------------ */
/* C3 + C4  Code lengths [P1 Methodology step 3; P2 key design 2].          */
/*                                                                          */
/* C3: Huffman's procedure written as its definition: while more than one   */
/* node is active, remove the smallest node by (count, id), then the next   */
/* smallest, and join them under a new node whose count is their sum.  The  */
/* length of a symbol is the depth of its leaf.                             */
/*                                                                          */
/* C4: if some depth exceeds max_len, move leaves up with the Adjust_BITS   */
/* procedure of [T81] (largest over-long depth first); each move keeps the  */
/* Kraft sum at exactly one.  Then, always, hand the lengths out again:     */
/* sort the present symbols by (count descending, symbol ascending) and     */
/* give the first bl_count[1] of them length 1, the next bl_count[2]        */
/* length 2, and so on.                                                     */
/*                                                                          */
/* max_len may be 1..63 here (the GPU library accepts 8..24); the test      */
/* suite uses small limits on tiny alphabets and large ones to see the      */
/* unlimited depths.  Returns REF_ERR_INVALID_ARG when 2^max_len is smaller */
/* than the number of present symbols.                                      */
/* ------------------------------------------------------------------------ */
int ref_code_lengths(const uint64_t *hist, int max_len, unsigned flags, uint8_t *len)
{
    uint64_t count[512];
    int parent[512];
    int active[512];
    int n_nodes = 256;
    int m = 0;

    if (max_len < 1 || max_len > 63) return REF_ERR_INVALID_ARG;

    for (int s = 0; s < 256; ++s) {
        count[s] = hist[s];
        if ((flags & REF_COVER_ALL) && count[s] == 0) count[s] = 1;
        active[s] = count[s] > 0;
        parent[s] = -1;
        len[s] = 0;
        if (active[s]) ++m;
    }
    if (m == 0) return REF_OK;                       /* C5: empty codebook  */
    {   /* node counts are sums of leaf counts: the total must stay below 2^63 */
        uint64_t total = 0;
        for (int s = 0; s < 256; ++s) {
            if (total + count[s] < total) return REF_ERR_INVALID_ARG;
            total += count[s];
        }
        if (total >= ((uint64_t)1 << 63)) return REF_ERR_INVALID_ARG;
    }
    if (max_len < 9 && (uint64_t)m > ((uint64_t)1 << max_len))
        return REF_ERR_INVALID_ARG;                  /* no prefix code fits */
    if (m == 1) {                                    /* C5: one symbol      */
        for (int s = 0; s < 256; ++s) if (active[s]) len[s] = 1;
        return REF_OK;
    }

    /* C3: m - 1 joins, each of the two smallest active nodes by (count, id). */
    for (int step = 0; step < m - 1; ++step) {
        int pick[2];
        for (int k = 0; k < 2; ++k) {
            int best = -1;
            for (int v = 0; v < n_nodes; ++v) {
                if (!active[v]) continue;
                if (best < 0 || count[v] < count[best] ||
                    (count[v] == count[best] && v < best))
                    best = v;
            }
            active[best] = 0;
            pick[k] = best;
        }
        count[n_nodes] = count[pick[0]] + count[pick[1]];
        parent[n_nodes] = -1;
        active[n_nodes] = 1;
        parent[pick[0]] = n_nodes;
        parent[pick[1]] = n_nodes;
        ++n_nodes;
    }

    /* Depth of each leaf = number of parent links up to the root. */
    int depth[256];
    int bl_count[REF_MAX_DEPTH];
    for (int d = 0; d < REF_MAX_DEPTH; ++d) bl_count[d] = 0;
    int max_depth = 0;
    for (int s = 0; s < 256; ++s) {
        depth[s] = 0;
        if (count[s] == 0) continue;
        int d = 0;
        for (int v = s; parent[v] >= 0; v = parent[v]) ++d;
        depth[s] = d;
        bl_count[d] += 1;
        if (d > max_depth) max_depth = d;
    }

    /* C4: Adjust_BITS, largest over-long depth first. */
    for (int i = max_depth; i > max_len; --i) {
        while (bl_count[i] > 0) {
            int j = i - 2;
            while (j > 0 && bl_count[j] == 0) --j;
            if (j <= 0) return REF_ERR_INVALID_ARG;  /* cannot happen when 2^max_len >= m */
            bl_count[i] -= 2;
            bl_count[i - 1] += 1;
            bl_count[j + 1] += 2;
            bl_count[j] -= 1;
        }
    }

    /* C4 step 3: reassign lengths by (count desc, symbol asc). */
    int order[256];
    int k = 0;
    for (int s = 0; s < 256; ++s) if (count[s] > 0) order[k++] = s;
    /* plain insertion sort on (count desc, symbol asc) */
    for (int a = 1; a < k; ++a) {
        int s = order[a];
        int b = a - 1;
        while (b >= 0 && (count[order[b]] < count[s] ||
                          (count[order[b]] == count[s] && order[b] > s))) {
            order[b + 1] = order[b];
            --b;
        }
        order[b + 1] = s;
    }
    int pos = 0;
    for (int L = 1; L <= max_len; ++L)
        for (int c = 0; c < bl_count[L]; ++c) len[order[pos++]] = (uint8_t)L;
    (void)depth;
    return pos == m ? REF_OK : REF_ERR_INVALID_ARG;
}

/* ------------------------------------------------------------------------ */
/* C6  Canonical codes [RFC1951 3.2.2].  bl[L] = number of symbols of      */
/* length L; next[1] = 0, next[L] = (next[L-1] + bl[L-1]) << 1; then each   */
/* symbol, in ascending order, takes next[len]++.  Returns                  */
/* REF_ERR_INVALID_ARG when the lengths over-subscribe the code space.      */
/* ------------------------------------------------------------------------ */
int ref_canonical_codes(const uint8_t *len, uint32_t *code)
{
    uint64_t bl[64];
    uint64_t next[64];
    for (int L = 0; L < 64; ++L) bl[L] = 0;
    for (int s = 0; s < 256; ++s) {
        if (len[s] > 32) return REF_ERR_INVALID_ARG;
        bl[len[s]] += 1;
    }
    bl[0] = 0;
    uint64_t c = 0;
    next[0] = 0;
    for (int L = 1; L <= 32; ++L) {
        c = (c + bl[L - 1]) << 1;
        next[L] = c;
        if (bl[L] > 0 && next[L] + bl[L] > ((uint64_t)1 << L)) return REF_ERR_INVALID_ARG;
    }
    for (int s = 0; s < 256; ++s) {
        code[s] = 0;
        if (len[s] == 0) continue;
        code[s] = (uint32_t)next[len[s]];
        next[len[s]] += 1;
    }
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* C7  Encode [P1 Methodology step 4; P2 framework stage 3].  Append each   */
/* symbol's code, most significant bit first, one bit at a time.  off[c]   */
/* is the bit position before symbol c * chunk_bytes; off[n_chunks] = T.    */
/* The payload must hold ceil(T/8) bytes; it is zeroed up to cap first.     */
/* ------------------------------------------------------------------------ */
int ref_encode(const uint8_t *in, uint64_t n, const uint8_t *len, const uint32_t *code,
               uint64_t chunk_bytes, uint8_t *payload, uint64_t cap, uint64_t *off)
{
    if (chunk_bytes == 0) return REF_ERR_INVALID_ARG;
    uint64_t n_chunks = (n + chunk_bytes - 1) / chunk_bytes;
    memset(payload, 0, (size_t)cap);
    uint64_t pos = 0;
    for (uint64_t i = 0; i < n; ++i) {
        if (i % chunk_bytes == 0) off[i / chunk_bytes] = pos;
        int L = len[in[i]];
        if (L == 0) return REF_ERR_SYMBOL_NOT_IN_CODEBOOK;
        for (int b = L - 1; b >= 0; --b) {
            if (pos / 8 >= cap) return REF_ERR_BUFFER_TOO_SMALL;
            if ((code[in[i]] >> b) & 1u) payload[pos / 8] |= (uint8_t)(0x80u >> (pos % 8));
            ++pos;
        }
    }
    off[n_chunks] = pos;
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* C8  Decode [P2 framework, decompression: read, Huffman-decode, restore]. */
/* Per chunk, from off[c]: read one bit at a time into (code, L) and accept */
/* when first_code[L] <= code < first_code[L] + bl[L]; the symbol is the    */
/* (code - first_code[L])-th symbol of length L in ascending order.  The    */
/* chunk must end exactly at off[c + 1].                                    */
/* ------------------------------------------------------------------------ */
int ref_decode(const uint8_t *payload, uint64_t payload_bytes, const uint64_t *off,
               uint64_t n, uint64_t chunk_bytes, const uint8_t *len, uint8_t *out)
{
    if (chunk_bytes == 0) return REF_ERR_INVALID_ARG;
    uint64_t bl[64], first_code[64], first_index[64];
    uint8_t sorted_symbols[256];
    int max_len = 0;
    for (int L = 0; L < 64; ++L) bl[L] = 0;
    for (int s = 0; s < 256; ++s) {
        bl[len[s]] += 1;
        if (len[s] > max_len) max_len = len[s];
    }
    bl[0] = 0;
    uint64_t c = 0, idx = 0;
    for (int L = 1; L < 64; ++L) {
        c = (c + bl[L - 1]) << 1;
        first_code[L] = c;
        first_index[L] = idx;
        idx += bl[L];
    }
    int k = 0;
    for (int L = 1; L <= max_len; ++L)
        for (int s = 0; s < 256; ++s)
            if (len[s] == L) sorted_symbols[k++] = (uint8_t)s;

    uint64_t n_chunks = (n + chunk_bytes - 1) / chunk_bytes;
    uint64_t total_bits = payload_bytes * 8;
    for (uint64_t ch = 0; ch < n_chunks; ++ch) {
        uint64_t pos = off[ch];
        uint64_t first = ch * chunk_bytes;
        uint64_t count = n - first < chunk_bytes ? n - first : chunk_bytes;
        for (uint64_t i = 0; i < count; ++i) {
            uint64_t cw = 0;
            int L = 0;
            for (;;) {
                if (pos >= total_bits) return REF_ERR_CORRUPT_STREAM;
                cw = (cw << 1) | ((payload[pos / 8] >> (7 - pos % 8)) & 1u);
                ++pos;
                ++L;
                if (L > max_len) return REF_ERR_CORRUPT_STREAM;
                if (bl[L] > 0 && cw >= first_code[L] && cw - first_code[L] < bl[L]) {
                    out[first + i] = sorted_symbols[first_index[L] + (cw - first_code[L])];
                    break;
                }
            }
        }
        if (pos != off[ch + 1]) return REF_ERR_CORRUPT_STREAM;
    }
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* C9  Byte grouping and delta [P2 framework stage 1 "byte grouping"; P2    */
/* English abstract "incremental delta compression"].                       */
/* ------------------------------------------------------------------------ */
void ref_bytegroup_split(const uint16_t *w, uint64_t n, uint8_t *hi, uint8_t *lo)
{
    for (uint64_t i = 0; i < n; ++i) {
        hi[i] = (uint8_t)(w[i] >> 8);
        lo[i] = (uint8_t)(w[i] & 0xffu);
    }
}

void ref_bytegroup_merge(const uint8_t *hi, const uint8_t *lo, uint64_t n, uint16_t *w)
{
    for (uint64_t i = 0; i < n; ++i) w[i] = (uint16_t)(((uint16_t)hi[i] << 8) | lo[i]);
}

void ref_delta_xor(const uint16_t *a, const uint16_t *b, uint64_t n, uint16_t *out)
{
    for (uint64_t i = 0; i < n; ++i) out[i] = (uint16_t)(a[i] ^ b[i]);
}

/* ------------------------------------------------------------------------ */
/* C10  Shannon entropy of a histogram in bits per symbol [P1 Key           */
/* contributions and Results: the Shannon limit the codebooks are measured  */
/* against].  H = -sum p log2 p over present symbols, in double.            */
/* ------------------------------------------------------------------------ */
double ref_entropy(const uint64_t *hist)
{
    double total = 0.0;
    for (int s = 0; s < 256; ++s) total += (double)hist[s];
    if (total == 0.0) return 0.0;
    double h = 0.0;
    for (int s = 0; s < 256; ++s) {
        if (hist[s] == 0) continue;
        double p = (double)hist[s] / total;
        h -= p * log2(p);
    }
    return h;
}

/* Total encoded bits T = sum over symbols of count * length (closed form). */
uint64_t ref_total_bits(const uint64_t *hist, const uint8_t *len)
{
    uint64_t t = 0;
    for (int s = 0; s < 256; ++s) t += hist[s] * (uint64_t)len[s];
    return t;
}
