/*
 * huff.h -- C ABI of libhuff: canonical Huffman coding of ML tensor bytes on
 * one GB300 (sm_103a).
 *
 * The calls follow the problem statements of two papers:
 *   [P1] "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
 *        Overview and Methodology steps 1-4: per-shard Huffman needs frequency
 *        analysis, codebook generation and codebook transmission for every
 *        shard; the single-stage scheme counts 8-bit symbols over warm-up
 *        batches, averages the distributions, builds one codebook once, keeps
 *        it on every accelerator and encodes later tensors with it alone.
 *   [P2] "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
 *        2505.09810), Method details / technical framework and the English
 *        abstract: byte-grouping of bf16 tensors, per-group frequency
 *        statistics, per-group Huffman trees and codes, decompression as the
 *        reverse (Huffman-decode, restore the byte groups), and incremental
 *        delta compression between snapshots.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless their name starts with h_.
 *   - The caller owns and allocates every buffer.  The library never
 *     allocates memory, never synchronises the device or the stream, and
 *     enqueues all its work on `stream` (0 = the legacy default stream).
 *   - The return value is a huff_status.  It reports argument errors found
 *     on the host (HUFF_ERR_INVALID_ARG, HUFF_ERR_BUFFER_TOO_SMALL) and
 *     launch failures (HUFF_ERR_CUDA).  Nothing is enqueued when it is not
 *     HUFF_OK.
 *   - Errors found by the GPU while the work runs (a symbol without a code,
 *     a full output buffer, a corrupt stream, a wait that ran out) are
 *     written to the caller's device int32 *status: the first error wins,
 *     later ones are dropped.  The caller zeroes *status before the call and
 *     reads it after synchronising the stream.  No kernel traps or asserts.
 *   - n == 0 is valid everywhere.
 *
 * Stream format (one byte stream, e.g. an int8 shard or one bf16 byte plane)
 *   - payload: the canonical code of each symbol appended most significant bit
 *     first; stream bit k is bit 7 - (k mod 8) of payload byte k / 8; bits
 *     after the last code up to the end of the last written 32-bit word are 0.
 *     T = total bits; the stream occupies ceil(T / 8) bytes.
 *   - chunk_bit_off[c] (uint64, c = 0..n_chunks): bit position where symbol
 *     c * chunk_bytes starts; chunk_bit_off[n_chunks] = T.  Chunks are not
 *     padded, so the payload does not depend on chunk_bytes; the offsets are
 *     the index that lets chunks decode independently.
 *   - codebook: transmitted as its 256 code lengths only (canonical codes).
 */
#ifndef HUFF_H_
#define HUFF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *huff_stream_t; /* the same handle as cudaStream_t */

typedef enum huff_status {
    HUFF_OK = 0,
    HUFF_ERR_INVALID_ARG = -1,            /* bad pointer, size, alignment, flag */
    HUFF_ERR_BUFFER_TOO_SMALL = -2,       /* output or workspace capacity */
    HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK = -3, /* encode met a symbol whose length is 0 */
    HUFF_ERR_CORRUPT_STREAM = -4,         /* decode: invalid code, chunk not ending at its offset, read past payload */
    HUFF_ERR_TIMEOUT = -5,                /* a bounded device-side wait gave up */
    HUFF_ERR_CUDA = -6,                   /* a CUDA runtime call or launch failed */
    HUFF_ERR_INVALID_CODEBOOK = -7        /* codebook not built, or lengths over-subscribe the code space */
} huff_status;

#define HUFF_MAX_LEN 24          /* longest code the library produces or accepts */
#define HUFF_MIN_MAX_LEN 8       /* smallest length limit that fits 256 symbols */
#define HUFF_COVER_ALL 1u        /* raise zero counts to 1 before building (fixed codebooks) */
#define HUFF_CHUNK_ALIGN 32      /* chunk_bytes must be a positive multiple of this (the encode's lanes
                                    take 32 byte-stream symbols or 16 bf16 elements of a tile) */
#define HUFF_MAX_CHUNK (1u << 30) /* and at most this: a chunk's symbol count fits an int with room */
#define HUFF_ALIGN 16            /* alignment (bytes) required of bulk device buffers */
#define HUFF_LUT_BITS 12         /* first-level decode table index width */
#define HUFF_LUT_SYMS 6          /* most symbols one decode-table entry holds */
#define HUFF_CODEBOOK_MAGIC 0x48554642u
#define HUFF_NOALLOC_MAX_SYMBOLS (1ull << 30) /* largest n huff_encode_noalloc accepts */

/*
 * Device-resident codebook, built by huff_build_codebook or imported by
 * huff_codebook_from_lengths.  Allocate sizeof(huff_codebook) bytes of device
 * memory (16-byte aligned).  len[] is the transmitted form; the rest is
 * derived from it.  magic == HUFF_CODEBOOK_MAGIC marks a finished codebook.
 */
typedef struct huff_codebook {
    uint32_t magic;            /* HUFF_CODEBOOK_MAGIC once complete */
    int32_t max_len;           /* length limit it was built with */
    int32_t n_symbols;         /* symbols with len > 0 */
    int32_t longest;           /* longest code length present */
    uint8_t len[256];          /* code length per symbol, 0 = no code */
    uint32_t code[256];        /* canonical code per symbol, right-aligned */
    uint32_t bl_count[32];     /* number of codes of each length */
    uint32_t first_code[32];   /* canonical value of the first code of each length */
    uint32_t first_index[32];  /* index in sorted_symbols of the first code of each length */
    uint8_t sorted_symbols[256]; /* symbols ordered by (length, symbol) */
    uint64_t lut[1u << HUFF_LUT_BITS]; /* decode table for the next 12 stream bits: the codes wholly inside
                                          them, greedily, at most 6: symbols (bits 0-47, first symbol in
                                          bits 0-7), count (bits 48-51), total length (bits 52-55);
                                          0 when the first code is longer than 12 bits */
} huff_codebook;

/* Per-stream quality figures (host helper). */
typedef struct huff_stats {
    uint64_t n;                /* symbols counted */
    uint64_t total_bits;       /* T = sum_s hist[s] * len[s] */
    double entropy_bits;       /* H = -sum p log2 p, bits per symbol */
    double mean_len;           /* T / n */
    double shannon_gap;        /* (T - n H) / (n H); 0 when n H == 0 */
} huff_stats;

/* ---------------------------------------------------------------- queries */

/* Library version as 0xMMmmpp. */
uint32_t huff_version(void);

/* Static text for a status code. */
const char *huff_status_string(int status);

/* sizeof(huff_codebook), for callers that cannot include this header. */
size_t huff_codebook_size(void);

/* Worst-case payload bytes for n symbols coded with lengths <= max_len,
 * rounded up to whole 32-bit words, plus 16 bytes of slack. */
size_t huff_encode_bound(size_t n, int max_len);

/* Workspace bytes huff_encode needs for n symbols on the current device (per
 * segment of 4 to 16 tiles of 1024 symbols, the size chosen from n and the SM
 * count: a lookback descriptor and the segment's boundary-word pair, plus a
 * segment counter; at most 16 bytes per 4096 symbols + 16).  chunk_bytes does
 * not change it today; it is an argument so the format can change without an
 * ABI break. */
size_t huff_workspace_size(size_t n, size_t chunk_bytes);

/* Number of chunks: ceil(n / chunk_bytes); 0 when n == 0. */
size_t huff_num_chunks(size_t n, size_t chunk_bytes);

/*
 * huff_pick_chunk -- a chunk size for n symbols (elements, for the fused bf16
 * calls) on the current device.  The decode runs one lane per chunk, all lanes
 * resident, at most L lanes per SM: the widest block whose shared memory fits
 * for the decode that will run (delta != 0: lmc_decode_bf16 with x0, whose x0
 * staging takes shared memory; L = 896 either way on a GPU with 227 KiB of
 * shared memory per block).  This returns the smallest multiple of
 * HUFF_CHUNK_ALIGN that gives at most L chunks per SM (at least 256, so that
 * the offsets, 8 bytes a chunk, stay within 1/32 of the symbols; at most
 * HUFF_MAX_CHUNK), so that one wave of blocks of nearly L lanes covers the
 * input on every SM.  (The chunk size is the
 * caller's choice on the pages' format; each chunk costs 8 bytes of offset
 * per stream.)  Returns 0 when the device cannot be queried.
 */
size_t huff_pick_chunk(size_t n, int delta);

/* ---------------------------------------------------------------- histogram */

/*
 * huff_histogram -- 256-bin symbol histogram [P1 Methodology step 1; P2
 * framework stage 2 "frequency statistics"].
 *   in        n symbols at in[0], in[stride], ..., in[(n-1)*stride]; stride is
 *             1 (a byte stream, int8 read as its two's-complement byte) or 2
 *             (one byte plane of a little-endian 16-bit array: pass base for
 *             the low plane, base + 1 for the high plane).  Any alignment.
 *   hist      uint64[256], device.  accumulate = 0 overwrites it; accumulate = 1
 *             adds to it, which is how the averaged warm-up distribution of P1
 *             Methodology step 2 is formed (the pooled sum; Huffman lengths are
 *             unchanged by scaling all counts, so the sum gives the mean's
 *             codebook).
 */
int huff_histogram(const uint8_t *in, size_t n, size_t stride, uint64_t *hist,
                   int accumulate, huff_stream_t stream);

/* ---------------------------------------------------------------- codebook */

/*
 * huff_build_codebook -- Huffman code lengths and canonical codes from a
 * histogram [P1 Methodology step 3 "build the Huffman codebook once"; P2 key
 * design 2 "Huffman tree construction"].  The pages do not fix tie-breaks or a
 * length limit; the rule used (and reproduced by the CPU oracle) is:
 *   1. flags & HUFF_COVER_ALL: counts of 0 become 1.
 *   2. Huffman's procedure: repeatedly join the two smallest nodes by
 *      (count, id), leaves having id = symbol and new nodes ids 256, 257, ...
 *   3. Lengths above max_len are repaired with the Adjust_BITS procedure of
 *      ITU-T T.81 Annex K.3 (without its reserved-code step).
 *   4. Lengths are handed out again by (count desc, symbol asc).
 *   5. Canonical codes as in RFC 1951 section 3.2.2.
 *   6. No present symbol: an empty codebook; one symbol: length 1, code 0.
 *   hist      uint64[256], device.
 *   max_len   8..24.
 *   cb        device huff_codebook, written completely (decode tables too).
 *   status    device int32; HUFF_ERR_INVALID_CODEBOOK if the build fails: the
 *             counts (after HUFF_COVER_ALL) must sum below 2^63, which every
 *             histogram of fewer than 2^63 symbols does.
 * Runs as one thread block.
 */
int huff_build_codebook(const uint64_t *hist, int max_len, unsigned flags,
                        huff_codebook *cb, int32_t *status, huff_stream_t stream);

/*
 * huff_build_codebooks -- huff_build_codebook for `count` histograms in one
 * launch (one thread block each): cbs[k] from hists[256 k .. 256 k + 255].
 * Used for the two byte planes of a bf16 tensor.
 *   hists     uint64[count * 256], device, 8-byte aligned.
 *   count     0..65535 (0: nothing is enqueued).
 *   cbs       huff_codebook[count], device, 16-byte aligned, contiguous.
 *   other arguments and status as in huff_build_codebook (status is shared).
 */
int huff_build_codebooks(const uint64_t *hists, size_t count, int max_len, unsigned flags,
                         huff_codebook *cbs, int32_t *status, huff_stream_t stream);

/*
 * Drift-adaptive refresh of a fixed codebook.  P1 builds its codebook once
 * from warm-up statistics and names distribution drift as the limitation of
 * that scheme, with adaptive codebooks as future work.  For a shard about to
 * be encoded with cb, huff_drift_check measures how far cb is from the
 * shard's own statistics and huff_build_codebook_if rebuilds cb from the
 * shard's histogram only when the check said so, without a host round trip.
 *
 * huff_drift_check -- with h the shard's histogram (n symbols, entropy H bits
 * per symbol), T = sum h[s] * len[s] its cost under cb and B = n * max(H, 1)
 * (the entropy bound, and at least one bit per symbol for any Huffman code
 * of bytes):  gap = (T - B) / B, +infinity when a present symbol has no
 * code, 0 for an empty shard.  Writes *flag = (gap > threshold) and, if gap
 * is not NULL, *gap (double).  All pointers device; threshold >= 0.
 */
int huff_drift_check(const uint64_t *hist, const huff_codebook *cb, double threshold, uint32_t *flag,
                     double *gap, huff_stream_t stream);

/*
 * huff_build_codebook_if -- huff_build_codebook when *flag != 0 (a device
 * word, e.g. from huff_drift_check); otherwise cb is left as it is.
 */
int huff_build_codebook_if(const uint64_t *hist, const uint32_t *flag, int max_len, unsigned flags,
                           huff_codebook *cb, int32_t *status, huff_stream_t stream);

/*
 * huff_codebook_from_lengths -- import a transmitted codebook [P1 Key
 * contributions: the codebook is stored on each accelerator, not exchanged per
 * batch; it travels once, as 256 lengths].
 *   h_len     HOST uint8[256]; copied before the call returns.
 *   max_len   8..24; every length must be <= max_len.
 *   cb        device huff_codebook; status gets HUFF_ERR_INVALID_CODEBOOK when
 *             the lengths over-subscribe the code space (Kraft sum > 1).
 */
int huff_codebook_from_lengths(const uint8_t *h_len, int max_len, huff_codebook *cb,
                               int32_t *status, huff_stream_t stream);

/* ---------------------------------------------------------------- encode / decode */

/*
 * huff_encode -- single-stage encode with a given codebook [P1 Methodology
 * step 4: tensors are encoded directly with the precomputed codebook; P2
 * framework stage 3 "Huffman coding", split into parallel tasks].
 *   in            n symbols, 16-byte aligned.
 *   cb            device codebook built or imported above.
 *   chunk_bytes   symbols per chunk, a positive multiple of HUFF_CHUNK_ALIGN,
 *                 at most HUFF_MAX_CHUNK (otherwise HUFF_ERR_INVALID_ARG).
 *   payload       16-byte aligned, payload_cap bytes; huff_encode_bound(n,
 *                 max_len) always suffices.  The stream needs ceil(T/32)*4
 *                 bytes; a shorter buffer gives HUFF_ERR_BUFFER_TOO_SMALL in
 *                 *status and a truncated payload.
 *   chunk_bit_off uint64[n_chunks + 1], device, 8-byte aligned.
 *   ws, ws_bytes  device workspace of at least huff_workspace_size(n,
 *                 chunk_bytes) bytes, 16-byte aligned; its contents need not be
 *                 initialised and are garbage afterwards.  Two encodes that run
 *                 at the same time need two workspaces.
 *   status        device int32: HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK,
 *                 HUFF_ERR_BUFFER_TOO_SMALL, HUFF_ERR_TIMEOUT,
 *                 HUFF_ERR_INVALID_CODEBOOK.
 * T = chunk_bit_off[n_chunks] after the stream completes.
 */
int huff_encode(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk_bytes,
                uint8_t *payload, size_t payload_cap, uint64_t *chunk_bit_off,
                void *ws, size_t ws_bytes, int32_t *status, huff_stream_t stream);

/*
 * huff_encode_noalloc -- huff_encode for callers that cannot allocate device
 * memory.  No counterpart in the papers: it is a deployment convenience.
 *
 * huff_encode needs a workspace of huff_workspace_size(n) bytes.  Some callers
 * have no way to provide one: a process whose device memory is owned entirely
 * by a framework's pool allocator (third-party cudaMalloc calls fail or break
 * its accounting), a latency-critical loop that must not call cudaMalloc or
 * cudaFree because they can synchronise the whole device, or a caller that
 * only holds the input and output buffers it was handed.  This entry point
 * takes the same inputs and outputs as huff_encode, without ws, and runs the
 * same kernels with a workspace that the library keeps in a fixed 2 MiB
 * device array.  Nothing is allocated per call.
 *   n             at most HUFF_NOALLOC_MAX_SYMBOLS (2^30) symbols; larger n
 *                 returns HUFF_ERR_BUFFER_TOO_SMALL and enqueues nothing.
 *   other arguments as in huff_encode; the output is identical to its output.
 * The array lives in every GPU that loads the library, until the process
 * exits.  Every call looks up the array's address on the current device
 * (cudaGetSymbolAddress: a host-side query that allocates nothing), so the
 * address stays right after cudaDeviceReset.  The first call on a device may
 * load the library's device code; make that first call before any stream
 * capture.  All calls share the one array:
 * calls whose work can overlap on the GPU (different streams, or several host
 * threads) race and corrupt each other's output; serialise them, or use
 * huff_encode with one workspace per stream.
 */
int huff_encode_noalloc(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk_bytes,
                        uint8_t *payload, size_t payload_cap, uint64_t *chunk_bit_off, int32_t *status,
                        huff_stream_t stream);

/*
 * huff_stream_copy -- copy a compressed stream to other device buffers, its
 * size read on the device ["Single-stage Huffman encoder for ML compression",
 * Practical impact: compressed tensors travel between accelerators that hold
 * the same fixed codebook, so nothing but the stream is exchanged].  With one
 * GPU this is the loopback link: encode -> copy -> decode with no host round
 * trip (the host never needs T).
 *   payload, chunk_bit_off, n_chunks   a stream as huff_encode writes it;
 *                 payload 16-byte aligned, payload_bytes long.
 *   dst_payload   dst_cap bytes, 16-byte aligned, not the source; receives
 *                 the stream through the end of its last 32-bit word:
 *                 min(4 ceil(T / 32), payload_bytes) bytes, T =
 *                 chunk_bit_off[n_chunks].
 *   dst_off       uint64[n_chunks + 1], 8-byte aligned, not the source.
 *   status        HUFF_ERR_BUFFER_TOO_SMALL when dst_cap is below that size;
 *                 HUFF_ERR_CORRUPT_STREAM when T > 8 payload_bytes.  Either
 *                 way nothing is copied.
 */
int huff_stream_copy(const uint8_t *payload, size_t payload_bytes, const uint64_t *chunk_bit_off,
                     size_t n_chunks, uint8_t *dst_payload, size_t dst_cap, uint64_t *dst_off,
                     int32_t *status, huff_stream_t stream);

/*
 * huff_decode -- chunked decode [P2 framework: decompression reads the data,
 * Huffman-decodes it and restores it; lossless, so the output equals the
 * encoder's input].
 *   payload       payload_bytes bytes, 16-byte aligned.  It is read in whole
 *                 16-byte units: the unit holding the last payload byte is
 *                 read whole, and no unit after it is read.  The unit's bytes
 *                 past payload_bytes never change the result.
 *   chunk_bit_off uint64[n_chunks + 1] as written by huff_encode.
 *   n, chunk_bytes the encoder's values.
 *   out           n bytes, 16-byte aligned.
 *   status        HUFF_ERR_CORRUPT_STREAM when a code is invalid, a chunk does
 *                 not end exactly at the next offset, an offset lies outside
 *                 the payload, or a chunk holds fewer than 1 or more than
 *                 HUFF_MAX_LEN bits per symbol;
 *                 HUFF_ERR_INVALID_CODEBOOK.
 */
int huff_decode(const uint8_t *payload, size_t payload_bytes, const uint64_t *chunk_bit_off,
                size_t n, size_t chunk_bytes, const huff_codebook *cb, uint8_t *out,
                int32_t *status, huff_stream_t stream);

/* ---------------------------------------------------------------- LMC byte grouping */

/*
 * lmc_bytegroup_split -- byte grouping of a 16-bit tensor [P2 framework stage 1
 * and key design 1; English abstract "byte-grouping"]: hi[i] = w[i] >> 8 (bf16:
 * sign and the 7 high exponent bits), lo[i] = w[i] & 0xff (lowest exponent bit
 * and the 7 mantissa bits).  w is little-endian uint16 (the bf16 bit pattern).
 */
int lmc_bytegroup_split(const uint16_t *w, size_t n, uint8_t *hi, uint8_t *lo,
                        huff_stream_t stream);

/* lmc_bytegroup_merge -- inverse of the split [P2 framework, decompression:
 * "restore the byte groups"]: w[i] = hi[i] << 8 | lo[i]. */
int lmc_bytegroup_merge(const uint8_t *hi, const uint8_t *lo, size_t n, uint16_t *w,
                        huff_stream_t stream);

/* lmc_delta_xor -- incremental delta between snapshots [P2 English abstract
 * "incremental delta compression"; the operator is not given on the pages and
 * is read as XOR of the bit patterns, which is exact for every value including
 * NaN, Inf and -0]: out[i] = a[i] ^ b[i].  Self-inverse; out may alias a or b. */
int lmc_delta_xor(const uint16_t *a, const uint16_t *b, size_t n, uint16_t *out,
                  huff_stream_t stream);

/*
 * lmc_bytegroup_split_w / lmc_bytegroup_merge_w -- byte planes of W-byte
 * words, W = 1, 2, 4 or 8: P2's byte grouping (framework stage 1, key design
 * 1) for other element widths (fp32: 4 planes, fp16 and bf16: 2, fp8: 1,
 * fp64: 8).  Plane p holds byte W-1-p of every word, most significant first;
 * for W = 2 plane 0 is lmc_bytegroup_split's hi.  Each plane is then an
 * ordinary byte stream for huff_histogram / huff_encode.
 *   in, out     n words of W bytes, little endian; any alignment (16-byte
 *               aligned pointers with n % 16 == 0 take the vector path).
 *   planes      plane p at planes + p * plane_stride (plane_stride >= n bytes, a
 *               multiple of 16 for the vector path); must not overlap in/out.
 *   width       1, 2, 4 or 8, else HUFF_ERR_INVALID_ARG.
 */
int lmc_bytegroup_split_w(const void *in, size_t n, int width, uint8_t *planes, size_t plane_stride,
                          huff_stream_t stream);
int lmc_bytegroup_merge_w(const uint8_t *planes, size_t n, int width, size_t plane_stride, void *out,
                          huff_stream_t stream);

/* ---------------------------------------------------------------- LMC fused bf16 paths */

/*
 * lmc_histogram_bf16 -- histograms of both byte planes of a bf16 tensor,
 * optionally of its XOR delta against x0, in one pass (P2 framework stages 1-2
 * fused).  Equal to lmc_delta_xor + lmc_bytegroup_split + huff_histogram on
 * each plane.
 *   w, x0     n uint16 values; x0 may be NULL (no delta).  Any alignment.
 *   hist_hi, hist_lo  uint64[256] each; accumulate as in huff_histogram.
 */
int lmc_histogram_bf16(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                       uint64_t *hist_lo, int accumulate, huff_stream_t stream);

/* Workspace bytes lmc_encode_bf16 needs for n elements: the per-segment
 * counts (lmc_segment_counts_size), the counted encode's workspace
 * (lmc_counted_workspace_size), each rounded up to 256 bytes, and 4 KiB for
 * the two histograms the counting pass also produces (about 32 MB for 2e9
 * elements). */
size_t lmc_workspace_size(size_t n, size_t chunk_bytes);

/*
 * lmc_encode_bf16 -- encode both byte planes of a bf16 tensor (optionally of
 * its XOR delta against x0) straight from the 16-bit words, each plane with
 * its own given codebook (P2 framework stages 1 and 3 fused; P1 Methodology
 * step 4, a codebook fixed in advance).  The outputs are byte-identical to
 * split + huff_encode per plane: plane streams (payload_hi, off_hi) and
 * (payload_lo, off_lo) with chunk_bytes elements per chunk.  Runs as two
 * passes over the input: lmc_histogram_bf16_counted's counting pass into the
 * workspace, then lmc_encode_bf16_counted under the given codebooks.  A
 * symbol present in the data without a code in its plane's codebook sets
 * HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK (the stream is then not usable).
 *   w, x0     16-byte aligned; x0 may be NULL.
 *   other arguments as in huff_encode, once per plane.
 */
int lmc_encode_bf16(const uint16_t *w, const uint16_t *x0, size_t n,
                    const huff_codebook *cb_hi, const huff_codebook *cb_lo, size_t chunk_bytes,
                    uint8_t *payload_hi, size_t cap_hi, uint64_t *off_hi,
                    uint8_t *payload_lo, size_t cap_lo, uint64_t *off_lo,
                    void *ws, size_t ws_bytes, int32_t *status, huff_stream_t stream);

/*
 * Counted per-shard path.  When the codebooks are built from the tensor's own
 * histograms (per-shard mode, P2 framework stages 2-3), the histogram pass
 * can also record both planes' counts per segment of S = lmc_count_segment(n)
 * elements.  lmc_encode_bf16_counted then derives every segment's bit offset
 * as sum(count * length) and encodes in one pass over the input, with no
 * counting pass and no waiting between CTAs.  Its outputs are byte-identical
 * to lmc_encode_bf16's.  (A GPU arrangement of the same method; the pages
 * have no separate step for it.)
 */
#define HUFF_COUNT_SEGMENT 131072 /* the least segment size S */

/*
 * lmc_count_segment -- S, the elements per counted segment for n elements on
 * the current device: HUFF_COUNT_SEGMENT while the counted encode's warps (20
 * per SM) outnumber segments of that size; otherwise the multiple of 512 in
 * [HUFF_COUNT_SEGMENT, 2 * HUFF_COUNT_SEGMENT) that gives every warp the same
 * number of segments.  lmc_histogram_bf16_counted and lmc_encode_bf16_counted
 * both use it, so both must run on devices with the same SM count.
 */
size_t lmc_count_segment(size_t n);

/* Bytes of the per-segment counts for n elements: 2048 * ceil(n / HUFF_COUNT_SEGMENT)
 * (enough for any S). */
size_t lmc_segment_counts_size(size_t n);

/* Workspace bytes lmc_encode_bf16_counted needs: 48 * ceil(n / HUFF_COUNT_SEGMENT) + 16. */
size_t lmc_counted_workspace_size(size_t n);

/*
 * lmc_histogram_bf16_counted -- lmc_histogram_bf16 that also writes
 * seg_counts[s][0][b] and seg_counts[s][1][b] (uint32): the counts of symbol
 * b in the high and low plane of elements [s * S, (s + 1) * S), S =
 * lmc_count_segment(n).
 *   w, x0       16-byte aligned; x0 may be NULL (no delta).
 *   hist_hi, hist_lo  uint64[256] each, overwritten.
 *   seg_counts  uint32 array of seg_counts_bytes >= lmc_segment_counts_size(n), 4-byte aligned.
 */
int lmc_histogram_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                               uint64_t *hist_lo, uint32_t *seg_counts, size_t seg_counts_bytes,
                               huff_stream_t stream);

/*
 * lmc_encode_bf16_counted -- lmc_encode_bf16 from the per-segment counts of
 * the same w (and x0) written by lmc_histogram_bf16_counted.  Counts that do
 * not match the data give a wrong stream; when a segment's bits differ from
 * the bits its counts give, status gets HUFF_ERR_INVALID_ARG.  A symbol
 * without a code still sets HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK.
 *   ws          ws_bytes >= lmc_counted_workspace_size(n), 16-byte aligned.
 *   other arguments as in lmc_encode_bf16.
 */
int lmc_encode_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n,
                            const huff_codebook *cb_hi, const huff_codebook *cb_lo, size_t chunk_bytes,
                            const uint32_t *seg_counts, size_t seg_counts_bytes,
                            uint8_t *payload_hi, size_t cap_hi, uint64_t *off_hi,
                            uint8_t *payload_lo, size_t cap_lo, uint64_t *off_lo,
                            void *ws, size_t ws_bytes, int32_t *status, huff_stream_t stream);

/*
 * lmc_decode_bf16 -- decode both planes and write the 16-bit words, optionally
 * XOR-ing x0 back in (P2 decompression: Huffman-decode, restore byte groups,
 * re-apply the delta).  out[i] = (hi[i] << 8 | lo[i]) ^ (x0 ? x0[i] : 0).
 *   out, x0   16-byte aligned; x0 may be NULL; out may not alias x0.
 *   other arguments as in huff_decode, once per plane.
 */
int lmc_decode_bf16(const uint8_t *payload_hi, size_t bytes_hi, const uint64_t *off_hi,
                    const uint8_t *payload_lo, size_t bytes_lo, const uint64_t *off_lo,
                    size_t n, size_t chunk_bytes, const huff_codebook *cb_hi,
                    const huff_codebook *cb_lo, const uint16_t *x0, uint16_t *out,
                    int32_t *status, huff_stream_t stream);

/* ---------------------------------------------------------------- host helpers */

/*
 * huff_code_stats -- quality figures of one stream [P1 Key contributions and
 * Results: compression is compared against per-shard Huffman and against the
 * Shannon limit].  h_hist: HOST uint64[256]; h_len: HOST uint8[256] code
 * lengths.  Returns HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK when a counted symbol has
 * no code.
 */
int huff_code_stats(const uint64_t *h_hist, const uint8_t *h_len, huff_stats *out);

/*
 * Serialised stream (a container) [P1 Methodology: with a fixed codebook the
 * per-message codebook is neither recomputed nor transmitted; P2 framework:
 * the compressed data and what decompression needs].  All fields little-endian,
 * on HOST memory, no padding:
 *   offset  0  uint32 magic HUFF_CONTAINER_MAGIC ("HUFC")
 *           4  uint16 version (1)
 *           6  uint16 flags: bit 0 set when the 256 code lengths follow the
 *                    header (per-shard mode); clear for a fixed codebook,
 *                    which the receiver already holds
 *           8  uint32 max_len the codebook was built with
 *          12  uint32 zero
 *          16  uint64 n (symbols)
 *          24  uint64 chunk_bytes
 *          32  uint64 n_chunks = huff_num_chunks(n, chunk_bytes)
 *          40  uint64 T (total bits) = chunk_bit_off[n_chunks]
 *          48  [uint8 len[256] when flag bit 0]
 *          then uint64 chunk_bit_off[n_chunks + 1], then the payload's first
 *          ceil(T / 8) bytes.
 */
#define HUFF_CONTAINER_MAGIC 0x43465548u
#define HUFF_CONTAINER_HEADER 48
#define HUFF_CONTAINER_LENGTHS 1u

/* Bytes of a container for n symbols, chunk_bytes, T bits; with_lengths: flag bit 0. */
size_t huff_container_size(size_t n, size_t chunk_bytes, uint64_t total_bits, int with_lengths);

/*
 * huff_container_write -- serialise a stream (HOST buffers; no device work).
 *   h_len     HOST uint8[256] code lengths, or NULL for a fixed codebook.
 *   h_off     HOST uint64[n_chunks + 1] chunk bit offsets; h_off[n_chunks] = T.
 *   h_payload HOST payload, at least ceil(T / 8) bytes.
 *   h_dst     HOST buffer of cap bytes; *written gets the container's size.
 * Returns HUFF_ERR_INVALID_ARG for a bad chunk size, offsets that are not
 * non-decreasing from 0, or lengths above max_len; HUFF_ERR_BUFFER_TOO_SMALL
 * when cap < huff_container_size(...).
 */
int huff_container_write(uint8_t *h_dst, size_t cap, size_t n, size_t chunk_bytes, int max_len,
                         const uint8_t *h_len, const uint64_t *h_off, const uint8_t *h_payload,
                         size_t *written);

/* A parsed container: the fields, and pointers into the parsed buffer. */
typedef struct huff_container_view {
    uint64_t n, chunk_bytes, n_chunks, total_bits;
    int32_t max_len;
    int32_t has_lengths;
    const uint8_t *len;       /* 256 lengths, or NULL */
    const uint8_t *off;       /* (n_chunks + 1) little-endian uint64, unaligned in general */
    const uint8_t *payload;   /* ceil(T / 8) bytes */
    uint64_t payload_bytes;
} huff_container_view;

/*
 * huff_container_parse -- check and view a container of size bytes (HOST; no
 * copy).  Returns HUFF_ERR_CORRUPT_STREAM when the magic, version, reserved
 * field or sizes do not agree, n_chunks is not huff_num_chunks(n,
 * chunk_bytes), the offsets do not rise from 0 to T, or a length exceeds
 * max_len; HUFF_ERR_INVALID_ARG for NULL pointers.
 */
int huff_container_parse(const uint8_t *h_src, size_t size, huff_container_view *view);

/* ---------------------------------------------------------------- test hook */

/*
 * huff_debug_wait -- runs one of the library's bounded device waits on its
 * own, so that a test can watch it run out without any fault: the waits of
 * the encode kernels (the decoupled lookback over segment descriptors, after
 * Merrill & Garland's single-pass scan, and the bulk-copy mbarrier waits)
 * give up after a poll limit and report HUFF_ERR_TIMEOUT instead of hanging.
 * (Failure handling around the method; the pages have no step for it.)
 *   kind 0   one warp looks back from segment seg over desc[0 .. seg) (device
 *            uint64 descriptors: flag in bits 62-63, 1 = aggregate, 2 =
 *            inclusive prefix, 0 = not yet published; bit count in bits
 *            0-61), n_desc >= seg >= 1.  A descriptor left at 0 makes the
 *            wait run out after `limit` polls, or at the first poll count
 *            divisible by 256 when *status already holds an error.
 *   kind 1   one warp waits on a fresh mbarrier that nothing arrives on and
 *            no copy targets, at most `limit` polls; desc is ignored.
 *   limit    1 .. 2^20 polls.
 *   out      device uint64[2]: the lookback's exclusive prefix (kind 0) and
 *            the number of polls made.
 *   status   device int32, caller-zeroed: HUFF_ERR_TIMEOUT when the wait ran
 *            out (the first error recorded stays).
 * Returns HUFF_ERR_INVALID_ARG for other arguments.  One launch of 32 threads
 * on `stream`; no allocation, no synchronisation.
 */
int huff_debug_wait(int kind, const uint64_t *desc, size_t n_desc, uint32_t seg, uint32_t limit, uint64_t *out,
                    int32_t *status, huff_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HUFF_H_ */
