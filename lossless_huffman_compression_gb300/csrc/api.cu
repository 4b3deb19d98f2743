// api.cu -- the extern "C" entry points of libhuff (include/huff.h).
//
// Host side only: argument checks, buffer sizing, and launches on the caller's
// stream.  No allocation, no synchronisation.
#include <cmath>
#include <cstddef>

#include "common.cuh"

using namespace huffk;

namespace {

// the decode kernels copy the table with 16-byte loads; the binding reads len[] at byte 16
static_assert(offsetof(huff_codebook, lut) % 16 == 0, "codebook lut must be 16-byte aligned");
static_assert(HUFF_COUNT_SEGMENT == huffk::kDirSegElems, "counted segment size");
static_assert(offsetof(huff_codebook, len) == 16 && offsetof(huff_codebook, code) == 272, "codebook layout");
static_assert(sizeof(huff_codebook) % 16 == 0, "codebook size");

constexpr size_t kMaxN = size_t(1) << 40;  // 1 Ti symbols: bit offsets stay far below 2^62
constexpr size_t kMaxCodebooks = 65535;     // one CTA per codebook in one launch

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline cudaStream_t cs(huff_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool chunk_ok(size_t chunk) { return chunk > 0 && chunk % HUFF_CHUNK_ALIGN == 0 && chunk <= HUFF_MAX_CHUNK; }

}  // namespace

extern "C" {

uint32_t huff_version(void) { return 0x010000u; }

const char *huff_status_string(int status) {
    switch (status) {
        case HUFF_OK: return "ok";
        case HUFF_ERR_INVALID_ARG: return "invalid argument";
        case HUFF_ERR_BUFFER_TOO_SMALL: return "buffer too small";
        case HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK: return "symbol not in codebook";
        case HUFF_ERR_CORRUPT_STREAM: return "corrupt stream";
        case HUFF_ERR_TIMEOUT: return "device wait timed out";
        case HUFF_ERR_CUDA: return "CUDA error";
        case HUFF_ERR_INVALID_CODEBOOK: return "invalid codebook";
        default: return "unknown status";
    }
}

size_t huff_codebook_size(void) { return sizeof(huff_codebook); }

size_t huff_num_chunks(size_t n, size_t chunk_bytes) {
    if (chunk_bytes == 0) return 0;
    return (n + chunk_bytes - 1) / chunk_bytes;
}

constexpr size_t kPickChunkMin = 256;

size_t huff_pick_chunk(size_t n, int delta) {
    int dev = 0, sms = 0, smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0 ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    // one full block of the decode's widest width on every SM: the smallest chunk size (in steps of
    // HUFF_CHUNK_ALIGN) that gives at most that many chunks
    const size_t lanes = static_cast<size_t>(sms) * static_cast<size_t>(decode_lanes(smem, delta != 0));
    size_t c = (n + lanes - 1) / lanes;
    c = (c + HUFF_CHUNK_ALIGN - 1) / HUFF_CHUNK_ALIGN * HUFF_CHUNK_ALIGN;
    if (c < kPickChunkMin) c = kPickChunkMin;  // offsets (8 bytes a chunk) stay within 1/32 of the symbols
    return c > HUFF_MAX_CHUNK ? HUFF_MAX_CHUNK : c;
}

size_t huff_encode_bound(size_t n, int max_len) {
    if (max_len < 1 || max_len > HUFF_MAX_LEN) max_len = HUFF_MAX_LEN;
    const size_t words = (n * static_cast<size_t>(max_len) + 31) / 32;
    return words * 4 + 16;
}

size_t huff_workspace_size(size_t n, size_t chunk_bytes) {
    (void)chunk_bytes;
    return enc_u8_workspace_words(n) * sizeof(uint64_t);
}

size_t lmc_workspace_size(size_t n, size_t chunk_bytes) {
    (void)chunk_bytes;
    return enc_bf16_given_ws_parts(n, nullptr, nullptr);
}

int huff_histogram(const uint8_t *in, size_t n, size_t stride, uint64_t *hist, int accumulate,
                   huff_stream_t stream) {
    if (hist == nullptr || !aligned(hist, 8) || (stride != 1 && stride != 2) || n > kMaxN ||
        (n > 0 && in == nullptr))
        return HUFF_ERR_INVALID_ARG;
    if (!accumulate) {
        const int st = launch_zero_u64(hist, 256, cs(stream));
        if (st != HUFF_OK) return st;
    }
    if (n == 0) return HUFF_OK;
    return launch_histogram(in, n, stride, hist, cs(stream));
}

int huff_build_codebook(const uint64_t *hist, int max_len, unsigned flags, huff_codebook *cb, int32_t *status,
                        huff_stream_t stream) {
    if (hist == nullptr || cb == nullptr || status == nullptr || !aligned(cb, 16) || !aligned(hist, 8) ||
        max_len < HUFF_MIN_MAX_LEN || max_len > HUFF_MAX_LEN || (flags & ~HUFF_COVER_ALL) != 0)
        return HUFF_ERR_INVALID_ARG;
    return launch_build_codebook(hist, max_len, flags, cb, status, nullptr, cs(stream));
}

int huff_build_codebooks(const uint64_t *hists, size_t count, int max_len, unsigned flags, huff_codebook *cbs,
                         int32_t *status, huff_stream_t stream) {
    if (count == 0) return HUFF_OK;
    if (hists == nullptr || cbs == nullptr || status == nullptr || !aligned(cbs, 16) || !aligned(hists, 8) ||
        count > kMaxCodebooks || max_len < HUFF_MIN_MAX_LEN || max_len > HUFF_MAX_LEN ||
        (flags & ~HUFF_COVER_ALL) != 0)
        return HUFF_ERR_INVALID_ARG;
    return launch_build_codebooks(hists, count, max_len, flags, cbs, status, nullptr, cs(stream));
}

int huff_stream_copy(const uint8_t *payload, size_t payload_bytes, const uint64_t *chunk_bit_off, size_t n_chunks,
                     uint8_t *dst_payload, size_t dst_cap, uint64_t *dst_off, int32_t *status,
                     huff_stream_t stream) {
    if (payload == nullptr || chunk_bit_off == nullptr || dst_payload == nullptr || dst_off == nullptr ||
        status == nullptr || !aligned(payload, HUFF_ALIGN) || !aligned(dst_payload, HUFF_ALIGN) ||
        !aligned(chunk_bit_off, 8) || !aligned(dst_off, 8) || dst_off == chunk_bit_off || dst_payload == payload)
        return HUFF_ERR_INVALID_ARG;
    return launch_stream_copy(payload, payload_bytes, chunk_bit_off, n_chunks, dst_payload, dst_cap, dst_off, status,
                              cs(stream));
}

int huff_drift_check(const uint64_t *hist, const huff_codebook *cb, double threshold, uint32_t *flag, double *gap,
                     huff_stream_t stream) {
    if (hist == nullptr || cb == nullptr || flag == nullptr || !aligned(hist, 8) || !aligned(cb, 16) ||
        !aligned(flag, 4) || (gap != nullptr && !aligned(gap, 8)) || !(threshold >= 0.0))
        return HUFF_ERR_INVALID_ARG;
    return launch_drift_check(hist, cb, threshold, flag, gap, cs(stream));
}

int huff_build_codebook_if(const uint64_t *hist, const uint32_t *flag, int max_len, unsigned flags,
                           huff_codebook *cb, int32_t *status, huff_stream_t stream) {
    if (hist == nullptr || flag == nullptr || cb == nullptr || status == nullptr || !aligned(cb, 16) ||
        !aligned(hist, 8) || !aligned(flag, 4) || max_len < HUFF_MIN_MAX_LEN || max_len > HUFF_MAX_LEN ||
        (flags & ~HUFF_COVER_ALL) != 0)
        return HUFF_ERR_INVALID_ARG;
    return launch_build_codebook(hist, max_len, flags, cb, status, flag, cs(stream));
}

int huff_codebook_from_lengths(const uint8_t *h_len, int max_len, huff_codebook *cb, int32_t *status,
                               huff_stream_t stream) {
    if (h_len == nullptr || cb == nullptr || status == nullptr || !aligned(cb, 16) ||
        max_len < HUFF_MIN_MAX_LEN || max_len > HUFF_MAX_LEN)
        return HUFF_ERR_INVALID_ARG;
    for (int s = 0; s < 256; ++s)
        if (h_len[s] > max_len) return HUFF_ERR_INVALID_ARG;
    // a pageable source is staged before cudaMemcpyAsync returns, so h_len may be reused at once
    if (cudaMemcpyAsync(cb->len, h_len, 256, cudaMemcpyHostToDevice, cs(stream)) != cudaSuccess)
        return HUFF_ERR_CUDA;
    return launch_codebook_from_lengths(max_len, cb, status, cs(stream));
}

int huff_encode(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk_bytes, uint8_t *payload,
                size_t payload_cap, uint64_t *chunk_bit_off, void *ws, size_t ws_bytes, int32_t *status,
                huff_stream_t stream) {
    if (cb == nullptr || chunk_bit_off == nullptr || status == nullptr || !chunk_ok(chunk_bytes) || n > kMaxN ||
        !aligned(cb, 16) || !aligned(chunk_bit_off, 8))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (in == nullptr || payload == nullptr || ws == nullptr || !aligned(in, HUFF_ALIGN) ||
                  !aligned(payload, HUFF_ALIGN) || !aligned(ws, HUFF_ALIGN)))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && ws_bytes < huff_workspace_size(n, chunk_bytes)) return HUFF_ERR_BUFFER_TOO_SMALL;
    return launch_encode_u8(in, n, cb, chunk_bytes, payload, payload_cap, chunk_bit_off, ws, status, cs(stream));
}

int huff_encode_noalloc(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk_bytes,
                        uint8_t *payload, size_t payload_cap, uint64_t *chunk_bit_off, int32_t *status,
                        huff_stream_t stream) {
    if (cb == nullptr || chunk_bit_off == nullptr || status == nullptr || !chunk_ok(chunk_bytes) ||
        !aligned(cb, 16) || !aligned(chunk_bit_off, 8))
        return HUFF_ERR_INVALID_ARG;
    if (n > HUFF_NOALLOC_MAX_SYMBOLS) return HUFF_ERR_BUFFER_TOO_SMALL;  // beyond the built-in scratch
    if (n > 0 && (in == nullptr || payload == nullptr || !aligned(in, HUFF_ALIGN) || !aligned(payload, HUFF_ALIGN)))
        return HUFF_ERR_INVALID_ARG;
    return launch_encode_u8_noalloc(in, n, cb, chunk_bytes, payload, payload_cap, chunk_bit_off, status,
                                    cs(stream));
}

int huff_decode(const uint8_t *payload, size_t payload_bytes, const uint64_t *chunk_bit_off, size_t n,
                size_t chunk_bytes, const huff_codebook *cb, uint8_t *out, int32_t *status,
                huff_stream_t stream) {
    if (cb == nullptr || status == nullptr || !chunk_ok(chunk_bytes) || n > kMaxN || !aligned(cb, 16))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (payload == nullptr || chunk_bit_off == nullptr || out == nullptr ||
                  !aligned(payload, HUFF_ALIGN) || !aligned(out, HUFF_ALIGN) || !aligned(chunk_bit_off, 8)))
        return HUFF_ERR_INVALID_ARG;
    return launch_decode_u8(payload, payload_bytes, chunk_bit_off, n, chunk_bytes, cb, out, status, cs(stream));
}

int lmc_bytegroup_split(const uint16_t *w, size_t n, uint8_t *hi, uint8_t *lo, huff_stream_t stream) {
    if (n > kMaxN || (n > 0 && (w == nullptr || hi == nullptr || lo == nullptr || !aligned(w, 2))))
        return HUFF_ERR_INVALID_ARG;
    return launch_split(w, n, hi, lo, cs(stream));
}

int lmc_bytegroup_merge(const uint8_t *hi, const uint8_t *lo, size_t n, uint16_t *w, huff_stream_t stream) {
    if (n > kMaxN || (n > 0 && (w == nullptr || hi == nullptr || lo == nullptr || !aligned(w, 2))))
        return HUFF_ERR_INVALID_ARG;
    return launch_merge(hi, lo, n, w, cs(stream));
}

int lmc_delta_xor(const uint16_t *a, const uint16_t *b, size_t n, uint16_t *out, huff_stream_t stream) {
    if (n > kMaxN || (n > 0 && (a == nullptr || b == nullptr || out == nullptr || !aligned(a, 2) ||
                                !aligned(b, 2) || !aligned(out, 2))))
        return HUFF_ERR_INVALID_ARG;
    return launch_xor(a, b, n, out, cs(stream));
}

int lmc_bytegroup_split_w(const void *in, size_t n, int width, uint8_t *planes, size_t plane_stride,
                          huff_stream_t stream) {
    if ((width != 1 && width != 2 && width != 4 && width != 8) || n > kMaxN || plane_stride < n ||
        (n > 0 && (in == nullptr || planes == nullptr)))
        return HUFF_ERR_INVALID_ARG;
    return launch_split_w(static_cast<const uint8_t *>(in), n, width, planes, plane_stride, cs(stream));
}

int lmc_bytegroup_merge_w(const uint8_t *planes, size_t n, int width, size_t plane_stride, void *out,
                          huff_stream_t stream) {
    if ((width != 1 && width != 2 && width != 4 && width != 8) || n > kMaxN || plane_stride < n ||
        (n > 0 && (out == nullptr || planes == nullptr)))
        return HUFF_ERR_INVALID_ARG;
    return launch_merge_w(planes, n, width, plane_stride, static_cast<uint8_t *>(out), cs(stream));
}

int lmc_histogram_bf16(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi, uint64_t *hist_lo,
                       int accumulate, huff_stream_t stream) {
    if (hist_hi == nullptr || hist_lo == nullptr || hist_hi == hist_lo || !aligned(hist_hi, 8) ||
        !aligned(hist_lo, 8) || n > kMaxN || (n > 0 && (w == nullptr || !aligned(w, 2))) ||
        (x0 != nullptr && !aligned(x0, 2)))
        return HUFF_ERR_INVALID_ARG;
    if (!accumulate) {
        int st = launch_zero_u64(hist_hi, 256, cs(stream));
        if (st == HUFF_OK) st = launch_zero_u64(hist_lo, 256, cs(stream));
        if (st != HUFF_OK) return st;
    }
    if (n == 0) return HUFF_OK;
    return launch_histogram_bf16(w, x0, n, hist_hi, hist_lo, cs(stream));
}

int lmc_encode_bf16(const uint16_t *w, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                    const huff_codebook *cb_lo, size_t chunk_bytes, uint8_t *payload_hi, size_t cap_hi,
                    uint64_t *off_hi, uint8_t *payload_lo, size_t cap_lo, uint64_t *off_lo, void *ws,
                    size_t ws_bytes, int32_t *status, huff_stream_t stream) {
    if (cb_hi == nullptr || cb_lo == nullptr || off_hi == nullptr || off_lo == nullptr || status == nullptr ||
        !chunk_ok(chunk_bytes) || n > kMaxN || !aligned(cb_hi, 16) || !aligned(cb_lo, 16) ||
        !aligned(off_hi, 8) || !aligned(off_lo, 8))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (w == nullptr || payload_hi == nullptr || payload_lo == nullptr || ws == nullptr ||
                  !aligned(w, HUFF_ALIGN) || (x0 != nullptr && !aligned(x0, HUFF_ALIGN)) ||
                  !aligned(payload_hi, HUFF_ALIGN) || !aligned(payload_lo, HUFF_ALIGN) || !aligned(ws, HUFF_ALIGN)))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && ws_bytes < lmc_workspace_size(n, chunk_bytes)) return HUFF_ERR_BUFFER_TOO_SMALL;
    return launch_encode_bf16(w, x0, n, cb_hi, cb_lo, chunk_bytes, payload_hi, cap_hi, off_hi, payload_lo, cap_lo,
                              off_lo, ws, status, cs(stream));
}

size_t lmc_segment_counts_size(size_t n) {
    return static_cast<size_t>(huffk::kSegCountWords) * 4 * ((n + HUFF_COUNT_SEGMENT - 1) / HUFF_COUNT_SEGMENT);
}

size_t lmc_count_segment(size_t n) { return huffk::count_seg_elems(n); }

size_t lmc_counted_workspace_size(size_t n) { return 48 * ((n + HUFF_COUNT_SEGMENT - 1) / HUFF_COUNT_SEGMENT) + 16; }

int lmc_histogram_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                               uint64_t *hist_lo, uint32_t *seg_counts, size_t seg_counts_bytes,
                               huff_stream_t stream) {
    if (hist_hi == nullptr || hist_lo == nullptr || hist_hi == hist_lo || !aligned(hist_hi, 8) ||
        !aligned(hist_lo, 8) || n > kMaxN)
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (w == nullptr || seg_counts == nullptr || !aligned(w, HUFF_ALIGN) ||
                  (x0 != nullptr && !aligned(x0, HUFF_ALIGN)) || !aligned(seg_counts, 4)))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && seg_counts_bytes < lmc_segment_counts_size(n)) return HUFF_ERR_BUFFER_TOO_SMALL;
    // both histograms zeroed by one launch when they are adjacent
    const bool adjacent = hist_lo == hist_hi + 256;
    int st = launch_zero_u64(hist_hi, adjacent ? 512 : 256, cs(stream));
    if (st == HUFF_OK && !adjacent) st = launch_zero_u64(hist_lo, 256, cs(stream));
    if (st != HUFF_OK || n == 0) return st;
    return launch_histogram_bf16_counted(w, x0, n, hist_hi, hist_lo, seg_counts, cs(stream));
}

int lmc_encode_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                            const huff_codebook *cb_lo, size_t chunk_bytes, const uint32_t *seg_counts,
                            size_t seg_counts_bytes, uint8_t *payload_hi, size_t cap_hi, uint64_t *off_hi,
                            uint8_t *payload_lo, size_t cap_lo, uint64_t *off_lo, void *ws, size_t ws_bytes,
                            int32_t *status, huff_stream_t stream) {
    if (cb_hi == nullptr || cb_lo == nullptr || off_hi == nullptr || off_lo == nullptr || status == nullptr ||
        !chunk_ok(chunk_bytes) || n > kMaxN || !aligned(cb_hi, 16) || !aligned(cb_lo, 16) ||
        !aligned(off_hi, 8) || !aligned(off_lo, 8))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (w == nullptr || payload_hi == nullptr || payload_lo == nullptr || ws == nullptr ||
                  seg_counts == nullptr || !aligned(w, HUFF_ALIGN) || (x0 != nullptr && !aligned(x0, HUFF_ALIGN)) ||
                  !aligned(payload_hi, HUFF_ALIGN) || !aligned(payload_lo, HUFF_ALIGN) || !aligned(ws, HUFF_ALIGN) ||
                  !aligned(seg_counts, 4)))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (ws_bytes < lmc_counted_workspace_size(n) || seg_counts_bytes < lmc_segment_counts_size(n)))
        return HUFF_ERR_BUFFER_TOO_SMALL;
    return launch_encode_bf16_counted(w, x0, n, cb_hi, cb_lo, chunk_bytes, seg_counts, payload_hi, cap_hi, off_hi,
                                      payload_lo, cap_lo, off_lo, ws, status, cs(stream));
}

int lmc_decode_bf16(const uint8_t *payload_hi, size_t bytes_hi, const uint64_t *off_hi, const uint8_t *payload_lo,
                    size_t bytes_lo, const uint64_t *off_lo, size_t n, size_t chunk_bytes,
                    const huff_codebook *cb_hi, const huff_codebook *cb_lo, const uint16_t *x0, uint16_t *out,
                    int32_t *status, huff_stream_t stream) {
    if (cb_hi == nullptr || cb_lo == nullptr || status == nullptr || !chunk_ok(chunk_bytes) || n > kMaxN ||
        !aligned(cb_hi, 16) || !aligned(cb_lo, 16))
        return HUFF_ERR_INVALID_ARG;
    if (n > 0 && (payload_hi == nullptr || payload_lo == nullptr || off_hi == nullptr || off_lo == nullptr ||
                  out == nullptr || !aligned(payload_hi, HUFF_ALIGN) || !aligned(payload_lo, HUFF_ALIGN) ||
                  !aligned(out, HUFF_ALIGN) || (x0 != nullptr && !aligned(x0, HUFF_ALIGN)) ||
                  !aligned(off_hi, 8) || !aligned(off_lo, 8) || x0 == out))
        return HUFF_ERR_INVALID_ARG;
    return launch_decode_bf16(payload_hi, bytes_hi, off_hi, payload_lo, bytes_lo, off_lo, n, chunk_bytes, cb_hi,
                              cb_lo, x0, out, status, cs(stream));
}

int huff_code_stats(const uint64_t *h_hist, const uint8_t *h_len, huff_stats *out) {
    if (h_hist == nullptr || h_len == nullptr || out == nullptr) return HUFF_ERR_INVALID_ARG;
    huff_stats r{};
    int st = HUFF_OK;
    for (int s = 0; s < 256; ++s) {
        r.n += h_hist[s];
        r.total_bits += h_hist[s] * h_len[s];
        if (h_hist[s] > 0 && h_len[s] == 0) st = HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK;
    }
    if (r.n > 0) {
        double h = 0.0;
        for (int s = 0; s < 256; ++s) {
            if (h_hist[s] == 0) continue;
            const double p = static_cast<double>(h_hist[s]) / static_cast<double>(r.n);
            h -= p * std::log2(p);
        }
        r.entropy_bits = h;
        r.mean_len = static_cast<double>(r.total_bits) / static_cast<double>(r.n);
        const double nh = static_cast<double>(r.n) * h;
        r.shannon_gap = nh > 0.0 ? (static_cast<double>(r.total_bits) - nh) / nh : 0.0;
    }
    *out = r;
    return st;
}


// ---------------------------------------------------------------- container (host only)

static void le_put(uint8_t *p, uint64_t v, int bytes) {
    for (int k = 0; k < bytes; ++k) p[k] = static_cast<uint8_t>(v >> (8 * k));
}
static uint64_t le_get(const uint8_t *p, int bytes) {
    uint64_t v = 0;
    for (int k = 0; k < bytes; ++k) v |= static_cast<uint64_t>(p[k]) << (8 * k);
    return v;
}

size_t huff_container_size(size_t n, size_t chunk_bytes, uint64_t total_bits, int with_lengths) {
    return HUFF_CONTAINER_HEADER + (with_lengths ? 256 : 0) + 8 * (huff_num_chunks(n, chunk_bytes) + 1) +
           static_cast<size_t>((total_bits + 7) / 8);
}

int huff_container_write(uint8_t *h_dst, size_t cap, size_t n, size_t chunk_bytes, int max_len,
                         const uint8_t *h_len, const uint64_t *h_off, const uint8_t *h_payload,
                         size_t *written) {
    if (h_dst == nullptr || h_off == nullptr || written == nullptr || !chunk_ok(chunk_bytes) || n > kMaxN ||
        max_len < 1 || max_len > HUFF_MAX_LEN)
        return HUFF_ERR_INVALID_ARG;
    const size_t nc = huff_num_chunks(n, chunk_bytes);
    if (h_off[0] != 0) return HUFF_ERR_INVALID_ARG;
    for (size_t c = 0; c < nc; ++c)
        if (h_off[c + 1] < h_off[c]) return HUFF_ERR_INVALID_ARG;
    const uint64_t T = h_off[nc];
    if (T > 0 && h_payload == nullptr) return HUFF_ERR_INVALID_ARG;
    if (h_len != nullptr)
        for (int s = 0; s < 256; ++s)
            if (h_len[s] > max_len) return HUFF_ERR_INVALID_ARG;
    const size_t size = huff_container_size(n, chunk_bytes, T, h_len != nullptr);
    if (cap < size) return HUFF_ERR_BUFFER_TOO_SMALL;
    uint8_t *p = h_dst;
    le_put(p, HUFF_CONTAINER_MAGIC, 4);
    le_put(p + 4, 1, 2);
    le_put(p + 6, h_len != nullptr ? HUFF_CONTAINER_LENGTHS : 0u, 2);
    le_put(p + 8, static_cast<uint64_t>(max_len), 4);
    le_put(p + 12, 0, 4);
    le_put(p + 16, n, 8);
    le_put(p + 24, chunk_bytes, 8);
    le_put(p + 32, nc, 8);
    le_put(p + 40, T, 8);
    p += HUFF_CONTAINER_HEADER;
    if (h_len != nullptr) {
        for (int s = 0; s < 256; ++s) p[s] = h_len[s];
        p += 256;
    }
    for (size_t c = 0; c <= nc; ++c, p += 8) le_put(p, h_off[c], 8);
    const size_t pb = static_cast<size_t>((T + 7) / 8);
    for (size_t i = 0; i < pb; ++i) p[i] = h_payload[i];
    *written = size;
    return HUFF_OK;
}

int huff_container_parse(const uint8_t *h_src, size_t size, huff_container_view *view) {
    if (h_src == nullptr || view == nullptr) return HUFF_ERR_INVALID_ARG;
    if (size < HUFF_CONTAINER_HEADER) return HUFF_ERR_CORRUPT_STREAM;
    if (le_get(h_src, 4) != HUFF_CONTAINER_MAGIC || le_get(h_src + 4, 2) != 1 || le_get(h_src + 12, 4) != 0)
        return HUFF_ERR_CORRUPT_STREAM;
    const uint64_t flags = le_get(h_src + 6, 2);
    const uint64_t max_len = le_get(h_src + 8, 4);
    const uint64_t n = le_get(h_src + 16, 8), chunk = le_get(h_src + 24, 8);
    const uint64_t nc = le_get(h_src + 32, 8), T = le_get(h_src + 40, 8);
    if ((flags & ~static_cast<uint64_t>(HUFF_CONTAINER_LENGTHS)) != 0 || max_len < 1 || max_len > HUFF_MAX_LEN ||
        !chunk_ok(chunk) || n > kMaxN || nc != huff_num_chunks(n, chunk) || T > static_cast<uint64_t>(n) * max_len)
        return HUFF_ERR_CORRUPT_STREAM;
    const bool has_len = (flags & HUFF_CONTAINER_LENGTHS) != 0;
    if (size != huff_container_size(n, chunk, T, has_len)) return HUFF_ERR_CORRUPT_STREAM;
    const uint8_t *p = h_src + HUFF_CONTAINER_HEADER;
    const uint8_t *len = nullptr;
    if (has_len) {
        len = p;
        for (int s = 0; s < 256; ++s)
            if (len[s] > max_len) return HUFF_ERR_CORRUPT_STREAM;
        p += 256;
    }
    const uint8_t *off = p;
    uint64_t prev = 0;
    for (uint64_t c = 0; c <= nc; ++c) {
        const uint64_t o = le_get(off + 8 * c, 8);
        if ((c == 0 && o != 0) || o < prev) return HUFF_ERR_CORRUPT_STREAM;
        prev = o;
    }
    if (prev != T) return HUFF_ERR_CORRUPT_STREAM;
    view->n = n;
    view->chunk_bytes = chunk;
    view->n_chunks = nc;
    view->total_bits = T;
    view->max_len = static_cast<int32_t>(max_len);
    view->has_lengths = has_len ? 1 : 0;
    view->len = len;
    view->off = off;
    view->payload = off + 8 * (nc + 1);
    view->payload_bytes = (T + 7) / 8;
    return HUFF_OK;
}

int huff_debug_wait(int kind, const uint64_t *desc, size_t n_desc, uint32_t seg, uint32_t limit, uint64_t *out,
                    int32_t *status, huff_stream_t stream) {
    if ((kind != 0 && kind != 1) || out == nullptr || status == nullptr || !aligned(out, 8) || limit == 0 ||
        limit > kSpinLimit)
        return HUFF_ERR_INVALID_ARG;
    if (kind == 0 && (desc == nullptr || !aligned(desc, 8) || seg == 0 || seg > n_desc))
        return HUFF_ERR_INVALID_ARG;
    return launch_wait_probe(kind, desc, seg, limit, out, status, cs(stream));
}

}  // extern "C"
