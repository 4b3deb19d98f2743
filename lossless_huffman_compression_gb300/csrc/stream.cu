// stream.cu -- moving a compressed stream between device buffers.
//
// "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
// Practical impact: with one fixed codebook on every accelerator, compressed
// tensors go between accelerators without a codebook exchange.  One process
// on one GPU stands in for the link with a device-to-device copy of the
// stream.  The stream's size is known only on the device (T =
// chunk_bit_off[n_chunks], written by the encode), so the copy reads T there
// and moves the stream's words (4 ceil(T / 32) bytes) and the n_chunks + 1
// offsets, with no host round trip between the encode and the decode.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) k_stream_copy(const uint8_t *__restrict__ src, size_t src_bytes,
                                                              const uint64_t *__restrict__ off, size_t n_chunks,
                                                              uint8_t *__restrict__ dst, size_t dst_cap,
                                                              uint64_t *__restrict__ dst_off, int32_t *status) {
    const uint64_t T = off[n_chunks];
    if (T > static_cast<uint64_t>(src_bytes) * 8) {  // a size the source buffer cannot hold
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, HUFF_ERR_CORRUPT_STREAM);
        return;
    }
    // the stream through the end of its last 32-bit word (the encode writes whole words), or
    // the whole source when that is shorter
    size_t bytes = static_cast<size_t>((T + 31) / 32) * 4;
    bytes = bytes < src_bytes ? bytes : src_bytes;
    if (bytes > dst_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
        return;
    }
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nt = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = tid; i <= n_chunks; i += nt) dst_off[i] = off[i];
    // src and dst are 16-byte aligned: whole 16-byte vectors, then the last bytes one by one
    const size_t nv = bytes / 16;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    for (size_t i = tid; i < nv; i += nt) d4[i] = __ldcs(s4 + i);
    for (size_t i = nv * 16 + tid; i < bytes; i += nt) dst[i] = src[i];
}

}  // namespace

int launch_stream_copy(const uint8_t *src, size_t src_bytes, const uint64_t *off, size_t n_chunks, uint8_t *dst,
                       size_t dst_cap, uint64_t *dst_off, int32_t *status, cudaStream_t s) {
    // the size is on the device: size the grid for the capacity, at most a few waves
    const size_t want = (dst_cap / 16 + kCopyThreads - 1) / kCopyThreads;
    const size_t most = static_cast<size_t>(dev_info().sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want > most ? most : want));
    k_stream_copy<<<grid, kCopyThreads, 0, s>>>(src, src_bytes, off, n_chunks, dst, dst_cap, dst_off, status);
    return launch_status();
}

}  // namespace huffk
