// bytegroup.cu -- byte grouping of 16-bit tensors and the XOR snapshot delta.
//
// "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
// 2505.09810): technical framework stage 1 and key design 1 (byte grouping;
// here the high and low byte of each bf16 word form two planes), the
// decompression step that restores the byte groups, and the English
// abstract's incremental delta compression between snapshots (read as XOR of
// the bit patterns).
//
// Streaming kernels: 16-byte vector loads and stores with byte permutes, grid
// sized to a few CTAs per SM with a grid-stride loop.  A scalar loop handles
// pointers that are not 16-byte aligned and the ragged end.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kStreamThreads = 256;

unsigned stream_grid(size_t items) {
    const size_t cap = static_cast<size_t>(dev_info().sms) * 8;
    size_t g = (items + kStreamThreads - 1) / kStreamThreads;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

__device__ __forceinline__ bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

__global__ void __launch_bounds__(kStreamThreads) k_split(const uint16_t *__restrict__ w, size_t n,
                                                          uint8_t *__restrict__ hi, uint8_t *__restrict__ lo) {
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (aligned16(w) && aligned16(hi) && aligned16(lo)) {
        const size_t nv = n / 16;  // 16 elements -> 32 bytes in, 16 + 16 bytes out
        const uint4 *src = reinterpret_cast<const uint4 *>(w);
        uint4 *dh = reinterpret_cast<uint4 *>(hi);
        uint4 *dl = reinterpret_cast<uint4 *>(lo);
        for (size_t i = tid; i < nv; i += stride) {
            const uint4 a = __ldcs(src + 2 * i);
            const uint4 b = __ldcs(src + 2 * i + 1);
            __stcs(dl + i, make_uint4(__byte_perm(a.x, a.y, 0x6420), __byte_perm(a.z, a.w, 0x6420),
                                      __byte_perm(b.x, b.y, 0x6420), __byte_perm(b.z, b.w, 0x6420)));
            __stcs(dh + i, make_uint4(__byte_perm(a.x, a.y, 0x7531), __byte_perm(a.z, a.w, 0x7531),
                                      __byte_perm(b.x, b.y, 0x7531), __byte_perm(b.z, b.w, 0x7531)));
        }
        done = nv * 16;
    }
    for (size_t i = done + tid; i < n; i += stride) {
        const uint16_t v = w[i];
        hi[i] = static_cast<uint8_t>(v >> 8);
        lo[i] = static_cast<uint8_t>(v & 0xffu);
    }
}

__global__ void __launch_bounds__(kStreamThreads) k_merge(const uint8_t *__restrict__ hi,
                                                          const uint8_t *__restrict__ lo, size_t n,
                                                          uint16_t *__restrict__ w) {
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (aligned16(w) && aligned16(hi) && aligned16(lo)) {
        const size_t nv = n / 16;
        const uint4 *sh = reinterpret_cast<const uint4 *>(hi);
        const uint4 *sl = reinterpret_cast<const uint4 *>(lo);
        uint4 *dst = reinterpret_cast<uint4 *>(w);
        for (size_t i = tid; i < nv; i += stride) {
            const uint4 h = __ldcs(sh + i);
            const uint4 l = __ldcs(sl + i);
            __stcs(dst + 2 * i, make_uint4(__byte_perm(l.x, h.x, 0x5140), __byte_perm(l.x, h.x, 0x7362),
                                           __byte_perm(l.y, h.y, 0x5140), __byte_perm(l.y, h.y, 0x7362)));
            __stcs(dst + 2 * i + 1, make_uint4(__byte_perm(l.z, h.z, 0x5140), __byte_perm(l.z, h.z, 0x7362),
                                               __byte_perm(l.w, h.w, 0x5140), __byte_perm(l.w, h.w, 0x7362)));
        }
        done = nv * 16;
    }
    for (size_t i = done + tid; i < n; i += stride)
        w[i] = static_cast<uint16_t>((static_cast<uint16_t>(hi[i]) << 8) | lo[i]);
}

__global__ void __launch_bounds__(kStreamThreads) k_xor(const uint16_t *a, const uint16_t *b, size_t n,
                                                        uint16_t *out) {
    // no __restrict__: out may alias a or b (each element is read before it is written by the same thread)
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (aligned16(a) && aligned16(b) && aligned16(out)) {
        const size_t nv = n / 8;
        const uint4 *va = reinterpret_cast<const uint4 *>(a);
        const uint4 *vb = reinterpret_cast<const uint4 *>(b);
        uint4 *vo = reinterpret_cast<uint4 *>(out);
        for (size_t i = tid; i < nv; i += stride) {
            const uint4 x = va[i];
            const uint4 y = vb[i];
            vo[i] = make_uint4(x.x ^ y.x, x.y ^ y.y, x.z ^ y.z, x.w ^ y.w);
        }
        done = nv * 8;
    }
    for (size_t i = done + tid; i < n; i += stride) out[i] = static_cast<uint16_t>(a[i] ^ b[i]);
}

// Byte planes of W-byte words (W = 1, 2, 4, 8): plane p holds byte W-1-p of
// every word (most significant first, so for IEEE floats plane 0 is the sign
// and the high exponent bits).  Plane p starts at planes + p * ps (ps >= n).  A thread moves 16
// words at a time: W 16-byte loads, one 16-byte store per plane.
template <int W>
__device__ __forceinline__ uint32_t byte_of(const uint32_t (&r)[4 * W], int b) {
    return (r[b >> 2] >> (8 * (b & 3))) & 0xffu;
}

template <int W>
__global__ void __launch_bounds__(kStreamThreads) k_split_w(const uint8_t *__restrict__ in, size_t n,
                                                            uint8_t *__restrict__ planes, size_t ps) {
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (aligned16(in) && aligned16(planes) && n % 16 == 0 && ps % 16 == 0) {
        const size_t nv = n / 16;
        for (size_t v = tid; v < nv; v += stride) {
            uint32_t r[4 * W];
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(in + (v * 16) * W) + j);
                r[4 * j] = a.x; r[4 * j + 1] = a.y; r[4 * j + 2] = a.z; r[4 * j + 3] = a.w;
            }
#pragma unroll
            for (int p = 0; p < W; ++p) {
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[q] = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[q] |= byte_of<W>(r, (4 * q + i) * W + (W - 1 - p)) << (8 * i);
                }
                __stcs(reinterpret_cast<uint4 *>(planes + p * ps + v * 16), make_uint4(o[0], o[1], o[2], o[3]));
            }
        }
        done = nv * 16;
    }
    for (size_t i = done + tid; i < n; i += stride)
#pragma unroll
        for (int p = 0; p < W; ++p) planes[p * ps + i] = in[i * W + (W - 1 - p)];
}

template <int W>
__global__ void __launch_bounds__(kStreamThreads) k_merge_w(const uint8_t *__restrict__ planes, size_t n,
                                                            size_t ps, uint8_t *__restrict__ out) {
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (aligned16(out) && aligned16(planes) && n % 16 == 0 && ps % 16 == 0) {
        const size_t nv = n / 16;
        for (size_t v = tid; v < nv; v += stride) {
            uint32_t pl[4 * W];  // 16 bytes of each plane
#pragma unroll
            for (int p = 0; p < W; ++p) {
                const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(planes + p * ps + v * 16));
                pl[4 * p] = a.x; pl[4 * p + 1] = a.y; pl[4 * p + 2] = a.z; pl[4 * p + 3] = a.w;
            }
#pragma unroll
            for (int j = 0; j < W; ++j) {  // output vector j: bytes 16 j .. 16 j + 15 of the 16 words
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[q] = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int b = 16 * j + 4 * q + i;  // byte b of the block = byte b % W of word b / W
                        const int p = W - 1 - b % W;
                        o[q] |= byte_of<W>(pl, 16 * p + b / W) << (8 * i);
                    }
                }
                __stcs(reinterpret_cast<uint4 *>(out + (v * 16) * W) + j, make_uint4(o[0], o[1], o[2], o[3]));
            }
        }
        done = nv * 16;
    }
    for (size_t i = done + tid; i < n; i += stride)
#pragma unroll
        for (int p = 0; p < W; ++p) out[i * W + (W - 1 - p)] = planes[p * ps + i];
}

}  // namespace

int launch_split(const uint16_t *w, size_t n, uint8_t *hi, uint8_t *lo, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    k_split<<<stream_grid(n / 16 + 1), kStreamThreads, 0, s>>>(w, n, hi, lo);
    return launch_status();
}

int launch_merge(const uint8_t *hi, const uint8_t *lo, size_t n, uint16_t *w, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    k_merge<<<stream_grid(n / 16 + 1), kStreamThreads, 0, s>>>(hi, lo, n, w);
    return launch_status();
}

int launch_xor(const uint16_t *a, const uint16_t *b, size_t n, uint16_t *out, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    k_xor<<<stream_grid(n / 8 + 1), kStreamThreads, 0, s>>>(a, b, n, out);
    return launch_status();
}

int launch_split_w(const uint8_t *in, size_t n, int width, uint8_t *planes, size_t ps, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const unsigned g = stream_grid(n / 16 + 1);
    switch (width) {
        case 1: k_split_w<1><<<g, kStreamThreads, 0, s>>>(in, n, planes, ps); break;
        case 2: k_split_w<2><<<g, kStreamThreads, 0, s>>>(in, n, planes, ps); break;
        case 4: k_split_w<4><<<g, kStreamThreads, 0, s>>>(in, n, planes, ps); break;
        case 8: k_split_w<8><<<g, kStreamThreads, 0, s>>>(in, n, planes, ps); break;
        default: return HUFF_ERR_INVALID_ARG;
    }
    return launch_status();
}

int launch_merge_w(const uint8_t *planes, size_t n, int width, size_t ps, uint8_t *out, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const unsigned g = stream_grid(n / 16 + 1);
    switch (width) {
        case 1: k_merge_w<1><<<g, kStreamThreads, 0, s>>>(planes, n, ps, out); break;
        case 2: k_merge_w<2><<<g, kStreamThreads, 0, s>>>(planes, n, ps, out); break;
        case 4: k_merge_w<4><<<g, kStreamThreads, 0, s>>>(planes, n, ps, out); break;
        case 8: k_merge_w<8><<<g, kStreamThreads, 0, s>>>(planes, n, ps, out); break;
        default: return HUFF_ERR_INVALID_ARG;
    }
    return launch_status();
}

}  // namespace huffk
