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

}  // namespace huffk
