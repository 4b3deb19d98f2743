// histogram.cu -- 256-bin symbol histograms.
//
// "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
// Methodology step 1 (8-bit symbol frequencies) and "Lossless Compression for
// LLM Tensor Incremental Snapshots" (arXiv 2505.09810), technical framework
// stage 2 (frequency statistics of the byte groups).
//
// Design: every CTA keeps 32 privatised copies of the 256 counters in shared
// memory, one per lane index, interleaved bin-major: copy c of bin b is word
// 32 b + c, so lane c only ever touches bank c.  Whatever symbols the lanes of
// a warp see, their 32 updates hit 32 distinct banks: no bank conflict and no
// address serialisation.  The fold sums a bin's 32 copies in an order rotated
// by the bin (thread b reads copy (k + b) mod 32 at step k), so the threads of
// a warp read 32 distinct banks too.  Input is read as 16-byte vectors, four
// per thread in flight.  At the end each CTA folds its copies and adds one
// uint64 per non-zero bin to global memory.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kHistPlaneWords = 256 * kHistCopies;  // one plane's 32 copies

// A lane's copy of the counters: bin b at word 32 b of the lane's column.
struct LaneCopy {
    uint32_t *p;
    __device__ __forceinline__ uint32_t &operator[](uint32_t b) const { return p[b << 5]; }
};

__device__ __forceinline__ void count_word(LaneCopy my, uint32_t w) {
    atomicAdd(&my[w & 0xffu], 1u);
    atomicAdd(&my[(w >> 8) & 0xffu], 1u);
    atomicAdd(&my[(w >> 16) & 0xffu], 1u);
    atomicAdd(&my[w >> 24], 1u);
}

// bytes 0 and 2 (par = 0) or 1 and 3 (par = 1) of a word
__device__ __forceinline__ void count_word_half(LaneCopy my, uint32_t w, int par) {
    w >>= 8 * par;
    atomicAdd(&my[w & 0xffu], 1u);
    atomicAdd(&my[(w >> 16) & 0xffu], 1u);
}

template <int STRIDE>
__device__ __forceinline__ void count_vec(LaneCopy my, uint4 v, int par) {
    if (STRIDE == 1) {
        count_word(my, v.x);
        count_word(my, v.y);
        count_word(my, v.z);
        count_word(my, v.w);
    } else {
        count_word_half(my, v.x, par);
        count_word_half(my, v.y, par);
        count_word_half(my, v.z, par);
        count_word_half(my, v.w, par);
    }
}

__device__ __forceinline__ void flush_copies(const uint32_t *sh, uint64_t *hist) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) {
        uint64_t s = 0;
#pragma unroll 8
        for (int c = 0; c < kHistCopies; ++c) s += sh[b * kHistCopies + ((c + b) & (kHistCopies - 1))];
        if (s) atomicAdd(reinterpret_cast<unsigned long long *>(&hist[b]), static_cast<unsigned long long>(s));
    }
}

template <int STRIDE>
__global__ void __launch_bounds__(kHistThreads) k_histogram(const uint8_t *__restrict__ in, size_t n,
                                                            uint64_t *__restrict__ hist) {
    extern __shared__ uint32_t sh[];
    for (int i = threadIdx.x; i < kHistPlaneWords; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const LaneCopy my{sh + (threadIdx.x & 31)};

    const size_t gtid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
    const uintptr_t base = reinterpret_cast<uintptr_t>(in);
    const uintptr_t end = base + (n ? (n - 1) * STRIDE + 1 : 0);
    const uintptr_t a0 = (base + 15) & ~uintptr_t(15);
    const uintptr_t a1 = end & ~uintptr_t(15);
    const int par = static_cast<int>(base & 1);

    if (n == 0) {
    } else if (a0 >= a1) {
        for (size_t i = gtid; i < n; i += nthreads) atomicAdd(&my[in[i * STRIDE]], 1u);
    } else {
        // ragged head and tail, one byte at a time
        for (uintptr_t a = base + gtid; a < a0; a += nthreads)
            if ((a - base) % STRIDE == 0) atomicAdd(&my[*reinterpret_cast<const uint8_t *>(a)], 1u);
        for (uintptr_t a = a1 + gtid; a < end; a += nthreads)
            if ((a - base) % STRIDE == 0) atomicAdd(&my[*reinterpret_cast<const uint8_t *>(a)], 1u);
        // aligned body, 16-byte vectors, four in flight per thread
        const uint4 *v = reinterpret_cast<const uint4 *>(a0);
        const size_t nv = (a1 - a0) / 16;
        size_t i = gtid;
        for (; i + 3 * nthreads < nv; i += 4 * nthreads) {
            uint4 x0 = __ldcs(v + i);
            uint4 x1 = __ldcs(v + i + nthreads);
            uint4 x2 = __ldcs(v + i + 2 * nthreads);
            uint4 x3 = __ldcs(v + i + 3 * nthreads);
            count_vec<STRIDE>(my, x0, par);
            count_vec<STRIDE>(my, x1, par);
            count_vec<STRIDE>(my, x2, par);
            count_vec<STRIDE>(my, x3, par);
        }
        for (; i < nv; i += nthreads) count_vec<STRIDE>(my, __ldcs(v + i), par);
    }
    __syncthreads();
    flush_copies(sh, hist);
}

// Both byte planes of 16-bit words, optionally of (w ^ x0).
__device__ __forceinline__ void count_pair(LaneCopy hi, LaneCopy lo, uint32_t w) {
    atomicAdd(&lo[w & 0xffu], 1u);
    atomicAdd(&hi[(w >> 8) & 0xffu], 1u);
    atomicAdd(&lo[(w >> 16) & 0xffu], 1u);
    atomicAdd(&hi[w >> 24], 1u);
}

template <bool XOR>
__global__ void __launch_bounds__(kHistThreads) k_histogram_bf16(const uint16_t *__restrict__ w,
                                                                 const uint16_t *__restrict__ x0, size_t n,
                                                                 uint64_t *__restrict__ hist_hi,
                                                                 uint64_t *__restrict__ hist_lo) {
    extern __shared__ uint32_t sh[];
    for (int i = threadIdx.x; i < 2 * kHistPlaneWords; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const LaneCopy hi{sh + (threadIdx.x & 31)};
    const LaneCopy lo{sh + kHistPlaneWords + (threadIdx.x & 31)};

    const size_t gtid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
    const uintptr_t base = reinterpret_cast<uintptr_t>(w);
    const bool vec_ok = !XOR || ((base ^ reinterpret_cast<uintptr_t>(x0)) & 15) == 0;
    // elements before the first 16-byte boundary of w
    size_t head = vec_ok ? ((16 - (base & 15)) & 15) / 2 : n;
    if (head > n) head = n;
    const size_t nv = (n - head) / 8;
    const size_t body_end = head + nv * 8;

    for (size_t i = gtid; i < head; i += nthreads) {
        uint32_t v = w[i] ^ (XOR ? x0[i] : 0);
        atomicAdd(&lo[v & 0xffu], 1u);
        atomicAdd(&hi[v >> 8], 1u);
    }
    for (size_t i = body_end + gtid; i < n; i += nthreads) {
        uint32_t v = w[i] ^ (XOR ? x0[i] : 0);
        atomicAdd(&lo[v & 0xffu], 1u);
        atomicAdd(&hi[v >> 8], 1u);
    }
    const uint4 *vw = reinterpret_cast<const uint4 *>(w + head);
    const uint4 *vx = reinterpret_cast<const uint4 *>(XOR ? x0 + head : w);
    size_t i = gtid;
    for (; i + nthreads < nv; i += 2 * nthreads) {
        uint4 a = __ldcs(vw + i);
        uint4 b = __ldcs(vw + i + nthreads);
        if (XOR) {
            uint4 c = __ldcs(vx + i);
            uint4 d = __ldcs(vx + i + nthreads);
            a.x ^= c.x; a.y ^= c.y; a.z ^= c.z; a.w ^= c.w;
            b.x ^= d.x; b.y ^= d.y; b.z ^= d.z; b.w ^= d.w;
        }
        count_pair(hi, lo, a.x); count_pair(hi, lo, a.y); count_pair(hi, lo, a.z); count_pair(hi, lo, a.w);
        count_pair(hi, lo, b.x); count_pair(hi, lo, b.y); count_pair(hi, lo, b.z); count_pair(hi, lo, b.w);
    }
    for (; i < nv; i += nthreads) {
        uint4 a = __ldcs(vw + i);
        if (XOR) {
            uint4 c = __ldcs(vx + i);
            a.x ^= c.x; a.y ^= c.y; a.z ^= c.z; a.w ^= c.w;
        }
        count_pair(hi, lo, a.x); count_pair(hi, lo, a.y); count_pair(hi, lo, a.z); count_pair(hi, lo, a.w);
    }
    __syncthreads();
    flush_copies(sh, hist_hi);
    flush_copies(sh + kHistPlaneWords, hist_lo);
}

// Both byte planes, per segment of seg_elems elements: each CTA takes whole
// segments; after a segment it folds its 32 copies into the segment's 512
// counts (high plane, then low plane), zeroes them, and keeps a running total
// per bin for the whole-tensor histograms.  Folding costs 0.25 shared-memory
// accesses per element.  w and x0 are 16-byte aligned.
template <bool XOR>
__global__ void __launch_bounds__(kHistThreads) k_histogram_bf16_counted(const uint16_t *__restrict__ w,
                                                                         const uint16_t *__restrict__ x0, size_t n,
                                                                         uint64_t *__restrict__ hist_hi,
                                                                         uint64_t *__restrict__ hist_lo,
                                                                         uint32_t *__restrict__ seg_counts,
                                                                         size_t seg_elems, uint32_t n_seg) {
    static_assert(kHistThreads == kSegCountWords, "one thread per (plane, bin)");
    extern __shared__ uint32_t sh[];
    const int tid = threadIdx.x;
    for (int i = tid; i < 2 * kHistPlaneWords; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const LaneCopy hi{sh + (tid & 31)};
    const LaneCopy lo{sh + kHistPlaneWords + (tid & 31)};
    const int fb = tid & 255;
    uint32_t *fold = sh + (tid >> 8) * kHistPlaneWords + fb * kHistCopies;  // this thread's bin, its 32 copies
    uint64_t total = 0;
    for (uint32_t seg = blockIdx.x; seg < n_seg; seg += gridDim.x) {
        const size_t first = static_cast<size_t>(seg) * seg_elems;
        const size_t cnt = n - first < seg_elems ? n - first : seg_elems;
        const size_t nv = cnt / 8;
        const uint4 *vw = reinterpret_cast<const uint4 *>(w + first);
        const uint4 *vx = reinterpret_cast<const uint4 *>(XOR ? x0 + first : w + first);
        size_t i = tid;
        for (; i + 3 * kHistThreads < nv; i += 4 * kHistThreads) {
            uint4 a[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] = __ldcs(vw + i + j * kHistThreads);
            if (XOR) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 c = __ldcs(vx + i + j * kHistThreads);
                    a[j].x ^= c.x; a[j].y ^= c.y; a[j].z ^= c.z; a[j].w ^= c.w;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                count_pair(hi, lo, a[j].x); count_pair(hi, lo, a[j].y);
                count_pair(hi, lo, a[j].z); count_pair(hi, lo, a[j].w);
            }
        }
        for (; i < nv; i += kHistThreads) {
            uint4 a = __ldcs(vw + i);
            if (XOR) {
                const uint4 c = __ldcs(vx + i);
                a.x ^= c.x; a.y ^= c.y; a.z ^= c.z; a.w ^= c.w;
            }
            count_pair(hi, lo, a.x); count_pair(hi, lo, a.y); count_pair(hi, lo, a.z); count_pair(hi, lo, a.w);
        }
        for (size_t e = nv * 8 + tid; e < cnt; e += kHistThreads) {
            const uint32_t v = w[first + e] ^ (XOR ? x0[first + e] : 0);
            atomicAdd(&lo[v & 0xffu], 1u);
            atomicAdd(&hi[v >> 8], 1u);
        }
        __syncthreads();
        uint32_t s = 0;
#pragma unroll 8
        for (int c = 0; c < kHistCopies; ++c) {
            s += fold[(c + fb) & (kHistCopies - 1)];
            fold[(c + fb) & (kHistCopies - 1)] = 0;
        }
        seg_counts[static_cast<size_t>(seg) * kSegCountWords + tid] = s;
        total += s;
        __syncthreads();
    }
    if (total)
        atomicAdd(reinterpret_cast<unsigned long long *>(tid < 256 ? &hist_hi[tid] : &hist_lo[tid - 256]),
                  static_cast<unsigned long long>(total));
}

__global__ void k_zero_u64(uint64_t *p, size_t count) {
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = 0;
}

template <typename K>
int hist_grid(K kernel, size_t smem, size_t work_items, int *grid) {
    DevInfo d = dev_info();
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return HUFF_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kHistThreads, smem) != cudaSuccess)
        return HUFF_ERR_CUDA;
    if (per_sm < 1) per_sm = 1;
    size_t want = (work_items + kHistThreads - 1) / kHistThreads;
    size_t cap = static_cast<size_t>(d.sms) * per_sm;
    *grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
    return HUFF_OK;
}

}  // namespace

DevInfo dev_info() {
    static DevInfo cache[64];
    static bool have[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && have[dev]) return cache[dev];
    DevInfo d{1, 48 * 1024};
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (dev >= 0 && dev < 64) {
        cache[dev] = d;
        have[dev] = true;
    }
    return d;
}

int launch_zero_u64(uint64_t *p, size_t count, cudaStream_t s) {
    if (count == 0) return HUFF_OK;
    size_t blocks = (count + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_zero_u64<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p, count);
    return launch_status();
}

int launch_histogram(const uint8_t *in, size_t n, size_t stride, uint64_t *hist, cudaStream_t s) {
    const size_t smem = kHistPlaneWords * sizeof(uint32_t);
    int grid = 1, st;
    if (stride == 1) {
        if ((st = hist_grid(k_histogram<1>, smem, n / 64 + 1, &grid)) != HUFF_OK) return st;
        k_histogram<1><<<grid, kHistThreads, smem, s>>>(in, n, hist);
    } else {
        if ((st = hist_grid(k_histogram<2>, smem, n / 32 + 1, &grid)) != HUFF_OK) return st;
        k_histogram<2><<<grid, kHistThreads, smem, s>>>(in, n, hist);
    }
    return launch_status();
}

int launch_histogram_bf16(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                          uint64_t *hist_lo, cudaStream_t s) {
    const size_t smem = 2 * kHistPlaneWords * sizeof(uint32_t);
    int grid = 1, st;
    if (x0 != nullptr) {
        if ((st = hist_grid(k_histogram_bf16<true>, smem, n / 16 + 1, &grid)) != HUFF_OK) return st;
        k_histogram_bf16<true><<<grid, kHistThreads, smem, s>>>(w, x0, n, hist_hi, hist_lo);
    } else {
        if ((st = hist_grid(k_histogram_bf16<false>, smem, n / 16 + 1, &grid)) != HUFF_OK) return st;
        k_histogram_bf16<false><<<grid, kHistThreads, smem, s>>>(w, nullptr, n, hist_hi, hist_lo);
    }
    return launch_status();
}

int launch_histogram_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                                  uint64_t *hist_lo, uint32_t *seg_counts, cudaStream_t s) {
    const size_t smem = 2 * kHistPlaneWords * sizeof(uint32_t);
    const size_t seg_elems = count_seg_elems(n);  // the counted encode's segments
    const size_t n_seg = (n + seg_elems - 1) / seg_elems;
    int grid = 1, st;
    if (x0 != nullptr) {
        if ((st = hist_grid(k_histogram_bf16_counted<true>, smem, n_seg * kHistThreads, &grid)) != HUFF_OK) return st;
        k_histogram_bf16_counted<true><<<grid, kHistThreads, smem, s>>>(w, x0, n, hist_hi, hist_lo, seg_counts,
                                                                         seg_elems, static_cast<uint32_t>(n_seg));
    } else {
        if ((st = hist_grid(k_histogram_bf16_counted<false>, smem, n_seg * kHistThreads, &grid)) != HUFF_OK)
            return st;
        k_histogram_bf16_counted<false><<<grid, kHistThreads, smem, s>>>(w, nullptr, n, hist_hi, hist_lo,
                                                                          seg_counts, seg_elems,
                                                                          static_cast<uint32_t>(n_seg));
    }
    return launch_status();
}

}  // namespace huffk
