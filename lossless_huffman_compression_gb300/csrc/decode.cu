// decode.cu -- chunked Huffman decode.
//
// "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
// 2505.09810), technical framework: decompression reads the data,
// Huffman-decodes it and restores the byte groups; key design 3: the work is
// split into tasks that run in parallel.  The chunk bit offsets written by the
// encoder are those tasks' entry points.
//
// GPU design: one thread per chunk (per chunk pair for the fused bf16 path).
// Each CTA copies the codebook's 4096-entry first-level table into shared
// memory; a 12-bit window of the bit buffer yields (length, symbol) for every
// code of up to 12 bits in one lookup, and longer codes (up to 24 bits) fall
// back to the canonical first_code / bl_count search.  The bit reader keeps 64
// bits in a register and refills 32 at a time from big-endian words; reads
// never pass the payload's end.  Symbols are gathered in registers and stored
// 16 bytes at a time.  Every chunk must end exactly at the next chunk's offset,
// otherwise HUFF_ERR_CORRUPT_STREAM is reported.
#include "common.cuh"

namespace huffk {

namespace {

struct DecTables {
    uint32_t lut[1u << HUFF_LUT_BITS];
    uint32_t bl_count[32];
    uint32_t first_code[32];
    uint32_t first_index[32];
    uint8_t sorted[256];
    int longest;
    int ok;
};

__device__ void load_tables(DecTables &T, const huff_codebook *cb) {
    const int tid = threadIdx.x;
    const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC;
    const uint4 *src = reinterpret_cast<const uint4 *>(cb->lut);
    uint4 *dst = reinterpret_cast<uint4 *>(T.lut);
    for (int i = tid; i < (1 << HUFF_LUT_BITS) / 4; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
    if (tid < 32) {
        T.bl_count[tid] = ok ? cb->bl_count[tid] : 0;
        T.first_code[tid] = ok ? cb->first_code[tid] : 0;
        T.first_index[tid] = ok ? cb->first_index[tid] : 0;
    }
    for (int i = tid; i < 256; i += blockDim.x) T.sorted[i] = ok ? cb->sorted_symbols[i] : 0;
    if (tid == 0) {
        T.longest = ok ? cb->longest : 0;
        T.ok = ok && cb->longest <= HUFF_MAX_LEN;
    }
}

struct BitReader {
    const uint32_t *words;
    size_t nbytes;
    size_t wi;     // next word to load
    uint64_t buf;  // upcoming bits, most significant first
    int nb;        // valid bits in buf

    __device__ __forceinline__ uint32_t word(size_t i) const {
        if (i * 4 + 4 <= nbytes) return bswap32(ld_nc_u32(words + i));
        uint32_t v = 0;
        const uint8_t *b = reinterpret_cast<const uint8_t *>(words);
        for (int j = 0; j < 4; ++j) {
            const size_t k = i * 4 + j;
            v = (v << 8) | (k < nbytes ? b[k] : 0u);
        }
        return v;
    }
    __device__ __forceinline__ void init(uint64_t pos) {
        wi = pos >> 5;
        buf = (static_cast<uint64_t>(word(wi)) << 32) | word(wi + 1);
        wi += 2;
        const int sk = static_cast<int>(pos & 31);
        buf <<= sk;
        nb = 64 - sk;
    }
    __device__ __forceinline__ void refill() {
        if (nb <= 32) {
            buf |= static_cast<uint64_t>(word(wi++)) << (32 - nb);
            nb += 32;
        }
    }
    __device__ __forceinline__ uint64_t pos() const { return static_cast<uint64_t>(wi) * 32 - nb; }
};

// One symbol; sets `bad` on an invalid code.
__device__ __forceinline__ uint32_t decode_sym(BitReader &r, const DecTables &T, bool &bad) {
    r.refill();
    const uint32_t e = T.lut[r.buf >> (64 - HUFF_LUT_BITS)];
    uint32_t L, sym;
    if (e != 0) {
        L = e >> 8;
        sym = e & 0xffu;
    } else {
        const uint32_t v = static_cast<uint32_t>(r.buf >> (64 - HUFF_MAX_LEN));
        L = 0;
        sym = 0;
        for (int l = HUFF_LUT_BITS + 1; l <= T.longest; ++l) {
            const uint32_t c = v >> (HUFF_MAX_LEN - l);
            const uint32_t d = c - T.first_code[l];
            if (d < T.bl_count[l]) {
                L = static_cast<uint32_t>(l);
                sym = T.sorted[T.first_index[l] + d];
                break;
            }
        }
        if (L == 0) {
            bad = true;
            L = 1;
        }
    }
    r.buf <<= L;
    r.nb -= static_cast<int>(L);
    return sym;
}

__device__ __forceinline__ bool chunk_bounds(const uint64_t *off, size_t c, size_t nbytes, uint64_t &start,
                                             uint64_t &end) {
    start = off[c];
    end = off[c + 1];
    return start <= end && end <= static_cast<uint64_t>(nbytes) * 8;
}

__global__ void __launch_bounds__(kDecThreads) k_decode_u8(const uint8_t *__restrict__ payload, size_t nbytes,
                                                           const uint64_t *__restrict__ off, size_t n,
                                                           size_t chunk, const huff_codebook *__restrict__ cb,
                                                           uint8_t *__restrict__ out, int32_t *status) {
    __shared__ __align__(16) DecTables T;
    load_tables(T, cb);
    __syncthreads();
    if (!T.ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= n_chunks) return;
    uint64_t start, end;
    if (!chunk_bounds(off, c, nbytes, start, end)) {
        set_status(status, HUFF_ERR_CORRUPT_STREAM);
        return;
    }
    BitReader r{reinterpret_cast<const uint32_t *>(payload), nbytes, 0, 0, 0};
    r.init(start);
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint8_t *o = out + first;
    bool bad = false;
    int k = 0;
    for (; k + 16 <= cnt; k += 16) {
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j >> 2] |= decode_sym(r, T, bad) << (8 * (j & 3));
        *reinterpret_cast<uint4 *>(o + k) = make_uint4(w[0], w[1], w[2], w[3]);
        if (r.pos() > end) break;  // corrupt: stop early, reported below
    }
    for (; k < cnt && r.pos() <= end; ++k) o[k] = static_cast<uint8_t>(decode_sym(r, T, bad));
    if (bad || r.pos() != end || k < cnt) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

template <bool XOR>
__global__ void __launch_bounds__(kDecThreads) k_decode_bf16(
    const uint8_t *__restrict__ pay_hi, size_t bytes_hi, const uint64_t *__restrict__ off_hi,
    const uint8_t *__restrict__ pay_lo, size_t bytes_lo, const uint64_t *__restrict__ off_lo, size_t n,
    size_t chunk, const huff_codebook *__restrict__ cb_hi, const huff_codebook *__restrict__ cb_lo,
    const uint16_t *__restrict__ x0, uint16_t *__restrict__ out, int32_t *status) {
    __shared__ __align__(16) DecTables Th;
    __shared__ __align__(16) DecTables Tl;
    load_tables(Th, cb_hi);
    load_tables(Tl, cb_lo);
    __syncthreads();
    if (!Th.ok || !Tl.ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= n_chunks) return;
    uint64_t sh, eh, sl, el;
    if (!chunk_bounds(off_hi, c, bytes_hi, sh, eh) || !chunk_bounds(off_lo, c, bytes_lo, sl, el)) {
        set_status(status, HUFF_ERR_CORRUPT_STREAM);
        return;
    }
    BitReader rh{reinterpret_cast<const uint32_t *>(pay_hi), bytes_hi, 0, 0, 0};
    BitReader rl{reinterpret_cast<const uint32_t *>(pay_lo), bytes_lo, 0, 0, 0};
    rh.init(sh);
    rl.init(sl);
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint16_t *o = out + first;
    const uint16_t *x = XOR ? x0 + first : nullptr;
    bool bad = false;
    int k = 0;
    for (; k + 8 <= cnt; k += 8) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t h0 = decode_sym(rh, Th, bad);
            const uint32_t l0 = decode_sym(rl, Tl, bad);
            const uint32_t h1 = decode_sym(rh, Th, bad);
            const uint32_t l1 = decode_sym(rl, Tl, bad);
            w[j] = l0 | (h0 << 8) | (l1 << 16) | (h1 << 24);
        }
        uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
        if (XOR) {
            const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(x + k));
            v.x ^= a.x; v.y ^= a.y; v.z ^= a.z; v.w ^= a.w;
        }
        __stcs(reinterpret_cast<uint4 *>(o + k), v);
        if (rh.pos() > eh || rl.pos() > el) break;
    }
    for (; k < cnt && rh.pos() <= eh && rl.pos() <= el; ++k) {
        const uint32_t h = decode_sym(rh, Th, bad);
        const uint32_t l = decode_sym(rl, Tl, bad);
        uint16_t v = static_cast<uint16_t>((h << 8) | l);
        if (XOR) v ^= x[k];
        o[k] = v;
    }
    if (bad || rh.pos() != eh || rl.pos() != el || k < cnt) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

}  // namespace

int launch_decode_u8(const uint8_t *payload, size_t bytes, const uint64_t *off, size_t n, size_t chunk,
                     const huff_codebook *cb, uint8_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const unsigned grid = static_cast<unsigned>((n_chunks + kDecThreads - 1) / kDecThreads);
    k_decode_u8<<<grid, kDecThreads, 0, s>>>(payload, bytes, off, n, chunk, cb, out, status);
    return launch_status();
}

int launch_decode_bf16(const uint8_t *pay_hi, size_t bytes_hi, const uint64_t *off_hi, const uint8_t *pay_lo,
                       size_t bytes_lo, const uint64_t *off_lo, size_t n, size_t chunk,
                       const huff_codebook *cb_hi, const huff_codebook *cb_lo, const uint16_t *x0,
                       uint16_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const unsigned grid = static_cast<unsigned>((n_chunks + kDecThreads - 1) / kDecThreads);
    if (x0 != nullptr)
        k_decode_bf16<true><<<grid, kDecThreads, 0, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo, n,
                                                         chunk, cb_hi, cb_lo, x0, out, status);
    else
        k_decode_bf16<false><<<grid, kDecThreads, 0, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo, n,
                                                          chunk, cb_hi, cb_lo, nullptr, out, status);
    return launch_status();
}

}  // namespace huffk
