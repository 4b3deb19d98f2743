// decode.cu -- chunked Huffman decode.
//
// "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
// 2505.09810), technical framework: decompression reads the data,
// Huffman-decodes it and restores the byte groups; key design 3: the work is
// split into tasks that run in parallel.  The chunk bit offsets written by the
// encoder are those tasks' entry points.
//
// GPU design:
//   * one thread per chunk (byte streams); for the fused bf16 path two
//     adjacent lanes share a chunk pair, one per byte plane, and swap 8
//     decoded bytes per round with a pair shuffle to form 16-bit words;
//   * the codebook's 4096-entry first-level table sits in shared memory; an
//     entry holds every code that fits completely in the 12-bit window (up
//     to three symbols, their count and their total length), so short codes
//     decode several symbols per lookup; codes longer than 12 bits take an
//     out-of-line canonical search (first_code / bl_count);
//   * the bit reader keeps 64 bits in a register, refills 32 at a time from a
//     128-bit queue, and always has the next 16-byte unit of the stream in
//     flight, so global-memory latency stays off the decode chain; reads
//     never pass the payload's end;
//   * decoded bytes gather in a 64-bit accumulator and leave as 8-byte
//     stores; x0 (for the XOR delta) is loaded one group of four rounds ahead.
// Every chunk must end exactly at the next chunk's offset, otherwise
// HUFF_ERR_CORRUPT_STREAM is reported.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kDecBlock = 256;

// 16-byte aligned (and sized) so that arrays of tables keep every lut 16-byte aligned for uint4 copies
struct __align__(16) DecTables {
    uint32_t lut[1u << HUFF_LUT_BITS];  // syms (24 bits) | count << 24 | total bits << 27
    uint32_t bl_count[32];
    uint32_t first_code[32];
    uint32_t first_index[32];
    uint8_t sorted[256];
    uint8_t len[256];
    int longest;
    int ok;
};
static_assert(sizeof(DecTables) % 16 == 0, "table arrays must keep 16-byte alignment");

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
    for (int i = tid; i < 256; i += blockDim.x) {
        T.sorted[i] = ok ? cb->sorted_symbols[i] : 0;
        T.len[i] = ok ? cb->len[i] : 0;
    }
    if (tid == 0) {
        T.longest = ok ? cb->longest : 0;
        T.ok = ok && cb->longest <= HUFF_MAX_LEN;
    }
}

// Bytes of a 16-byte unit past the payload's end read as zero.
__device__ __noinline__ uint4 load_unit_tail(const uint8_t *p, size_t nbytes, size_t u) {
    uint32_t w[4] = {0, 0, 0, 0};
    for (int k = 0; k < 16; ++k) {
        const size_t i = u * 16 + k;
        if (i < nbytes) w[k >> 2] |= static_cast<uint32_t>(p[i]) << (8 * (k & 3));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

struct BitReader {
    const uint8_t *p;
    size_t nbytes;
    size_t ui;        // next 16-byte unit to fetch
    uint64_t buf;     // upcoming bits, most significant first
    int nb;           // valid bits in buf
    uint64_t qh, ql;  // queued big-endian words not yet in buf
    int qn;           // words left in the queue
    uint4 nxt;        // the unit after the queue, in flight

    __device__ __forceinline__ uint4 load_unit(size_t u) const {
        if (u * 16 + 16 <= nbytes) {
            uint4 v;
            asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "l"(p + u * 16));
            return v;
        }
        return load_unit_tail(p, nbytes, u);
    }
    __device__ __forceinline__ void enqueue(uint4 v) {
        qh = (static_cast<uint64_t>(bswap32(v.x)) << 32) | bswap32(v.y);
        ql = (static_cast<uint64_t>(bswap32(v.z)) << 32) | bswap32(v.w);
        qn = 4;
    }
    __device__ __forceinline__ uint32_t pop() {
        const uint32_t w = static_cast<uint32_t>(qh >> 32);
        qh = (qh << 32) | (ql >> 32);
        ql <<= 32;
        if (--qn == 0) {
            enqueue(nxt);
            nxt = load_unit(ui++);
        }
        return w;
    }
    __device__ __forceinline__ void init(uint64_t pos) {
        const size_t u = pos >> 7;
        enqueue(load_unit(u));
        nxt = load_unit(u + 1);
        ui = u + 2;
        for (uint32_t k = 0; k < ((pos >> 5) & 3u); ++k) pop();
        buf = static_cast<uint64_t>(pop()) << 32;
        buf |= pop();
        const int sk = static_cast<int>(pos & 31u);
        buf <<= sk;
        nb = 64 - sk;
    }
    __device__ __forceinline__ void refill() {
        if (nb <= 32) {
            buf |= static_cast<uint64_t>(pop()) << (32 - nb);
            nb += 32;
        }
    }
    __device__ __forceinline__ void consume(uint32_t bits) {
        buf <<= bits;
        nb -= static_cast<int>(bits);
    }
    // bits consumed from the start of the payload
    __device__ __forceinline__ uint64_t pos() const {
        return static_cast<uint64_t>(ui - 1) * 128 - 32 * static_cast<uint64_t>(qn) - static_cast<uint64_t>(nb);
    }
};

// Canonical search for a code longer than the table's 12 bits; L = 0 if none matches.
__device__ __noinline__ uint32_t long_code(uint64_t buf, const DecTables *T, uint32_t *L) {
    const uint32_t v = static_cast<uint32_t>(buf >> (64 - HUFF_MAX_LEN));
    for (int l = HUFF_LUT_BITS + 1; l <= T->longest; ++l) {
        const uint32_t c = v >> (HUFF_MAX_LEN - l);
        const uint32_t d = c - T->first_code[l];
        if (d < T->bl_count[l]) {
            *L = static_cast<uint32_t>(l);
            return T->sorted[T->first_index[l] + d];
        }
    }
    *L = 0;
    return 0;
}

// Pending decoded bytes: byte k of the stream order is byte k of (a0, a1).
struct Pend {
    uint64_t a0, a1;
    int fill;
};

// Decode one table lookup's worth of symbols (1..3, never more than rem > 0).
__device__ __forceinline__ void take(BitReader &r, const DecTables &T, Pend &o, int &rem, bool &bad) {
    r.refill();
    const uint32_t e = T.lut[r.buf >> (64 - HUFF_LUT_BITS)];
    uint32_t c = (e >> 24) & 3u;
    uint32_t bits = e >> 27;
    uint32_t v = e & 0xffffffu;
    if (c == 0) {
        uint32_t L;
        v = long_code(r.buf, &T, &L);
        if (L == 0) {
            bad = true;
            L = 1;
        }
        c = 1;
        bits = L;
    } else if (static_cast<int>(c) > rem) {
        c = static_cast<uint32_t>(rem);
        bits = T.len[v & 0xffu] + (c == 2 ? T.len[(v >> 8) & 0xffu] : 0u);
        v &= c == 1 ? 0xffu : 0xffffu;
    }
    r.consume(bits);
    rem -= static_cast<int>(c);
    const int f = o.fill;
    o.a0 |= static_cast<uint64_t>(v) << (8 * f);
    if (f + static_cast<int>(c) > 8) o.a1 |= static_cast<uint64_t>(v) >> (8 * (8 - f));
    o.fill = f + static_cast<int>(c);
}

__device__ __forceinline__ void shift8(Pend &o) {
    o.a0 = o.a1;
    o.a1 = 0;
    o.fill -= 8;
}

__device__ __forceinline__ bool chunk_bounds(const uint64_t *off, size_t c, size_t nbytes, uint64_t &start,
                                             uint64_t &end) {
    start = off[c];
    end = off[c + 1];
    return start <= end && end <= static_cast<uint64_t>(nbytes) * 8;
}

__global__ void __launch_bounds__(kDecBlock) k_decode_u8(const uint8_t *__restrict__ payload, size_t nbytes,
                                                         const uint64_t *__restrict__ off, size_t n, size_t chunk,
                                                         const huff_codebook *__restrict__ cb,
                                                         uint8_t *__restrict__ out, int32_t *status) {
    __shared__ DecTables T;
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
    BitReader r;
    r.p = payload;
    r.nbytes = nbytes;
    r.init(start);
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint8_t *o = out + first;
    bool bad = false;
    int rem = cnt;
    Pend pd{0, 0, 0};
    int written = 0;
    while (rem > 0) {
        take(r, T, pd, rem, bad);  // fill < 8 before, <= 10 after
        if (pd.fill >= 8) {
            *reinterpret_cast<uint64_t *>(o + written) = pd.a0;
            written += 8;
            shift8(pd);
        }
    }
    for (int k = 0; k < pd.fill; ++k) o[written + k] = static_cast<uint8_t>(pd.a0 >> (8 * k));
    if (bad || r.pos() != end) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

// Lanes 2c (high plane) and 2c + 1 (low plane) decode chunk c of their plane.
template <bool XOR>
__global__ void __launch_bounds__(kDecBlock) k_decode_bf16(
    const uint8_t *__restrict__ pay_hi, size_t bytes_hi, const uint64_t *__restrict__ off_hi,
    const uint8_t *__restrict__ pay_lo, size_t bytes_lo, const uint64_t *__restrict__ off_lo, size_t n,
    size_t chunk, const huff_codebook *__restrict__ cb_hi, const huff_codebook *__restrict__ cb_lo,
    const uint16_t *__restrict__ x0, uint16_t *__restrict__ out, int32_t *status) {
    __shared__ DecTables Tb[2];
    load_tables(Tb[0], cb_hi);
    load_tables(Tb[1], cb_lo);
    __syncthreads();
    if (!Tb[0].ok || !Tb[1].ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const size_t g = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t c = g >> 1;
    const int plane = static_cast<int>(g & 1);  // 0: high byte, 1: low byte
    if (c >= n_chunks) return;                   // both lanes of a pair leave together
    const unsigned pair = 3u << (threadIdx.x & 30u);
    const DecTables &T = Tb[plane];
    const uint8_t *pay = plane ? pay_lo : pay_hi;
    const size_t nbytes = plane ? bytes_lo : bytes_hi;
    const uint64_t *off = plane ? off_lo : off_hi;
    uint64_t start, end;
    const bool ok = chunk_bounds(off, c, nbytes, start, end);
    if (!ok) set_status(status, HUFF_ERR_CORRUPT_STREAM);
    if (__any_sync(pair, !ok)) return;
    BitReader r;
    r.p = pay;
    r.nbytes = nbytes;
    r.init(start);
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint16_t *o = out + first;
    const uint16_t *x = XOR ? x0 + first : nullptr;
    bool bad = false;
    int rem = cnt;
    Pend pd{0, 0, 0};
    // x0 words of this lane (4 elements per round) for the current and the next group of 4 rounds
    uint64_t xq[4] = {0, 0, 0, 0}, xn[4] = {0, 0, 0, 0};
    if (XOR) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int base = 8 * q + 4 * plane;
            if (base + 4 <= cnt) xq[q] = __ldcs(reinterpret_cast<const unsigned long long *>(x + base));
        }
    }
    for (int k = 0; k < cnt; k += 32) {
        if (XOR) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int base = k + 32 + 8 * q + 4 * plane;
                if (base + 4 <= cnt) xn[q] = __ldcs(reinterpret_cast<const unsigned long long *>(x + base));
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int kk = k + 8 * q;
            if (kk < cnt) {
                const int want = cnt - kk < 8 ? cnt - kk : 8;
                while (pd.fill < want) take(r, T, pd, rem, bad);
                const uint64_t mine = pd.a0;
                const uint64_t other = __shfl_xor_sync(pair, mine, 1);
                const uint64_t hi8 = plane ? other : mine;
                const uint64_t lo8 = plane ? mine : other;
                // element j = lo byte j | hi byte j << 8; the high lane writes elements 0-3, the low lane 4-7
                const uint32_t l32 = static_cast<uint32_t>(plane ? lo8 >> 32 : lo8);
                const uint32_t h32 = static_cast<uint32_t>(plane ? hi8 >> 32 : hi8);
                uint64_t wv = (static_cast<uint64_t>(__byte_perm(l32, h32, 0x7362)) << 32) |
                              __byte_perm(l32, h32, 0x5140);
                const int base = kk + 4 * plane;
                if (base + 4 <= cnt) {
                    if (XOR) wv ^= xq[q];
                    __stcs(reinterpret_cast<unsigned long long *>(o + base), static_cast<unsigned long long>(wv));
                } else {
                    for (int j = 0; j < 4 && base + j < cnt; ++j) {
                        uint16_t v = static_cast<uint16_t>(wv >> (16 * j));
                        if (XOR) v ^= x[base + j];
                        o[base + j] = v;
                    }
                }
                if (want == 8) shift8(pd);
                else pd.fill = 0;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) xq[q] = xn[q];
    }
    if (bad || r.pos() != end) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

}  // namespace

int launch_decode_u8(const uint8_t *payload, size_t bytes, const uint64_t *off, size_t n, size_t chunk,
                     const huff_codebook *cb, uint8_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const unsigned grid = static_cast<unsigned>((n_chunks + kDecBlock - 1) / kDecBlock);
    k_decode_u8<<<grid, kDecBlock, 0, s>>>(payload, bytes, off, n, chunk, cb, out, status);
    return launch_status();
}

int launch_decode_bf16(const uint8_t *pay_hi, size_t bytes_hi, const uint64_t *off_hi, const uint8_t *pay_lo,
                       size_t bytes_lo, const uint64_t *off_lo, size_t n, size_t chunk,
                       const huff_codebook *cb_hi, const huff_codebook *cb_lo, const uint16_t *x0,
                       uint16_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const unsigned grid = static_cast<unsigned>((2 * n_chunks + kDecBlock - 1) / kDecBlock);
    if (x0 != nullptr)
        k_decode_bf16<true><<<grid, kDecBlock, 0, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo, n,
                                                       chunk, cb_hi, cb_lo, x0, out, status);
    else
        k_decode_bf16<false><<<grid, kDecBlock, 0, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo, n,
                                                        chunk, cb_hi, cb_lo, nullptr, out, status);
    return launch_status();
}

}  // namespace huffk
