// decode.cu -- chunked Huffman decode.
//
// "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
// 2505.09810), technical framework: decompression reads the data,
// Huffman-decodes it and restores the byte groups; key design 3: the work is
// split into tasks that run in parallel.  The chunk bit offsets written by the
// encoder are those tasks' entry points.
//
// GPU design:
//   * the codebook's 4096-entry first-level table sits in shared memory; an
//     entry lists every code that lies wholly inside a 12-bit window (up to
//     six symbols, their count and their total length), so short codes decode
//     several symbols per lookup; codes longer than 12 bits take an
//     out-of-line canonical search (first_code / bl_count);
//   * the bit reader keeps 64 bits in a register, refills 32 at a time from a
//     128-bit queue, and always has the next two 16-byte units of the stream
//     in flight, so global-memory latency stays off the decode chain; reads
//     never pass the payload's end;
//   * byte streams: one thread per chunk, decoded bytes leave as 8-byte stores;
//   * fused bf16: one thread per chunk pair decodes 64 symbols of each byte
//     plane per segment into private shared-memory rows (one lookup per loop
//     iteration, stores predicated, so the lanes of a warp stay in step),
//     then merges them into 16-bit words, XORs x0 (loaded before the
//     segment's decode, so its latency hides behind it) and stores 128 bytes;
//     no barrier couples the threads.
// Every chunk must end exactly at the next chunk's offset, otherwise
// HUFF_ERR_CORRUPT_STREAM is reported.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kDecBlock = 256;

// 16-byte aligned (and sized) so that arrays of tables keep every lut 16-byte aligned for uint4 copies
struct __align__(16) DecTables {
    uint64_t lut[1u << HUFF_LUT_BITS];  // syms (48 bits) | count << 48 | total bits << 52
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
    for (int i = tid; i < (1 << HUFF_LUT_BITS) / 2; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
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
    uint32_t bh, bl;  // upcoming bits (64, most significant first): bh = first 32
    int nb;           // valid bits in (bh, bl)
    uint64_t qh, ql;  // queued big-endian words not yet in the bit buffer
    int qn;           // words left in the queue
    uint4 nxt, nxt2;  // the two units after the queue, in flight

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
            nxt = nxt2;
            nxt2 = load_unit(ui++);
        }
        return w;
    }
    __device__ __forceinline__ void init(uint64_t pos) {
        const size_t u = pos >> 7;
        enqueue(load_unit(u));
        nxt = load_unit(u + 1);
        nxt2 = load_unit(u + 2);
        ui = u + 3;
        for (uint32_t k = 0; k < ((pos >> 5) & 3u); ++k) pop();
        bh = pop();
        bl = pop();
        nb = 64;
        consume(static_cast<uint32_t>(pos & 31u));
    }
    // drop `bits` (< 32) leading bits
    __device__ __forceinline__ void consume(uint32_t bits) {
        bh = __funnelshift_l(bl, bh, bits);
        bl <<= bits;
        nb -= static_cast<int>(bits);
    }
    __device__ __forceinline__ void refill() {
        if (nb <= 32) {
            const uint32_t w = pop();
            const int s = 32 - nb;  // free bits in bl, 0..32
            if (s == 32) {
                bh = w;  // nb == 0: every bit of the buffer is free
            } else {
                bh |= s ? (w >> (32 - s)) : 0u;
                bl |= w << s;
            }
            nb += 32;
        }
    }
    __device__ __forceinline__ uint64_t top64() const { return (static_cast<uint64_t>(bh) << 32) | bl; }
    // bits consumed from the start of the payload
    __device__ __forceinline__ uint64_t pos() const {
        return static_cast<uint64_t>(ui - 2) * 128 - 32 * static_cast<uint64_t>(qn) - static_cast<uint64_t>(nb);
    }
};

// Canonical search for a code longer than the table's 12 bits: returns
// (length << 8) | symbol, length 0 if no code matches.
__device__ __noinline__ uint32_t long_code(uint32_t top, const DecTables *T) {
    const uint32_t v = top >> (32 - HUFF_MAX_LEN);
    for (int l = HUFF_LUT_BITS + 1; l <= T->longest; ++l) {
        const uint32_t c = v >> (HUFF_MAX_LEN - l);
        const uint32_t d = c - T->first_code[l];
        if (d < T->bl_count[l]) return (static_cast<uint32_t>(l) << 8) | T->sorted[T->first_index[l] + d];
    }
    return 0;
}

// The rare case where a table entry holds more symbols than the chunk has
// left: the total length of its first c symbols.
__device__ __noinline__ uint32_t clamped_bits(uint64_t v, uint32_t c, const DecTables *T) {
    uint32_t bits = 0;
    for (uint32_t k = 0; k < c; ++k) bits += T->len[(v >> (8 * k)) & 0xffu];
    return bits;
}

// Pending decoded bytes: byte k of the stream order is byte k of (a0, a1).
struct Pend {
    uint64_t a0, a1;
    int fill;  // < 8 before a take, <= 7 + HUFF_LUT_SYMS after
};

// Decode one table lookup's worth of symbols (1..HUFF_LUT_SYMS, never more than rem > 0).
__device__ __forceinline__ void take(BitReader &r, const DecTables &T, Pend &o, int &rem, bool &bad) {
    r.refill();
    const uint64_t e = T.lut[r.bh >> (32 - HUFF_LUT_BITS)];
    uint32_t c = static_cast<uint32_t>(e >> 48) & 15u;
    uint32_t bits = static_cast<uint32_t>(e >> 52) & 15u;
    uint64_t v = e & 0xffffffffffffull;
    if (c == 0) {
        const uint32_t lc = long_code(r.bh, &T);
        uint32_t L = lc >> 8;
        if (L == 0) {
            bad = true;
            L = 1;
        }
        v = lc & 0xffu;
        c = 1;
        bits = L;
    } else if (static_cast<int>(c) > rem) {
        c = static_cast<uint32_t>(rem);
        bits = clamped_bits(v, c, &T);
        v &= (1ull << (8 * c)) - 1ull;
    }
    r.consume(bits);
    rem -= static_cast<int>(c);
    const int f = o.fill;
    o.a0 |= v << (8 * f);
    if (f + static_cast<int>(c) > 8) o.a1 |= v >> (8 * (8 - f));
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
    while (rem > 0) {  // one lookup per iteration keeps the lanes in step
        take(r, T, pd, rem, bad);
        if (pd.fill >= 8) {
            *reinterpret_cast<uint64_t *>(o + written) = pd.a0;
            written += 8;
            shift8(pd);
        }
    }
    while (pd.fill >= 8) {
        *reinterpret_cast<uint64_t *>(o + written) = pd.a0;
        written += 8;
        shift8(pd);
    }
    for (int k = 0; k < pd.fill; ++k) o[written + k] = static_cast<uint8_t>(pd.a0 >> (8 * k));
    if (bad || r.pos() != end) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

constexpr int kSegB = 64;                                    // elements per lane per segment
constexpr int kRowB = kSegB + 8;                              // staging row pitch (spreads the lanes' rows over banks)
constexpr size_t kBf16Smem = 2 * sizeof(DecTables) + size_t(2) * kDecBlock * kRowB;

// Decode one plane's symbols up to `target` into its staging row (row byte k
// = stream symbol seg0 + k).  Every iteration does one table lookup and, when
// 8 bytes are ready, one 8-byte store: the lanes of a warp run the same
// instructions and only the trip count differs.  Symbols decoded past
// `target` stay in the accumulator for the next segment.
__device__ __forceinline__ void decode_row(BitReader &r, const DecTables &T, Pend &pd, int &rem, int &written,
                                           int target, int seg0, uint8_t *row, bool &bad) {
    while (written < target) {
        if (rem > 0) take(r, T, pd, rem, bad);  // fill <= 7 before, <= 13 after
        if (pd.fill >= 8) {
            *reinterpret_cast<uint64_t *>(row + (written - seg0)) = pd.a0;
            written += 8;
            shift8(pd);
        } else if (rem == 0) {
            *reinterpret_cast<uint64_t *>(row + (written - seg0)) = pd.a0;
            written += pd.fill;
            pd.fill = 0;
            pd.a0 = 0;
        }
    }
}

// Each thread owns one chunk pair: per segment it decodes 64 symbols of the
// high-byte plane, then 64 of the low-byte plane, into two private
// shared-memory rows, then merges them into 16-bit words, XORs x0 and stores
// 128 bytes.  Long segments let the lanes' varying symbols-per-lookup even
// out before the warp's lanes meet again.  No barrier couples the threads, and every lane of a warp runs
// the same plane at the same time.
template <bool XOR>
__global__ void __launch_bounds__(kDecBlock) k_decode_bf16(
    const uint8_t *__restrict__ pay_hi, size_t bytes_hi, const uint64_t *__restrict__ off_hi,
    const uint8_t *__restrict__ pay_lo, size_t bytes_lo, const uint64_t *__restrict__ off_lo, size_t n,
    size_t chunk, const huff_codebook *__restrict__ cb_hi, const huff_codebook *__restrict__ cb_lo,
    const uint16_t *__restrict__ x0, uint16_t *__restrict__ out, int32_t *status) {
    extern __shared__ __align__(16) uint8_t dsm[];
    DecTables *Tb = reinterpret_cast<DecTables *>(dsm);
    load_tables(Tb[0], cb_hi);
    load_tables(Tb[1], cb_lo);
    __syncthreads();
    if (!Tb[0].ok || !Tb[1].ok) {
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
    uint8_t *hrow = dsm + 2 * sizeof(DecTables) + static_cast<size_t>(threadIdx.x) * kRowB;
    uint8_t *lrow = hrow + static_cast<size_t>(kDecBlock) * kRowB;
    BitReader rh, rl;
    rh.p = pay_hi;
    rh.nbytes = bytes_hi;
    rh.init(sh);
    rl.p = pay_lo;
    rl.nbytes = bytes_lo;
    rl.init(sl);
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint16_t *o = out + first;
    const uint16_t *x = XOR ? x0 + first : nullptr;
    bool bad = false;
    int remh = cnt, reml = cnt, wh = 0, wl = 0;
    Pend ph{0, 0, 0}, pl{0, 0, 0};
    for (int seg0 = 0; seg0 < cnt; seg0 += kSegB) {
        const int target = cnt - seg0 < kSegB ? cnt : seg0 + kSegB;
        const bool full = target == seg0 + kSegB;
        uint4 xq[kSegB / 8];  // x0 of the whole segment, in flight while the planes decode
        if (XOR && full) {
#pragma unroll
            for (int g = 0; g < kSegB / 8; ++g) xq[g] = __ldcs(reinterpret_cast<const uint4 *>(x + seg0) + g);
        }
        decode_row(rh, Tb[0], ph, remh, wh, target, seg0, hrow, bad);
        decode_row(rl, Tb[1], pl, reml, wl, target, seg0, lrow, bad);
#pragma unroll
        for (int g = 0; g < kSegB / 8; ++g) {
            const int e0 = seg0 + 8 * g;  // first of this group's 8 elements
            if (e0 >= target) break;
            const uint2 h = *reinterpret_cast<const uint2 *>(hrow + 8 * g);
            const uint2 l = *reinterpret_cast<const uint2 *>(lrow + 8 * g);
            uint4 v = make_uint4(__byte_perm(l.x, h.x, 0x5140), __byte_perm(l.x, h.x, 0x7362),
                                 __byte_perm(l.y, h.y, 0x5140), __byte_perm(l.y, h.y, 0x7362));
            if (e0 + 8 <= target) {
                if (XOR) {
                    const uint4 xv = full ? xq[g] : __ldcs(reinterpret_cast<const uint4 *>(x + e0));
                    v.x ^= xv.x; v.y ^= xv.y; v.z ^= xv.z; v.w ^= xv.w;
                }
                __stcs(reinterpret_cast<uint4 *>(o + e0), v);
            } else {
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (e0 + k < target) {
                        uint16_t val = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
                        if (XOR) val ^= x[e0 + k];
                        o[e0 + k] = val;
                    }
                }
            }
        }
    }
    if (bad || rh.pos() != eh || rl.pos() != el) set_status(status, HUFF_ERR_CORRUPT_STREAM);
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
    const unsigned grid = static_cast<unsigned>((n_chunks + kDecBlock - 1) / kDecBlock);
    if (x0 != nullptr) {
        if (cudaFuncSetAttribute(k_decode_bf16<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kBf16Smem)) != cudaSuccess)
            return HUFF_ERR_CUDA;
        k_decode_bf16<true><<<grid, kDecBlock, kBf16Smem, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo,
                                                               n, chunk, cb_hi, cb_lo, x0, out, status);
    } else {
        if (cudaFuncSetAttribute(k_decode_bf16<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kBf16Smem)) != cudaSuccess)
            return HUFF_ERR_CUDA;
        k_decode_bf16<false><<<grid, kDecBlock, kBf16Smem, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo,
                                                                off_lo, n, chunk, cb_hi, cb_lo, nullptr, out,
                                                                status);
    }
    return launch_status();
}

}  // namespace huffk
