// encode.cu -- single-pass chunked Huffman encode.
//
// "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
// Methodology step 4: tensors are encoded directly with a precomputed
// codebook, with no per-batch analysis.  "Lossless Compression for LLM Tensor
// Incremental Snapshots" (arXiv 2505.09810), technical framework stage 3
// (Huffman coding of each byte group) and key design 3 (split into tasks that
// run in parallel).
//
// Output format: codes appended MSB first into one contiguous stream; the bit
// offset of every chunk start is recorded so chunks decode independently.
//
// GPU design (one pass over the input):
//   * persistent CTAs claim 8 KiB input tiles from an atomic counter, so a
//     tile's predecessors are always claimed by running CTAs;
//   * each CTA keeps a 3-stage ring of tiles in flight, fetched with 1-D bulk
//     copies (cp.async.bulk) completing on mbarriers;
//   * (code << 8 | len) comes from a shared-memory table replicated kLutRep
//     times so that lanes with different symbols spread over more banks;
//   * a block scan gives each thread its bit offset inside the tile; the tile
//     publishes its bit count and finds its global bit offset with a
//     warp-wide decoupled lookback (Merrill & Garland, "Single-pass Parallel
//     Prefix Scan with Decoupled Look-back", 2016);
//   * codes are packed into a tile-local shared-memory bit buffer while the
//     lookback is in flight (only the partial words at thread boundaries use
//     shared atomics), then written out shifted by the tile's bit phase with
//     coalesced 32-bit stores;
//   * the word that straddles two tiles is owned by the later tile: each tile
//     publishes its trailing partial word and its successor ORs it in.
//   The fused bf16 variant reads 16-bit words (and optionally x0, for the XOR
//   delta), and encodes the high and low byte planes as two streams in the
//   same pass.  All waits are bounded; a wait that runs out sets
//   HUFF_ERR_TIMEOUT and the kernel carries on to completion.
#include "common.cuh"

namespace huffk {

namespace {

struct EncPlane {
    const huff_codebook *cb;
    uint32_t *payload;  // 32-bit words; payload byte 4w + j = bits 31-8j .. 24-8j of word w
    size_t cap_words;
    uint64_t *off;
    uint64_t *desc;  // per-tile lookback descriptors
    uint64_t *tail;  // per-tile trailing partial word (kTailValid | word)
};

template <bool BF16, bool XOR>
struct EncCfg {
    static constexpr int kPlanes = BF16 ? 2 : 1;
    static constexpr int kSyms = BF16 ? kEncBf16ElemsPerThread : kEncU8SymsPerThread;  // per plane, per thread
    static constexpr int kTileSyms = kEncThreads * kSyms;
    static constexpr int kTileBytes = 8192;  // per input array
    static constexpr int kInputs = XOR ? 2 : 1;
    static constexpr int kBufWords = kTileSyms * HUFF_MAX_LEN / 32 + 4;
    static constexpr int kLutWords = 256 * kLutRep;
    static constexpr size_t kMiscBytes = 256;
    static constexpr size_t kRingBytes = size_t(kEncStages) * kInputs * kTileBytes;
    static constexpr size_t kLutBytes = size_t(kPlanes) * kLutWords * 4;
    static constexpr size_t kBufBytes = size_t(kPlanes) * kBufWords * 4;
    static constexpr size_t kSmem = kMiscBytes + kRingBytes + kLutBytes + kBufBytes;
    static_assert(kTileSyms * (BF16 ? 2 : 1) == kTileBytes, "tile geometry");
};

struct Misc {
    uint64_t mbar[kEncStages];
    uint64_t warp_sum[kEncThreads / 32];
    uint64_t prefix[2];
    uint32_t tile_q[kEncStages];
    uint32_t prev_words[2];
    int32_t bad_codebook;
};
static_assert(sizeof(Misc) <= 256, "misc area");

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Warp-wide decoupled lookback for tile t of one stream; returns the tile's
// exclusive bit offset.  Called by all 32 lanes of one warp.
__device__ uint64_t lookback(uint64_t *desc, uint32_t t, uint64_t total, int lane, int32_t *status) {
    if (t == 0) {
        if (lane == 0) st_release(&desc[0], kFlagPrefix | total);
        return 0;
    }
    if (lane == 0) st_release(&desc[t], kFlagAggregate | total);
    uint64_t excl = 0;
    int64_t base = static_cast<int64_t>(t) - 1;
    unsigned spins = 0;
    for (;;) {
        const int64_t idx = base - lane;
        const uint64_t d = idx >= 0 ? ld_acquire(&desc[idx]) : kFlagPrefix;
        const uint32_t flag = static_cast<uint32_t>(d >> 62);
        const unsigned pmask = __ballot_sync(0xffffffffu, flag == 2);
        const unsigned zmask = __ballot_sync(0xffffffffu, flag == 0);
        // lanes up to and including the nearest inclusive prefix must all be published
        const unsigned need = pmask ? ((pmask & (0u - pmask)) << 1) - 1u : 0xffffffffu;
        if ((zmask & need) == 0) {
            const uint64_t v = ((need >> lane) & 1u) ? (d & kValueMask) : 0;
            excl += warp_sum_u64(v);
            if (pmask) break;
            base -= 32;
        } else {
            ++spins;
            const bool give_up = spins > kSpinLimit || ((spins & 255u) == 0 && error_recorded(status));
            if (__any_sync(0xffffffffu, give_up)) {
                if (lane == 0 && spins > kSpinLimit) set_status(status, HUFF_ERR_TIMEOUT);
                break;
            }
            __nanosleep(20);
        }
    }
    if (lane == 0) st_release(&desc[t], kFlagPrefix | (excl + total));
    return excl;
}

// Pack `count` (code << 8 | len) entries starting at tile-local bit `start`.
// Words wholly inside this thread's bits are stored; the partial words at
// either end are OR-ed (the buffer is zero before packing).
template <int N>
__device__ __forceinline__ void pack_bits(uint32_t *buf, uint32_t start, const uint32_t (&e)[N]) {
    uint64_t acc = 0;
    uint32_t nb = start & 31u;
    uint32_t w = start >> 5;
    bool first_partial = nb != 0;
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const uint32_t L = e[k] & 0xffu;
        acc = (acc << L) | (e[k] >> 8);
        nb += L;
        if (nb >= 32) {
            nb -= 32;
            const uint32_t word = static_cast<uint32_t>(acc >> nb);
            if (first_partial) {
                atomicOr(&buf[w], word);
                first_partial = false;
            } else {
                buf[w] = word;
            }
            ++w;
        }
    }
    if (nb > 0) atomicOr(&buf[w], static_cast<uint32_t>(acc << (32 - nb)));
}

// Global word i of a tile whose bits start at phase ph, from the tile-local buffer.
__device__ __forceinline__ uint32_t shifted_word(const uint32_t *buf, uint32_t i, uint32_t ph) {
    if (ph == 0) return buf[i];
    const uint32_t lo = buf[i] >> ph;
    return i == 0 ? lo : (lo | (buf[i - 1] << (32 - ph)));
}

__device__ __forceinline__ void put_word(const EncPlane &p, uint64_t gw, uint32_t v, int32_t *status) {
    if (gw < p.cap_words)
        p.payload[gw] = bswap32(v);
    else
        set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
}

template <bool BF16, bool XOR>
__device__ __forceinline__ void issue_tile(uint8_t *ring, uint64_t *mbar, int s, uint32_t t, const uint8_t *in,
                                           const uint8_t *in2, size_t n) {
    using C = EncCfg<BF16, XOR>;
    const size_t first = static_cast<size_t>(t) * C::kTileSyms;
    const size_t cnt = n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms);
    const uint32_t bytes = static_cast<uint32_t>(cnt * (BF16 ? 2 : 1)) & ~15u;
    mbar_arrive_expect_tx(&mbar[s], bytes * C::kInputs);
    if (bytes) {
        const size_t src = first * (BF16 ? 2 : 1);
        uint8_t *dst = ring + size_t(s) * C::kInputs * C::kTileBytes;
        bulk_g2s(dst, in + src, bytes, &mbar[s]);
        if (XOR) bulk_g2s(dst + C::kTileBytes, in2 + src, bytes, &mbar[s]);
    }
}

template <bool BF16, bool XOR>
__global__ void __launch_bounds__(kEncThreads) k_encode(const uint8_t *__restrict__ in,
                                                        const uint8_t *__restrict__ in2, size_t n, EncPlane p0,
                                                        EncPlane p1, size_t chunk, uint32_t n_tiles,
                                                        unsigned *tile_ctr, int32_t *status) {
    using C = EncCfg<BF16, XOR>;
    extern __shared__ __align__(128) uint8_t smem[];
    Misc *ms = reinterpret_cast<Misc *>(smem);
    uint8_t *ring = smem + C::kMiscBytes;
    uint32_t *lut = reinterpret_cast<uint32_t *>(ring + C::kRingBytes);
    uint32_t *bufs = lut + C::kPlanes * C::kLutWords;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // code table: entry (s * kLutRep + r) = (code << 8) | len, 0 when the symbol has no code
    if (tid == 0) ms->bad_codebook = 0;
    __syncthreads();
#pragma unroll
    for (int p = 0; p < C::kPlanes; ++p) {
        const huff_codebook *cb = p == 0 ? p0.cb : p1.cb;
        const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC;
        if (!ok && tid == 0) ms->bad_codebook = 1;
        for (int i = tid; i < C::kLutWords; i += kEncThreads) {
            const int s = i / kLutRep;
            const uint32_t L = ok ? cb->len[s] : 0u;
            lut[p * C::kLutWords + i] = (L >= 1 && L <= HUFF_MAX_LEN) ? ((cb->code[s] << 8) | L) : 0u;
        }
    }
    for (int i = tid; i < C::kPlanes * C::kBufWords; i += kEncThreads) bufs[i] = 0;
    if (tid == 0) {
        for (int s = 0; s < kEncStages; ++s) mbar_init(&ms->mbar[s], 1);
        ms->prev_words[0] = ms->prev_words[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (ms->bad_codebook && tid == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
    if (tid == 0) {
        for (int s = 0; s < kEncStages; ++s) {
            const uint32_t t = atomicAdd(tile_ctr, 1u);
            ms->tile_q[s] = t;
            if (t < n_tiles) issue_tile<BF16, XOR>(ring, ms->mbar, s, t, in, in2, n);
        }
    }
    __syncthreads();

    const size_t n_chunks = (n + chunk - 1) / chunk;
    for (uint32_t iter = 0;; ++iter) {
        const int s = static_cast<int>(iter % kEncStages);
        const uint32_t t = *reinterpret_cast<volatile uint32_t *>(&ms->tile_q[s]);
        if (t >= n_tiles) break;
        if (!mbar_wait(&ms->mbar[s], (iter / kEncStages) & 1u)) {
            if (tid == 0) set_status(status, HUFF_ERR_TIMEOUT);
        }

        // ---- my 32 input bytes (and x0's) from the ring
        const size_t first = static_cast<size_t>(t) * C::kTileSyms;
        const int tile_n = static_cast<int>(n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms));
        const uint8_t *stage = ring + size_t(s) * C::kInputs * C::kTileBytes;
        uint32_t wv[8];
        {
            const uint4 a = *reinterpret_cast<const uint4 *>(stage + tid * 32);
            const uint4 b = *reinterpret_cast<const uint4 *>(stage + tid * 32 + 16);
            wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
            wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
            if (XOR) {
                const uint4 c = *reinterpret_cast<const uint4 *>(stage + C::kTileBytes + tid * 32);
                const uint4 d = *reinterpret_cast<const uint4 *>(stage + C::kTileBytes + tid * 32 + 16);
                wv[0] ^= c.x; wv[1] ^= c.y; wv[2] ^= c.z; wv[3] ^= c.w;
                wv[4] ^= d.x; wv[5] ^= d.y; wv[6] ^= d.z; wv[7] ^= d.w;
            }
        }
        const int es = BF16 ? 2 : 1;
        const int tile_bytes = tile_n * es;
        const int tma_bytes = tile_bytes & ~15;
        if (tid * 32 + 32 > tma_bytes && tid * 32 < tile_bytes) {
            // ragged end of the last tile: bytes the bulk copy did not cover come from global memory
            for (int k = 0; k < 32; ++k) {
                const int b = tid * 32 + k;
                if (b < tma_bytes) continue;
                uint32_t v = 0;
                if (b < tile_bytes) {
                    v = in[first * es + b];
                    if (XOR) v ^= in2[first * es + b];
                }
                wv[k >> 2] = (wv[k >> 2] & ~(0xffu << (8 * (k & 3)))) | (v << (8 * (k & 3)));
            }
        }
        __syncthreads();  // (A) stage consumed, tile_q[s] read, previous tile's buffers read
        if (tid == 0) {
            const uint32_t nt = atomicAdd(tile_ctr, 1u);
            ms->tile_q[s] = nt;
            if (nt < n_tiles) {
                fence_proxy_async_smem();
                issue_tile<BF16, XOR>(ring, ms->mbar, s, nt, in, in2, n);
            }
        }
#pragma unroll
        for (int p = 0; p < C::kPlanes; ++p)
            for (uint32_t i = tid; i < ms->prev_words[p]; i += kEncThreads) bufs[p * C::kBufWords + i] = 0;

        // ---- code lookup
        const int nvalid = tile_n - tid * C::kSyms < 0 ? 0 : (tile_n - tid * C::kSyms > C::kSyms ? C::kSyms : tile_n - tid * C::kSyms);
        const int r = lane & (kLutRep - 1);
        uint32_t e0[C::kSyms];
        uint32_t e1[BF16 ? C::kSyms : 1];
        uint32_t bits0 = 0, bits1 = 0, mn = 0xffffffffu;
        if (BF16) {
#pragma unroll
            for (int k = 0; k < C::kSyms; ++k) {
                const uint32_t v = (wv[k >> 1] >> (16 * (k & 1))) & 0xffffu;
                uint32_t hi = lut[(v >> 8) * kLutRep + r];
                uint32_t lo = lut[C::kLutWords + (v & 0xffu) * kLutRep + r];
                if (k >= nvalid) hi = lo = 0;
                else mn = min(mn, min(hi, lo));
                e0[k] = hi;
                e1[k] = lo;
                bits0 += hi & 0xffu;
                bits1 += lo & 0xffu;
            }
        } else {
#pragma unroll
            for (int k = 0; k < C::kSyms; ++k) {
                const uint32_t sym = (wv[k >> 2] >> (8 * (k & 3))) & 0xffu;
                uint32_t v = lut[sym * kLutRep + r];
                if (k >= nvalid) v = 0;
                else mn = min(mn, v);
                e0[k] = v;
                bits0 += v & 0xffu;
            }
        }
        if (nvalid > 0 && mn == 0) set_status(status, HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK);

        // ---- block scan of (bits_hi << 32 | bits_lo)
        const uint64_t mine = BF16 ? ((uint64_t(bits0) << 32) | bits1) : uint64_t(bits0);
        uint64_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) ms->warp_sum[warp] = incl;
        __syncthreads();  // (B)
        uint64_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kEncThreads / 32; ++w) {
            const uint64_t ws = ms->warp_sum[w];
            before += w < warp ? ws : 0;
            total += ws;
        }
        const uint64_t excl = before + incl - mine;
        const uint32_t excl0 = BF16 ? uint32_t(excl >> 32) : uint32_t(excl);
        const uint32_t excl1 = uint32_t(excl);
        const uint32_t tot0 = BF16 ? uint32_t(total >> 32) : uint32_t(total);
        const uint32_t tot1 = uint32_t(total);

        // ---- lookback (warp p for plane p) overlapped with packing by the other warps
        if (warp < C::kPlanes) {
            const uint64_t pre = lookback(warp == 0 ? p0.desc : p1.desc, t, warp == 0 ? tot0 : tot1, lane, status);
            if (lane == 0) ms->prefix[warp] = pre;
        }
        pack_bits(bufs, excl0, e0);
        if (BF16) pack_bits(bufs + C::kBufWords, excl1, e1);
        __syncthreads();  // (C) buffers and prefixes complete

        // ---- chunk offsets
#pragma unroll
        for (int p = 0; p < C::kPlanes; ++p) {
            const uint64_t pre = ms->prefix[p];
            const size_t g = first + size_t(tid) * C::kSyms;
            uint64_t *off = p == 0 ? p0.off : p1.off;
            if (nvalid > 0 && g % chunk == 0) off[g / chunk] = pre + (p == 0 ? excl0 : excl1);
            if (tid == 0 && t + 1 == n_tiles) off[n_chunks] = pre + (p == 0 ? tot0 : tot1);
        }

        // ---- shifted write-out
#pragma unroll
        for (int p = 0; p < C::kPlanes; ++p) {
            const EncPlane &P = p == 0 ? p0 : p1;
            const uint32_t *buf = bufs + p * C::kBufWords;
            const uint64_t pre = ms->prefix[p];
            const uint32_t ph = static_cast<uint32_t>(pre & 31u);
            const uint64_t g0 = pre >> 5;
            const uint32_t tot = p == 0 ? tot0 : tot1;
            const uint32_t nfull = (ph + tot) >> 5;  // complete global words touched by this tile
            const bool has_tail = ((ph + tot) & 31u) != 0;
            for (uint32_t i = (ph ? 1u : 0u) + tid; i < nfull; i += kEncThreads)
                put_word(P, g0 + i, shifted_word(buf, i, ph), status);
            if (tid == 32 * p) {
                uint32_t pt = 0;
                if (ph) {
                    // the head word straddles the predecessor: wait for its trailing bits
                    uint64_t v = 0;
                    for (unsigned k = 0;; ++k) {
                        v = ld_acquire(&P.tail[t - 1]);
                        if (v & kTailValid) break;
                        if (k > kSpinLimit) {
                            set_status(status, HUFF_ERR_TIMEOUT);
                            break;
                        }
                        if ((k & 255u) == 255u && error_recorded(status)) break;
                        __nanosleep(20);
                    }
                    pt = static_cast<uint32_t>(v);
                }
                const uint32_t head = pt | shifted_word(buf, 0, ph);
                uint32_t tail_word = 0;
                if (has_tail) tail_word = nfull == 0 ? head : shifted_word(buf, nfull, ph);
                st_release(&P.tail[t], kTailValid | tail_word);
                if (ph && nfull >= 1) put_word(P, g0, head, status);
                if (has_tail && t + 1 == n_tiles) put_word(P, g0 + nfull, tail_word, status);
                ms->prev_words[p] = (tot + 31) >> 5;
            }
        }
    }
}

template <bool BF16, bool XOR>
int run_encode(const uint8_t *in, const uint8_t *in2, size_t n, const EncPlane &p0, const EncPlane &p1,
               size_t chunk, uint32_t n_tiles, unsigned *ctr, int32_t *status, cudaStream_t s) {
    using C = EncCfg<BF16, XOR>;
    auto kern = k_encode<BF16, XOR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) !=
        cudaSuccess)
        return HUFF_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kEncThreads, C::kSmem) != cudaSuccess)
        return HUFF_ERR_CUDA;
    if (per_sm < 1) return HUFF_ERR_CUDA;
    const DevInfo d = dev_info();
    size_t grid = static_cast<size_t>(d.sms) * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    kern<<<static_cast<unsigned>(grid), kEncThreads, C::kSmem, s>>>(in, in2, n, p0, p1, chunk, n_tiles, ctr,
                                                                    status);
    return launch_status();
}

__global__ void k_encode_empty(uint64_t *off0, uint64_t *off1) {
    off0[0] = 0;
    if (off1) off1[0] = 0;
}

}  // namespace

size_t enc_u8_tiles(size_t n) { return (n + kEncU8Tile - 1) / kEncU8Tile; }
size_t enc_bf16_tiles(size_t n) { return (n + kEncBf16Tile - 1) / kEncBf16Tile; }

int launch_encode_u8(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk, uint8_t *payload,
                     size_t cap, uint64_t *off, void *ws, int32_t *status, cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off, nullptr);
        return launch_status();
    }
    const size_t tiles = enc_u8_tiles(n);
    uint64_t *w = static_cast<uint64_t *>(ws);
    int st = launch_zero_u64(w, 2 * tiles + 2, s);
    if (st != HUFF_OK) return st;
    EncPlane p0{cb, reinterpret_cast<uint32_t *>(payload), cap / 4, off, w, w + tiles};
    EncPlane p1 = p0;
    unsigned *ctr = reinterpret_cast<unsigned *>(w + 2 * tiles);
    return run_encode<false, false>(in, nullptr, n, p0, p1, chunk, static_cast<uint32_t>(tiles), ctr, status, s);
}

int launch_encode_bf16(const uint16_t *w16, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                       const huff_codebook *cb_lo, size_t chunk, uint8_t *pay_hi, size_t cap_hi, uint64_t *off_hi,
                       uint8_t *pay_lo, size_t cap_lo, uint64_t *off_lo, void *ws, int32_t *status,
                       cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off_hi, off_lo);
        return launch_status();
    }
    const size_t tiles = enc_bf16_tiles(n);
    uint64_t *w = static_cast<uint64_t *>(ws);
    int st = launch_zero_u64(w, 4 * tiles + 2, s);
    if (st != HUFF_OK) return st;
    EncPlane p0{cb_hi, reinterpret_cast<uint32_t *>(pay_hi), cap_hi / 4, off_hi, w, w + tiles};
    EncPlane p1{cb_lo, reinterpret_cast<uint32_t *>(pay_lo), cap_lo / 4, off_lo, w + 2 * tiles, w + 3 * tiles};
    unsigned *ctr = reinterpret_cast<unsigned *>(w + 4 * tiles);
    const uint8_t *a = reinterpret_cast<const uint8_t *>(w16);
    if (x0 != nullptr)
        return run_encode<true, true>(a, reinterpret_cast<const uint8_t *>(x0), n, p0, p1, chunk,
                                      static_cast<uint32_t>(tiles), ctr, status, s);
    return run_encode<true, false>(a, nullptr, n, p0, p1, chunk, static_cast<uint32_t>(tiles), ctr, status, s);
}

}  // namespace huffk
