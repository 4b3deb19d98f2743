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
//   * a persistent, cooperatively launched grid (all CTAs co-resident) walks
//     8 KiB input tiles round-robin: CTA b takes tiles b, b + G, b + 2G, ...;
//   * each CTA keeps a ring of tiles in flight, fetched with 1-D bulk copies
//     (cp.async.bulk) that complete on mbarriers;
//   * 8 consumer warps look up (code << 8 | len) in a shared-memory table
//     replicated kLutRep times (lanes with different symbols spread over more
//     banks), scan the per-thread bit counts, publish the tile's bit count,
//     and pack the codes into a tile-local bit buffer (double-buffered);
//   * a ninth, scheduler warp issues the bulk copies and, one iteration
//     behind, resolves each tile's global bit offset with a decoupled
//     lookback (Merrill & Garland, "Single-pass Parallel Prefix Scan with
//     Decoupled Look-back", 2016) over a window of 384 predecessor
//     descriptors read with independent relaxed loads, so the lookback costs
//     one memory round trip and hides behind the next tile's work;
//   * the consumers then write the previous tile's whole 32-bit words,
//     shifted by its bit phase, with coalesced stores, and its chunk offsets;
//   * the two partial words at each tile boundary are left in the workspace
//     and written by a small fix-up kernel, so no CTA ever waits for another
//     CTA's output.
//   The fused bf16 variant reads 16-bit words (and optionally x0, for the XOR
//   delta) and encodes the high and low byte planes as two streams in one
//   pass.  All waits are bounded; a wait that runs out sets HUFF_ERR_TIMEOUT
//   and the kernel carries on to completion.
#include <mutex>

#include "common.cuh"

namespace huffk {

// Workspace for huff_encode_noalloc: two 64-bit words per 8 KiB tile, enough
// for HUFF_NOALLOC_MAX_SYMBOLS symbols.  Every GPU that loads the library
// keeps these 2 MiB until the process exits; all calls share them.
constexpr size_t kNoAllocScratchWords = 2 * (HUFF_NOALLOC_MAX_SYMBOLS / kEncU8Tile);
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocScratchWords];

namespace {

constexpr int kConsumers = kEncThreads;           // 8 consumer warps
constexpr int kThreads = kConsumers + 32;         // + 1 scheduler warp
constexpr int kLookbackPerLane = 12;              // descriptors per lane per lookback step
constexpr int kBarAll = 1;                        // named barrier: all 288 threads
constexpr int kBarCons = 2;                       // named barrier: the 256 consumers

struct EncPlane {
    const huff_codebook *cb;
    uint32_t *payload;  // 32-bit words; payload byte 4w + j = bits 31-8j .. 24-8j of word w
    size_t cap_words;
    uint64_t *off;
    uint64_t *desc;     // per-tile lookback descriptors (zeroed before the launch)
    uint64_t *edge;     // per-tile boundary words: head bits << 32 | tail bits
};

template <bool BF16, bool XOR>
struct EncCfg {
    static constexpr int kPlanes = BF16 ? 2 : 1;
    static constexpr int kSyms = BF16 ? kEncBf16ElemsPerThread : kEncU8SymsPerThread;  // per plane, per thread
    static constexpr int kTileSyms = kConsumers * kSyms;
    static constexpr int kTileBytes = 8192;  // per input array
    static constexpr int kInputs = XOR ? 2 : 1;
    static constexpr int kBufWords = kTileSyms * HUFF_MAX_LEN / 32 + 4;
    static constexpr int kLutWords = 256 * kLutRep;
    static constexpr size_t kMiscBytes = 512;
    static constexpr size_t kRingBytes = size_t(kEncStages) * kInputs * kTileBytes;
    static constexpr size_t kLutBytes = size_t(kPlanes) * kLutWords * 4;
    static constexpr size_t kBufBytes = size_t(2) * kPlanes * kBufWords * 4;  // two slots
    static constexpr size_t kSmem = kMiscBytes + kRingBytes + kLutBytes + kBufBytes;
    static_assert(kTileSyms * (BF16 ? 2 : 1) == kTileBytes, "tile geometry");
};

struct Misc {
    uint64_t full[kEncStages];
    uint64_t warp_sum[kConsumers / 32];
    uint64_t prefix[2][2];  // [slot][plane] exclusive bit offset, from the scheduler
    uint32_t total[2][2];   // [slot][plane] tile bit count, from the consumers
    int32_t bad_codebook;
};
static_assert(sizeof(Misc) <= 512, "misc area");

__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Decoupled lookback for tile t of one stream, by one full warp, over windows
// of 32 * kLookbackPerLane predecessors; returns the exclusive bit offset.
// The tile's own aggregate is already published.
__device__ uint64_t lookback(const uint64_t *desc, uint32_t t, int lane, int32_t *status) {
    if (t == 0) return 0;
    uint64_t excl = 0;
    int64_t base = static_cast<int64_t>(t) - 1;
    unsigned spins = 0;
    for (;;) {
        uint64_t d[kLookbackPerLane];
#pragma unroll
        for (int j = 0; j < kLookbackPerLane; ++j) {
            const int64_t idx = base - (j * 32 + lane);
            d[j] = idx >= 0 ? ld_relaxed(&desc[idx]) : kFlagPrefix;
        }
        // nearest inclusive prefix in the window (distance q = 32 j + lane)
        int qp = -1;
        bool zero_before = false;  // an unpublished descriptor at distance <= qp (or anywhere, if none)
#pragma unroll
        for (int j = 0; j < kLookbackPerLane; ++j) {
            const unsigned pm = __ballot_sync(0xffffffffu, (d[j] >> 62) == 2);
            const unsigned zm = __ballot_sync(0xffffffffu, (d[j] >> 62) == 0);
            if (qp < 0) {
                if (pm) {
                    const int l = __ffs(pm) - 1;
                    qp = j * 32 + l;
                    const unsigned upto = l == 31 ? 0xffffffffu : ((2u << l) - 1u);
                    zero_before |= (zm & upto) != 0;
                } else {
                    zero_before |= zm != 0;
                }
            }
        }
        if (!zero_before) {
            uint64_t v = 0;
#pragma unroll
            for (int j = 0; j < kLookbackPerLane; ++j) {
                const int q = j * 32 + lane;
                if (qp < 0 || q <= qp) v += d[j] & kValueMask;
            }
            excl += warp_sum_u64(v);
            if (qp >= 0) break;
            base -= 32 * kLookbackPerLane;
        } else {
            ++spins;
            const bool give_up = spins > kSpinLimit || ((spins & 255u) == 0 && error_recorded(status));
            if (__any_sync(0xffffffffu, give_up)) {
                if (lane == 0 && spins > kSpinLimit) set_status(status, HUFF_ERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
    }
    return excl;
}

// Pack N (code << 8 | len) entries starting at tile-local bit `start`.
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

__device__ __forceinline__ void put_word(uint32_t *payload, size_t cap_words, uint64_t gw, uint32_t v,
                                         int32_t *status) {
    if (gw < cap_words)
        payload[gw] = bswap32(v);
    else
        set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
}

template <bool BF16, bool XOR>
__device__ __forceinline__ void issue_tile(uint8_t *ring, uint64_t *full, int s, uint32_t t, const uint8_t *in,
                                           const uint8_t *in2, size_t n) {
    using C = EncCfg<BF16, XOR>;
    const size_t first = static_cast<size_t>(t) * C::kTileSyms;
    const size_t cnt = n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms);
    const uint32_t bytes = static_cast<uint32_t>(cnt * (BF16 ? 2 : 1)) & ~15u;
    mbar_arrive_expect_tx(&full[s], bytes * C::kInputs);
    if (bytes) {
        const size_t src = first * (BF16 ? 2 : 1);
        uint8_t *dst = ring + size_t(s) * C::kInputs * C::kTileBytes;
        bulk_g2s(dst, in + src, bytes, &full[s]);
        if (XOR) bulk_g2s(dst + C::kTileBytes, in2 + src, bytes, &full[s]);
    }
}

// State a consumer carries from a tile's packing to its write-out one iteration later.
struct Pending {
    uint32_t tile;
    uint32_t excl0, excl1;  // this thread's bit offset inside the tile, per plane
    uint32_t tot0, tot1;    // tile bit counts, per plane
    int nvalid;
};

template <bool BF16, bool XOR>
__device__ __forceinline__ void write_out(const Pending &pd, const uint32_t *bufs, const Misc *ms, int slot,
                                          const EncPlane &p0, const EncPlane &p1, size_t chunk, int tid,
                                          int32_t *status) {
    using C = EncCfg<BF16, XOR>;
#pragma unroll
    for (int p = 0; p < C::kPlanes; ++p) {
        const EncPlane &P = p == 0 ? p0 : p1;
        const uint32_t *buf = bufs + (slot * C::kPlanes + p) * C::kBufWords;
        const uint64_t pre = ms->prefix[slot][p];
        const uint32_t ph = static_cast<uint32_t>(pre & 31u);
        const uint64_t g0 = pre >> 5;
        const uint32_t tot = p == 0 ? pd.tot0 : pd.tot1;
        const uint32_t nfull = (ph + tot) >> 5;
        // whole words of this tile
        for (uint32_t i = (ph ? 1u : 0u) + tid; i < nfull; i += kConsumers)
            put_word(P.payload, P.cap_words, g0 + i, shifted_word(buf, i, ph), status);
        // chunk offsets
        const size_t g = static_cast<size_t>(pd.tile) * C::kTileSyms + size_t(tid) * C::kSyms;
        if (pd.nvalid > 0 && g % chunk == 0) P.off[g / chunk] = pre + (p == 0 ? pd.excl0 : pd.excl1);
        // boundary words for the fix-up kernel: this tile's bits in its first and last partial words
        if (tid == 32 * p) {
            const uint32_t head = ph ? shifted_word(buf, 0, ph) : 0u;
            const uint32_t tail = ((ph + tot) & 31u) ? shifted_word(buf, nfull, ph) : 0u;
            P.edge[pd.tile] = (static_cast<uint64_t>(head) << 32) | tail;
        }
    }
}

template <bool BF16, bool XOR>
__global__ void __launch_bounds__(kThreads) k_encode(const uint8_t *__restrict__ in, const uint8_t *__restrict__ in2,
                                                     size_t n, EncPlane p0, EncPlane p1, size_t chunk,
                                                     uint32_t n_tiles, int32_t *status) {
    using C = EncCfg<BF16, XOR>;
    extern __shared__ __align__(128) uint8_t smem[];
    Misc *ms = reinterpret_cast<Misc *>(smem);
    uint8_t *ring = smem + C::kMiscBytes;
    uint32_t *lut = reinterpret_cast<uint32_t *>(ring + C::kRingBytes);
    uint32_t *bufs = lut + C::kPlanes * C::kLutWords;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t G = gridDim.x;
    const uint32_t b = blockIdx.x;
    const uint32_t n_iter = b < n_tiles ? (n_tiles - 1 - b) / G + 1 : 0;

    // code table: entry (s * kLutRep + r) = (code << 8) | len, 0 when the symbol has no code
    if (tid == 0) ms->bad_codebook = 0;
    __syncthreads();
#pragma unroll
    for (int p = 0; p < C::kPlanes; ++p) {
        const huff_codebook *cb = p == 0 ? p0.cb : p1.cb;
        const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC;
        if (!ok && tid == 0) ms->bad_codebook = 1;
        for (int i = tid; i < C::kLutWords; i += kThreads) {
            const int s = i / kLutRep;
            const uint32_t L = ok ? cb->len[s] : 0u;
            lut[p * C::kLutWords + i] = (L >= 1 && L <= HUFF_MAX_LEN) ? ((cb->code[s] << 8) | L) : 0u;
        }
    }
    for (int i = tid; i < 2 * C::kPlanes * C::kBufWords; i += kThreads) bufs[i] = 0;
    if (tid == 0) {
        for (int s = 0; s < kEncStages; ++s) mbar_init(&ms->full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (ms->bad_codebook && tid == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);

    if (warp == kConsumers / 32) {
        // ------------------------------------------------ scheduler warp
        if (lane == 0)
            for (uint32_t i = 0; i < n_iter && i < uint32_t(kEncStages); ++i)
                issue_tile<BF16, XOR>(ring, ms->full, static_cast<int>(i), i * G + b, in, in2, n);
        for (uint32_t i = 0; i <= n_iter; ++i) {
            if (i >= 1) {
                const uint32_t t = (i - 1) * G + b;
                const int slot = (i - 1) & 1;
#pragma unroll
                for (int p = 0; p < C::kPlanes; ++p) {
                    uint64_t *desc = p == 0 ? p0.desc : p1.desc;
                    const uint64_t pre = lookback(desc, t, lane, status);
                    if (lane == 0) {
                        ms->prefix[slot][p] = pre;
                        if (t != 0) st_relaxed(&desc[t], kFlagPrefix | (pre + ms->total[slot][p]));
                    }
                }
            }
            bar_sync(kBarAll, kThreads);
            // stage i % kEncStages was consumed before this barrier: refill it
            if (lane == 0 && i + kEncStages < n_iter) {
                fence_proxy_async_smem();
                issue_tile<BF16, XOR>(ring, ms->full, static_cast<int>(i % kEncStages), (i + kEncStages) * G + b,
                                      in, in2, n);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    Pending prev{};
    for (uint32_t i = 0; i < n_iter; ++i) {
        const int s = static_cast<int>(i % kEncStages);
        const uint32_t t = i * G + b;
        if (!mbar_wait(&ms->full[s], (i / kEncStages) & 1u)) {
            if (tid == 0) set_status(status, HUFF_ERR_TIMEOUT);
        }
        const size_t first = static_cast<size_t>(t) * C::kTileSyms;
        const int tile_n = static_cast<int>(n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms));
        const uint8_t *stage = ring + size_t(s) * C::kInputs * C::kTileBytes;
        uint32_t wv[8];
        {
            const uint4 a = *reinterpret_cast<const uint4 *>(stage + tid * 32);
            const uint4 c = *reinterpret_cast<const uint4 *>(stage + tid * 32 + 16);
            wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
            wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
            if (XOR) {
                const uint4 d = *reinterpret_cast<const uint4 *>(stage + C::kTileBytes + tid * 32);
                const uint4 e = *reinterpret_cast<const uint4 *>(stage + C::kTileBytes + tid * 32 + 16);
                wv[0] ^= d.x; wv[1] ^= d.y; wv[2] ^= d.z; wv[3] ^= d.w;
                wv[4] ^= e.x; wv[5] ^= e.y; wv[6] ^= e.z; wv[7] ^= e.w;
            }
        }
        const int es = BF16 ? 2 : 1;
        const int tile_bytes = tile_n * es;
        const int tma_bytes = tile_bytes & ~15;
        if (tid * 32 + 32 > tma_bytes && tid * 32 < tile_bytes) {
            // ragged end of the last tile: bytes the bulk copy did not cover come from global memory
            for (int k = 0; k < 32; ++k) {
                const int bb = tid * 32 + k;
                if (bb < tma_bytes) continue;
                uint32_t v = 0;
                if (bb < tile_bytes) {
                    v = in[first * es + bb];
                    if (XOR) v ^= in2[first * es + bb];
                }
                wv[k >> 2] = (wv[k >> 2] & ~(0xffu << (8 * (k & 3)))) | (v << (8 * (k & 3)));
            }
        }

        // ---- code lookup
        const int nvalid = tile_n - tid * C::kSyms < 0
                               ? 0
                               : (tile_n - tid * C::kSyms > C::kSyms ? C::kSyms : tile_n - tid * C::kSyms);
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

        // ---- block scan of (bits_hi << 32 | bits_lo) over the consumers
        const uint64_t mine = BF16 ? ((uint64_t(bits0) << 32) | bits1) : uint64_t(bits0);
        uint64_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) ms->warp_sum[warp] = incl;
        bar_sync(kBarCons, kConsumers);
        uint64_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kConsumers / 32; ++w) {
            const uint64_t ws = ms->warp_sum[w];
            before += w < warp ? ws : 0;
            total += ws;
        }
        const uint64_t excl = before + incl - mine;
        const int slot = static_cast<int>(i & 1u);
        Pending cur;
        cur.tile = t;
        cur.excl0 = BF16 ? uint32_t(excl >> 32) : uint32_t(excl);
        cur.excl1 = uint32_t(excl);
        cur.tot0 = BF16 ? uint32_t(total >> 32) : uint32_t(total);
        cur.tot1 = uint32_t(total);
        cur.nvalid = nvalid;
        if (tid == 0) {
            // tile 0 knows its prefix (0); every other tile publishes its aggregate
            const uint64_t f = t == 0 ? kFlagPrefix : kFlagAggregate;
            st_relaxed(&p0.desc[t], f | cur.tot0);
            if (BF16) st_relaxed(&p1.desc[t], f | cur.tot1);
            ms->total[slot][0] = cur.tot0;
            ms->total[slot][1] = cur.tot1;
        }

        // ---- pack into slot i & 1
        pack_bits(bufs + (slot * C::kPlanes) * C::kBufWords, cur.excl0, e0);
        if (BF16) pack_bits(bufs + (slot * C::kPlanes + 1) * C::kBufWords, cur.excl1, e1);

        bar_sync(kBarAll, kThreads);  // prefix of tile i-1 resolved; this tile packed; stage s consumed
        if (i >= 1) {
            const int ps = static_cast<int>((i - 1) & 1u);
            write_out<BF16, XOR>(prev, bufs, ms, ps, p0, p1, chunk, tid, status);
            bar_sync(kBarCons, kConsumers);
#pragma unroll
            for (int p = 0; p < C::kPlanes; ++p) {
                uint32_t *buf = bufs + (ps * C::kPlanes + p) * C::kBufWords;
                const uint32_t used = ((p == 0 ? prev.tot0 : prev.tot1) + 31u) / 32u + 1u;
                for (uint32_t k = tid; k < used; k += kConsumers) buf[k] = 0;
            }
        }
        prev = cur;
    }
    bar_sync(kBarAll, kThreads);  // the last tile's prefix is resolved
    if (n_iter >= 1) write_out<BF16, XOR>(prev, bufs, ms, static_cast<int>((n_iter - 1) & 1u), p0, p1, chunk, tid,
                                          status);
}

// Boundary words: the word where tile t-1 ends and tile t begins holds bits of
// both; the stream's last, partial word holds the end of the last tile.
__global__ void k_encode_fixup(EncPlane p0, EncPlane p1, int planes, uint32_t n_tiles, size_t n_chunks,
                               int32_t *status) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_tiles) return;
    for (int p = 0; p < planes; ++p) {
        const EncPlane &P = p == 0 ? p0 : p1;
        const uint64_t start = t ? (P.desc[t - 1] & kValueMask) : 0;
        const uint64_t end = P.desc[t] & kValueMask;
        const uint64_t e = P.edge[t];
        const uint32_t ph = static_cast<uint32_t>(start & 31u);
        if (ph) {
            const uint32_t prev_tail = static_cast<uint32_t>(P.edge[t - 1]);
            put_word(P.payload, P.cap_words, start >> 5, prev_tail | static_cast<uint32_t>(e >> 32), status);
        }
        if (t + 1 == n_tiles) {
            const bool own_word = (end & 31u) && !(ph && (end >> 5) == (start >> 5));
            if (own_word) put_word(P.payload, P.cap_words, end >> 5, static_cast<uint32_t>(e), status);
            P.off[n_chunks] = end;
        }
    }
}

template <bool BF16, bool XOR>
int run_encode(const uint8_t *in, const uint8_t *in2, size_t n, EncPlane p0, EncPlane p1, size_t chunk,
               uint32_t n_tiles, int32_t *status, cudaStream_t s) {
    using C = EncCfg<BF16, XOR>;
    auto kern = k_encode<BF16, XOR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) !=
        cudaSuccess)
        return HUFF_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, C::kSmem) != cudaSuccess)
        return HUFF_ERR_CUDA;
    if (per_sm < 1) return HUFF_ERR_CUDA;
    const DevInfo d = dev_info();
    size_t grid = static_cast<size_t>(d.sms) * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    size_t chunk_arg = chunk;
    void *args[] = {(void *)&in, (void *)&in2, (void *)&n, (void *)&p0, (void *)&p1, (void *)&chunk_arg,
                    (void *)&n_tiles, (void *)&status};
    // cooperative launch: every CTA is resident at once, so the round-robin lookback always makes progress
    if (cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(static_cast<unsigned>(grid)),
                                    dim3(kThreads), args, C::kSmem, s) != cudaSuccess)
        return HUFF_ERR_CUDA;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    k_encode_fixup<<<(n_tiles + 255) / 256, 256, 0, s>>>(p0, p1, C::kPlanes, n_tiles, n_chunks, status);
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
    int st = launch_zero_u64(w, tiles, s);  // descriptors only; edge words are always written
    if (st != HUFF_OK) return st;
    EncPlane p0{cb, reinterpret_cast<uint32_t *>(payload), cap / 4, off, w, w + tiles};
    EncPlane p1 = p0;
    return run_encode<false, false>(in, nullptr, n, p0, p1, chunk, static_cast<uint32_t>(tiles), status, s);
}

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (host code only sees a host-side stand-in under the array's name).
static uint64_t *noalloc_scratch_address() {
    static std::mutex mu;
    static uint64_t *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<uint64_t *>(p);
    }
    return addr[dev];
}

int launch_encode_u8_noalloc(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk, uint8_t *payload,
                             size_t cap, uint64_t *off, int32_t *status, cudaStream_t s) {
    if (2 * enc_u8_tiles(n) > kNoAllocScratchWords) return HUFF_ERR_BUFFER_TOO_SMALL;
    uint64_t *ws = noalloc_scratch_address();
    if (ws == nullptr) return HUFF_ERR_CUDA;
    // the same path as huff_encode; it zeroes the descriptors it needs before the encode kernel runs
    return launch_encode_u8(in, n, cb, chunk, payload, cap, off, ws, status, s);
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
    // layout: desc_hi, desc_lo (zeroed), edge_hi, edge_lo
    int st = launch_zero_u64(w, 2 * tiles, s);
    if (st != HUFF_OK) return st;
    EncPlane p0{cb_hi, reinterpret_cast<uint32_t *>(pay_hi), cap_hi / 4, off_hi, w, w + 2 * tiles};
    EncPlane p1{cb_lo, reinterpret_cast<uint32_t *>(pay_lo), cap_lo / 4, off_lo, w + tiles, w + 3 * tiles};
    const uint8_t *a = reinterpret_cast<const uint8_t *>(w16);
    if (x0 != nullptr)
        return run_encode<true, true>(a, reinterpret_cast<const uint8_t *>(x0), n, p0, p1, chunk,
                                      static_cast<uint32_t>(tiles), status, s);
    return run_encode<true, false>(a, nullptr, n, p0, p1, chunk, static_cast<uint32_t>(tiles), status, s);
}

}  // namespace huffk
