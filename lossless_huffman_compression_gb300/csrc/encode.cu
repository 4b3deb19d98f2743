// encode.cu -- chunked Huffman encode.
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
// GPU design (two passes over each segment, the second from L2):
//   * the input is cut into 8 KiB tiles and segments of kSegTiles tiles;
//     persistent CTAs take segments from an atomic counter;
//   * pass 1 streams a segment's tiles from HBM into a shared-memory ring with
//     1-D bulk copies (cp.async.bulk on mbarriers, L2 policy evict_last), looks
//     up each symbol's code length and keeps every thread's bit count;
//   * the CTA publishes the segment's bit count, claims its next segment, and
//     one warp resolves the segment's global bit offset with a decoupled
//     lookback (Merrill & Garland, "Single-pass Parallel Prefix Scan with
//     Decoupled Look-back", 2016) over windows of 320 segment descriptors;
//     one lookback per segment, so its latency is amortised over 8 tiles;
//   * pass 2 streams the same tiles again (now from L2, evict_first), looks
//     up (code << 8 | len) in a shared-memory table replicated kLutRep times
//     (lanes with different symbols spread over more banks), scans the stored
//     per-thread counts, packs the codes into a tile-local bit buffer with
//     32-bit funnel shifts (each thread's symbols as two independent halves
//     per plane, so two to four packing chains interleave), and writes whole
//     32-bit words shifted to the tile's bit phase
//     with coalesced stores; the CTA carries each tile's last partial word
//     into the next tile of the segment itself;
//   * the two partial words at each segment boundary are left in the
//     workspace and written by a small fix-up kernel, so no CTA ever waits for
//     another CTA's output.
//   The fused bf16 variant reads 16-bit words (and optionally x0, for the XOR
//   delta) and encodes the high and low byte planes as two streams in one
//   pass.  All waits are bounded; a wait that runs out sets HUFF_ERR_TIMEOUT
//   and the kernel carries on to completion.
#include <mutex>

#include "common.cuh"

namespace huffk {

// Workspace for huff_encode_noalloc, sized like huff_workspace_size for
// HUFF_NOALLOC_MAX_SYMBOLS symbols.  Every GPU that loads the library keeps
// these 2 MiB until the process exits; all calls share them.
constexpr size_t kNoAllocScratchWords = 2 * (HUFF_NOALLOC_MAX_SYMBOLS / kEncU8Tile) + 2;
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocScratchWords];

namespace {

constexpr int kThreads = kEncThreads;  // 8 warps
constexpr int kSegTiles = 8;           // tiles per segment
constexpr int kStages = 3;             // bulk-copy ring depth
constexpr int kLookbackPerLane = 10;   // descriptors per lane per lookback step (window 320)

struct EncPlane {
    const huff_codebook *cb;
    uint32_t *payload;  // 32-bit words; payload byte 4w + j = bits 31-8j .. 24-8j of word w
    size_t cap_words;
    uint64_t *off;
    uint64_t *desc;     // per-segment lookback descriptors (zeroed before the launch)
    uint64_t *edge;     // per-segment boundary words: head bits << 32 | tail bits
};

template <bool BF16, bool XOR>
struct EncCfg {
    static constexpr int kPlanes = BF16 ? 2 : 1;
    static constexpr int kSyms = BF16 ? kEncBf16ElemsPerThread : kEncU8SymsPerThread;  // per plane, per thread
    static constexpr int kTileSyms = kThreads * kSyms;
    static constexpr int kTileBytes = 8192;  // per input array
    static constexpr int kInputs = XOR ? 2 : 1;
    static constexpr int kBufWords = kTileSyms * HUFF_MAX_LEN / 32 + 4;
    static constexpr int kLutWords = 256 * kLutRep;
    static constexpr size_t kMiscBytes = 512;
    static constexpr size_t kRingBytes = size_t(kStages) * kInputs * kTileBytes;
    static constexpr size_t kLutBytes = size_t(kPlanes) * kLutWords * 4;
    static constexpr size_t kBufBytes = size_t(kPlanes) * kBufWords * 4;
    static constexpr size_t kCntBytes = size_t(kSegTiles) * kThreads * 4;
    static constexpr size_t kSmem = kMiscBytes + kRingBytes + kLutBytes + kBufBytes + kCntBytes;
    static_assert(kTileSyms * (BF16 ? 2 : 1) == kTileBytes && kTileSyms <= 8192, "tile geometry");
};

struct Misc {
    uint64_t full[kStages];
    uint64_t warp_sum[kThreads / 32];
    uint64_t prefix[2];      // [plane] segment bit counts, handed to the lookback warp
    uint64_t run[2];         // [plane] bit offset of the current tile
    uint32_t carry[2];       // [plane] bits of the previous tile in the word the current tile starts in
    uint32_t seg_head[2];    // [plane] the segment's bits in its first, partial word
    uint32_t segq[2];        // segment of round r at [r & 1]
    int32_t bad_codebook;
    uint64_t chunk_q;        // the current tile's first element is element chunk_r of chunk chunk_q
    uint32_t chunk_r;
};
static_assert(sizeof(Misc) <= 512, "misc area");

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void load_window(const uint64_t *desc, int64_t base, int lane,
                                            uint64_t (&d)[kLookbackPerLane]) {
#pragma unroll
    for (int j = 0; j < kLookbackPerLane; ++j) {
        const int64_t idx = base - (j * 32 + lane);
        d[j] = idx >= 0 ? ld_relaxed(&desc[idx]) : kFlagPrefix;
    }
}

// Decoupled lookback for segment t of one stream, by one full warp, over
// windows of 32 * kLookbackPerLane predecessors; returns the exclusive bit
// offset.  The segment's own aggregate is already published.  d holds the
// first window, already loaded (two streams' first windows fly together).
__device__ uint64_t lookback(const uint64_t *desc, uint32_t t, int lane, int32_t *status,
                             uint64_t (&d)[kLookbackPerLane]) {
    if (t == 0) return 0;
    uint64_t excl = 0;
    int64_t base = static_cast<int64_t>(t) - 1;
    unsigned spins = 0;
    for (bool first = true;; first = false) {
        if (!first) load_window(desc, base, lane, d);
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
            __nanosleep(64);
        }
    }
    return excl;
}

// Packs (code << 8 | len) entries, len <= 24 in the low 5 bits, into a
// tile-local bit buffer from bit `start` on.  The pending bits sit in the
// 64-bit pair (hi, lo); since len < 32, 32-bit funnel shifts move them, and
// the entry itself serves as the shift count (funnel shifts use its low 5
// bits).  A word wholly inside this thread's bits is stored under a
// predicate (no branch, no atomic); the first word, which may hold bits of
// earlier threads, is kept in a register and OR-ed in by finish() together
// with the last, partial word (the buffer is zero before packing).
struct Packer {
    uint32_t *buf;
    uint32_t hi, lo;  // pending bits: the low `nb` bits of hi:lo
    uint32_t nb;
    uint32_t w;       // next buffer word
    uint32_t w0;      // the first word
    uint32_t head;    // the first word's bits, once complete
    bool first;       // the first word is not complete yet

    __device__ __forceinline__ void begin(uint32_t *b, uint32_t start) {
        buf = b;
        hi = lo = 0;
        nb = start & 31u;
        w = w0 = start >> 5;
        head = 0;
        first = true;
    }
    __device__ __forceinline__ void push(uint32_t e) {
        hi = __funnelshift_l(lo, hi, e);
        lo = __funnelshift_l(0u, lo, e) | (e >> 8);
        nb += e & 31u;
        const bool full = nb >= 32;
        nb -= full ? 32u : 0u;
        const uint32_t word = __funnelshift_r(lo, hi, nb);
        if (full && !first) buf[w] = word;
        head = (full && first) ? word : head;
        first = first && !full;
        w += full ? 1u : 0u;
    }
    // Two codes at once when together they are at most 31 bits.
    __device__ __forceinline__ void push2(uint32_t ea, uint32_t eb, uint32_t L) {  // L = both lengths
        const uint32_t code = ((ea >> 8) << (eb & 31u)) | (eb >> 8);
        hi = __funnelshift_l(lo, hi, L);
        lo = (lo << L) | code;
        nb += L;
        const bool full = nb >= 32;
        nb -= full ? 32u : 0u;
        const uint32_t word = __funnelshift_r(lo, hi, nb);
        if (full && !first) buf[w] = word;
        head = (full && first) ? word : head;
        first = first && !full;
        w += full ? 1u : 0u;
    }
    __device__ __forceinline__ void finish() {
        if (!first) atomicOr(&buf[w0], head);
        if (nb > 0) atomicOr(&buf[w], lo << (32 - nb));
    }
};

// Chunk starts among a tile's per-thread groups.  Chunks are multiples of 256
// elements and a thread's group is 16 or 32, so a group starts a chunk or lies
// inside one.  With the tile's position in its chunk (q, r) kept by thread 0,
// a thread's distance d = r + first-of-group < chunk + 8192 (a tile is at
// most 8192 symbols) is divided exactly by a multiply-high when chunk < 8192
// (magic = ceil(2^32 / chunk); exact since d * chunk < 2^32) or by one
// compare when chunk >= 8192 (then d < 2 chunk).
struct ChunkDiv {
    uint32_t chunk;  // < 2^31
    uint32_t magic;  // 0 when chunk >= 8192
    __device__ __forceinline__ uint32_t div(uint32_t d) const {
        return magic ? __umulhi(d, magic) : (d >= chunk ? 1u : 0u);
    }
};

__host__ inline ChunkDiv make_chunk_div(size_t chunk) {
    const uint32_t c = static_cast<uint32_t>(chunk);
    return ChunkDiv{c, c < 8192 ? static_cast<uint32_t>(((1ull << 32) + c - 1) / c) : 0u};
}

// Thread 0, before a tile: its first element's chunk and offset in it
// (incrementally from the previous tile of the same segment).
__device__ __forceinline__ void chunk_position(Misc *ms, const ChunkDiv &cd, size_t first, bool seg_start,
                                               uint32_t tile_syms) {
    if (seg_start) {
        ms->chunk_q = first / cd.chunk;
        ms->chunk_r = static_cast<uint32_t>(first % cd.chunk);
    } else {
        const uint32_t d = ms->chunk_r + tile_syms;
        const uint32_t k = cd.div(d);
        ms->chunk_q += k;
        ms->chunk_r = d - k * cd.chunk;
    }
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

// Job q of a CTA: round r = q / (2 kSegTiles) works on segment segq[r & 1];
// its first kSegTiles jobs are pass 1, the next kSegTiles pass 2.
template <bool BF16, bool XOR>
__device__ __forceinline__ void issue_job(uint8_t *ring, Misc *ms, uint32_t q, uint32_t n_seg, uint32_t n_tiles,
                                          const uint8_t *in, const uint8_t *in2, size_t n) {
    using C = EncCfg<BF16, XOR>;
    const uint32_t r = q / (2 * kSegTiles);
    const uint32_t w = q % (2 * kSegTiles);
    const uint32_t seg = ms->segq[r & 1];
    if (seg >= n_seg) return;  // the consumers stop before this job
    const int s = static_cast<int>(q % kStages);
    const uint32_t t = seg * kSegTiles + (w % kSegTiles);
    uint32_t bytes = 0;
    size_t first = 0;
    if (t < n_tiles) {
        first = static_cast<size_t>(t) * C::kTileSyms;
        const size_t cnt = n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms);
        bytes = static_cast<uint32_t>(cnt * (BF16 ? 2 : 1)) & ~15u;
    }
    mbar_arrive_expect_tx(&ms->full[s], bytes * C::kInputs);
    if (bytes) {
        const uint64_t pol = w < kSegTiles ? l2_policy_evict_last() : l2_policy_evict_first();
        const size_t src = first * (BF16 ? 2 : 1);
        uint8_t *dst = ring + size_t(s) * C::kInputs * C::kTileBytes;
        bulk_g2s_hint(dst, in + src, bytes, &ms->full[s], pol);
        if (XOR) bulk_g2s_hint(dst + C::kTileBytes, in2 + src, bytes, &ms->full[s], pol);
    }
}

// This thread's 32 input bytes (16-bit words XOR x0 for the fused delta) of the tile in a stage.
template <bool BF16, bool XOR>
__device__ __forceinline__ void read_tile(const uint8_t *stage, int tid, size_t first, int tile_n,
                                          const uint8_t *in, const uint8_t *in2, uint32_t (&wv)[8]) {
    using C = EncCfg<BF16, XOR>;
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
}

// (code << 8 | len) of this thread's symbols; symbols past the tile's end get 0.
// mn ends at 0 when a valid symbol has no code.
template <bool BF16, bool XOR, bool COUNT>
__device__ __forceinline__ void lookup(const uint32_t *lut_r, const uint32_t (&wv)[8], bool full, int nvalid,
                                       uint32_t (&e0)[EncCfg<BF16, XOR>::kSyms],
                                       uint32_t (&e1)[BF16 ? EncCfg<BF16, XOR>::kSyms : 1], uint32_t &bits0,
                                       uint32_t &bits1, uint32_t &mn) {
    using C = EncCfg<BF16, XOR>;
    bits0 = bits1 = 0;
    mn = 0xffffffffu;
    if (full) {
#pragma unroll
        for (int k = 0; k < C::kSyms; ++k) {
            if (BF16) {
                const uint32_t w2 = wv[k >> 1];
                const uint32_t hi = lut_r[__byte_perm(w2, 0, 0x4441 + 2 * (k & 1)) * kLutRep];
                const uint32_t lo = lut_r[C::kLutWords + __byte_perm(w2, 0, 0x4440 + 2 * (k & 1)) * kLutRep];
                mn = min(mn, min(hi, lo));
                e0[k] = hi;
                e1[BF16 ? k : 0] = lo;
                if (COUNT) {
                    bits0 += hi & 31u;
                    bits1 += lo & 31u;
                }
            } else {
                const uint32_t v = lut_r[__byte_perm(wv[k >> 2], 0, 0x4440 + (k & 3)) * kLutRep];
                mn = min(mn, v);
                e0[k] = v;
                if (COUNT) bits0 += v & 31u;
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < C::kSyms; ++k) {
            if (BF16) {
                const uint32_t v = (wv[k >> 1] >> (16 * (k & 1))) & 0xffffu;
                uint32_t hi = lut_r[(v >> 8) * kLutRep];
                uint32_t lo = lut_r[C::kLutWords + (v & 0xffu) * kLutRep];
                if (k >= nvalid) hi = lo = 0;
                else mn = min(mn, min(hi, lo));
                e0[k] = hi;
                e1[BF16 ? k : 0] = lo;
                if (COUNT) {
                    bits0 += hi & 31u;
                    bits1 += lo & 31u;
                }
            } else {
                const uint32_t sym = (wv[k >> 2] >> (8 * (k & 3))) & 0xffu;
                uint32_t v = lut_r[sym * kLutRep];
                if (k >= nvalid) v = 0;
                else mn = min(mn, v);
                e0[k] = v;
                if (COUNT) bits0 += v & 31u;
            }
        }
    }
}

template <bool BF16, bool XOR>
__global__ void __launch_bounds__(kThreads, 2) k_encode(const uint8_t *__restrict__ in, const uint8_t *__restrict__ in2,
                                                     size_t n, EncPlane p0, EncPlane p1, ChunkDiv cdiv,
                                                     uint32_t n_tiles, unsigned *seg_ctr, int32_t *status) {
    using C = EncCfg<BF16, XOR>;
    extern __shared__ __align__(128) uint8_t smem[];
    Misc *ms = reinterpret_cast<Misc *>(smem);
    uint8_t *ring = smem + C::kMiscBytes;
    uint32_t *lut = reinterpret_cast<uint32_t *>(ring + C::kRingBytes);
    uint32_t *bufs = lut + C::kPlanes * C::kLutWords;
    uint32_t *cnt = bufs + C::kPlanes * C::kBufWords;  // [kSegTiles][kThreads] hi << 16 | lo

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t n_seg = (n_tiles + kSegTiles - 1) / kSegTiles;

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
    for (int i = tid; i < C::kPlanes * C::kBufWords; i += kThreads) bufs[i] = 0;
    uint32_t issued = 0;  // next job to issue (thread 0 only)
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&ms->full[s], 1);
        fence_mbar_init();
        ms->segq[0] = atomicAdd(seg_ctr, 1u);
        ms->segq[1] = 0xffffffffu;
        for (; issued < uint32_t(kStages); ++issued) issue_job<BF16, XOR>(ring, ms, issued, n_seg, n_tiles, in, in2, n);
    }
    __syncthreads();
    if (ms->bad_codebook && tid == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
    const uint32_t *lut_r = lut + (lane & (kLutRep - 1));

    for (uint32_t r = 0;; ++r) {
        const uint32_t seg = ms->segq[r & 1];
        if (seg >= n_seg) break;
        const uint32_t t_first = seg * kSegTiles;
        const int seg_tiles = static_cast<int>(n_tiles - t_first < uint32_t(kSegTiles) ? n_tiles - t_first : kSegTiles);
        const uint32_t q0 = r * 2 * kSegTiles;

        // ---------------- pass 1: bit counts per thread and per tile
        uint32_t sum0 = 0, sum1 = 0, mn_all = 0xffffffffu;
        for (int k = 0; k < kSegTiles; ++k) {
            const uint32_t q = q0 + k;
            const int s = static_cast<int>(q % kStages);
            if (!mbar_wait(&ms->full[s], (q / kStages) & 1u) && tid == 0) set_status(status, HUFF_ERR_TIMEOUT);
            if (k < seg_tiles) {
                const uint32_t t = t_first + k;
                const size_t first = static_cast<size_t>(t) * C::kTileSyms;
                const int tile_n = static_cast<int>(n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms));
                uint32_t wv[8];
                read_tile<BF16, XOR>(ring + size_t(s) * C::kInputs * C::kTileBytes, tid, first, tile_n, in, in2, wv);
                const int nvalid = tile_n - tid * C::kSyms < 0
                                       ? 0
                                       : (tile_n - tid * C::kSyms > C::kSyms ? C::kSyms : tile_n - tid * C::kSyms);
                uint32_t e0[C::kSyms], e1[BF16 ? C::kSyms : 1], b0, b1, mn;
                lookup<BF16, XOR, true>(lut_r, wv, tile_n == C::kTileSyms, nvalid, e0, e1, b0, b1, mn);
                if (nvalid > 0) mn_all = min(mn_all, mn);
                cnt[k * kThreads + tid] = (b0 << 16) | b1;
                sum0 += b0;
                sum1 += b1;
            }
            __syncthreads();  // stage s consumed
            if (tid == 0) issue_job<BF16, XOR>(ring, ms, issued++, n_seg, n_tiles, in, in2, n);
        }
        if (mn_all == 0) set_status(status, HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK);

        // ---------------- segment bit count, publish, claim the next segment
        const uint64_t v = warp_sum_u64((static_cast<uint64_t>(sum0) << 32) | sum1);
        if (lane == 0) ms->warp_sum[warp] = v;
        __syncthreads();
        if (tid == 0) {
            uint64_t tot = 0;
            for (int w = 0; w < kThreads / 32; ++w) tot += ms->warp_sum[w];
            const uint64_t tot0 = tot >> 32;
            const uint64_t tot1 = tot & 0xffffffffull;
            const uint64_t f = seg == 0 ? kFlagPrefix : kFlagAggregate;
            st_relaxed(&p0.desc[seg], f | tot0);
            if (BF16) st_relaxed(&p1.desc[seg], f | tot1);
            ms->segq[(r + 1) & 1] = atomicAdd(seg_ctr, 1u);
            ms->prefix[0] = tot0;  // the totals, handed to warp 0
            ms->prefix[1] = tot1;
        }
        __syncthreads();
        if (warp == 0) {
            const uint64_t tot0 = ms->prefix[0], tot1 = ms->prefix[1];
            uint64_t w0[kLookbackPerLane], w1[kLookbackPerLane];
            load_window(p0.desc, static_cast<int64_t>(seg) - 1, lane, w0);
            if (BF16) load_window(p1.desc, static_cast<int64_t>(seg) - 1, lane, w1);
            const uint64_t pre0 = lookback(p0.desc, seg, lane, status, w0);
            const uint64_t pre1 = BF16 ? lookback(p1.desc, seg, lane, status, w1) : 0;
            if (lane == 0) {
                if (seg != 0) {
                    st_relaxed(&p0.desc[seg], kFlagPrefix | (pre0 + tot0));
                    if (BF16) st_relaxed(&p1.desc[seg], kFlagPrefix | (pre1 + tot1));
                }
                ms->run[0] = pre0;
                ms->run[1] = pre1;
                ms->carry[0] = ms->carry[1] = 0;
                ms->seg_head[0] = ms->seg_head[1] = 0;
            }
        }
        __syncthreads();

        // ---------------- pass 2: pack and write, tile after tile
        for (int k = 0; k < kSegTiles; ++k) {
            const uint32_t q = q0 + kSegTiles + k;
            const int s = static_cast<int>(q % kStages);
            if (!mbar_wait(&ms->full[s], (q / kStages) & 1u) && tid == 0) set_status(status, HUFF_ERR_TIMEOUT);
            if (k < seg_tiles) {
                const uint32_t t = t_first + k;
                const size_t first = static_cast<size_t>(t) * C::kTileSyms;
                const int tile_n = static_cast<int>(n - first < size_t(C::kTileSyms) ? n - first : size_t(C::kTileSyms));
                uint32_t wv[8];
                read_tile<BF16, XOR>(ring + size_t(s) * C::kInputs * C::kTileBytes, tid, first, tile_n, in, in2, wv);
                const int nvalid = tile_n - tid * C::kSyms < 0
                                       ? 0
                                       : (tile_n - tid * C::kSyms > C::kSyms ? C::kSyms : tile_n - tid * C::kSyms);
                uint32_t e0[C::kSyms], e1[BF16 ? C::kSyms : 1], b0, b1, mn;
                lookup<BF16, XOR, false>(lut_r, wv, tile_n == C::kTileSyms, nvalid, e0, e1, b0, b1, mn);
                // each pair's total length, once: the bit counts, the pair check and the packing use it
                uint32_t L0[C::kSyms / 2], L1[BF16 ? C::kSyms / 2 : 1], longest_pair = 0;
#pragma unroll
                for (int j = 0; j < C::kSyms / 2; ++j) {
                    L0[j] = (e0[2 * j] & 31u) + (e0[2 * j + 1] & 31u);
                    b0 += L0[j];
                    longest_pair = max(longest_pair, L0[j]);
                    if (BF16) {
                        L1[BF16 ? j : 0] = (e1[BF16 ? 2 * j : 0] & 31u) + (e1[BF16 ? 2 * j + 1 : 0] & 31u);
                        b1 += L1[BF16 ? j : 0];
                        longest_pair = max(longest_pair, L1[BF16 ? j : 0]);
                    }
                }
                // block scan of the counts kept from pass 1
                const uint32_t c = cnt[k * kThreads + tid];
                const uint64_t mine = (static_cast<uint64_t>(c >> 16) << 32) | (c & 0xffffu);
                uint64_t incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (lane == 31) ms->warp_sum[warp] = incl;
                if (tid == 0) chunk_position(ms, cdiv, first, k == 0, C::kTileSyms);
                __syncthreads();  // stage s consumed; warp sums ready
                if (tid == 0) issue_job<BF16, XOR>(ring, ms, issued++, n_seg, n_tiles, in, in2, n);
                uint64_t before = 0, total = 0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) {
                    const uint64_t ws = ms->warp_sum[w];
                    before += w < warp ? ws : 0;
                    total += ws;
                }
                const uint64_t excl = before + incl - mine;
                const uint32_t excl0 = uint32_t(excl >> 32);
                const uint32_t excl1 = uint32_t(excl);
                const uint32_t tot0 = uint32_t(total >> 32);
                const uint32_t tot1 = uint32_t(total);
                Packer pk0, pk1;
                pk0.begin(bufs, excl0);
                if (BF16) pk1.begin(bufs + C::kBufWords, excl1);
                // pairs of codes at most 31 bits long go in one step; a warp with a longer pair
                // anywhere packs its codes one by one
                if (__any_sync(0xffffffffu, longest_pair > 31u)) {
#pragma unroll
                    for (int j = 0; j < C::kSyms; ++j) {
                        pk0.push(e0[j]);
                        if (BF16) pk1.push(e1[BF16 ? j : 0]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C::kSyms; j += 2) {
                        pk0.push2(e0[j], e0[j + 1], L0[j / 2]);
                        if (BF16) pk1.push2(e1[BF16 ? j : 0], e1[BF16 ? j + 1 : 0], L1[BF16 ? j / 2 : 0]);
                    }
                }
                pk0.finish();
                if (BF16) pk1.finish();
                __syncthreads();  // buffers packed
                // write the tile's words at its global bit offset
                uint64_t next_run = 0;  // thread 32 p: plane p's offset after this tile
#pragma unroll
                for (int p = 0; p < C::kPlanes; ++p) {
                    const EncPlane &P = p == 0 ? p0 : p1;
                    const uint32_t *buf = bufs + p * C::kBufWords;
                    const uint64_t pre = ms->run[p];
                    const uint32_t ph = static_cast<uint32_t>(pre & 31u);
                    const uint64_t g0 = pre >> 5;
                    const uint32_t tot = p == 0 ? tot0 : tot1;
                    const uint32_t nfull = (ph + tot) >> 5;
                    for (uint32_t i = (ph ? 1u : 0u) + tid; i < nfull; i += kThreads)
                        put_word(P.payload, P.cap_words, g0 + i, shifted_word(buf, i, ph), status);
                    const size_t g = first + size_t(tid) * C::kSyms;
                    if (nvalid > 0) {
                        const uint32_t d = ms->chunk_r + static_cast<uint32_t>(tid) * C::kSyms;
                        const uint32_t kq = cdiv.div(d);
                        if (kq * cdiv.chunk == d) P.off[ms->chunk_q + kq] = pre + (p == 0 ? excl0 : excl1);
                    }
                    if (tid == 32 * p) {
                        // the word this tile starts in, and the one it ends in
                        const uint32_t head = ph ? shifted_word(buf, 0, ph) : 0u;
                        uint32_t combined = head;
                        if (ph) {
                            if (k == 0) {
                                ms->seg_head[p] = head;  // the segment's first word: the fix-up kernel's
                            } else {
                                combined |= ms->carry[p];
                                if (nfull >= 1) put_word(P.payload, P.cap_words, g0, combined, status);
                            }
                        }
                        uint32_t tail = 0;
                        if ((ph + tot) & 31u) tail = nfull == 0 ? (ph ? combined : buf[0]) : shifted_word(buf, nfull, ph);
                        ms->carry[p] = tail;  // read only by this thread
                        next_run = pre + tot;
                        if (k == seg_tiles - 1)
                            P.edge[seg] = (static_cast<uint64_t>(ms->seg_head[p]) << 32) | tail;
                    }
                }
                __syncthreads();  // everyone has read the buffers and the running offsets
                if (tid == 0) ms->run[0] = next_run;
                if (BF16 && tid == 32) ms->run[1] = next_run;
#pragma unroll
                for (int p = 0; p < C::kPlanes; ++p) {
                    uint32_t *buf = bufs + p * C::kBufWords;
                    const uint32_t used = ((p == 0 ? tot0 : tot1) + 31u) / 32u + 1u;
                    for (uint32_t i = tid; i < used; i += kThreads) buf[i] = 0;
                }
            } else {
                __syncthreads();  // stage s consumed (an empty job)
                if (tid == 0) issue_job<BF16, XOR>(ring, ms, issued++, n_seg, n_tiles, in, in2, n);
            }
        }
    }
}

// ------------------------------------------------------------------ counted path (bf16, per shard)
//
// When the histogram pass has recorded each plane's counts per segment of
// kDirSegTiles tiles, every segment's bit count is sum(count * length): a
// scan gives each segment's offset before the encode starts.  The encode then
// reads its input once (no counting pass) and no CTA waits for another.

// Bits of each segment per plane (sum of count x length over its recorded
// counts, a warp per segment, one wave of CTAs) and their inclusive prefix.  The last CTA to
// finish its segments (a ticket counter) scans all segments' bits: thread t
// of its 1024 sums a run of consecutive segments, a block scan combines the
// runs, and each thread writes its run's prefixes as the descriptors.
constexpr int kSegScanThreads = 1024;

__global__ void __launch_bounds__(kSegScanThreads) k_seg_bits_scan(const uint32_t *__restrict__ seg_counts,
                                                                   uint32_t n_seg, const huff_codebook *cb_hi,
                                                                   const huff_codebook *cb_lo, uint32_t *bits,
                                                                   uint64_t *desc_hi, uint64_t *desc_lo,
                                                                   unsigned *done, int32_t *status) {
    __shared__ uint8_t len[kSegCountWords];
    __shared__ uint64_t wsum[2][kSegScanThreads / 32];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kSegCountWords; i += blockDim.x) {
        const huff_codebook *cb = i < 256 ? cb_hi : cb_lo;
        len[i] = cb->magic == HUFF_CODEBOOK_MAGIC ? cb->len[i & 255] : 0;
    }
    __syncthreads();
    for (uint32_t seg = blockIdx.x * (kSegScanThreads / 32) + warp; seg < n_seg;
         seg += gridDim.x * (kSegScanThreads / 32)) {
        const uint32_t *h = seg_counts + static_cast<size_t>(seg) * kSegCountWords;
        uint64_t b0 = 0, b1 = 0;
        bool missing = false;
#pragma unroll
        for (int j = lane; j < 256; j += 32) {
            const uint32_t c0 = h[j], c1 = h[256 + j];
            const uint32_t l0 = len[j], l1 = len[256 + j];
            b0 += static_cast<uint64_t>(c0) * l0;
            b1 += static_cast<uint64_t>(c1) * l1;
            missing |= (c0 && !l0) || (c1 && !l1);
        }
        b0 = warp_sum_u64(b0);
        b1 = warp_sum_u64(b1);
        if (__any_sync(0xffffffffu, missing) && lane == 0) set_status(status, HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK);
        if (lane == 0) {  // a segment has at most 131 072 * 24 bits per plane: 32-bit counts
            bits[seg] = static_cast<uint32_t>(b0);
            bits[n_seg + seg] = static_cast<uint32_t>(b1);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // the last CTA: thread tid sums segments [lo, hi) of both planes (up to kRun of them held in
    // registers, their loads all in flight at once; longer runs are read twice)
    constexpr uint32_t kRun = 16;
    const uint32_t K = (n_seg + kSegScanThreads - 1) / kSegScanThreads;
    const uint32_t lo = tid * K < n_seg ? tid * K : n_seg;
    const uint32_t hi = lo + K < n_seg ? lo + K : n_seg;
    uint32_t v0[kRun], v1[kRun];
    uint64_t s0 = 0, s1 = 0;
    if (K <= kRun) {
#pragma unroll
        for (uint32_t j = 0; j < kRun; ++j) {
            const bool in = lo + j < hi;
            v0[j] = in ? __ldcg(&bits[lo + j]) : 0u;
            v1[j] = in ? __ldcg(&bits[n_seg + lo + j]) : 0u;
        }
#pragma unroll
        for (uint32_t j = 0; j < kRun; ++j) {
            s0 += v0[j];
            s1 += v1[j];
        }
    } else {
        for (uint32_t i = lo; i < hi; ++i) {
            s0 += __ldcg(&bits[i]);
            s1 += __ldcg(&bits[n_seg + i]);
        }
    }
    uint64_t i0 = s0, i1 = s1;  // inclusive scan across the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y0 = __shfl_up_sync(0xffffffffu, i0, o);
        const uint64_t y1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
            i0 += y0;
            i1 += y1;
        }
    }
    if (lane == 31) {
        wsum[0][warp] = i0;
        wsum[1][warp] = i1;
    }
    __syncthreads();
    if (warp == 0) {
        uint64_t u0 = wsum[0][lane], u1 = wsum[1][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y0 = __shfl_up_sync(0xffffffffu, u0, o);
            const uint64_t y1 = __shfl_up_sync(0xffffffffu, u1, o);
            if (lane >= o) {
                u0 += y0;
                u1 += y1;
            }
        }
        wsum[0][lane] = u0;
        wsum[1][lane] = u1;
    }
    __syncthreads();
    uint64_t r0 = i0 - s0 + (warp ? wsum[0][warp - 1] : 0);  // exclusive prefix of this run
    uint64_t r1 = i1 - s1 + (warp ? wsum[1][warp - 1] : 0);
    if (K <= kRun) {
#pragma unroll
        for (uint32_t j = 0; j < kRun; ++j) {
            if (lo + j < hi) {
                r0 += v0[j];
                r1 += v1[j];
                desc_hi[lo + j] = kFlagPrefix | r0;
                desc_lo[lo + j] = kFlagPrefix | r1;
            }
        }
    } else {
        for (uint32_t i = lo; i < hi; ++i) {
            r0 += __ldcg(&bits[i]);
            r1 += __ldcg(&bits[n_seg + i]);
            desc_hi[i] = kFlagPrefix | r0;
            desc_lo[i] = kFlagPrefix | r1;
        }
    }
}

// One warp per segment.  With every segment's bit offset known before the
// launch, a segment depends on no other segment and on no other warp, so a
// warp encodes whole segments alone, tile after tile (512 elements, 16 per
// lane), with its own bulk-copy ring and bit buffers: no block barrier on
// the path.  Per tile:
//   * lookups: the code table has a 256-byte row per byte value, holding 32
//     (code, length) slots: slot 16 p + lane % 16 for plane p.  One byte
//     permute makes the entry's address from an input byte and the lane's
//     slot, and the 16 lanes of a half-warp always read 16 different bank
//     pairs, whatever the symbols;
//   * the codes of consecutive symbols are joined into groups of 2, 4 or 8
//     while every group of the warp fits in 31 bits (one warp vote per plane
//     and tile picks the largest such size); a group is appended as one code;
//   * a warp scan of the lanes' bit counts gives each lane its start bit;
//     each lane stores the words it completes, and after that ORs its last,
//     partial word into the buffer.  The first word a lane completes holds
//     zeros where earlier lanes' bits go; those lanes OR their last words
//     into it afterwards.  The word the tile ends in is zeroed first, since
//     no lane completes it;
//   * complete words go out byte-swapped at the tile's global word; the word
//     the tile ends in stays in a register and lane 0 of the next tile starts
//     its bits behind it.
namespace wenc {
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kLaneElems = 16;
constexpr int kTile = 32 * kLaneElems;                                 // 512 elements
constexpr uint32_t kTilesPerSeg = static_cast<uint32_t>(kDirSegElems / kTile);  // 256
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kTile * 2;                             // the tile of w, then of x0
constexpr int kBufWords = 392;                                         // a tile's bits of one plane
constexpr size_t kTableBytes = 256 * 256;
constexpr size_t kRingBytes = size_t(kWarps) * kStages * kStageBytes;
constexpr size_t kBufBytes = size_t(kWarps) * 2 * kBufWords * 4;
constexpr size_t kBarBytes = size_t(kWarps) * kStages * 8;
constexpr size_t kSmem = kTableBytes + kRingBytes + kBufBytes + kBarBytes;
static_assert(kDirSegElems % kTile == 0, "segments of whole tiles");
static_assert((kBufWords - 1) * 32 >= 31 + kTile * HUFF_MAX_LEN + 32 && kBufWords % 4 == 0,
              "tile buffer, and a last slot no tile uses");
static_assert(kSmem <= 227 * 1024, "one CTA per SM");
}  // namespace wenc

// Table entry at byte address a (row = byte value, slot from the permute).
__device__ __forceinline__ uint2 wtab(const uint8_t *tab, uint32_t a) {
    return *reinterpret_cast<const uint2 *>(tab + a);
}

// Byte-permute selectors: byte 0 <- the lane's slot offset, byte 1 <- the
// symbol byte (row), bytes 2-3 <- zero.  Element 2j of a lane is the low half
// of its word j: high plane byte 1, low plane byte 0; element 2j+1 the high
// half: bytes 3 and 2.
constexpr uint32_t kSelHiA = 0x5514, kSelHiB = 0x5534, kSelLoA = 0x5504, kSelLoB = 0x5524;

// (code, length) of each pair of a lane's symbols in both planes; symbols at
// or past nvalid count as empty codes when RAGGED.
template <bool RAGGED>
__device__ __forceinline__ void wlookup(const uint8_t *tab, const uint32_t (&wv)[8], uint32_t kbh, uint32_t kbl,
                                        int nvalid, uint32_t (&m)[2][8], uint32_t (&L)[2][8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint2 ha = wtab(tab, __byte_perm(wv[j], kbh, kSelHiA));
        uint2 hb = wtab(tab, __byte_perm(wv[j], kbh, kSelHiB));
        uint2 la = wtab(tab, __byte_perm(wv[j], kbl, kSelLoA));
        uint2 lb = wtab(tab, __byte_perm(wv[j], kbl, kSelLoB));
        if (RAGGED) {
            if (2 * j >= nvalid) ha = la = make_uint2(0u, 0u);
            if (2 * j + 1 >= nvalid) hb = lb = make_uint2(0u, 0u);
        }
        m[0][j] = (ha.x << hb.y) | hb.x;  // meaningful while the pair fits 32 bits
        L[0][j] = ha.y + hb.y;
        m[1][j] = (la.x << lb.y) | lb.x;
        L[1][j] = la.y + lb.y;
    }
}

// A lane's bits of one plane in one tile.  Pending bits: the low nb bits of
// hi:lo (nb < 32 between appends); append(code, len) takes len <= 31.
// BUFWORDS: the tile buffer's size; its last slot is never part of a tile.
template <int BUFWORDS>
struct WPackerT {
    uint32_t hi, lo, nb, w;
    // A word that is not complete yet goes to the buffer's last slot, which no
    // tile uses: a plain store instead of a branch.
    __device__ __forceinline__ void append(uint32_t *buf, uint32_t code, uint32_t len) {
        hi = __funnelshift_l(lo, hi, len);
        lo = (lo << len) | code;
        nb += len;
        const bool full = nb >= 32;
        nb &= 31u;
        buf[full ? w : uint32_t(BUFWORDS - 1)] = __funnelshift_r(lo, hi, nb);
        w += full ? 1u : 0u;
    }
    // The last, partial word (an OR of zero when there is none).
    __device__ __forceinline__ void tail(uint32_t *buf) const {
        atomicOr(&buf[w], nb ? lo << (32u - nb) : 0u);
    }
};
using WPacker = WPackerT<wenc::kBufWords>;

// A lane's 16 elements (32 bytes, XOR x0 for the delta) straight from global
// memory; bytes at or past tile_n elements read as zero.
template <bool XOR>
__device__ __forceinline__ void wload_global(const uint8_t *in, const uint8_t *in2, size_t first, int lane,
                                             int tile_n, uint32_t (&wv)[8]) {
    const size_t b0 = (first + static_cast<size_t>(lane) * wenc::kLaneElems) * 2;
    if (tile_n == wenc::kTile) {
        const uint4 a = *reinterpret_cast<const uint4 *>(in + b0);
        const uint4 c = *reinterpret_cast<const uint4 *>(in + b0 + 16);
        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
        wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
        if (XOR) {
            const uint4 d = *reinterpret_cast<const uint4 *>(in2 + b0);
            const uint4 e = *reinterpret_cast<const uint4 *>(in2 + b0 + 16);
            wv[0] ^= d.x; wv[1] ^= d.y; wv[2] ^= d.z; wv[3] ^= d.w;
            wv[4] ^= e.x; wv[5] ^= e.y; wv[6] ^= e.z; wv[7] ^= e.w;
        }
    } else {
        const int tile_bytes = tile_n * 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = 0;
        for (int kk = 0; kk < 32; ++kk) {
            const int bb = lane * 32 + kk;
            if (bb >= tile_bytes) break;
            uint32_t v = in[first * 2 + bb];
            if (XOR) v ^= in2[first * 2 + bb];
            wv[kk >> 2] |= v << (8 * (kk & 3));
        }
    }
}

// Appends a lane's 16 symbols of one plane in the largest group size that fits
// 31 bits for every lane of the warp (warp-uniform branches).
template <bool XOR>
__device__ __forceinline__ void wpack(WPacker &pk, uint32_t *buf, const uint32_t (&m)[8], const uint32_t (&L)[8],
                                      const uint8_t *tab, uint32_t kb, uint32_t sel_a, uint32_t sel_b,
                                      const uint8_t *in, const uint8_t *in2, size_t first, int lane, int tile_n,
                                      int nvalid) {
    uint32_t Q[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) Q[q] = L[2 * q] + L[2 * q + 1];
    const uint32_t O0 = Q[0] + Q[1], O1 = Q[2] + Q[3];
    if (!__any_sync(0xffffffffu, max(O0, O1) > 31u)) {
        uint32_t M4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) M4[q] = (m[2 * q] << L[2 * q + 1]) | m[2 * q + 1];
        pk.append(buf, (M4[0] << Q[1]) | M4[1], O0);
        pk.append(buf, (M4[2] << Q[3]) | M4[3], O1);
    } else if (!__any_sync(0xffffffffu, max(max(Q[0], Q[1]), max(Q[2], Q[3])) > 31u)) {
#pragma unroll
        for (int q = 0; q < 4; ++q) pk.append(buf, (m[2 * q] << L[2 * q + 1]) | m[2 * q + 1], Q[q]);
    } else {
        uint32_t lmax = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) lmax = max(lmax, L[j]);
        if (!__any_sync(0xffffffffu, lmax > 31u)) {
#pragma unroll
            for (int j = 0; j < 8; ++j) pk.append(buf, m[j], L[j]);
        } else {
            // some pair is longer than 31 bits: one symbol at a time, read and looked up again
            uint32_t wv[8];
            wload_global<XOR>(in, in2, first, lane, tile_n, wv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint2 a = wtab(tab, __byte_perm(wv[j], kb, sel_a));
                uint2 b = wtab(tab, __byte_perm(wv[j], kb, sel_b));
                if (2 * j >= nvalid) a = make_uint2(0u, 0u);
                if (2 * j + 1 >= nvalid) b = make_uint2(0u, 0u);
                pk.append(buf, a.x, a.y);
                pk.append(buf, b.x, b.y);
            }
        }
    }
}

// Lane 0's copy job for tile kk of this warp's sequence counted from segment
// seg (which has `tiles` tiles); kk may run past that segment's end into the
// warp's next one.  No job when the sequence ends first.
template <bool XOR>
__device__ __forceinline__ void wissue(uint8_t *ring, uint64_t *bar, uint32_t stage, uint32_t seg, uint32_t kk,
                                       uint32_t tiles, uint32_t nw, uint32_t n_seg, uint32_t n_tiles,
                                       uint32_t last_bytes, const uint8_t *in, const uint8_t *in2, uint64_t pol) {
    if (kk >= tiles) {
        kk -= tiles;
        seg += nw;
        if (seg >= n_seg) return;
        const uint32_t rest = n_tiles - seg * wenc::kTilesPerSeg;
        if (kk >= (rest < wenc::kTilesPerSeg ? rest : wenc::kTilesPerSeg)) return;
    }
    const uint32_t t = seg * wenc::kTilesPerSeg + kk;
    const uint32_t bytes = t == n_tiles - 1 ? last_bytes : uint32_t(wenc::kTile * 2);  // every tile whole but the last
    const size_t src = static_cast<size_t>(t) * (wenc::kTile * 2);
    uint8_t *dst = ring + stage * wenc::kStageBytes;
    mbar_arrive_expect_tx(&bar[stage], bytes * (XOR ? 2u : 1u));
    if (bytes) {
        bulk_g2s_hint(dst, in + src, bytes, &bar[stage], pol);
        if (XOR) bulk_g2s_hint(dst + wenc::kTile * 2, in2 + src, bytes, &bar[stage], pol);
    }
}

// Complete words [skip, nfull) of a tile's buffer to dst (byte-swapped: the
// stream is a byte sequence, most significant bit first).
__device__ __forceinline__ void wwrite(uint32_t *dst, const uint32_t *buf, uint32_t skip, uint32_t nfull, int lane) {
#pragma unroll 1
    for (uint32_t i = skip + lane; i < nfull; i += 32) dst[i] = bswap32(buf[i]);
}

template <bool XOR>
__global__ void __launch_bounds__(wenc::kThreads, 1)
    k_encode_counted(const uint8_t *__restrict__ in, const uint8_t *__restrict__ in2, size_t n, EncPlane p0,
                     EncPlane p1, ChunkDiv cdiv, uint32_t n_tiles, uint32_t n_seg, int32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint8_t *tab = smem;
    uint8_t *ring = smem + wenc::kTableBytes + size_t(warp) * wenc::kStages * wenc::kStageBytes;
    uint32_t *buf0 = reinterpret_cast<uint32_t *>(smem + wenc::kTableBytes + wenc::kRingBytes) + warp * 2 * wenc::kBufWords;
    uint32_t *buf1 = buf0 + wenc::kBufWords;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + wenc::kTableBytes + wenc::kRingBytes + wenc::kBufBytes) + warp * wenc::kStages;

    // code table: row = byte value, slot = 16 plane + copy; entry (code, length), (0, 0) without a code
    const bool ok0 = p0.cb->magic == HUFF_CODEBOOK_MAGIC, ok1 = p1.cb->magic == HUFF_CODEBOOK_MAGIC;
    for (int i = tid; i < 256 * 32; i += wenc::kThreads) {
        const int sym = i >> 5;
        const bool lo_plane = (i & 31) >= 16;
        const huff_codebook *cb = lo_plane ? p1.cb : p0.cb;
        const uint32_t len = (lo_plane ? ok1 : ok0) ? cb->len[sym] : 0u;
        const bool has = len >= 1 && len <= HUFF_MAX_LEN;
        reinterpret_cast<uint2 *>(smem)[i] = make_uint2(has ? cb->code[sym] : 0u, has ? len : 0u);
    }
    if (tid == 0 && !(ok0 && ok1)) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
    if (lane == 0) {
        for (int s = 0; s < wenc::kStages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();  // the table and the barriers are ready

    const uint32_t nw = gridDim.x * wenc::kWarps;
    const uint32_t gw = static_cast<uint32_t>(warp) * gridDim.x + blockIdx.x;  // round r: segment r nw + gw
    const uint64_t pol = l2_policy_evict_first();
    const uint32_t last_n = static_cast<uint32_t>(n - static_cast<size_t>(n_tiles - 1) * wenc::kTile);  // 1..512
    const uint32_t last_bytes = (last_n * 2) & ~15u;
    if (lane == 0 && gw < n_seg) {  // the first kStages tiles of the warp's sequence
        const uint32_t rest = n_tiles - gw * wenc::kTilesPerSeg;
        const uint32_t tiles0 = rest < wenc::kTilesPerSeg ? rest : wenc::kTilesPerSeg;
        for (int j = 0; j < wenc::kStages; ++j)
            wissue<XOR>(ring, bar, j, gw, j, tiles0, nw, n_seg, n_tiles, last_bytes, in, in2, pol);
    }
    const uint32_t kbh = static_cast<uint32_t>(lane & 15) << 3;
    const uint32_t kbl = kbh + 128u;
    uint32_t cstage = 0, cphase = 0;

    for (uint32_t r = 0;; ++r) {
        const uint32_t seg = r * nw + gw;
        if (seg >= n_seg) break;
        const uint32_t t0 = seg * wenc::kTilesPerSeg;
        const uint32_t tiles = n_tiles - t0 < wenc::kTilesPerSeg ? n_tiles - t0 : wenc::kTilesPerSeg;
        // Bit positions inside the segment are 32-bit (a segment has at most 131072 * 24 bits): pos =
        // the segment's phase in its first word + bits so far; word pos >> 5 of the segment is global
        // word (start >> 5) + (pos >> 5).
        const uint64_t start0 = seg ? (p0.desc[seg - 1] & kValueMask) : 0;
        const uint64_t start1 = seg ? (p1.desc[seg - 1] & kValueMask) : 0;
        uint32_t *const dst0 = p0.payload + (start0 >> 5);
        uint32_t *const dst1 = p1.payload + (start1 >> 5);
        // bits this segment may write before its plane's capacity ends
        const uint64_t room0 = start0 >> 5 < p0.cap_words ? (p0.cap_words - (start0 >> 5)) * 32 : 0;
        const uint64_t room1 = start1 >> 5 < p1.cap_words ? (p1.cap_words - (start1 >> 5)) * 32 : 0;
        const uint32_t lim0 = room0 < 0xffffffffull ? static_cast<uint32_t>(room0) : 0xffffffffu;
        const uint32_t lim1 = room1 < 0xffffffffull ? static_cast<uint32_t>(room1) : 0xffffffffu;
        uint32_t pos0 = static_cast<uint32_t>(start0 & 31u), pos1 = static_cast<uint32_t>(start1 & 31u);
        uint32_t carry0 = 0, carry1 = 0, head0 = 0, head1 = 0;
        const size_t seg_first = static_cast<size_t>(t0) * wenc::kTile;
        // the next chunk start: to_next elements ahead, chunk number next_q
        const uint32_t cr = static_cast<uint32_t>(seg_first % cdiv.chunk);
        uint64_t next_q = seg_first / cdiv.chunk + (cr ? 1u : 0u);
        uint32_t to_next = cr ? cdiv.chunk - cr : 0u;
        for (uint32_t k = 0; k < tiles; ++k) {
            const int tile_n = t0 + k == n_tiles - 1 ? static_cast<int>(last_n) : wenc::kTile;
            if (!mbar_wait(&bar[cstage], cphase) && lane == 0) set_status(status, HUFF_ERR_TIMEOUT);
            const uint8_t *st = ring + cstage * wenc::kStageBytes;
            uint32_t wv[8];
            {
                const uint4 a = *reinterpret_cast<const uint4 *>(st + lane * 32);
                const uint4 c = *reinterpret_cast<const uint4 *>(st + lane * 32 + 16);
                wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
                if (XOR) {
                    const uint4 d = *reinterpret_cast<const uint4 *>(st + wenc::kTile * 2 + lane * 32);
                    const uint4 e = *reinterpret_cast<const uint4 *>(st + wenc::kTile * 2 + lane * 32 + 16);
                    wv[0] ^= d.x; wv[1] ^= d.y; wv[2] ^= d.z; wv[3] ^= d.w;
                    wv[4] ^= e.x; wv[5] ^= e.y; wv[6] ^= e.z; wv[7] ^= e.w;
                }
            }
            const int nvalid = tile_n - lane * wenc::kLaneElems < 0
                                   ? 0
                                   : (tile_n - lane * wenc::kLaneElems > wenc::kLaneElems ? wenc::kLaneElems
                                                                                          : tile_n - lane * wenc::kLaneElems);
            if (tile_n < wenc::kTile) {
                // the last tile: bytes past the bulk copy's 16-byte multiple come from global memory
                const size_t first = seg_first + static_cast<size_t>(k) * wenc::kTile;
                const int tile_bytes = tile_n * 2, tma_bytes = tile_bytes & ~15;
                for (int kk = 0; kk < 32; ++kk) {
                    const int bb = lane * 32 + kk;
                    if (bb < tma_bytes) continue;
                    uint32_t v = 0;
                    if (bb < tile_bytes) {
                        v = in[first * 2 + bb];
                        if (XOR) v ^= in2[first * 2 + bb];
                    }
                    wv[kk >> 2] = (wv[kk >> 2] & ~(0xffu << (8 * (kk & 3)))) | (v << (8 * (kk & 3)));
                }
            }
            consumed(wv);
            __syncwarp();  // every lane has read the stage
            if (lane == 0) fence_proxy_async_smem();  // the reads before the bulk copy that refills the stage
            // the stage is free again: lane 0 refills it with the tile kStages further on
            if (lane == 0)
                wissue<XOR>(ring, bar, cstage, seg, k + wenc::kStages, tiles, nw, n_seg, n_tiles, last_bytes, in, in2,
                            pol);
            cstage = cstage + 1 == uint32_t(wenc::kStages) ? 0u : cstage + 1;
            cphase ^= cstage == 0 ? 1u : 0u;

            uint32_t m[2][8], L[2][8];
            if (tile_n == wenc::kTile)
                wlookup<false>(tab, wv, kbh, kbl, wenc::kLaneElems, m, L);
            else
                wlookup<true>(tab, wv, kbh, kbl, nvalid, m, L);
            uint32_t b0 = 0, b1 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                b0 += L[0][j];
                b1 += L[1][j];
            }
            // warp scan of (high plane bits << 16 | low plane bits): a lane has at most
            // 16 * 24 bits per plane, a warp at most 12288
            const uint32_t mine = (b0 << 16) | b1;
            uint32_t incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t excl = incl - mine;
            const uint32_t ex0 = excl >> 16, ex1 = excl & 0xffffu, tot0 = tot >> 16, tot1 = tot & 0xffffu;

            // chunk starts in this tile (chunks are multiples of 256 elements, so a chunk starts
            // at the first element of some lane)
            if (to_next < wenc::kTile) {
                do {
                    if (static_cast<uint32_t>(lane) * wenc::kLaneElems == to_next && to_next < uint32_t(tile_n)) {
                        p0.off[next_q] = start0 + (pos0 - (start0 & 31u)) + ex0;
                        p1.off[next_q] = start1 + (pos1 - (start1 & 31u)) + ex1;
                    }
                    to_next += cdiv.chunk;
                    ++next_q;
                } while (to_next < wenc::kTile);
            }
            to_next -= wenc::kTile;

            const uint32_t ph0 = pos0 & 31u, ph1 = pos1 & 31u;
            const uint32_t end0 = ph0 + tot0, end1 = ph1 + tot1;
            // the words the tile ends in: no lane completes them (all lanes store the same zero)
            buf0[end0 >> 5] = 0;
            buf1[end1 >> 5] = 0;
            WPacker q0, q1;
            {
                const uint32_t s0 = ph0 + ex0, s1 = ph1 + ex1;
                q0.hi = q1.hi = 0;
                q0.nb = s0 & 31u;
                q0.w = s0 >> 5;
                q1.nb = s1 & 31u;
                q1.w = s1 >> 5;
                // lane 0 starts with the previous tile's bits of the word it starts in
                q0.lo = lane == 0 ? __funnelshift_rc(carry0, 0u, 32u - ph0) : 0u;
                q1.lo = lane == 0 ? __funnelshift_rc(carry1, 0u, 32u - ph1) : 0u;
            }
            {
                const size_t first = seg_first + static_cast<size_t>(k) * wenc::kTile;
                wpack<XOR>(q0, buf0, m[0], L[0], tab, kbh, kSelHiA, kSelHiB, in, in2, first, lane, tile_n, nvalid);
                wpack<XOR>(q1, buf1, m[1], L[1], tab, kbl, kSelLoA, kSelLoB, in, in2, first, lane, tile_n, nvalid);
            }
            __syncwarp();  // whole words stored
            q0.tail(buf0);
            q1.tail(buf1);
            __syncwarp();  // partial words ORed in
            const uint32_t nf0 = end0 >> 5, nf1 = end1 >> 5;
            // a segment's first word, when it starts inside one, is the fix-up kernel's to write
            const uint32_t sk0 = (k == 0 && ph0) ? 1u : 0u, sk1 = (k == 0 && ph1) ? 1u : 0u;
            if (pos0 + tot0 <= lim0 && pos1 + tot1 <= lim1) {
                wwrite(dst0 + (pos0 >> 5), buf0, sk0, nf0, lane);
                wwrite(dst1 + (pos1 >> 5), buf1, sk1, nf1, lane);
            } else if (lane == 0) {
                set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
            }
            if (k == 0) {
                head0 = ph0 ? buf0[0] : 0u;
                head1 = ph1 ? buf1[0] : 0u;
            }
            carry0 = buf0[nf0];  // zero when the tile ends on a word boundary
            carry1 = buf1[nf1];
            pos0 += tot0;
            pos1 += tot1;
            __syncwarp();  // buffers read before the next tile writes them
        }
        if (lane == 0) {
            p0.edge[seg] = (static_cast<uint64_t>(head0) << 32) | carry0;
            p1.edge[seg] = (static_cast<uint64_t>(head1) << 32) | carry1;
            // the bits written must be the bits the counts gave this segment
            if (start0 - (start0 & 31u) + pos0 != (p0.desc[seg] & kValueMask) ||
                start1 - (start1 & 31u) + pos1 != (p1.desc[seg] & kValueMask))
                set_status(status, HUFF_ERR_INVALID_ARG);
        }
    }
}

// ------------------------------------------------------------------ byte streams, one warp per segment
//
// With a given codebook (the fixed one, or a shard's own), a segment's bit
// count is not known before its symbols are read, so a warp makes two passes
// over each segment of seg_tiles tiles (16; down to 4 for small inputs, so
// that there are segments for every warp): it streams the tiles in (L2 policy
// evict_last) and counts their bits, publishes the count and looks back over
// the earlier segments' descriptors for its offset (decoupled lookback), then
// streams the same tiles again from L2 (evict_first) and packs them as the
// counted bf16 encode does, one plane of 32 symbols per lane.  Segments are
// claimed in order from a counter, and a warp claims its next segment only
// three tiles before the end of its current one (its copy jobs run three
// tiles ahead): a claimed segment is started right away, so the segments a
// lookback waits on are being counted at the same time, not queued behind
// another segment.  A symbol without a code has the table length 0x1000, so a
// tile's count shows it; such a segment sets the status and is not packed.
namespace wenc8 {
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kLaneSyms = 32;
constexpr int kTile = 32 * kLaneSyms;  // 1024 symbols
constexpr int kSegTilesMax = 16;       // 16 384 symbols per segment for large inputs
constexpr int kSegTilesMin = 4;        // at least kStages + 1 tiles, for the claim three tiles before the end
constexpr int kStages = 3;
constexpr int kStageBytes = kTile;
constexpr int kBufWords = 776;
constexpr uint32_t kNoCode = 0x1000;   // table length of a symbol without a code
constexpr size_t kTableBytes = 256 * 256;
constexpr size_t kRingBytes = size_t(kWarps) * kStages * kStageBytes;
constexpr size_t kBufBytes = size_t(kWarps) * kBufWords * 4;
constexpr size_t kBarBytes = size_t(kWarps) * kStages * 8;
constexpr size_t kSmem = kTableBytes + kRingBytes + kBufBytes + kBarBytes;
static_assert((kBufWords - 1) * 32 >= 31 + kTile * HUFF_MAX_LEN + 32 && kBufWords % 4 == 0, "tile buffer");
static_assert(kLaneSyms * HUFF_MAX_LEN < int(kNoCode), "a lane's count stays below the no-code mark");
static_assert(kSegTilesMin > kStages, "a full segment claims its successor three tiles before its end");
}  // namespace wenc8

using WPacker8 = WPackerT<wenc8::kBufWords>;

// Lane 0's copy-job cursor: pass p (0 count, 1 pack) of tile k of segment
// seg; p == 2 once the segment's jobs are all issued (the next segment is
// taken from the claim when its first job is due).
struct Job8 {
    uint32_t seg, k, pass;
};

__device__ __forceinline__ uint32_t seg_tiles8(uint32_t seg, uint32_t n_tiles, uint32_t st) {
    const uint32_t rest = n_tiles - seg * st;
    return rest < st ? rest : st;
}

// Issue the cursor's job into `stage` and advance it; seg_next is the warp's
// claim of its next segment (0xffffffff until made), taken when the current
// segment's jobs are done.
__device__ __forceinline__ void wissue8(uint8_t *ring, uint64_t *bar, uint32_t stage, Job8 &j, uint32_t &seg_next,
                                        uint32_t n_seg, uint32_t n_tiles, uint32_t st, uint32_t last_bytes,
                                        const uint8_t *in, uint64_t pol_keep, uint64_t pol_drop) {
    if (j.pass == 2) {
        j.seg = seg_next;
        j.pass = 0;
        j.k = 0;
        seg_next = 0xffffffffu;  // taken: the next claim replaces it
    }
    if (j.seg >= n_seg) return;
    const uint32_t t = j.seg * st + j.k;
    const uint32_t bytes = t == n_tiles - 1 ? last_bytes : uint32_t(wenc8::kTile);
    mbar_arrive_expect_tx(&bar[stage], bytes);
    if (bytes)
        bulk_g2s_hint(ring + stage * wenc8::kStageBytes, in + static_cast<size_t>(t) * wenc8::kTile, bytes, &bar[stage],
                      j.pass ? pol_drop : pol_keep);
    if (++j.k == seg_tiles8(j.seg, n_tiles, st)) {
        j.k = 0;
        ++j.pass;
    }
}

// A lane's 32 symbols: pairs of consecutive symbols as (code, length).
template <bool RAGGED>
__device__ __forceinline__ void wlookup8(const uint8_t *tab, const uint32_t (&wv)[8], uint32_t kb, int nvalid,
                                         uint32_t (&m)[16], uint32_t (&L)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t word = wv[j >> 1];
        const uint32_t sa = (j & 1) ? 0x5524u : 0x5504u, sb = (j & 1) ? 0x5534u : 0x5514u;
        uint2 a = wtab(tab, __byte_perm(word, kb, sa));
        uint2 b = wtab(tab, __byte_perm(word, kb, sb));
        if (RAGGED) {
            if (2 * j >= nvalid) a = make_uint2(0u, 0u);
            if (2 * j + 1 >= nvalid) b = make_uint2(0u, 0u);
        }
        m[j] = (a.x << b.y) | b.x;
        L[j] = a.y + b.y;
    }
}

// A lane's 32 bytes of a tile from global memory (bytes at or past tile_n read as zero).
__device__ __forceinline__ void wload8(const uint8_t *in, size_t first, int lane, int tile_n, uint32_t (&wv)[8]) {
    const size_t b0 = first + static_cast<size_t>(lane) * wenc8::kLaneSyms;
    if (tile_n == wenc8::kTile) {  // in is 16-byte aligned and first a multiple of 1024
        const uint4 a = *reinterpret_cast<const uint4 *>(in + b0);
        const uint4 c = *reinterpret_cast<const uint4 *>(in + b0 + 16);
        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
        wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
        return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) wv[j] = 0;
    for (int k = 0; k < wenc8::kLaneSyms; ++k) {
        const int bb = lane * wenc8::kLaneSyms + k;
        if (bb >= tile_n) break;
        wv[k >> 2] |= static_cast<uint32_t>(in[b0 + k]) << (8 * (k & 3));
    }
}

// Appends a lane's 32 symbols in the largest group size that fits 31 bits for every lane.
__device__ __forceinline__ void wpack8(WPacker8 &pk, uint32_t *buf, const uint32_t (&m)[16], const uint32_t (&L)[16],
                                       const uint8_t *tab, uint32_t kb, const uint8_t *in, size_t first, int lane,
                                       int tile_n, int nvalid) {
    uint32_t Q[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) Q[q] = L[2 * q] + L[2 * q + 1];
    uint32_t O[4];
#pragma unroll
    for (int o = 0; o < 4; ++o) O[o] = Q[2 * o] + Q[2 * o + 1];
    if (!__any_sync(0xffffffffu, max(max(O[0], O[1]), max(O[2], O[3])) > 31u)) {
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            const uint32_t qa = (m[4 * o] << L[4 * o + 1]) | m[4 * o + 1];
            const uint32_t qb = (m[4 * o + 2] << L[4 * o + 3]) | m[4 * o + 3];
            pk.append(buf, (qa << Q[2 * o + 1]) | qb, O[o]);
        }
    } else {
        uint32_t qmax = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) qmax = max(qmax, Q[q]);
        if (!__any_sync(0xffffffffu, qmax > 31u)) {
#pragma unroll
            for (int q = 0; q < 8; ++q) pk.append(buf, (m[2 * q] << L[2 * q + 1]) | m[2 * q + 1], Q[q]);
        } else {
            uint32_t lmax = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) lmax = max(lmax, L[j]);
            if (!__any_sync(0xffffffffu, lmax > 31u)) {
#pragma unroll
                for (int j = 0; j < 16; ++j) pk.append(buf, m[j], L[j]);
            } else {
                // some pair is longer than 31 bits: one symbol at a time, read and looked up again
                uint32_t wv[8];
                wload8(in, first, lane, tile_n, wv);
#pragma unroll
                for (int k = 0; k < wenc8::kLaneSyms; ++k) {
                    uint2 e = wtab(tab, __byte_perm(wv[k >> 2], kb, 0x5504u + 0x10u * (k & 3)));
                    if (k >= nvalid) e = make_uint2(0u, 0u);
                    pk.append(buf, e.x, e.y);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(wenc8::kThreads, 1)
    k_encode_u8w(const uint8_t *__restrict__ in, size_t n, EncPlane P, uint32_t chunk, uint32_t n_tiles,
                 uint32_t st, uint32_t n_seg, unsigned *seg_ctr, int32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint8_t *tab = smem;
    uint8_t *ring = smem + wenc8::kTableBytes + size_t(warp) * wenc8::kStages * wenc8::kStageBytes;
    uint32_t *buf = reinterpret_cast<uint32_t *>(smem + wenc8::kTableBytes + wenc8::kRingBytes) + warp * wenc8::kBufWords;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + wenc8::kTableBytes + wenc8::kRingBytes + wenc8::kBufBytes) +
                    warp * wenc8::kStages;

    // code table: row = byte value, slot = lane; entry (code, length); no code: (0, kNoCode)
    const bool ok = P.cb->magic == HUFF_CODEBOOK_MAGIC;
    for (int i = tid; i < 256 * 32; i += wenc8::kThreads) {
        const int sym = i >> 5;
        const uint32_t len = ok ? P.cb->len[sym] : 0u;
        const bool has = len >= 1 && len <= HUFF_MAX_LEN;
        reinterpret_cast<uint2 *>(smem)[i] = make_uint2(has ? P.cb->code[sym] : 0u, has ? len : wenc8::kNoCode);
    }
    if (tid == 0 && !ok) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
    if (lane == 0) {
        for (int s = 0; s < wenc8::kStages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol_keep = l2_policy_evict_last(), pol_drop = l2_policy_evict_first();
    const uint32_t last_n = static_cast<uint32_t>(n - static_cast<size_t>(n_tiles - 1) * wenc8::kTile);  // 1..1024
    const uint32_t last_bytes = last_n & ~15u;
    const uint32_t kb = static_cast<uint32_t>(lane) << 3;
    // the warp's segment (claimed in order), lane 0's copy-job cursor
    uint32_t seg = 0;
    if (lane == 0) seg = atomicAdd(seg_ctr, 1u);
    seg = __shfl_sync(0xffffffffu, seg, 0);
    Job8 job{seg, 0, 0};
    uint32_t job_next = 0xffffffffu;  // lane 0: the next segment, once claimed
    if (lane == 0)
        for (int s = 0; s < wenc8::kStages; ++s)
            wissue8(ring, bar, s, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep, pol_drop);
    uint32_t cstage = 0, cphase = 0;

    auto next_stage = [&]() {
        cstage = cstage + 1 == uint32_t(wenc8::kStages) ? 0u : cstage + 1;
        cphase ^= cstage == 0 ? 1u : 0u;
    };
    // a lane's 32 bytes of the tile in the current stage (global memory for bytes past the bulk copy)
    auto read_stage = [&](size_t first, int tile_n, uint32_t (&wv)[8]) {
        if (!mbar_wait(&bar[cstage], cphase) && lane == 0) set_status(status, HUFF_ERR_TIMEOUT);
        const uint8_t *st = ring + cstage * wenc8::kStageBytes;
        const uint4 a = *reinterpret_cast<const uint4 *>(st + lane * 32);
        const uint4 c = *reinterpret_cast<const uint4 *>(st + lane * 32 + 16);
        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
        wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
        if (tile_n < wenc8::kTile) {
            const int tma = tile_n & ~15;
            for (int k = 0; k < 32; ++k) {
                const int bb = lane * 32 + k;
                if (bb < tma) continue;
                const uint32_t v = bb < tile_n ? in[first + bb] : 0u;
                wv[k >> 2] = (wv[k >> 2] & ~(0xffu << (8 * (k & 3)))) | (v << (8 * (k & 3)));
            }
        }
        consumed(wv);
        __syncwarp();  // every lane has read the stage
        if (lane == 0) fence_proxy_async_smem();  // the reads before the bulk copy that refills the stage
    };

    while (seg < n_seg) {
        const uint32_t tiles = seg_tiles8(seg, n_tiles, st);
        const size_t seg_first = static_cast<size_t>(seg) * st * wenc8::kTile;
        // ---------------- pass 1: the segment's bits
        uint32_t bits = 0;
        bool no_code = false;
        for (uint32_t k = 0; k < tiles; ++k) {
            const size_t first = seg_first + static_cast<size_t>(k) * wenc8::kTile;
            const int tile_n = seg * st + k == n_tiles - 1 ? static_cast<int>(last_n) : wenc8::kTile;
            uint32_t wv[8];
            read_stage(first, tile_n, wv);
            if (lane == 0) wissue8(ring, bar, cstage, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep,
                                    pol_drop);
            next_stage();
            const int nvalid = tile_n - lane * 32 < 0 ? 0 : (tile_n - lane * 32 > 32 ? 32 : tile_n - lane * 32);
            uint32_t b = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint32_t y = wtab(tab, __byte_perm(wv[j >> 2], kb, 0x5504u + 0x10u * (j & 3))).y;
                b += j < nvalid ? y : 0u;
            }
            no_code |= b >= wenc8::kNoCode;  // a lane's tile counts at most 32 * 24 bits
            bits += b;
        }
        // a symbol without a code shows as a tile count of 0x1000 or more in some lane
        const bool missing = __any_sync(0xffffffffu, no_code);
        uint64_t seg_bits = static_cast<uint64_t>(missing ? 0u : bits);
        seg_bits = warp_sum_u64(seg_bits);
        if (missing && lane == 0) set_status(status, HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK);
        // publish, look back
        if (lane == 0) st_relaxed(&P.desc[seg], (seg == 0 ? kFlagPrefix : kFlagAggregate) | seg_bits);
        uint64_t start = 0;
        if (seg != 0) {
            uint64_t wnd[kLookbackPerLane];
            load_window(P.desc, static_cast<int64_t>(seg) - 1, lane, wnd);
            start = lookback(P.desc, seg, lane, status, wnd);
            if (lane == 0) st_relaxed(&P.desc[seg], kFlagPrefix | (start + seg_bits));
        }
        // ---------------- pass 2: pack, tile after tile
        uint32_t *const dst = P.payload + (start >> 5);
        const uint64_t room = start >> 5 < P.cap_words ? (P.cap_words - (start >> 5)) * 32 : 0;
        const uint32_t lim = room < 0xffffffffull ? static_cast<uint32_t>(room) : 0xffffffffu;
        uint32_t pos = static_cast<uint32_t>(start & 31u);
        uint32_t carry = 0, head = 0;
        const uint32_t cr = static_cast<uint32_t>(seg_first % chunk);
        uint64_t next_q = seg_first / chunk + (cr ? 1u : 0u);
        uint32_t to_next = cr ? chunk - cr : 0u;
        uint32_t seg_next = 0xffffffffu;
        for (uint32_t k = 0; k < tiles; ++k) {
            const size_t first = seg_first + static_cast<size_t>(k) * wenc8::kTile;
            const int tile_n = seg * st + k == n_tiles - 1 ? static_cast<int>(last_n) : wenc8::kTile;
            if (k + wenc8::kStages == tiles) {  // the copy job about to be issued is the next segment's first
                uint32_t claim = 0;
                if (lane == 0) job_next = claim = atomicAdd(seg_ctr, 1u);
                seg_next = __shfl_sync(0xffffffffu, claim, 0);
            }
            uint32_t wv[8];
            read_stage(first, tile_n, wv);
            if (lane == 0) wissue8(ring, bar, cstage, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep,
                                    pol_drop);
            next_stage();
            if (missing) continue;  // the status is set; this segment's stream is not written
            const int nvalid = tile_n - lane * 32 < 0 ? 0 : (tile_n - lane * 32 > 32 ? 32 : tile_n - lane * 32);
            uint32_t m[16], L[16];
            if (tile_n == wenc8::kTile)
                wlookup8<false>(tab, wv, kb, 32, m, L);
            else
                wlookup8<true>(tab, wv, kb, nvalid, m, L);
            uint32_t b = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) b += L[j];
            uint32_t incl = b;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t excl = incl - b;
            if (to_next < uint32_t(wenc8::kTile)) {
                do {
                    if (static_cast<uint32_t>(lane) * wenc8::kLaneSyms == to_next && to_next < uint32_t(tile_n))
                        P.off[next_q] = start + (pos - (start & 31u)) + excl;
                    to_next += chunk;
                    ++next_q;
                } while (to_next < uint32_t(wenc8::kTile));
            }
            to_next -= wenc8::kTile;
            const uint32_t ph = pos & 31u, end = ph + tot;
            buf[end >> 5] = 0;  // the word the tile ends in: no lane completes it
            WPacker8 q;
            {
                const uint32_t s0 = ph + excl;
                q.hi = 0;
                q.nb = s0 & 31u;
                q.w = s0 >> 5;
                q.lo = lane == 0 ? __funnelshift_rc(carry, 0u, 32u - ph) : 0u;
            }
            wpack8(q, buf, m, L, tab, kb, in, first, lane, tile_n, nvalid);
            __syncwarp();
            q.tail(buf);
            __syncwarp();
            const uint32_t nf = end >> 5;
            const uint32_t sk = (k == 0 && ph) ? 1u : 0u;
            if (pos + tot <= lim) {
                wwrite(dst + (pos >> 5), buf, sk, nf, lane);
            } else if (lane == 0) {
                set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
            }
            if (k == 0) head = ph ? buf[0] : 0u;
            carry = buf[nf];
            pos += tot;
            __syncwarp();
        }
        if (lane == 0) P.edge[seg] = (static_cast<uint64_t>(head) << 32) | carry;
        // a segment of fewer than kStages tiles is the last one: no next segment then
        seg = seg_next;
    }
}

// Boundary words: the word where segment t-1 ends and segment t begins holds
// bits of both; the stream's last, partial word holds the end of the last
// segment.
__global__ void k_encode_fixup(EncPlane p0, EncPlane p1, int planes, uint32_t n_seg, size_t n_chunks,
                               int32_t *status) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_seg) return;
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
        if (t + 1 == n_seg) {
            const bool own_word = (end & 31u) && !(ph && (end >> 5) == (start >> 5));
            if (own_word) put_word(P.payload, P.cap_words, end >> 5, static_cast<uint32_t>(e), status);
            P.off[n_chunks] = end;
        }
    }
}

template <bool BF16, bool XOR>
int run_encode(const uint8_t *in, const uint8_t *in2, size_t n, EncPlane p0, EncPlane p1, size_t chunk,
               uint32_t n_tiles, unsigned *seg_ctr, int32_t *status, cudaStream_t s) {
    using C = EncCfg<BF16, XOR>;
    auto kern = k_encode<BF16, XOR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) !=
        cudaSuccess)
        return HUFF_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, C::kSmem) != cudaSuccess)
        return HUFF_ERR_CUDA;
    if (per_sm < 1) return HUFF_ERR_CUDA;
    const uint32_t n_seg = (n_tiles + kSegTiles - 1) / kSegTiles;
    const DevInfo d = dev_info();
    size_t grid = static_cast<size_t>(d.sms) * per_sm;
    if (grid > n_seg) grid = n_seg;
    // segments are claimed in order by CTAs that are already running, so every segment a
    // lookback waits for belongs to a resident CTA and the grid needs no co-residency
    kern<<<static_cast<unsigned>(grid), kThreads, C::kSmem, s>>>(in, in2, n, p0, p1, make_chunk_div(chunk), n_tiles,
                                                                  seg_ctr, status);
    if (cudaGetLastError() != cudaSuccess) return HUFF_ERR_CUDA;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    k_encode_fixup<<<(n_seg + 255) / 256, 256, 0, s>>>(p0, p1, C::kPlanes, n_seg, n_chunks, status);
    return launch_status();
}

__global__ void k_encode_empty(uint64_t *off0, uint64_t *off1) {
    off0[0] = 0;
    if (off1) off1[0] = 0;
}

}  // namespace

// Tiles per segment of the byte-stream encode: 16 when there are at least 8192
// tiles per 16 of them (two segments and more for every warp of a large GPU),
// fewer down to 4 for smaller inputs, so that small inputs still fill the GPU.
size_t enc_u8_seg_tiles(size_t n) {
    const size_t tiles = (n + wenc8::kTile - 1) / wenc8::kTile;
    size_t st = tiles / 8192;
    if (st < size_t(wenc8::kSegTilesMin)) st = wenc8::kSegTilesMin;
    if (st > size_t(wenc8::kSegTilesMax)) st = wenc8::kSegTilesMax;
    return st;
}

// Workspace words of the byte-stream encode: descriptor and edge word per segment, and a counter.
size_t enc_u8_workspace_words(size_t n) {
    const size_t tiles = (n + wenc8::kTile - 1) / wenc8::kTile;
    const size_t st = enc_u8_seg_tiles(n);
    return 2 * ((tiles + st - 1) / st) + 2;
}
size_t enc_bf16_tiles(size_t n) { return (n + kEncBf16Tile - 1) / kEncBf16Tile; }

int launch_encode_u8(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk, uint8_t *payload,
                     size_t cap, uint64_t *off, void *ws, int32_t *status, cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off, nullptr);
        return launch_status();
    }
    const size_t tiles = (n + wenc8::kTile - 1) / wenc8::kTile;
    const size_t seg_tiles = enc_u8_seg_tiles(n);
    const size_t segs = (tiles + seg_tiles - 1) / seg_tiles;
    uint64_t *w = static_cast<uint64_t *>(ws);
    // layout: segment descriptors, segment counter (both zeroed), edge words (written before they are read);
    // 2 segs + 1 words, within huff_workspace_size
    int st = launch_zero_u64(w, segs + 1, s);
    if (st != HUFF_OK) return st;
    EncPlane p0{cb, reinterpret_cast<uint32_t *>(payload), cap / 4, off, w, w + segs + 1};
    unsigned *ctr = reinterpret_cast<unsigned *>(w + segs);
    if (cudaFuncSetAttribute(k_encode_u8w, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(wenc8::kSmem)) != cudaSuccess)
        return HUFF_ERR_CUDA;
    // one CTA of 16 warps per SM, fewer when there are fewer segments than warps
    const size_t sms = static_cast<size_t>(dev_info().sms);
    size_t grid = (segs + wenc8::kWarps - 1) / wenc8::kWarps;
    if (grid > sms) grid = sms;
    k_encode_u8w<<<static_cast<unsigned>(grid), wenc8::kThreads, wenc8::kSmem, s>>>(
        in, n, p0, static_cast<uint32_t>(chunk), static_cast<uint32_t>(tiles), static_cast<uint32_t>(seg_tiles),
        static_cast<uint32_t>(segs), ctr, status);
    if (cudaGetLastError() != cudaSuccess) return HUFF_ERR_CUDA;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    k_encode_fixup<<<static_cast<unsigned>((segs + 255) / 256), 256, 0, s>>>(p0, p0, 1, static_cast<uint32_t>(segs),
                                                                              n_chunks, status);
    return launch_status();
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
    if (enc_u8_workspace_words(n) > kNoAllocScratchWords) return HUFF_ERR_BUFFER_TOO_SMALL;
    uint64_t *ws = noalloc_scratch_address();
    if (ws == nullptr) return HUFF_ERR_CUDA;
    // the same path as huff_encode; it zeroes what must start at zero before the encode kernel runs
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
    const size_t segs = (tiles + kSegTiles - 1) / kSegTiles;
    uint64_t *w = static_cast<uint64_t *>(ws);
    // layout: desc_hi, desc_lo, segment counter (zeroed), edge_hi, edge_lo
    int st = launch_zero_u64(w, 2 * segs + 1, s);
    if (st != HUFF_OK) return st;
    EncPlane p0{cb_hi, reinterpret_cast<uint32_t *>(pay_hi), cap_hi / 4, off_hi, w, w + 2 * segs + 1};
    EncPlane p1{cb_lo, reinterpret_cast<uint32_t *>(pay_lo), cap_lo / 4, off_lo, w + segs, w + 3 * segs + 1};
    unsigned *ctr = reinterpret_cast<unsigned *>(w + 2 * segs);
    const uint8_t *a = reinterpret_cast<const uint8_t *>(w16);
    if (x0 != nullptr)
        return run_encode<true, true>(a, reinterpret_cast<const uint8_t *>(x0), n, p0, p1, chunk,
                                      static_cast<uint32_t>(tiles), ctr, status, s);
    return run_encode<true, false>(a, nullptr, n, p0, p1, chunk, static_cast<uint32_t>(tiles), ctr, status, s);
}

int launch_encode_bf16_counted(const uint16_t *w16, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                               const huff_codebook *cb_lo, size_t chunk, const uint32_t *seg_counts,
                               uint8_t *pay_hi, size_t cap_hi, uint64_t *off_hi, uint8_t *pay_lo, size_t cap_lo,
                               uint64_t *off_lo, void *ws, int32_t *status, cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off_hi, off_lo);
        return launch_status();
    }
    const size_t tiles = enc_bf16_tiles(n);
    const size_t segs = (tiles + kDirSegTiles - 1) / kDirSegTiles;
    uint64_t *w = static_cast<uint64_t *>(ws);
    // layout: desc_hi, desc_lo, edge_hi, edge_lo, 32-bit bits (2 x segs), ticket counter (zeroed)
    EncPlane p0{cb_hi, reinterpret_cast<uint32_t *>(pay_hi), cap_hi / 4, off_hi, w, w + 2 * segs};
    EncPlane p1{cb_lo, reinterpret_cast<uint32_t *>(pay_lo), cap_lo / 4, off_lo, w + segs, w + 3 * segs};
    uint32_t *bits = reinterpret_cast<uint32_t *>(w + 4 * segs);
    unsigned *ticket = reinterpret_cast<unsigned *>(w + 6 * segs);
    int zst = launch_zero_u64(w + 6 * segs, 1, s);
    if (zst != HUFF_OK) return zst;
    const DevInfo d = dev_info();
    {
        size_t blocks = (segs + kSegScanThreads / 32 - 1) / (kSegScanThreads / 32);
        if (blocks > static_cast<size_t>(d.sms)) blocks = static_cast<size_t>(d.sms);  // one wave
        k_seg_bits_scan<<<static_cast<unsigned>(blocks), kSegScanThreads, 0, s>>>(seg_counts, static_cast<uint32_t>(segs), cb_hi, cb_lo,
                                                            bits, p0.desc, p1.desc, ticket, status);
        if (cudaGetLastError() != cudaSuccess) return HUFF_ERR_CUDA;
    }
    const uint8_t *a = reinterpret_cast<const uint8_t *>(w16);
    const uint8_t *b = reinterpret_cast<const uint8_t *>(x0);
    const size_t wtiles = (n + wenc::kTile - 1) / wenc::kTile;
    auto run = [&](auto kern) -> int {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(wenc::kSmem)) !=
            cudaSuccess)
            return HUFF_ERR_CUDA;
        // one CTA of 16 warps per SM; a warp takes whole segments, so fewer CTAs when there are few
        size_t grid = static_cast<size_t>(d.sms);
        if (grid > segs) grid = segs;
        kern<<<static_cast<unsigned>(grid), wenc::kThreads, wenc::kSmem, s>>>(
            a, b, n, p0, p1, make_chunk_div(chunk), static_cast<uint32_t>(wtiles), static_cast<uint32_t>(segs), status);
        return cudaGetLastError() == cudaSuccess ? HUFF_OK : HUFF_ERR_CUDA;
    };
    int st = x0 != nullptr ? run(k_encode_counted<true>) : run(k_encode_counted<false>);
    if (st != HUFF_OK) return st;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    k_encode_fixup<<<static_cast<unsigned>((segs + 127) / 128), 128, 0, s>>>(p0, p1, 2, static_cast<uint32_t>(segs),
                                                                            n_chunks, status);
    return launch_status();
}

}  // namespace huffk
