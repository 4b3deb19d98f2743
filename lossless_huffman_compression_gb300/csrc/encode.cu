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
// GPU design: one warp encodes a whole segment, with its own ring of 1-D
// bulk copies (cp.async.bulk on mbarriers) that stages the segment's tiles in
// shared memory, a conflict-free code table, and warp-level scans and packing
// (no block barrier on the path).  A segment's bit offset comes either from
// counts recorded before the encode (the counted bf16 encode: per-segment
// plane counts from the histogram pass give sum(count x length) and one scan
// over all segments) or from a decoupled lookback over the segments before it
// (the byte-stream encode, which counts a segment's bits in a first pass over
// its tiles and packs them in a second pass, from L2: Merrill & Garland,
// "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016).  The
// two partial words at each segment boundary are left in the workspace and
// written by a small fix-up kernel, so no warp ever waits for another warp's
// output.  All waits are bounded: a wait that runs out sets HUFF_ERR_TIMEOUT;
// a warp whose copy wait ran out issues no further copies, gives each copy it
// has in flight one more bounded wait, and stops.
#include "common.cuh"

namespace huffk {

// Workspace for huff_encode_noalloc, sized like huff_workspace_size for
// HUFF_NOALLOC_MAX_SYMBOLS symbols.  Every GPU that loads the library keeps
// these 2 MiB until the process exits; all calls share them.
// (2 MiB: twice the byte-stream encode's need at that size, 2 words per
// segment of 16 tiles of 1024 symbols plus the counter.)
constexpr size_t kNoAllocScratchWords = 2 * (HUFF_NOALLOC_MAX_SYMBOLS / 8192) + 2;
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocScratchWords];

namespace {

constexpr int kLookbackPerLane = 10;   // descriptors per lane per lookback step (window 320)

struct EncPlane {
    const huff_codebook *cb;
    uint32_t *payload;  // 32-bit words; payload byte 4w + j = bits 31-8j .. 24-8j of word w
    size_t cap_words;
    uint64_t *off;
    uint64_t *desc;     // per-segment lookback descriptors (zeroed before the launch)
    uint64_t *edge;     // per-segment boundary words: head bits << 32 | tail bits
};

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
// At most `limit` polls of an unpublished window (the spin count is left in
// `polls`); the wait also stops at a poll count divisible by 256 once any
// error is recorded, so one failure does not hold every later segment for
// the full limit.
__device__ uint64_t lookback(const uint64_t *desc, uint32_t t, int lane, int32_t *status,
                             uint64_t (&d)[kLookbackPerLane], unsigned limit, unsigned &polls) {
    unsigned spins = 0;
    polls = 0;
    if (t == 0) return 0;
    uint64_t excl = 0;
    int64_t base = static_cast<int64_t>(t) - 1;
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
            const bool give_up = spins > limit || ((spins & 255u) == 0 && error_recorded(status));
            if (__any_sync(0xffffffffu, give_up)) {
                if (lane == 0 && spins > limit) set_status(status, HUFF_ERR_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    }
    polls = spins;
    return excl;
}


// The chunk size, as the encode kernels take it (chunks are multiples of 32
// symbols, so a chunk starts at the first symbol of some lane's group: 16
// bf16 elements or 32 byte-stream symbols a lane).
struct ChunkDiv {
    uint32_t chunk;  // < 2^31
};

__host__ inline ChunkDiv make_chunk_div(size_t chunk) {
    return ChunkDiv{static_cast<uint32_t>(chunk)};
}

__device__ __forceinline__ void put_word(uint32_t *payload, size_t cap_words, uint64_t gw, uint32_t v,
                                         int32_t *status) {
    if (gw < cap_words)
        payload[gw] = bswap32(v);
    else
        set_status(status, HUFF_ERR_BUFFER_TOO_SMALL);
}

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
        if (lane == 0) {  // a segment has fewer than 512 * 512 * 24 bits per plane: 32-bit counts
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
constexpr int kWarps = 20;  // 5 per scheduler: 6.6 % faster than 16 (4 per scheduler, 3 stages) on the snapshot
constexpr int kThreads = 32 * kWarps;
constexpr int kLaneElems = 16;
constexpr int kTile = 32 * kLaneElems;                                 // 512 elements
constexpr uint32_t kMinSegTiles = static_cast<uint32_t>(kDirSegElems / kTile);  // 256
constexpr int kStages = 2;   // two suffice (3 measured the same), which is what makes room for 20 warps
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
// Returns whether a job was issued on the stage.
template <bool XOR>
__device__ __forceinline__ bool wissue(uint8_t *ring, uint64_t *bar, uint32_t stage, uint32_t seg, uint32_t kk,
                                       uint32_t tiles, uint32_t nw, uint32_t n_seg, uint32_t n_tiles,
                                       uint32_t seg_tiles, uint32_t last_bytes, const uint8_t *in,
                                       const uint8_t *in2, uint64_t pol) {
    if (kk >= tiles) {
        kk -= tiles;
        seg += nw;
        if (seg >= n_seg) return false;
        const uint32_t rest = n_tiles - seg * seg_tiles;
        if (kk >= (rest < seg_tiles ? rest : seg_tiles)) return false;
    }
    const uint32_t t = seg * seg_tiles + kk;
    const uint32_t bytes = t == n_tiles - 1 ? last_bytes : uint32_t(wenc::kTile * 2);  // every tile whole but the last
    const size_t src = static_cast<size_t>(t) * (wenc::kTile * 2);
    uint8_t *dst = ring + stage * wenc::kStageBytes;
    mbar_arrive_expect_tx(&bar[stage], bytes * (XOR ? 2u : 1u));
    if (bytes) {
        bulk_g2s_hint(dst, in + src, bytes, &bar[stage], pol);
        if (XOR) bulk_g2s_hint(dst + wenc::kTile * 2, in2 + src, bytes, &bar[stage], pol);
    }
    return true;
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
                     EncPlane p1, ChunkDiv cdiv, uint32_t n_tiles, uint32_t seg_tiles, uint32_t n_seg,
                     int32_t *status) {
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
    uint32_t inflight = 0;  // lane 0: stages with a job issued and not yet waited for
    if (lane == 0 && gw < n_seg) {  // the first kStages tiles of the warp's sequence
        const uint32_t rest = n_tiles - gw * seg_tiles;
        const uint32_t tiles0 = rest < seg_tiles ? rest : seg_tiles;
        for (int j = 0; j < wenc::kStages; ++j)
            if (wissue<XOR>(ring, bar, j, gw, j, tiles0, nw, n_seg, n_tiles, seg_tiles, last_bytes, in, in2, pol))
                inflight |= 1u << j;
    }
    const uint32_t kbh = static_cast<uint32_t>(lane & 15) << 3;
    const uint32_t kbl = kbh + 128u;
    uint32_t cstage = 0, cphase = 0;

    for (uint32_t r = 0;; ++r) {
        const uint32_t seg = r * nw + gw;
        if (seg >= n_seg) break;
        const uint32_t t0 = seg * seg_tiles;
        const uint32_t tiles = n_tiles - t0 < seg_tiles ? n_tiles - t0 : seg_tiles;
        // Bit positions inside the segment are 32-bit (a segment has fewer than 512 tiles, at most
        // 511 * 512 * 24 bits): pos =
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
            if (!__all_sync(0xffffffffu, mbar_wait(&bar[cstage], cphase))) {
                // the copy never arrived: no further copies; wait for those in flight, then stop
                if (lane == 0) set_status(status, HUFF_ERR_TIMEOUT);
                drain_ring(bar, wenc::kStages, __shfl_sync(0xffffffffu, inflight, 0), cstage, cphase);
                return;
            }
            inflight &= ~(1u << cstage);
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
            if (lane == 0 && wissue<XOR>(ring, bar, cstage, seg, k + wenc::kStages, tiles, nw, n_seg, n_tiles,
                                         seg_tiles, last_bytes, in, in2, pol))
                inflight |= 1u << cstage;
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

            // chunk starts in this tile (chunks are multiples of 32 elements, so a chunk starts
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
constexpr int kWarps = 24;  // 6 per scheduler: 6 to 13 % faster than 16 from 16 MiB to 1 GiB
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
static_assert(kSmem <= 227 * 1024, "one CTA per SM");
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
// Returns whether a job was issued on the stage.
__device__ __forceinline__ bool wissue8(uint8_t *ring, uint64_t *bar, uint32_t stage, Job8 &j, uint32_t &seg_next,
                                        uint32_t n_seg, uint32_t n_tiles, uint32_t st, uint32_t last_bytes,
                                        const uint8_t *in, uint64_t pol_keep, uint64_t pol_drop) {
    if (j.pass == 2) {
        j.seg = seg_next;
        j.pass = 0;
        j.k = 0;
        seg_next = 0xffffffffu;  // taken: the next claim replaces it
    }
    if (j.seg >= n_seg) return false;
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
    return true;
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
    uint32_t inflight = 0;  // lane 0: stages with a job issued and not yet waited for
    if (lane == 0)
        for (int s = 0; s < wenc8::kStages; ++s)
            if (wissue8(ring, bar, s, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep, pol_drop))
                inflight |= 1u << s;
    uint32_t cstage = 0, cphase = 0;

    auto next_stage = [&]() {
        cstage = cstage + 1 == uint32_t(wenc8::kStages) ? 0u : cstage + 1;
        cphase ^= cstage == 0 ? 1u : 0u;
    };
    // a lane's 32 bytes of the tile in the current stage (global memory for bytes past the bulk copy);
    // false when the stage's copy never arrived (the warp must then stop: see the callers)
    auto read_stage = [&](size_t first, int tile_n, uint32_t (&wv)[8]) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar[cstage], cphase))) {
            if (lane == 0) set_status(status, HUFF_ERR_TIMEOUT);
            drain_ring(bar, wenc8::kStages, __shfl_sync(0xffffffffu, inflight, 0), cstage, cphase);
            return false;
        }
        inflight &= ~(1u << cstage);
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
        return true;
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
            if (!read_stage(first, tile_n, wv)) return;
            if (lane == 0 && wissue8(ring, bar, cstage, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep,
                                     pol_drop))
                inflight |= 1u << cstage;
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
            unsigned polls;
            start = lookback(P.desc, seg, lane, status, wnd, kSpinLimit, polls);
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
            if (!read_stage(first, tile_n, wv)) return;
            if (lane == 0 && wissue8(ring, bar, cstage, job, job_next, n_seg, n_tiles, st, last_bytes, in, pol_keep,
                                     pol_drop))
                inflight |= 1u << cstage;
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

// The bounded waits on their own (huff_debug_wait): one warp runs the
// lookback of segment `seg` over desc[0 .. seg) (kind 0), or waits on an
// mbarrier that nothing arrives on and no copy targets (kind 1), with at most
// `limit` polls; out[0] = the lookback's exclusive prefix, out[1] = the polls
// made.
__global__ void k_wait_probe(int kind, const uint64_t *desc, uint32_t seg, unsigned limit, uint64_t *out,
                             int32_t *status) {
    __shared__ uint64_t bar;
    const int lane = threadIdx.x & 31;
    if (kind == 0) {
        uint64_t wnd[kLookbackPerLane];
        load_window(desc, static_cast<int64_t>(seg) - 1, lane, wnd);
        unsigned polls = 0;
        const uint64_t excl = lookback(desc, seg, lane, status, wnd, limit, polls);
        if (lane == 0) {
            out[0] = excl;
            out[1] = polls;
        }
        return;
    }
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    unsigned polls = 0;
    bool ok = false;
    while (!ok && polls < limit) {  // the same bounded wait, one poll per round, counted
        ok = mbar_wait(&bar, 0, 1);
        ++polls;
    }
    if (lane == 0) {
        if (!ok) set_status(status, HUFF_ERR_TIMEOUT);
        out[0] = 0;
        out[1] = polls;
    }
}

__global__ void k_encode_empty(uint64_t *off0, uint64_t *off1) {
    off0[0] = 0;
    if (off1) off1[0] = 0;
}

}  // namespace

int launch_wait_probe(int kind, const uint64_t *desc, uint32_t seg, unsigned limit, uint64_t *out, int32_t *status,
                      cudaStream_t s) {
    k_wait_probe<<<1, 32, 0, s>>>(kind, desc, seg, limit, out, status);
    return launch_status();
}

// Tiles per segment of the byte-stream encode: the fewest rounds of segments
// over the GPU's encode warps (one CTA of wenc8::kWarps per SM) that segments
// of at most 16 tiles allow, and then the fewest tiles per segment that keep
// to those rounds, so that the last round has (nearly) every warp busy; at
// least 4 tiles.  A 16 MiB input on 152 SMs: 5-tile segments in one round of
// 3277 of the 3648 warps; large inputs: 16.
size_t enc_u8_seg_tiles(size_t n) {
    const size_t tiles = (n + wenc8::kTile - 1) / wenc8::kTile;
    const size_t warps = static_cast<size_t>(dev_info().sms) * wenc8::kWarps;
    const size_t rounds = (tiles + size_t(wenc8::kSegTilesMax) * warps - 1) / (size_t(wenc8::kSegTilesMax) * warps);
    size_t st = rounds ? (tiles + rounds * warps - 1) / (rounds * warps) : 0;
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
    // one CTA of wenc8::kWarps warps per SM, fewer CTAs only when there are fewer segments than SMs: the
    // warps claim segments from the counter, so a small input spreads over as many SMs as it has segments
    // (the warps that claim none leave)
    const size_t sms = static_cast<size_t>(dev_info().sms);
    const size_t grid = segs < sms ? segs : sms;
    k_encode_u8w<<<static_cast<unsigned>(grid), wenc8::kThreads, wenc8::kSmem, s>>>(
        in, n, p0, static_cast<uint32_t>(chunk), static_cast<uint32_t>(tiles), static_cast<uint32_t>(seg_tiles),
        static_cast<uint32_t>(segs), ctr, status);
    if (cudaGetLastError() != cudaSuccess) return HUFF_ERR_CUDA;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    k_encode_fixup<<<static_cast<unsigned>((segs + 255) / 256), 256, 0, s>>>(p0, p0, 1, static_cast<uint32_t>(segs),
                                                                              n_chunks, status);
    return launch_status();
}

// Device address of g_noalloc_scratch on the current device (host code only
// sees a host-side stand-in under the array's name).  Looked up on every call:
// the query allocates nothing, and a cached address would go stale when the
// device's context is torn down and made again (cudaDeviceReset).
static uint64_t *noalloc_scratch_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return static_cast<uint64_t *>(p);
}

int launch_encode_u8_noalloc(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk, uint8_t *payload,
                             size_t cap, uint64_t *off, int32_t *status, cudaStream_t s) {
    if (enc_u8_workspace_words(n) > kNoAllocScratchWords) return HUFF_ERR_BUFFER_TOO_SMALL;
    uint64_t *ws = noalloc_scratch_address();
    if (ws == nullptr) return HUFF_ERR_CUDA;
    // the same path as huff_encode; it zeroes what must start at zero before the encode kernel runs
    return launch_encode_u8(in, n, cb, chunk, payload, cap, off, ws, status, s);
}

// Elements per counted segment for n elements: kDirSegElems (256 tiles) while the counted encode's warps
// (one CTA of wenc::kWarps per SM) outnumber such segments; otherwise the whole number of tiles (at least 256,
// fewer than 512) that gives every warp the same number of segments, so that no warp's last segment
// runs while most of its SM's warps are done.
size_t count_seg_elems(size_t n) {
    const size_t tiles = (n + wenc::kTile - 1) / wenc::kTile;
    const size_t warps = static_cast<size_t>(dev_info().sms) * wenc::kWarps;
    const size_t rounds = tiles / (static_cast<size_t>(wenc::kMinSegTiles) * warps);
    if (rounds == 0) return kDirSegElems;
    const size_t st = (tiles + warps * rounds - 1) / (warps * rounds);
    return st * wenc::kTile;
}

// bf16 with given codebooks (the fixed-codebook mode): the counted histogram pass records both planes'
// counts per segment, and the one-pass counted encode then gives every segment its bit offset from
// sum(count x length) under the given codebooks (a symbol present without a code is reported by that
// sum).  The input is read twice from HBM (it is larger than L2), by two kernels that each run near
// their own bound.  Workspace (lmc_workspace_size): segment counts, the counted encode's workspace,
// then the two histograms the counting pass also produces.
size_t enc_bf16_given_ws_parts(size_t n, size_t *counted_off, size_t *hist_off) {
    const size_t segs = (n + kDirSegElems - 1) / kDirSegElems;
    const size_t counts = (static_cast<size_t>(kSegCountWords) * 4 * segs + 255) / 256 * 256;
    const size_t counted = (48 * segs + 16 + 255) / 256 * 256;
    if (counted_off) *counted_off = counts;
    if (hist_off) *hist_off = counts + counted;
    return counts + counted + 512 * sizeof(uint64_t);
}

int launch_encode_bf16(const uint16_t *w16, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                       const huff_codebook *cb_lo, size_t chunk, uint8_t *pay_hi, size_t cap_hi, uint64_t *off_hi,
                       uint8_t *pay_lo, size_t cap_lo, uint64_t *off_lo, void *ws, int32_t *status,
                       cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off_hi, off_lo);
        return launch_status();
    }
    size_t counted_off = 0, hist_off = 0;
    enc_bf16_given_ws_parts(n, &counted_off, &hist_off);
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *seg_counts = reinterpret_cast<uint32_t *>(w);
    uint64_t *hist = reinterpret_cast<uint64_t *>(w + hist_off);
    int st = launch_zero_u64(hist, 512, s);
    if (st != HUFF_OK) return st;
    st = launch_histogram_bf16_counted(w16, x0, n, hist, hist + 256, seg_counts, s);
    if (st != HUFF_OK) return st;
    return launch_encode_bf16_counted(w16, x0, n, cb_hi, cb_lo, chunk, seg_counts, pay_hi, cap_hi, off_hi, pay_lo,
                                      cap_lo, off_lo, w + counted_off, status, s);
}

int launch_encode_bf16_counted(const uint16_t *w16, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                               const huff_codebook *cb_lo, size_t chunk, const uint32_t *seg_counts,
                               uint8_t *pay_hi, size_t cap_hi, uint64_t *off_hi, uint8_t *pay_lo, size_t cap_lo,
                               uint64_t *off_lo, void *ws, int32_t *status, cudaStream_t s) {
    if (n == 0) {
        k_encode_empty<<<1, 1, 0, s>>>(off_hi, off_lo);
        return launch_status();
    }
    const size_t seg_elems = count_seg_elems(n);
    const size_t segs = (n + seg_elems - 1) / seg_elems;  // at most ceil(n / kDirSegElems): the workspace's size
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
        // one CTA of wenc::kWarps warps per SM; a warp takes whole segments, so fewer CTAs when there are few
        size_t grid = static_cast<size_t>(d.sms);
        if (grid > segs) grid = segs;
        kern<<<static_cast<unsigned>(grid), wenc::kThreads, wenc::kSmem, s>>>(
            a, b, n, p0, p1, make_chunk_div(chunk), static_cast<uint32_t>(wtiles),
            static_cast<uint32_t>(seg_elems / wenc::kTile), static_cast<uint32_t>(segs), status);
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
