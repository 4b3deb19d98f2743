// decode.cu -- chunked Huffman decode.
//
// "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
// 2505.09810), technical framework: decompression reads the data,
// Huffman-decodes it and restores the byte groups; key design 3: the work is
// split into tasks that run in parallel.  The chunk bit offsets written by the
// encoder are those tasks' entry points.
//
// GPU design:
//   * one lane per chunk (per chunk pair for bf16), every lane of the grid
//     resident at once; the block size follows the chunk count.  With fewer
//     than 768 chunks per SM, byte streams instead give each chunk a team of
//     1 to 28 warps whose threads take slices of its bits and find their
//     code boundaries by self-synchronisation (the section on fewer chunks
//     below).  With at most 448 lanes per SM the fused bf16 decode steps
//     both planes of a lane in one loop;
//   * shared tables per plane: a window table of 2^W 64-bit entries (W = 12
//     for the high plane, 13 for the low plane and byte streams), each
//     listing the codes wholly inside the next W bits (up to six symbols,
//     their count and total length), a secondary table for longer codes and
//     the canonical arrays for when that table would not fit (byte streams
//     count the length limits a window reaches; the bf16 planes search);
//   * the bit reader keeps 64 bits in two registers and refills 32 at a time
//     from a queue of the current 16-byte unit of the stream; units are read
//     whole, the payload's last unit standing in for any unit past it;
//   * a step is one predicated basic block: a table lookup plus a second,
//     dependent one when both fit 8 symbols, then (bf16 planes) a third on
//     the bits after them when its codes lie within the buffer's valid bits
//     (its symbols emitted as a second round of the pending-word logic; up
//     to 14 symbols a step), or, on a plane with a 1-bit code, a run of that code as long
//     as the zero bits on top of the window (up to 32); on a plane without
//     one, while every lane of the warp has room for a full step in its
//     chunk and its ring, steps run without the per-step checks;
//   * the fused bf16 decode of a high plane with a 1-bit code (a snapshot
//     delta's, about 98 % one symbol) takes at most one other code per step
//     and then the whole run of the 1-bit code after it, into a ring that
//     already holds that code's symbol (no stores for runs); it has its own
//     kernel, which also stages x0 in shared memory a segment ahead;
//   * decoded bytes go to per-lane shared rings in segments; the warp steps
//     until every lane has its segment (a lane that is ahead decodes into
//     the ring's free part), then merges 8 lanes' segments per pass into
//     16-bit words, XORs x0 (staged, or prefetched to L2 before the segments'
//     decode with a merge's four loads issued together) and stores 16 bytes
//     per lane; while every chunk of the warp has the same length (all warps
//     but the last one of a ragged input), the merge skips the per-lane
//     bounds.
// Every chunk must end exactly at the next chunk's offset, otherwise
// HUFF_ERR_CORRUPT_STREAM is reported.
#include <algorithm>
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kSecMax = 2048;  // secondary-table entries per plane

// Shared decode tables of one codebook for a W-bit window (W = 12: the
// codebook's own table; W = 13: built from it in the prologue).  16-byte
// aligned and sized, so tables placed back to back stay aligned.
// The W-bit table: one 64-bit entry per window (syms (48 bits) | count << 48 | total bits << 52; 0: the
// first code is longer than W bits), or, split (SPLIT), at most 4 symbols per window in a 32-bit word
// (first symbol in the low byte) and count | total bits << 3 in a byte: 5 bytes per window instead of 8.
template <int W, bool SPLIT>
struct LutStore {
    uint64_t lut[1u << W];
};
template <int W>
struct LutStore<W, true> {
    uint32_t syms[1u << W];
    uint8_t meta[1u << W];
};
constexpr int kSplitSyms = 4;  // symbols a split entry holds

template <int W, int SEC = kSecMax, bool SPLIT = false>
struct __align__(16) DecTables : LutStore<W, SPLIT> {
    uint16_t sec[SEC];      // codes longer than W bits: symbol | length << 8 (0: no code)
    uint64_t run;           // the 1-bit code's symbol in all 8 bytes (when there is one)
    uint32_t bl_count[32];
    uint32_t first_code[32];
    uint32_t first_index[32];
    uint32_t lim[32];       // 24-bit windows below lim[l] start with a code of at most l bits (all ones past the longest)
    uint8_t sorted[256];
    uint8_t len[256];
    int longest;
    int ok;
    int has_run;    // a 1-bit code exists: 8 leading zero bits are 8 of its symbol
    int sec_k;      // bits after the W-bit window that index sec (0: no code is longer than W bits)
    int sec_first;  // first W-bit prefix of the long codes (they fill the top of the code space)
    int sec_ok;     // sec holds every long code; otherwise the canonical search decodes them
};
static_assert(sizeof(DecTables<12>) % 16 == 0 && sizeof(DecTables<13, kSecMax, true>) % 16 == 0,
              "tables keep 16-byte alignment");

// Entry i of the W-bit table: its symbols (first in the low byte, the rest zero), their count and total
// bits.
template <int W, int SEC, bool SPLIT>
__device__ __forceinline__ void lut_get(const DecTables<W, SEC, SPLIT> &T, uint32_t i, uint64_t &v, uint32_t &c,
                                        uint32_t &bits) {
    if constexpr (SPLIT) {
        const uint32_t m = T.meta[i];
        v = T.syms[i];
        c = m & 7u;
        bits = m >> 3;
    } else {
        const uint64_t e = T.lut[i];
        const uint32_t eh = static_cast<uint32_t>(e >> 32);
        c = (eh >> 16) & 15u;
        bits = eh >> 20;
        v = e & 0xffffffffffffull;
    }
}

// Tables of a plane with a 1-bit code, for the run decode below: the
// canonical arrays and, for each 10-bit window, the first code's symbol and
// length (symbol | length << 8; 0 when that code is longer than 10 bits,
// which the canonical search then decodes).
constexpr int kZWin = 10;
struct __align__(16) RunTables {
    uint64_t run;  // the 1-bit code's symbol in all 8 bytes
    uint32_t bl_count[32];
    uint32_t first_code[32];
    uint32_t first_index[32];
    uint8_t sorted[256];
    int longest;
    int ok;
    uint16_t zf[1u << kZWin];
};

// The low plane next to a run-decoded high plane: a split 13-bit table (at
// most 4 symbols per window, which changes the symbols a three-lookup step
// takes by less than 0.1 % on a snapshot delta's low plane) and a smaller
// secondary table, so that the rings and the x0 staging of 896 lanes fit next
// to them (7 warps on each of the SM's 4 schedulers).
constexpr int kSecRun = 1024;
using LoTables = DecTables<13, kSecMax, true>;  // the low plane beside a table-decoded high plane: split too
using LoTablesRun = DecTables<13, kSecRun, true>;
static_assert(sizeof(RunTables) % 16 == 0 && sizeof(LoTablesRun) % 16 == 0, "tables keep 16-byte alignment");
constexpr size_t kBf16Tables = sizeof(DecTables<12>) + sizeof(LoTables);
constexpr size_t kBf16RunTables = sizeof(RunTables) + sizeof(LoTablesRun);

// Canonical codes fill the code space in order of length, so the codes of at
// most l bits are the 24-bit windows below (first_code[l] + bl_count[l]) <<
// (24 - l), and a window's code length is one more than the number of lengths
// whose limit it reaches.  All ones past the longest code.
__device__ __forceinline__ uint32_t code_limit(const huff_codebook *cb, bool ok, int l) {
    if (!ok || l > cb->longest) return 0xffffffffu;
    if (l == 0) return 0;
    return (cb->first_code[l] + cb->bl_count[l]) << (HUFF_MAX_LEN - l);
}

// Phase 1 of loading a codebook: the W-bit table, the canonical arrays and
// the header.  For W = 13 an entry is the 12-bit entry of its first 12 bits
// plus, when it holds fewer than the maximum number of symbols, the one code
// that ends exactly at the 13th bit (a code ending earlier would already be
// in the 12-bit entry, and no code is shorter than 1 bit).
template <int W, int SEC, bool SPLIT>
__device__ void load_table_a(DecTables<W, SEC, SPLIT> &T, const huff_codebook *cb) {
    static_assert(W == HUFF_LUT_BITS || W == HUFF_LUT_BITS + 1, "12- or 13-bit window");
    static_assert(!SPLIT || W == HUFF_LUT_BITS + 1, "split tables have 13-bit windows");
    const int tid = threadIdx.x;
    const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC;
    if constexpr (W == HUFF_LUT_BITS && !SPLIT) {
        const uint4 *src = reinterpret_cast<const uint4 *>(cb->lut);
        uint4 *dst = reinterpret_cast<uint4 *>(T.lut);
        for (int i = tid; i < (1 << W) / 2; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
    } else {
        for (int i = tid; i < (1 << W); i += blockDim.x) {
            uint64_t e = 0;
            if (ok) {
                e = cb->lut[i >> 1];
                const uint32_t c = static_cast<uint32_t>(e >> 48) & 15u;
                const uint32_t bits = static_cast<uint32_t>(e >> 52) & 15u;
                if (c < HUFF_LUT_SYMS) {
                    const uint32_t r = static_cast<uint32_t>(W) - bits;  // 1..W
                    const uint32_t v = static_cast<uint32_t>(i) & ((1u << r) - 1u);
                    const uint32_t nc = cb->bl_count[r];
                    const uint32_t d = v - cb->first_code[r];
                    if (nc != 0 && d < nc) {
                        const uint64_t sym = cb->sorted_symbols[cb->first_index[r] + d];
                        e = (e & 0xffffffffffffull) | (sym << (8 * c)) | (static_cast<uint64_t>(c + 1) << 48) |
                            (static_cast<uint64_t>(W) << 52);
                    }
                }
            }
            if constexpr (SPLIT) {
                // the first kSplitSyms symbols and their bits
                uint32_t c = static_cast<uint32_t>(e >> 48) & 15u;
                uint32_t bits = static_cast<uint32_t>(e >> 52) & 15u;
                if (c > static_cast<uint32_t>(kSplitSyms)) {
                    c = kSplitSyms;
                    bits = 0;
                    for (int k = 0; k < kSplitSyms; ++k) bits += cb->len[(e >> (8 * k)) & 0xffu];
                }
                T.syms[i] = static_cast<uint32_t>(e);
                T.meta[i] = static_cast<uint8_t>(c | (bits << 3));
            } else {
                T.lut[i] = e;
            }
        }
    }
    uint4 *sz = reinterpret_cast<uint4 *>(T.sec);
    for (int i = tid; i < SEC / 8; i += blockDim.x) sz[i] = make_uint4(0, 0, 0, 0);
    if (tid < 32) {
        T.bl_count[tid] = ok ? cb->bl_count[tid] : 0;
        T.first_code[tid] = ok ? cb->first_code[tid] : 0;
        T.first_index[tid] = ok ? cb->first_index[tid] : 0;
        T.lim[tid] = code_limit(cb, ok, tid);
    }
    for (int i = tid; i < 256; i += blockDim.x) {
        T.sorted[i] = ok ? cb->sorted_symbols[i] : 0;
        T.len[i] = ok ? cb->len[i] : 0;
    }
    if (tid == 0) {
        const int longest = ok ? cb->longest : 0;
        T.longest = longest;
        T.ok = ok && longest <= HUFF_MAX_LEN;
        T.has_run = ok && cb->bl_count[1] > 0;
        T.run = (ok ? static_cast<uint64_t>(cb->sorted_symbols[0]) : 0ull) * 0x0101010101010101ull;
        const int k = longest > W ? longest - W : 0;
        const int first = k ? static_cast<int>(cb->first_code[W + 1] >> 1) : (1 << W);
        T.sec_k = k;
        T.sec_first = first;
        T.sec_ok = k == 0 || (first <= (1 << W) && (static_cast<long long>((1 << W) - first) << k) <= SEC);
    }
}

// Phase 2 (after a barrier): the secondary table for codes longer than the
// window.  Canonical codes place every code longer than W bits after all
// shorter ones, so their W-bit prefixes are the contiguous range
// [first_code[W + 1] / 2, 2^W); sec holds, per prefix, 2^k entries
// (k = longest - W) indexed by the next k bits.
template <int W, int SEC, bool SPLIT>
__device__ void load_table_b(DecTables<W, SEC, SPLIT> &T, const huff_codebook *cb) {
    if (!T.ok || T.sec_k == 0 || !T.sec_ok) return;
    const int k = T.sec_k;
    for (int sym = threadIdx.x; sym < 256; sym += blockDim.x) {
        const int L = T.len[sym];
        if (L <= W) continue;
        const uint32_t base = (cb->code[sym] << (W + k - L)) - (static_cast<uint32_t>(T.sec_first) << k);
        const uint16_t ent = static_cast<uint16_t>(sym | (L << 8));
        for (uint32_t j = 0; j < (1u << (W + k - L)); ++j) T.sec[base + j] = ent;
    }
}

// Bit reader: 64 upcoming bits in (bh, bl), most significant first, and the
// words of the current 16-byte unit of the stream not taken yet (a queue: the
// next word is always cur.x).  The payload pointer and size are passed to
// every call that may load, so they stay kernel parameters rather than
// registers.
//
// Unit u of the payload, read whole; past the last unit that holds a payload
// byte, that last unit again.  The payload is 16-byte aligned, so a unit that
// holds one of its bytes lies in pages it occupies: every read is of mapped
// memory, with no bounds branch.  Bytes past the payload's end (in its last
// unit, or a repeated unit) only ever enter a lookup window beyond the end
// of a valid stream, where the symbol count clamps every entry and no
// decoded symbol depends on them.  Only lanes that decode load (nbytes >= 1:
// a chunk of cnt symbols holds at least cnt bits).
__device__ __forceinline__ uint4 load_unit(const uint8_t *p, size_t nbytes, size_t u) {
    const size_t last = (nbytes - 1) >> 4;
    const uint8_t *a = p + (u < last ? u : last) * 16;
    // a lane reads its chunk 16 bytes at a time over the whole kernel while x0 and the output stream
    // past: keep the payload's lines in L2 ahead of them (x0 and out are evict-first)
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(a), "l"(pol));
    return v;
}

// Canonical search for a code longer than the table's W bits: returns
// (length << 8) | symbol, length 0 if no code matches.
// The window's code length counted against the limits (no loop-carried
// search), then its symbol from the canonical arrays.  The caller knows the
// first code is longer than W bits.
template <int W, class Tab>
__device__ __forceinline__ uint32_t long_code_lim(uint32_t top, const Tab &T, int longest) {
    const uint32_t v = top >> (32 - HUFF_MAX_LEN);
    uint32_t L = W + 1;
#pragma unroll
    for (int l = W + 1; l < HUFF_MAX_LEN; ++l) L += v >= T.lim[l] ? 1u : 0u;
    const uint32_t d = (v >> (HUFF_MAX_LEN - L)) - T.first_code[L];
    if (L > static_cast<uint32_t>(longest) || d >= T.bl_count[L]) return 0;
    return (L << 8) | T.sorted[T.first_index[L] + d];
}

template <int W, int SEC, bool SPLIT>
__device__ __noinline__ uint32_t long_code(uint32_t top, const DecTables<W, SEC, SPLIT> *T) {
    return long_code_lim<W>(top, *T, T->longest);
}

// The same by a search over the lengths.  The fused bf16 decode uses this one:
// its planes rarely have codes past the window, and the counting form
// measured 1.2 % slower there (a different register allocation around the
// call); the byte-stream decodes, whose fixed codebooks often meet data they
// were not built for (codes of 17 to 24 bits), use the count.
template <int W, class Tab>
__device__ __noinline__ uint32_t long_code_search(uint32_t top, const Tab *T) {
    const uint32_t v = top >> (32 - HUFF_MAX_LEN);
    for (int l = W + 1; l <= T->longest; ++l) {
        const uint32_t c = v >> (HUFF_MAX_LEN - l);
        const uint32_t d = c - T->first_code[l];
        if (d < T->bl_count[l]) return (static_cast<uint32_t>(l) << 8) | T->sorted[T->first_index[l] + d];
    }
    return 0;
}

// The rare case where a table entry holds more symbols than the chunk has
// left: the total length of its first c symbols.
template <int W, int SEC, bool SPLIT>
__device__ __noinline__ uint32_t clamped_bits(uint64_t v, uint32_t c, const DecTables<W, SEC, SPLIT> *T) {
    uint32_t bits = 0;
    for (uint32_t k = 0; k < c; ++k) bits += T->len[(v >> (8 * k)) & 0xffu];
    return bits;
}

// ------------------------------------------------------------------ per-lane plane decoder
//
// A lane decodes one chunk of one byte plane into a private ring of RING
// bytes in shared memory.  The warp works in segments of kSeg symbols per
// lane: it keeps stepping until every lane has stored its segment, and a lane
// that is ahead keeps decoding into the ring's free slots instead of idling,
// so the lanes' varying symbols-per-lookup cost little SIMT efficiency.  Then
// the warp copies the segment out cooperatively, so global stores are whole
// sectors.  A step is one straight-line table lookup; only codes longer than
// the 12-bit window (one secondary-table load) and a chunk's last symbols
// leave it.
constexpr int kSeg = 32;       // symbols per lane per segment (multiple of 16)
constexpr int kRing = 64;      // ring bytes per lane per plane (power of two)
constexpr int kStepMax = 8;    // symbols a table step may add (a run step: up to 32, within the ring's room)
constexpr int kFastSteps = 2;  // steps per unchecked block on a plane without runs
constexpr int kStepMax3 = 14;  // symbols a three-lookup step may add (8 from the first two, 6 from the third)
static_assert(kRing >= kSeg + kFastSteps * kStepMax3, "a lane at its segment's start has room for a fast block");
constexpr int kMaxBlock = 896;   // 72 registers per thread; 152 SMs x 896 lanes cover 16 KiB chunks of 2e9 elements in one wave
constexpr int kPairBlock = 448;  // at most this many lanes per SM: the fused bf16 decode steps both planes in one loop
static_assert(kRing >= kSeg + 7 + 2 * kStepMax && (kRing & (kRing - 1)) == 0 && kSeg % 16 == 0, "ring geometry");
static_assert(HUFF_LUT_SYMS <= kStepMax, "a table entry must fit one step");

struct PlaneDec {
    uint32_t bh, bl;  // upcoming bits, most significant first
    int nb;           // valid bits in (bh, bl); >= 33 after a refill
    int qi;           // words of the current unit taken so far
    uint4 cur;        // the current unit's words not taken yet, from cur.x on (raw little-endian)
    size_t ui;        // index of the unit after cur
    uint64_t a0;      // pending decoded bytes: byte k of the stream order is byte k of a0
    int fill;         // pending symbols, < 8 between steps (< 4 on a plane stepped with three lookups)
    int st;           // symbols stored to the ring (a multiple of 8, or of 4 with three lookups, until
                      // the chunk is complete)

    __device__ __forceinline__ void refill(const uint8_t *p, size_t nbytes) {
        const bool rf = nb <= 32;
        // cur.x is always the next word; a refill moves the queue down one word
        const uint32_t w = rf ? bswap32(cur.x) : 0u;
        bh |= __funnelshift_rc(w, 0u, static_cast<uint32_t>(nb));       // w >> nb (0 when nb >= 32)
        bl |= __funnelshift_lc(0u, w, static_cast<uint32_t>(32 - nb));  // w << (32 - nb)
        nb += rf ? 32 : 0;
        if (rf) {
            cur.x = cur.y;
            cur.y = cur.z;
            cur.z = cur.w;
        }
        qi += rf ? 1 : 0;
        if (qi == 4) {
            cur = load_unit(p, nbytes, ui++);
            qi = 0;
        }
    }
    __device__ __forceinline__ void consume(uint32_t bits) {  // bits <= 32
        bh = __funnelshift_lc(bl, bh, bits);
        bl = __funnelshift_lc(0u, bl, bits);
        nb -= static_cast<int>(bits);
    }
    __device__ __forceinline__ void start(const uint8_t *p, size_t nbytes, uint64_t pos) {
        const size_t u = pos >> 7;
        cur = load_unit(p, nbytes, u);
        ui = u + 1;
        qi = static_cast<int>((pos >> 5) & 3u);
        for (int k = 0; k < qi; ++k) {  // words of the unit before the start
            cur.x = cur.y;
            cur.y = cur.z;
            cur.z = cur.w;
        }
        bh = bl = 0;
        nb = 0;
        refill(p, nbytes);
        refill(p, nbytes);
        consume(static_cast<uint32_t>(pos & 31u));
    }
    // bits consumed from the start of the payload
    __device__ __forceinline__ uint64_t pos() const {
        return 32 * (static_cast<uint64_t>(ui - 1) * 4 + static_cast<uint64_t>(qi)) - static_cast<uint64_t>(nb);
    }
};

// The rare cases of a step: a code longer than the table's window (or no
// code at all: a corrupt stream), and an entry with more symbols than the
// chunk has left.
template <int W, bool LIM, int SEC, bool SPLIT>
__device__ __forceinline__ void step_rare(const DecTables<W, SEC, SPLIT> &T, uint32_t win, uint32_t top, int rem, uint32_t &c,
                                       uint32_t &bits, uint64_t &v, bool &bad) {
    if (c == 0) {
        uint32_t L = 0, sym = 0;
        if (T.sec_ok) {
            if (T.sec_k > 0 && static_cast<int>(win) >= T.sec_first) {
                const int k = T.sec_k;
                const uint32_t idx = ((win - static_cast<uint32_t>(T.sec_first)) << k) |
                                     ((top >> (32 - W - k)) & ((1u << k) - 1u));
                const uint32_t e2 = T.sec[idx];
                L = e2 >> 8;
                sym = e2 & 0xffu;
            }
        } else {
            const uint32_t lc = LIM ? long_code(top, &T) : long_code_search<W>(top, &T);
            L = lc >> 8;
            sym = lc & 0xffu;
        }
        if (L == 0) {
            bad = true;
            L = 1;
        }
        c = 1;
        bits = L;
        v = sym;
    }
    if (static_cast<int>(c) > rem) {
        c = static_cast<uint32_t>(rem);
        bits = clamped_bits(v, c, &T);
        v &= (1ull << (8 * c)) - 1ull;
    }
}

// Append c symbols (v's low c bytes, the rest zero) to the pending bytes of a
// plane whose pending part is at most 3 bytes (the low word of a0), storing
// every completed 4-byte word: only 32-bit shifts.
template <int RING>
__device__ __forceinline__ void put4(PlaneDec &s, uint8_t *ring, uint32_t swz, uint64_t v, uint32_t c) {
    const uint32_t sh = 8u * static_cast<uint32_t>(s.fill);  // fill <= 3
    const uint32_t vl = static_cast<uint32_t>(v), vh = static_cast<uint32_t>(v >> 32);
    const uint32_t w0 = static_cast<uint32_t>(s.a0) | (vl << sh);
    const uint32_t w1 = __funnelshift_l(vl, vh, sh);
    const uint32_t w2 = __funnelshift_l(vh, 0u, sh);
    const int nf = s.fill + static_cast<int>(c);
    if (nf >= 4) *reinterpret_cast<uint32_t *>(ring + ((s.st & (RING - 1)) ^ swz)) = w0;
    if (nf >= 8) *reinterpret_cast<uint32_t *>(ring + (((s.st + 4) & (RING - 1)) ^ swz)) = w1;
    s.a0 = nf >= 8 ? w2 : (nf >= 4 ? w1 : w0);
    s.st += nf & ~3;
    s.fill = nf & 3;
}

// One step: if the chunk has symbols left and the ring has room, one table
// lookup, or, for a plane with a 1-bit code, a run of that code as long as
// the zero bits on top of the window (up to 32, the chunk's rest and the
// ring's room) when that beats a lookup; then up to four 8-byte stores.
// `limit` = the first symbol position whose slot still holds unmerged data.
template <int RING, bool RUN, int W, bool LIM, bool FAST = false, bool THIRD = false, int SEC = kSecMax, bool SPLIT = false>
__device__ __forceinline__ void step(PlaneDec &s, const uint8_t *p, size_t nbytes, const DecTables<W, SEC, SPLIT> &T,
                                     uint8_t *ring, uint32_t swz, int cnt, int limit, uint64_t run, bool &bad) {
    static_assert(!(RUN && THIRD), "a third lookup is for planes without runs");
    static_assert(!(RUN && FAST), "a run step may add more symbols than a fast block reserves");
    // Predicated rather than branched: a lane with nothing to do (its chunk
    // is complete or its ring is full) takes a step of zero bits and zero
    // symbols, so the step stays one basic block.
    // FAST: the caller has checked that the chunk and the ring have room for this step
    const int rem = FAST ? (1 << 20) : cnt - s.st - s.fill;
    const int room = FAST ? (1 << 20) : limit - s.st - s.fill;
    const bool go = FAST || (rem > 0 && room >= (THIRD ? kStepMax3 : kStepMax));
    s.refill(p, nbytes);
    const uint32_t win = s.bh >> (32 - W);
    uint32_t c, bits;
    uint64_t v;
    lut_get(T, win, v, c, bits);
    bool is_run = false;
    if (RUN) {
        // the 1-bit code is all zeros: clz(bh) symbols of it are next (bh holds >= 33 valid bits)
        const int cr = min(min(static_cast<int>(__clz(s.bh)), rem), room);
        // at least 8 (more than a lookup gives), so a run always completes the pending word and the
        // first stored word takes run bytes in every position the pending bytes leave
        is_run = cr >= kStepMax;
        c = is_run ? static_cast<uint32_t>(cr) : c;
        bits = is_run ? static_cast<uint32_t>(cr) : bits;
        v = is_run ? run : v;
    }
    const bool simple = c != 0 && static_cast<int>(c) <= rem;
    if (go && !simple) step_rare<W, LIM>(T, win, s.bh, rem, c, bits, v, bad);
    if (!RUN) {
        // a second, dependent lookup on the bits after the first entry, taken when the first entry was
        // simple (at least 20 valid bits remain) and the two entries together are at most 8 symbols
        // within the chunk; otherwise those bits wait for the next step
        const uint32_t top2 = __funnelshift_l(s.bl, s.bh, bits);
        uint32_t c2, b2;
        uint64_t v2;
        lut_get(T, top2 >> (32 - W), v2, c2, b2);
        const bool take2 = simple && c2 != 0 && c + c2 <= static_cast<uint32_t>(kStepMax) &&
                           static_cast<int>(c + c2) <= rem;
        v |= take2 ? v2 << (8 * c) : 0ull;
        bits += take2 ? b2 : 0u;
        c += take2 ? c2 : 0u;
    }
    c = go ? c : 0u;
    bits = go ? bits : 0u;
    v = go ? v : 0ull;
    s.consume(bits);
    if constexpr (THIRD) {
        // pending bytes kept below a word, so both rounds' appends use 32-bit shifts only; then a third
        // lookup on the bits after the first two entries, taken when the step went the simple way and
        // its codes lie within the valid bits and the chunk, appended as a second round
        put4<RING>(s, ring, swz, v, c);
        uint32_t c3, b3;
        uint64_t v3;
        lut_get(T, s.bh >> (32 - W), v3, c3, b3);
        const bool take3 = go && simple && c3 != 0 && static_cast<int>(b3) <= s.nb &&
                           static_cast<int>(c + c3) <= rem;
        s.consume(take3 ? b3 : 0u);
        put4<RING>(s, ring, swz, take3 ? v3 : 0ull, take3 ? c3 : 0u);
        return;
    }
    const int f = s.fill;
    const uint64_t a = s.a0 | (v << (8 * f));
    const int nf = f + static_cast<int>(c);
    const bool full = nf >= 8;
    if (full) *reinterpret_cast<uint64_t *>(ring + ((s.st & (RING - 1)) ^ swz)) = a;
    if (RUN) {
        if (nf >= 16) *reinterpret_cast<uint64_t *>(ring + (((s.st + 8) & (RING - 1)) ^ swz)) = run;
        if (nf >= 24) *reinterpret_cast<uint64_t *>(ring + (((s.st + 16) & (RING - 1)) ^ swz)) = run;
        if (nf >= 32) *reinterpret_cast<uint64_t *>(ring + (((s.st + 24) & (RING - 1)) ^ swz)) = run;
    }
    // the bytes that did not fit: a lookup's last nf - 8 bytes, or nf % 8 run bytes
    const int keep = (RUN && is_run) ? 8 * (nf & 7) : 8 * f;
    s.a0 = full ? (v >> 1) >> (63 - keep) : a;
    s.st += nf & ~7;
    s.fill = nf & 7;
}

__device__ __forceinline__ void plane_start(PlaneDec &s, const uint8_t *pay, size_t nbytes, uint64_t start, int cnt) {
    if (cnt > 0) {
        s.start(pay, nbytes, start);
    } else {  // no chunk: 64 valid bits, so the reader never refills and never loads
        s.bh = s.bl = 0;
        s.nb = 64;
        s.qi = 0;
        s.cur = make_uint4(0, 0, 0, 0);
        s.ui = 0;
    }
    s.a0 = 0;
    s.fill = 0;
    s.st = 0;
}

// Decode until every lane of the warp has stored symbols [.., need) into its
// RING-byte ring (a lane whose chunk is complete stores its last partial word).
template <int RING, bool RUN, int W, bool LIM, int SEC, bool THIRD = false, bool SPLIT = false>
__device__ __forceinline__ void fill_segment_t(PlaneDec &s, const uint8_t *p, size_t nbytes, const DecTables<W, SEC, SPLIT> &T,
                                               uint8_t *ring, uint32_t swz, int cnt, int need, int limit,
                                               bool &bad) {
    const uint64_t run = RUN ? T.run : 0ull;
    if (!RUN) {
        // while every lane's chunk and ring have room for kFastSteps unchecked steps (a table step adds
        // at most kStepMax symbols, a three-lookup step kStepMax3), take them without the per-step checks
        constexpr int kFast = kFastSteps;
        constexpr int kNeed = THIRD ? kFastSteps * kStepMax3 : kFastSteps * kStepMax;
        while (__all_sync(0xffffffffu, limit - s.st - s.fill >= kNeed && cnt - s.st - s.fill >= kNeed) &&
               __any_sync(0xffffffffu, s.st < need)) {
#pragma unroll
            for (int k = 0; k < kFast; ++k)
                step<RING, false, W, LIM, true, THIRD, SEC, SPLIT>(s, p, nbytes, T, ring, swz, cnt, limit, run, bad);
        }
    }
    while (__any_sync(0xffffffffu, s.st < need && s.st + s.fill != cnt))
        step<RING, RUN, W, LIM, false, THIRD && !RUN, SEC, SPLIT>(s, p, nbytes, T, ring, swz, cnt, limit, run, bad);
    if (s.fill > 0 && s.st + s.fill == cnt) {
        if (THIRD && !RUN)  // pending part below a word, st a multiple of 4
            *reinterpret_cast<uint32_t *>(ring + ((s.st & (RING - 1)) ^ swz)) = static_cast<uint32_t>(s.a0);
        else
            *reinterpret_cast<uint64_t *>(ring + ((s.st & (RING - 1)) ^ swz)) = s.a0;
        s.st = cnt;
        s.fill = 0;
        s.a0 = 0;
    }
}

// Both planes of a lane in one loop, a step of each per pass, both steps
// predicated in one block: two independent dependency chains per lane, for
// launches with few lanes per SM (where issue slots are idle).  A plane that
// is ahead keeps decoding into its ring's room or takes empty steps.
template <int RING, bool RUN_H, bool RUN_L>
__device__ __forceinline__ void fill_pair_t(PlaneDec &h, PlaneDec &l, const uint8_t *ph, size_t nh, const uint8_t *pl,
                                            size_t nl, const DecTables<12> &Th, const LoTables &Tl,
                                            uint8_t *hring, uint8_t *lring, uint32_t swz, int cnt, int need,
                                            int limit, bool &bad) {
    const uint64_t run_h = RUN_H ? Th.run : 0ull, run_l = RUN_L ? Tl.run : 0ull;
    while (__any_sync(0xffffffffu,
                      (h.st < need && h.st + h.fill != cnt) || (l.st < need && l.st + l.fill != cnt))) {
        step<RING, RUN_H, 12, false>(h, ph, nh, Th, hring, swz, cnt, limit, run_h, bad);
        step<RING, RUN_L, 13, false>(l, pl, nl, Tl, lring, swz, cnt, limit, run_l, bad);
    }
    for (int q = 0; q < 2; ++q) {  // a chunk's last partial words
        PlaneDec &s = q ? l : h;
        uint8_t *ring = q ? lring : hring;
        if (s.fill > 0 && s.st + s.fill == cnt) {
            *reinterpret_cast<uint64_t *>(ring + ((s.st & (RING - 1)) ^ swz)) = s.a0;
            s.st = cnt;
            s.fill = 0;
            s.a0 = 0;
        }
    }
}

template <int RING>
__device__ __forceinline__ void fill_pair(PlaneDec &h, PlaneDec &l, const uint8_t *ph, size_t nh, const uint8_t *pl,
                                          size_t nl, const DecTables<12> &Th, const LoTables &Tl,
                                          uint8_t *hring, uint8_t *lring, uint32_t swz, int cnt, int need, int limit,
                                          bool &bad) {
    if (Th.has_run) {
        if (Tl.has_run)
            fill_pair_t<RING, true, true>(h, l, ph, nh, pl, nl, Th, Tl, hring, lring, swz, cnt, need, limit, bad);
        else
            fill_pair_t<RING, true, false>(h, l, ph, nh, pl, nl, Th, Tl, hring, lring, swz, cnt, need, limit, bad);
    } else {
        if (Tl.has_run)
            fill_pair_t<RING, false, true>(h, l, ph, nh, pl, nl, Th, Tl, hring, lring, swz, cnt, need, limit, bad);
        else
            fill_pair_t<RING, false, false>(h, l, ph, nh, pl, nl, Th, Tl, hring, lring, swz, cnt, need, limit, bad);
    }
}

template <int RING, bool LIM, bool THIRD = false, int W, int SEC, bool SPLIT>
__device__ __forceinline__ void fill_segment(PlaneDec &s, const uint8_t *p, size_t nbytes, const DecTables<W, SEC, SPLIT> &T,
                                             uint8_t *ring, uint32_t swz, int cnt, int need, int limit, bool &bad) {
    if (T.has_run)
        fill_segment_t<RING, true, W, LIM, SEC, false, SPLIT>(s, p, nbytes, T, ring, swz, cnt, need, limit, bad);
    else
        fill_segment_t<RING, false, W, LIM, SEC, THIRD, SPLIT>(s, p, nbytes, T, ring, swz, cnt, need, limit, bad);
}

// ------------------------------------------------------------------ planes with a 1-bit code
//
// A plane whose most frequent symbol has a 1-bit code (the high plane of a
// snapshot delta: that symbol is 0 for about 98 % of elements) is decoded as
// runs.  The lane's ring holds that symbol in every slot not yet decoded
// (filled at the start, and again by the merge after it reads a segment), so
// a run costs no store at all.  One step takes at most one other code (it
// starts with a 1 bit: the 1-bit code is 0; its symbol is stored as one byte)
// and then the run of 1-bit codes after it: as many as the zero bits on top of
// the buffer, up to the valid bits, the chunk's rest and the ring's room; then
// a second such round, when the next code is in the first-code table and
// within the valid bits (a warp-level simulation of the snapshot's high plane:
// 1.13 steps per 32-symbol segment instead of 1.81).  No symbols are ever
// pending: st counts the symbols placed.

// The run tables of a codebook with a 1-bit code (every thread of the block
// takes part).
__device__ void load_run_tables(RunTables &T, const huff_codebook *cb) {
    const int tid = threadIdx.x;
    const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC && cb->longest <= HUFF_MAX_LEN;
    if (tid < 32) {
        T.bl_count[tid] = ok ? cb->bl_count[tid] : 0;
        T.first_code[tid] = ok ? cb->first_code[tid] : 0;
        T.first_index[tid] = ok ? cb->first_index[tid] : 0;
    }
    for (int i = tid; i < 256; i += blockDim.x) T.sorted[i] = ok ? cb->sorted_symbols[i] : 0;
    // the codebook's 12-bit table gives each window's first symbol; its code is taken when it is at most
    // kZWin bits long
    for (int i = tid; i < (1 << kZWin); i += blockDim.x) {
        uint32_t v = 0;
        if (ok) {
            const uint64_t e = cb->lut[static_cast<size_t>(i) << (HUFF_LUT_BITS - kZWin)];
            const uint32_t sym = static_cast<uint32_t>(e & 0xffu);
            const uint32_t L = cb->len[sym];
            if (((e >> 48) & 15u) != 0 && L <= static_cast<uint32_t>(kZWin)) v = sym | (L << 8);
        }
        T.zf[i] = static_cast<uint16_t>(v);
    }
    if (tid == 0) {
        T.longest = ok ? cb->longest : 0;
        T.ok = ok;
        T.run = (ok ? static_cast<uint64_t>(cb->sorted_symbols[0]) : 0ull) * 0x0101010101010101ull;
    }
}

// Shift the 64-bit buffer (bh, bl) left by r bits, 0 <= r <= 64.
__device__ __forceinline__ void consume64(PlaneDec &s, uint32_t r) {
    const uint32_t r1 = r < 32 ? r : 32u;  // first up to 32 bits, then the rest
    const uint32_t r2 = r - r1;
    uint32_t bh = __funnelshift_lc(s.bl, s.bh, r1);
    uint32_t bl = __funnelshift_lc(0u, s.bl, r1);
    bh = __funnelshift_lc(bl, bh, r2);
    bl = __funnelshift_lc(0u, bl, r2);
    s.bh = bh;
    s.bl = bl;
    s.nb -= static_cast<int>(r);
}

template <int RING>
__device__ __forceinline__ void step_zrun(PlaneDec &s, const uint8_t *p, size_t nbytes, const RunTables &T,
                                          uint8_t *ring, uint32_t swz, int cnt, int limit, bool &bad) {
    const int rem = cnt - s.st;
    const int room = limit - s.st;
    const bool go = rem > 0 && room > 0;
    s.refill(p, nbytes);
    // another code first, when the top bit is 1
    const bool nz = go && static_cast<int32_t>(s.bh) < 0;
    const uint32_t f = T.zf[s.bh >> (32 - kZWin)];
    uint32_t L = f >> 8, sym = f & 0xffu;
    if (__any_sync(0xffffffffu, nz && L == 0)) {  // a code longer than the window (or none: corrupt)
        if (nz && L == 0) {
            const uint32_t lc = long_code_search<kZWin>(s.bh, &T);
            L = lc >> 8;
            sym = lc & 0xffu;
            if (L == 0) {
                bad = true;
                L = 1;
            }
        }
    }
    if (nz) ring[(s.st & (RING - 1)) ^ swz] = static_cast<uint8_t>(sym);
    const int one = nz ? 1 : 0;
    s.consume(nz ? L : 0u);
    // then the run: the zero bits on top, within the valid bits, the chunk and the ring
    const uint32_t z = s.bh != 0 ? __clz(s.bh) : 32u + __clz(s.bl);  // 64 when the buffer is all zeros
    int r = min(min(static_cast<int>(z), s.nb), min(rem, room) - one);
    r = go ? r : 0;
    consume64(s, static_cast<uint32_t>(r));
    s.st += one + r;
    // a second round: the next code (when the first-code table has it and it lies within the valid
    // bits) and the run after it
    const int rem2 = cnt - s.st, room2 = limit - s.st;
    const bool go2 = go && rem2 > 0 && room2 > 0;
    const bool top1 = static_cast<int32_t>(s.bh) < 0;
    const uint32_t f2 = T.zf[s.bh >> (32 - kZWin)];
    const uint32_t L2 = f2 >> 8;
    const bool nz2 = go2 && top1 && L2 != 0 && static_cast<int>(L2) <= s.nb;
    if (nz2) ring[(s.st & (RING - 1)) ^ swz] = static_cast<uint8_t>(f2 & 0xffu);
    const int one2 = nz2 ? 1 : 0;
    s.consume(nz2 ? L2 : 0u);
    const uint32_t z2 = s.bh != 0 ? __clz(s.bh) : 32u + __clz(s.bl);
    int r2 = min(min(static_cast<int>(z2), s.nb), min(rem2, room2) - one2);
    r2 = (go2 && (nz2 || !top1)) ? r2 : 0;
    consume64(s, static_cast<uint32_t>(r2));
    s.st += one2 + r2;
}

// Steps until every lane of the warp has placed symbols [.., need).
template <int RING>
__device__ __forceinline__ void fill_zrun(PlaneDec &s, const uint8_t *p, size_t nbytes, const RunTables &T,
                                          uint8_t *ring, uint32_t swz, int cnt, int need, int limit, bool &bad) {
    while (__any_sync(0xffffffffu, s.st < need && s.st != cnt))
        step_zrun<RING>(s, p, nbytes, T, ring, swz, cnt, limit, bad);
}

// The chunk's bit range lies in the payload and holds between one and
// HUFF_MAX_LEN bits per symbol.
__device__ __forceinline__ bool chunk_bounds(const uint64_t *off, size_t c, size_t nbytes, int cnt, uint64_t &start,
                                             uint64_t &end) {
    start = off[c];
    end = off[c + 1];
    return start <= end && end <= static_cast<uint64_t>(nbytes) * 8 && end - start >= static_cast<uint64_t>(cnt) &&
           end - start <= static_cast<uint64_t>(cnt) * HUFF_MAX_LEN;
}

// Launch geometry: one lane per chunk (pair), blocks spread over every SM.
__host__ int decode_block(size_t n_chunks, int sms) {
    size_t per_sm = (n_chunks + static_cast<size_t>(sms) - 1) / static_cast<size_t>(sms);
    per_sm = (per_sm + 31) / 32 * 32;
    return static_cast<int>(per_sm > static_cast<size_t>(kMaxBlock) ? kMaxBlock : per_sm);
}

// ------------------------------------------------------------------ byte streams
//
// Lane ring: 2 * kRing bytes (one plane, twice the slack); swizzled by lane
// parity so that the copy-out's reads of 8 lanes' segments spread over the banks.
constexpr int kRingU8 = 2 * kRing;
// Byte streams often meet data their (fixed) codebook was not built for, where
// most symbols have codes of 17 to 24 bits: a secondary table of 16 Ki entries
// (32 KiB; the block's rings leave room for it) holds all of them when their
// 13-bit prefixes are few, so such a code costs one lookup.  The 13-bit table
// is split (at most 4 symbols a window; 2 to 3 % faster on the sweep's
// streams than the 64-bit entries).
constexpr int kSecU8 = 16384;
using U8Tables = DecTables<13, kSecU8, true>;
constexpr int kSegU8 = 2 * kSeg;
static_assert(kRingU8 >= kSegU8 + 7 + 2 * kStepMax && (kRingU8 & (kRingU8 - 1)) == 0 && kSegU8 % 16 == 0,
              "byte-stream ring geometry");

__global__ void __launch_bounds__(kMaxBlock, 1) k_decode_u8(const uint8_t *__restrict__ payload, size_t nbytes,
                                                           const uint64_t *__restrict__ off, size_t n, size_t chunk,
                                                           const huff_codebook *__restrict__ cb,
                                                           uint8_t *__restrict__ out, int32_t *status, int spread) {
    extern __shared__ __align__(16) uint8_t dsm[];
    U8Tables &T = *reinterpret_cast<U8Tables *>(dsm);
    load_table_a(T, cb);
    __syncthreads();
    load_table_b(T, cb);
    __syncthreads();
    if (!T.ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    const int lane = threadIdx.x & 31;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    // a warp takes 32 consecutive chunks; with spread (1), the warps of a block take groups spread over the
    // input (group warp * gridDim.x + block), so that blocks, and the SMs they run on, meet every part of
    // it alike where there are too few waves of blocks for the block scheduler to even them out; by rank
    // (2), block b takes the range of consecutive chunks with the b-th most bits, so that the block
    // scheduler, which starts blocks in index order, starts the costly ones first and ends on cheap ones
    size_t blk = blockIdx.x;
    if (spread == 2) {
        uint64_t *cost = reinterpret_cast<uint64_t *>(dsm + sizeof(U8Tables) + static_cast<size_t>(blockDim.x) * kRingU8);
        uint32_t *pick = reinterpret_cast<uint32_t *>(cost + gridDim.x);
        if (threadIdx.x == 0) *pick = blockIdx.x;  // (the ranks are a permutation: some thread overwrites it)
        for (uint32_t r = threadIdx.x; r < gridDim.x; r += blockDim.x) {
            const size_t a = static_cast<size_t>(r) * blockDim.x, b = min(a + blockDim.x, n_chunks);
            cost[r] = off[b] - off[a];
        }
        __syncthreads();
        for (uint32_t r = threadIdx.x; r < gridDim.x; r += blockDim.x) {
            const uint64_t kr = cost[r];
            uint32_t rank = 0;
            for (uint32_t q = 0; q < gridDim.x; ++q) {
                const uint64_t kq = cost[q];
                rank += (kq > kr || (kq == kr && q < r)) ? 1u : 0u;
            }
            if (rank == blockIdx.x) *pick = r;
        }
        __syncthreads();
        blk = *pick;
    }
    const size_t c = spread == 1 ? (static_cast<size_t>(threadIdx.x >> 5) * gridDim.x + blockIdx.x) * 32 + lane
                                 : blk * blockDim.x + threadIdx.x;
    const size_t c0 = c - lane;  // the warp's first chunk
    uint64_t start = 0, end = 0;
    int cnt = 0;
    if (c < n_chunks) {
        const size_t first = c * chunk;
        const int want = static_cast<int>(n - first < chunk ? n - first : chunk);
        if (chunk_bounds(off, c, nbytes, want, start, end))
            cnt = want;
        else
            set_status(status, HUFF_ERR_CORRUPT_STREAM);
    }
    uint8_t *rings = dsm + sizeof(U8Tables) + static_cast<size_t>(threadIdx.x - lane) * kRingU8;
    uint8_t *ring = rings + lane * kRingU8;
    const uint32_t swz = (lane & 1) ? kRingU8 / 2 : 0;
    PlaneDec s;
    plane_start(s, payload, nbytes, start, cnt);
    bool bad = false;
    const int warp_cnt = __reduce_max_sync(0xffffffffu, cnt);
    const bool whole = __all_sync(0xffffffffu, cnt == warp_cnt);  // every chunk of the warp has the same length
    for (int seg0 = 0; seg0 < warp_cnt; seg0 += kSegU8) {
        // (no third lookup here: on the sweep's drifted data, where long codes dominate, it measured slower)
        fill_segment<kRingU8, true>(s, payload, nbytes, T, ring, swz, cnt, min(cnt, seg0 + kSegU8), seg0 + kRingU8, bad);
        __syncwarp();
        // copy-out: 8 lanes' segments per pass, 16 bytes per lane
        if (whole && seg0 + kSegU8 <= warp_cnt) {  // every lane's segment is complete: no per-lane bounds
            // pass i: source lane 8 i + lane / 4 (same parity as lane / 4), 8 i chunks further on
            const int s0 = lane >> 2;
            const int e0 = seg0 + 16 * (lane & 3);
            const uint8_t *src = rings + s0 * kRingU8 + ((e0 & (kRingU8 - 1)) ^ ((s0 & 1) ? kRingU8 / 2 : 0));
            uint8_t *dst = out + (c0 + s0) * chunk + e0;
            const size_t ds = 8 * chunk;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                __stcs(reinterpret_cast<uint4 *>(dst + i * ds), *reinterpret_cast<const uint4 *>(src + i * 8 * kRingU8));
            __syncwarp();
            continue;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int sl = 8 * i + (lane >> 2);
            const int e0 = seg0 + 16 * (lane & 3);
            const int cs = __shfl_sync(0xffffffffu, cnt, sl);
            if (e0 < cs) {
                const uint8_t *src =
                    rings + sl * kRingU8 + ((e0 & (kRingU8 - 1)) ^ ((sl & 1) ? kRingU8 / 2 : 0));
                uint8_t *dst = out + (c0 + sl) * chunk + e0;
                const uint4 v = *reinterpret_cast<const uint4 *>(src);
                if (e0 + 16 <= cs) {  // out is 16-byte aligned and chunk a multiple of 32
                    __stcs(reinterpret_cast<uint4 *>(dst), v);
                } else {
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    for (int k = 0; k < cs - e0; ++k) dst[k] = static_cast<uint8_t>(w[k >> 2] >> (8 * (k & 3)));
                }
            }
        }
        __syncwarp();
    }
    if (cnt > 0 && (bad || s.pos() != off[c + 1])) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

// A slice's output bytes, stored as aligned 8-byte words.  Its first and
// last words may hold other slices' bytes, so those two are written byte by
// byte (the slice's own bytes only); every word between them in one store.
struct WordOut {
    uint8_t *w;     // the aligned word being filled
    uint64_t acc;   // its bytes so far, byte k of the word in byte k
    uint32_t f;     // position of the next byte in the word
    uint32_t f0;    // the slice's first byte in the word (nonzero only in the slice's first word)
    uint64_t left;  // bytes the slice may still write
    __device__ __forceinline__ void init(uint8_t *o, uint64_t room) {
        f0 = f = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(o) & 7u);
        w = o - f;
        acc = 0;
        left = room;
    }
    __device__ __forceinline__ void bytes(uint32_t upto) {  // bytes [f0, upto) of the word
        for (uint32_t k = f0; k < upto; ++k) w[k] = static_cast<uint8_t>(acc >> (8 * k));
    }
    __device__ __forceinline__ void put(uint64_t v, uint32_t c) {  // c <= 6 bytes, v's higher bytes zero
        if (c > left) {  // only a corrupt chunk decodes more symbols than it holds
            c = static_cast<uint32_t>(left);
            v &= (1ull << (8 * c)) - 1ull;
        }
        left -= c;
        acc |= v << (8 * f);
        const uint32_t nf = f + c;
        if (nf >= 8) {  // the word is complete (f >= 2 here, so the carry shift is 16..48)
            if (f0 == 0)
                *reinterpret_cast<uint64_t *>(w) = acc;
            else
                bytes(8);
            w += 8;
            f0 = 0;
            acc = v >> (8 * (8 - f));
            f = nf - 8;
        } else {
            f = nf;
        }
    }
    __device__ __forceinline__ void finish() {
        if (f > f0) bytes(f);
    }
};

// ------------------------------------------------------------------ byte streams, few chunks
//
// With fewer chunks than the GPU has lanes to spare, one lane per chunk
// leaves most of the GPU idle.  Then a CTA takes one chunk and splits its bit
// range into S slices, one thread each (S = blockDim.x).  It relies on
// Huffman codes being self-synchronising: a decode started at an arbitrary
// bit usually falls onto the true code boundaries within a few codes (the
// observation behind Klein and Wiseman's parallel decoding and the GPU
// decoder of Weissenberger and Schmidt).  Three walks over the slice:
//   1. from the slice's first bit (a true boundary for slice 0; slices start
//      on multiples of the code lengths' greatest common divisor, so for a
//      code of one length every slice does) to the first boundary of that
//      walk at or after the slice's end: the exit;
//   2. from the previous slice's exit, counting the codes that start in the
//      slice, to a new exit; repeated while any exit changes.  Slice 0 starts
//      at the chunk's offset, so after round r slices 0..r are exact and a
//      round that changes nothing has every exit exact: at most S + 1 rounds,
//      whatever the code (one that never resynchronises costs a round per
//      slice);
//   3. a block scan of the counts gives each slice its first output index;
//      each slice decodes again from its entry and stores its symbols.
// The chunk is valid when the counts add up to its symbol count and the last
// slice's exit is the next chunk's offset.
constexpr int kSplitMinSyms = 16;  // symbols per slice at least, where the chunk allows 32 slices

// The split decode's copy of a codebook's canonical arrays (shared memory).
struct SplitTab {
    uint32_t lim[32];
    uint32_t first_code[32];
    uint32_t first_index[32];
    uint32_t bl_count[32];
    uint8_t sorted[256];
};

// The codes that start in [pos, lim): their count, and with WRITE the symbols
// stored to out[0, room).  pos ends at the walk's first boundary at or after
// lim.  Every iteration takes at least one bit, so a walk over corrupt data
// ends as well; `bad` notes bits that are no code.
// Positions are relative to the slice's first bit (32 bits: a chunk holds at
// most 2^30 * 24 bits and has at least 32 slices).
template <bool WRITE>
__device__ uint32_t split_walk(PlaneDec &s, const uint8_t *p, size_t nbytes, const huff_codebook *cb,
                               const SplitTab &tab, int longest, uint32_t &pos, uint32_t lim, uint8_t *out,
                               uint64_t room, bool &bad) {
    uint32_t n = 0;
    WordOut wo;
    if (WRITE) wo.init(out, room);
    while (pos < lim) {
        s.refill(p, nbytes);
        const uint64_t e = __ldg(&cb->lut[s.bh >> (32 - HUFF_LUT_BITS)]);
        uint32_t c = static_cast<uint32_t>(e >> 48) & 15u;
        uint32_t bits = static_cast<uint32_t>(e >> 52) & 15u;
        uint64_t v = e & 0xffffffffffffull;
        if (c == 0) {  // the first code is longer than the table's window (or no code)
            const uint32_t lc = long_code_lim<HUFF_LUT_BITS>(s.bh, tab, longest);
            bits = lc >> 8;
            v = lc & 0xffu;
            c = 1;
            if (bits == 0) {
                bad = true;
                bits = 1;
            }
        } else if (pos + bits > lim) {  // codes past lim in the entry: only the first starts before it
            c = 1;
            v &= 0xffu;
            bits = __ldg(&cb->len[v]);
        }
        if (WRITE) wo.put(v, c);
        n += c;
        pos += bits;
        s.consume(bits);
    }
    if (WRITE) wo.finish();
    return n;
}

__global__ void __launch_bounds__(1024) k_decode_u8_split(const uint8_t *__restrict__ payload, size_t nbytes,
                                                         const uint64_t *__restrict__ off, size_t n, size_t chunk,
                                                         const huff_codebook *__restrict__ cb,
                                                         uint8_t *__restrict__ out, int32_t *status) {
    extern __shared__ __align__(16) uint8_t dsm[];
    const int S = blockDim.x;
    const int k = threadIdx.x;
    uint64_t *ex = reinterpret_cast<uint64_t *>(dsm);          // slice exits, S
    uint64_t *wsum = ex + S;                                    // per-warp count sums, 32
    SplitTab &tab = *reinterpret_cast<SplitTab *>(wsum + 32);
    const int longest = cb->longest;
    if (cb->magic != HUFF_CODEBOOK_MAGIC || longest < 1 || longest > HUFF_MAX_LEN) {
        if (k == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    const size_t c = blockIdx.x;
    const size_t first = c * chunk;
    const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
    uint64_t start = 0, end = 0;
    if (!chunk_bounds(off, c, nbytes, cnt, start, end)) {  // the same for the whole CTA
        if (k == 0) set_status(status, HUFF_ERR_CORRUPT_STREAM);
        return;
    }
    // slice boundaries on multiples of g, the greatest common divisor of the code lengths, from the chunk's
    // start: a code whose lengths share a divisor (all 8 bits, say) then starts every slice on a boundary
    uint32_t g = 0;
    for (int l = 1; l <= longest; ++l) {
        if (__ldg(&cb->bl_count[l]) == 0) continue;
        uint32_t a = static_cast<uint32_t>(l), b = g;
        while (b) {
            const uint32_t t = a % b;
            a = b;
            b = t;
        }
        g = a;
    }
    if (g == 0) g = 1;
    if (k < 32) {
        tab.lim[k] = code_limit(cb, true, k);
        tab.first_code[k] = cb->first_code[k];
        tab.first_index[k] = cb->first_index[k];
        tab.bl_count[k] = cb->bl_count[k];
    }
    for (int i = k; i < 256; i += S) tab.sorted[i] = cb->sorted_symbols[i];
    __syncthreads();
    const uint64_t span = end - start;
    const auto bound = [&](int j) -> uint64_t {
        if (j >= S) return end;
        const uint64_t b = span * static_cast<uint64_t>(j) / static_cast<uint64_t>(S);
        return start + b / g * g;
    };
    const uint64_t lo = bound(k);
    const uint64_t hi = bound(k + 1);
    PlaneDec s;
    bool unsynced = false;  // walks 1 and 2 may start off the code boundaries: bits that are no code mean nothing
    bool bad = false;       // walk 3 starts on them
    // 1. from the slice's first bit
    // (every entry and exit of slice k is at or after lo: an exit is at or after its own slice's end)
    const uint32_t rl = static_cast<uint32_t>(hi - lo);
    uint64_t pos = lo;
    if (lo < hi) {
        s.start(payload, nbytes, lo);
        uint32_t rp = 0;
        split_walk<false>(s, payload, nbytes, cb, tab, longest, rp, rl, nullptr, 0, unsynced);
        pos = lo + rp;
    }
    ex[k] = pos;
    __syncthreads();
    // 2. from the previous slice's exit until no exit changes
    uint64_t entry = start, mine = 0;
    for (int round = 0; round <= S; ++round) {
        entry = k == 0 ? start : ex[k - 1];
        pos = entry;
        mine = 0;
        if (entry < hi) {
            s.start(payload, nbytes, entry);
            uint32_t rp = static_cast<uint32_t>(entry - lo);
            mine = split_walk<false>(s, payload, nbytes, cb, tab, longest, rp, rl, nullptr, 0, unsynced);
            pos = lo + rp;
        }
        const bool changed = pos != ex[k];
        __syncthreads();  // every slice has read its entry
        ex[k] = pos;
        if (!__syncthreads_or(changed)) break;
    }
    // 3. output indices: exclusive scan of the counts over the block
    const int lane = k & 31, warp = k >> 5;
    uint64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = S >> 5;
        uint64_t w = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) wsum[lane] = w;  // inclusive sums of whole warps
    }
    __syncthreads();
    const uint64_t base = incl - mine + (warp ? wsum[warp - 1] : 0);
    const uint64_t total = wsum[(S >> 5) - 1];
    if (k == 0 && (total != static_cast<uint64_t>(cnt) || ex[S - 1] != end)) set_status(status, HUFF_ERR_CORRUPT_STREAM);
    if (entry < hi && base < static_cast<uint64_t>(cnt)) {
        s.start(payload, nbytes, entry);
        uint32_t rp = static_cast<uint32_t>(entry - lo);
        split_walk<true>(s, payload, nbytes, cb, tab, longest, rp, rl, out + first + base,
                         static_cast<uint64_t>(cnt) - base, bad);
    }
    if (bad) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

// ------------------------------------------------------------------ byte streams, fewer chunks
//
// With fewer chunks than one lane each needs to fill the GPU (or to balance
// it: the chunks' decode costs can differ several times), a team of TW warps
// (TW = 1 while there are enough chunks, up to the whole CTA when they are
// few) decodes a chunk in rounds of TW * 32 slices of B bits, one per
// thread.  Each slice is walked once from its first bit, which need not be a
// code boundary (Huffman codes are self-synchronising: a walk started
// anywhere falls onto the true boundaries within a few codes, as Klein and
// Wiseman's parallel decoding and Weissenberger and Schmidt's GPU decoder
// use).  The walk stages the symbols of the codes that start in the slice in
// the thread's area of shared memory, and notes where its first kWsList
// table steps start and how many symbols came before each.  Then each thread
// goes on past its slice's end, one code at a time, until a code starts
// where a noted step of the next slice starts: from there on the two walks
// are the same, so once this slice is exact the next one is exact from that
// step, and the codes in between are this slice's (staged after its own).
// The walk that reaches no noted step (about one slice in a few thousand on
// the data measured) leaves the next slice to be walked again from this
// slice's exit; its own end may then move, so the slice after it checks
// again (slice 0 starts on the round's exact entry, and pass i makes slice i
// exact).  A scan of the slices' counts places each slice's symbols, which
// each thread copies from its area to the output.
// B follows the chunk's mean code length so that a slice holds about
// kWsTarget symbols (with a team of several warps, no more than gives every
// slice of one round some bits); a slice with more than its area holds (a
// skewed part of a chunk) is decoded once more from its entry, writing
// straight to the output.  Slices start on multiples of the code lengths'
// greatest common divisor from the chunk's start: a code of one length (all
// 8 bits, say) then starts every slice on a boundary.
// A CTA per SM of kWsWarps warps shares one copy of the tables; its teams
// take chunks blockIdx.x, blockIdx.x + gridDim.x, ... (interleaved, so every
// CTA meets every part of the input alike) from a shared counter, a chunk at
// a time and the largest (most bits) first, so teams that drew cheap chunks
// take more of them and the share ends on cheap ones (the 16 GiB sweep at
// 1 MiB chunks: 205 -> 231 GB/s against taking them in order).
constexpr int kWsWarps = 28;              // warps per CTA (7 per scheduler)
constexpr int kWsStage = 84;              // staged symbols per slice
constexpr int kWsStride = kWsStage + 4;   // bytes between two threads' areas (a word of padding read by the copy)
constexpr int kWsTarget = 56;             // symbols a slice is sized for
constexpr int kWsList = 24;               // steps noted per walk
static_assert(kWsStage % 4 == 0 && 4 * kWsList <= 255, "staging geometry");

// A thread's step notes: where its first walk's first kWsList steps start
// (relative to the slice's first bit) and the symbols before each; entry i
// of a team's slice l at i * (slices per round) + l.
struct WsNotes {
    uint16_t *pos;
    uint8_t *cnt;
};

// The first code of the window: its symbol and length (length 0 when the bits are no code).
__device__ __forceinline__ void ws_code(const PlaneDec &s, const U8Tables &T, uint32_t &L, uint32_t &sym) {
    const uint32_t win = s.bh >> (32 - 13);
    uint64_t v;
    uint32_t c, bits;
    lut_get(T, win, v, c, bits);
    if (c != 0) {
        sym = static_cast<uint32_t>(v) & 0xffu;
        L = T.len[sym];
        return;
    }
    L = 0;
    sym = 0;
    if (T.sec_ok) {
        if (T.sec_k > 0 && static_cast<int>(win) >= T.sec_first) {
            const int k = T.sec_k;
            const uint32_t e2 = T.sec[((win - static_cast<uint32_t>(T.sec_first)) << k) |
                                      ((s.bh >> (32 - 13 - k)) & ((1u << k) - 1u))];
            L = e2 >> 8;
            sym = e2 & 0xffu;
        }
    } else {
        const uint32_t lc = long_code(s.bh, &T);
        L = lc >> 8;
        sym = lc & 0xffu;
    }
}

// One walk over [pos, lim) (positions relative to the round's entry; lo = the
// slice's first bit): the count of the codes that start in it, and their
// symbols: staged (the first kWsStage; NOTE: with the first kWsList steps
// noted) or, DIRECT, written to dst[0, room).  pos ends at the walk's exit;
// badpos is the last position (relative to lo) where the bits were no code.
template <bool DIRECT, bool NOTE, int NS, bool TWO = false>
__device__ __forceinline__ uint32_t ws_walk(PlaneDec &s_io, const uint8_t *p, size_t nbytes, const U8Tables &T,
                                         uint32_t &pos, uint32_t lo, uint32_t lim, uint8_t *stg, WsNotes nt,
                                         int &nsteps, int &badpos, uint8_t *dst, uint64_t room) {
    PlaneDec s = s_io;  // a private copy, so that the stores below cannot alias the reader's state
    const int seck = T.sec_k, secf = T.sec_first;
    const bool use_sec = T.sec_ok;
    uint32_t n = 0;
    uint32_t a = 0;  // pending staged bytes (fewer than 4)
    int fill = 0, st = 0, steps = 0;
    WordOut wo;
    if (DIRECT) wo.init(dst, room);
    while (pos < lim) {
        s.refill(p, nbytes);
        const uint32_t win = s.bh >> (32 - 13);
        uint64_t v;
        uint32_t c, bits;
        lut_get(T, win, v, c, bits);
        if (NOTE && steps < kWsList) {
            nt.pos[steps * NS] = static_cast<uint16_t>(pos - lo);
            nt.cnt[steps * NS] = static_cast<uint8_t>(n);
        }
        ++steps;
        // a code longer than the window: the secondary table's entry, looked up on every step (a
        // predicated load rather than a branch that splits the warp where long and short codes mix)
        uint32_t L2 = 0, sym2 = 0;
        if (use_sec) {
            const bool inr = seck > 0 && static_cast<int>(win) >= secf;
            const uint32_t idx =
                inr ? ((win - static_cast<uint32_t>(secf)) << seck) | ((s.bh >> (32 - 13 - seck)) & ((1u << seck) - 1u))
                    : 0u;
            const uint32_t e2 = T.sec[idx];
            L2 = inr ? e2 >> 8 : 0u;
            sym2 = e2 & 0xffu;
        } else if (c == 0) {
            const uint32_t lc = long_code(s.bh, &T);
            L2 = lc >> 8;
            sym2 = lc & 0xffu;
        }
        const bool lng = c == 0;
        if (lng && L2 == 0) badpos = static_cast<int>(pos - lo);  // no code
        v = lng ? sym2 : v;
        bits = lng ? max(L2, 1u) : bits;
        c = lng ? 1u : c;
        const bool cut = c > 1 && pos + bits > lim;
        if (cut) {  // codes past lim in the entry: only the first starts before it
            v &= 0xffu;
            c = 1;
            bits = T.len[v];
        }
        if constexpr (TWO && !DIRECT) {
            // short codes: a second lookup on the bits after a simple first entry, when its codes end by lim
            const uint32_t top2 = __funnelshift_l(s.bl, s.bh, bits);
            uint64_t v2;
            uint32_t c2, b2;
            lut_get(T, top2 >> (32 - 13), v2, c2, b2);
            const bool take2 = !lng && !cut && c2 != 0 && pos + bits + b2 <= lim;
            v |= take2 ? v2 << (8 * c) : 0ull;
            bits += take2 ? b2 : 0u;
            c += take2 ? c2 : 0u;
        }
        bits = max(bits, 1u);  // only a corrupt codebook has a zero-length entry: every step moves on
        if (DIRECT) {
            wo.put(v, c);
        } else {
            const uint32_t sh = 8u * static_cast<uint32_t>(fill);
            const uint32_t vl = static_cast<uint32_t>(v);
            const uint32_t w0 = a | (vl << sh);
            const int nf = fill + static_cast<int>(c);  // <= 7 (<= 11 with a second lookup)
            if (nf >= 4 && st + 4 <= kWsStage) *reinterpret_cast<uint32_t *>(stg + st) = w0;
            if constexpr (TWO) {
                const uint32_t vh = static_cast<uint32_t>(v >> 32);
                const uint32_t w1 = __funnelshift_l(vl, vh, sh);
                if (nf >= 8 && st + 8 <= kWsStage) *reinterpret_cast<uint32_t *>(stg + st + 4) = w1;
                a = nf >= 8 ? __funnelshift_l(vh, 0u, sh) : (nf >= 4 ? w1 : w0);
                st += nf & ~3;
            } else {
                a = nf >= 4 ? __funnelshift_l(vl, 0u, sh) : w0;  // the bytes past the completed word
                st += nf >= 4 ? 4 : 0;
            }
            fill = nf & 3;
        }
        n += c;
        pos += bits;
        s.consume(bits);
    }
    if (DIRECT)
        wo.finish();
    else if (fill > 0 && st + 4 <= kWsStage)
        *reinterpret_cast<uint32_t *>(stg + st) = a;
    nsteps = min(steps, kWsList);
    s_io = s;
    return n;
}

// From the walk's exit pos (the reader is there), codes one at a time until
// one starts where a noted step of the next slice starts (npos: its notes,
// nns of them, relative to its first bit nlo): returns that step, or -1 when
// the codes pass its last note.  The codes' symbols are staged from stg[n]
// on, m of them; pb notes bits that are no code.
template <int NS>
__device__ __forceinline__ int ws_over(PlaneDec &s_io, const uint8_t *p, size_t nbytes, const U8Tables &T, uint32_t pos,
                                    uint32_t nlo, const uint16_t *npos, int nns, uint8_t *stg, uint32_t n,
                                    uint32_t &m, bool &pb) {
    PlaneDec s = s_io;
    int j = 0;
    m = 0;
    for (;;) {
        const uint32_t d = pos - nlo;
        while (j < nns && npos[j * NS] < d) ++j;
        if (j == nns) break;
        if (npos[j * NS] == d) {
            s_io = s;
            return j;
        }
        s.refill(p, nbytes);
        uint32_t L, sym;
        ws_code(s, T, L, sym);
        if (L == 0) {
            pb = true;
            L = 1;
        }
        if (n + m < static_cast<uint32_t>(kWsStage)) stg[n + m] = static_cast<uint8_t>(sym);
        ++m;
        pos += L;
        s.consume(L);
    }
    s_io = s;
    return -1;
}

// Bytes stg[from, from + len) to dst[0, len): 4-byte stores between a head
// and a tail of single bytes.  Reads stay below from + len rounded up to a
// word, plus one word (the area's padding).
__device__ __forceinline__ void ws_copy(const uint8_t *stg, uint32_t from, uint32_t len, uint8_t *dst) {
    const uint32_t head = min(len, (4u - static_cast<uint32_t>(reinterpret_cast<uintptr_t>(dst) & 3u)) & 3u);
    uint32_t i = 0;
    for (; i < head; ++i) dst[i] = stg[from + i];
    for (; i + 4 <= len; i += 4) {
        const uint32_t at = from + i, wa = at & ~3u;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(stg + wa);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(stg + wa + 4);
        *reinterpret_cast<uint32_t *>(dst + i) = __funnelshift_r(w0, w1, 8u * (at & 3u));
    }
    for (; i < len; ++i) dst[i] = stg[from + i];
}

// A team of TW warps decodes one chunk at a time; slice i of a round goes to
// the team's thread i.  Exchanges between neighbouring slices, the count
// scan and broadcasts use warp shuffles within one warp (TW = 1) and shared
// memory with the team's own named barrier otherwise.
template <int TW>
struct WsTeam {
    uint32_t *xa, *xb;  // L words each: values exchanged between neighbouring slices
    uint32_t *xw;       // 32 words: warp totals and broadcasts
    int tl, lane, wt, id;  // thread in the team, lane, warp in the team, team in the CTA
    __device__ __forceinline__ void sync() const {
        if constexpr (TW == 1)
            __syncwarp();
        else
            asm volatile("barrier.sync %0, %1;" ::"r"(id + 1), "n"(TW * 32) : "memory");
    }
    __device__ __forceinline__ bool any(bool p) const {
        if constexpr (TW == 1) {
            return __any_sync(0xffffffffu, p);
        } else {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\tbarrier.red.or.pred b, %2, %3, a;\n\t"
                "selp.u32 %0, 1, 0, b;\n\t}"
                : "=r"(r)
                : "r"(static_cast<uint32_t>(p)), "r"(id + 1), "n"(TW * 32)
                : "memory");
            return r != 0;
        }
    }
    // the previous slice's values (slice 0 gets its own)
    __device__ __forceinline__ void prev2(uint32_t &a, uint32_t &b) const {
        if constexpr (TW == 1) {
            a = __shfl_up_sync(0xffffffffu, a, 1);
            b = __shfl_up_sync(0xffffffffu, b, 1);
        } else {
            xa[tl] = a;
            xb[tl] = b;
            sync();
            const int q = tl ? tl - 1 : 0;
            a = xa[q];
            b = xb[q];
            sync();
        }
    }
    // the next slice's value (the last slice gets its own)
    __device__ __forceinline__ uint32_t next(uint32_t v) const {
        if constexpr (TW == 1) {
            return __shfl_down_sync(0xffffffffu, v, 1);
        } else {
            xa[tl] = v;
            sync();
            const uint32_t r = xa[tl + 1 < TW * 32 ? tl + 1 : tl];
            sync();
            return r;
        }
    }
    __device__ __forceinline__ uint32_t from(uint32_t v, int src) const {
        if constexpr (TW == 1) {
            return __shfl_sync(0xffffffffu, v, src);
        } else {
            if (tl == src) xw[0] = v;
            sync();
            const uint32_t r = xw[0];
            sync();
            return r;
        }
    }
    // exclusive prefix sum over the team's slices, and their total
    __device__ __forceinline__ uint32_t scan(uint32_t v, uint32_t &total) const {
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if constexpr (TW == 1) {
            total = __shfl_sync(0xffffffffu, incl, 31);
            return incl - v;
        } else {
            if (lane == 31) xw[wt] = incl;
            sync();
            uint32_t before = 0, all = 0;
            for (int w = 0; w < TW; ++w) {
                const uint32_t t = xw[w];
                all += t;
                before += w < wt ? t : 0u;
            }
            sync();
            total = all;
            return before + incl - v;
        }
    }
};

// Shared memory of one team: the lanes' areas, the step notes and the exchange words.
template <int TW>
__host__ __device__ constexpr size_t ws_team_bytes() {
    return static_cast<size_t>(TW) * 32 * (kWsStride + 3 * kWsList + 8) + 32 * 4;
}
constexpr int kWsOrder = 768;  // chunks a CTA orders by size (its share below kWsMaxPerSm chunks per SM)
template <int TW>
__host__ size_t ws_smem() {
    return sizeof(U8Tables) + static_cast<size_t>(kWsWarps / TW) * ws_team_bytes<TW>() + 16 + 2 * kWsOrder;
}

template <int TW>
__global__ void __launch_bounds__(kWsWarps * 32, 1) k_decode_u8_ws(const uint8_t *__restrict__ payload, size_t nbytes,
                                                                  const uint64_t *__restrict__ off, size_t n,
                                                                  size_t chunk, const huff_codebook *__restrict__ cb,
                                                                  uint8_t *__restrict__ out, int32_t *status) {
    static_assert(kWsWarps % TW == 0 && (TW == 1 || kWsWarps / TW <= 15), "teams divide the CTA; one named barrier each");
    constexpr int L = TW * 32;
    extern __shared__ __align__(16) uint8_t dsm[];
    U8Tables &T = *reinterpret_cast<U8Tables *>(dsm);
    const int warp = threadIdx.x >> 5;
    WsTeam<TW> tm;
    tm.lane = threadIdx.x & 31;
    tm.wt = warp % TW;
    tm.id = warp / TW;
    tm.tl = tm.wt * 32 + tm.lane;
    const int tl = tm.tl;
    uint8_t *const tbase = dsm + sizeof(U8Tables) + static_cast<size_t>(tm.id) * ws_team_bytes<TW>();
    uint8_t *const stg = tbase + tl * kWsStride;
    WsNotes nt;
    nt.pos = reinterpret_cast<uint16_t *>(tbase + L * kWsStride) + tl;
    nt.cnt = tbase + L * kWsStride + L * 2 * kWsList + tl;
    tm.xa = reinterpret_cast<uint32_t *>(tbase + L * (kWsStride + 3 * kWsList));
    tm.xb = tm.xa + L;
    tm.xw = tm.xb + L;
    int *next = reinterpret_cast<int *>(dsm + sizeof(U8Tables) + static_cast<size_t>(kWsWarps / TW) * ws_team_bytes<TW>());
    load_table_a(T, cb);
    if (threadIdx.x == 0) *next = 0;
    __syncthreads();
    load_table_b(T, cb);
    __syncthreads();
    if (!T.ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        return;
    }
    // g: the greatest common divisor of the code lengths
    uint32_t g = 0;
    for (int l = 1; l <= T.longest; ++l) {
        if (T.bl_count[l] == 0) continue;
        uint32_t x = static_cast<uint32_t>(l), y = g;
        while (y) {
            const uint32_t t = x % y;
            x = y;
            y = t;
        }
        g = x;
    }
    if (g == 0) g = 1;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    // the CTA's share, chunks blockIdx.x + gridDim.x j, taken largest first (by their bits): the team that
    // takes the share's last chunks then takes cheap ones, and the teams finish closer together
    const uint32_t share =
        n_chunks > blockIdx.x ? static_cast<uint32_t>((n_chunks - blockIdx.x + gridDim.x - 1) / gridDim.x) : 0u;
    uint16_t *order = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(next) + 16);
    const bool ordered = share <= static_cast<uint32_t>(kWsOrder);
    if (ordered) {
        uint64_t *key = reinterpret_cast<uint64_t *>(dsm + sizeof(U8Tables));  // the areas, not in use yet
        for (uint32_t i = threadIdx.x; i < share; i += blockDim.x) {
            const size_t c = blockIdx.x + static_cast<size_t>(i) * gridDim.x;
            key[i] = off[c + 1] - off[c];
        }
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < share; i += blockDim.x) {  // rank: larger first, then by index
            const uint64_t ki = key[i];
            uint32_t r = 0;
            for (uint32_t q = 0; q < share; ++q) {
                const uint64_t kq = key[q];
                r += (kq > ki || (kq == ki && q < i)) ? 1u : 0u;
            }
            order[r] = static_cast<uint16_t>(i);
        }
        __syncthreads();
    }
    bool bad = false;
    for (;;) {
        uint32_t jc = 0;
        if (tl == 0) jc = static_cast<uint32_t>(atomicAdd(next, 1));
        jc = tm.from(jc, 0);
        if (jc >= share) break;
        if (ordered) jc = order[jc];
        const size_t c = blockIdx.x + static_cast<size_t>(jc) * gridDim.x;
        if (c >= n_chunks) break;
        const size_t first = c * chunk;
        const int cnt = static_cast<int>(n - first < chunk ? n - first : chunk);
        uint64_t start = 0, end = 0;
        if (!chunk_bounds(off, c, nbytes, cnt, start, end)) {
            if (tl == 0) set_status(status, HUFF_ERR_CORRUPT_STREAM);
            continue;
        }
        // slice length: about kWsTarget symbols at the chunk's mean code length (a team of several warps:
        // no more than gives every slice of one round some bits), at least 32 bits, a multiple of g
        const uint64_t span = end - start;
        uint32_t B = static_cast<uint32_t>(span * kWsTarget / static_cast<uint64_t>(cnt));
        if (TW > 1) {
            const uint64_t fit = (span + L - 1) / L;
            if (fit < B) B = static_cast<uint32_t>(fit);
        }
        B = max(B, 32u);
        B = (B + g - 1) / g * g;
        // short codes (a mean of at most 6 bits): a second lookup a step (N(0, 8) bytes at 64 and 256 KiB
        // chunks: +10 and +9 %); longer ones gain nothing from it and pay for it
        const bool two = span <= 6ull * static_cast<uint64_t>(cnt);
        uint8_t *const dst0 = out + first;
        uint64_t entry = start, written = 0;
        while (entry < end) {
            const uint64_t left = end - entry;
            const uint32_t rlen = left < static_cast<uint64_t>(L) * B ? static_cast<uint32_t>(left) : L * B;
            const uint32_t lo = static_cast<uint32_t>(tl) * B;
            const uint32_t hi = tl == L - 1 ? rlen : min(lo + B, rlen);
            const bool act = lo < rlen;
            const int last = static_cast<int>((rlen - 1) / B);  // the last slice with bits
            const bool has_next = tl < last;
            PlaneDec s;
            uint32_t ex = lo, cntw = 0;
            int ns = 0, badpos = -1;
            if (act) {
                s.start(payload, nbytes, entry + lo);
                cntw = two ? ws_walk<false, true, L, true>(s, payload, nbytes, T, ex, lo, hi, stg, nt, ns, badpos, nullptr, 0)
                           : ws_walk<false, true, L>(s, payload, nbytes, T, ex, lo, hi, stg, nt, ns, badpos, nullptr, 0);
            }
            tm.sync();  // every slice's notes are in place
            const int ns_next = static_cast<int>(tm.next(static_cast<uint32_t>(ns)));
            // past the slice's end until the next slice's walk is met
            uint32_t m = 0;
            bool pb = false;
            int met = -1;
            if (has_next) met = ws_over<L>(s, payload, nbytes, T, ex, hi, nt.pos + 1, ns_next, stg, cntw, m, pb);
            // each slice's entry: from the previous slice's meeting step (M), or walked again from its exit (R)
            uint32_t skip = 0, ent = lo, seen_e = 0xffffffffu;
            int seen_met = -2;
            bool first_walk = true, used_m = false, own_bad = false, settled = false;
            for (int pass = 0; pass <= L; ++pass) {
                uint32_t e = ex, mpu = static_cast<uint32_t>(met);
                tm.prev2(e, mpu);
                int mp = static_cast<int>(mpu);
                if (tl == 0) {
                    e = 0;
                    mp = 0;  // slice 0 starts on the round's entry, its first noted step
                }
                const bool todo = act && (e != seen_e || mp != seen_met);
                settled = !tm.any(todo);
                if (settled) break;
                if (!todo) continue;
                seen_e = e;
                seen_met = mp;
                if (e >= hi) {  // no code starts in the slice (only the last one can be this short)
                    skip = cntw;
                    ent = e;
                    used_m = false;
                    own_bad = false;
                    continue;
                }
                if (mp >= 0 && first_walk) {
                    skip = nt.cnt[mp * L];
                    ent = lo + nt.pos[mp * L];
                    used_m = true;
                    own_bad = badpos >= static_cast<int>(ent - lo);
                    continue;
                }
                // walk the slice again from its exact entry, then past its end again
                s.start(payload, nbytes, entry + e);
                ex = e;
                badpos = -1;
                int n2 = 0;
                cntw = two ? ws_walk<false, false, L, true>(s, payload, nbytes, T, ex, lo, hi, stg, nt, n2, badpos, nullptr, 0)
                           : ws_walk<false, false, L>(s, payload, nbytes, T, ex, lo, hi, stg, nt, n2, badpos, nullptr, 0);
                skip = 0;
                ent = e;
                used_m = false;
                first_walk = false;
                own_bad = badpos >= 0;
                pb = false;
                met = has_next ? ws_over<L>(s, payload, nbytes, T, ex, hi, nt.pos + 1, ns_next, stg, cntw, m, pb) : -1;
            }
            if (!settled) bad = true;  // cannot happen: pass i makes slice i exact
            // this slice's codes past its end are its own when the next slice starts at the meeting step
            const bool next_m = tm.next(used_m ? 1u : 0u) != 0 && has_next;
            if (act && (own_bad || (next_m && pb))) bad = true;
            const uint32_t own = act ? cntw - skip : 0u;
            const uint32_t cw = own + (next_m ? m : 0u);
            const bool thru = act && ent >= hi;
            const uint32_t rex = tm.from(thru ? ent : ex, last);
            uint32_t total = 0;
            const uint64_t o = written + tm.scan(cw, total);
            uint32_t len = cw;
            if (o >= static_cast<uint64_t>(cnt))
                len = 0;
            else if (o + len > static_cast<uint64_t>(cnt))
                len = static_cast<uint32_t>(cnt - o);  // only a corrupt chunk holds more symbols than cnt
            if (len > 0) {
                if (skip + cw > static_cast<uint32_t>(kWsStage)) {  // more than the staging area holds
                    // from the slice's entry to where the next slice starts
                    uint32_t lim = hi;
                    if (next_m) lim = hi + nt.pos[met * L + 1];
                    s.start(payload, nbytes, entry + ent);
                    uint32_t rp = ent;
                    int n2 = 0, b2 = -1;
                    ws_walk<true, false, L>(s, payload, nbytes, T, rp, lo, lim, nullptr, nt, n2, b2, dst0 + o, len);
                } else {
                    ws_copy(stg, skip, len, dst0 + o);
                }
            }
            written += total;
            entry += rex;
            tm.sync();  // the notes and areas are reused by the next round
        }
        if (tl == 0 && (written != static_cast<uint64_t>(cnt) || entry != end)) set_status(status, HUFF_ERR_CORRUPT_STREAM);
    }
    if (bad) set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

// The byte-stream decode's mode: 0, one lane per chunk; -1, a CTA per chunk
// with three walks per slice (the split decode above); otherwise TW, a team
// of TW warps per chunk.
// One lane per chunk from kWsMaxPerSm chunks per SM.  Below, teams: the
// fewest warps per team that leave at most about a tenth of the teams
// without a chunk, provided a chunk is at least kWsMinRounds rounds of the
// team (a round costs the same however few slices have bits); otherwise one
// lane per chunk from 256 chunks per SM, the split decode below that.
// Measured (CUDA events, one call): the 16 GiB sweep (fixed codebook) at
// 1 MiB chunks (108 per SM) 231 GB/s with a warp per chunk against 97 with
// the split decode, at 256 KiB (431 per SM) 238 against 146 with one lane per
// chunk, at 128 KiB (862 per SM) 237 against 258; 1024 chunks (6.7 per SM): 1 GiB of
// the sweep at 1 MiB chunks 161 to 183 GB/s with teams of 4 to 28 warps
// against 98 split, 256 MiB of N(0, 8) bytes at 256 KiB 281 (4 warps)
// against 222 split, 64 MiB at 64 KiB (9 rounds of 4 warps) 227 against 214
// split, 16 MiB at 16 KiB (2.3 rounds) 130 against 161 split; 64 chunks of
// 16 KiB: 45 us with teams of 14 or 28 warps against 37 split.
constexpr size_t kWsMaxPerSm = 768;
constexpr size_t kWsMinRounds = 4;
__host__ int u8_mode(size_t n_chunks, size_t chunk, int sms) {
    if (n_chunks >= static_cast<size_t>(sms) * kWsMaxPerSm) return 0;
    int tw = kWsWarps;
    for (int d : {1, 2, 4, 7, 14})
        if (10 * static_cast<size_t>(sms) * (kWsWarps / d) <= 11 * n_chunks) {
            tw = d;
            break;
        }
    if (chunk >= kWsMinRounds * static_cast<size_t>(tw) * 32 * kWsTarget) return tw;
    return n_chunks >= static_cast<size_t>(sms) * 256 ? 0 : -1;
}

// Threads per chunk for the split decode, or 0 when one lane per chunk fills the GPU.
__host__ int split_threads(size_t n_chunks, size_t chunk, int sms) {
    // the split decode walks every slice three times, so it pays where one lane per chunk would leave the
    // SMs with fewer than about a third of the lanes they need to run at full rate (several hundred); it
    // takes the chunks too small for a team of warps (u8_mode)
    const size_t lanes = static_cast<size_t>(sms) * 256;
    if (n_chunks >= lanes) return 0;
    size_t t = (4 * lanes + n_chunks - 1) / n_chunks;     // about 1024 threads per SM in all
    t = (t + 31) / 32 * 32;
    const size_t by_syms = chunk / kSplitMinSyms / 32 * 32;  // slices of kSplitMinSyms symbols at least
    if (t > by_syms) t = by_syms;
    if (t > 1024) t = 1024;
    if (t < 32) t = 32;
    return static_cast<int>(t);
}

// ------------------------------------------------------------------ fused bf16
//
// One lane per chunk pair decodes both planes into two rings (128 bytes per
// lane: the high ring in the half given by the lane's parity, the low ring in
// the other; each ring's two 32-byte halves swapped on every second lane
// pair), then the warp merges 8 lanes' segments per pass: bytes to 16-bit
// words, XOR x0, 16-byte streaming stores.
//
// Three cases, each its own kernel (ZR), so that each keeps its own register
// allocation: 0, the high plane decoded by table lookups (or both planes
// stepped together, PAIR); 1, the high plane has a 1-bit code and is decoded
// as runs; 2, the same with x0 staged in shared memory: each lane copies its
// chunk's next 64 bytes of x0 (one segment) with four asynchronous 16-byte
// copies (cp.async, no registers held) right after the merge that used the
// previous ones, so the merge finds x0 waiting instead of waiting for it (it
// is read a segment's decode after its copies were issued).  The run-decoded
// cases carry the high plane's run tables (no window table) and the low
// plane's split table with a smaller secondary table, which is what leaves
// room for the staging area of up to 896 lanes.
constexpr int kStageLane = kSeg * 2;  // bytes of x0 per lane per segment

template <bool XOR, bool PAIR, int ZR, class TH, class TL>
__device__ __forceinline__ void decode_bf16_body(const TH &Th, const TL &Tl, uint8_t *rings_base, uint8_t *stage_base,
                                                 const uint8_t *__restrict__ pay_hi,
                                                 size_t bytes_hi, const uint64_t *__restrict__ off_hi,
                                                 const uint8_t *__restrict__ pay_lo, size_t bytes_lo,
                                                 const uint64_t *__restrict__ off_lo, size_t n, size_t chunk,
                                                 const uint16_t *__restrict__ x0, uint16_t *__restrict__ out,
                                                 int32_t *status) {
    constexpr bool zrun = ZR >= 1;
    constexpr bool stage = ZR == 2 && XOR;
    const int lane = threadIdx.x & 31;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t c0 = c - lane;
    uint64_t sh = 0, eh = 0, sl = 0, el = 0;
    int cnt = 0;
    if (c < n_chunks) {
        const size_t first = c * chunk;
        const int want = static_cast<int>(n - first < chunk ? n - first : chunk);
        if (chunk_bounds(off_hi, c, bytes_hi, want, sh, eh) && chunk_bounds(off_lo, c, bytes_lo, want, sl, el))
            cnt = want;
        else
            set_status(status, HUFF_ERR_CORRUPT_STREAM);
    }
    uint8_t *rings = rings_base + static_cast<size_t>(threadIdx.x - lane) * (2 * kRing);
    uint8_t *hring = rings + lane * (2 * kRing) + ((lane & 1) ? kRing : 0);
    uint8_t *lring = rings + lane * (2 * kRing) + ((lane & 1) ? 0 : kRing);
    const uint32_t swz = (lane & 2) ? kRing / 2 : 0;
    PlaneDec h, l;
    plane_start(h, pay_hi, bytes_hi, sh, cnt);
    plane_start(l, pay_lo, bytes_lo, sl, cnt);
    bool bad = false;
    const int warp_cnt = __reduce_max_sync(0xffffffffu, cnt);
    const bool whole = __all_sync(0xffffffffu, cnt == warp_cnt);  // every chunk of the warp has the same length
    // a high plane with a 1-bit code is decoded as runs into a ring that holds that code's symbol
    const uint2 run2 = make_uint2(static_cast<uint32_t>(Th.run), static_cast<uint32_t>(Th.run >> 32));
    if (zrun) {
#pragma unroll
        for (int k = 0; k < kRing; k += 8) *reinterpret_cast<uint2 *>(hring + k) = run2;
    }
    // x0 staging (warp-uniform): the warp's 2 KiB area, lane q's chunk at 64 q (32-bit shared addresses),
    // filled by each lane's own asynchronous 16-byte copies; xf: staging in use
    const uint32_t xst = stage ? smem_u32(stage_base) + (threadIdx.x - lane) * kStageLane : 0u;
    // (a warp past the last chunk has every count 0 and is whole too: it stages nothing; inside the
    // full-segment merge below, where warp_cnt >= kSeg, xf is exactly `stage`)
    const bool xf = stage && whole && warp_cnt >= kSeg;
    const auto stage_issue = [&](int seg) {  // x0 of segment [seg, seg + kSeg) of this lane's chunk
        const uint16_t *src = x0 + c * chunk + seg;
#pragma unroll
        for (int k = 0; k < kStageLane / 16; ++k)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(xst + lane * kStageLane + 16 * k),
                         "l"(src + 8 * k)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (xf) stage_issue(0);
    for (int seg0 = 0; seg0 < warp_cnt; seg0 += kSeg) {
        if (XOR && !xf && seg0 < cnt && (seg0 & 63) == 0) {  // one 128-byte line of x0 per two segments
            const uint16_t *xp = x0 + c * chunk + seg0;
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(xp));
        }
        const int need = min(cnt, seg0 + kSeg);
        if constexpr (PAIR) {
            fill_pair<kRing>(h, l, pay_hi, bytes_hi, pay_lo, bytes_lo, Th, Tl, hring, lring, swz, cnt, need, seg0 + kRing,
                             bad);
        } else {
            // the high plane as runs (ZR >= 1) or by three-lookup steps (ZR == 0: no 1-bit code, the kernel's
            // case); the low plane by three-lookup steps in every case (a 1-bit code there is decoded correctly
            // by its table entries, only without the run shortcut), so each kernel holds one fill loop per plane
            if constexpr (zrun)
                fill_zrun<kRing>(h, pay_hi, bytes_hi, Th, hring, swz, cnt, need, seg0 + kRing, bad);
            else
                fill_segment_t<kRing, false, 12, false, kSecMax, true, false>(h, pay_hi, bytes_hi, Th, hring, swz, cnt,
                                                                            need, seg0 + kRing, bad);
            fill_segment_t<kRing, false, 13, false, zrun ? kSecRun : kSecMax, true, true>(l, pay_lo, bytes_lo, Tl, lring,
                                                                                         swz, cnt, need, seg0 + kRing,
                                                                                         bad);
        }
        __syncwarp();
        if (whole && seg0 + kSeg <= warp_cnt) {
            // every lane's segment is complete: no per-lane bounds
            const size_t g0 = (c0 + (lane >> 2)) * chunk + seg0 + 8 * (lane & 3);  // pass i: + 8 i chunk
            const size_t gs = 8 * chunk;
            const int q0 = lane >> 2;
            uint4 xv[4];
            if constexpr (stage) {  // whole: the staging is in use (xf)
                // this lane's copies have landed (issued a segment's decode ago); then every lane's
                asm volatile("cp.async.wait_all;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(xv[i].x), "=r"(xv[i].y), "=r"(xv[i].z), "=r"(xv[i].w)
                                 : "r"(xst + (8 * i + q0) * kStageLane + 16 * (lane & 3))
                                 : "memory");
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    xv[i] = XOR ? __ldcs(reinterpret_cast<const uint4 *>(x0 + g0 + i * gs)) : make_uint4(0, 0, 0, 0);
            }
            const uint32_t o = ((seg0 + 8 * (lane & 3)) & (kRing - 1)) ^ ((q0 & 2) ? kRing / 2 : 0);
            uint8_t *hr = rings + q0 * (2 * kRing) + ((q0 & 1) ? kRing : 0) + o;
            const uint8_t *lr = rings + q0 * (2 * kRing) + ((q0 & 1) ? 0 : kRing) + o;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint2 hv = *reinterpret_cast<const uint2 *>(hr + i * 8 * (2 * kRing));
                const uint2 lv = *reinterpret_cast<const uint2 *>(lr + i * 8 * (2 * kRing));
                if (zrun) *reinterpret_cast<uint2 *>(hr + i * 8 * (2 * kRing)) = run2;
                uint4 v = make_uint4(__byte_perm(lv.x, hv.x, 0x5140), __byte_perm(lv.x, hv.x, 0x7362),
                                     __byte_perm(lv.y, hv.y, 0x5140), __byte_perm(lv.y, hv.y, 0x7362));
                v.x ^= xv[i].x;
                v.y ^= xv[i].y;
                v.z ^= xv[i].z;
                v.w ^= xv[i].w;
                __stcs(reinterpret_cast<uint4 *>(out + g0 + i * gs), v);
            }
            if (stage && seg0 + 2 * kSeg <= warp_cnt) {
                // every lane has read its staged x0 (the values fed the stores above): refill the area
                __syncwarp();
                stage_issue(seg0 + kSeg);
            }
        } else {
            // merge: 8 lanes' segments per pass, 8 elements (16 output bytes) per lane; the four passes'
            // x0 loads are issued together, ahead of the shared-memory reads
            uint4 xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int q = 8 * i + (lane >> 2);
                const int e0 = seg0 + 8 * (lane & 3);
                xv[i] = make_uint4(0, 0, 0, 0);
                if (XOR && e0 + 8 <= __shfl_sync(0xffffffffu, cnt, q))
                    xv[i] = __ldcs(reinterpret_cast<const uint4 *>(x0 + (c0 + q) * chunk + e0));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int q = 8 * i + (lane >> 2);  // source lane
                const int e0 = seg0 + 8 * (lane & 3);
                const int cs = __shfl_sync(0xffffffffu, cnt, q);
                if (e0 < cs) {
                    uint8_t *qr = rings + q * (2 * kRing);
                    const uint32_t o = (e0 & (kRing - 1)) ^ ((q & 2) ? kRing / 2 : 0);
                    const uint2 hv = *reinterpret_cast<const uint2 *>(qr + ((q & 1) ? kRing : 0) + o);
                    const uint2 lv = *reinterpret_cast<const uint2 *>(qr + ((q & 1) ? 0 : kRing) + o);
                    if (zrun) *reinterpret_cast<uint2 *>(qr + ((q & 1) ? kRing : 0) + o) = run2;
                    uint4 v = make_uint4(__byte_perm(lv.x, hv.x, 0x5140), __byte_perm(lv.x, hv.x, 0x7362),
                                         __byte_perm(lv.y, hv.y, 0x5140), __byte_perm(lv.y, hv.y, 0x7362));
                    const size_t g = (c0 + q) * chunk + e0;  // first element of this group
                    if (e0 + 8 <= cs) {  // x0 and out are 16-byte aligned, chunk a multiple of 32
                        v.x ^= xv[i].x;
                        v.y ^= xv[i].y;
                        v.z ^= xv[i].z;
                        v.w ^= xv[i].w;
                        __stcs(reinterpret_cast<uint4 *>(out + g), v);
                    } else {
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (e0 + k < cs) {
                                uint16_t val = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
                                if (XOR) val ^= x0[g + k];
                                out[g + k] = val;
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
    if (cnt > 0 && (bad || h.pos() != off_hi[c + 1] || l.pos() != off_lo[c + 1]))
        set_status(status, HUFF_ERR_CORRUPT_STREAM);
}

// Shared memory of each case for a block of `block` lanes.
__host__ size_t bf16_smem(int zr, int block) {
    const size_t b = static_cast<size_t>(block);
    if (zr == 0) return kBf16Tables + b * (2 * kRing);
    const size_t s = kBf16RunTables + b * (2 * kRing);
    return zr == 1 ? s : s + b * kStageLane;
}

// ZR (with one lane per chunk pair): 1 and 2 decode streams whose high plane
// has a 1-bit code (as runs; 2 stages x0), 0 those without.  Two kernels are
// launched, one after the other (0 and 1 or 2); the one whose case does not
// hold returns at once (the host cannot read the codebook).
template <bool XOR, bool PAIR, int ZR>
__global__ void __launch_bounds__(PAIR ? kPairBlock : kMaxBlock, 1) k_decode_bf16(
    const uint8_t *__restrict__ pay_hi, size_t bytes_hi, const uint64_t *__restrict__ off_hi,
    const uint8_t *__restrict__ pay_lo, size_t bytes_lo, const uint64_t *__restrict__ off_lo, size_t n,
    size_t chunk, const huff_codebook *__restrict__ cb_hi, const huff_codebook *__restrict__ cb_lo,
    const uint16_t *__restrict__ x0, uint16_t *__restrict__ out, int32_t *status) {
    if (!PAIR) {
        const bool has_run = cb_hi->magic == HUFF_CODEBOOK_MAGIC && cb_hi->longest <= HUFF_MAX_LEN &&
                             cb_hi->bl_count[1] > 0;
        if (has_run != (ZR >= 1)) return;  // the other kernel's case
    }
    extern __shared__ __align__(16) uint8_t dsm[];
    if constexpr (ZR >= 1) {
        // high plane: run tables; low plane: a 13-bit table with a smaller secondary table
        RunTables &Th = *reinterpret_cast<RunTables *>(dsm);
        LoTablesRun &Tl = *reinterpret_cast<LoTablesRun *>(dsm + sizeof(RunTables));
        load_run_tables(Th, cb_hi);
        load_table_a(Tl, cb_lo);
        __syncthreads();
        load_table_b(Tl, cb_lo);
        __syncthreads();
        if (!Th.ok || !Tl.ok) {
            if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
            return;
        }
        uint8_t *rings = dsm + kBf16RunTables;
        uint8_t *stage = rings + static_cast<size_t>(blockDim.x) * (2 * kRing);
        decode_bf16_body<XOR, PAIR, ZR>(Th, Tl, rings, stage, pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo,
                                        n, chunk, x0, out, status);
    } else {
        // high plane: the codebook's 12-bit table; low plane: a 13-bit table
        DecTables<12> &Th = *reinterpret_cast<DecTables<12> *>(dsm);
        LoTables &Tl = *reinterpret_cast<LoTables *>(dsm + sizeof(DecTables<12>));
        load_table_a(Th, cb_hi);
        load_table_a(Tl, cb_lo);
        __syncthreads();
        load_table_b(Th, cb_hi);
        load_table_b(Tl, cb_lo);
        __syncthreads();
        if (!Th.ok || !Tl.ok) {
            if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, HUFF_ERR_INVALID_CODEBOOK);
            return;
        }
        decode_bf16_body<XOR, PAIR, 0>(Th, Tl, dsm + kBf16Tables, nullptr, pay_hi, bytes_hi, off_hi, pay_lo,
                                       bytes_lo, off_lo, n, chunk, x0, out, status);
    }
}

}  // namespace

// The most lanes per block (whole warps, at most kMaxBlock) whose decode fits
// in max_smem bytes of shared memory: with an XOR delta, the fused bf16
// decode's case with x0 staged; without, every other case.
int decode_lanes(int max_smem, bool delta) {
    const auto need = [delta](int b) {
        if (delta) return bf16_smem(2, b);
        const size_t u8 = sizeof(U8Tables) + static_cast<size_t>(b) * kRingU8;
        return std::max(std::max(bf16_smem(0, b), bf16_smem(1, b)), u8);
    };
    int b = kMaxBlock;
    while (b > 32 && need(b) > static_cast<size_t>(max_smem)) b -= 32;
    return b;
}

// Measured on the 16 GiB sweep (blocks of 896 consecutive chunks lie in one 256 MiB segment), GB/s:
// at 128 KiB chunks (one wave) spread blocks 258, ranked ranges 234, consecutive 234; at 64 KiB (1.93
// waves) ranked 273, spread 265, consecutive 246; at 16 KiB (7.7 waves) ranked 346, consecutive 335,
// spread 268 (each spread block waits for its slowest warp).  Ranking costs each block a pass over the
// launch's block ranges, hence its limit.
constexpr int kSpreadWaves = 1;
constexpr unsigned kRankBlocks = 2048;
constexpr size_t kRankChunk = 4096;

int launch_decode_u8(const uint8_t *payload, size_t bytes, const uint64_t *off, size_t n, size_t chunk,
                     const huff_codebook *cb, uint8_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const int sms = dev_info().sms;
    const int tw = u8_mode(n_chunks, chunk, sms);
    if (tw < 0) {
        const int split = split_threads(n_chunks, chunk, sms);
        const size_t smem = (static_cast<size_t>(split) + 32) * sizeof(uint64_t) + sizeof(SplitTab);
        k_decode_u8_split<<<static_cast<unsigned>(n_chunks), split, smem, s>>>(payload, bytes, off, n, chunk, cb, out,
                                                                              status);
        return launch_status();
    }
    const size_t teams = static_cast<size_t>(kWsWarps / (tw > 0 ? tw : 1));  // per CTA
    const unsigned grid = static_cast<unsigned>(std::min<size_t>(sms, (n_chunks + teams - 1) / teams));
    const auto ws = [&](auto kern, size_t smem) -> int {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return HUFF_ERR_CUDA;
        kern<<<grid, kWsWarps * 32, smem, s>>>(payload, bytes, off, n, chunk, cb, out, status);
        return launch_status();
    };
    switch (tw) {
        case 1: return ws(k_decode_u8_ws<1>, ws_smem<1>());
        case 2: return ws(k_decode_u8_ws<2>, ws_smem<2>());
        case 4: return ws(k_decode_u8_ws<4>, ws_smem<4>());
        case 7: return ws(k_decode_u8_ws<7>, ws_smem<7>());
        case 14: return ws(k_decode_u8_ws<14>, ws_smem<14>());
        case 28: return ws(k_decode_u8_ws<28>, ws_smem<28>());
        default: break;
    }
    const int block = decode_block(n_chunks, sms);
    const unsigned blocks = static_cast<unsigned>((n_chunks + block - 1) / block);
    // blocks take spread chunks when they run in at most kSpreadWaves waves, ranges by rank up to
    // kRankBlocks blocks of chunks of at least kRankChunk symbols (a block's ranking pass then costs
    // under 1 % of its decode)
    const int spread = blocks <= static_cast<unsigned>(kSpreadWaves * sms)
                           ? 1
                           : (blocks <= kRankBlocks && chunk >= kRankChunk ? 2 : 0);
    const size_t smem = sizeof(U8Tables) + static_cast<size_t>(block) * kRingU8 +
                        (spread == 2 ? static_cast<size_t>(blocks) * 8 + 16 : 0);
    if (cudaFuncSetAttribute(k_decode_u8, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return HUFF_ERR_CUDA;
    k_decode_u8<<<blocks, block, smem, s>>>(payload, bytes, off, n, chunk, cb, out, status, spread);
    return launch_status();
}

int launch_decode_bf16(const uint8_t *pay_hi, size_t bytes_hi, const uint64_t *off_hi, const uint8_t *pay_lo,
                       size_t bytes_lo, const uint64_t *off_lo, size_t n, size_t chunk,
                       const huff_codebook *cb_hi, const huff_codebook *cb_lo, const uint16_t *x0,
                       uint16_t *out, int32_t *status, cudaStream_t s) {
    if (n == 0) return HUFF_OK;
    const size_t n_chunks = (n + chunk - 1) / chunk;
    const DevInfo d = dev_info();
    const int block = decode_block(n_chunks, d.sms);
    const unsigned grid = static_cast<unsigned>((n_chunks + block - 1) / block);
    const auto go = [&](auto kern, int zr, const uint16_t *x) -> int {
        const size_t smem = bf16_smem(zr, block);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return HUFF_ERR_CUDA;
        kern<<<grid, block, smem, s>>>(pay_hi, bytes_hi, off_hi, pay_lo, bytes_lo, off_lo, n, chunk, cb_hi, cb_lo, x,
                                       out, status);
        return cudaGetLastError() == cudaSuccess ? HUFF_OK : HUFF_ERR_CUDA;
    };
    // few lanes per SM: both planes stepped in one loop; otherwise the kernels of the high plane's two
    // cases (with and without a 1-bit code), of which one returns at once; with x0, the run case stages
    // x0 in shared memory when the block's staging area fits
    const bool pair = block <= kPairBlock;
    int st;
    if (x0 != nullptr) {
        if (pair) {
            st = go(k_decode_bf16<true, true, 0>, 0, x0);
        } else {
            const bool fits = bf16_smem(2, block) <= static_cast<size_t>(d.max_smem_optin);
            st = fits ? go(k_decode_bf16<true, false, 2>, 2, x0) : go(k_decode_bf16<true, false, 1>, 1, x0);
            if (st == HUFF_OK) st = go(k_decode_bf16<true, false, 0>, 0, x0);
        }
    } else {
        if (pair) {
            st = go(k_decode_bf16<false, true, 0>, 0, nullptr);
        } else {
            st = go(k_decode_bf16<false, false, 1>, 1, nullptr);
            if (st == HUFF_OK) st = go(k_decode_bf16<false, false, 0>, 0, nullptr);
        }
    }
    return st;
}

}  // namespace huffk
