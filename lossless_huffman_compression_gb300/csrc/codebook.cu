// codebook.cu -- code lengths, canonical codes and decode tables, one CTA.
//
// "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
// Methodology step 3: the Huffman codebook is built once from the averaged
// distribution.  "Lossless Compression for LLM Tensor Incremental Snapshots"
// (arXiv 2505.09810), key design 2: efficient Huffman tree construction.
//
// The pages fix neither the tie-break nor a length limit nor how codes are
// assigned; the rule implemented here is:
//   (count, id) order with leaves id = symbol and new nodes 256, 257, ...;
//   ITU-T T.81 Annex K.3 Adjust_BITS repair down to max_len (no reserved
//   code); lengths handed out again by (count desc, symbol asc);
//   RFC 1951 3.2.2 canonical codes.
//
// GPU design: 256 threads, one per symbol.  The present symbols are ranked by
// (count, symbol) with an all-pairs comparison (256 x 256 compares spread over
// the block), which turns Huffman's procedure into the two-queue form: sorted
// leaves plus a FIFO of new nodes, whose counts come out non-decreasing with
// increasing ids, so the FIFO is itself in (count, id) order and every step
// takes the same two nodes as a (count, id) heap would.  The 255 joins are
// inherently serial and run on one thread (a few microseconds, once per
// codebook); depths, counting, reassignment, code assignment and the 4096
// entry decode table are spread over the block.
#include "common.cuh"

namespace huffk {

namespace {

constexpr int kT = 256;

// Codes, ranks, decode tables and the header from 256 lengths in shared
// memory.  Requires every length <= max_len <= 24.
__device__ void finish_codebook(const uint8_t *lens, int max_len, huff_codebook *cb, int32_t *status) {
    __shared__ uint32_t blc[34];
    __shared__ uint32_t fc[34];
    __shared__ uint32_t fi[34];
    __shared__ uint8_t srt[256];
    __shared__ int s_bad, s_nsym, s_longest;
    const int t = threadIdx.x;
    if (t < 34) blc[t] = 0;
    if (t == 0) {
        s_bad = 0;
        s_longest = 0;
    }
    srt[t] = 0;
    __syncthreads();
    const int L = lens[t];
    if (L > 0) {
        atomicAdd(&blc[L], 1u);
        atomicMax(&s_longest, L);
    }
    __syncthreads();
    if (t == 0) {
        uint64_t code = 0;
        uint32_t idx = 0;
        blc[0] = 0;
        fc[0] = 0;
        fi[0] = 0;
        for (int l = 1; l <= 32; ++l) {
            code = (code + blc[l - 1]) << 1;
            fc[l] = static_cast<uint32_t>(code);
            fi[l] = idx;
            idx += blc[l];
            if (blc[l] > 0 && code + blc[l] > (1ull << l)) s_bad = 1;  // over-subscribed
        }
        s_nsym = static_cast<int>(idx);
    }
    __syncthreads();
    if (s_bad) {
        if (t == 0) {
            cb->magic = 0;
            set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        }
        return;
    }
    uint32_t code = 0;
    if (L > 0) {
        uint32_t r = 0;
        for (int u = 0; u < t; ++u) r += (lens[u] == L);
        code = fc[L] + r;
        srt[fi[L] + r] = static_cast<uint8_t>(t);
    }
    cb->len[t] = static_cast<uint8_t>(L);
    cb->code[t] = code;
    if (t < 32) {
        cb->bl_count[t] = blc[t];
        cb->first_code[t] = fc[t];
        cb->first_index[t] = fi[t];
    }
    __syncthreads();
    cb->sorted_symbols[t] = srt[t];
    // first-level decode table: entry i lists the codes that lie wholly inside the 12-bit window i,
    // greedily from its first bit, at most HUFF_LUT_SYMS: symbols (8 bits each, first in the low
    // byte), their count << 48 and their total length << 52; 0 when the first code is longer than 12 bits.
    // Built in two passes: first the code that starts each window (its symbol and length, 0 when it
    // is longer than 12 bits), then each entry as a chain through that table: after pos bits, the
    // window shifted left by pos (zeros behind) starts with the next code exactly when that code's
    // length is at most 12 - pos, since then all its bits are real bits of the window.
    __shared__ uint16_t first_code_of[1 << HUFF_LUT_BITS];  // symbol | length << 8
    for (int i = t; i < (1 << HUFF_LUT_BITS); i += kT) {
        uint32_t e = 0;
        for (uint32_t l = 1; l <= HUFF_LUT_BITS; ++l) {
            const uint32_t c = static_cast<uint32_t>(i) >> (HUFF_LUT_BITS - l);
            if (blc[l] > 0 && c >= fc[l] && c - fc[l] < blc[l]) {
                e = srt[fi[l] + (c - fc[l])] | (l << 8);
                break;
            }
        }
        first_code_of[i] = static_cast<uint16_t>(e);
    }
    __syncthreads();
    for (int i = t; i < (1 << HUFF_LUT_BITS); i += kT) {
        uint64_t syms = 0;
        uint32_t count = 0, pos = 0;
        while (count < HUFF_LUT_SYMS) {
            const uint32_t e = first_code_of[(static_cast<uint32_t>(i) << pos) & ((1u << HUFF_LUT_BITS) - 1u)];
            const uint32_t l = e >> 8;
            if (l == 0 || l + pos > HUFF_LUT_BITS) break;
            syms |= static_cast<uint64_t>(e & 0xffu) << (8 * count);
            ++count;
            pos += l;
        }
        cb->lut[i] = count ? (syms | (static_cast<uint64_t>(count) << 48) | (static_cast<uint64_t>(pos) << 52)) : 0ull;
    }
    __syncthreads();
    if (t == 0) {
        cb->max_len = max_len;
        cb->n_symbols = s_nsym;
        cb->longest = s_longest;
        __threadfence();
        cb->magic = HUFF_CODEBOOK_MAGIC;
    }
}

// One CTA per codebook: CTA b builds cbs[b] from hists[256 b .. 256 b + 255].
__global__ void __launch_bounds__(kT) k_build_codebook(const uint64_t *__restrict__ hists, int max_len,
                                                       unsigned flags, huff_codebook *__restrict__ cbs,
                                                       int32_t *status, const uint32_t *__restrict__ when) {
    if (when != nullptr && *when == 0) return;  // conditional rebuild: the codebook stays as it is
    const uint64_t *hist = hists + 256 * static_cast<size_t>(blockIdx.x);
    huff_codebook *cb = cbs + blockIdx.x;
    __shared__ uint64_t cnt[256];
    __shared__ uint64_t leaf_cnt[256];
    __shared__ uint64_t int_cnt[256];
    __shared__ uint16_t leaf_parent[256];
    __shared__ uint16_t int_parent[256];
    __shared__ uint16_t int_depth[256];
    __shared__ uint32_t bl[260];
    __shared__ uint8_t lens[256];
    __shared__ int s_maxdepth, s_fail;

    const int t = threadIdx.x;
    uint64_t c = hist[t];
    if ((flags & HUFF_COVER_ALL) && c == 0) c = 1;
    cnt[t] = c;
    int_cnt[t] = 0;
    bl[t] = 0;
    if (t < 4) bl[256 + t] = 0;
    lens[t] = 0;
    if (t == 0) {
        s_maxdepth = 0;
        s_fail = 0;
    }
    const int m = __syncthreads_count(c > 0);

    if (m >= 2) {
        // rank of each present symbol by (count asc, symbol asc)
        if (c > 0) {
            int r = 0;
            for (int u = 0; u < 256; ++u) {
                const uint64_t cu = cnt[u];
                r += (cu > 0) && (cu < c || (cu == c && u < t));
            }
            leaf_cnt[r] = c;
        }
        __syncthreads();
        {
            // the counts must sum below 2^63 so that no node count can overflow: sum the high and
            // low 32-bit halves separately (no overflow in either), then compare
            uint64_t h = c >> 32, l = c & 0xffffffffull;
            for (int o = 16; o > 0; o >>= 1) {
                h += __shfl_xor_sync(0xffffffffu, h, o);
                l += __shfl_xor_sync(0xffffffffu, l, o);
            }
            if ((t & 31) == 0) {
                atomicAdd(reinterpret_cast<unsigned long long *>(&int_cnt[0]), static_cast<unsigned long long>(h));
                atomicAdd(reinterpret_cast<unsigned long long *>(&int_cnt[1]), static_cast<unsigned long long>(l));
            }
        }
        __syncthreads();
        if (t == 0 && int_cnt[0] + (int_cnt[1] >> 32) >= (1ull << 31)) s_fail = 1;
        __syncthreads();
        if (s_fail) {
            if (t == 0) {
                cb->magic = 0;
                set_status(status, HUFF_ERR_INVALID_CODEBOOK);
            }
            return;
        }
        if (t == 0) {
            // two-queue Huffman: leaves (sorted) against new nodes (FIFO); a leaf wins a count tie.
            // The heads of both queues and the entries behind them sit in registers (an empty slot
            // holds kNone, above every count), so the next shared-memory load is one pop ahead of
            // its use and the serial chain is compares and adds.
            constexpr uint64_t kNone = ~0ull;
            int li = 0, ii = 0;
            uint64_t l0 = leaf_cnt[0], l1 = m > 1 ? leaf_cnt[1] : kNone;
            uint64_t i0 = kNone, i1 = kNone;
            for (int k = 0; k < m - 1; ++k) {
                uint64_t sum = 0;
#pragma unroll
                for (int pick = 0; pick < 2; ++pick) {
                    if (l0 <= i0) {  // l0 < kNone here: at least two nodes are left in all
                        leaf_parent[li] = static_cast<uint16_t>(k);
                        sum += l0;
                        ++li;
                        l0 = l1;
                        l1 = li + 1 < m ? leaf_cnt[li + 1] : kNone;
                    } else {
                        int_parent[ii] = static_cast<uint16_t>(k);
                        sum += i0;
                        ++ii;
                        i0 = i1;
                        i1 = ii + 1 < k ? int_cnt[ii + 1] : kNone;
                    }
                }
                int_cnt[k] = sum;
                // the new node joins the queue: as its head or right behind it
                if (ii == k) i0 = sum;
                else if (ii + 1 == k) i1 = sum;
            }
        }
        __syncthreads();
        {
            // depths of new nodes by pointer jumping: the root is node m - 2 (its own ancestor, depth 0);
            // after round r a node's depth counts its first 2^r ancestors and anc skips to the next ones
            __shared__ uint16_t anc[256];
            const int k = t;
            uint32_t dk = 0, ak = 0;
            if (k < m - 1) {
                ak = k == m - 2 ? static_cast<uint32_t>(k) : int_parent[k];
                dk = k == m - 2 ? 0u : 1u;
                int_depth[k] = static_cast<uint16_t>(dk);
                anc[k] = static_cast<uint16_t>(ak);
            }
            __syncthreads();
            for (int r = 0; r < 8; ++r) {  // 2^8 >= 255 ancestors
                uint32_t nd = dk, na = ak;
                if (k < m - 1) {
                    nd = dk + int_depth[ak];
                    na = anc[ak];
                }
                __syncthreads();
                if (k < m - 1) {
                    dk = nd;
                    ak = na;
                    int_depth[k] = static_cast<uint16_t>(dk);
                    anc[k] = static_cast<uint16_t>(ak);
                }
                __syncthreads();
            }
        }
        if (t < m) {
            const int d = int_depth[leaf_parent[t]] + 1;
            atomicAdd(&bl[d], 1u);
            atomicMax(&s_maxdepth, d);
        }
        __syncthreads();
        if (t == 0 && s_maxdepth > max_len) {
            // Adjust_BITS, largest over-long depth first; each move keeps the Kraft sum at 1
            for (int i = s_maxdepth; i > max_len; --i) {
                while (bl[i] > 0) {
                    int j = i - 2;
                    while (j > 0 && bl[j] == 0) --j;
                    if (j <= 0) {
                        s_fail = 1;
                        break;
                    }
                    bl[i] -= 2;
                    bl[i - 1] += 1;
                    bl[j + 1] += 2;
                    bl[j] -= 1;
                }
                if (s_fail) break;
            }
        }
        __syncthreads();
        if (s_fail) {
            if (t == 0) {
                cb->magic = 0;
                set_status(status, HUFF_ERR_INVALID_CODEBOOK);
            }
            return;
        }
        // hand the lengths out again by (count desc, symbol asc)
        if (c > 0) {
            int r = 0;
            for (int u = 0; u < 256; ++u) {
                const uint64_t cu = cnt[u];
                r += (cu > 0) && (cu > c || (cu == c && u < t));
            }
            uint32_t cum = 0;
            for (int L = 1; L <= max_len; ++L) {
                cum += bl[L];
                if (static_cast<uint32_t>(r) < cum) {
                    lens[t] = static_cast<uint8_t>(L);
                    break;
                }
            }
        }
    } else if (m == 1) {
        if (c > 0) lens[t] = 1;
    }
    __syncthreads();
    finish_codebook(lens, max_len, cb, status);
}

// Drift of a shard against the codebook in use (P1 Limitations: a fixed
// codebook degrades when the distribution drifts; refreshing it is P1's
// future work).  The shard costs T = sum h * len bits under the codebook;
// its own entropy bounds any code from below by n H bits, and a Huffman
// code of bytes by n bits (at least one bit per symbol), so the bound is
// B = n max(H, 1).  gap = (T - B) / B; a symbol without a code makes the gap
// infinite; an empty shard has gap 0.  *flag = gap > threshold.
__global__ void __launch_bounds__(kT) k_drift_check(const uint64_t *__restrict__ hist,
                                                    const huff_codebook *__restrict__ cb, double threshold,
                                                    uint32_t *__restrict__ flag, double *__restrict__ gap_out) {
    __shared__ uint64_t s_n[kT / 32], s_bits[kT / 32];
    __shared__ double s_h[kT / 32];
    __shared__ int s_missing;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) s_missing = 0;
    __syncthreads();
    const bool ok = cb->magic == HUFF_CODEBOOK_MAGIC;
    const uint64_t h = hist[t];
    const uint64_t L = ok ? cb->len[t] : 0;
    if (h > 0 && L == 0) s_missing = 1;
    uint64_t n = h, bits = h * L;
    for (int o = 16; o > 0; o >>= 1) {
        n += __shfl_xor_sync(0xffffffffu, n, o);
        bits += __shfl_xor_sync(0xffffffffu, bits, o);
    }
    if (lane == 0) {
        s_n[warp] = n;
        s_bits[warp] = bits;
    }
    __syncthreads();
    uint64_t N = 0, T = 0;
    for (int w = 0; w < kT / 32; ++w) {
        N += s_n[w];
        T += s_bits[w];
    }
    double e = 0.0;  // -p log2 p of this symbol
    if (h > 0) {
        const double p = static_cast<double>(h) / static_cast<double>(N);
        e = -p * log2(p);
    }
    for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
    if (lane == 0) s_h[warp] = e;
    __syncthreads();
    if (t == 0) {
        double H = 0.0;
        for (int w = 0; w < kT / 32; ++w) H += s_h[w];
        double g = 0.0;
        if (s_missing) {
            g = __longlong_as_double(0x7ff0000000000000ll);  // +infinity
        } else if (N > 0) {
            const double B = static_cast<double>(N) * (H > 1.0 ? H : 1.0);
            g = (static_cast<double>(T) - B) / B;
        }
        if (gap_out != nullptr) *gap_out = g;
        *flag = g > threshold ? 1u : 0u;
    }
}

__global__ void __launch_bounds__(kT) k_codebook_from_lengths(int max_len, huff_codebook *__restrict__ cb,
                                                              int32_t *status) {
    __shared__ uint8_t lens[256];
    __shared__ int s_bad;
    const int t = threadIdx.x;
    if (t == 0) s_bad = 0;
    __syncthreads();
    const int L = cb->len[t];
    if (L > max_len) s_bad = 1;
    lens[t] = static_cast<uint8_t>(L);
    __syncthreads();
    if (s_bad) {
        if (t == 0) {
            cb->magic = 0;
            set_status(status, HUFF_ERR_INVALID_CODEBOOK);
        }
        return;
    }
    finish_codebook(lens, max_len, cb, status);
}

}  // namespace

int launch_build_codebook(const uint64_t *hist, int max_len, unsigned flags, huff_codebook *cb,
                          int32_t *status, const uint32_t *when, cudaStream_t s) {
    return launch_build_codebooks(hist, 1, max_len, flags, cb, status, when, s);
}

int launch_build_codebooks(const uint64_t *hists, size_t count, int max_len, unsigned flags, huff_codebook *cbs,
                           int32_t *status, const uint32_t *when, cudaStream_t s) {
    if (count == 0) return HUFF_OK;
    k_build_codebook<<<static_cast<unsigned>(count), kT, 0, s>>>(hists, max_len, flags, cbs, status, when);
    return launch_status();
}

int launch_drift_check(const uint64_t *hist, const huff_codebook *cb, double threshold, uint32_t *flag,
                       double *gap, cudaStream_t s) {
    k_drift_check<<<1, kT, 0, s>>>(hist, cb, threshold, flag, gap);
    return launch_status();
}

int launch_codebook_from_lengths(int max_len, huff_codebook *cb, int32_t *status, cudaStream_t s) {
    k_codebook_from_lengths<<<1, kT, 0, s>>>(max_len, cb, status);
    return launch_status();
}

}  // namespace huffk
