// common.cuh -- device helpers and internal launch interface of libhuff.
//
// Everything here is internal to the library; the public ABI is include/huff.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "huff.h"

namespace huffk {

// ----------------------------------------------------------------- tuning constants
// Counted (per-shard) bf16 path: the histogram pass records each plane's
// counts per segment (at least kDirSegElems elements; count_seg_elems), so
// the encode knows every segment's bit offset before it starts and reads its
// input once.
constexpr size_t kDirSegElems = 131072;          // least bf16 elements per counted segment
constexpr int kSegCountWords = 512;              // [hi 256 | lo 256] per segment
constexpr int kHistThreads = 512;
constexpr int kHistCopies = 32;                  // one histogram copy per lane
constexpr unsigned kSpinLimit = 1u << 20;        // bounded waits (polls) before HUFF_ERR_TIMEOUT

// lookback descriptor: flag in the top two bits, value in the low 62
constexpr uint64_t kFlagAggregate = 1ull << 62;
constexpr uint64_t kFlagPrefix = 2ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;
constexpr uint64_t kTailValid = 1ull << 32;

// ----------------------------------------------------------------- device helpers
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Relaxed (unordered) 64-bit accesses: single-copy atomic, so a descriptor that
// packs its flag with its value needs no acquire/release; independent relaxed
// loads can all be in flight at once.
__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_nc_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t bswap32(uint32_t x) { return __byte_perm(x, 0, 0x0123); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The 8 words have arrived in registers: the shared-memory loads that produced
// them are complete (an empty instruction that consumes them), so a bulk copy
// issued after a barrier cannot overwrite the stage under a pending load.
__device__ __forceinline__ void consumed(const uint32_t (&v)[8]) {
    asm volatile("" ::"r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policies for bulk copies: keep (data read again soon) or drop first (last use).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache-policy hint.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// True once any error is recorded: waits stop early so one failure cannot
// turn into a long chain of per-tile timeouts.
__device__ __forceinline__ bool error_recorded(const int32_t *status) {
    return status != nullptr && *reinterpret_cast<const volatile int32_t *>(status) != 0;
}

// Bounded wait on an mbarrier phase: at most `limit` polls; false when the
// limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned limit = kSpinLimit) {
    for (unsigned i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(32);
    }
    return false;
}

// A warp's copy ring after one of its waits ran out: every lane waits once
// more (bounded) on each stage whose copy may still be in flight (bit s of
// `inflight`), so that the warp does not leave while a bulk copy is still
// writing its shared memory.  Stages before `cstage` in the ring complete in
// the next lap (parity cphase ^ 1), the others in this one.
__device__ __forceinline__ void drain_ring(uint64_t *bar, int stages, uint32_t inflight, uint32_t cstage,
                                           uint32_t cphase) {
    for (int s = 0; s < stages; ++s)
        if (inflight & (1u << s)) mbar_wait(&bar[s], static_cast<uint32_t>(s) < cstage ? cphase ^ 1u : cphase);
}

// ----------------------------------------------------------------- launchers (host)
// Each returns a huff_status; arguments are already validated by the ABI layer.
struct DevInfo {
    int sms;
    int max_smem_optin;
};
DevInfo dev_info();
// Elements per counted segment for n elements on the current device (encode.cu).
size_t count_seg_elems(size_t n);
// Widest decode block that fits in max_smem bytes, with or without an XOR delta (decode.cu).
int decode_lanes(int max_smem, bool delta);

int launch_zero_u64(uint64_t *p, size_t count, cudaStream_t s);
int launch_histogram(const uint8_t *in, size_t n, size_t stride, uint64_t *hist, cudaStream_t s);
int launch_histogram_bf16(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                          uint64_t *hist_lo, cudaStream_t s);
int launch_build_codebook(const uint64_t *hist, int max_len, unsigned flags, huff_codebook *cb,
                          int32_t *status, const uint32_t *when, cudaStream_t s);
int launch_build_codebooks(const uint64_t *hists, size_t count, int max_len, unsigned flags, huff_codebook *cbs,
                           int32_t *status, const uint32_t *when, cudaStream_t s);
int launch_drift_check(const uint64_t *hist, const huff_codebook *cb, double threshold, uint32_t *flag,
                       double *gap, cudaStream_t s);
int launch_codebook_from_lengths(int max_len, huff_codebook *cb, int32_t *status, cudaStream_t s);

size_t enc_u8_seg_tiles(size_t n);
size_t enc_u8_workspace_words(size_t n);
size_t enc_bf16_given_ws_parts(size_t n, size_t *counted_off, size_t *hist_off);
int launch_encode_u8(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk,
                     uint8_t *payload, size_t cap, uint64_t *off, void *ws, int32_t *status,
                     cudaStream_t s);
int launch_encode_u8_noalloc(const uint8_t *in, size_t n, const huff_codebook *cb, size_t chunk,
                             uint8_t *payload, size_t cap, uint64_t *off, int32_t *status, cudaStream_t s);
int launch_histogram_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, uint64_t *hist_hi,
                                  uint64_t *hist_lo, uint32_t *seg_counts, cudaStream_t s);
int launch_encode_bf16_counted(const uint16_t *w, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                               const huff_codebook *cb_lo, size_t chunk, const uint32_t *seg_counts,
                               uint8_t *pay_hi, size_t cap_hi, uint64_t *off_hi, uint8_t *pay_lo, size_t cap_lo,
                               uint64_t *off_lo, void *ws, int32_t *status, cudaStream_t s);
int launch_encode_bf16(const uint16_t *w, const uint16_t *x0, size_t n, const huff_codebook *cb_hi,
                       const huff_codebook *cb_lo, size_t chunk, uint8_t *pay_hi, size_t cap_hi,
                       uint64_t *off_hi, uint8_t *pay_lo, size_t cap_lo, uint64_t *off_lo, void *ws,
                       int32_t *status, cudaStream_t s);
int launch_decode_u8(const uint8_t *payload, size_t bytes, const uint64_t *off, size_t n, size_t chunk,
                     const huff_codebook *cb, uint8_t *out, int32_t *status, cudaStream_t s);
int launch_decode_bf16(const uint8_t *pay_hi, size_t bytes_hi, const uint64_t *off_hi,
                       const uint8_t *pay_lo, size_t bytes_lo, const uint64_t *off_lo, size_t n,
                       size_t chunk, const huff_codebook *cb_hi, const huff_codebook *cb_lo,
                       const uint16_t *x0, uint16_t *out, int32_t *status, cudaStream_t s);
int launch_split(const uint16_t *w, size_t n, uint8_t *hi, uint8_t *lo, cudaStream_t s);
int launch_merge(const uint8_t *hi, const uint8_t *lo, size_t n, uint16_t *w, cudaStream_t s);
int launch_xor(const uint16_t *a, const uint16_t *b, size_t n, uint16_t *out, cudaStream_t s);
int launch_split_w(const uint8_t *in, size_t n, int width, uint8_t *planes, size_t ps, cudaStream_t s);
int launch_stream_copy(const uint8_t *src, size_t src_bytes, const uint64_t *off, size_t n_chunks, uint8_t *dst,
                       size_t dst_cap, uint64_t *dst_off, int32_t *status, cudaStream_t s);
int launch_merge_w(const uint8_t *planes, size_t n, int width, size_t ps, uint8_t *out, cudaStream_t s);
int launch_wait_probe(int kind, const uint64_t *desc, uint32_t seg, unsigned limit, uint64_t *out, int32_t *status,
                      cudaStream_t s);

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? HUFF_OK : HUFF_ERR_CUDA;
}

}  // namespace huffk
