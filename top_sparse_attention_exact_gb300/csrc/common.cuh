// common.cuh -- internal definitions shared by the sm_103a kernels of the
// ReTopK / Exact Top-K decode library.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/retopk.h"

namespace retopk {

constexpr int kD = 128;             // head dimension (the only one supported)
constexpr int kHistBits = 11;       // first-level radix digit of the exact scan
constexpr int kHistBins = 1 << kHistBits;
constexpr int kMaxGroup = 16;       // query heads per KV head
constexpr int kMaxLen = 1 << 20;    // rows per sequence (candidate bitmap in smem)
constexpr int kMaxK = 4096;
constexpr int kMaxC = 256;
constexpr int kStageCap = 12288;    // candidates staged in shared memory by finalize
constexpr int kMaxSeg = 64;         // filter CTAs (segments) per head
constexpr int kMaxSeqGroups = 512;  // B * Hkv handled by one scan launch
constexpr int kMaxCand = 20480;     // R*K + W (the candidate list lives in smem)

// Per-sequence control words.
enum { SEQ_HEAD = 0, SEQ_COUNT = 1, SEQ_TDEC = 2, SEQ_DONE = 3, SEQ_WORDS = 4 };
// Counters per sequence.
enum { CNT_REUSE = 0, CNT_FALLBACK = 1, CNT_REFRESH = 2, CNT_SUM_M = 3, CNT_MAX_M = 4, CNT_WORDS = 5 };

// Device-side view of one context's workspace (or of a stateless exact call).
struct Work {
    int B, Hq, Hkv, G, max_len, K, C, W, R, T_r;
    float tau;
    int cand_stride;   // per-head capacity of cand_idx / cand_key
    int n_filter;      // filter CTAs (segments) per head
    int n_scan;        // scan CTAs per (b, h_kv)
    int sc_stride;     // row stride of `scores` (max_len rounded up to 16)
    // query-support cache (decode contexts only)
    uint16_t *fifo_q;
    int32_t *fifo_sup;
    int32_t *fifo_len;
    int32_t *seq;
    unsigned long long *counters;
    // per-step scratch
    int32_t *path;       // [B*Hq] (NULL: every head takes the exact path)
    float *rho_max;      // [B*Hq]
    int32_t *topR;       // [B*Hq*R]
    int32_t *M;          // [B*Hq]
    int32_t *cand_idx;   // [B*Hq*cand_stride]
    uint32_t *cand_key;  // [B*Hq*cand_stride]
    int32_t *seg_count;  // [B*Hq*n_filter]
    float *scores;       // [B*Hq*sc_stride]
    uint32_t *hist;      // [B*Hq*kHistBins]
    int32_t *support;    // [B*Hq*K]
    int32_t *sup_len;    // [B*Hq]
    float *out_f32;      // [B*Hq*kD]
    uint32_t *status;    // [1]
};

// Order-preserving map float -> uint32 (larger float -> larger key).  -0 is
// folded onto +0 by the caller (x + 0.0f) so equal scores get equal keys.
__device__ __forceinline__ uint32_t f2key(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// Composite selection key: score first, then lower index first.
__device__ __forceinline__ unsigned long long key64(uint32_t k, int32_t idx)
{
    return ((unsigned long long)k << 32) | (unsigned long long)(uint32_t)(~(uint32_t)idx);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Streaming 16-byte load (evict-first): the K rows of a scan are read once.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_isum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Effective length of sequence b for a launch (len_off < 0 during cache
// initialisation, where the causal prefix of a prompt position is scored).
// Clamped to the cache capacity so that a bad length can never index past it.
__device__ __forceinline__ int seq_len(const int32_t *seqlens, int b, int len_off, int max_len)
{
    int L = seqlens[b] + len_off;
    L = L > max_len ? max_len : L;
    return L < 0 ? 0 : L;
}

// ---- host-side launchers (one per kernel family) -------------------------
struct QSrc {              // where the query of (b, h) lives
    const uint16_t *q;
    long long b_stride, h_stride;   // in elements
};

// ev0 / ev1 (optional) are recorded immediately around the kernel launch.
cudaError_t launch_scan(const Work &w, QSrc q, const uint16_t *k_cache, const int32_t *seqlens,
                        int len_off, cudaStream_t st, cudaEvent_t ev0 = nullptr, cudaEvent_t ev1 = nullptr);
cudaError_t launch_filter(const Work &w, const int32_t *seqlens, int len_off, cudaStream_t st);
cudaError_t launch_finalize(const Work &w, QSrc q, const uint16_t *v_cache, const int32_t *seqlens,
                            int len_off, int mode, int init_slot, uint16_t *out, int32_t *idx_out,
                            cudaStream_t st);
cudaError_t launch_reuse(const Work &w, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *seqlens, uint16_t *out, cudaStream_t st);
cudaError_t launch_append(const Work &w, const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *k_cache, uint16_t *v_cache, int32_t *seqlens, cudaStream_t st);
cudaError_t launch_init_done(const Work &w, cudaStream_t st);
cudaError_t launch_selftest_wait(uint32_t *status, long long limit, cudaStream_t st);
cudaError_t configure_kernels();   // one-time function attributes (smem opt-in)
int scan_ctas_per_sm();

enum { FIN_DECODE = 0, FIN_EXACT = 1, FIN_INIT = 2 };

}  // namespace retopk
