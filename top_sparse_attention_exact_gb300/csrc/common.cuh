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
constexpr int kMaxLen = 1 << 23;    // rows per sequence
constexpr long long kMaxRows = 1ll << 29;   // B * Hkv * max_len (the scan's TMA row coordinate is 32-bit)
constexpr int kMaxK = 4096;
constexpr int kMaxC = 256;
constexpr int kExactCluster = 8;    // CTAs (candidate segments) per exact-path head
constexpr int kMaxSeqGroups = 512;  // B * Hkv handled by one scan launch
constexpr int kMaxCand = 18432;     // R*K + W (the candidate lists live in smem)
// scores per window of the exact select (67.5 KiB): one window per CTA up to
// 138K keys at 8 CTAs per head, and two CTAs of the select (115,712 bytes of
// shared memory at K = 2048) per 228 KB SM up to K = 2048
constexpr int kSliceCap = 17280;
constexpr int kPfMaxHeads = 64;     // decode steps with the exact-head prefilter: at most this many heads
constexpr size_t kMaxDynSmem = 227 * 1024;   // dynamic shared memory of one CTA

// Per-sequence control words.
// (next slot, live entries, decode steps done, unused); `snap` holds the same
// three words as the path decision saw them, for the rest of the step.
enum { SEQ_HEAD = 0, SEQ_COUNT = 1, SEQ_TDEC = 2, SEQ_WORDS = 4 };
// Counters per sequence.
enum { CNT_REUSE = 0, CNT_FALLBACK = 1, CNT_REFRESH = 2, CNT_SUM_M = 3, CNT_MAX_M = 4, CNT_WORDS = 5 };

// Device-side view of one context's workspace (or of a stateless exact call).
struct Work {
    int B, Hq, Hkv, G, max_len, K, C, W, R, T_r;
    float tau;
    int retrieval;     // RETOPK_RETRIEVE_*
    int cand_stride;   // per-head capacity of cand_idx / cand_key
    int n_scan;        // scan CTAs per (b, h_kv)
    int cluster;       // CTAs per head in the back end (finish / select kernels): 1, 2, 4 or 8
    int sc_stride;     // row stride of `scores` (max_len rounded up to 16)
    // query-support cache (decode contexts only)
    uint16_t *fifo_q;
    int32_t *fifo_sup;
    int32_t *fifo_len;
    int32_t *seq;
    int32_t *snap;       // [B*SEQ_WORDS] this step's view of `seq`
    unsigned long long *counters;
    // per-step scratch
    int32_t *path;       // [B*Hq] (NULL: every head takes the exact path)
    float *rho_max;      // [B*Hq]
    int32_t *topR;       // [B*Hq*R]
    uint16_t *q_stage;   // [B*Hq*d] device copy of q for retopk_decode_step_host
    int32_t *M;          // [B*Hq]
    int32_t *cand_idx;   // [B*Hq*cand_stride]
    uint32_t *cand_key;  // [B*Hq*cand_stride]
    float *scores;       // [B*Hq*sc_stride]
    // Exact-head prefilter of long-history decode steps (8 CTAs per head, a
    // CTA's share of the scores longer than one window, at most kPfMaxHeads
    // heads): per (head, rank, window) its first-digit candidate count, and
    // per (head, rank) the second-digit histogram of its digit-T1 keys
    int prefilter;       // decode steps run it
    int pf_nw;           // windows per rank at max_len (0: no arrays)
    int32_t *pf_cnt;     // [B*Hq*kExactCluster*pf_nw]
    uint32_t *pf_h2;     // [B*Hq*kExactCluster*256], cleared with the histogram
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

// ---- mbarrier / bulk-copy helpers (inline PTX) --------------------------------
constexpr long long kWaitCycles = 4000000000LL;   // bounded waits: ~2 s at 2 GHz
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; returns false (and flags the status word) on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          long long limit = kWaitCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            atomicOr(status, RETOPK_STATUS_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while its predecessor on the stream is still running; pdl_wait() returns once
// the predecessor grid has completed and its memory operations are visible
// (at once for a plain launch).  pdl_trigger() lets this grid's successor
// launch before this grid ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with the programmatic-serialization attribute (and a cluster of
// cluster_x CTAs along x when cluster_x > 1).
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// 1-D bulk copy global -> shared (TMA), completing on `bar`.  dst, src 16-byte
// aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Range check of a gathered K / V row.  A build with RETOPK_CHECKED defined
// checks every row index a kernel gathers against the sequence's length
// before the load; a violation sets RETOPK_STATUS_GATHER and the row is
// skipped (read as zeros), never a trap.  Other builds compile the check away:
// every gathered index comes from a scan or a candidate list over [0, L).
#ifdef RETOPK_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ bool row_ok(int32_t idx, int L, uint32_t *status)
{
    if (!kChecked || (uint32_t)idx < (uint32_t)L)
        return true;
    atomicOr(status, RETOPK_STATUS_GATHER);
    return false;
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
                        int len_off, cudaStream_t st, int max_stages = 6);
cudaError_t launch_exact_select(const Work &w, QSrc q, const uint16_t *v_cache, const int32_t *seqlens,
                                int len_off, int mode, int init_slot, uint16_t *out, int32_t *idx_out,
                                cudaStream_t st);
cudaError_t launch_fidelity(const uint16_t *q, const uint16_t *k, const int32_t *S, const int32_t *Sh,
                            const uint16_t *o, const uint16_t *oh, float *out, uint32_t *status, int B, int Hq,
                            int Hkv, int max_len, int K, cudaStream_t st);
cudaError_t launch_overlap(const int32_t *S, const int32_t *others, int rows, int R, int K, float *out,
                           cudaStream_t st);
cudaError_t launch_decide(const Work &w, const uint16_t *q, uint16_t *q_copy, const uint16_t *k_new,
                          const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache, int32_t *seqlens,
                          cudaStream_t st);
cudaError_t launch_finish(const Work &w, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *seqlens, uint16_t *out, cudaStream_t st);
cudaError_t launch_append(const Work &w, const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *k_cache, uint16_t *v_cache, int32_t *seqlens, cudaStream_t st);
cudaError_t launch_init_done(const Work &w, cudaStream_t st);
cudaError_t launch_clear_words(void *p, size_t bytes, cudaStream_t st);
cudaError_t launch_prefilter(const Work &w, const int32_t *seqlens, cudaStream_t st);
cudaError_t launch_selftest_wait(uint32_t *status, long long limit, cudaStream_t st);
int scan_ctas_per_sm();

enum { FIN_DECODE = 0, FIN_EXACT = 1, FIN_INIT = 2 };

}  // namespace retopk
