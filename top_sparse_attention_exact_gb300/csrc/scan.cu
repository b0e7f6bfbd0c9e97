// scan.cu -- full-history QK scan of the exact path (ReTopK paper, §Problem
// Setup Eq. (4): e_i = q . k_i / sqrt(d) for every cached key) fused with the
// first radix digit of the global Top-K (§Motivation Eq. (1)).
//
// Work: every (sequence, KV head) group that has at least one query head on
// the exact path this step contributes ceil(L_b / 128) tiles of 128 key rows.
// The tiles of all active groups are split evenly over a persistent grid of
// one CTA per SM, so a step with a single exact group still streams with the
// whole GPU.  Each K row leaves HBM once per group and is scored against
// every exact query head of the group.
//
// Pipeline (per CTA): one producer thread issues one 2-D tensor copy (TMA)
// per tile -- 256 half rows of 128 bytes, a contiguous 32 KiB block -- into a
// ring of shared-memory stages, with the 128-byte swizzle and an evict-first
// L2 policy; eight
// consumer warps wait on the stage's mbarrier, read their 16 rows as mma
// A fragments (conflict-free thanks to the swizzle), multiply them with the
// group's queries on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate) and release the stage.  Every wait is bounded: on expiry the
// kernel sets RETOPK_STATUS_TIMEOUT, drains its copies and returns.
//
// Fragment layout: the contraction dimension is permuted identically for A
// (keys) and B (queries) so that each thread's fragment elements of a row
// form whole 16-byte chunks: lane (g, t) holds chunks 4j+t (j = 0..3) of
// rows g and g+8; in k-step s the logical columns {2t, 2t+1, 2t+8, 2t+9}
// are the physical elements (s>>1)*32 + t*8 + (s&1)*4 + {0,1,2,3}.
//
// Epilogue: fp32 scores go to the workspace, and an 11-bit histogram of
// their order-preserving keys is kept per exact head in shared memory and
// flushed to global memory when the CTA leaves a group -- from the top bin
// down to where this CTA alone holds min(K, L) keys, which keeps the global
// histogram exact from the Top-K threshold digit up (flush_hist).
#include <cuda.h>

#include <algorithm>

#include "common.cuh"

namespace retopk {

constexpr int kTileRows = 128;
constexpr int kStageBytes = kTileRows * kD * 2;          // 32 KiB
constexpr int kConsumerWarps = 8;
constexpr int kScanThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxGroups = kMaxSeqGroups;                // B * Hkv

struct ScanArgs {
    const uint16_t *q;
    long long q_b_stride, q_h_stride;
    const int32_t *seqlens;
    const int32_t *path;
    float *scores;
    uint32_t *hist;
    uint32_t *status;
    int B, Hq, Hkv, G, max_len, sc_stride, len_off, stages, K;
    float scale;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)),
          "l"(policy)
        : "memory");
}

// fp32 store with an L2 evict-last policy: the scores are re-read right after
// the scan while the K stream (evict-first) passes through L2.
__device__ __forceinline__ void st_keep(float *p, float v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Adds the shared-memory histograms of the exact heads in `mask` (G heads of
// kHistBins bins) into global memory: 16-byte shared loads, one atomic per
// non-empty bin.  Called by the 256 consumer threads.
__device__ __forceinline__ void flush_hist_all(const uint32_t *hist_s, uint32_t *hg, int G, uint32_t mask, int tid)
{
    constexpr int kVec = kHistBins / 4;
    for (int i4 = tid; i4 < G * kVec; i4 += 256) {
        if (!((mask >> (i4 / kVec)) & 1u))
            continue;
        const uint4 h = reinterpret_cast<const uint4 *>(hist_s)[i4];
        uint32_t *d = hg + 4 * i4;
        if (h.x)
            atomicAdd(d + 0, h.x);
        if (h.y)
            atomicAdd(d + 1, h.y);
        if (h.z)
            atomicAdd(d + 2, h.z);
        if (h.w)
            atomicAdd(d + 3, h.w);
    }
}

// The same, when the CTA holds many keys of many exact heads: only the top of
// a histogram is used -- the select takes from it the digit T1 of the
// need-th largest score, and the bins from T1 up must be complete.  If this
// CTA alone holds `need` keys at or above digit th, the global T1 is >= th;
// so each CTA flushing its bins from the top down to its own th keeps every
// bin >= T1 exact.  Consumer warp w takes heads w, w + 8, ...: 128 bins per
// step from the top (lane 0 the highest four), one atomic per nonzero bin,
// until the step in which its running count reaches need.  Fewer atomics than
// flush_hist_all when each head holds several times `need` keys here (one
// warp per head is slower when only one or two heads are exact).
__device__ __forceinline__ void flush_hist_top(const uint32_t *hist_s, uint32_t *hg, int G, uint32_t mask, int need,
                                               int tid)
{
    const int lane = tid & 31, warp = tid >> 5;
    for (int n = warp; n < G; n += kConsumerWarps) {
        if (!((mask >> n) & 1u))
            continue;
        const uint32_t *hs = hist_s + (size_t)n * kHistBins;
        uint32_t *hd = hg + (size_t)n * kHistBins;
        int run = 0;
        for (int top = kHistBins; top > 0 && run < need; top -= 128) {   // warp-uniform
            const int base = top - 4 * (lane + 1);
            const uint4 h = *reinterpret_cast<const uint4 *>(hs + base);
            if (h.x)
                atomicAdd(hd + base, h.x);
            if (h.y)
                atomicAdd(hd + base + 1, h.y);
            if (h.z)
                atomicAdd(hd + base + 2, h.z);
            if (h.w)
                atomicAdd(hd + base + 3, h.w);
            run += warp_isum((int)(h.x + h.y + h.z + h.w));
        }
    }
}

// The group's histograms into global memory: the top-only flush when this CTA
// scored at least 4 * need rows of the group for at least four exact heads.
__device__ __forceinline__ void flush_hist(const uint32_t *hist_s, uint32_t *hg, int G, uint32_t mask, int need,
                                           int rows, int tid)
{
    if (rows >= 4 * need && __popc(mask) >= 4)
        flush_hist_top(hist_s, hg, G, mask, need, tid);
    else
        flush_hist_all(hist_s, hg, G, mask, tid);
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Fragment row g reads tile row row_perm(g) (and +8): g = 0..7 -> 0 2 1 3 4 6 5 7.
// The two fragment rows of a quarter warp (g = 2p, 2p+1) then map to half rows
// whose swizzle phases differ by 4, so every 128-bit shared load is free of
// bank conflicts.
__device__ __forceinline__ int row_perm(int g) { return (g & 4) | ((g & 1) << 1) | ((g >> 1) & 1); }

struct ScanShared {
    uint64_t full[8];
    uint64_t empty[8];
    int timed_out;                  // a pipeline wait expired (copies may still be in flight)
    int n_groups;
    int total_tiles;
    int grp_first[kMaxGroups + 1];  // prefix of tiles over groups b * Hkv + hk
    uint32_t grp_mask[kMaxGroups];
};

template <int NT>
__global__ void __launch_bounds__(kScanThreads, 1)
    scan_kernel(const __grid_constant__ CUtensorMap kmap, const ScanArgs a)
{
    extern __shared__ __align__(1024) unsigned char scan_smem[];
    __shared__ ScanShared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const int S = a.stages;
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(scan_smem) + 1023) & ~uintptr_t(1023));
    uint32_t *hist_s = reinterpret_cast<uint32_t *>(ring + (size_t)S * kStageBytes);   // [G][kHistBins]

    // ---- set-up that needs nothing from the previous kernel
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
        for (int s2 = 0; s2 < S; ++s2) {
            mbar_init(&sh.full[s2], 1);
            mbar_init(&sh.empty[s2], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.timed_out = 0;
    }
    // Without a path decision (the stateless exact step, cache initialisation)
    // nothing the tiles or the tile list read comes from the previous kernel
    // (the histogram clear, itself a plain launch behind everything earlier):
    // the copies start at once and only the histogram flush waits for it.
    // A decode step's scan needs the decision (and the appended K row) first.
    const bool early = a.path == nullptr;
    if (!early)
        pdl_wait();
    pdl_trigger();
    // ---- active groups and their tile ranges (every CTA computes the same
    //      list): groups with no exact head get zero tiles
    const int NG = a.B * a.Hkv;
    for (int i = tid; i < NG; i += kScanThreads) {
        const int b = i / a.Hkv, hk = i % a.Hkv;
        uint32_t mask = 0;
        if (!a.path) {
            mask = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
        } else {
            const int32_t *pp = a.path + b * a.Hq + hk * G;
            for (int j = 0; j < G; ++j)
                mask |= (pp[j] != 0 ? 1u : 0u) << j;
        }
        const int L = seq_len(a.seqlens, b, a.len_off, a.max_len);
        sh.grp_mask[i] = mask;
        sh.grp_first[i + 1] = (mask && L > 0) ? (L + kTileRows - 1) / kTileRows : 0;
    }
    if (tid == 0)
        sh.grp_first[0] = 0;
    __syncthreads();
    // inclusive prefix over the per-group tile counts (one warp, NG <= 512)
    if (warp == 0) {
        int carry = 0;
        for (int base = 1; base <= NG; base += 32) {
            const int i = base + lane;
            int v = (i <= NG) ? sh.grp_first[i] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o)
                    v += y;
            }
            if (i <= NG)
                sh.grp_first[i] = v + carry;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            sh.n_groups = NG;
            sh.total_tiles = carry;
        }
    }
    __syncthreads();
    const int T = sh.total_tiles;
    const int t_begin = (int)(((long long)T * blockIdx.x) / gridDim.x);
    const int t_end = (int)(((long long)T * (blockIdx.x + 1)) / gridDim.x);

    if (warp == kConsumerWarps) {
        // ================= producer =================
        if (lane == 0 && t_begin < t_end) {
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            int gi = 0;
            bool ok = true;
            for (int it = 0, tile = t_begin; tile < t_end && ok; ++it, ++tile) {
                while (tile >= sh.grp_first[gi + 1])
                    ++gi;
                const int s = it % S;
                if (it >= S)
                    ok = mbar_wait(&sh.empty[s], ((it / S) - 1) & 1, a.status);
                if (!ok)
                    break;
                const int row = gi * a.max_len + (tile - sh.grp_first[gi]) * kTileRows;
                unsigned char *dst = ring + (size_t)s * kStageBytes;
                mbar_expect_tx(&sh.full[s], kStageBytes);
                tma_load_2d(dst, &kmap, 0, 2 * row, &sh.full[s], policy);
            }
            if (!ok)
                sh.timed_out = 1;
        }
    } else {
        // ================= consumers =================
        const int g = lane >> 2, t = lane & 3;
        uint64_t keep;
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
        int gi = -1;
        int grp_rows = 0;   // rows of the current group this CTA has scored (flush heuristic)
        uint32_t mask = 0;
        int b = 0, hk = 0, L = 0;
        uint4 qf[NT][4];
        bool ok = true;
        bool nonfinite = false;   // a score that is NaN or +-inf (reported once per thread)
        for (int it = 0, tile = t_begin; tile < t_end; ++it, ++tile) {
            int ng = gi < 0 ? 0 : gi;
            while (tile >= sh.grp_first[ng + 1])
                ++ng;
            if (ng != gi) {
                consumer_sync();
                if (gi >= 0) {   // flush the previous group's histogram
                    if (early)
                        pdl_wait();   // the histograms are cleared
                    flush_hist(hist_s, a.hist + (size_t)(b * a.Hq + hk * G) * kHistBins, G, mask, min(a.K, L),
                               grp_rows, tid);
                    consumer_sync();
                }
                gi = ng;
                grp_rows = 0;
                mask = sh.grp_mask[gi];
                b = gi / a.Hkv;
                hk = gi % a.Hkv;
                L = seq_len(a.seqlens, b, a.len_off, a.max_len);
                for (int i4 = tid; i4 < G * (kHistBins / 4); i4 += kConsumerWarps * 32)
                    if ((mask >> (i4 / (kHistBins / 4))) & 1u)
                        reinterpret_cast<uint4 *>(hist_s)[i4] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int n = nt * 8 + g;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (n < G) {
                            const uint4 *qp = reinterpret_cast<const uint4 *>(
                                a.q + b * a.q_b_stride + (long long)(hk * G + n) * a.q_h_stride);
                            qf[nt][j] = qp[j * 4 + t];
                        } else {
                            qf[nt][j] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                consumer_sync();
            }
            const int s = it % S;
            if (ok)
                ok = mbar_wait(&sh.full[s], (it / S) & 1, a.status);
            if (!ok)
                continue;   // keep walking the tiles so the named barriers still match
            const unsigned char *st = ring + (size_t)s * kStageBytes;
            const int base = (tile - sh.grp_first[gi]) * kTileRows;   // first row of the tile
            grp_rows += kTileRows;
            const int rl0 = warp * 16 + row_perm(g), rl1 = rl0 + 8;    // rows within the tile
            uint4 x0[4], x1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // half row h = j>>1 of key row r is box row 2r+h; its 16-byte
                // chunk cc sits at position cc ^ ((2r+h) & 7)
                const int hr0 = 2 * rl0 + (j >> 1), hr1 = 2 * rl1 + (j >> 1), cc = ((j & 1) << 2) + t;
                x0[j] = *reinterpret_cast<const uint4 *>(st + hr0 * 128 + ((cc ^ (hr0 & 7)) << 4));
                x1[j] = *reinterpret_cast<const uint4 *>(st + hr1 * 128 + ((cc ^ (hr1 & 7)) << 4));
            }
            const int r0 = base + rl0, r1 = base + rl1;
            float *sc_base = a.scores + (size_t)(b * a.Hq + hk * G) * a.sc_stride;
            float c[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int j = ks >> 1;
                    const bool hi = ks & 1;
                    mma_bf16_16816(c[nt], hi ? x0[j].z : x0[j].x, hi ? x1[j].z : x1[j].x,
                                   hi ? x0[j].w : x0[j].y, hi ? x1[j].w : x1[j].y, hi ? qf[nt][j].z : qf[nt][j].x,
                                   hi ? qf[nt][j].w : qf[nt][j].y);
                }
            }
            // the stage's rows have been consumed by the MMAs: hand it back
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.empty[s]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // c[0]: (row r0, head 2t)  c[1]: (r0, 2t+1)  c[2]: (r1, 2t)  c[3]: (r1, 2t+1)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = nt * 8 + 2 * t + (e & 1);
                    const int r = (e < 2) ? r0 : r1;
                    if (n < G && r < L && ((mask >> n) & 1u)) {
                        const float sc = c[nt][e] * a.scale + 0.0f;
                        nonfinite |= !(fabsf(sc) <= 3.402823466e38f);
                        st_keep(&sc_base[(size_t)n * a.sc_stride + r], sc, keep);
                        atomicAdd(&hist_s[n * kHistBins + (f2key(sc) >> (32 - kHistBits))], 1u);
                    }
                }
            }
        }
        consumer_sync();
        if (early)
            pdl_wait();   // the histograms are cleared
        if (gi >= 0)
            flush_hist(hist_s, a.hist + (size_t)(b * a.Hq + hk * G) * kHistBins, G, mask, min(a.K, L), grp_rows,
                       tid);
        if (nonfinite)
            atomicOr(a.status, RETOPK_STATUS_NONFINITE);
        if (!ok)
            sh.timed_out = 1;
    }
    __syncthreads();
    // Drain: every issued copy has landed before shared memory is released.
    // On the normal path the consumers waited on each one; only after an
    // expired wait can copies still be in flight.
    if (tid == kConsumerWarps * 32 && sh.timed_out) {
        const int n = t_end - t_begin;
        for (int s = 0; s < S && s < n; ++s) {
            const int last = s + ((n - 1 - s) / S) * S;     // last issue index that used stage s
            mbar_wait(&sh.full[s], (last / S) & 1, a.status);
        }
    }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on, gives up after `limit` cycles, flags RETOPK_STATUS_TIMEOUT and
// returns -- the path every pipeline wait of the scan takes on expiry.
__global__ void selftest_wait_kernel(uint32_t *status, long long limit)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait(&bar, 0, status, limit);
    }
}

cudaError_t launch_selftest_wait(uint32_t *status, long long limit, cudaStream_t st)
{
    selftest_wait_kernel<<<1, 32, 0, st>>>(status, limit);
    return cudaGetLastError();
}

// ---- host side --------------------------------------------------------------
static size_t hist_bytes(int G) { return (size_t)G * kHistBins * sizeof(uint32_t); }

static int stages_for(int G)
{
    const size_t budget = 227 * 1024 - sizeof(ScanShared) - 1024 - hist_bytes(G);
    int s = (int)(budget / kStageBytes);
    return s > 6 ? 6 : (s < 2 ? 2 : s);
}

static size_t scan_smem_bytes(int G) { return 1024 + (size_t)stages_for(G) * kStageBytes + hist_bytes(G); }

int scan_ctas_per_sm() { return 1; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// K cache viewed as a 2-D tensor of 128-byte half rows: [2*B*Hkv*max_len, 64
// elements].  One box of 256 half rows is one contiguous 32 KiB tile.
static cudaError_t make_kmap(CUtensorMap *map, const uint16_t *k, int B, int Hkv, int max_len)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kD / 2, (cuuint64_t)2 * B * Hkv * max_len};
    cuuint64_t strides[1] = {(cuuint64_t)kD};            // 128 bytes per half row
    cuuint32_t box[2] = {64, 2 * kTileRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(k), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_scan(const Work &w, QSrc q, const uint16_t *k_cache, const int32_t *seqlens,
                        int len_off, cudaStream_t st, int max_stages)
{
    if ((size_t)w.B * w.Hkv > (size_t)kMaxGroups)
        return cudaErrorInvalidValue;
    CUtensorMap map;
    cudaError_t e = make_kmap(&map, k_cache, w.B, w.Hkv, w.max_len);
    if (e != cudaSuccess)
        return e;
    ScanArgs a;
    a.q = q.q;
    a.q_b_stride = q.b_stride;
    a.q_h_stride = q.h_stride;
    a.seqlens = seqlens;
    a.path = w.path;
    a.scores = w.scores;
    a.hist = w.hist;
    a.status = w.status;
    a.B = w.B;
    a.Hq = w.Hq;
    a.Hkv = w.Hkv;
    a.G = w.G;
    a.max_len = w.max_len;
    a.sc_stride = w.sc_stride;
    a.len_off = len_off;
    a.K = w.K;
    a.stages = std::max(2, std::min(stages_for(w.G), max_stages));
    a.scale = 1.0f / sqrtf((float)kD);
    const size_t smem = 1024 + (size_t)a.stages * kStageBytes + hist_bytes(w.G);
    if (w.G <= 8)
        return launch_pdl(scan_kernel<1>, dim3(w.n_scan), dim3(kScanThreads), smem, st, 1, map, a);
    return launch_pdl(scan_kernel<2>, dim3(w.n_scan), dim3(kScanThreads), smem, st, 1, map, a);
}

cudaError_t configure_scan()
{
    size_t m1 = 0, m2 = 0;   // the largest request of each instantiation
    for (int G = 1; G <= kMaxGroup; ++G)
        (G <= 8 ? m1 : m2) = std::max(G <= 8 ? m1 : m2, scan_smem_bytes(G));
    // the whole unified cache as shared memory: a decode-step scan CTA leaves
    // room for a CTA of the concurrent reuse kernel only under that split
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(scan_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m2);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(scan_kernel<1>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(scan_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

}  // namespace retopk
