// select_body.cuh -- the exact path's global Top-K and sparse softmax-value
// aggregation (ReTopK paper, §Motivation Eq. (1), §Recall-Before-Rerank
// Eq. (12), and §Complexity and GPU Implementation: the paths differ only in
// support discovery, so this back end mirrors the reuse kernel's).
//
// exact_select_kernel: one cluster of CL CTAs (CL = 1, 2, 4 or 8, at most
// kExactCluster: chosen per configuration so that one wave of clusters covers
// the heads) per exact-path
// (sequence, query head), after the scan has written the head's fp32 scores
// and its 11-bit score histogram.
//   1. Every rank finds the threshold digit T1 -- the largest digit whose
//      suffix count reaches min(K, L) -- from the histogram, and compacts the
//      keys of its 1/CL slice whose digit is >= T1 (only they can
//      be in the Exact Top-K support), in ascending index order, into its own
//      shared memory (up to kLocCap of them) and into its segment of the
//      global candidate arrays.  The slice arrives in shared memory by one
//      bulk copy (TMA) per 17K scores, issued before the histogram is read;
//      every wait on it is bounded.
//   2. Ranks exchange their counts and second-digit histograms through
//      distributed shared memory; after a cluster barrier every rank knows the
//      second digit T2 and each rank's number of final candidates (keys at or
//      above the prefix (T1, T2)).  While every rank's candidates fit its
//      shared memory, each rank pulls them (one warp per source rank);
//      otherwise each rank compacts its own final candidates (from its shared
//      memory, then its global segment) with all its threads and writes them
//      into every rank's staging list at its offset, followed by a second
//      cluster barrier.  Every rank then runs the same radix select on
//      (score, lower index first) and stable compaction: identical ascending
//      supports in every rank.
//   3. Each rank aggregates 1/CL of the support's V rows with the
//      common max and pushes (weighted sum, sum of weights) to rank 0, which
//      normalises, writes the output and -- on decode / init -- inserts
//      (q_t, S_t) into the query-support cache (Eq. (5)).
// The phases are latency-bound chains over a few thousand elements per CTA,
// so the kernel runs 16 warps per CTA (two CTAs per SM) and keeps two
// independent shared-memory loads in flight per lane in the filter.
#pragma once

#include <cooperative_groups.h>

#include <algorithm>
#include <cstddef>

#include "topk.cuh"

namespace cg = cooperative_groups;

namespace retopk {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelStageCap = 8192;                 // candidates staged in shared memory
constexpr int kLocCap = 1024;                      // candidates a rank keeps in its own shared memory
constexpr int kBlkGroups = 32;                     // filter block: 32 groups of four scores
constexpr int kMaxBlk = (kSliceCap / 4 + kBlkGroups - 1) / kBlkGroups;
static_assert(kMaxBlk <= kSelThreads, "one block count per thread");
constexpr int kSub = 13;                           // key bits [kSub, 32 - kHistBits): second-level digit
constexpr int kSubBins = 1 << (32 - kHistBits - kSub);
static_assert(kSubBins == 256, "second-level digit is 8 bits");
// the score slice, the candidate staging arrays and the per-warp value
// partials share one region (they are live in phases 1, 2 and 3)
constexpr size_t kSelRegionBytes = (size_t)kSliceCap * 4 > (size_t)kSelStageCap * 8 ? (size_t)kSliceCap * 4
                                                                                   : (size_t)kSelStageCap * 8;
// the per-warp value partials use the region's start once the staging
// arrays are dead
static_assert((size_t)kSelWarps * kD * 4 <= kSelRegionBytes, "value partials fit the region");
static_assert(kHistBins == 4 * kSelThreads, "one uint4 of histogram per thread");
constexpr int kMaxTie = 128;                       // tied keys one warp ranks (four per lane)
static_assert(kMaxBlk * kBlkGroups >= kMaxTie * 8, "the tie list fits the filter masks");

struct SelArgs {
    Work w;
    const uint16_t *q;
    long long q_b_stride, q_h_stride;
    const uint16_t *v;
    const int32_t *seqlens;
    uint16_t *out;
    int32_t *idx_out;
    int len_off, mode, init_slot;
};

struct SelShared {
    uint64_t bar;                                  // bulk-copy completion (score slices)
    int T1, T2, above2;
    int wcnt[kSelWarps];                           // final candidates per rank (phase 2)
    // filter: bit e of group g = score 4g + e passes; in phase 2 the tied
    // keys' composite keys (tie list, at most kMaxTie)
    alignas(16) uint8_t gmask[kMaxBlk * kBlkGroups];
    int bcnt[kMaxBlk], boff[kMaxBlk];              // candidates per block, and their first position
    int cnt[kExactCluster];                        // candidates per rank
    int off[kExactCluster + 1];                    // final candidates: offsets per rank
    alignas(16) uint32_t h2[kSubBins];             // this rank's digit-T1 keys by second-level digit
    alignas(16) uint32_t h2all[kExactCluster][kSubBins];   // every rank's h2 (pushed by the ranks)
    SelectShared sel;
    int ntie;                                      // final candidates sharing the prefix (T1, T2)
    unsigned long long tie_thr;                    // the rem-th largest of them
    uint32_t kmax;
    float zw[kSelWarps];
    alignas(16) float part_o[kExactCluster][kD];   // rank 0 receives every rank's partial
    float part_z[kExactCluster];
};
static_assert(offsetof(SelShared, h2) % 16 == 0 && offsetof(SelShared, h2all) % 16 == 0, "vector stores");
// the per-CTA state leads the dynamic shared memory, the regions follow
constexpr size_t kSelSharedBytes = (sizeof(SelShared) + 127) & ~size_t(127);

// Dynamic shared memory of one select CTA for a given K.
inline size_t sel_smem_bytes(int K)
{
    return kSelSharedBytes + kSelRegionBytes + (size_t)kLocCap * 8 + (size_t)((K + 3) & ~3) * 8;
}

// Bit e of the result: f2key(score e of s) >= tkey, the scores given by their
// raw bits.  For tkey >= 2^31 (threshold >= +0) that is "bits as signed int >=
// tkey - 2^31", otherwise "bits as unsigned <= ~tkey" (t: that right-hand
// side); both restate the order of f2key for every bit pattern.
template <bool kNonNeg>
__device__ __forceinline__ unsigned ge4(uint4 s, uint32_t t)
{
    if (kNonNeg)
        return ((int)s.x >= (int)t ? 1u : 0u) | ((int)s.y >= (int)t ? 2u : 0u) | ((int)s.z >= (int)t ? 4u : 0u) |
               ((int)s.w >= (int)t ? 8u : 0u);
    return (s.x <= t ? 1u : 0u) | (s.y <= t ? 2u : 0u) | (s.z <= t ? 4u : 0u) | (s.w <= t ? 8u : 0u);
}

// Filter pass 1 over one chunk (n scores, nfull full groups of four, ng groups,
// nblk blocks of kBlkGroups groups): warp w takes blocks w, w + kSelWarps, ...
// two at a time; gmask[g] bit e = score 4g + e passes, bcnt[blk] = the block's
// count (one reduction per block: warp votes cost more than the compares).
template <bool kNonNeg>
__device__ __forceinline__ void filter_masks(const uint4 *s4, int nblk, int ng, int nfull, int n, uint32_t t,
                                             uint8_t *gmask, int *bcnt)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned tail = (1u << (n & 3)) - 1u;
    auto masks = [&](int bk) {
        const int g = bk * kBlkGroups + lane;
        unsigned m = 0u;
        if (bk < nblk) {
            if (g < ng) {
                m = ge4<kNonNeg>(s4[g], t);
                if (g >= nfull)
                    m &= tail;
            }
            gmask[g] = (uint8_t)m;   // every group of a block, zero past the last
        }
        return m;
    };
    for (int bk = warp; bk < nblk; bk += 2 * kSelWarps) {   // warp-uniform trip count
        const unsigned ma = masks(bk), mb = masks(bk + kSelWarps);
        const int ca = (int)__reduce_add_sync(0xffffffffu, (unsigned)__popc(ma));
        const int cb = (int)__reduce_add_sync(0xffffffffu, (unsigned)__popc(mb));
        if (lane == 0)
            bcnt[bk] = ca;
        if (lane == 1 && bk + kSelWarps < nblk)
            bcnt[bk + kSelWarps] = cb;
    }
}

// ---- the select's rare paths, kept out of line -----------------------------
// They run only when many keys tie at the 19-bit prefix, when the histograms
// disagree with the scores, or for long histories.  Out of line, the common
// path's code stays short and contiguous: after an L2 flush a lone exact
// head's cluster fetches it from device memory phase by phase.

// The threshold of the `need` largest staged candidates by the full radix
// select (no usable second digit).
static __device__ __noinline__ unsigned long long staged_full_select(int N2, int need, const int32_t *st_idx,
                                                              const uint32_t *st_key, SelectShared &sel)
{
    auto get = [&](int j, int32_t &idx, uint32_t &k) {
        idx = st_idx[j];
        k = st_key[j];
    };
    return radix_select_threshold<kSelThreads>(N2, need, get, sel);
}

// The threshold among the staged candidates sharing the 19-bit prefix when
// more than 32 share it: radix refinement below the prefix.
static __device__ __noinline__ unsigned long long staged_refine(int N2, int rem, uint32_t p19, const int32_t *st_idx,
                                                         const uint32_t *st_key, SelectShared &sel)
{
    auto get = [&](int j, int32_t &idx, uint32_t &k) {
        idx = st_idx[j];
        k = st_key[j];
    };
    return radix_refine<kSelThreads>(N2, rem, (unsigned long long)p19 << (32 + kSub), 32 + kSub, get, sel);
}

// More final candidates than the staging holds: select among all candidates in
// place, in the global segments (offsets off[] of the unfiltered per-rank
// lists), compact the support into sup_i / sup_k and leave its maximum key in
// kmax.  Returns the support's length.
static __device__ __noinline__ int global_select(int N, int need, int K, int seg, int ranks, const int *off,
                                                 const int32_t *gi, const uint32_t *gk, int32_t *sup_i,
                                                 uint32_t *sup_k, SelectShared &sel, uint32_t *kmax)
{
    auto get = [&](int j, int32_t &idx, uint32_t &k) {
        int r = 0;
        while (r + 1 < ranks && off[r + 1] <= j)
            ++r;
        const int o = r * seg + (j - off[r]);
        idx = gi[o];
        k = gk[o];
    };
    const unsigned long long thr = radix_select_threshold<kSelThreads>(N, need, get, sel);
    const int n = stable_compact<kSelThreads, 4>(N, thr, get, K, sup_i, sup_k, sel.warp_tot);
    __syncthreads();
    uint32_t km = 0u;
    for (int j = threadIdx.x; j < n; j += kSelThreads)
        km = max(km, sup_k[j]);
    km = __reduce_max_sync(0xffffffffu, km);
    if ((threadIdx.x & 31) == 0)
        atomicMax(kmax, km);
    return n;
}

// Long-history decode steps: the exact-head prefilter (prefilter.cu) has
// listed this rank's first-digit candidates window by window -- window v's
// count in pf_cnt, its candidates at offset v * kSliceCap of the rank's global
// segment -- and their second-digit histogram in pf_h2.  Compacts the lists
// in place into positions 0 .. count-1 (the first kLocCap also into shared
// memory) and loads the histogram into sh.h2.  Entry j of the compacted list
// comes from position >= j, so batches of kSelThreads * 4 entries, each read
// in full (every load of a batch in flight at once) before it is written, in
// order, never clobber an entry not yet read.  Returns the rank's count.
static __device__ __noinline__ int gather_prefiltered(const Work &w, int bh, int rank, int range, int32_t *loc_i,
                                                      uint32_t *loc_k, int32_t *oi, uint32_t *ok, SelShared &sh)
{
    constexpr int kPer = 4;
    const int tid = threadIdx.x;
    const int nw = (range + kSliceCap - 1) / kSliceCap;   // <= pf_nw <= kMaxBlk
    const int32_t *pc = w.pf_cnt + ((size_t)bh * kExactCluster + rank) * w.pf_nw;
    const int cv = tid < nw ? pc[tid] : 0;
    int total;
    const int pre = block_excl_scan<kSelThreads>(cv, sh.sel.warp_tot, total);
    if (tid < nw)
        sh.boff[tid] = pre;
    if (tid < kSubBins)
        sh.h2[tid] = w.pf_h2[((size_t)bh * kExactCluster + rank) * kSubBins + tid];
    __syncthreads();
    for (int j0 = 0; j0 < total; j0 += kSelThreads * kPer) {   // uniform trip count
        int32_t ix[kPer];
        uint32_t k[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int j = j0 + u * kSelThreads + tid;
            ix[u] = 0;
            k[u] = 0u;
            if (j < total) {
                int lo = 0, hi = nw - 1;   // the window holding entry j: last v with boff[v] <= j
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (sh.boff[mid] <= j)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int src = lo * kSliceCap + (j - sh.boff[lo]);
                ix[u] = oi[src];
                k[u] = ok[src];
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int j = j0 + u * kSelThreads + tid;
            if (j < total) {
                if (j < kLocCap) {
                    loc_i[j] = ix[u];
                    loc_k[j] = k[u];
                }
                oi[j] = ix[u];
                ok[j] = k[u];
            }
        }
        __syncthreads();
    }
    return total;
}

// One exact-path head per cluster of CL CTAs of kSelThreads threads; `smem`
// is the CTA's dynamic shared memory (sel_smem_bytes).
template <int CL>
__device__ __forceinline__ void exact_select_body(const SelArgs &a, unsigned char *smem)
{
    static_assert(CL == 1 || CL == 2 || CL == 4 || CL == 8, "cluster of 1, 2, 4 or 8 CTAs");
    SelShared &sh = *reinterpret_cast<SelShared *>(smem);
    unsigned char *xs = smem + kSelSharedBytes;
    cg::cluster_group cluster = cg::this_cluster();
    const Work &w = a.w;
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq, h = bh % w.Hq, hk = h / w.G;
    const int path = (a.mode == FIN_DECODE) ? w.path[bh] : RETOPK_PATH_FALLBACK;
    if (path == RETOPK_PATH_REUSE)
        return;                                    // a reuse head (uniform over the cluster)
    // Until the wait for the scan below, only what the scan does not write:
    // the lengths, the ring snapshot and q (written before the scan passed its
    // own wait, or by the caller before the step), and shared-memory set-up.
    const bool insert = a.mode == FIN_DECODE || a.mode == FIN_INIT;   // into the query-support cache
    const size_t e_slot = insert ? (size_t)bh * w.C + (a.mode == FIN_INIT ? a.init_slot : w.snap[b * SEQ_WORDS + SEQ_HEAD])
                                 : 0;
    if (insert && rank == 0 && tid < kD / 8) {     // q_t into its slot (Eq. (5)), off the critical path
        const uint16_t *qrow = a.q + b * a.q_b_stride + (long long)h * a.q_h_stride;
        reinterpret_cast<uint4 *>(w.fifo_q + e_slot * kD)[tid] = reinterpret_cast<const uint4 *>(qrow)[tid];
    }
    const int L = seq_len(a.seqlens, b, a.len_off, w.max_len);
    const int need = min(w.K, L);
    const int seg = (((L + CL - 1) / CL) + 15) & ~15;
    const int start = min(L, rank * seg), end = min(L, start + seg);
    const float *sc = w.scores + (size_t)bh * w.sc_stride;
    int32_t *oi = w.cand_idx + (size_t)bh * w.cand_stride + (size_t)rank * seg;
    uint32_t *ok = w.cand_key + (size_t)bh * w.cand_stride + (size_t)rank * seg;

    float *slice = reinterpret_cast<float *>(xs);                          // [kSliceCap], phase 1
    int32_t *st_idx = reinterpret_cast<int32_t *>(xs);                     // [kSelStageCap], phase 2
    uint32_t *st_key = reinterpret_cast<uint32_t *>(st_idx + kSelStageCap);
    float(*red)[kD] = reinterpret_cast<float(*)[kD]>(xs);                  // [kSelWarps][kD], phase 3
    int32_t *loc_i = reinterpret_cast<int32_t *>(xs + kSelRegionBytes);    // [kLocCap]
    uint32_t *loc_k = reinterpret_cast<uint32_t *>(loc_i + kLocCap);
    const int Kp = (w.K + 3) & ~3;
    int32_t *sup_i = reinterpret_cast<int32_t *>(loc_k + kLocCap);         // [Kp]
    uint32_t *sup_k = reinterpret_cast<uint32_t *>(sup_i + Kp);

    // ---- 1. this rank's slice of scores (one bulk copy per kSliceCap scores, issued
    //         first) while the threshold digit is found from the histogram ---
    if (tid == 0) {
        mbar_init(&sh.bar, 1);
        sh.ntie = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.kmax = 0u;
        sh.T1 = 0;
        sh.T2 = 0;
        sh.above2 = -1;   // stays -1 unless digit T2 is found
    }
    if (tid < kSubBins)
        sh.h2[tid] = 0u;
    __syncthreads();
    pdl_wait();                                    // the scan's scores and histogram
    // copies [c0, c0 + n & ~3) by TMA; the <= 3 trailing scores by plain loads
    auto issue = [&](int c0, int n) {
        const int nb = n & ~3;
        if (tid == 0 && nb > 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier reads of the buffer
            mbar_expect_tx(&sh.bar, (uint32_t)nb * 4u);
            bulk_load(slice, sc + c0, (uint32_t)nb * 4u, &sh.bar);
        }
        if (tid < n - nb)
            slice[nb + tid] = sc[c0 + nb + tid];
    };
    // decode steps of long histories: the prefilter kernel has listed this
    // rank's first-digit candidates window by window
    const bool prefiltered = a.mode == FIN_DECODE && w.prefilter;
    if (!prefiltered)
        issue(start, min(end - start, kSliceCap));
    const uint4 hv = reinterpret_cast<const uint4 *>(w.hist + (size_t)bh * kHistBins)[tid];   // digits [4t, 4t+4)
    {
        const int part = (int)(hv.x + hv.y + hv.z + hv.w);
        int tot;
        const int below = block_excl_scan<kSelThreads>(part, sh.sel.warp_tot, tot);
        const int above = tot - below - part;
        if (need > 0 && above < need && above + part >= need) {
            const uint32_t c4[4] = {hv.x, hv.y, hv.z, hv.w};
            int acc = above;
            for (int i = 3; i >= 0; --i) {
                acc += (int)c4[i];
                if (acc >= need) {
                    sh.T1 = tid * 4 + i;
                    break;
                }
            }
        }
    }
    __syncthreads();
    const int T1 = sh.T1;
    const uint32_t tkey = (uint32_t)T1 << (32 - kHistBits);   // smallest key whose digit is T1
    // f2key(x) >= tkey as one compare on the raw bits of x (ge4)
    const uint32_t tcmp = tkey >= 0x80000000u ? (tkey & 0x7fffffffu) : ~tkey;
    int count = 0;
    uint32_t parity = 0;
    if (prefiltered)
        count = gather_prefiltered(w, bh, rank, end - start, loc_i, loc_k, oi, ok, sh);
    for (int c0 = start; c0 < end && !prefiltered; c0 += kSliceCap) {   // uniform trip count
        const int n = min(end - c0, kSliceCap);
        if (c0 != start)
            issue(c0, n);
        if ((n & ~3) > 0 && !mbar_wait(&sh.bar, parity, w.status)) {
            if (tid == 0)   // the copy may still be in flight: wait once more before reusing the buffer
                mbar_wait(&sh.bar, parity, w.status);
        }
        parity ^= 1u;
        __syncthreads();                                  // trailing plain loads visible
        // blocks of 32 groups of four scores (128 scores) go round-robin to the
        // warps -- candidates cluster by position, so contiguous ranges would
        // leave a few warps with all of them.  Pass 1: per block, the four
        // ballots "score 4g + e passes" (lane = g mod 32) and their count.
        const int nfull = n >> 2, ng = (n + 3) >> 2, nblk = (ng + kBlkGroups - 1) / kBlkGroups;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(slice);
        if (tkey >= 0x80000000u)
            filter_masks<true>(s4, nblk, ng, nfull, n, tcmp, sh.gmask, sh.bcnt);
        else
            filter_masks<false>(s4, nblk, ng, nfull, n, tcmp, sh.gmask, sh.bcnt);
        __syncthreads();
        int total;
        {
            const int c = tid < nblk ? sh.bcnt[tid] : 0;
            const int ex = block_excl_scan<kSelThreads>(c, sh.sel.warp_tot, total);
            if (tid < nblk)
                sh.boff[tid] = count + ex;
        }
        __syncthreads();
        // pass 2: the candidates' indices, in ascending order, from the masks
        {
            const unsigned lt = (1u << lane) - 1u;
            for (int bk = warp; bk < nblk; bk += kSelWarps) {   // warp-uniform
                if (sh.bcnt[bk] == 0)
                    continue;
                const unsigned m = sh.gmask[bk * kBlkGroups + lane];   // 0 past the chunk's last group
                const int c = __popc(m);
                const unsigned b0 = __ballot_sync(0xffffffffu, c & 1), b1 = __ballot_sync(0xffffffffu, c & 2),
                               b2 = __ballot_sync(0xffffffffu, c & 4);
                int p = sh.boff[bk] + __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if ((m >> e) & 1u) {
                        const int idx = c0 + 4 * (bk * kBlkGroups + lane) + e;
                        if (p < kLocCap)
                            loc_i[p] = idx;
                        else
                            oi[p] = idx;
                        ++p;
                    }
                }
            }
        }
        __syncthreads();                                  // the chunk's candidate indices are listed
        // the whole block: keys, the global copy of the list, and the
        // second-level histogram of the digit-T1 keys (one atomic per distinct
        // bin per warp) -- candidates cluster, so this is not left to the warp
        // that found them
        for (int jb = count; jb < count + total; jb += kSelThreads) {   // block-uniform trip count
            const int j = jb + tid;
            int bin = -1;
            if (j < count + total) {
                const int idx = j < kLocCap ? loc_i[j] : oi[j];
                const uint32_t k = f2key(slice[idx - c0]);
                if (j < kLocCap) {
                    loc_k[j] = k;
                    oi[j] = idx;
                }
                ok[j] = k;
                if ((k >> (32 - kHistBits)) == (uint32_t)T1)
                    bin = (int)((k >> kSub) & (kSubBins - 1));
            }
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(same) - 1)
                atomicAdd(&sh.h2[bin], (uint32_t)__popc(same));
        }
        count += total;
        __syncthreads();                                  // before the next chunk overwrites the slice
    }
    if (tid < CL)
        cluster.map_shared_rank(&sh.cnt[0], tid)[rank] = count;
    {   // this rank's second-level histogram to every rank: one uint4 per thread
        static_assert(kExactCluster * kSubBins / 4 == kSelThreads, "push layout");
        const int r = tid / (kSubBins / 4), q4 = tid % (kSubBins / 4);
        if (r < CL)
            reinterpret_cast<uint4 *>(cluster.map_shared_rank(&sh.h2all[rank][0], r))[q4] =
                reinterpret_cast<const uint4 *>(sh.h2)[q4];
    }
    cluster.sync();   // every rank's candidates (shared and global), count and histogram are visible

    // ---- 2. all candidates, identical Top-K in every rank ---------------------
    // The second-level digit T2 (key bits [kSub, 21)) within digit T1: the
    // largest whose suffix count over the cluster, plus the keys above digit
    // T1, reaches min(K, L).  Only keys with (key >> kSub) >= (T1, T2) can be
    // selected.  Thread t (< kSubBins) takes bin kSubBins - 1 - t.
    int N = 0;
#pragma unroll
    for (int r = 0; r < CL; ++r)
        N += sh.cnt[r];
    {
        uint32_t hsum = 0u;
        if (tid < kSubBins) {
#pragma unroll
            for (int r = 0; r < CL; ++r)
                hsum += sh.h2all[r][kSubBins - 1 - tid];
        }
        int tot;
        const int excl = block_excl_scan<kSelThreads>((int)hsum, sh.sel.warp_tot, tot);
        const int need2 = need - (N - tot);            // keys of digit T1 still to select
        if (tid < kSubBins && excl < need2 && excl + (int)hsum >= need2) {
            sh.T2 = kSubBins - 1 - tid;
            sh.above2 = (N - tot) + excl;              // keys above prefix (T1, T2)
        }
    }
    __syncthreads();
    const uint32_t p19 = ((uint32_t)T1 << 8) | (uint32_t)sh.T2;
    // final candidates per rank: its keys above digit T1 plus its digit-T1 keys
    // whose second-level digit is >= T2 (warp r counts rank r)
    if (warp < CL) {
        int all = 0, ge = 0;
#pragma unroll
        for (int i = 0; i < kSubBins / 32; ++i) {
            const int d = lane * (kSubBins / 32) + i;
            const int x = (int)sh.h2all[warp][d];
            all += x;
            ge += d >= sh.T2 ? x : 0;
        }
        all = warp_isum(all);
        ge = warp_isum(ge);
        if (lane == 0)
            sh.wcnt[warp] = sh.cnt[warp] - all + ge;
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int r = 0; r < CL; ++r) {
            sh.off[r] = acc;
            acc += sh.wcnt[r];
        }
        sh.off[CL] = acc;
    }
    __syncthreads();
    const int N2 = sh.off[CL];
    const int32_t *gi = w.cand_idx + (size_t)bh * w.cand_stride;
    const uint32_t *gk = w.cand_key + (size_t)bh * w.cand_stride;
    const bool staged = N2 <= kSelStageCap;
    // Every rank's candidates in its shared memory: warp r of each rank pulls
    // rank r's final candidates in order.  Some rank past kLocCap (long
    // histories): each rank pushes its own, compacted by all its threads.
    int cmax = 0;
#pragma unroll
    for (int r = 0; r < CL; ++r)
        cmax = max(cmax, sh.cnt[r]);
    const bool push = cmax > kLocCap;
    if (staged && !push && warp < CL) {
        // warp r gathers rank r's final candidates in order from its shared memory
        const int r = warp, cr = sh.cnt[r];
        const int32_t *pi = cluster.map_shared_rank(loc_i, r);
        const uint32_t *pk = cluster.map_shared_rank(loc_k, r);
        const unsigned lt = (1u << lane) - 1u;
        int dst = sh.off[r];
        uint32_t km = 0u;   // the largest key: the support's maximum (Eq. (12)'s shift)
        for (int j0 = 0; j0 < cr; j0 += 4 * 32) {
            int32_t ii[4];
            uint32_t kk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * 32 + lane;
                ii[u] = j < cr ? pi[j] : 0;
                kk[u] = j < cr ? pk[j] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool take = (j0 + u * 32 + lane < cr) && (kk[u] >> kSub) >= p19;
                const unsigned bal = __ballot_sync(0xffffffffu, take);
                if (take) {
                    st_idx[dst + __popc(bal & lt)] = ii[u];
                    st_key[dst + __popc(bal & lt)] = kk[u];
                    km = max(km, kk[u]);
                }
                dst += __popc(bal);
            }
        }
        km = __reduce_max_sync(0xffffffffu, km);
        if (lane == 0)
            atomicMax(&sh.kmax, km);
    }
    if (staged && !push)
        for (int i = tid; i < 512; i += kSelThreads)
            (&sh.sel.hist[0][0])[i] = 0u;
    if (staged && push) {
        // this rank compacts its own final candidates (stable, all threads; the
        // first kLocCap from shared memory, the rest from its global segment)
        // and writes them into every rank's staging list at off[rank]
        const int cr = sh.cnt[rank], o0 = sh.off[rank], o1 = sh.off[rank + 1];
        int got = 0;
        for (int base = 0; base < cr; base += kSelThreads * 4) {   // block-uniform trip count
            const int j0 = base + tid * 4;
            int32_t ii[4];
            uint32_t kk[4];
            int c = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u;
                ii[u] = 0;
                kk[u] = 0u;
                if (j < cr) {
                    ii[u] = j < kLocCap ? loc_i[j] : oi[j];
                    kk[u] = j < kLocCap ? loc_k[j] : ok[j];
                    c += (kk[u] >> kSub) >= p19;
                }
            }
            int total;
            int d = o0 + got + block_excl_scan<kSelThreads>(c, sh.sel.warp_tot, total);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j0 + u < cr && (kk[u] >> kSub) >= p19) {
                    if (d < o1) {   // the histogram's count bounds the rank's range
#pragma unroll
                        for (int r2 = 0; r2 < CL; ++r2) {
                            cluster.map_shared_rank(st_idx, r2)[d] = ii[u];
                            cluster.map_shared_rank(st_key, r2)[d] = kk[u];
                        }
                    }
                    ++d;
                }
            }
            got += total;
        }
        for (int i = tid; i < 512; i += kSelThreads)
            (&sh.sel.hist[0][0])[i] = 0u;
        cluster.sync();   // every rank's final candidates are staged in every rank
        uint32_t km = 0u;   // the largest key: the support's maximum (Eq. (12)'s shift)
        for (int j = tid; j < N2; j += kSelThreads)
            km = max(km, st_key[j]);
        km = __reduce_max_sync(0xffffffffu, km);
        if (lane == 0)
            atomicMax(&sh.kmax, km);
    }
    __syncthreads();
    auto get_staged = [&](int j, int32_t &idx, uint32_t &k) {
        idx = st_idx[j];
        k = st_key[j];
    };
    const uint16_t *vb = a.v + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
    int n;
    unsigned long long thr = 0ull;
    if (staged) {
        // every key above prefix (T1, T2) is in; the need - above2 others come
        // from the keys with that prefix.  Those few are listed (in the filter
        // masks' space, dead by now) and ranked by one warp, four per lane
        // (composite keys are distinct); more than kMaxTie of them take the
        // radix refinement, and a histogram that disagreed with the scores (no
        // T2 found) falls back to the full select.
        const int rem = need - sh.above2;
        unsigned long long *tie = reinterpret_cast<unsigned long long *>(sh.gmask);
        if (N2 > need && sh.above2 >= 0) {
            for (int j = tid; j < N2; j += kSelThreads) {
                const uint32_t k = st_key[j];
                if ((k >> kSub) == p19) {
                    const int s = atomicAdd(&sh.ntie, 1);
                    if (s < kMaxTie)
                        tie[s] = key64(k, st_idx[j]);
                }
            }
            __syncthreads();
            if (sh.ntie <= kMaxTie) {
                if (warp == 0) {
                    const int nt = sh.ntie;
                    for (int q = 0; 32 * q < nt; ++q) {   // warp-uniform
                        const int me = 32 * q + lane;
                        const unsigned long long mine = me < nt ? tie[me] : 0ull;
                        int rk = 0;   // how many tied keys are larger
                        for (int i = 0; i < nt; ++i)
                            rk += tie[i] > mine;
                        if (me < nt && rk == rem - 1)
                            sh.tie_thr = mine;
                    }
                }
                __syncthreads();
            }
        }
        thr = N2 <= need           ? 0ull
              : sh.above2 < 0      ? staged_full_select(N2, need, st_idx, st_key, sh.sel)
              : sh.ntie <= kMaxTie ? sh.tie_thr
                                   : staged_refine(N2, rem, p19, st_idx, st_key, sh.sel);
        n = stable_compact<kSelThreads, 4>(N2, thr, get_staged, w.K, sup_i, sup_k, sh.sel.warp_tot);
    } else {
        // more than kSelStageCap final candidates: select among all of them
        // in place, in global memory (offsets of the unfiltered segments)
        if (tid == 0) {
            int acc = 0;
            for (int r = 0; r < CL; ++r) {
                sh.off[r] = acc;
                acc += sh.cnt[r];
            }
            sh.off[CL] = acc;
        }
        __syncthreads();
        n = global_select(N, need, w.K, seg, CL, sh.off, gi, gk, sup_i, sup_k, sh.sel, &sh.kmax);
    }
    __syncthreads();
    const float m = key2f(sh.kmax);
    {   // the support (identical in every rank), written 1/CL per rank
        const int kper = (w.K + CL - 1) / CL;
        const int j0 = rank * kper, j1 = min(w.K, j0 + kper);
        for (int jj = j0 + tid; jj < j1; jj += kSelThreads) {
            const int32_t v = jj < n ? sup_i[jj] : -1;
            if (a.idx_out)
                a.idx_out[(size_t)bh * w.K + jj] = v;
            if (w.support)
                w.support[(size_t)bh * w.K + jj] = v;
            if (insert)
                w.fifo_sup[e_slot * w.K + jj] = v;
        }
        if (rank == 0 && tid == 0) {
            if (a.mode == FIN_DECODE)
                w.M[bh] = L;                       // an exact head "considers" every key
            if (w.support)
                w.sup_len[bh] = n;
            if (insert)
                w.fifo_len[e_slot] = n;
            if (a.mode == FIN_DECODE)
                count_head(w, b, path, N);
        }
    }

    // ---- 3. this rank's share of the value rows (Eq. (12)) -------------------
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float zsum = 0.f;
    if (a.mode != FIN_INIT) {   // cache initialisation needs the support only
        const int vper = (n + CL - 1) / CL;
        const int vs = min(n, rank * vper), ve = min(n, vs + vper);
        value_partial<8>(vb, sup_i, sup_k, vs + warp, ve, kSelWarps, m, acc, zsum, L, w.status);
    }
    *reinterpret_cast<float4 *>(&red[warp][lane * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0)
        sh.zw[warp] = zsum;
    __syncthreads();
    if (tid < kD) {
        float o = 0.f;
#pragma unroll
        for (int ww = 0; ww < kSelWarps; ++ww)
            o += red[ww][tid];
        cluster.map_shared_rank(&sh.part_o[0][0], 0)[rank * kD + tid] = o;
    }
    if (tid == kD) {
        float z = 0.f;
#pragma unroll
        for (int ww = 0; ww < kSelWarps; ++ww)
            z += sh.zw[ww];
        cluster.map_shared_rank(&sh.part_z[0], 0)[rank] = z;
    }
    cluster.sync();   // partials at rank 0; no rank reads a peer's shared memory after this
    if (rank != 0 || a.mode == FIN_INIT)
        return;

    // ---- rank 0: the output ----------------------------------------------------
    if (tid < kD) {
        float o = 0.f, Z = 0.f;
#pragma unroll
        for (int r = 0; r < CL; ++r) {
            o += sh.part_o[r][tid];
            Z += sh.part_z[r];
        }
        o = (n > 0) ? o / Z : 0.f;
        a.out[(size_t)bh * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        if (w.out_f32)
            w.out_f32[(size_t)bh * kD + tid] = o;
    }
}


}  // namespace retopk
