// prefilter.cu -- the first-digit filter of the exact heads of a long-history
// decode step, spread over the whole GPU (ReTopK paper, §Motivation Eq. (1):
// only keys whose first radix digit reaches the threshold digit T1 can be in
// the Exact Top-K support).
//
// A decode step at a long history usually has one or two exact heads, whose
// select runs on one cluster of 8 CTAs: each CTA would filter its 1/8 of the
// scores window by window (kSliceCap scores each, dozens of windows at
// millions of keys) while the rest of the GPU idles.  Between the scan and
// the finish kernel, this persistent kernel takes the (exact head, rank,
// window) items instead, one per CTA at a time: it finds T1 from the head's
// histogram (as the select does), copies the window into shared memory
// (TMA), lists the window's candidates (index and key, ascending) at offset
// window * kSliceCap of the rank's global candidate segment, writes their
// count, and adds their second-digit counts to the rank's histogram pf_h2.
// The select then only compacts each rank's lists (select_body.cuh,
// "prefiltered").  Used when the context has 8 CTAs per head, more than one
// window per CTA at max_len and at most kPfMaxHeads heads.
#include "select_body.cuh"

namespace retopk {

struct PfArgs {
    Work w;
    const int32_t *seqlens;
};

struct PfShared {
    int nlist;
    int list[kPfMaxHeads];   // the exact heads, in order
};

__global__ void __launch_bounds__(kSelThreads, 2) prefilter_kernel(PfArgs a)
{
    extern __shared__ __align__(128) unsigned char pf_smem[];
    __shared__ PfShared ps;
    SelShared &sh = *reinterpret_cast<SelShared *>(pf_smem);
    float *slice = reinterpret_cast<float *>(pf_smem + kSelSharedBytes);
    const Work &w = a.w;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&sh.bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();      // the scan's scores and histograms, the decision's paths
    pdl_trigger();   // the finish kernel may launch: its exact heads wait for this grid
    if (tid == 0) {
        int n = 0;
        for (int bh = 0; bh < w.B * w.Hq; ++bh)
            if (w.path[bh] != RETOPK_PATH_REUSE)
                ps.list[n++] = bh;
        ps.nlist = n;
    }
    __syncthreads();
    const int per_head = kExactCluster * w.pf_nw;
    const int items = ps.nlist * per_head;
    uint32_t parity = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {   // block-uniform
        const int bh = ps.list[it / per_head], x = it % per_head, r = x / w.pf_nw, v = x % w.pf_nw;
        const int b = bh / w.Hq;
        const int L = seq_len(a.seqlens, b, 0, w.max_len);
        const int need = min(w.K, L);
        const int seg = (((L + kExactCluster - 1) / kExactCluster) + 15) & ~15;   // as the select's ranks
        const int rs = min(L, r * seg), re = min(L, rs + seg);
        const int c0 = rs + v * kSliceCap;
        int32_t *cnt_out = w.pf_cnt + ((size_t)bh * kExactCluster + r) * w.pf_nw + v;
        if (c0 >= re) {
            if (tid == 0)
                *cnt_out = 0;
            continue;
        }
        const int n = min(re - c0, kSliceCap);
        const float *sc = w.scores + (size_t)bh * w.sc_stride;
        int32_t *oi = w.cand_idx + (size_t)bh * w.cand_stride + (size_t)r * seg + (size_t)v * kSliceCap;
        uint32_t *ok = w.cand_key + (size_t)bh * w.cand_stride + (size_t)r * seg + (size_t)v * kSliceCap;
        uint32_t *h2 = w.pf_h2 + ((size_t)bh * kExactCluster + r) * kSubBins;
        // the window into shared memory (the <= 3 trailing scores by plain loads)
        const int nb = n & ~3;
        if (tid == 0 && nb > 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier reads of the buffer
            mbar_expect_tx(&sh.bar, (uint32_t)nb * 4u);
            bulk_load(slice, sc + c0, (uint32_t)nb * 4u, &sh.bar);
        }
        if (tid < n - nb)
            slice[nb + tid] = sc[c0 + nb + tid];
        // T1 from the head's histogram
        if (tid == 0)
            sh.T1 = 0;
        __syncthreads();
        const uint4 hv = reinterpret_cast<const uint4 *>(w.hist + (size_t)bh * kHistBins)[tid];
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
        const uint32_t T1 = (uint32_t)sh.T1;
        const uint32_t tkey = T1 << (32 - kHistBits);
        const uint32_t tcmp = tkey >= 0x80000000u ? (tkey & 0x7fffffffu) : ~tkey;
        if (nb > 0 && !mbar_wait(&sh.bar, parity, w.status)) {
            if (tid == 0)   // the copy may still be in flight: wait once more before reusing the buffer
                mbar_wait(&sh.bar, parity, w.status);
        }
        if (nb > 0)
            parity ^= 1u;
        __syncthreads();   // trailing plain loads visible
        // pass 1: per block of 128 scores, the candidate masks and their count
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
                sh.boff[tid] = ex;
        }
        __syncthreads();
        // pass 2: index and key of every candidate, ascending, and the
        // second digit of the digit-T1 keys
        const unsigned lt = (1u << lane) - 1u;
        for (int bk = warp; bk < nblk; bk += kSelWarps) {   // warp-uniform
            if (sh.bcnt[bk] == 0)
                continue;
            const unsigned m = sh.gmask[bk * kBlkGroups + lane];
            const int c = __popc(m);
            const unsigned b0 = __ballot_sync(0xffffffffu, c & 1), b1 = __ballot_sync(0xffffffffu, c & 2),
                           b2 = __ballot_sync(0xffffffffu, c & 4);
            int p = sh.boff[bk] + __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if ((m >> e) & 1u) {
                    const int loc = 4 * (bk * kBlkGroups + lane) + e;
                    const uint32_t k = f2key(slice[loc]);
                    oi[p] = c0 + loc;
                    ok[p] = k;
                    if ((k >> (32 - kHistBits)) == T1)
                        atomicAdd(&h2[(k >> kSub) & (kSubBins - 1)], 1u);
                    ++p;
                }
            }
        }
        if (tid == 0)
            *cnt_out = total;
        __syncthreads();   // before the next item overwrites the window
    }
}

cudaError_t launch_prefilter(const Work &w, const int32_t *seqlens, cudaStream_t st)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return cudaErrorInvalidValue;
    const long long items = (long long)w.B * w.Hq * kExactCluster * w.pf_nw;
    const int grid = (int)std::max(1LL, std::min<long long>(items, 2LL * sms));
    const PfArgs a{w, seqlens};
    return launch_pdl(prefilter_kernel, dim3(grid), dim3(kSelThreads), kSelSharedBytes + (size_t)kSliceCap * 4, st, 1,
                      a);
}

cudaError_t configure_prefilter()
{
    cudaError_t e = cudaFuncSetAttribute(prefilter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kSelSharedBytes + (size_t)kSliceCap * 4));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefilter_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

}  // namespace retopk
