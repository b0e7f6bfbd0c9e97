// finish.cu -- the back end of a decode step, after the path decision and the
// scan: one cluster of w.cluster CTAs (1, 2, 4 or 8) per (sequence, query
// head) serves the head on its path (ReTopK paper, Eq. (13)):
//   reuse   -> reuse_body (reuse_body.cuh): Eqs. (8)-(12) over the candidates
//              A_t, then the cache insertion;
//   exact   -> exact_select_body (select_body.cuh): Eq. (1) over the scan's
//              scores, Eq. (12), then the cache insertion.
// Both kinds of head run side by side in one launch (the path is uniform over
// a cluster); the two bodies overlay the same dynamic shared memory.
#include <algorithm>

#include "reuse_body.cuh"
#include "select_body.cuh"

namespace retopk {

static_assert(kReuseThreads == kSelThreads && kReuseCluster == kExactCluster, "one launch shape for both paths");

// the exact select fits for every K; the reuse path's size depends on max_len,
// R*K + W and the cluster size together and is checked per configuration
// (finish_smem_bytes_for)
static_assert(kSelSharedBytes + kSelRegionBytes + (size_t)kLocCap * 8 + (size_t)kMaxK * 8 <= kMaxDynSmem,
              "the exact select fits one CTA's shared memory for every K");

template <int CL>
__global__ void __launch_bounds__(kSelThreads, 2) finish_kernel(SelArgs sa, ReuseArgs ra)
{
    extern __shared__ __align__(128) unsigned char fin_smem[];
    // Launched programmatically after the scan, so it may start while the scan
    // runs.  A reuse head needs nothing from the scan: what it reads was
    // written by the decision and the append, which completed before the scan
    // passed its own wait (the scan lets this grid launch only after that).
    // An exact head waits for the scan inside exact_select_body.
    const Work &w = sa.w;
    // The next grid on the stream (the next step's or the next layer's
    // decision) may launch now: it only prefetches before its own wait, which
    // returns once this grid has completed.
    pdl_trigger();
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y % w.Hq == 0) {
        // the ring advance of Eq. (5) (slot, live count, t_dec): nothing later
        // in this step reads `seq`, every head takes its slot from `snap`
        const int b = blockIdx.y / w.Hq;
        const int *sn = w.snap + b * SEQ_WORDS;
        int *sq = w.seq + b * SEQ_WORDS;
        sq[SEQ_HEAD] = (sn[SEQ_HEAD] + 1) % w.C;
        sq[SEQ_COUNT] = min(sn[SEQ_COUNT] + 1, w.C);
        sq[SEQ_TDEC] = sn[SEQ_TDEC] + 1;
    }
    if (w.path[blockIdx.y] == RETOPK_PATH_REUSE)   // uniform over the cluster
        reuse_body<CL>(ra, fin_smem);
    else
        exact_select_body<CL>(sa, fin_smem);
    // Reuse heads never wait for the grid before this one (the scan, or the
    // exact-head prefilter), so on a step without exact heads nothing would.
    // One CTA waiting before it exits keeps this grid from completing before
    // that one: the next step's decision, which waits for this grid, then
    // never overlaps a kernel of this step that still reads the paths.
    if (blockIdx.x == 0 && blockIdx.y == 0)
        pdl_wait();
}

size_t finish_smem_bytes_for(int max_len, int K, int RKW, int CL)
{
    return std::max(sel_smem_bytes(K), reuse_smem_bytes(max_len, RKW, CL));
}

static size_t finish_smem_bytes(const Work &w)
{
    return finish_smem_bytes_for(w.max_len, w.K, w.R * w.K + w.W, w.cluster);
}

cudaError_t launch_finish(const Work &w, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *seqlens, uint16_t *out, cudaStream_t st)
{
    SelArgs sa;
    sa.w = w;
    sa.q = q;
    sa.q_b_stride = (long long)w.Hq * kD;
    sa.q_h_stride = kD;
    sa.v = v_cache;
    sa.seqlens = seqlens;
    sa.out = out;
    sa.idx_out = nullptr;
    sa.len_off = 0;
    sa.mode = FIN_DECODE;
    sa.init_slot = 0;
    const ReuseArgs ra{w, q, k_cache, v_cache, seqlens, out, 1.0f / sqrtf((float)kD)};
    const dim3 grid(w.cluster, w.B * w.Hq), block(kSelThreads);
    const size_t smem = finish_smem_bytes(w);
    switch (w.cluster) {
    case 1: return launch_pdl(finish_kernel<1>, grid, block, smem, st, 1, sa, ra);
    case 2: return launch_pdl(finish_kernel<2>, grid, block, smem, st, 2, sa, ra);
    case 4: return launch_pdl(finish_kernel<4>, grid, block, smem, st, 4, sa, ra);
    case 8: return launch_pdl(finish_kernel<8>, grid, block, smem, st, 8, sa, ra);
    default: return cudaErrorInvalidValue;
    }
}

template <int CL>
static cudaError_t configure_one()
{
    cudaError_t e =
        cudaFuncSetAttribute(finish_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(finish_kernel<CL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t configure_finish()
{
    cudaError_t e = configure_one<1>();
    if (e == cudaSuccess)
        e = configure_one<2>();
    if (e == cudaSuccess)
        e = configure_one<4>();
    if (e == cudaSuccess)
        e = configure_one<8>();
    return e;
}

}  // namespace retopk
