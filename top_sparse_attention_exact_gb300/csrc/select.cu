// select.cu -- the exact path's select kernel for the stateless Exact Top-K
// step and the cache initialisation (ReTopK paper, §Motivation Eq. (1),
// §Recall-Before-Rerank Eq. (12)): one cluster of kExactCluster CTAs per
// (sequence, query head) runs exact_select_body (select_body.cuh) after the
// scan.  Decode steps run the same body inside the fused finish kernel.
#include "select_body.cuh"

namespace retopk {

__global__ void __launch_bounds__(kSelThreads, 2) exact_select_kernel(SelArgs a)
{
    extern __shared__ __align__(128) unsigned char sel_smem[];
    exact_select_body(a, sel_smem);
}


cudaError_t launch_exact_select(const Work &w, QSrc q, const uint16_t *v_cache, const int32_t *seqlens,
                                int len_off, int mode, int init_slot, uint16_t *out, int32_t *idx_out,
                                cudaStream_t st)
{
    SelArgs a;
    a.w = w;
    a.q = q.q;
    a.q_b_stride = q.b_stride;
    a.q_h_stride = q.h_stride;
    a.v = v_cache;
    a.seqlens = seqlens;
    a.out = out;
    a.idx_out = idx_out;
    a.len_off = len_off;
    a.mode = mode;
    a.init_slot = init_slot;
    return launch_pdl(exact_select_kernel, dim3(kExactCluster, w.B * w.Hq), dim3(kSelThreads), sel_smem_bytes(w.K), st, kExactCluster,
                      a);
}

cudaError_t configure_select()
{
    cudaError_t e = cudaFuncSetAttribute(exact_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sel_smem_bytes(kMaxK));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(exact_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

}  // namespace retopk
