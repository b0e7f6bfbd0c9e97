// select.cu -- the exact path's select kernel for the stateless Exact Top-K
// step and the cache initialisation (ReTopK paper, §Motivation Eq. (1),
// §Recall-Before-Rerank Eq. (12)): one cluster of w.cluster CTAs (1, 2, 4 or
// 8) per (sequence, query head) runs exact_select_body (select_body.cuh)
// after the scan.  Decode steps run the same body inside the fused finish
// kernel.
#include "select_body.cuh"

namespace retopk {

template <int CL>
__global__ void __launch_bounds__(kSelThreads, 2) exact_select_kernel(SelArgs a)
{
    extern __shared__ __align__(128) unsigned char sel_smem[];
    pdl_trigger();   // the next grid on the stream waits for this one before it reads anything
    exact_select_body<CL>(a, sel_smem);
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
    const dim3 grid(w.cluster, w.B * w.Hq), block(kSelThreads);
    const size_t smem = sel_smem_bytes(w.K);
    switch (w.cluster) {
    case 1: return launch_pdl(exact_select_kernel<1>, grid, block, smem, st, 1, a);
    case 2: return launch_pdl(exact_select_kernel<2>, grid, block, smem, st, 2, a);
    case 4: return launch_pdl(exact_select_kernel<4>, grid, block, smem, st, 4, a);
    case 8: return launch_pdl(exact_select_kernel<8>, grid, block, smem, st, 8, a);
    default: return cudaErrorInvalidValue;
    }
}

template <int CL>
static cudaError_t configure_one()
{
    cudaError_t e = cudaFuncSetAttribute(exact_select_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sel_smem_bytes(kMaxK));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(exact_select_kernel<CL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t configure_select()
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
