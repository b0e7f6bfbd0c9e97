// scan.cu -- full-history QK scan of the exact path (ReTopK paper, §Problem
// Setup Eq. (4): e_i = q . k_i / sqrt(d) for every cached key) fused with the
// first radix digit of the global Top-K (§Motivation Eq. (1)).
//
// One CTA streams a contiguous range of K rows of one (sequence, KV head)
// and scores them against every query head of the GQA group that takes the
// exact path this step, so each K row leaves HBM once per group.  The grouped
// product [16 keys x 128] x [128 x 8 heads] is a dense contraction, so it
// runs on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// Loads go straight from global memory into the A fragments.  The
// contraction dimension is permuted identically for A (keys) and B (queries)
// so that each thread's fragment elements of a key row are contiguous: lane
// (g, t) holds bytes [j*64 + t*16, +16) of rows g and g+8 for j = 0..3, which
// makes every warp load eight fully used 64-byte row segments (no shared
// memory staging, no bank conflicts).  In k-step s the logical columns
// {2t, 2t+1, 2t+8, 2t+9} map to physical elements
// (s>>1)*32 + t*8 + (s&1)*4 + {0,1,2,3}.
//
// Epilogue: scores (fp32) are written to the workspace, and an 11-bit
// histogram of their order-preserving keys is accumulated per head in shared
// memory and flushed with one global atomic per non-empty bin.
#include "common.cuh"

namespace retopk {

struct ScanArgs {
    const uint16_t *q;
    long long q_b_stride, q_h_stride;
    const uint16_t *k;
    const int32_t *seqlens;
    const int32_t *path;
    float *scores;
    uint32_t *hist;
    int Hq, Hkv, G, max_len, n_split, len_off;
    float scale;
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>
__global__ void __launch_bounds__(256) scan_kernel(ScanArgs a)
{
    extern __shared__ uint32_t hist_s[];   // [G][kHistBins]
    const int b = blockIdx.z, hk = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int G = a.G;

    uint32_t mask = 0;
    for (int n = 0; n < G; ++n)
        if (!a.path || a.path[b * a.Hq + hk * G + n] != 0)
            mask |= 1u << n;
    if (!mask)
        return;

    const int L = seq_len(a.seqlens, b, a.len_off, a.max_len);
    const int chunk = (((L + a.n_split - 1) / a.n_split) + 15) & ~15;
    const int start = split * chunk;
    const int end = min(L, start + chunk);
    if (start >= end)
        return;

    for (int i = tid; i < G * kHistBins; i += blockDim.x)
        if ((mask >> (i / kHistBins)) & 1u)
            hist_s[i] = 0;

    // B fragments: query head n = nt*8 + g of the group, same column permutation
    uint4 qf[NT][4];
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
    __syncthreads();

    const uint16_t *kb = a.k + ((size_t)(b * a.Hkv + hk) * a.max_len) * kD;
    float *sc_base = a.scores + (size_t)(b * a.Hq + hk * G) * a.max_len;

    for (int tile = start + warp * 16; tile < end; tile += 8 * 16) {
        const int r0 = tile + g, r1 = tile + g + 8;
        const int l0 = min(r0, end - 1), l1 = min(r1, end - 1);
        const uint4 *p0 = reinterpret_cast<const uint4 *>(kb + (size_t)l0 * kD);
        const uint4 *p1 = reinterpret_cast<const uint4 *>(kb + (size_t)l1 * kD);
        uint4 x0[4], x1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x0[j] = ld_stream(p0 + j * 4 + t);
            x1[j] = ld_stream(p1 + j * 4 + t);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int j = s >> 1;
                const bool hi = s & 1;
                const uint32_t a0 = hi ? x0[j].z : x0[j].x;
                const uint32_t a2 = hi ? x0[j].w : x0[j].y;
                const uint32_t a1 = hi ? x1[j].z : x1[j].x;
                const uint32_t a3 = hi ? x1[j].w : x1[j].y;
                const uint32_t b0 = hi ? qf[nt][j].z : qf[nt][j].x;
                const uint32_t b1 = hi ? qf[nt][j].w : qf[nt][j].y;
                mma_bf16_16816(c, a0, a1, a2, a3, b0, b1);
            }
            // c[0]: (row r0, head 2t)  c[1]: (r0, 2t+1)  c[2]: (r1, 2t)  c[3]: (r1, 2t+1)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = nt * 8 + 2 * t + (e & 1);
                const int r = (e < 2) ? r0 : r1;
                if (n < G && r < end && ((mask >> n) & 1u)) {
                    const float sc = c[e] * a.scale + 0.0f;
                    sc_base[(size_t)n * a.max_len + r] = sc;
                    atomicAdd(&hist_s[n * kHistBins + (f2key(sc) >> (32 - kHistBits))], 1u);
                }
            }
        }
    }
    __syncthreads();
    uint32_t *hg = a.hist + (size_t)(b * a.Hq + hk * G) * kHistBins;
    for (int i = tid; i < G * kHistBins; i += blockDim.x) {
        if ((mask >> (i / kHistBins)) & 1u) {
            const uint32_t v = hist_s[i];
            if (v)
                atomicAdd(&hg[i], v);
        }
    }
}

static size_t scan_smem(int G) { return (size_t)G * kHistBins * sizeof(uint32_t); }

int scan_ctas_per_sm()
{
    static int cached = 0;
    if (!cached) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_kernel<1>, 256, scan_smem(8)) != cudaSuccess || n < 1)
            n = 1;
        cached = n;
    }
    return cached;
}

cudaError_t launch_scan(const Work &w, QSrc q, const uint16_t *k_cache, const int32_t *seqlens,
                        int len_off, cudaStream_t st)
{
    ScanArgs a;
    a.q = q.q;
    a.q_b_stride = q.b_stride;
    a.q_h_stride = q.h_stride;
    a.k = k_cache;
    a.seqlens = seqlens;
    a.path = w.path;
    a.scores = w.scores;
    a.hist = w.hist;
    a.Hq = w.Hq;
    a.Hkv = w.Hkv;
    a.G = w.G;
    a.max_len = w.max_len;
    a.n_split = w.n_scan;
    a.len_off = len_off;
    a.scale = 1.0f / sqrtf((float)kD);
    dim3 grid(w.n_scan, w.Hkv, w.B);
    const size_t smem = scan_smem(w.G);
    if (w.G <= 8)
        scan_kernel<1><<<grid, 256, smem, st>>>(a);
    else
        scan_kernel<2><<<grid, 256, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t configure_scan()
{
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)scan_smem(8));
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(scan_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)scan_smem(kMaxGroup));
}

}  // namespace retopk
