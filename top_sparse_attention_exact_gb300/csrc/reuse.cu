// reuse.cu -- the path decision of one decode step (ReTopK paper,
// §Recall-Before-Rerank Selection and §Reliable Reuse): one CTA per
// (sequence, query head) computes
//   Eq. (6)  the cosine of q_t to each cached query,
//   Eq. (7)  Top-R (ties to the older entry) and rho_max,
//   Eq. (13) the path (refresh / similarity fallback / reuse),
// and publishes them to global memory; for an exact-path head it also clears
// the head's score histogram for the scan.  The scan then streams the groups
// with an exact head, and the finish kernel serves every head: the reuse path
// (reuse_body.cuh) or the exact select (select_body.cuh).
#include "reuse_body.cuh"

namespace retopk {

constexpr int kDecideThreads = 256;
static_assert(kMaxC <= kDecideThreads, "one cache entry per thread");

struct DecideArgs {
    Work w;
    const uint16_t *q;
    // when not null, each CTA copies its head's q row here (the step's later
    // kernels read q from this device copy; q itself may be host memory)
    uint16_t *q_copy;
    // the token's K/V rows when the append is fused into this launch (else null)
    const uint16_t *k_new, *v_new;
    uint16_t *k_cache, *v_cache;
    int32_t *seqlens;
};

struct DecideShared {
    float qf[kD];
    float dot[kMaxC];      // by slot
    float nrm[kMaxC];      // by slot
    float rho[kMaxC];      // by live position (0 = oldest)
    int topr[kMaxC + 1];   // live positions by rank
    float nq;
};

// Eqs. (6), (7), (13) for one (sequence, query head) per CTA.
__global__ void __launch_bounds__(kDecideThreads) decide_kernel(DecideArgs a)
{
    __shared__ DecideShared sh;
    {   // the head's cached queries (C rows of 256 bytes in the workspace)
        // into the L2 while the grid before this one (the previous step's or
        // layer's back end) finishes: a hint only, every value is read after
        // the wait
        const char *fq = reinterpret_cast<const char *>(a.w.fifo_q + (size_t)blockIdx.x * a.w.C * kD);
        for (int i = threadIdx.x; i < a.w.C * kD * 2 / 128; i += kDecideThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(fq + (size_t)i * 128));
    }
    pdl_wait();      // the previous step is done with the caches, lengths and ring
    pdl_trigger();   // the scan may set up while the decision runs
    const Work &w = a.w;
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq;
    if (a.k_new && bh % w.Hq == 0) {
        // the fused append: head 0's CTA writes sequence b's new K/V rows at
        // row L and sets L += 1 (no other CTA of this launch reads L)
        const int L = a.seqlens[b];
        if (L >= w.max_len) {
            if (tid == 0)
                atomicOr(w.status, RETOPK_STATUS_KV_FULL);
        } else {
            constexpr int kPer = kD / 8;   // uint4 per row
            for (int i = tid; i < 2 * w.Hkv * kPer; i += kDecideThreads) {
                const int which = i / (w.Hkv * kPer), r = i % (w.Hkv * kPer), hk = r / kPer, c = r % kPer;
                const uint4 *src = reinterpret_cast<const uint4 *>((which ? a.v_new : a.k_new) + ((size_t)b * w.Hkv + hk) * kD);
                uint4 *dst = reinterpret_cast<uint4 *>((which ? a.v_cache : a.k_cache) +
                                                       (((size_t)b * w.Hkv + hk) * w.max_len + L) * kD);
                dst[c] = src[c];
            }
            if (tid == 0)
                a.seqlens[b] = L + 1;
        }
    }
    const int *sq = w.seq + b * SEQ_WORDS;
    const int head = sq[SEQ_HEAD], count = sq[SEQ_COUNT], done = sq[SEQ_TDEC];
    const int t_dec = done + 1;
    if (tid == 0 && bh % w.Hq == 0) {   // the step's view of the ring, for the finish kernel
        int *sn = w.snap + b * SEQ_WORDS;
        sn[SEQ_HEAD] = head;
        sn[SEQ_COUNT] = count;
        sn[SEQ_TDEC] = done;
    }
    if (tid < kD)
        sh.qf[tid] = __uint_as_float(((uint32_t)a.q[(size_t)bh * kD + tid]) << 16);
    if (a.q_copy && tid < kD / 8)
        reinterpret_cast<uint4 *>(a.q_copy + (size_t)bh * kD)[tid] =
            reinterpret_cast<const uint4 *>(a.q + (size_t)bh * kD)[tid];
    const uint2 qraw = *reinterpret_cast<const uint2 *>(a.q + (size_t)bh * kD + lane * 4);
    const float q0 = bf16lo(qraw.x), q1 = bf16hi(qraw.x), q2 = bf16lo(qraw.y), q3 = bf16hi(qraw.y);
    for (int s0 = warp * 4; s0 < w.C; s0 += (kDecideThreads / 32) * 4) {
        uint2 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            raw[u] = (s0 + u < w.C)
                         ? *reinterpret_cast<const uint2 *>(w.fifo_q + ((size_t)bh * w.C + s0 + u) * kD + lane * 4)
                         : make_uint2(0u, 0u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float x0 = bf16lo(raw[u].x), x1 = bf16hi(raw[u].x), x2 = bf16lo(raw[u].y), x3 = bf16hi(raw[u].y);
            float dq = q0 * x0 + q1 * x1 + q2 * x2 + q3 * x3;
            float nc = x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
            dq = warp_sum(dq);
            nc = warp_sum(nc);
            if (lane == 0 && s0 + u < w.C) {
                sh.dot[s0 + u] = dq;
                sh.nrm[s0 + u] = nc;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            s += sh.qf[lane * 4 + c] * sh.qf[lane * 4 + c];
        s = warp_sum(s);
        if (lane == 0)
            sh.nq = s;
    }
    __syncthreads();
    // Eq. (6) for live entry c (0 = oldest) in slot (head - count + c) mod C
    for (int c = tid; c < count; c += kDecideThreads) {
        const int slot = ((head - count + c) % w.C + w.C) % w.C;
        const float nc = sh.nrm[slot], dq = sh.dot[slot];
        sh.rho[c] = (sh.nq > 0.f && nc > 0.f) ? dq / (sqrtf(sh.nq) * sqrtf(nc)) : -INFINITY;
    }
    __syncthreads();
    // Eq. (7): Top-R by (rho desc, older first); or the R newest entries
    if (w.retrieval == RETOPK_RETRIEVE_RECENT) {
        const int nr = min(w.R, count);
        for (int r = tid; r < nr; r += kDecideThreads)
            sh.topr[r] = count - 1 - r;
        __syncthreads();
        if (tid == 0) {   // rho_max over the retrieved entries
            float m = -INFINITY;
            for (int r = 0; r < nr; ++r)
                m = fmaxf(m, sh.rho[count - 1 - r]);
            sh.nq = m;    // (|q|^2 is not needed any more)
        }
    }
    for (int c = tid; c < count && w.retrieval != RETOPK_RETRIEVE_RECENT; c += kDecideThreads) {
        const float r = sh.rho[c];
        int rk = 0;
#pragma unroll 8
        for (int c2 = 0; c2 < count; ++c2) {
            const float r2 = sh.rho[c2];
            rk += (r2 > r) || (r2 == r && c2 < c);
        }
        sh.topr[rk] = c;
    }
    __syncthreads();
    const float rmax = count == 0 ? -INFINITY : (w.retrieval == RETOPK_RETRIEVE_RECENT ? sh.nq : sh.rho[sh.topr[0]]);
    const bool refresh = (w.T_r > 0) && (t_dec % w.T_r == 0);   // Eq. (13), checked first
    const int p = refresh ? RETOPK_PATH_REFRESH : (!(rmax >= w.tau) ? RETOPK_PATH_FALLBACK : RETOPK_PATH_REUSE);
    if (tid == 0) {
        w.path[bh] = p;
        w.rho_max[bh] = rmax;
    }
    for (int r = tid; r < w.R; r += kDecideThreads)
        w.topR[(size_t)bh * w.R + r] = r < count ? sh.topr[r] : -1;
    if (p != RETOPK_PATH_REUSE) {   // exact head: a clean histogram for the scan
        uint4 *hg = reinterpret_cast<uint4 *>(w.hist + (size_t)bh * kHistBins);
        for (int i = tid; i < kHistBins / 4; i += kDecideThreads)
            hg[i] = make_uint4(0u, 0u, 0u, 0u);
        if (w.prefilter) {          // and for the prefilter's second-digit histograms
            uint4 *h2 = reinterpret_cast<uint4 *>(w.pf_h2 + (size_t)bh * kExactCluster * 256);
            for (int i = tid; i < kExactCluster * 256 / 4; i += kDecideThreads)
                h2[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

cudaError_t launch_decide(const Work &w, const uint16_t *q, uint16_t *q_copy, const uint16_t *k_new,
                          const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache, int32_t *seqlens,
                          cudaStream_t st)
{
    const DecideArgs a{w, q, q_copy, k_new, v_new, k_cache, v_cache, seqlens};
    return launch_pdl(decide_kernel, dim3(w.B * w.Hq), dim3(kDecideThreads), 0, st, 1, a);
}


}  // namespace retopk
