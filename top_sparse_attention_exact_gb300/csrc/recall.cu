// recall.cu -- the reuse path's support discovery (ReTopK paper,
// §Recall-Before-Rerank Selection and §Reliable Reuse), plus the KV append.
//
//   recall_kernel  per (sequence, query head): cosine of q_t to every cached
//                  query (Eq. (6)), Top-R with ties to the older entry and
//                  rho_max (Eq. (7)), the path rule (Eq. (13)); on reuse, the
//                  candidate set A_t = Unique(retrieved supports U recent
//                  window) (Eqs. (8)-(9)) built in a shared-memory bitmap of
//                  L bits and emitted in ascending order.  Exact heads get
//                  their score histogram cleared for the scan.
//   rerank_kernel  exact scores q_t . k_i / sqrt(d) of the candidate keys only
//                  (Eq. (10)), gathered straight from the K cache with
//                  16-byte loads (half a warp per key row).
//   append_kernel  writes the new token's key and value rows and advances L.
#include "common.cuh"

namespace retopk {

struct RecallArgs {
    Work w;
    const uint16_t *q;
    const int32_t *seqlens;
};

__global__ void __launch_bounds__(256) recall_kernel(RecallArgs a)
{
    extern __shared__ uint32_t bitmap[];
    __shared__ float qf[kD];
    __shared__ float rho[kMaxC];
    __shared__ int topr[kMaxC];
    __shared__ int warp_tot[9];
    __shared__ float nq_s;
    __shared__ int path_s;
    const Work &w = a.w;
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq;
    const int L = seq_len(a.seqlens, b, 0, w.max_len);
    const int *sq = w.seq + b * SEQ_WORDS;
    const int head = sq[SEQ_HEAD], count = sq[SEQ_COUNT];
    const int t_dec = sq[SEQ_TDEC] + 1;

    if (tid < kD)
        qf[tid] = __uint_as_float(((uint32_t)a.q[(size_t)bh * kD + tid]) << 16);
    __syncthreads();
    if (warp == 0) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            s += qf[lane * 4 + c] * qf[lane * 4 + c];
        s = warp_sum(s);
        if (lane == 0)
            nq_s = s;
    }
    __syncthreads();
    const float nq = nq_s;
    // Eq. (6): rho_c = D(q, q_c) / sqrt(D(q,q) D(q_c,q_c)), live entry c oldest first
    for (int c = warp; c < count; c += 8) {
        const int slot = ((head - count + c) % w.C + w.C) % w.C;
        const uint2 raw = *reinterpret_cast<const uint2 *>(w.fifo_q + ((size_t)bh * w.C + slot) * kD + lane * 4);
        const float x0 = bf16lo(raw.x), x1 = bf16hi(raw.x), x2 = bf16lo(raw.y), x3 = bf16hi(raw.y);
        float dqc = qf[lane * 4] * x0 + qf[lane * 4 + 1] * x1 + qf[lane * 4 + 2] * x2 + qf[lane * 4 + 3] * x3;
        float ncc = x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
        dqc = warp_sum(dqc);
        ncc = warp_sum(ncc);
        if (lane == 0)
            rho[c] = (nq > 0.f && ncc > 0.f) ? (float)((double)dqc / sqrt((double)nq * (double)ncc))
                                              : -INFINITY;
    }
    __syncthreads();
    // Eq. (7): Top-R by (rho desc, older first); rank by counting
    for (int c = tid; c < count; c += blockDim.x) {
        const float r = rho[c];
        int rank = 0;
        for (int c2 = 0; c2 < count; ++c2) {
            const float r2 = rho[c2];
            rank += (r2 > r) || (r2 == r && c2 < c);
        }
        topr[rank] = c;
    }
    __syncthreads();
    if (tid == 0) {
        const float rmax = count > 0 ? rho[topr[0]] : -INFINITY;
        // Eq. (13): refresh first, then the similarity fallback (strict <)
        const bool refresh = (w.T_r > 0) && (t_dec % w.T_r == 0);
        const int p = refresh ? RETOPK_PATH_REFRESH : (!(rmax >= w.tau) ? RETOPK_PATH_FALLBACK : RETOPK_PATH_REUSE);
        path_s = p;
        w.path[bh] = p;
        w.rho_max[bh] = rmax;
    }
    for (int r = tid; r < w.R; r += blockDim.x)
        w.topR[(size_t)bh * w.R + r] = r < count ? topr[r] : -1;
    __syncthreads();
    if (path_s != RETOPK_PATH_REUSE) {
        uint32_t *hg = w.hist + (size_t)bh * kHistBins;
        for (int i = tid; i < kHistBins; i += blockDim.x)
            hg[i] = 0u;
        if (tid == 0)
            w.M[bh] = L;
        return;
    }
    // Eqs. (8)-(9): bitmap union of the window and the retrieved supports
    const int nwords = (L + 31) >> 5;
    for (int i = tid; i < nwords; i += blockDim.x)
        bitmap[i] = 0u;
    __syncthreads();
    const int lo = max(0, L - w.W);
    for (int i = lo + tid; i < L; i += blockDim.x)
        atomicOr(&bitmap[i >> 5], 1u << (i & 31));
    const int nr = min(w.R, count);
    for (int r = 0; r < nr; ++r) {
        const int slot = ((head - count + topr[r]) % w.C + w.C) % w.C;
        const size_t e = (size_t)bh * w.C + slot;
        const int len = w.fifo_len[e];
        const int32_t *sp = w.fifo_sup + e * w.K;
        for (int j = tid; j < len; j += blockDim.x) {
            const int i = sp[j];
            if (i >= 0 && i < L)
                atomicOr(&bitmap[i >> 5], 1u << (i & 31));
            else
                atomicOr(w.status, RETOPK_STATUS_BAD_INDEX);
        }
    }
    __syncthreads();
    // ascending emission: each thread owns a contiguous run of words
    const int wpt = (nwords + blockDim.x - 1) / blockDim.x;
    const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
    int mine = 0;
    for (int i = w0; i < w1; ++i)
        mine += __popc(bitmap[i]);
    // block exclusive scan of `mine` (8 warps)
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_tot[warp] = x;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i < 8; ++i) {
            const int v = warp_tot[i];
            warp_tot[i] = acc;
            acc += v;
        }
        warp_tot[8] = acc;
    }
    __syncthreads();
    int pos = warp_tot[warp] + x - mine;
    int32_t *out = w.cand_idx + (size_t)bh * w.cand_stride;
    for (int i = w0; i < w1; ++i) {
        uint32_t bits = bitmap[i];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            out[pos++] = (i << 5) + bit;
            bits &= bits - 1;
        }
    }
    if (tid == 0)
        w.M[bh] = warp_tot[8];
}

cudaError_t launch_recall(const Work &w, const uint16_t *q, const int32_t *seqlens, cudaStream_t st)
{
    RecallArgs a{w, q, seqlens};
    const size_t smem = (size_t)((w.max_len + 31) / 32) * 4;
    recall_kernel<<<w.B * w.Hq, 256, smem, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
struct RerankArgs {
    const int32_t *path;
    const int32_t *M;
    const int32_t *cand_idx;
    uint32_t *cand_key;
    const uint16_t *q;
    const uint16_t *k;
    const int32_t *seqlens;
    int Hq, Hkv, G, max_len, cand_stride, n_split;
    float scale;
};

__global__ void __launch_bounds__(256) rerank_kernel(RerankArgs a)
{
    const int bh = blockIdx.y, split = blockIdx.x, tid = threadIdx.x;
    if (a.path[bh] != RETOPK_PATH_REUSE)
        return;
    const int b = bh / a.Hq, hk = (bh % a.Hq) / a.G;
    const int M = a.M[bh];
    const int per = (M + a.n_split - 1) / a.n_split;
    const int start = split * per, end = min(M, start + per);
    if (start >= end)
        return;
    const int hw = tid >> 4, hl = tid & 15;
    const uint4 qv = reinterpret_cast<const uint4 *>(a.q + (size_t)bh * kD)[hl];
    const float q0 = bf16lo(qv.x), q1 = bf16hi(qv.x), q2 = bf16lo(qv.y), q3 = bf16hi(qv.y);
    const float q4 = bf16lo(qv.z), q5 = bf16hi(qv.z), q6 = bf16lo(qv.w), q7 = bf16hi(qv.w);
    const uint16_t *kb = a.k + ((size_t)(b * a.Hkv + hk) * a.max_len) * kD;
    const int32_t *ci = a.cand_idx + (size_t)bh * a.cand_stride;
    uint32_t *ck = a.cand_key + (size_t)bh * a.cand_stride;
    for (int j0 = start + hw; j0 < end; j0 += 16 * 4) {
        uint4 kv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * 16;
            if (j < end)
                kv[u] = reinterpret_cast<const uint4 *>(kb + (size_t)ci[j] * kD)[hl];
            else
                kv[u] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float s = q0 * bf16lo(kv[u].x) + q1 * bf16hi(kv[u].x) + q2 * bf16lo(kv[u].y) +
                      q3 * bf16hi(kv[u].y) + q4 * bf16lo(kv[u].z) + q5 * bf16hi(kv[u].z) +
                      q6 * bf16lo(kv[u].w) + q7 * bf16hi(kv[u].w);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);
            const int j = j0 + u * 16;
            if (hl == 0 && j < end)
                ck[j] = f2key(s * a.scale + 0.0f);
        }
    }
}

cudaError_t launch_rerank(const Work &w, const uint16_t *q, const uint16_t *k_cache,
                          const int32_t *seqlens, cudaStream_t st)
{
    RerankArgs a;
    a.path = w.path;
    a.M = w.M;
    a.cand_idx = w.cand_idx;
    a.cand_key = w.cand_key;
    a.q = q;
    a.k = k_cache;
    a.seqlens = seqlens;
    a.Hq = w.Hq;
    a.Hkv = w.Hkv;
    a.G = w.G;
    a.max_len = w.max_len;
    a.cand_stride = w.cand_stride;
    a.n_split = w.n_rerank;
    a.scale = 1.0f / sqrtf((float)kD);
    dim3 grid(w.n_rerank, w.B * w.Hq);
    rerank_kernel<<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
__global__ void append_kernel(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                              uint16_t *v_cache, int32_t *seqlens, uint32_t *status, int Hkv,
                              int max_len)
{
    const int b = blockIdx.x;
    const int L = seqlens[b];
    if (L >= max_len) {
        if (threadIdx.x == 0)
            atomicOr(status, RETOPK_STATUS_KV_FULL);
        return;
    }
    const int per_row = kD / 8;   // uint4 per row
    for (int i = threadIdx.x; i < 2 * Hkv * per_row; i += blockDim.x) {
        const int which = i / (Hkv * per_row);
        const int r = i % (Hkv * per_row);
        const int hk = r / per_row, c = r % per_row;
        const uint4 *src = reinterpret_cast<const uint4 *>((which ? v_new : k_new) + ((size_t)b * Hkv + hk) * kD);
        uint4 *dst = reinterpret_cast<uint4 *>((which ? v_cache : k_cache) +
                                               (((size_t)b * Hkv + hk) * max_len + L) * kD);
        dst[c] = src[c];
    }
    __syncthreads();
    if (threadIdx.x == 0)
        seqlens[b] = L + 1;
}

cudaError_t launch_append(const Work &w, const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *k_cache, uint16_t *v_cache, int32_t *seqlens, cudaStream_t st)
{
    append_kernel<<<w.B, 128, 0, st>>>(k_new, v_new, k_cache, v_cache, seqlens, w.status, w.Hkv, w.max_len);
    return cudaGetLastError();
}

// After cache initialisation: C entries in slots 0..C-1, next slot 0, t_dec 0.
__global__ void init_done_kernel(int32_t *seq, unsigned long long *counters, int B, int C)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        seq[b * SEQ_WORDS + SEQ_HEAD] = 0;
        seq[b * SEQ_WORDS + SEQ_COUNT] = C;
        seq[b * SEQ_WORDS + SEQ_TDEC] = 0;
        seq[b * SEQ_WORDS + SEQ_DONE] = 0;
        for (int i = 0; i < CNT_WORDS; ++i)
            counters[(size_t)b * CNT_WORDS + i] = 0ull;
    }
}

cudaError_t launch_init_done(const Work &w, cudaStream_t st)
{
    init_done_kernel<<<(w.B + 127) / 128, 128, 0, st>>>(w.seq, w.counters, w.B, w.C);
    return cudaGetLastError();
}

cudaError_t configure_recall(int max_len_words_bytes)
{
    return cudaFuncSetAttribute(recall_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_len_words_bytes);
}

}  // namespace retopk
