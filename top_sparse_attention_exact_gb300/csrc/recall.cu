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
//                  The same kernel then computes the exact scores
//                  q_t . k_i / sqrt(d) of the candidate keys only (Eq. (10)),
//                  gathered straight from the K cache with 16-byte loads (half
//                  a warp per key row); several CTAs share one head's
//                  candidates.
//   append_kernel  writes the new token's key and value rows and advances L.
#include "common.cuh"

namespace retopk {

struct RecallArgs {
    Work w;
    const uint16_t *q;
    const uint16_t *k;
    const int32_t *seqlens;
    float scale;
};

constexpr int kRecallThreads = 256;
constexpr int kRerankRows = 8;       // key rows per half-warp per round

// grid (n_rerank, B*Hq).  Every CTA of a head recomputes the (cheap, exactly
// reproducible) recall and candidate set; CTA x then scores candidates
// [x*per, (x+1)*per).  CTA 0 publishes path, rho_max, R_t, M_t and A_t.
__global__ void __launch_bounds__(kRecallThreads) recall_kernel(RecallArgs a)
{
    extern __shared__ uint32_t rsm[];   // bitmap [ceil(L/32)] then A_t [R*K+W]
    __shared__ float qf[kD];
    __shared__ float rho[kMaxC];
    __shared__ int topr[kMaxC];
    __shared__ int flen[kMaxC];
    __shared__ float dot_s[kMaxC];
    __shared__ float nrm_s[kMaxC];
    __shared__ int warp_tot[9];
    __shared__ float nq_s;
    __shared__ int path_s;
    const Work &w = a.w;
    const int bh = blockIdx.y, split = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq, hk = (bh % w.Hq) / w.G;
    const int L = seq_len(a.seqlens, b, 0, w.max_len);
    const int *sq = w.seq + b * SEQ_WORDS;
    const int head = sq[SEQ_HEAD], count = sq[SEQ_COUNT];
    const int t_dec = sq[SEQ_TDEC] + 1;
    uint32_t *bitmap = rsm;
    const int nwords = (L + 31) >> 5;
    int32_t *cand_s = reinterpret_cast<int32_t *>(rsm + ((w.max_len + 31) >> 5));

    if (tid < kD)
        qf[tid] = __uint_as_float(((uint32_t)a.q[(size_t)bh * kD + tid]) << 16);
    for (int c = tid; c < count; c += kRecallThreads) {
        const int slot = ((head - count + c) % w.C + w.C) % w.C;
        flen[c] = w.fifo_len[(size_t)bh * w.C + slot];
    }
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
    // Eq. (6): rho_c = D(q, q_c) / sqrt(D(q,q) D(q_c,q_c)), live entry c oldest
    // first; each warp loads up to 4 cached queries at once
    for (int c0 = warp * 4; c0 < count; c0 += 8 * 4) {
        uint2 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u;
            const int slot = ((head - count + c) % w.C + w.C) % w.C;
            raw[u] = (c < count) ? *reinterpret_cast<const uint2 *>(w.fifo_q + ((size_t)bh * w.C + slot) * kD + lane * 4)
                                 : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float x0 = bf16lo(raw[u].x), x1 = bf16hi(raw[u].x), x2 = bf16lo(raw[u].y), x3 = bf16hi(raw[u].y);
            float dqc = qf[lane * 4] * x0 + qf[lane * 4 + 1] * x1 + qf[lane * 4 + 2] * x2 + qf[lane * 4 + 3] * x3;
            float ncc = x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
            dqc = warp_sum(dqc);
            ncc = warp_sum(ncc);
            if (lane == 0 && c0 + u < count) {
                dot_s[c0 + u] = dqc;
                nrm_s[c0 + u] = ncc;
            }
        }
    }
    __syncthreads();
    const float nq = nq_s;
    for (int c = tid; c < count; c += kRecallThreads) {
        const float ncc = nrm_s[c], dqc = dot_s[c];
        rho[c] = (nq > 0.f && ncc > 0.f) ? (float)((double)dqc / sqrt((double)nq * (double)ncc)) : -INFINITY;
    }
    __syncthreads();
    // Eq. (7): Top-R by (rho desc, older first); rank by counting
    for (int c = tid; c < count; c += kRecallThreads) {
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
        if (split == 0) {
            w.path[bh] = p;
            w.rho_max[bh] = rmax;
        }
    }
    if (split == 0)
        for (int r = tid; r < w.R; r += kRecallThreads)
            w.topR[(size_t)bh * w.R + r] = r < count ? topr[r] : -1;
    // Eqs. (8)-(9): bitmap union of the window and the retrieved supports
    for (int i = tid; i < nwords; i += kRecallThreads)
        bitmap[i] = 0u;
    __syncthreads();
    if (path_s != RETOPK_PATH_REUSE) {
        if (split == 0) {
            uint32_t *hg = w.hist + (size_t)bh * kHistBins;
            for (int i = tid; i < kHistBins; i += kRecallThreads)
                hg[i] = 0u;
            if (tid == 0)
                w.M[bh] = L;
        }
        return;
    }
    const int lo = max(0, L - w.W);
    for (int i = lo + tid; i < L; i += kRecallThreads)
        atomicOr(&bitmap[i >> 5], 1u << (i & 31));
    const int nr = min(w.R, count);
    for (int r = 0; r < nr; ++r) {
        const int c = topr[r];
        const int slot = ((head - count + c) % w.C + w.C) % w.C;
        const int len = flen[c];
        const int32_t *sp = w.fifo_sup + ((size_t)bh * w.C + slot) * w.K;
        for (int j0 = tid; j0 < len; j0 += kRecallThreads * 4) {
            int id[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kRecallThreads;
                id[u] = j < len ? sp[j] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kRecallThreads;
                if (j < len) {
                    const int i = id[u];
                    if (i >= 0 && i < L)
                        atomicOr(&bitmap[i >> 5], 1u << (i & 31));
                    else if (split == 0)
                        atomicOr(w.status, RETOPK_STATUS_BAD_INDEX);
                }
            }
        }
    }
    __syncthreads();
    // ascending emission into shared memory: each thread owns a run of words
    const int wpt = (nwords + kRecallThreads - 1) / kRecallThreads;
    const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
    int mine = 0;
    for (int i = w0; i < w1; ++i)
        mine += __popc(bitmap[i]);
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
        for (int i = 0; i < kRecallThreads / 32; ++i) {
            const int v = warp_tot[i];
            warp_tot[i] = acc;
            acc += v;
        }
        warp_tot[8] = acc;
    }
    __syncthreads();
    int pos = warp_tot[warp] + x - mine;
    for (int i = w0; i < w1; ++i) {
        uint32_t bits = bitmap[i];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            cand_s[pos++] = (i << 5) + bit;
            bits &= bits - 1;
        }
    }
    __syncthreads();
    const int M = warp_tot[8];
    int32_t *ci = w.cand_idx + (size_t)bh * w.cand_stride;
    if (split == 0) {
        for (int j = tid; j < M; j += kRecallThreads)
            ci[j] = cand_s[j];
        if (tid == 0)
            w.M[bh] = M;
    }
    // Eq. (10): exact scores of this CTA's candidate slice, half a warp per key
    // row, kRerankRows rows in flight per half-warp
    const int per = (M + gridDim.x - 1) / gridDim.x;
    const int start = split * per, end = min(M, start + per);
    const int hw = tid >> 4, hl = tid & 15;
    const float *qq = qf + hl * 8;
    const uint16_t *kb = a.k + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
    uint32_t *ck = w.cand_key + (size_t)bh * w.cand_stride;
    for (int j0 = start + hw; j0 < end; j0 += (kRecallThreads / 16) * kRerankRows) {
        uint4 kv[kRerankRows];
#pragma unroll
        for (int u = 0; u < kRerankRows; ++u) {
            const int j = j0 + u * (kRecallThreads / 16);
            kv[u] = (j < end) ? reinterpret_cast<const uint4 *>(kb + (size_t)cand_s[j] * kD)[hl]
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kRerankRows; ++u) {
            float s = qq[0] * bf16lo(kv[u].x) + qq[1] * bf16hi(kv[u].x) + qq[2] * bf16lo(kv[u].y) +
                      qq[3] * bf16hi(kv[u].y) + qq[4] * bf16lo(kv[u].z) + qq[5] * bf16hi(kv[u].z) +
                      qq[6] * bf16lo(kv[u].w) + qq[7] * bf16hi(kv[u].w);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);
            const int j = j0 + u * (kRecallThreads / 16);
            if (hl == 0 && j < end)
                ck[j] = f2key(s * a.scale + 0.0f);
        }
    }
}

static size_t recall_smem_bytes(int max_len, int RKW)
{
    return (size_t)((max_len + 31) >> 5) * 4 + (size_t)RKW * 4;
}

cudaError_t launch_recall(const Work &w, const uint16_t *q, const uint16_t *k_cache, const int32_t *seqlens,
                          cudaStream_t st)
{
    RecallArgs a{w, q, k_cache, seqlens, 1.0f / sqrtf((float)kD)};
    dim3 grid(w.n_rerank, w.B * w.Hq);
    recall_kernel<<<grid, kRecallThreads, recall_smem_bytes(w.max_len, w.R * w.K + w.W), st>>>(a);
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

cudaError_t configure_recall()
{
    // the largest request: max_len = 2^20 keys and R*K+W = kMaxC*kMaxK/16 candidates
    return cudaFuncSetAttribute(recall_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

size_t recall_smem_need(int max_len, int RKW) { return recall_smem_bytes(max_len, RKW); }

}  // namespace retopk
