// select.cu -- Top-K selection and sparse softmax-value aggregation, shared by
// the reuse and the exact path (ReTopK paper, §Complexity and GPU
// Implementation: the two paths differ only in support discovery).
//
//   filter_kernel    exact heads: reads the 11-bit score histogram built by
//                    the scan, finds the digit that holds the K-th largest
//                    score, and compacts every key whose digit is >= it, in
//                    ascending index order, one segment per CTA.  Only these
//                    keys can belong to the Exact Top-K support (Eq. (1)).
//   finalize_kernel  per exact-path (sequence, query head): Top-K (Eq. (1))
//                    over the filter's candidate list by radix select on a
//                    64-bit key (score, then lower index), stable compaction
//                    so the support comes out in ascending index order,
//                    softmax over its scores and the weighted sum of the V
//                    rows (Eq. (12)), the bf16 output, and -- on decode
//                    steps -- insertion of (q_t, support) into the
//                    query-support cache (Eq. (5)) and the t_dec advance.
//
// Both kernels are latency-bound at batch 1, so every thread issues all of its
// global loads before it consumes any of them, and the number of block-wide
// barriers is kept small.
#include "topk.cuh"

namespace retopk {

// ---------------------------------------------------------------------------
struct FilterArgs {
    const int32_t *seqlens;
    const int32_t *path;
    const float *scores;
    const uint32_t *hist;
    int32_t *cand_idx;
    uint32_t *cand_key;
    int32_t *seg_count;
    int Hq, max_len, sc_stride, K, n_filter, cand_stride, len_off;
};

constexpr int kFilterThreads = 256;
constexpr int kFilterPer = 32;                       // scores per thread per chunk

__global__ void __launch_bounds__(kFilterThreads) filter_kernel(FilterArgs a)
{
    __shared__ int warp_tot[33];
    __shared__ __align__(16) uint32_t hist_s[kHistBins];   // filled with 16-byte stores
    __shared__ int T1_s;
    const int bh = blockIdx.y, s = blockIdx.x, tid = threadIdx.x;
    const int b = bh / a.Hq;
    if (a.path && a.path[bh] == 0)
        return;
    const int L = seq_len(a.seqlens, b, a.len_off, a.max_len);
    const int need = min(a.K, L);
    const int seg = (((L + a.n_filter - 1) / a.n_filter) + 15) & ~15;
    const int start = s * seg;
    const int end = min(L, start + seg);
    const float *sc = a.scores + (size_t)bh * a.sc_stride;

    // issue the first chunk's score loads and the histogram loads together
    auto load_chunk = [&](int i0, uint32_t (&key)[kFilterPer]) {
        if (i0 + kFilterPer <= end) {
#pragma unroll
            for (int v = 0; v < kFilterPer / 4; ++v) {
                const float4 f = reinterpret_cast<const float4 *>(sc + i0)[v];
                key[4 * v + 0] = f2key(f.x);
                key[4 * v + 1] = f2key(f.y);
                key[4 * v + 2] = f2key(f.z);
                key[4 * v + 3] = f2key(f.w);
            }
        } else {
#pragma unroll
            for (int e = 0; e < kFilterPer; ++e)
                key[e] = (i0 + e < end) ? f2key(sc[i0 + e]) : 0u;
        }
    };
    uint32_t key[kFilterPer];
    load_chunk(start + tid * kFilterPer, key);
    {
        const uint4 *hg = reinterpret_cast<const uint4 *>(a.hist + (size_t)bh * kHistBins);
        uint4 hv[kHistBins / 4 / kFilterThreads];
#pragma unroll
        for (int u = 0; u < kHistBins / 4 / kFilterThreads; ++u)
            hv[u] = hg[tid + u * kFilterThreads];
#pragma unroll
        for (int u = 0; u < kHistBins / 4 / kFilterThreads; ++u)
            reinterpret_cast<uint4 *>(hist_s)[tid + u * kFilterThreads] = hv[u];
    }
    if (tid == 0)
        T1_s = 0;
    __syncthreads();
    // threshold digit T1: the largest digit whose suffix count reaches `need`;
    // thread t owns the 8 digits [8t, 8t+8)
    constexpr int per = kHistBins / kFilterThreads;
    int part = 0;
#pragma unroll
    for (int i = 0; i < per; ++i)
        part += (int)hist_s[tid * per + i];
    int tot;
    const int below = block_excl_scan<kFilterThreads>(part, warp_tot, tot);
    const int above = tot - below - part;
    if (need > 0 && above < need && above + part >= need) {
        int acc = above;
        for (int i = per - 1; i >= 0; --i) {
            acc += (int)hist_s[tid * per + i];
            if (acc >= need) {
                T1_s = tid * per + i;
                break;
            }
        }
    }
    __syncthreads();
    const uint32_t T1 = (uint32_t)T1_s;

    int32_t *oi = a.cand_idx + (size_t)bh * a.cand_stride + start;
    uint32_t *ok = a.cand_key + (size_t)bh * a.cand_stride + start;
    int count = 0;
    for (int chunk = start; chunk < end; chunk += kFilterThreads * kFilterPer) {   // uniform trip count
        const int i0 = chunk + tid * kFilterPer;
        if (chunk != start)
            load_chunk(i0, key);
        int n = 0;
#pragma unroll
        for (int e = 0; e < kFilterPer; ++e)
            n += (i0 + e < end) && ((key[e] >> (32 - kHistBits)) >= T1);
        int total;
        int pos = count + block_excl_scan<kFilterThreads>(n, warp_tot, total);
#pragma unroll
        for (int e = 0; e < kFilterPer; ++e) {
            if ((i0 + e < end) && ((key[e] >> (32 - kHistBits)) >= T1)) {
                oi[pos] = i0 + e;
                ok[pos] = key[e];
                ++pos;
            }
        }
        count += total;
    }
    if (tid == 0)
        a.seg_count[(size_t)bh * a.n_filter + s] = count;
}

cudaError_t launch_filter(const Work &w, const int32_t *seqlens, int len_off, cudaStream_t st)
{
    FilterArgs a;
    a.seqlens = seqlens;
    a.path = w.path;
    a.scores = w.scores;
    a.hist = w.hist;
    a.cand_idx = w.cand_idx;
    a.cand_key = w.cand_key;
    a.seg_count = w.seg_count;
    a.Hq = w.Hq;
    a.max_len = w.max_len;
    a.sc_stride = w.sc_stride;
    a.K = w.K;
    a.n_filter = w.n_filter;
    a.cand_stride = w.cand_stride;
    a.len_off = len_off;
    dim3 grid(w.n_filter, w.B * w.Hq);
    filter_kernel<<<grid, kFilterThreads, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
struct FinArgs {
    Work w;
    const uint16_t *q;
    long long q_b_stride, q_h_stride;
    const uint16_t *v;
    const int32_t *seqlens;
    uint16_t *out;
    int32_t *idx_out;
    int len_off, mode, init_slot;
};

constexpr int kFinThreads = 1024;
constexpr int kFinWarps = kFinThreads / 32;

struct FinShared {
    int seg_off[kMaxSeg + 1];
    SelectShared sel;
    uint32_t kmax;
    float Z_w[kFinWarps];
    int slot;
};

// Candidate j of the head's virtual list (segments concatenated in order).
struct CandView {
    const int32_t *gi;
    const uint32_t *gk;
    const int32_t *si;
    const uint32_t *sk;
    const int *seg_off;
    int nseg, seg;
    bool staged;
    __device__ __forceinline__ int goff(int j) const
    {
        int lo = 0, hi = nseg - 1;            // last segment with seg_off[s] <= j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seg_off[mid] <= j)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo * seg + (j - seg_off[lo]);
    }
    __device__ __forceinline__ void get(int j, int32_t &idx, uint32_t &key) const
    {
        if (staged) {
            idx = si[j];
            key = sk[j];
        } else {
            const int o = goff(j);
            idx = gi[o];
            key = gk[o];
        }
    }
};

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(FinArgs a)
{
    extern __shared__ __align__(16) unsigned char fin_smem[];
    __shared__ FinShared sh;
    const Work &w = a.w;
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq, h = bh % w.Hq, hk = h / w.G;
    const int L = seq_len(a.seqlens, b, a.len_off, w.max_len);
    const int path = (a.mode == FIN_DECODE) ? w.path[bh] : RETOPK_PATH_FALLBACK;
    if (path == RETOPK_PATH_REUSE)
        return;   // the reuse kernel has served this head

    int32_t *st_idx = reinterpret_cast<int32_t *>(fin_smem);                  // [kStageCap]
    uint32_t *st_key = reinterpret_cast<uint32_t *>(st_idx + kStageCap);      // [kStageCap]
    const int Kp = (w.K + 3) & ~3;                                            // keeps `red` 16-byte aligned
    int32_t *sup_i = reinterpret_cast<int32_t *>(st_key + kStageCap);         // [Kp]
    uint32_t *sup_k = reinterpret_cast<uint32_t *>(sup_i + Kp);               // [Kp]
    float *red = reinterpret_cast<float *>(sup_k + Kp);                       // [kFinWarps][kD]

    // ---- candidate segments written by the filter kernel ---------------------
    const int nseg = w.n_filter;
    const int seg = (((L + w.n_filter - 1) / w.n_filter) + 15) & ~15;
    if (warp == 0) {
        // nseg <= 64: two counts per lane, warp-wide inclusive scan
        const int c0 = (2 * lane < nseg) ? w.seg_count[(size_t)bh * nseg + 2 * lane] : 0;
        const int c1 = (2 * lane + 1 < nseg) ? w.seg_count[(size_t)bh * nseg + 2 * lane + 1] : 0;
        int x = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        const int ex = x - c0 - c1;
        if (2 * lane <= nseg)
            sh.seg_off[2 * lane] = ex;
        if (2 * lane + 1 <= nseg)
            sh.seg_off[2 * lane + 1] = ex + c0;
    }
    __syncthreads();
    const int N = sh.seg_off[nseg];
    const int need = min(w.K, N);
    const int32_t *gi = w.cand_idx + (size_t)bh * w.cand_stride;
    const uint32_t *gk = w.cand_key + (size_t)bh * w.cand_stride;
    CandView cv{gi, gk, st_idx, st_key, sh.seg_off, nseg, seg, N <= kStageCap};
    if (cv.staged) {
#pragma unroll 4
        for (int j = tid; j < N; j += kFinThreads) {
            const int o = (nseg == 1) ? j : cv.goff(j);
            st_idx[j] = gi[o];
            st_key[j] = gk[o];
        }
    }
    __syncthreads();

    // ---- Eq. (1): the K best candidates, ascending index order ---------------
    auto get = [&](int j, int32_t &idx, uint32_t &key) { cv.get(j, idx, key); };
    const unsigned long long thr = radix_select_threshold<kFinThreads>(N, need, get, sh.sel);
    const int n = stable_compact<kFinThreads>(N, thr, get, w.K, sup_i, sup_k, sh.sel.warp_tot);

    // ---- softmax over the support and value aggregation (Eq. (12)) --------
    if (tid == 0)
        sh.kmax = 0u;
    __syncthreads();
    {
        uint32_t km = 0u;
        for (int j = tid; j < n; j += kFinThreads)
            km = max(km, sup_k[j]);
        km = __reduce_max_sync(0xffffffffu, km);
        if (lane == 0)
            atomicMax(&sh.kmax, km);
    }
    __syncthreads();
    const float m = key2f(sh.kmax);
    const uint16_t *vb = a.v + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float zsum = 0.f;
    if (a.mode != FIN_INIT)   // cache initialisation needs the support only
        value_partial(vb, sup_i, sup_k, warp, n, kFinWarps, m, acc, zsum);
    *reinterpret_cast<float4 *>(red + warp * kD + lane * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0)
        sh.Z_w[warp] = zsum;
    if ((a.mode == FIN_DECODE || a.mode == FIN_INIT) && tid == 0)
        sh.slot = (a.mode == FIN_INIT) ? a.init_slot : w.seq[b * SEQ_WORDS + SEQ_HEAD];
    __syncthreads();
    if (a.mode != FIN_INIT && tid < kD) {
        float o = 0.f, Z = 0.f;
#pragma unroll 8
        for (int ww = 0; ww < kFinWarps; ++ww) {
            o += red[ww * kD + tid];
            Z += sh.Z_w[ww];
        }
        o = (n > 0) ? o / Z : 0.f;
        a.out[(size_t)bh * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        if (w.out_f32)
            w.out_f32[(size_t)bh * kD + tid] = o;
    }

    // ---- support outputs, cache insertion ----------------------------------
    if (a.idx_out) {
        for (int jj = tid; jj < w.K; jj += kFinThreads)
            a.idx_out[(size_t)bh * w.K + jj] = jj < n ? sup_i[jj] : -1;
    }
    if (w.support) {
        for (int jj = tid; jj < w.K; jj += kFinThreads)
            w.support[(size_t)bh * w.K + jj] = jj < n ? sup_i[jj] : -1;
        if (tid == 0)
            w.sup_len[bh] = n;
    }
    if (a.mode == FIN_DECODE || a.mode == FIN_INIT) {
        const int slot = sh.slot;
        const size_t e = (size_t)bh * w.C + slot;
        const uint16_t *qrow = a.q + b * a.q_b_stride + (long long)h * a.q_h_stride;
        if (tid < kD / 8)
            reinterpret_cast<uint4 *>(w.fifo_q + e * kD)[tid] = reinterpret_cast<const uint4 *>(qrow)[tid];
        for (int jj = tid; jj < w.K; jj += kFinThreads)
            w.fifo_sup[e * w.K + jj] = jj < n ? sup_i[jj] : -1;
        if (tid == 0)
            w.fifo_len[e] = n;
    }
    if (a.mode == FIN_DECODE && tid == 0)
        finish_head(w, b, path, N);
}

static size_t fin_smem_bytes(int K)
{
    return (size_t)kStageCap * 8 + (size_t)((K + 3) & ~3) * 8 + (size_t)kFinWarps * kD * 4;
}

cudaError_t launch_finalize(const Work &w, QSrc q, const uint16_t *v_cache, const int32_t *seqlens,
                            int len_off, int mode, int init_slot, uint16_t *out, int32_t *idx_out,
                            cudaStream_t st)
{
    FinArgs a;
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
    finalize_kernel<<<w.B * w.Hq, kFinThreads, fin_smem_bytes(w.K), st>>>(a);
    return cudaGetLastError();
}

cudaError_t configure_select()
{
    return cudaFuncSetAttribute(finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)fin_smem_bytes(kMaxK));
}

}  // namespace retopk
