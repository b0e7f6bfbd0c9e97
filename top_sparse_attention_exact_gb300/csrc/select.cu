// select.cu -- Top-K selection and sparse softmax-value aggregation, shared by
// the reuse and the exact path (ReTopK paper, §Complexity and GPU
// Implementation: the two paths differ only in support discovery).
//
//   filter_kernel    exact heads: reads the 11-bit score histogram built by
//                    the scan, finds the digit that holds the K-th largest
//                    score, and compacts every key whose digit is >= it, in
//                    ascending index order, one segment per CTA.  Only these
//                    keys can belong to the Exact Top-K support (Eq. (1)).
//   finalize_kernel  per (sequence, query head): exact Top-K (Eq. (1) or
//                    Eq. (11)) over the candidate list by radix select on a
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
#include "common.cuh"

namespace retopk {

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one int per thread (NT threads, NT % 32 == 0).
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < NT / 32 ? warp_tot[lane] : 0;
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += y;
        }
        if (lane < NT / 32)
            warp_tot[lane] = s - w;
        if (lane == NT / 32 - 1)
            warp_tot[32] = s;
    }
    __syncthreads();
    const int r = warp_tot[warp] + x - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

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

constexpr int kFilterThreads = 512;
constexpr int kFilterPer = 16;                       // scores per thread per chunk

__global__ void __launch_bounds__(kFilterThreads) filter_kernel(FilterArgs a)
{
    __shared__ int warp_tot[33];
    __shared__ int T1_s;
    const int bh = blockIdx.y, s = blockIdx.x, tid = threadIdx.x;
    const int b = bh / a.Hq;
    if (a.path && a.path[bh] == 0)
        return;
    const int L = seq_len(a.seqlens, b, a.len_off, a.max_len);
    const int need = min(a.K, L);

    // threshold digit T1: the largest digit whose suffix count reaches `need`
    constexpr int per = kHistBins / kFilterThreads;   // 4 bins per thread
    static_assert(per == 4, "one uint4 of bins per thread");
    const uint4 hv = reinterpret_cast<const uint4 *>(a.hist + (size_t)bh * kHistBins)[tid];
    const int part = (int)(hv.x + hv.y + hv.z + hv.w);
    if (tid == 0)
        T1_s = 0;
    int tot;
    const int below = block_excl_scan<kFilterThreads>(part, warp_tot, tot);   // bins under mine
    const int above = tot - below - part;                                      // bins over mine
    if (need > 0 && above < need && above + part >= need) {
        int acc = above;
        const uint32_t hb[4] = {hv.x, hv.y, hv.z, hv.w};
        for (int i = per - 1; i >= 0; --i) {
            acc += (int)hb[i];
            if (acc >= need) {
                T1_s = tid * per + i;
                break;
            }
        }
    }
    __syncthreads();
    const uint32_t T1 = (uint32_t)T1_s;

    const int seg = (((L + a.n_filter - 1) / a.n_filter) + 15) & ~15;
    const int start = s * seg;
    const int end = min(L, start + seg);
    const float *sc = a.scores + (size_t)bh * a.sc_stride;
    int32_t *oi = a.cand_idx + (size_t)bh * a.cand_stride + start;
    uint32_t *ok = a.cand_key + (size_t)bh * a.cand_stride + start;
    int count = 0;
    for (int chunk = start; chunk < end; chunk += kFilterThreads * kFilterPer) {   // uniform trip count
        const int i0 = chunk + tid * kFilterPer;
        uint32_t key[kFilterPer];
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
    int warp_tot[33];
    uint32_t hist[2][256];
    int digit, above, cnt_d;
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

    int32_t *st_idx = reinterpret_cast<int32_t *>(fin_smem);                  // [kStageCap]
    uint32_t *st_key = reinterpret_cast<uint32_t *>(st_idx + kStageCap);      // [kStageCap]
    const int Kp = (w.K + 3) & ~3;                                            // keeps `red` 16-byte aligned
    int32_t *sup_i = reinterpret_cast<int32_t *>(st_key + kStageCap);         // [Kp]
    uint32_t *sup_k = reinterpret_cast<uint32_t *>(sup_i + Kp);               // [Kp]
    float *red = reinterpret_cast<float *>(sup_k + Kp);                       // [kFinWarps][kD]

    // ---- candidate segments (reuse: one list of M_t; exact: filter segments)
    int nseg, seg;
    if (path == RETOPK_PATH_REUSE) {
        nseg = 1;
        seg = 0;
        if (tid == 0) {
            sh.seg_off[0] = 0;
            sh.seg_off[1] = w.M[bh];
        }
    } else {
        nseg = w.n_filter;
        seg = (((L + w.n_filter - 1) / w.n_filter) + 15) & ~15;
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
    for (int i = tid; i < 512; i += kFinThreads)
        (&sh.hist[0][0])[i] = 0u;
    __syncthreads();

    // ---- radix select of the `need` largest composite keys (8-bit digits) --
    unsigned long long thr = 0ull;
    if (N > need) {
        unsigned long long prefix = 0ull;
        int rem = need;
        int buf = 0;
        for (int shift = 56; shift >= 0; shift -= 8, buf ^= 1) {
            const unsigned long long hmask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
            uint32_t *hist = sh.hist[buf];
            for (int j = tid; j < N; j += kFinThreads) {
                int32_t idx;
                uint32_t key;
                cv.get(j, idx, key);
                const unsigned long long k64 = key64(key, idx);
                if (((k64 ^ prefix) & hmask) == 0ull)
                    atomicAdd(&hist[(k64 >> shift) & 255ull], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                int c8[8];
                int t8 = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c8[i] = (int)hist[lane * 8 + i];
                    t8 += c8[i];
                }
                int sfx = t8;   // inclusive suffix over lanes >= lane
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_down_sync(0xffffffffu, sfx, o);
                    if (lane + o < 32)
                        sfx += y;
                }
                int above = sfx - t8;
                if (above < rem && rem <= sfx) {
                    for (int i = 7; i >= 0; --i) {
                        if (above + c8[i] >= rem) {
                            sh.digit = lane * 8 + i;
                            sh.above = above;
                            sh.cnt_d = c8[i];
                            break;
                        }
                        above += c8[i];
                    }
                }
            } else if (warp == 1) {
                // clear the other buffer for the next pass
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    sh.hist[buf ^ 1][lane * 8 + i] = 0u;
            }
            __syncthreads();
            rem -= sh.above;
            prefix |= (unsigned long long)sh.digit << shift;
            if (sh.cnt_d == rem)
                break;                 // every key with this prefix is selected
        }
        thr = prefix;
    }

    // ---- stable compaction: the support in ascending index order -----------
    int got = 0;
    for (int base = 0; base < N; base += kFinThreads) {
        const int j = base + tid;
        int32_t idx = 0;
        uint32_t key = 0;
        int flag = 0;
        if (j < N) {
            cv.get(j, idx, key);
            flag = key64(key, idx) >= thr;
        }
        int total;
        const int pos = block_excl_scan<kFinThreads>(flag, sh.warp_tot, total);
        if (flag && got + pos < w.K) {
            sup_i[got + pos] = idx;
            sup_k[got + pos] = key;
        }
        got += total;
    }
    const int n = min(got, w.K);

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
    if (a.mode != FIN_INIT) {   // cache initialisation needs the support only
        // warp `warp` owns support rows warp, warp+32, ...; 16 loads in flight per lane
        for (int j0 = warp; j0 < n; j0 += kFinWarps * 16) {
            uint2 vv[16];
            float p[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int j = j0 + u * kFinWarps;
                if (j < n) {
                    vv[u] = *reinterpret_cast<const uint2 *>(vb + (size_t)sup_i[j] * kD + lane * 4);
                    p[u] = expf(key2f(sup_k[j]) - m);
                } else {
                    vv[u] = make_uint2(0u, 0u);
                    p[u] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                zsum += p[u];
                acc[0] += p[u] * bf16lo(vv[u].x);
                acc[1] += p[u] * bf16hi(vv[u].x);
                acc[2] += p[u] * bf16lo(vv[u].y);
                acc[3] += p[u] * bf16hi(vv[u].y);
            }
        }
    }
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
    if (a.mode == FIN_DECODE && tid == 0) {
        unsigned long long *cnt = w.counters + (size_t)b * CNT_WORDS;
        atomicAdd(&cnt[path == RETOPK_PATH_REUSE ? CNT_REUSE
                       : path == RETOPK_PATH_FALLBACK ? CNT_FALLBACK : CNT_REFRESH], 1ull);
        if (path == RETOPK_PATH_REUSE) {
            atomicAdd(&cnt[CNT_SUM_M], (unsigned long long)N);
            atomicMax(&cnt[CNT_MAX_M], (unsigned long long)N);
        }
        // the last head of the sequence to finish advances the ring and t_dec
        __threadfence();
        const int prev = atomicAdd(&w.seq[b * SEQ_WORDS + SEQ_DONE], 1);
        if (prev == w.Hq - 1) {
            __threadfence();
            int *sq = w.seq + b * SEQ_WORDS;
            const int head = *(volatile int *)&sq[SEQ_HEAD];
            const int count = *(volatile int *)&sq[SEQ_COUNT];
            sq[SEQ_HEAD] = (head + 1) % w.C;
            sq[SEQ_COUNT] = min(count + 1, w.C);
            sq[SEQ_TDEC] = *(volatile int *)&sq[SEQ_TDEC] + 1;
            sq[SEQ_DONE] = 0;
        }
    }
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
