// reuse.cu -- the whole ReTopK reuse path of one decode step in one kernel
// (ReTopK paper, §Recall-Before-Rerank Selection, §Reliable Reuse and
// §Complexity and GPU Implementation: cache matching, Top-R retrieval,
// candidate union and dedup, indexed rerank, Top-K, indexed softmax-value
// aggregation and cache update, fused).
//
// One cluster of kReuseCluster CTAs serves one (sequence, query head).  Every
// CTA of the cluster recomputes the cheap, exactly reproducible front half:
//   Eq. (6)  cosine of q_t to each cached query,
//   Eq. (7)  Top-R (ties to the older entry) and rho_max,
//   Eq. (13) the path (refresh / similarity fallback / reuse),
//   Eqs. (8)-(9) the candidate set A_t (window U retrieved supports) through a
//            shared-memory bitmap of L bits, emitted in ascending order,
// so that the cluster agrees on A_t without communication.  The work that
// touches HBM is split across the cluster:
//   Eq. (10) each CTA scores 1/kReuseCluster of the candidate keys (K rows
//            gathered straight from the cache) and pushes the scores into
//            every peer's shared memory (distributed shared memory);
//   Eq. (11) after a cluster barrier each CTA holds all M_t scores and runs
//            the same radix select -> identical support S_t;
//   Eq. (12) each CTA aggregates 1/kReuseCluster of the support's V rows with
//            the common max, pushes (sum of weights, weighted sum) to rank 0;
// after a second barrier rank 0 normalises, writes the output and inserts
// (q_t, S_t) into the query-support cache (Eq. (5)).
// Heads on the exact path only publish their path here (and clear their score
// histogram for the scan); the scan and exact-select kernels serve them.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstddef>

#include "topk.cuh"

namespace cg = cooperative_groups;

namespace retopk {

constexpr int kReuseThreads = 256;
constexpr int kReuseWarps = kReuseThreads / 32;
constexpr int kReuseCluster = 8;
constexpr int kRerankRows = 8;        // key rows in flight per half-warp

struct ReuseArgs {
    Work w;
    const uint16_t *q;
    const uint16_t *k;
    const uint16_t *v;
    const int32_t *seqlens;
    uint16_t *out;
    float scale;
};

struct ReuseShared {
    float qf[kD];
    float dot[kMaxC];      // by slot
    float nrm[kMaxC];      // by slot
    int flen[kMaxC];       // by slot
    float rho[kMaxC];      // by live position (0 = oldest)
    int topr[kMaxC + 1];   // live positions by rank
    int pre[kMaxC + 1];    // prefix of the retrieved supports' lengths
    float nq;
    int path;
    int sup_off[kMaxC];    // cache offset of each retrieved support
    int wcount[kReuseWarps];
    uint32_t kmax;
    SelectShared sel;
    alignas(16) float red[kReuseWarps][kD];          // written with 16-byte stores
    float zw[kReuseWarps];
    alignas(16) float part_o[kReuseCluster][kD];     // rank 0 receives every rank's partial
    float part_z[kReuseCluster];
};
static_assert(offsetof(ReuseShared, red) % 16 == 0, "16-byte stores into red");
static_assert(offsetof(ReuseShared, part_o) % 16 == 0, "partials aligned");

__global__ void __launch_bounds__(kReuseThreads) reuse_kernel(ReuseArgs a)
{
    extern __shared__ __align__(16) uint32_t rsm[];
    __shared__ ReuseShared sh;
    cg::cluster_group cluster = cg::this_cluster();
    const Work &w = a.w;
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq, h = bh % w.Hq, hk = h / w.G;
    const int RKW = w.R * w.K + w.W;
    uint32_t *region = rsm;                                           // bitmap, then the scores
    const int region_words = max((w.max_len + 31) >> 5, RKW);
    int32_t *cand = reinterpret_cast<int32_t *>(rsm + region_words);  // A_t, then S_t
    uint32_t *keys = region;

    // ---- front half: every load issued before any is consumed ----------------
    const int L = seq_len(a.seqlens, b, 0, w.max_len);
    const int *sq = w.seq + b * SEQ_WORDS;
    const int head = sq[SEQ_HEAD], count = sq[SEQ_COUNT];
    const int t_dec = sq[SEQ_TDEC] + 1;
    if (tid < kD)
        sh.qf[tid] = __uint_as_float(((uint32_t)a.q[(size_t)bh * kD + tid]) << 16);
    for (int s = tid; s < w.C; s += kReuseThreads)
        sh.flen[s] = w.fifo_len[(size_t)bh * w.C + s];
    const uint2 qraw = *reinterpret_cast<const uint2 *>(a.q + (size_t)bh * kD + lane * 4);
    const float q0 = bf16lo(qraw.x), q1 = bf16hi(qraw.x), q2 = bf16lo(qraw.y), q3 = bf16hi(qraw.y);
    for (int s0 = warp * 4; s0 < w.C; s0 += kReuseWarps * 4) {
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
    for (int c = tid; c < count; c += kReuseThreads) {
        const int slot = ((head - count + c) % w.C + w.C) % w.C;
        const float nc = sh.nrm[slot], dq = sh.dot[slot];
        sh.rho[c] = (sh.nq > 0.f && nc > 0.f) ? dq / (sqrtf(sh.nq) * sqrtf(nc)) : -INFINITY;
    }
    __syncthreads();
    // Eq. (7): Top-R by (rho desc, older first)
    for (int c = tid; c < count; c += kReuseThreads) {
        const float r = sh.rho[c];
        int rk = 0;
        for (int c2 = 0; c2 < count; ++c2) {
            const float r2 = sh.rho[c2];
            rk += (r2 > r) || (r2 == r && c2 < c);
        }
        sh.topr[rk] = c;
    }
    __syncthreads();
    const int nr = min(w.R, count);
    if (tid == 0) {
        const float rmax = count > 0 ? sh.rho[sh.topr[0]] : -INFINITY;
        const bool refresh = (w.T_r > 0) && (t_dec % w.T_r == 0);   // Eq. (13), checked first
        const int p = refresh ? RETOPK_PATH_REFRESH : (!(rmax >= w.tau) ? RETOPK_PATH_FALLBACK : RETOPK_PATH_REUSE);
        sh.path = p;
        if (rank == 0) {
            w.path[bh] = p;
            w.rho_max[bh] = rmax;
        }
        int acc = 0;   // prefix of the retrieved supports' lengths
        for (int r = 0; r < nr; ++r) {
            sh.pre[r] = acc;
            acc += sh.flen[((head - count + sh.topr[r]) % w.C + w.C) % w.C];
        }
        sh.pre[nr] = acc;
    }
    if (rank == 0)
        for (int r = tid; r < w.R; r += kReuseThreads)
            w.topR[(size_t)bh * w.R + r] = r < count ? sh.topr[r] : -1;
    const int nwords = (L + 31) >> 5;
    for (int i = tid; i < nwords; i += kReuseThreads)
        region[i] = 0u;
    __syncthreads();
    if (sh.path != RETOPK_PATH_REUSE) {          // uniform over the whole cluster
        if (rank == 0) {
            uint32_t *hg = w.hist + (size_t)bh * kHistBins;
            for (int i = tid; i < kHistBins; i += kReuseThreads)
                hg[i] = 0u;
            if (tid == 0)
                w.M[bh] = L;
        }
        return;
    }

    // ---- Eqs. (8)-(9): candidate bitmap -------------------------------------
    // recent window [lo, L): one thread per bitmap word
    const int lo = max(0, L - w.W);
    if (lo < L) {
        for (int wd = (lo >> 5) + tid; wd <= ((L - 1) >> 5); wd += kReuseThreads) {
            const int a0 = max(lo, wd << 5) - (wd << 5), a1 = min(L, (wd << 5) + 32) - (wd << 5);
            const uint32_t msk = (a1 - a0 == 32) ? 0xffffffffu : (((1u << (a1 - a0)) - 1u) << a0);
            atomicOr(&region[wd], msk);
        }
    }
    // thread t walks a contiguous run of the concatenated (ascending) support
    // lists, so neighbouring indices share a bitmap word: OR them in a register
    // and issue one shared atomic per word change
    const int T = sh.pre[nr];
    if (tid < nr)
        sh.sup_off[tid] = (int)(((size_t)bh * w.C + (((head - count + sh.topr[tid]) % w.C + w.C) % w.C)) * w.K);
    __syncthreads();
    {
        const int per_t = (T + kReuseThreads - 1) / kReuseThreads;
        const int e_begin = min(T, tid * per_t), e_end = min(T, e_begin + per_t);
        int r = 0;
        while (r + 1 < nr && sh.pre[r + 1] <= e_begin)
            ++r;
        uint32_t cur_w = 0xffffffffu, cur_m = 0u;
        for (int e0 = e_begin; e0 < e_end; e0 += 8) {
            int id[8];
            int rr = r;
#pragma unroll
            for (int u = 0; u < 8; ++u) {      // 8 loads in flight
                const int e = e0 + u;
                id[u] = -1;
                if (e < e_end) {
                    while (rr + 1 < nr && sh.pre[rr + 1] <= e)
                        ++rr;
                    id[u] = w.fifo_sup[(size_t)sh.sup_off[rr] + (e - sh.pre[rr])];
                }
            }
            r = rr;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (e0 + u >= e_end)
                    break;
                const int i = id[u];
                if (i >= 0 && i < L) {
                    const uint32_t wd = (uint32_t)i >> 5, bit = 1u << (i & 31);
                    if (wd != cur_w) {
                        if (cur_m)
                            atomicOr(&region[cur_w], cur_m);
                        cur_w = wd;
                        cur_m = 0u;
                    }
                    cur_m |= bit;
                } else if (rank == 0) {
                    atomicOr(w.status, RETOPK_STATUS_BAD_INDEX);
                }
            }
        }
        if (cur_m)
            atomicOr(&region[cur_w], cur_m);
    }
    __syncthreads();
    // ascending emission.  Warp v owns a contiguous range of bitmap words and
    // walks it 32 words at a time, lane l taking word l of each chunk, so that
    // dense stretches (a retrieved topic run) are shared by all lanes.
    const int chunks = (nwords + kReuseWarps * 32 - 1) / (kReuseWarps * 32);   // per warp
    const int wbeg = warp * chunks * 32;
    int mine = 0;
    for (int k = 0; k < chunks; ++k) {
        const int i = wbeg + k * 32 + lane;
        mine += (i < nwords) ? __popc(region[i]) : 0;
    }
    mine = warp_isum(mine);
    if (lane == 0)
        sh.wcount[warp] = mine;
    __syncthreads();
    int pos = 0, M = 0;
    for (int v = 0; v < kReuseWarps; ++v) {
        pos += (v < warp) ? sh.wcount[v] : 0;
        M += sh.wcount[v];
    }
    for (int k = 0; k < chunks; ++k) {
        const int i = wbeg + k * 32 + lane;
        uint32_t bits = (i < nwords) ? region[i] : 0u;
        if (!__any_sync(0xffffffffu, bits != 0u))
            continue;                      // most chunks are empty
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        int p = pos + incl - c;
        while (bits) {
            const int bit = __ffs(bits) - 1;
            cand[p++] = (i << 5) + bit;
            bits &= bits - 1;
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncthreads();
    if (rank == 0) {
        int32_t *ci = w.cand_idx + (size_t)bh * w.cand_stride;
        for (int j = tid; j < M; j += kReuseThreads)
            ci[j] = cand[j];
        if (tid == 0)
            w.M[bh] = M;
    }

    // ---- Eq. (10): this rank's slice of the candidate scores -----------------
    const int per = (M + kReuseCluster - 1) / kReuseCluster;
    const int cs = min(M, rank * per), ce = min(M, cs + per);
    {
        // half-warp hw scores rows jb + hw + 16u; the loop bound is the same for
        // every thread so that the full-warp shuffles below always have all 32
        // lanes present
        constexpr int kHalfWarps = kReuseThreads / 16;
        const int hw = tid >> 4, hl = tid & 15;
        const float *qq = sh.qf + hl * 8;
        const uint16_t *kb = a.k + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
        for (int jb = cs; jb < ce; jb += kHalfWarps * kRerankRows) {
            uint4 kv[kRerankRows];
#pragma unroll
            for (int u = 0; u < kRerankRows; ++u) {
                const int j = jb + hw + u * kHalfWarps;
                kv[u] = (j < ce) ? reinterpret_cast<const uint4 *>(kb + (size_t)cand[j] * kD)[hl]
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
                const int j = jb + hw + u * kHalfWarps;
                if (hl == 0 && j < ce)
                    keys[j] = f2key(s * a.scale + 0.0f);
            }
        }
    }
    // every CTA of the cluster is past its bitmap before any score is pushed
    // into the (shared) region that held it
    cluster.sync();
    // push the slice into every peer
    for (int e = tid; e < (ce - cs) * (kReuseCluster - 1); e += kReuseThreads) {
        const int p = e / (ce - cs), j = cs + e % (ce - cs);
        const int peer = p < rank ? p : p + 1;
        cluster.map_shared_rank(keys, peer)[j] = keys[j];
    }
    cluster.sync();   // every CTA now holds all M scores

    // ---- Eq. (11): identical Top-K in every CTA ------------------------------
    const int need = min(w.K, M);
    auto get = [&](int j, int32_t &idx, uint32_t &key) {
        idx = cand[j];
        key = keys[j];
    };
    const unsigned long long thr = radix_select_threshold<kReuseThreads>(M, need, get, sh.sel);
    const int n = stable_compact<kReuseThreads>(M, thr, get, w.K, cand, keys, sh.sel.warp_tot);
    int32_t *sup_i = cand;
    uint32_t *sup_k = keys;
    if (tid == 0)
        sh.kmax = 0u;
    __syncthreads();
    {
        uint32_t km = 0u;
        for (int j = tid; j < n; j += kReuseThreads)
            km = max(km, sup_k[j]);
        km = __reduce_max_sync(0xffffffffu, km);
        if (lane == 0)
            atomicMax(&sh.kmax, km);
    }
    __syncthreads();
    const float m = key2f(sh.kmax);

    // ---- Eq. (12): this rank's share of the value rows -----------------------
    const int vper = (n + kReuseCluster - 1) / kReuseCluster;
    const int vs = min(n, rank * vper), ve = min(n, vs + vper);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float zsum = 0.f;
    const uint16_t *vb = a.v + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
    value_partial(vb, sup_i, sup_k, vs + warp, ve, kReuseWarps, m, acc, zsum);
    *reinterpret_cast<float4 *>(&sh.red[warp][lane * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0)
        sh.zw[warp] = zsum;
    __syncthreads();
    if (tid < kD) {
        float o = 0.f;
#pragma unroll
        for (int ww = 0; ww < kReuseWarps; ++ww)
            o += sh.red[ww][tid];
        cluster.map_shared_rank(&sh.part_o[0][0], 0)[rank * kD + tid] = o;
    }
    if (tid == kD) {
        float z = 0.f;
#pragma unroll
        for (int ww = 0; ww < kReuseWarps; ++ww)
            z += sh.zw[ww];
        cluster.map_shared_rank(&sh.part_z[0], 0)[rank] = z;
    }
    cluster.sync();
    if (rank != 0)
        return;

    // ---- rank 0: output, cache insertion, bookkeeping -------------------------
    if (tid < kD) {
        float o = 0.f, Z = 0.f;
#pragma unroll
        for (int r = 0; r < kReuseCluster; ++r) {
            o += sh.part_o[r][tid];
            Z += sh.part_z[r];
        }
        o = (n > 0) ? o / Z : 0.f;
        a.out[(size_t)bh * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        w.out_f32[(size_t)bh * kD + tid] = o;
    }
    const int slot = head;
    const size_t e = (size_t)bh * w.C + slot;
    if (tid < kD / 8)
        reinterpret_cast<uint4 *>(w.fifo_q + e * kD)[tid] = reinterpret_cast<const uint4 *>(a.q + (size_t)bh * kD)[tid];
    for (int jj = tid; jj < w.K; jj += kReuseThreads) {
        const int32_t v = jj < n ? sup_i[jj] : -1;
        w.fifo_sup[e * w.K + jj] = v;
        w.support[(size_t)bh * w.K + jj] = v;
    }
    if (tid == 0) {
        w.fifo_len[e] = n;
        w.sup_len[bh] = n;
        finish_head(w, b, RETOPK_PATH_REUSE, M);
    }
}

static size_t reuse_smem_bytes(int max_len, int RKW)
{
    const size_t region = (size_t)std::max((max_len + 31) >> 5, RKW);
    return (region + (size_t)RKW) * 4;
}

cudaError_t launch_reuse(const Work &w, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *seqlens, uint16_t *out, cudaStream_t st)
{
    ReuseArgs a{w, q, k_cache, v_cache, seqlens, out, 1.0f / sqrtf((float)kD)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kReuseCluster, w.B * w.Hq, 1);
    cfg.blockDim = dim3(kReuseThreads, 1, 1);
    cfg.dynamicSmemBytes = reuse_smem_bytes(w.max_len, w.R * w.K + w.W);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kReuseCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reuse_kernel, a);
}

cudaError_t configure_reuse()
{
    return cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)reuse_smem_bytes(kMaxLen, kMaxCand));
}

}  // namespace retopk
