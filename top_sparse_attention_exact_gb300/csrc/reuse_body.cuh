// reuse_body.cuh -- the reuse path of one decode step for one (sequence,
// query head) per cluster of CL CTAs (CL = 1, 2, 4 or 8, at most
// kReuseCluster; chosen per configuration) (ReTopK paper,
// §Recall-Before-Rerank Selection, §Reliable Reuse and §Complexity and GPU
// Implementation: candidate union and dedup, indexed rerank, Top-K, indexed
// softmax-value aggregation and cache update), after the path decision.
//
// The candidate set A_t (Eqs. (8)-(9): window U the retrieved supports) is
// built through a bitmap over the key positions split across the cluster:
// rank r owns the positions [r*S, (r+1)*S) (S = L/CL rounded up to
// 32), sets the bits of the window and support entries in that range in its
// own shared memory, and lists its candidates in ascending order.  After one
// cluster barrier every rank concatenates the eight lists in rank order
// (distributed shared memory reads), so the cluster agrees on A_t, ascending.
// The work that touches HBM is split across the cluster:
//   Eq. (10) each CTA scores 1/CL of the candidate keys (K rows
//            gathered straight from the cache) and pushes the scores into
//            every peer's shared memory (distributed shared memory);
//   Eq. (11) after a cluster barrier each CTA holds all M_t scores and runs
//            the same radix select -> identical support S_t;
//   Eq. (12) each CTA aggregates 1/CL of the support's V rows with
//            the common max, pushes (sum of weights, weighted sum) to rank 0;
// after a second barrier rank 0 normalises, writes the output and inserts
// (q_t, S_t) into the query-support cache (Eq. (5)).
#pragma once

#include <cooperative_groups.h>

#include <algorithm>
#include <cstddef>

#include "topk.cuh"

namespace retopk {

namespace cg = cooperative_groups;

constexpr int kReuseThreads = 512;
constexpr int kReuseWarps = kReuseThreads / 32;
constexpr int kReuseCluster = 8;
static_assert(kMaxC <= kReuseThreads, "one cache entry per thread");

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
    int pre[kMaxC + 1];    // prefix of the retrieved supports' lengths
    int sup_off[kMaxC];    // cache offset of each retrieved support
    int wcount[kReuseWarps];
    int ncand;             // this rank's candidates (read by the peers)
    int cpre[kReuseCluster + 1];   // prefix of the ranks' candidate counts
    uint32_t kmax;
    SelectShared sel;
};
// value-phase scratch (after the scores are exchanged)
struct ReuseTail {
    float red[kReuseWarps][kD];          // written with 16-byte stores
    float zw[kReuseWarps];
    alignas(16) float part_o[kReuseCluster][kD];   // rank 0 receives every rank's partial
    float part_z[kReuseCluster];
};
static_assert(offsetof(ReuseTail, part_o) % 16 == 0, "partials aligned");
constexpr int kReuseTailWords = (int)((sizeof(ReuseTail) + 15) / 16 * 4);

// Dynamic shared memory of the reuse path, in 4-byte words after ReuseShared:
//   [0, A)        the rank's bitmap slice; then the M_t scores (keys)
//   [A, A + Bw)   the rank's list of candidates; then the ReuseTail
//   [A + Bw, +RKW) A_t, then S_t (cand)
// with A = max(S/32, RKW) rounded up to 4 and Bw = max(RKW, kReuseTailWords).
constexpr size_t kReuseSharedBytes = (sizeof(ReuseShared) + 127) & ~size_t(127);

// positions per rank of the split bitmap: L / CL rounded up to 32
__host__ __device__ __forceinline__ int reuse_span(int L, int CL)
{
    return (((L + CL - 1) / CL) + 31) & ~31;
}
__host__ __device__ __forceinline__ int reuse_words_a(int max_len, int RKW, int CL)
{
    const int s = reuse_span(max_len, CL) >> 5;
    return ((s > RKW ? s : RKW) + 3) & ~3;
}
__host__ __device__ __forceinline__ int reuse_words_b(int RKW)
{
    return RKW > kReuseTailWords ? RKW : kReuseTailWords;
}

inline size_t reuse_smem_bytes(int max_len, int RKW, int CL)
{
    return kReuseSharedBytes + ((size_t)reuse_words_a(max_len, RKW, CL) + reuse_words_b(RKW) + (size_t)RKW) * 4;
}

// Eqs. (8)-(12) and the cache insertion for one reuse head per cluster of
// CL CTAs of kReuseThreads threads; `smem` is the CTA's dynamic shared memory
// (reuse_smem_bytes).
template <int CL>
__device__ __forceinline__ void reuse_body(const ReuseArgs &a, unsigned char *smem)
{
    static_assert(CL == 1 || CL == 2 || CL == 4 || CL == 8, "cluster of 1, 2, 4 or 8 CTAs");
    // key rows in flight per half-warp: twice as many when one or two CTAs
    // carry the head (large batches, where the candidates per CTA are many)
    constexpr int kRerankRows = CL <= 2 ? 8 : 4;
    ReuseShared &sh = *reinterpret_cast<ReuseShared *>(smem);
    uint32_t *rsm = reinterpret_cast<uint32_t *>(smem + kReuseSharedBytes);
    cg::cluster_group cluster = cg::this_cluster();
    const Work &w = a.w;
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / w.Hq, h = bh % w.Hq, hk = h / w.G;
    if (w.path[bh] != RETOPK_PATH_REUSE)
        return;                                   // uniform over the cluster
    const int RKW = w.R * w.K + w.W;
    const int wa = reuse_words_a(w.max_len, RKW, CL), wb = reuse_words_b(RKW);
    uint32_t *region = rsm;                                           // bitmap slice, then the scores
    uint32_t *keys = region;
    int32_t *loc = reinterpret_cast<int32_t *>(rsm + wa);             // this rank's candidates
    ReuseTail &tl = *reinterpret_cast<ReuseTail *>(rsm + wa);         // (after the score exchange)
    int32_t *cand = reinterpret_cast<int32_t *>(rsm + wa + wb);       // A_t, then S_t

    // ---- the decision's outputs: retrieved entries and their supports --------
    const int L = seq_len(a.seqlens, b, 0, w.max_len);
    const int *sq = w.snap + b * SEQ_WORDS;   // the ring as the decision saw it
    const int head = sq[SEQ_HEAD], count = sq[SEQ_COUNT];
    const int nr = min(w.R, count);
    const size_t e_slot = (size_t)bh * w.C + head;   // this step's cache entry (Eq. (5))
    if (tid < kD)
        sh.qf[tid] = __uint_as_float(((uint32_t)a.q[(size_t)bh * kD + tid]) << 16);
    if (rank == 0 && tid < kD / 8)   // q_t into its slot, off the critical path (only the decision reads fifo_q)
        reinterpret_cast<uint4 *>(w.fifo_q + e_slot * kD)[tid] = reinterpret_cast<const uint4 *>(a.q + (size_t)bh * kD)[tid];
    {   // slots, lengths and prefix of the nr (<= C <= kReuseThreads) retrieved supports
        int len = 0, off = 0;
        if (tid < nr) {
            const int pos = w.topR[(size_t)bh * w.R + tid];
            const int slot = ((head - count + pos) % w.C + w.C) % w.C;
            len = w.fifo_len[(size_t)bh * w.C + slot];
            off = (int)(((size_t)bh * w.C + slot) * w.K);
        }
        int tot;
        const int ex = block_excl_scan<kReuseThreads>(len, sh.sel.warp_tot, tot);
        if (tid < nr) {
            sh.pre[tid] = ex;
            sh.sup_off[tid] = off;
        }
        if (tid == 0)
            sh.pre[nr] = tot;
    }
    // this rank's positions [r_lo, r_hi) (r_lo a multiple of 32)
    const int r_lo = min(L, rank * reuse_span(L, CL)), r_hi = min(L, r_lo + reuse_span(L, CL));
    const int nwords = (r_hi - r_lo + 31) >> 5;
    for (int i = tid; i < nwords; i += kReuseThreads)
        region[i] = 0u;
    __syncthreads();

    // ---- Eqs. (8)-(9): candidate bitmap (this rank's slice) -----------------
    // recent window [lo, L): one thread per bitmap word
    const int lo = max(r_lo, L - w.W);
    if (lo < r_hi) {
        for (int wd = ((lo - r_lo) >> 5) + tid; wd <= ((r_hi - 1 - r_lo) >> 5); wd += kReuseThreads) {
            const int p0 = r_lo + (wd << 5);
            const int a0 = max(lo, p0) - p0, a1 = min(r_hi, p0 + 32) - p0;
            const uint32_t msk = (a1 - a0 == 32) ? 0xffffffffu : (((1u << (a1 - a0)) - 1u) << a0);
            atomicOr(&region[wd], msk);
        }
    }
    // thread t walks a contiguous run of the concatenated (ascending) support
    // lists, so neighbouring indices share a bitmap word: OR them in a register
    // and issue one shared atomic per word change (entries of this rank only)
    const int T = sh.pre[nr];
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
                if (i >= r_lo && i < r_hi) {
                    const uint32_t wd = (uint32_t)(i - r_lo) >> 5, bit = 1u << (i & 31);
                    if (wd != cur_w) {
                        if (cur_m)
                            atomicOr(&region[cur_w], cur_m);
                        cur_w = wd;
                        cur_m = 0u;
                    }
                    cur_m |= bit;
                } else if ((i < 0 || i >= L) && rank == 0) {
                    atomicOr(w.status, RETOPK_STATUS_BAD_INDEX);
                }
            }
        }
        if (cur_m)
            atomicOr(&region[cur_w], cur_m);
    }
    __syncthreads();
    // ascending emission of this rank's list.  Warp v owns a contiguous range
    // of bitmap words and walks it 32 words at a time, lane l taking word l of
    // each chunk, so that dense stretches (a retrieved topic run) are shared
    // by all lanes.
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
    int pos = 0, Mr = 0;
    for (int v = 0; v < kReuseWarps; ++v) {
        pos += (v < warp) ? sh.wcount[v] : 0;
        Mr += sh.wcount[v];
    }
    if (tid == 0)
        sh.ncand = Mr;
    const unsigned lt = (1u << lane) - 1u;
    for (int k = 0; k < chunks; ++k) {
        const int i = wbeg + k * 32 + lane;
        const uint32_t bits = (i < nwords) ? region[i] : 0u;
        unsigned nz = __ballot_sync(0xffffffffu, bits != 0u);
        if (!nz)
            continue;                      // most chunks are empty
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const int excl = pos + incl - c;
        // the whole warp expands one non-empty word at a time, lane l its bit l
        // (dense runs of retrieved supports fill whole words)
        while (nz) {                       // warp-uniform
            const int src = __ffs(nz) - 1;
            nz &= nz - 1u;
            const uint32_t wb = __shfl_sync(0xffffffffu, bits, src);
            const int base = __shfl_sync(0xffffffffu, excl, src);
            if ((wb >> lane) & 1u)
                loc[base + __popc(wb & lt)] = r_lo + ((wbeg + k * 32 + src) << 5) + lane;
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    // every rank's list and count are complete, and every bitmap is dead (the
    // peers' scores may now land in the region that held it)
    cluster.sync();
    if (tid < CL)
        sh.cpre[tid + 1] = *cluster.map_shared_rank(&sh.ncand, tid);
    __syncthreads();
    if (tid == 0) {
        sh.cpre[0] = 0;
        for (int r = 0; r < CL; ++r)
            sh.cpre[r + 1] += sh.cpre[r];
    }
    __syncthreads();
    const int M = sh.cpre[CL];
    {   // A_t = the ranks' lists in rank order; four peer loads in flight
        for (int j0 = tid; j0 < M; j0 += 4 * kReuseThreads) {
            int32_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kReuseThreads;
                v[u] = 0;
                if (j < M) {
                    int r = 0;
#pragma unroll
                    for (int q = 1; q < CL; ++q)
                        r += j >= sh.cpre[q];
                    v[u] = cluster.map_shared_rank(loc, r)[j - sh.cpre[r]];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kReuseThreads;
                if (j < M)
                    cand[j] = v[u];
            }
        }
        int32_t *ci = w.cand_idx + (size_t)bh * w.cand_stride + sh.cpre[rank];
        for (int j = tid; j < Mr; j += kReuseThreads)
            ci[j] = loc[j];
        if (rank == 0 && tid == 0)
            w.M[bh] = M;
    }
    __syncthreads();

    // ---- Eq. (10): this rank's slice of the candidate scores -----------------
    const int per = (M + CL - 1) / CL;
    const int cs = min(M, rank * per), ce = min(M, cs + per);
    {
        // half-warp hw scores rows jb + hw + 16u; the loop bound is the same for
        // every thread so that the full-warp shuffles below always have all 32
        // lanes present
        constexpr int kHalfWarps = kReuseThreads / 16;
        const int hw = tid >> 4, hl = tid & 15;
        const float *qq = sh.qf + hl * 8;
        const uint16_t *kb = a.k + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
        bool nonfinite = false;
        for (int jb = cs; jb < ce; jb += kHalfWarps * kRerankRows) {
            uint4 kv[kRerankRows];
#pragma unroll
            for (int u = 0; u < kRerankRows; ++u) {
                const int j = jb + hw + u * kHalfWarps;
                kv[u] = (j < ce && row_ok(cand[j], L, w.status))
                            ? reinterpret_cast<const uint4 *>(kb + (size_t)cand[j] * kD)[hl]
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
                if (hl == 0 && j < ce) {
                    const float sc = s * a.scale + 0.0f;
                    nonfinite |= !(fabsf(sc) <= 3.402823466e38f);
                    keys[j] = f2key(sc);
                }
            }
        }
        if (nonfinite)
            atomicOr(w.status, RETOPK_STATUS_NONFINITE);
    }
    __syncthreads();   // the slice's scores are written
    // push the slice into every peer (each is past its bitmap: cluster barrier above)
    for (int e = tid; e < (ce - cs) * (CL - 1); e += kReuseThreads) {
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
    const int n = stable_compact<kReuseThreads, 4>(M, thr, get, w.K, cand, keys, sh.sel.warp_tot);
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
    {   // S_t (identical in every rank), written 1/CL per rank; every
        // rank of the cluster is past its reads of the retrieved supports
        const int kper = (w.K + CL - 1) / CL;
        const int j0 = rank * kper, j1 = min(w.K, j0 + kper);
        for (int jj = j0 + tid; jj < j1; jj += kReuseThreads) {
            const int32_t v = jj < n ? sup_i[jj] : -1;
            w.fifo_sup[e_slot * w.K + jj] = v;
            w.support[(size_t)bh * w.K + jj] = v;
        }
        if (rank == 0 && tid == 0) {
            w.fifo_len[e_slot] = n;
            w.sup_len[bh] = n;
            count_head(w, b, RETOPK_PATH_REUSE, M);
        }
    }

    // ---- Eq. (12): this rank's share of the value rows -----------------------
    const int vper = (n + CL - 1) / CL;
    const int vs = min(n, rank * vper), ve = min(n, vs + vper);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float zsum = 0.f;
    const uint16_t *vb = a.v + ((size_t)(b * w.Hkv + hk) * w.max_len) * kD;
    value_partial<8>(vb, sup_i, sup_k, vs + warp, ve, kReuseWarps, m, acc, zsum, L, w.status);
    *reinterpret_cast<float4 *>(&tl.red[warp][lane * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0)
        tl.zw[warp] = zsum;
    __syncthreads();
    if (tid < kD) {
        float o = 0.f;
#pragma unroll
        for (int ww = 0; ww < kReuseWarps; ++ww)
            o += tl.red[ww][tid];
        cluster.map_shared_rank(&tl.part_o[0][0], 0)[rank * kD + tid] = o;
    }
    if (tid == kD) {
        float z = 0.f;
#pragma unroll
        for (int ww = 0; ww < kReuseWarps; ++ww)
            z += tl.zw[ww];
        cluster.map_shared_rank(&tl.part_z[0], 0)[rank] = z;
    }
    cluster.sync();
    if (rank != 0)
        return;

    // ---- rank 0: the output ----------------------------------------------------
    if (tid < kD) {
        float o = 0.f, Z = 0.f;
#pragma unroll
        for (int r = 0; r < CL; ++r) {
            o += tl.part_o[r][tid];
            Z += tl.part_z[r];
        }
        o = (n > 0) ? o / Z : 0.f;
        a.out[(size_t)bh * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        w.out_f32[(size_t)bh * kD + tid] = o;
    }

}

}  // namespace retopk
