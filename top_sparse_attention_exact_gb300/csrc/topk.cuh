// topk.cuh -- block-wide building blocks of the Top-K selection shared by the
// reuse-path kernel and the exact-path select kernel (ReTopK paper, Eq. (1)
// and Eq. (11): the K best keys by score, ties to the lower index).
//
// Candidates are visited through a callable get(j, idx, key) returning the
// key index and the order-preserving score key of candidate j.
#pragma once

#include "common.cuh"

namespace retopk {

// Exclusive scan of one int per thread over an NT-thread block.  warp_tot
// needs 33 ints of shared memory.  Three barriers; every thread must call it.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int &total)
{
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
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

struct SelectShared {
    uint32_t hist[2][256];
    int digit, above, cnt_d;
    int warp_tot[33];
    unsigned long long kand[32], kor[32];
};

// Radix refinement of a select threshold: the keys whose bits [top, 64) equal
// those of `prefix` compete for `rem` (>= 1) slots (keys above the prefix are
// already selected); 8-bit digits, most significant first, stopping as soon
// as every key sharing the current prefix is selected.  On entry sh.hist[0]
// is zero and a barrier has passed since.  Returns the threshold (identical
// in every thread).
template <int NT, class Get>
__device__ unsigned long long radix_refine(int N, int rem, unsigned long long prefix, int top, Get get,
                                          SelectShared &sh)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int buf = 0;
    for (int hi = top; hi > 0; hi -= 8, buf ^= 1) {
        const int lo = hi > 8 ? hi - 8 : 0;          // digit = bits [lo, hi)
        const unsigned long long hmask = (hi >= 64) ? 0ull : (~0ull << hi);
        const unsigned dmask = (1u << (hi - lo)) - 1u;
        uint32_t *hist = sh.hist[buf];
        for (int j = tid; j < N; j += NT) {
            int32_t idx;
            uint32_t key;
            get(j, idx, key);
            const unsigned long long k64 = key64(key, idx);
            if (((k64 ^ prefix) & hmask) == 0ull)
                atomicAdd(&hist[(unsigned)(k64 >> lo) & dmask], 1u);
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
#pragma unroll
            for (int i = 0; i < 8; ++i)   // the other buffer, for the next pass
                sh.hist[buf ^ 1][lane * 8 + i] = 0u;
        }
        __syncthreads();
        rem -= sh.above;
        prefix |= (unsigned long long)sh.digit << lo;
        if (sh.cnt_d == rem)
            break;
    }
    return prefix;
}

// Threshold of the `need` largest composite keys key64(key, idx) among N
// candidates: a radix select that starts at the highest bit where the
// candidates differ (the bits above are common to all of them).  Returns thr
// with |{j : key64_j >= thr}| == need; 0 when N <= need.  Identical in every
// thread.
template <int NT, class Get>
__device__ unsigned long long radix_select_threshold(int N, int need, Get get, SelectShared &sh)
{
    if (N <= need)
        return 0ull;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // common prefix: AND and OR of all keys
    unsigned long long kand = ~0ull, kor = 0ull;
    for (int j = tid; j < N; j += NT) {
        int32_t idx;
        uint32_t key;
        get(j, idx, key);
        const unsigned long long k64 = key64(key, idx);
        kand &= k64;
        kor |= k64;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kand &= __shfl_xor_sync(0xffffffffu, kand, o);
        kor |= __shfl_xor_sync(0xffffffffu, kor, o);
    }
    if (lane == 0) {
        sh.kand[warp] = kand;
        sh.kor[warp] = kor;
    }
    for (int i = tid; i < 512; i += NT)
        (&sh.hist[0][0])[i] = 0u;
    __syncthreads();
    kand = ~0ull;
    kor = 0ull;
    for (int v = 0; v < NT / 32; ++v) {
        kand &= sh.kand[v];
        kor |= sh.kor[v];
    }
    const unsigned long long diff = kand ^ kor;      // nonzero: the indices differ
    const int top = 64 - __clzll(diff);              // bits [top, 64) are common
    const unsigned long long prefix = (top >= 64) ? 0ull : (kand & (~0ull << top));
    return radix_refine<NT>(N, need, prefix, top, get, sh);
}

// Stable compaction of the candidates with key64 >= thr, in candidate order,
// into out_i / out_k (at most cap entries).  Thread t handles E consecutive
// candidates of each NT*E chunk, so one block scan covers the chunk.  The
// outputs may alias the candidate arrays read by `get` (positions written never
// exceed the position read, and every read of a chunk precedes its writes).
// Returns the count.  The last chunk's writes are not followed by a barrier:
// synchronise the block before other threads read the outputs.
template <int NT, int E = 8, class Get>
__device__ int stable_compact(int N, unsigned long long thr, Get get, int cap, int32_t *out_i,
                              uint32_t *out_k, int *warp_tot)
{
    int got = 0;
    for (int base = 0; base < N; base += NT * E) {
        const int j0 = base + threadIdx.x * E;
        int32_t idx[E];
        uint32_t key[E];
        int c = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            idx[e] = 0;
            key[e] = 0u;
            if (j0 + e < N) {
                get(j0 + e, idx[e], key[e]);
                c += key64(key[e], idx[e]) >= thr;
            }
        }
        int total;
        int pos = got + block_excl_scan<NT>(c, warp_tot, total);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (j0 + e < N && key64(key[e], idx[e]) >= thr) {
                if (pos < cap) {
                    out_i[pos] = idx[e];
                    out_k[pos] = key[e];
                }
                ++pos;
            }
        }
        got += total;
    }
    return got < cap ? got : cap;
}

// Softmax-weighted partial sum over support rows [j0, j1) (stride `step` per
// warp): lane l accumulates dims 4l..4l+3 with weights exp(score - m).
// U rows in flight per lane.  L and status serve the checked build's range
// check of the row indices (row_ok).
template <int U = 16>
__device__ __forceinline__ void value_partial(const uint16_t *vb, const int32_t *sup_i, const uint32_t *sup_k,
                                              int j0, int j1, int step, float m, float (&acc)[4], float &zsum,
                                              int L, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    for (int jb = j0; jb < j1; jb += step * U) {
        uint2 vv[U];
        float p[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = jb + u * step;
            if (j < j1 && row_ok(sup_i[j], L, status)) {
                vv[u] = *reinterpret_cast<const uint2 *>(vb + (size_t)sup_i[j] * kD + lane * 4);
                p[u] = expf(key2f(sup_k[j]) - m);
            } else {
                vv[u] = make_uint2(0u, 0u);
                p[u] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            zsum += p[u];
            acc[0] += p[u] * bf16lo(vv[u].x);
            acc[1] += p[u] * bf16hi(vv[u].x);
            acc[2] += p[u] * bf16lo(vv[u].y);
            acc[3] += p[u] * bf16hi(vv[u].y);
        }
    }
}

// Per-sequence counters after a decode step of one head (one thread; no
// result is waited for): the head's path, and on the reuse path |A_t|.
__device__ __forceinline__ void count_head(const Work &w, int b, int path, int M)
{
    unsigned long long *cnt = w.counters + (size_t)b * CNT_WORDS;
    atomicAdd(&cnt[path == RETOPK_PATH_REUSE ? CNT_REUSE : path == RETOPK_PATH_FALLBACK ? CNT_FALLBACK : CNT_REFRESH],
              1ull);
    if (path == RETOPK_PATH_REUSE) {
        atomicAdd(&cnt[CNT_SUM_M], (unsigned long long)M);
        atomicMax(&cnt[CNT_MAX_M], (unsigned long long)M);
    }
}

}  // namespace retopk
