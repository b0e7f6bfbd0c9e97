// fidelity.cu -- attention-support fidelity of a decode step (ReTopK paper,
// §Experiments "Attention-support fidelity" with Figs. 5-6, and §Motivation
// Eq. (2)): how well the support a decode step used (the reranked support on
// the reuse path) matches the Exact Top-K support of the same query.  A
// diagnostic run beside the decode loop ("exact shadow"), not part of it.
//
// One CTA per (sequence, query head): both supports (ascending, -1 padded)
// are loaded, their scores recomputed from q and the K rows, and
//   m[0] support recall      |Sh n S| / |S|
//   m[1] retained mass       sum over Sh n S of p, p = softmax over S
//   m[2] output cosine       cos(oh, o) of the two bf16 head outputs
//   m[3] distribution cosine sum over Sh n S of p ph / (|p| |ph|)
// are written in fp32.  The supports come from the caller: an entry outside
// [0, max_len) (other than the -1 padding after the valid ones) would address
// past the cache, so its row is not read; it scores 0 and sets
// RETOPK_STATUS_GATHER.
#include "common.cuh"

namespace retopk {

constexpr int kFidThreads = 256;
constexpr int kFidWarps = kFidThreads / 32;

struct FidArgs {
    const uint16_t *q;       // [B, Hq, d]
    const uint16_t *k;       // [B, Hkv, max_len, d]
    const int32_t *S;        // [B, Hq, K] exact support
    const int32_t *Sh;       // [B, Hq, K] judged support
    const uint16_t *o;       // [B, Hq, d] exact output
    const uint16_t *oh;      // [B, Hq, d] judged output
    float *out;              // [B, Hq, 4]
    uint32_t *status;
    int Hq, Hkv, max_len, K;
    float scale;
};

struct FidShared {
    float acc[8];            // mS, mh, ZS, Zh, p2, ph2, mass, cross (reduced in place)
    int nS, nh, common;
};

__device__ __forceinline__ void atomic_max_f(float *a, float v)
{
    // order-preserving integer max on the float's key
    atomicMax(reinterpret_cast<unsigned *>(a), f2key(v));
}

__global__ void __launch_bounds__(kFidThreads) fidelity_kernel(FidArgs a)
{
    extern __shared__ __align__(16) unsigned char fsm[];
    __shared__ FidShared sh;
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = bh / a.Hq, h = bh % a.Hq, hk = h / (a.Hq / a.Hkv);
    int32_t *S = reinterpret_cast<int32_t *>(fsm);      // [K]
    int32_t *Sh = S + a.K;                              // [K]
    float *eS = reinterpret_cast<float *>(Sh + a.K);    // [K]
    float *eh = eS + a.K;                               // [K]
    if (tid < 8)
        sh.acc[tid] = 0.f;
    if (tid == 0) {
        sh.nS = 0;
        sh.nh = 0;
        sh.common = 0;
        // maxima are kept as order-preserving keys
        reinterpret_cast<unsigned *>(sh.acc)[0] = 0u;
        reinterpret_cast<unsigned *>(sh.acc)[1] = 0u;
    }
    __syncthreads();
    int cS = 0, ch = 0;
    for (int j = tid; j < a.K; j += kFidThreads) {
        const int32_t s = a.S[(size_t)bh * a.K + j], t = a.Sh[(size_t)bh * a.K + j];
        S[j] = s;
        Sh[j] = t;
        cS += s >= 0;
        ch += t >= 0;
    }
    cS = warp_isum(cS);
    ch = warp_isum(ch);
    if (lane == 0) {
        atomicAdd(&sh.nS, cS);
        atomicAdd(&sh.nh, ch);
    }
    __syncthreads();
    const int nS = sh.nS, nh = sh.nh;   // the valid entries lead each list
    // scores of both supports: one K row per warp step, 8 bytes per lane
    const uint16_t *kb = a.k + ((size_t)(b * a.Hkv + hk) * a.max_len) * kD;
    const uint2 qr = *reinterpret_cast<const uint2 *>(a.q + (size_t)bh * kD + lane * 4);
    for (int j = warp; j < nS + nh; j += kFidWarps) {
        const int row = j < nS ? S[j] : Sh[j - nS];
        const bool in = (uint32_t)row < (uint32_t)a.max_len;
        if (!in && lane == 0)
            atomicOr(a.status, RETOPK_STATUS_GATHER);
        const uint2 kr = in ? *reinterpret_cast<const uint2 *>(kb + (size_t)row * kD + lane * 4) : make_uint2(0u, 0u);
        float e = bf16lo(qr.x) * bf16lo(kr.x) + bf16hi(qr.x) * bf16hi(kr.x) + bf16lo(qr.y) * bf16lo(kr.y) +
                  bf16hi(qr.y) * bf16hi(kr.y);
        e = warp_sum(e) * a.scale;
        if (lane == 0) {
            if (j < nS) {
                eS[j] = e;
                atomic_max_f(&sh.acc[0], e);
            } else {
                eh[j - nS] = e;
                atomic_max_f(&sh.acc[1], e);
            }
        }
    }
    __syncthreads();
    const float mS = key2f(reinterpret_cast<unsigned *>(sh.acc)[0]);
    const float mh = key2f(reinterpret_cast<unsigned *>(sh.acc)[1]);
    float zS = 0.f, zh = 0.f;
    for (int j = tid; j < nS; j += kFidThreads)
        zS += expf(eS[j] - mS);
    for (int j = tid; j < nh; j += kFidThreads)
        zh += expf(eh[j] - mh);
    zS = warp_sum(zS);
    zh = warp_sum(zh);
    if (lane == 0) {
        atomicAdd(&sh.acc[2], zS);
        atomicAdd(&sh.acc[3], zh);
    }
    __syncthreads();
    const float ZS = sh.acc[2], Zh = sh.acc[3];
    float p2 = 0.f, ph2 = 0.f, mass = 0.f, cross = 0.f;
    int common = 0;
    for (int j = tid; j < nS; j += kFidThreads) {
        const float p = expf(eS[j] - mS) / ZS;
        p2 += p * p;
    }
    for (int j = tid; j < nh; j += kFidThreads) {
        const float ph = expf(eh[j] - mh) / Zh;
        ph2 += ph * ph;
        int lo = 0, hi = nS;   // Sh[j] in the ascending S?
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (S[mid] < Sh[j])
                lo = mid + 1;
            else
                hi = mid;
        }
        if (lo < nS && S[lo] == Sh[j]) {
            const float p = expf(eS[lo] - mS) / ZS;
            ++common;
            mass += p;
            cross += p * ph;
        }
    }
    p2 = warp_sum(p2);
    ph2 = warp_sum(ph2);
    mass = warp_sum(mass);
    cross = warp_sum(cross);
    common = warp_isum(common);
    if (lane == 0) {
        atomicAdd(&sh.acc[4], p2);
        atomicAdd(&sh.acc[5], ph2);
        atomicAdd(&sh.acc[6], mass);
        atomicAdd(&sh.acc[7], cross);
        atomicAdd(&sh.common, common);
    }
    __syncthreads();
    if (warp == 0) {   // output cosine over the d = 128 values
        float oo = 0.f, hh = 0.f, oh = 0.f;
        for (int c = lane; c < kD; c += 32) {
            const float x = __uint_as_float((uint32_t)a.o[(size_t)bh * kD + c] << 16);
            const float y = __uint_as_float((uint32_t)a.oh[(size_t)bh * kD + c] << 16);
            oo += x * x;
            hh += y * y;
            oh += x * y;
        }
        oo = warp_sum(oo);
        hh = warp_sum(hh);
        oh = warp_sum(oh);
        if (lane == 0) {
            float *m = a.out + (size_t)bh * 4;
            m[0] = nS > 0 ? (float)sh.common / (float)nS : 1.f;
            m[1] = sh.acc[6];
            m[2] = (oo > 0.f && hh > 0.f) ? oh / (sqrtf(oo) * sqrtf(hh)) : 0.f;
            m[3] = (sh.acc[4] > 0.f && sh.acc[5] > 0.f) ? sh.acc[7] / (sqrtf(sh.acc[4]) * sqrtf(sh.acc[5])) : 0.f;
        }
    }
}

cudaError_t launch_fidelity(const uint16_t *q, const uint16_t *k, const int32_t *S, const int32_t *Sh,
                            const uint16_t *o, const uint16_t *oh, float *out, uint32_t *status, int B, int Hq,
                            int Hkv, int max_len, int K, cudaStream_t st)
{
    FidArgs a{q, k, S, Sh, o, oh, out, status, Hq, Hkv, max_len, K, 1.0f / sqrtf((float)kD)};
    fidelity_kernel<<<B * Hq, kFidThreads, (size_t)K * 16, st>>>(a);
    return cudaGetLastError();
}

// ---- support overlap and coverage (§Motivation Eqs. (2)-(3)) ----------------
// One CTA per row: S [rows, K] and the R supports others [rows, R, K], each
// ascending and -1 padded.  out[row] = (Overlap(S, others[0]),
// Coverage(S, union of others)), both over K.  Membership is a binary search
// over the valid prefix of each list; the union is never materialised.
constexpr int kOvThreads = 256;

__device__ __forceinline__ int valid_len(const int32_t *s, int K)
{
    int lo = 0, hi = K;   // entries >= 0 come first, then the -1 padding
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s[mid] >= 0)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ bool contains(const int32_t *s, int n, int32_t x)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s[mid] < x)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo < n && s[lo] == x;
}

__global__ void __launch_bounds__(kOvThreads) overlap_kernel(const int32_t *S, const int32_t *others, int R, int K,
                                                             float *out)
{
    __shared__ int lens[kMaxC + 1];
    __shared__ int cnt[2][kOvThreads / 32];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *s = S + (size_t)row * K;
    const int32_t *o = others + (size_t)row * R * K;
    for (int r = tid; r <= R; r += kOvThreads)
        lens[r] = valid_len(r < R ? o + (size_t)r * K : s, K);
    __syncthreads();
    const int ns = lens[R];
    int first = 0, any = 0;
    for (int j = tid; j < ns; j += kOvThreads) {
        const int32_t x = s[j];
        bool in_first = false, in_any = false;
        for (int r = 0; r < R && !in_any; ++r) {
            const bool c = contains(o + (size_t)r * K, lens[r], x);
            in_first |= (r == 0) && c;
            in_any |= c;
        }
        first += in_first;
        any += in_any;
    }
    first = warp_isum(first);
    any = warp_isum(any);
    if (lane == 0) {
        cnt[0][warp] = first;
        cnt[1][warp] = any;
    }
    __syncthreads();
    if (tid < 2) {
        int c = 0;
        for (int i = 0; i < kOvThreads / 32; ++i)
            c += cnt[tid][i];
        out[(size_t)row * 2 + tid] = (float)c / (float)K;
    }
}

cudaError_t launch_overlap(const int32_t *S, const int32_t *others, int rows, int R, int K, float *out,
                           cudaStream_t st)
{
    overlap_kernel<<<rows, kOvThreads, 0, st>>>(S, others, R, K, out);
    return cudaGetLastError();
}

cudaError_t configure_fidelity()
{
    return cudaFuncSetAttribute(fidelity_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxK * 16);
}

}  // namespace retopk
