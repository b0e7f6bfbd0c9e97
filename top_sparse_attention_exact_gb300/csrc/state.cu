// state.cu -- small per-step state kernels: appending the new token's key and
// value rows (and advancing L on the device), and finishing the cache
// initialisation (ReTopK paper, §Recall-Before-Rerank: the cache is
// initialised from the final C prompt tokens).
#include <algorithm>

#include "common.cuh"

namespace retopk {

__global__ void append_kernel(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                              uint16_t *v_cache, int32_t *seqlens, uint32_t *status, int Hkv,
                              int max_len)
{
    pdl_wait();      // the previous step is done with the caches and the lengths
    pdl_trigger();
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
    return launch_pdl(append_kernel, dim3(w.B), dim3(128), 0, st, 1, k_new, v_new, k_cache, v_cache, seqlens,
                      w.status, w.Hkv, w.max_len);
}

// After cache initialisation: C entries in slots 0..C-1, next slot 0, t_dec 0.
__global__ void init_done_kernel(int32_t *seq, unsigned long long *counters, int B, int C)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        seq[b * SEQ_WORDS + SEQ_HEAD] = 0;
        seq[b * SEQ_WORDS + SEQ_COUNT] = C;
        seq[b * SEQ_WORDS + SEQ_TDEC] = 0;
        for (int i = 0; i < CNT_WORDS; ++i)
            counters[(size_t)b * CNT_WORDS + i] = 0ull;
    }
}

// Zeroes n4 uint4 words (the exact step's histograms).  Launched
// programmatically, so its CTAs may become resident while the previous kernel
// drains; it waits for that kernel (which may still read the words) before it
// writes, then lets the scan that follows start (the scan reads nothing this
// kernel writes before its own wait for this grid, ahead of its flush).
__global__ void clear_words_kernel(uint4 *p, long long n4)
{
    pdl_wait();
    pdl_trigger();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t launch_clear_words(void *p, size_t bytes, cudaStream_t st)
{
    const long long n4 = (long long)(bytes / 16);
    const int blocks = (int)std::min<long long>(152, (n4 + 255) / 256);
    return launch_pdl(clear_words_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, st, 1,
                      reinterpret_cast<uint4 *>(p), n4);
}

cudaError_t launch_init_done(const Work &w, cudaStream_t st)
{
    init_done_kernel<<<(w.B + 127) / 128, 128, 0, st>>>(w.seq, w.counters, w.B, w.C);
    return cudaGetLastError();
}

}  // namespace retopk
