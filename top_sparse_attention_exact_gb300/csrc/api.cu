// api.cu -- the C ABI declared in include/retopk.h: argument checking,
// workspace layout and the launch sequence of each entry point.  No device
// memory is allocated here; every buffer lives in the caller's workspace.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace retopk {
cudaError_t configure_scan();
cudaError_t configure_select();
cudaError_t configure_finish();
size_t finish_smem_bytes_for(int max_len, int K, int RKW, int CL);
cudaError_t configure_fidelity();
cudaError_t configure_prefilter();
}  // namespace retopk

using namespace retopk;

// State of retopk_decode_step_host: pinned and device staging for the step's
// inputs and output, and the step captured as a CUDA graph for one binding of
// the caches and lengths (captured again when the binding changes).
struct HostStep {
    unsigned char *pin;     // pinned, mapped: q | k_new | v_new | out
    unsigned char *pin_d;   // its device address
    size_t o_k, o_v, o_out, bytes;
    cudaStream_t cap;       // capture stream
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    const void *k_cache, *v_cache, *seqlens;
};

struct retopk_ctx {
    retopk_config cfg;
    Work w;
    void *ws;
    size_t ws_bytes;
    int device;
    HostStep hs;
};

namespace {

constexpr size_t kAlign = 256;

struct Layout {
    size_t off[32];
    int n = 0;
    size_t total = 0;
    size_t add(size_t bytes)
    {
        total = (total + kAlign - 1) / kAlign * kAlign;
        const size_t o = total;
        total += bytes;
        off[n++] = o;
        return o;
    }
};

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_rc(cudaError_t e)
{
    if (e == cudaSuccess)
        return RETOPK_OK;
    g_last_cuda_error = e;
    return RETOPK_ERR_CUDA;
}

// Both the SM count and the kernels' attributes (cudaFuncSetAttribute) belong
// to a device: they are kept per device, for the device current at the call.
constexpr int kMaxDevices = 64;

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return -1;
    return dev;
}

int sm_count()
{
    static std::atomic<int> n[kMaxDevices];
    const int dev = current_device();
    if (dev < 0)
        return 1;
    int v = n[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
            v = 1;
        n[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int ensure_configured()
{
    static std::once_flag once[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    const int dev = current_device();
    if (dev < 0)
        return RETOPK_ERR_UNSUPPORTED;
    std::call_once(once[dev], [dev] {
        cudaError_t e = configure_scan();
        if (e == cudaSuccess)
            e = configure_select();
        if (e == cudaSuccess)
            e = configure_finish();
        if (e == cudaSuccess)
            e = configure_fidelity();
        if (e == cudaSuccess)
            e = configure_prefilter();
        err[dev] = e;
    });
    return cuda_rc(err[dev]);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Per-head capacity of the candidate arrays: the segments of an exact head
// (one per CTA of its cluster, each a multiple of 16 entries; the largest over
// every cluster size, so the workspace does not depend on it) or a reuse
// head's A_t.
int cand_stride_for(int max_len, int RKW)
{
    int s = RKW;
    for (int cl = 1; cl <= kExactCluster; cl <<= 1)
        s = std::max(s, ((((max_len + cl - 1) / cl) + 15) & ~15) * cl);
    return (s + 63) & ~63;
}

// CTAs per head in the back end (see retopk_config.cluster): the largest of 8,
// 4, 2, 1 whose B*Hq clusters fit one wave at two CTAs per SM (fewer CTAs per
// head cost latency per head but save whole waves of clusters once the batch
// has many heads), raised while the reuse path's shared memory would not fit.
int cluster_for(const retopk_config &c, bool stateful)
{
    if (c.cluster)
        return c.cluster;
    const long long heads = (long long)c.batch * c.n_q_heads, slots = 2LL * sm_count();
    int cl = kExactCluster;
    while (cl > 1 && heads * cl > slots)
        cl >>= 1;
    while (stateful && cl < kExactCluster &&
           finish_smem_bytes_for(c.max_len, c.K, c.R * c.K + c.W, cl) > kMaxDynSmem)
        cl <<= 1;
    return cl;
}

// The per-context state of a decode context: the query-support cache of
// Eq. (5), the ring words, the counters and the sticky status word.  Fills the
// pointers when base != NULL; returns the bytes.
size_t plan_state(const retopk_config &c, Work *w, char *base)
{
    const size_t BH = (size_t)c.batch * c.n_q_heads;
    Layout L;
    const size_t o_fq = L.add(BH * c.C * kD * 2);
    const size_t o_fs = L.add(BH * c.C * c.K * 4);
    const size_t o_fl = L.add(BH * c.C * 4);
    const size_t o_seq = L.add((size_t)c.batch * SEQ_WORDS * 4);
    const size_t o_cnt = L.add((size_t)c.batch * CNT_WORDS * 8);
    const size_t o_st = L.add(16);
    if (base && w) {
        w->fifo_q = (uint16_t *)(base + o_fq);
        w->fifo_sup = (int32_t *)(base + o_fs);
        w->fifo_len = (int32_t *)(base + o_fl);
        w->seq = (int32_t *)(base + o_seq);
        w->counters = (unsigned long long *)(base + o_cnt);
        w->status = (uint32_t *)(base + o_st);
    }
    return L.total + kAlign;
}

// The per-step scratch: written and read within one step (plus the last
// step's diagnostics), so the steps of several contexts that never overlap on
// the GPU can share it.  `stateful` adds the decode-only buffers; a stateless
// exact step also keeps its status word here.  Fills the sizes (and, when
// base != NULL, the pointers); returns the bytes.
size_t plan_scratch(const retopk_config &c, bool stateful, Work *w, char *base)
{
    const int RKW = stateful ? c.R * c.K + c.W : 0;
    const int cand_stride = cand_stride_for(c.max_len, RKW);
    const int sc_stride = (c.max_len + 15) & ~15;
    const size_t BH = (size_t)c.batch * c.n_q_heads;
    Layout L;
    size_t o_snap = 0, o_path = 0, o_rho = 0, o_topr = 0, o_qs = 0, o_st = 0;
    if (stateful) {
        o_snap = L.add((size_t)c.batch * SEQ_WORDS * 4);
        o_path = L.add(BH * 4);
        o_rho = L.add(BH * 4);
        o_topr = L.add(BH * c.R * 4);
        o_qs = L.add(BH * kD * 2);
    } else {
        o_st = L.add(16);
    }
    const size_t o_M = L.add(BH * 4);
    const size_t o_ci = L.add(BH * cand_stride * 4);
    const size_t o_ck = L.add(BH * cand_stride * 4);
    const size_t o_sc = L.add(BH * (size_t)sc_stride * 4);
    const size_t o_h = L.add(BH * kHistBins * 4);
    // the exact-head prefilter's arrays (decode contexts whose CTAs at 8 per
    // head hold more than one window of scores)
    const int seg8 = (((c.max_len + kExactCluster - 1) / kExactCluster) + 15) & ~15;
    const int pf_nw = stateful && seg8 > kSliceCap ? (seg8 + kSliceCap - 1) / kSliceCap : 0;
    size_t o_pfc = 0, o_pfh = 0;
    if (pf_nw) {
        o_pfc = L.add(BH * kExactCluster * pf_nw * 4);
        o_pfh = L.add(BH * kExactCluster * 256 * 4);
    }
    const size_t o_sup = L.add(BH * c.K * 4);
    const size_t o_sl = L.add(BH * 4);
    const size_t o_of = L.add(BH * kD * 4);
    if (w) {
        w->cand_stride = cand_stride;
        w->sc_stride = sc_stride;
        w->pf_nw = pf_nw;
    }
    if (base && w) {
        if (stateful) {
            w->snap = (int32_t *)(base + o_snap);
            w->path = (int32_t *)(base + o_path);
            w->rho_max = (float *)(base + o_rho);
            w->topR = (int32_t *)(base + o_topr);
            w->q_stage = (uint16_t *)(base + o_qs);
        } else {
            w->status = (uint32_t *)(base + o_st);
        }
        w->M = (int32_t *)(base + o_M);
        w->cand_idx = (int32_t *)(base + o_ci);
        w->cand_key = (uint32_t *)(base + o_ck);
        w->scores = (float *)(base + o_sc);
        w->pf_cnt = pf_nw ? (int32_t *)(base + o_pfc) : nullptr;
        w->pf_h2 = pf_nw ? (uint32_t *)(base + o_pfh) : nullptr;
        w->hist = (uint32_t *)(base + o_h);
        w->support = (int32_t *)(base + o_sup);
        w->sup_len = (int32_t *)(base + o_sl);
        w->out_f32 = (float *)(base + o_of);
    }
    return L.total + kAlign;
}

// The configuration's scalar fields in a Work (no buffers).
Work work_of(const retopk_config &c)
{
    Work x;
    memset(&x, 0, sizeof x);
    x.B = c.batch;
    x.Hq = c.n_q_heads;
    x.Hkv = c.n_kv_heads;
    x.G = c.n_q_heads / c.n_kv_heads;
    x.max_len = c.max_len;
    x.K = c.K;
    x.C = c.C;
    x.W = c.W;
    x.R = c.R;
    x.T_r = c.T_r;
    x.tau = c.tau;
    x.retrieval = c.retrieval;
    return x;
}

// One workspace holding everything: a decode context's state then its
// scratch, or a stateless exact step's scratch.  Fills the pointers when
// base != NULL; returns the bytes.
size_t plan(const retopk_config &c, bool stateful, Work *w, char *base)
{
    Work x = work_of(c);
    const size_t ns = stateful ? plan_state(c, &x, base) : 0;
    const size_t nt = plan_scratch(c, stateful, &x, base ? base + ns : nullptr);
    if (w)
        *w = x;
    return ns + nt;
}

int check_dims(int B, int Hq, int Hkv, int d, int max_len, int K)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || max_len < 1 || K < 1)
        return RETOPK_ERR_INVALID;
    if (Hq % Hkv != 0)
        return RETOPK_ERR_INVALID;
    if (d != kD || Hq / Hkv > kMaxGroup || max_len > kMaxLen || K > kMaxK || (long long)B * Hkv > kMaxSeqGroups ||
        (long long)B * Hkv * max_len > kMaxRows)
        return RETOPK_ERR_UNSUPPORTED;
    return RETOPK_OK;
}

int check_cfg(const retopk_config *c)
{
    if (!c)
        return RETOPK_ERR_INVALID;
    int e = check_dims(c->batch, c->n_q_heads, c->n_kv_heads, c->head_dim, c->max_len, c->K);
    if (e)
        return e;
    if (c->C < 1 || c->C > kMaxC || c->R < 1 || c->R > c->C || c->W < 0 || c->T_r < 0)
        return RETOPK_ERR_INVALID;
    if (c->cluster != 0 && c->cluster != 1 && c->cluster != 2 && c->cluster != 4 && c->cluster != 8)
        return RETOPK_ERR_INVALID;
    if ((long long)c->R * c->K + c->W > kMaxCand)
        return RETOPK_ERR_UNSUPPORTED;
    // the reuse path's bitmap slice and candidate lists share one CTA's shared
    // memory (the slice is smallest with 8 CTAs per head, which the automatic
    // choice falls back to); the query-support cache is addressed with 32-bit
    // offsets
    if (finish_smem_bytes_for(c->max_len, c->K, c->R * c->K + c->W, c->cluster ? c->cluster : kExactCluster) >
            kMaxDynSmem ||
        (long long)c->batch * c->n_q_heads * c->C * c->K > INT32_MAX)
        return RETOPK_ERR_UNSUPPORTED;
    if (isnan(c->tau))
        return RETOPK_ERR_INVALID;
    if (c->retrieval != RETOPK_RETRIEVE_SIMILAR && c->retrieval != RETOPK_RETRIEVE_RECENT)
        return RETOPK_ERR_INVALID;
    return RETOPK_OK;
}


// ---- optional scan timing -------------------------------------------------
// Optional per-kernel timing.  With profiling on, every launch of a decode or
// exact step is bracketed by two CUDA events on its stream.  Outside stream
// capture the events are recorded eagerly and consumed by the next read; under
// capture they become event-record nodes of the graph (cudaEventRecordExternal)
// and are kept, so every replay re-times them and every read reports the last
// replay.
struct Mark {
    int id;
    cudaEvent_t a, b;
    bool graph;
};
struct Prof {
    std::mutex mu;
    bool on = false;
    std::vector<Mark> marks;
} g_prof;

bool capturing(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive;
}

void record(cudaEvent_t e, cudaStream_t st, bool graph)
{
    if (graph)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}

// Runs `launch` (returning cudaError_t) between two profiling events.
template <class F>
cudaError_t timed(int id, cudaStream_t st, F launch)
{
    if (!g_prof.on)
        return launch();
    Mark m{id, nullptr, nullptr, capturing(st)};
    if (cudaEventCreate(&m.a) != cudaSuccess || cudaEventCreate(&m.b) != cudaSuccess) {
        if (m.a)
            cudaEventDestroy(m.a);
        return launch();
    }
    record(m.a, st, m.graph);
    const cudaError_t e = launch();
    record(m.b, st, m.graph);
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.marks.push_back(m);
    return e;
}

int run_scan(const Work &w, QSrc q, const uint16_t *k, const int32_t *sl, int off, cudaStream_t st)
{
    return cuda_rc(timed(RETOPK_PROF_SCAN, st, [&] { return launch_scan(w, q, k, sl, off, st); }));
}

// The scan is persistent: one CTA per SM shares the tiles of every active group.
int n_scan_for(int B, int Hkv, int max_len)
{
    const long long tiles = (long long)B * Hkv * ((max_len + 127) / 128);
    return (int)std::max(1LL, std::min<long long>(sm_count() * scan_ctas_per_sm(), tiles));
}

// Scratch of exact_topk_attention_step_noalloc: 16 MiB held by every GPU that
// loads the library, for as long as the process lives.  Every call shares it,
// so calls that overlap on the GPU race.
constexpr size_t kNoallocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array on the current device, looked up once per
// device (with that device current) on the first call made there.
int noalloc_scratch(void **out)
{
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return cuda_rc(ce);
    if (dev < 0 || dev >= kMaxDevices)
        return RETOPK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (ce != cudaSuccess)
            return cuda_rc(ce);
        addr[dev] = p;
    }
    *out = addr[dev];
    return RETOPK_OK;
}

}  // namespace

extern "C" {

size_t retopk_workspace_bytes(const retopk_config *cfg)
{
    if (check_cfg(cfg))
        return 0;
    return plan(*cfg, true, nullptr, nullptr);
}

size_t retopk_state_workspace_bytes(const retopk_config *cfg)
{
    if (check_cfg(cfg))
        return 0;
    return plan_state(*cfg, nullptr, nullptr);
}

size_t retopk_scratch_bytes(const retopk_config *cfg)
{
    if (check_cfg(cfg))
        return 0;
    return plan_scratch(*cfg, true, nullptr, nullptr);
}

int retopk_create_shared(const retopk_config *cfg, void *d_state, size_t state_bytes, void *d_scratch,
                         size_t scratch_bytes, retopk_ctx **out)
{
    int e = check_cfg(cfg);
    if (e)
        return e;
    if (!out || !d_state || !d_scratch)
        return RETOPK_ERR_INVALID;
    const size_t ns = plan_state(*cfg, nullptr, nullptr), nt = plan_scratch(*cfg, true, nullptr, nullptr);
    if (((uintptr_t)d_state & (kAlign - 1)) != 0 || ((uintptr_t)d_scratch & (kAlign - 1)) != 0 ||
        state_bytes < ns || scratch_bytes < nt)
        return RETOPK_ERR_WORKSPACE;
    if ((e = ensure_configured()))
        return e;
    retopk_ctx *c = (retopk_ctx *)calloc(1, sizeof(retopk_ctx));
    if (!c)
        return RETOPK_ERR_INVALID;
    c->cfg = *cfg;
    c->ws = d_state;
    c->ws_bytes = state_bytes;
    cudaGetDevice(&c->device);
    c->w = work_of(*cfg);
    plan_state(*cfg, &c->w, (char *)d_state);
    plan_scratch(*cfg, true, &c->w, (char *)d_scratch);
    c->w.n_scan = n_scan_for(cfg->batch, cfg->n_kv_heads, cfg->max_len);
    c->w.cluster = cluster_for(*cfg, true);
    c->w.prefilter = c->w.pf_nw > 0 && c->w.cluster == kExactCluster && (long long)cfg->batch * cfg->n_q_heads <= kPfMaxHeads;
    // the state starts at zero; the scratch holds nothing a step reads before writing it
    cudaError_t ce = cudaMemset(d_state, 0, ns);
    if (ce == cudaSuccess)
        ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) {
        free(c);
        return cuda_rc(ce);
    }
    *out = c;
    return RETOPK_OK;
}

int retopk_create(const retopk_config *cfg, void *d_workspace, size_t bytes, retopk_ctx **out)
{
    int e = check_cfg(cfg);
    if (e)
        return e;
    if (!out || !d_workspace)
        return RETOPK_ERR_INVALID;
    if (((uintptr_t)d_workspace & (kAlign - 1)) != 0 || bytes < plan(*cfg, true, nullptr, nullptr))
        return RETOPK_ERR_WORKSPACE;
    if ((e = ensure_configured()))
        return e;
    retopk_ctx *c = (retopk_ctx *)calloc(1, sizeof(retopk_ctx));
    if (!c)
        return RETOPK_ERR_INVALID;
    c->cfg = *cfg;
    c->ws = d_workspace;
    c->ws_bytes = bytes;
    cudaGetDevice(&c->device);
    plan(*cfg, true, &c->w, (char *)d_workspace);
    c->w.n_scan = n_scan_for(cfg->batch, cfg->n_kv_heads, cfg->max_len);
    c->w.cluster = cluster_for(*cfg, true);
    c->w.prefilter = c->w.pf_nw > 0 && c->w.cluster == kExactCluster && (long long)cfg->batch * cfg->n_q_heads <= kPfMaxHeads;
    cudaError_t ce = cudaMemset(d_workspace, 0, plan(*cfg, true, nullptr, nullptr));
    if (ce == cudaSuccess)
        ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) {
        free(c);
        return cuda_rc(ce);
    }
    *out = c;
    return RETOPK_OK;
}

namespace {

void release_host_step(HostStep &h)
{
    if (h.exec)
        cudaGraphExecDestroy(h.exec);
    if (h.graph)
        cudaGraphDestroy(h.graph);
    if (h.cap)
        cudaStreamDestroy(h.cap);
    if (h.pin)
        cudaFreeHost(h.pin);
    memset(&h, 0, sizeof h);
}

}  // namespace

int retopk_destroy(retopk_ctx *ctx)
{
    if (!ctx)
        return RETOPK_ERR_INVALID;
    release_host_step(ctx->hs);
    free(ctx);
    return RETOPK_OK;
}

int retopk_init_cache(retopk_ctx *ctx, const retopk_bf16 *q_last, const retopk_bf16 *k_cache,
                      const int32_t *d_prompt_len, void *stream)
{
    if (!ctx || !q_last || !k_cache || !d_prompt_len)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q_last) || !aligned16(k_cache))
        return RETOPK_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    const Work &w0 = ctx->w;
    std::vector<int32_t> L0(w0.B);
    cudaError_t ce = cudaMemcpyAsync(L0.data(), d_prompt_len, sizeof(int32_t) * w0.B, cudaMemcpyDeviceToHost, st);
    if (ce == cudaSuccess)
        ce = cudaStreamSynchronize(st);
    if (ce != cudaSuccess)
        return cuda_rc(ce);
    for (int b = 0; b < w0.B; ++b)
        if (L0[b] < w0.C || L0[b] > w0.max_len)
            return RETOPK_ERR_INVALID;
    // every head takes the exact path during initialisation
    Work w = w0;
    w.path = nullptr;
    QSrc qs{q_last, (long long)w.Hq * w.C * kD, (long long)w.C * kD};
    for (int c = 0; c < w.C; ++c) {
        const int off = c + 1 - w.C;   // causal prefix 0..L0-C+c
        QSrc qc{qs.q + (size_t)c * kD, qs.b_stride, qs.h_stride};
        int e;
        if ((e = cuda_rc(cudaMemsetAsync(w.hist, 0, (size_t)w.B * w.Hq * kHistBins * 4, st))))
            return e;
        if ((e = run_scan(w, qc, k_cache, d_prompt_len, off, st)))
            return e;
        if ((e = cuda_rc(launch_exact_select(w, qc, k_cache, d_prompt_len, off, FIN_INIT, c, nullptr, nullptr, st))))
            return e;
    }
    return cuda_rc(launch_init_done(w0, st));
}

int retopk_append_kv(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                     retopk_bf16 *k_cache, retopk_bf16 *v_cache, int32_t *d_seqlens, void *stream)
{
    if (!ctx || !k_new || !v_new || !k_cache || !v_cache || !d_seqlens)
        return RETOPK_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return RETOPK_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    return cuda_rc(timed(RETOPK_PROF_APPEND, st,
                         [&] { return launch_append(ctx->w, k_new, v_new, k_cache, v_cache, d_seqlens, st); }));
}

namespace {

// decide (with the append when k_new != null) -> scan -> finish.  With q_dev
// != null the decision reads q where it is (e.g. mapped host memory) and
// copies it to q_dev, from which the scan and the finish read it.
int decode_step(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new, const retopk_bf16 *q,
                retopk_bf16 *k_cache, retopk_bf16 *v_cache, int32_t *d_seqlens, retopk_bf16 *out,
                cudaStream_t st, retopk_bf16 *q_dev = nullptr)
{
    const Work &w = ctx->w;
    const retopk_bf16 *qk = q_dev ? q_dev : q;   // q as the scan and the finish read it
    QSrc qs{qk, (long long)w.Hq * kD, kD};
    int e;
    if ((e = cuda_rc(timed(RETOPK_PROF_DECIDE, st, [&] {
             return launch_decide(w, q, q_dev, k_new, v_new, k_cache, v_cache, d_seqlens, st);
         }))))
        return e;
    if ((e = run_scan(w, qs, k_cache, d_seqlens, 0, st)))
        return e;
    if (w.prefilter && (e = cuda_rc(launch_prefilter(w, d_seqlens, st))))
        return e;
    return cuda_rc(timed(RETOPK_PROF_FINISH, st,
                         [&] { return launch_finish(w, qk, k_cache, v_cache, d_seqlens, out, st); }));
}

}  // namespace

int retopk_decode_step(retopk_ctx *ctx, const retopk_bf16 *q, const retopk_bf16 *k_cache,
                       const retopk_bf16 *v_cache, const int32_t *d_seqlens, retopk_bf16 *out,
                       void *stream)
{
    if (!ctx || !q || !k_cache || !v_cache || !d_seqlens || !out)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return RETOPK_ERR_ALIGN;
    // path decision (Eqs. (6), (7), (13)); the scan of the groups with an exact
    // head; every head's back end in one launch.  Nothing is written through
    // the cache or length pointers without an append.
    return decode_step(ctx, nullptr, nullptr, q, const_cast<retopk_bf16 *>(k_cache),
                       const_cast<retopk_bf16 *>(v_cache), const_cast<int32_t *>(d_seqlens), out,
                       (cudaStream_t)stream);
}

int retopk_decode_step_kv(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                          const retopk_bf16 *q, retopk_bf16 *k_cache, retopk_bf16 *v_cache,
                          int32_t *d_seqlens, retopk_bf16 *out, void *stream)
{
    if (!ctx || !k_new || !v_new || !q || !k_cache || !v_cache || !d_seqlens || !out)
        return RETOPK_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out))
        return RETOPK_ERR_ALIGN;
    return decode_step(ctx, k_new, v_new, q, k_cache, v_cache, d_seqlens, out, (cudaStream_t)stream);
}

int retopk_decode_step_host(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                            const retopk_bf16 *q, retopk_bf16 *k_cache, retopk_bf16 *v_cache,
                            int32_t *d_seqlens, retopk_bf16 *out, void *stream)
{
    if (!ctx || !k_new || !v_new || !q || !k_cache || !v_cache || !d_seqlens || !out)
        return RETOPK_ERR_INVALID;
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return RETOPK_ERR_ALIGN;
    HostStep &h = ctx->hs;
    const Work &w = ctx->w;
    const size_t nq = (size_t)w.B * w.Hq * kD * 2, nkv = (size_t)w.B * w.Hkv * kD * 2;
    cudaStream_t st = (cudaStream_t)stream;
    if (capturing(st))   // a synchronous call with host copies cannot be captured
        return RETOPK_ERR_INVALID;
    cudaError_t ce = cudaSuccess;
    if (!h.pin) {
        auto up = [](size_t x) { return (x + kAlign - 1) / kAlign * kAlign; };
        h.o_k = up(nq);
        h.o_v = h.o_k + up(nkv);
        h.o_out = h.o_v + up(nkv);
        h.bytes = h.o_out + up(nq);
        ce = cudaHostAlloc((void **)&h.pin, h.bytes, cudaHostAllocMapped);
        if (ce == cudaSuccess)
            ce = cudaHostGetDevicePointer((void **)&h.pin_d, h.pin, 0);
        if (ce == cudaSuccess)
            ce = cudaStreamCreateWithFlags(&h.cap, cudaStreamNonBlocking);
        if (ce != cudaSuccess) {
            release_host_step(h);
            return cuda_rc(ce);
        }
    }
    if (!h.exec || h.k_cache != k_cache || h.v_cache != v_cache || h.seqlens != d_seqlens) {
        // capture the decode step on the mapped staging: the decision reads the
        // token's q, k_new, v_new across the host link (copying q to device
        // memory for the later kernels) and the finish writes the output there
        if (h.exec) {
            cudaGraphExecDestroy(h.exec);
            h.exec = nullptr;
        }
        if (h.graph) {
            cudaGraphDestroy(h.graph);
            h.graph = nullptr;
        }
        ce = cudaStreamBeginCapture(h.cap, cudaStreamCaptureModeThreadLocal);
        if (ce != cudaSuccess)
            return cuda_rc(ce);
        const int e = decode_step(ctx, (const retopk_bf16 *)(h.pin_d + h.o_k), (const retopk_bf16 *)(h.pin_d + h.o_v),
                                  (const retopk_bf16 *)h.pin_d, k_cache, v_cache, d_seqlens,
                                  (retopk_bf16 *)(h.pin_d + h.o_out), h.cap, w.q_stage);
        cudaGraph_t g = nullptr;
        ce = cudaStreamEndCapture(h.cap, &g);
        if (e) {
            if (g)
                cudaGraphDestroy(g);
            return e;
        }
        if (ce == cudaSuccess)
            ce = cudaGraphInstantiate(&h.exec, g, 0);
        if (ce != cudaSuccess) {
            if (g)
                cudaGraphDestroy(g);
            h.exec = nullptr;
            return cuda_rc(ce);
        }
        h.graph = g;
        h.k_cache = k_cache;
        h.v_cache = v_cache;
        h.seqlens = d_seqlens;
    }
    memcpy(h.pin, q, nq);
    memcpy(h.pin + h.o_k, k_new, nkv);
    memcpy(h.pin + h.o_v, v_new, nkv);
    ce = cudaGraphLaunch(h.exec, st);
    if (ce == cudaSuccess)
        ce = cudaStreamSynchronize(st);
    if (ce != cudaSuccess)
        return cuda_rc(ce);
    memcpy(out, h.pin + h.o_out, nq);
    return RETOPK_OK;
}

int retopk_fidelity(retopk_ctx *ctx, const retopk_bf16 *q, const retopk_bf16 *k_cache, const int32_t *exact_idx,
                    const retopk_bf16 *out_exact, const retopk_bf16 *out, float *metrics, void *stream)
{
    if (!ctx || !q || !k_cache || !exact_idx || !out_exact || !out || !metrics)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(out_exact) || !aligned16(out))
        return RETOPK_ERR_ALIGN;
    const Work &w = ctx->w;
    return cuda_rc(launch_fidelity(q, k_cache, exact_idx, w.support, out_exact, out, metrics, w.status, w.B, w.Hq,
                                   w.Hkv, w.max_len, w.K, (cudaStream_t)stream));
}

int retopk_support_overlap(const int32_t *S, const int32_t *others, int rows, int R, int K, float *out,
                           void *stream)
{
    if (!S || !others || !out || rows < 1 || R < 1 || R > kMaxC || K < 1 || K > kMaxK)
        return RETOPK_ERR_INVALID;
    return cuda_rc(launch_overlap(S, others, rows, R, K, out, (cudaStream_t)stream));
}

int retopk_get_diagnostics(retopk_ctx *ctx, int32_t *path, float *rho_max, int32_t *topR, int32_t *M,
                           int32_t *cand, int32_t *support, int32_t *sup_len, float *out_f32,
                           void *stream)
{
    if (!ctx)
        return RETOPK_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    const Work &w = ctx->w;
    const size_t BH = (size_t)w.B * w.Hq;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void *dst, const void *src, size_t n) {
        if (dst && e == cudaSuccess)
            e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st);
    };
    cp(path, w.path, BH * 4);
    cp(rho_max, w.rho_max, BH * 4);
    cp(topR, w.topR, BH * w.R * 4);
    cp(M, w.M, BH * 4);
    cp(support, w.support, BH * w.K * 4);
    cp(sup_len, w.sup_len, BH * 4);
    cp(out_f32, w.out_f32, BH * kD * 4);
    if (cand && e == cudaSuccess) {
        const size_t cap = (size_t)w.R * w.K + w.W;
        e = cudaMemcpy2DAsync(cand, cap * 4, w.cand_idx, (size_t)w.cand_stride * 4, cap * 4, BH,
                              cudaMemcpyDeviceToHost, st);
    }
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_rc(e);
    if (cand) {
        // entries past M_t (and every entry of exact heads) are not part of A_t
        std::vector<int32_t> Mh(BH), ph(BH);
        cudaMemcpy(Mh.data(), w.M, BH * 4, cudaMemcpyDeviceToHost);
        cudaMemcpy(ph.data(), w.path, BH * 4, cudaMemcpyDeviceToHost);
        const size_t cap = (size_t)w.R * w.K + w.W;
        for (size_t i = 0; i < BH; ++i) {
            const size_t m = ph[i] == RETOPK_PATH_REUSE ? std::min<size_t>(cap, (size_t)Mh[i]) : 0;
            for (size_t j = m; j < cap; ++j)
                cand[i * cap + j] = -1;
        }
    }
    return RETOPK_OK;
}

int retopk_get_counters(retopk_ctx *ctx, int64_t counts[5], void *stream)
{
    if (!ctx || !counts)
        return RETOPK_ERR_INVALID;
    const Work &w = ctx->w;
    std::vector<unsigned long long> h((size_t)w.B * CNT_WORDS);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t ce = cudaMemcpyAsync(h.data(), w.counters, h.size() * 8, cudaMemcpyDeviceToHost, st);
    if (ce == cudaSuccess)
        ce = cudaStreamSynchronize(st);
    if (ce != cudaSuccess)
        return cuda_rc(ce);
    for (int i = 0; i < 5; ++i)
        counts[i] = 0;
    for (int b = 0; b < w.B; ++b) {
        for (int i = 0; i < 4; ++i)
            counts[i] += (int64_t)h[(size_t)b * CNT_WORDS + i];
        counts[4] = std::max<int64_t>(counts[4], (int64_t)h[(size_t)b * CNT_WORDS + CNT_MAX_M]);
    }
    return RETOPK_OK;
}

size_t retopk_state_bytes(const retopk_ctx *ctx)
{
    if (!ctx)
        return 0;
    const Work &w = ctx->w;
    const size_t BHC = (size_t)w.B * w.Hq * w.C;
    return BHC * kD * 2 + BHC * w.K * 4 + BHC * 4 + (size_t)w.B * 3 * 4;
}

static int state_copy(retopk_ctx *ctx, void *host, size_t bytes, cudaStream_t st, bool to_host)
{
    const Work &w = ctx->w;
    if (!host || bytes != retopk_state_bytes(ctx))
        return RETOPK_ERR_STATE;
    const size_t BHC = (size_t)w.B * w.Hq * w.C;
    char *p = (char *)host;
    const cudaMemcpyKind kd = to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void *dev, size_t n) {
        if (e == cudaSuccess)
            e = to_host ? cudaMemcpyAsync(p, dev, n, kd, st) : cudaMemcpyAsync(dev, p, n, kd, st);
        p += n;
    };
    cp(w.fifo_q, BHC * kD * 2);
    cp(w.fifo_sup, BHC * w.K * 4);
    cp(w.fifo_len, BHC * 4);
    // seq words: the device keeps 4 per sequence, the buffer 3
    std::vector<int32_t> seq((size_t)w.B * SEQ_WORDS);
    if (e == cudaSuccess && to_host) {
        e = cudaMemcpyAsync(seq.data(), w.seq, seq.size() * 4, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
        for (int b = 0; b < w.B; ++b)
            memcpy(p + b * 12, &seq[(size_t)b * SEQ_WORDS], 12);
    } else if (e == cudaSuccess) {
        for (int b = 0; b < w.B; ++b) {
            memcpy(&seq[(size_t)b * SEQ_WORDS], p + b * 12, 12);
        }
        e = cudaMemcpyAsync(w.seq, seq.data(), seq.size() * 4, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    return cuda_rc(e);
}

int retopk_export_state(retopk_ctx *ctx, void *host_buf, size_t bytes, void *stream)
{
    if (!ctx)
        return RETOPK_ERR_INVALID;
    return state_copy(ctx, host_buf, bytes, (cudaStream_t)stream, true);
}

int retopk_import_state(retopk_ctx *ctx, const void *host_buf, size_t bytes, void *stream)
{
    if (!ctx)
        return RETOPK_ERR_INVALID;
    const Work &w = ctx->w;
    // validate before touching the device: slots, counts and support indices
    const size_t BHC = (size_t)w.B * w.Hq * w.C;
    if (!host_buf || bytes != retopk_state_bytes(ctx))
        return RETOPK_ERR_STATE;
    const char *p = (const char *)host_buf;
    const int32_t *len = (const int32_t *)(p + BHC * kD * 2 + BHC * w.K * 4);
    const int32_t *seq = len + BHC;
    const int32_t *sup = (const int32_t *)(p + BHC * kD * 2);
    for (size_t i = 0; i < BHC; ++i) {
        if (len[i] < 0 || len[i] > w.K)
            return RETOPK_ERR_STATE;
        // a support is a set of key positions, stored ascending
        const int32_t *si = sup + i * w.K;
        if (len[i] > 0 && si[0] < 0)
            return RETOPK_ERR_STATE;
        for (int j = 1; j < len[i]; ++j)
            if (si[j] <= si[j - 1])
                return RETOPK_ERR_STATE;
    }
    for (int b = 0; b < w.B; ++b)
        if (seq[b * 3] < 0 || seq[b * 3] >= w.C || seq[b * 3 + 1] < 0 || seq[b * 3 + 1] > w.C ||
            seq[b * 3 + 2] < 0)
            return RETOPK_ERR_STATE;
    return state_copy(ctx, const_cast<void *>(host_buf), bytes, (cudaStream_t)stream, false);
}

int retopk_get_status(retopk_ctx *ctx, uint32_t *bits, int clear, void *stream)
{
    if (!ctx || !bits)
        return RETOPK_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(bits, ctx->w.status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear)
        e = cudaMemsetAsync(ctx->w.status, 0, 4, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    return cuda_rc(e);
}

int retopk_selftest_wait(retopk_ctx *ctx, int64_t wait_cycles, void *stream)
{
    if (!ctx || wait_cycles < 0 || wait_cycles > 8000000000LL)
        return RETOPK_ERR_INVALID;
    return cuda_rc(launch_selftest_wait(ctx->w.status, (long long)wait_cycles, (cudaStream_t)stream));
}

const char *retopk_cuda_error_string(void)
{
    return g_last_cuda_error == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(g_last_cuda_error);
}

const char *retopk_strerror(int code)
{
    switch (code) {
    case RETOPK_OK: return "ok";
    case RETOPK_ERR_INVALID: return "invalid argument";
    case RETOPK_ERR_UNSUPPORTED: return "unsupported size (head_dim must be 128; group, K, C or max_len too large)";
    case RETOPK_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case RETOPK_ERR_CUDA: return "CUDA runtime error";
    case RETOPK_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case RETOPK_ERR_STATE: return "state buffer of the wrong size or with invalid contents";
    case RETOPK_ERR_SCRATCH: return "sizes need more scratch than the library's 16 MiB static array";
    default: return "unknown error";
    }
}

size_t exact_topk_workspace_bytes(int B, int Hq, int Hkv, int d, int max_len, int K)
{
    if (check_dims(B, Hq, Hkv, d, max_len, K))
        return 0;
    retopk_config c{B, Hq, Hkv, d, max_len, K, 1, 0, 1, 0, 0.f};
    return plan(c, false, nullptr, nullptr);
}

}  // extern "C"

namespace {

// The device view of a stateless exact step's workspace (both halves use it).
int exact_work(int B, int Hq, int Hkv, int d, int max_len, int K, void *d_workspace, size_t bytes, Work *w)
{
    int e = check_dims(B, Hq, Hkv, d, max_len, K);
    if (e)
        return e;
    if (!d_workspace)
        return RETOPK_ERR_INVALID;
    retopk_config c{B, Hq, Hkv, d, max_len, K, 1, 0, 1, 0, 0.f};
    const size_t need = plan(c, false, nullptr, nullptr);
    if (((uintptr_t)d_workspace & (kAlign - 1)) != 0 || bytes < need)
        return RETOPK_ERR_WORKSPACE;
    if ((e = ensure_configured()))
        return e;
    plan(c, false, w, (char *)d_workspace);
    w->n_scan = n_scan_for(B, Hkv, max_len);
    w->cluster = cluster_for(c, false);
    w->out_f32 = nullptr;
    w->support = nullptr;
    return RETOPK_OK;
}

// Eq. (4) for every key of every (b, h) into the workspace's scores, with the
// first radix digit's histograms (cleared first).
int exact_scan_half(const Work &w, const retopk_bf16 *q, const retopk_bf16 *k_cache, const int32_t *d_seqlens,
                    cudaStream_t st)
{
    int e;
    if ((e = cuda_rc(timed(RETOPK_PROF_CLEAR, st, [&] {
             return launch_clear_words(w.hist, (size_t)w.B * w.Hq * kHistBins * 4, st);
         }))))
        return e;
    return run_scan(w, QSrc{q, (long long)w.Hq * kD, kD}, k_cache, d_seqlens, 0, st);
}

// Eq. (1) over the scores the scan half left in the workspace, then Eq. (12).
int exact_select_half(const Work &w, const retopk_bf16 *q, const retopk_bf16 *v_cache, const int32_t *d_seqlens,
                      retopk_bf16 *out, int32_t *idx_out, cudaStream_t st)
{
    return cuda_rc(timed(RETOPK_PROF_SELECT, st, [&] {
        return launch_exact_select(w, QSrc{q, (long long)w.Hq * kD, kD}, v_cache, d_seqlens, 0, FIN_EXACT, 0, out,
                                   idx_out, st);
    }));
}

}  // namespace

extern "C" {

int exact_topk_attention_step(const retopk_bf16 *q, const retopk_bf16 *k_cache, const retopk_bf16 *v_cache,
                              const int32_t *d_seqlens, int B, int Hq, int Hkv, int d, int max_len, int K,
                              retopk_bf16 *out, int32_t *idx_out, void *d_workspace, size_t bytes,
                              void *stream)
{
    int e = check_dims(B, Hq, Hkv, d, max_len, K);
    if (e)
        return e;
    if (!q || !k_cache || !v_cache || !d_seqlens || !out || !d_workspace)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return RETOPK_ERR_ALIGN;
    Work w;
    if ((e = exact_work(B, Hq, Hkv, d, max_len, K, d_workspace, bytes, &w)))
        return e;
    cudaStream_t st = (cudaStream_t)stream;
    if ((e = exact_scan_half(w, q, k_cache, d_seqlens, st)))
        return e;
    return exact_select_half(w, q, v_cache, d_seqlens, out, idx_out, st);
}

int exact_topk_scan(const retopk_bf16 *q, const retopk_bf16 *k_cache, const int32_t *d_seqlens, int B, int Hq,
                    int Hkv, int d, int max_len, int K, void *d_workspace, size_t bytes, void *stream)
{
    int e = check_dims(B, Hq, Hkv, d, max_len, K);
    if (e)
        return e;
    if (!q || !k_cache || !d_seqlens || !d_workspace)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache))
        return RETOPK_ERR_ALIGN;
    Work w;
    if ((e = exact_work(B, Hq, Hkv, d, max_len, K, d_workspace, bytes, &w)))
        return e;
    return exact_scan_half(w, q, k_cache, d_seqlens, (cudaStream_t)stream);
}

int exact_topk_select(const retopk_bf16 *q, const retopk_bf16 *v_cache, const int32_t *d_seqlens, int B, int Hq,
                      int Hkv, int d, int max_len, int K, retopk_bf16 *out, int32_t *idx_out, void *d_workspace,
                      size_t bytes, void *stream)
{
    int e = check_dims(B, Hq, Hkv, d, max_len, K);
    if (e)
        return e;
    if (!q || !v_cache || !d_seqlens || !out || !d_workspace)
        return RETOPK_ERR_INVALID;
    if (!aligned16(q) || !aligned16(v_cache) || !aligned16(out))
        return RETOPK_ERR_ALIGN;
    Work w;
    if ((e = exact_work(B, Hq, Hkv, d, max_len, K, d_workspace, bytes, &w)))
        return e;
    return exact_select_half(w, q, v_cache, d_seqlens, out, idx_out, (cudaStream_t)stream);
}

// ---- allocation-free Exact Top-K step ---------------------------------------
// For callers that cannot allocate device memory at all: code running where
// allocation is forbidden or unavailable (inside a decode loop that must not
// touch the allocator, under an external memory manager that owns every byte
// of the device, or from a plain C host that has no allocator of its own to
// hand out a workspace).  The scratch the exact path needs lives in one
// file-scope device array instead of a caller-provided workspace.
int exact_topk_attention_step_noalloc(const retopk_bf16 *q, const retopk_bf16 *k_cache,
                                      const retopk_bf16 *v_cache, const int32_t *d_seqlens, int B, int Hq,
                                      int Hkv, int d, int max_len, int K, retopk_bf16 *out, int32_t *idx_out,
                                      void *stream)
{
    int e = check_dims(B, Hq, Hkv, d, max_len, K);
    if (e)
        return e;
    retopk_config c{B, Hq, Hkv, d, max_len, K, 1, 0, 1, 0, 0.f};
    if (plan(c, false, nullptr, nullptr) > kNoallocScratchBytes)
        return RETOPK_ERR_SCRATCH;
    void *scratch = nullptr;
    if ((e = noalloc_scratch(&scratch)))
        return e;
    // the existing exact path, with its workspace carved from the static array
    // (it clears the only buffer that must start at zero, the score histogram)
    return exact_topk_attention_step(q, k_cache, v_cache, d_seqlens, B, Hq, Hkv, d, max_len, K, out, idx_out,
                                     scratch, kNoallocScratchBytes, stream);
}

int retopk_profile_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.on = on != 0;
    return RETOPK_OK;
}

int retopk_profile_read(int64_t launches[RETOPK_PROF_KERNELS], double ms[RETOPK_PROF_KERNELS])
{
    if (!launches || !ms)
        return RETOPK_ERR_INVALID;
    for (int i = 0; i < RETOPK_PROF_KERNELS; ++i) {
        launches[i] = 0;
        ms[i] = 0.0;
    }
    std::lock_guard<std::mutex> lk(g_prof.mu);
    int rc = RETOPK_OK;
    std::vector<Mark> keep;
    for (auto &m : g_prof.marks) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(m.b);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&t, m.a, m.b);
        if (e == cudaSuccess && m.id >= 0 && m.id < RETOPK_PROF_KERNELS) {
            launches[m.id] += 1;
            ms[m.id] += t;
        } else if (e != cudaSuccess && !m.graph) {
            rc = cuda_rc(e);
        }
        if (m.graph) {
            keep.push_back(m);
        } else {
            cudaEventDestroy(m.a);
            cudaEventDestroy(m.b);
        }
    }
    g_prof.marks.swap(keep);
    return rc;
}

int retopk_profile_reset(void)
{
    std::lock_guard<std::mutex> lk(g_prof.mu);
    for (auto &m : g_prof.marks) {
        cudaEventDestroy(m.a);
        cudaEventDestroy(m.b);
    }
    g_prof.marks.clear();
    return RETOPK_OK;
}

}  // extern "C"
