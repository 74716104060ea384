// gcl_api.cu -- the C ABI: argument checks, launch plans, error reporting.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths
// on Ascend NPUs", section "API proposal": externally supplied metadata must
// match the expected shape and layout, and an unsupported request must fail
// clearly instead of falling back.  Every check here runs on the host before
// anything is enqueued; launch shapes depend only on the sizes, never on
// device data, so each call can be captured in a CUDA graph.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gcl_internal.cuh"
#include "transition.cuh"

namespace gcl {

static thread_local char g_err[512];

gcl_status_t fail(gcl_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

gcl_status_t cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return GCL_OK;
    return fail(GCL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
    static std::atomic<int> cache[64];                // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static gcl_status_t check_common(const char *fn, const void *q, const void *k, const void *v,
                                 const float *g, const void *beta, const int32_t *cu,
                                 int64_t t_max, int32_t n_max, int32_t H, int32_t K, int32_t V,
                                 int32_t bt, int32_t dtype) {
    if (!q || !k || !v || !g || !beta || !cu)
        return fail(GCL_ERR_INVALID_ARG, "%s: q, k, v, g, beta and cu_seqlens are required", fn);
    if (t_max < 1 || t_max >= (int64_t(1) << 31) || n_max < 1 || H < 1)
        return fail(GCL_ERR_INVALID_ARG, "%s: need 1 <= t_max < 2^31, n_max >= 1, H >= 1", fn);
    if (bt != kChunk && bt != 32)
        return fail(GCL_ERR_UNSUPPORTED, "%s: chunk size bt=%d (implemented: 32 and 64)", fn, bt);
    if ((K != 64 && K != 128) || (V != 64 && V != 128))
        return fail(GCL_ERR_UNSUPPORTED, "%s: K=%d V=%d (supported: 64 or 128 each)", fn, K, V);
    if (dtype != GCL_F32 && dtype != GCL_BF16 && dtype != GCL_F16)
        return fail(GCL_ERR_UNSUPPORTED, "%s: dtype %d (supported: GCL_F32, GCL_BF16, GCL_F16)", fn, dtype);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(cu))
        return fail(GCL_ERR_INVALID_ARG, "%s: every buffer must be 16-byte aligned", fn);
    return GCL_OK;
}

// The kernels' per-chunk records start on 1 KiB boundaries of the workspace (full cache lines
// for every TMA row); the queried sizes include the slack for aligning the caller's pointer.
constexpr size_t kWsAlign = 1024;

static void align_ws(void *ws, size_t bytes, void **out, size_t *out_bytes) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
    const uintptr_t a = (b + kWsAlign - 1) & ~(uintptr_t)(kWsAlign - 1);
    *out = reinterpret_cast<void *>(a);
    *out_bytes = bytes > a - b ? bytes - (a - b) : 0;
}

// Forward workspace: the minimum (W form) or what the fastest launch plan uses.
static size_t fwd_ws(const gcl_fwd_args *a, int variant, bool fastest) {
    const int64_t ntm = gcl_nt_max(a->t_max, a->n_max, a->bt);
    if (ntm <= 0 || a->H <= 0 || a->n_max <= 0) return 0;
    if (!fwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt)) {
        // the CUDA cores: the single kernel needs none; the split plan holds its records
        const size_t rec = fwd_simt_split_bytes(a->K, a->V, a->bt, ntm, a->H);
        return fastest && rec > 0 ? rec + kWsAlign : 0;
    }
    // the fused plan keeps everything on chip; a training forward's fastest plan is the
    // transition form (its records serve the backward), its least the fused plan
    if (fwd_tc_runs_fused(variant, a->n_max, a->H, a->h_save != nullptr, 0, ntm) &&
        (!a->h_save || !fastest))
        return 0;
    // the transition form, with the segment buffers when the fastest plan is segmented
    const size_t seg = fastest ? fwd_seg_workspace_bytes(ntm, a->n_max, a->H) : 0;
    if (variant == kKDA || a->dtype == GCL_F16)     // the transition form only (no W form)
        return fwd_tc_t_workspace_bytes(ntm, a->H) + seg + kWsAlign;
    if (fastest && (fwd_tc_prefers_transition(a->n_max, a->H) || a->h_save))
        return fwd_tc_t_workspace_bytes(ntm, a->H) + seg + kWsAlign;
    return fwd_tc_workspace_bytes(ntm, a->H) + kWsAlign;
}

static gcl_status_t run_fwd(const gcl_fwd_args *a, gcl_stream_t stream, int variant) {
    const char *fn = variant == kGDN ? "gdn_chunk_fwd" : "kda_chunk_fwd";
    if (!a) return fail(GCL_ERR_INVALID_ARG, "%s: args is NULL", fn);
    gcl_status_t st = check_common(fn, a->q, a->k, a->v, a->g, a->beta, a->cu_seqlens, a->t_max,
                                   a->n_max, a->H, a->K, a->V, a->bt, a->dtype);
    if (st != GCL_OK) return st;
    if (a->h_save && !a->chunk_offsets)
        return fail(GCL_ERR_INVALID_ARG, "%s: h_save needs chunk_offsets", fn);
    const bool tc = fwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt);
    const int64_t ntm = gcl_nt_max(a->t_max, a->n_max, a->bt);
    if (tc) {
        if (!a->chunk_indices || !a->chunk_offsets)
            return fail(GCL_ERR_INVALID_ARG,
                        "%s: chunk_indices and chunk_offsets are required for bf16 K=V=128", fn);
        const size_t need = fwd_ws(a, variant, false);
        if (need > 0 && (!a->workspace || a->workspace_bytes < need))
            return fail(GCL_ERR_CAPACITY,
                        "%s: workspace of at least %zu bytes needed (%zu for the fastest "
                        "plan), %zu given",
                        fn, need, fwd_ws(a, variant, true),
                        a->workspace ? a->workspace_bytes : (size_t)0);
        if (a->workspace && !aligned16(a->workspace))
            return fail(GCL_ERR_INVALID_ARG, "%s: every buffer must be 16-byte aligned", fn);
    }
    if ((a->o && !aligned16(a->o)) || (a->ht && !aligned16(a->ht)) ||
        (a->h0 && !aligned16(a->h0)) || (a->h_save && !aligned16(a->h_save)))
        return fail(GCL_ERR_INVALID_ARG, "%s: every buffer must be 16-byte aligned", fn);
    FwdParams p{};
    p.q = a->q; p.k = a->k; p.v = a->v; p.g = a->g; p.beta = a->beta; p.h0 = a->h0;
    p.cu_seqlens = a->cu_seqlens; p.chunk_indices = a->chunk_indices;
    p.chunk_offsets = a->chunk_offsets; p.seq_order = a->seq_order;
    p.o = a->o; p.ht = a->ht; p.h_save = a->h_save; p.dev_status = a->dev_status;
    p.workspace = nullptr;
    p.workspace_bytes = 0;
    if (a->workspace) {
        if (!aligned16(a->workspace))
            return fail(GCL_ERR_INVALID_ARG, "%s: every buffer must be 16-byte aligned", fn);
        align_ws(a->workspace, a->workspace_bytes, &p.workspace, &p.workspace_bytes);
    }
    p.t_max = a->t_max; p.n_max = a->n_max; p.H = a->H; p.K = a->K; p.V = a->V; p.bt = a->bt;
    p.nt_max = ntm;
    p.scale = a->scale;
    p.dtype = a->dtype;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = tc ? launch_fwd_tc(p, variant, s) : launch_fwd_simt(p, variant, a->dtype, s);
    return cuda_check(e, fn);
}


static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Backward workspace: dS' per chunk [nt_max, H, K, V] fp32; without saved states also
// the recomputed states (same shape) and the forward's own workspace; on the tensor-core
// path also the transition-form records the state-gradient sweep reads.
// KDA runs the backward on the CUDA cores (its recompute forward may use the tensor cores).
// The forward's records, when the caller hands over the workspace of a forward that ran the
// transition plan (decided from the sizes alone, as the forward decided), else NULL.
static const uint8_t *fwd_records(const gcl_bwd_args *a, int variant, int64_t ntm) {
    if (!a->h_save || !a->fwd_workspace || !bwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt))
        return nullptr;
    void *w = nullptr;
    size_t wb = 0;
    align_ws(const_cast<void *>(a->fwd_workspace), a->fwd_workspace_bytes, &w, &wb);
    if (!fwd_tc_runs_transition(variant, a->n_max, a->H, true, wb, ntm)) return nullptr;
    return static_cast<const uint8_t *>(w);
}

static size_t bwd_ws(const gcl_bwd_args *a, int variant) {
    const int64_t ntm = gcl_nt_max(a->t_max, a->n_max, a->bt);
    if (ntm <= 0 || a->H <= 0 || a->K <= 0 || a->V <= 0) return 0;
    const bool tc_fwd = bwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt);
    const bool tc = variant == kGDN && tc_fwd;
    const size_t per = align256(sizeof(float) * (size_t)ntm * a->H * a->K * a->V);
    // tensor-core sweep (GDN and KDA bf16 K = V = 128): transition records (unless the
    // forward's, or the state recompute's, are reused); GDN's tensor-core chunk gradients also
    // a scratch record per chunk and head
    const bool own_records = tc_fwd && a->h_save && !fwd_records(a, variant, ntm);
    const size_t rec = !tc_fwd ? 0
                       : (own_records ? align256(transition_record_bytes(ntm, a->H)) : 0) + kWsAlign +
                             (tc ? align256(bwd_grad_tc_scratch_bytes(ntm, a->H)) : 0);
    if (a->h_save) return per + rec;
    // the state recompute runs the transition plan, whose records the sweep then reads
    const size_t fw = !tc_fwd ? 0 : align256(fwd_tc_t_workspace_bytes(ntm, a->H)) + kWsAlign;
    return 2 * per + fw + rec;
}

}  // namespace gcl

using namespace gcl;

static gcl_status_t run_bwd(const gcl_bwd_args *a, gcl_stream_t stream, int variant) {
    g_err[0] = 0;
    const char *fn = variant == kGDN ? "gdn_chunk_bwd" : "kda_chunk_bwd";
    if (!a) return fail(GCL_ERR_INVALID_ARG, "%s: args is NULL", fn);
    gcl_status_t st = check_common(fn, a->q, a->k, a->v, a->g, a->beta, a->cu_seqlens, a->t_max,
                                   a->n_max, a->H, a->K, a->V, a->bt, a->dtype);
    if (st != GCL_OK) return st;
    if (!a->d_o || !a->chunk_indices || !a->chunk_offsets || !a->dq || !a->dk || !a->dv ||
        !a->dg || !a->dbeta)
        return fail(GCL_ERR_INVALID_ARG,
                    "%s: d_o, chunk_indices, chunk_offsets, dq, dk, dv, dg, dbeta are required",
                    fn);
    const size_t need = bwd_ws(a, variant);
    if (!a->workspace || a->workspace_bytes < need)
        return fail(GCL_ERR_CAPACITY, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    if (!aligned16(a->workspace) || !aligned16(a->d_o) || !aligned16(a->dq) ||
        !aligned16(a->dk) || !aligned16(a->dv) || !aligned16(a->dg) || !aligned16(a->dbeta))
        return fail(GCL_ERR_INVALID_ARG, "%s: every buffer must be 16-byte aligned", fn);
    const int64_t ntm = gcl_nt_max(a->t_max, a->n_max, a->bt);
    const size_t per = align256(sizeof(float) * (size_t)ntm * a->H * a->K * a->V);
    char *ws = static_cast<char *>(a->workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    BwdParams p{};
    p.q = a->q; p.k = a->k; p.v = a->v; p.g = a->g; p.beta = a->beta; p.h0 = a->h0;
    p.d_o = a->d_o; p.dht = a->dht; p.cu_seqlens = a->cu_seqlens;
    p.chunk_indices = a->chunk_indices; p.chunk_offsets = a->chunk_offsets;
    p.dh = reinterpret_cast<float *>(ws);
    p.dq = a->dq; p.dk = a->dk; p.dv = a->dv; p.dg = a->dg; p.dbeta = a->dbeta; p.dh0 = a->dh0;
    p.dev_status = a->dev_status;
    p.t_max = a->t_max; p.nt_max = ntm; p.n_max = a->n_max;
    p.H = a->H; p.K = a->K; p.V = a->V; p.bt = a->bt; p.scale = a->scale;
    const bool tc_fwd = bwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt);
    const bool tc = variant == kGDN && tc_fwd;        // tensor-core backward: GDN
    FwdParams f{};
    f.q = a->q; f.k = a->k; f.v = a->v; f.g = a->g; f.beta = a->beta; f.h0 = a->h0;
    f.cu_seqlens = a->cu_seqlens; f.chunk_indices = a->chunk_indices;
    f.chunk_offsets = a->chunk_offsets; f.seq_order = nullptr;
    f.o = nullptr; f.ht = nullptr; f.h_save = nullptr; f.dev_status = a->dev_status;
    f.t_max = a->t_max; f.n_max = a->n_max; f.H = a->H; f.K = a->K; f.V = a->V; f.bt = a->bt;
    f.nt_max = ntm;
    f.scale = a->scale;
    f.dtype = a->dtype;
    const size_t fw = !tc_fwd ? 0 : align256(fwd_tc_t_workspace_bytes(ntm, a->H)) + kWsAlign;
    const size_t used = a->h_save ? per : 2 * per + fw;
    const uint8_t *records = fwd_records(a, variant, ntm);    // the training forward's
    if (a->h_save) {
        p.h = a->h_save;
    } else {
        float *h = reinterpret_cast<float *>(ws + per);
        f.h_save = h;
        f.workspace = nullptr;
        f.workspace_bytes = 0;
        if (tc_fwd)     // the transition plan: its records serve the sweep below
            align_ws(ws + 2 * per, fw - 1, &f.workspace, &f.workspace_bytes);
        cudaError_t e = tc_fwd ? launch_fwd_tc(f, variant, s) : launch_fwd_simt(f, variant, a->dtype, s);
        if ((st = cuda_check(e, variant == kKDA ? "kda_chunk_bwd (state recompute)"
                                                : "gdn_chunk_bwd (state recompute)")) != GCL_OK)
            return st;
        if (tc_fwd) records = static_cast<const uint8_t *>(f.workspace);
        f.h_save = nullptr;
        p.h = h;
    }
    if (tc_fwd) {   // transition-form records, then the state-gradient sweep on the tensor cores
        void *rec = nullptr;
        size_t rec_bytes = 0;
        align_ws(ws + used, a->workspace_bytes - used, &rec, &rec_bytes);
        const size_t own = records ? 0 : align256(transition_record_bytes(ntm, a->H));
        if (rec_bytes < own + (tc ? bwd_grad_tc_scratch_bytes(ntm, a->H) : 0))
            return fail(GCL_ERR_CAPACITY, "%s: workspace too small for the sweep records", fn);
        cudaError_t e = cudaSuccess;
        if (!records) {
            e = variant == kKDA ? launch_prep_kda(f, static_cast<uint8_t *>(rec), s)
                                : launch_prep_t(f, static_cast<uint8_t *>(rec), s);
            records = static_cast<const uint8_t *>(rec);
        }
        if (e == cudaSuccess) e = launch_bwd_sweep_t(p, records, variant == kKDA, s);
        if ((st = cuda_check(e, variant == kKDA ? "kda_chunk_bwd (state-gradient sweep)"
                                                : "gdn_chunk_bwd (state-gradient sweep)")) != GCL_OK)
            return st;
        if (variant == kKDA) return cuda_check(launch_bwd_simt_kda(p, a->dtype, true, s), fn);
        // chunk gradients on the tensor cores; their scratch follows the records (if any)
        float *scratch = reinterpret_cast<float *>(static_cast<uint8_t *>(rec) + own);
        return cuda_check(launch_bwd_grad_tc(p, scratch, s), fn);
    }
    if (variant == kKDA) return cuda_check(launch_bwd_simt_kda(p, a->dtype, false, s), fn);
    return cuda_check(launch_bwd_simt(p, a->dtype, false, s), fn);
}

extern "C" {

const char *gcl_last_error(void) { return g_err; }

const char *gcl_status_string(int32_t s) {
    switch (s) {
        case GCL_OK: return "GCL_OK";
        case GCL_ERR_INVALID_ARG: return "GCL_ERR_INVALID_ARG";
        case GCL_ERR_UNSUPPORTED: return "GCL_ERR_UNSUPPORTED";
        case GCL_ERR_CAPACITY: return "GCL_ERR_CAPACITY";
        case GCL_ERR_CUDA: return "GCL_ERR_CUDA";
        default: return "unknown";
    }
}

int64_t gcl_nt_max(int64_t t_max, int64_t n_max, int32_t bt) {
    if (t_max <= 0 || n_max <= 0 || bt <= 0) return -1;
    return (t_max + bt - 1) / bt + n_max - 1;
}

gcl_status_t chunk_meta_build(const int32_t *cu_seqlens, int32_t n_max, int64_t t_max,
                              int32_t bt, int64_t nt_max, int32_t *chunk_indices,
                              int32_t *chunk_offsets, int32_t *seq_order, int32_t *dev_status,
                              gcl_stream_t stream) {
    g_err[0] = 0;
    if (!cu_seqlens || !chunk_indices || !chunk_offsets || !dev_status)
        return fail(GCL_ERR_INVALID_ARG,
                    "chunk_meta_build: cu_seqlens, chunk_indices, chunk_offsets, dev_status "
                    "are required");
    if (n_max < 1 || t_max < 1 || t_max >= (int64_t(1) << 31) || bt < 1)
        return fail(GCL_ERR_INVALID_ARG,
                    "chunk_meta_build: need n_max >= 1, 1 <= t_max < 2^31, bt >= 1");
    if (nt_max != gcl_nt_max(t_max, n_max, bt))
        return fail(GCL_ERR_INVALID_ARG, "chunk_meta_build: nt_max=%lld, expected %lld",
                    (long long)nt_max, (long long)gcl_nt_max(t_max, n_max, bt));
    return cuda_check(launch_chunk_meta(cu_seqlens, n_max, t_max, bt, nt_max, chunk_indices,
                                        chunk_offsets, seq_order, dev_status,
                                        static_cast<cudaStream_t>(stream)),
                      "chunk_meta_build");
}

gcl_status_t chunk_meta_build_i64(const int64_t *cu_seqlens, int32_t n_max, int64_t t_max,
                                  int32_t bt, int64_t nt_max, int32_t *cu_seqlens32,
                                  int32_t *chunk_indices, int32_t *chunk_offsets, int32_t *seq_order,
                                  int32_t *dev_status, gcl_stream_t stream) {
    g_err[0] = 0;
    if (!cu_seqlens || !cu_seqlens32 || !chunk_indices || !chunk_offsets || !dev_status)
        return fail(GCL_ERR_INVALID_ARG,
                    "chunk_meta_build_i64: cu_seqlens, cu_seqlens32, chunk_indices, chunk_offsets, "
                    "dev_status are required");
    if (n_max < 1 || t_max < 1 || t_max >= (int64_t(1) << 31) || bt < 1)
        return fail(GCL_ERR_INVALID_ARG,
                    "chunk_meta_build_i64: need n_max >= 1, 1 <= t_max < 2^31, bt >= 1");
    if (nt_max != gcl_nt_max(t_max, n_max, bt))
        return fail(GCL_ERR_INVALID_ARG, "chunk_meta_build_i64: nt_max=%lld, expected %lld",
                    (long long)nt_max, (long long)gcl_nt_max(t_max, n_max, bt));
    return cuda_check(launch_chunk_meta_i64(cu_seqlens, n_max, t_max, bt, nt_max, cu_seqlens32,
                                            chunk_indices, chunk_offsets, seq_order, dev_status,
                                            static_cast<cudaStream_t>(stream)),
                      "chunk_meta_build_i64");
}

size_t gcl_fwd_workspace_bytes(const gcl_fwd_args *args) {
    if (!args) return 0;
    return fwd_ws(args, kGDN, true);
}

size_t gcl_fwd_workspace_min_bytes(const gcl_fwd_args *args) {
    if (!args) return 0;
    return fwd_ws(args, kGDN, false);
}
size_t gcl_kda_fwd_workspace_bytes(const gcl_fwd_args *args) {
    if (!args) return 0;
    return fwd_ws(args, kKDA, true);
}

static int32_t fwd_plan(const gcl_fwd_args *a, int variant) {
    if (!a) return -1;
    if (check_common("plan", a->q, a->k, a->v, a->g, a->beta, a->cu_seqlens, a->t_max, a->n_max,
                     a->H, a->K, a->V, a->bt, a->dtype) != GCL_OK)
        return -1;
    void *w = nullptr;
    size_t wb = 0;
    if (a->workspace) align_ws(a->workspace, a->workspace_bytes, &w, &wb);
    if (!fwd_tc_supported(variant, a->dtype, a->K, a->V, a->bt)) {
        const size_t rec = fwd_simt_split_bytes(a->K, a->V, a->bt, gcl_nt_max(a->t_max, a->n_max, a->bt), a->H);
        return rec > 0 && w && wb >= rec && a->chunk_indices && a->chunk_offsets ? GCL_PLAN_CUDA_CORES_SPLIT
                                                                                  : GCL_PLAN_CUDA_CORES;
    }
    return fwd_tc_plan(variant, a->n_max, a->H, a->h_save != nullptr, wb,
                       gcl_nt_max(a->t_max, a->n_max, a->bt), a->dtype);
}

int32_t gcl_fwd_plan(const gcl_fwd_args *args) { return fwd_plan(args, kGDN); }
int32_t gcl_kda_fwd_plan(const gcl_fwd_args *args) { return fwd_plan(args, kKDA); }

int32_t gcl_fwd_chain_segments(int64_t t_max, int32_t n_max, int32_t H, int32_t bt) {
    const int64_t ntm = gcl_nt_max(t_max, n_max, bt);
    if (ntm <= 0 || H <= 0 || bt != kChunk) return 0;
    return fwd_seg_count(ntm, n_max, H);
}

gcl_status_t gdn_chunk_fwd(const gcl_fwd_args *args, gcl_stream_t stream) {
    g_err[0] = 0;
    return run_fwd(args, stream, kGDN);
}

gcl_status_t kda_chunk_fwd(const gcl_fwd_args *args, gcl_stream_t stream) {
    g_err[0] = 0;
    return run_fwd(args, stream, kKDA);
}

size_t gcl_kda_bwd_workspace_bytes(const gcl_bwd_args *a) {
    if (!a) return 0;
    return bwd_ws(a, kKDA);
}

size_t gcl_bwd_workspace_bytes(const gcl_bwd_args *a) {
    if (!a) return 0;
    return bwd_ws(a, kGDN);
}

gcl_status_t gdn_chunk_bwd(const gcl_bwd_args *a, gcl_stream_t stream) { return run_bwd(a, stream, kGDN); }
gcl_status_t kda_chunk_bwd(const gcl_bwd_args *a, gcl_stream_t stream) { return run_bwd(a, stream, kKDA); }


// ---------------------------------------------------------------- causal_conv1d
static gcl_status_t conv_check(const char *fn, const gcl_conv_args *a, bool backward) {
    if (!a) return fail(GCL_ERR_INVALID_ARG, "%s: args is NULL", fn);
    if (!a->x || !a->weight || !a->cu_seqlens || !a->chunk_indices)
        return fail(GCL_ERR_INVALID_ARG, "%s: x, weight, cu_seqlens and chunk_indices are required", fn);
    if (!backward && !a->y) return fail(GCL_ERR_INVALID_ARG, "%s: y is required", fn);
    if (backward && (!a->dy || !a->dx || !a->dweight))
        return fail(GCL_ERR_INVALID_ARG, "%s: dy, dx and dweight are required", fn);
    if (a->t_max < 1 || a->t_max >= (int64_t(1) << 31) || a->n_max < 1)
        return fail(GCL_ERR_INVALID_ARG, "%s: need 1 <= t_max < 2^31 and n_max >= 1", fn);
    if (a->bt != kChunk)
        return fail(GCL_ERR_UNSUPPORTED, "%s: chunk size bt=%d (implemented: 64)", fn, a->bt);
    if (a->W < 2 || a->W > 4)
        return fail(GCL_ERR_UNSUPPORTED, "%s: W=%d taps (supported: 2, 3, 4)", fn, a->W);
    if (a->D < 8 || a->D % 8 != 0)
        return fail(GCL_ERR_UNSUPPORTED, "%s: D=%d channels (a positive multiple of 8)", fn, a->D);
    if (a->dtype != GCL_F32 && a->dtype != GCL_BF16)
        return fail(GCL_ERR_UNSUPPORTED, "%s: dtype %d (supported: GCL_F32, GCL_BF16)", fn, a->dtype);
    if (a->activation != GCL_ACT_NONE && a->activation != GCL_ACT_SILU)
        return fail(GCL_ERR_UNSUPPORTED, "%s: activation %d (supported: none, SiLU)", fn, a->activation);
    if (!aligned16(a->x) || (a->y && !aligned16(a->y)) || (a->residual && !aligned16(a->residual)) ||
        (a->dy && !aligned16(a->dy)) || (a->dx && !aligned16(a->dx)) ||
        (backward && a->workspace && !aligned16(a->workspace)))
        return fail(GCL_ERR_INVALID_ARG, "%s: x, y, residual, dy, dx and the workspace must be 16-byte aligned", fn);
    return GCL_OK;
}

static ConvLaunch conv_launch(const gcl_conv_args *a) {
    ConvLaunch c{};
    c.x = a->x; c.w = a->weight; c.bias = a->bias; c.residual = a->residual; c.h0 = a->h0;
    c.dy = a->dy; c.y = a->y; c.ht = a->ht; c.dht = a->dht;
    c.dx = a->dx; c.dw = a->dweight; c.dbias = a->dbias; c.dh0 = a->dh0;
    c.partial = static_cast<float *>(a->workspace);
    c.cu_seqlens = a->cu_seqlens; c.chunk_indices = a->chunk_indices; c.dev_status = a->dev_status;
    c.t_max = a->t_max; c.nt_max = gcl_nt_max(a->t_max, a->n_max, a->bt); c.n_max = a->n_max;
    c.D = a->D; c.W = a->W; c.activation = a->activation; c.dtype = a->dtype;
    return c;
}

gcl_status_t causal_conv1d_fwd(const gcl_conv_args *a, gcl_stream_t stream) {
    g_err[0] = 0;
    const char *fn = "causal_conv1d_fwd";
    gcl_status_t st = conv_check(fn, a, false);
    if (st != GCL_OK) return st;
    return cuda_check(launch_conv_fwd(conv_launch(a), static_cast<cudaStream_t>(stream)), fn);
}

size_t gcl_causal_conv1d_bwd_workspace_bytes(const gcl_conv_args *a) {
    if (!a || a->D <= 0 || a->W < 2 || a->W > 4 || a->n_max < 1 || a->t_max < 1 || a->bt < 1) return 0;
    return conv_bwd_workspace_bytes(gcl_nt_max(a->t_max, a->n_max, a->bt), a->D, a->W);
}

gcl_status_t causal_conv1d_bwd(const gcl_conv_args *a, gcl_stream_t stream) {
    g_err[0] = 0;
    const char *fn = "causal_conv1d_bwd";
    gcl_status_t st = conv_check(fn, a, true);
    if (st != GCL_OK) return st;
    const size_t need = gcl_causal_conv1d_bwd_workspace_bytes(a);
    if (!a->workspace || a->workspace_bytes < need)
        return fail(GCL_ERR_CAPACITY, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    return cuda_check(launch_conv_bwd(conv_launch(a), static_cast<cudaStream_t>(stream)), fn);
}

}  // extern "C"
