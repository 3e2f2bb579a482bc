// Host side of the C ABI declared in include/gdn.h: argument validation,
// workspace carving, algorithm choice and the launch sequence.
#include <atomic>
#include <cstring>

#include "gdn_internal.h"

namespace gdn {

namespace {
std::atomic<uint64_t> g_armed_stall{0};
}  // namespace

uint64_t take_armed_stall() { return g_armed_stall.exchange(0); }

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_problem(const gdn_problem *p) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->B <= 0 || p->H <= 0 || p->T < 0 || p->K <= 0 || p->V <= 0) return GDN_ERR_INVALID_ARG;
    if (p->dtype != GDN_F32 && p->dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (p->algo != GDN_ALGO_AUTO && p->algo != GDN_ALGO_SIMT && p->algo != GDN_ALGO_TC &&
        p->algo != GDN_ALGO_TC_SINGLE && p->algo != GDN_ALGO_TC_WIDE)
        return GDN_ERR_INVALID_ARG;
    if (p->flags & ~kKnownFlags) return GDN_ERR_INVALID_ARG;
    const bool tc = p->algo == GDN_ALGO_TC || p->algo == GDN_ALGO_TC_SINGLE || p->algo == GDN_ALGO_TC_WIDE;
    // per-channel decay: the CUDA-core pipeline or the two-kernel tensor-core form
    if ((p->flags & GDN_FLAG_PER_CHANNEL_DECAY) && tc && p->algo != GDN_ALGO_TC)
        return GDN_ERR_UNSUPPORTED;
    if (p->K != 64 && p->K != 128) return GDN_ERR_UNSUPPORTED;
    if (p->V % 64 != 0 || p->V > 256) return GDN_ERR_UNSUPPORTED;
    // Every index is computed in 64 bits; B*T*H rows must still fit a grid.
    if (num_chunks(p->T) > 65535 * 64LL) return GDN_ERR_UNSUPPORTED;
    if (p->H > 65535 || p->B > 65535) return GDN_ERR_UNSUPPORTED;
    if (tc && !tc_supported(p->K, p->V, static_cast<gdn_dtype>(p->dtype)))
        return GDN_ERR_UNSUPPORTED;
    if (p->algo == GDN_ALGO_TC_WIDE && p->V % 128 != 0) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

TcForm tc_form(gdn_algo algo) {
    return algo == GDN_ALGO_TC_SINGLE ? TcForm::kSingle : algo == GDN_ALGO_TC_WIDE ? TcForm::kWide : TcForm::kTwo;
}

gdn_algo resolve_algo(const gdn_problem *p) {
    if (p->algo != GDN_ALGO_AUTO) return static_cast<gdn_algo>(p->algo);
    return tc_supported(p->K, p->V, static_cast<gdn_dtype>(p->dtype)) ? GDN_ALGO_TC
                                                                       : GDN_ALGO_SIMT;
}

bool per_channel(const gdn_problem *p) { return p->flags & GDN_FLAG_PER_CHANNEL_DECAY; }

// Front-end region: g_cum (one fp32 per token-head, or per token-head-channel
// with per-channel decay) and rk (one per token-head).
size_t g_cum_bytes(const gdn_problem *p) {
    const size_t per = (p->flags & GDN_FLAG_PER_CHANNEL_DECAY) ? p->K : 1;
    return align_up(static_cast<size_t>(p->B) * p->T * p->H * per * sizeof(float));
}
size_t front_bytes(const gdn_problem *p) {
    return g_cum_bytes(p) + align_up(static_cast<size_t>(p->B) * p->T * p->H * sizeof(float));
}

size_t body_bytes(const gdn_problem *p, gdn_algo algo) {
    if (p->T == 0) return 0;
    const size_t front = front_bytes(p);
    if (algo == GDN_ALGO_TC && per_channel(p)) {
        // with 'auto' also room for the CUDA-core pipeline, which serves a call
        // asking for the stage exports (the per-channel tensor-core form has
        // only A diag(beta))
        const size_t kda = kda_tc_workspace_bytes(p->B, p->T, p->H, p->K, p->V);
        const size_t simt = simt_workspace_bytes(p->B, p->T, p->H, p->K, p->V);
        return front + ((p->algo == GDN_ALGO_AUTO && simt > kda) ? simt : kda);
    }
    if (algo == GDN_ALGO_TC || algo == GDN_ALGO_TC_WIDE)
        return front + tc_workspace_bytes(p->B, p->T, p->H, p->K, p->V);
    if (algo == GDN_ALGO_TC_SINGLE) return front;   // A stays in the kernel
    return front + simt_workspace_bytes(p->B, p->T, p->H, p->K, p->V);
}

gdn_status run(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g,
               const float *beta, float scale, const float *h0, void *o, float *h_final,
               void *workspace, size_t workspace_bytes, const gdn_stage_exports *ex,
               const Marks &marks, cudaStream_t stream, const gdn_output_norm *norm = nullptr) {
    gdn_status st = check_problem(p);
    if (st != GDN_OK) return st;
    const bool empty = p->T == 0;
    if (!empty && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if (norm && (!norm->gate || !norm->weight || !(norm->eps >= 0.f))) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, beta, h0, o, h_final, workspace,
                          norm ? norm->gate : nullptr, norm ? norm->weight : nullptr};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return GDN_ERR_ALIGNMENT;
    gdn_algo algo = resolve_algo(p);
    const bool kda_tc = algo == GDN_ALGO_TC && per_channel(p);
    // the per-channel tensor-core form exports only A diag(beta); with 'auto'
    // a call asking for more runs on the CUDA-core pipeline, for which
    // workspace_bytes reserved room
    const bool simt_only = ex && (ex->A || ex->w || ex->u || ex->v_new || ex->h);
    if (kda_tc && simt_only) {
        if (p->algo != GDN_ALGO_AUTO) return GDN_ERR_UNSUPPORTED;
        algo = GDN_ALGO_SIMT;
    }
    if (ex && (algo == GDN_ALGO_TC || algo == GDN_ALGO_TC_WIDE) &&
        (ex->A || ex->w || ex->u || ex->v_new || ex->h))
        return GDN_ERR_UNSUPPORTED;
    // the single-kernel form keeps A on chip and has no output stage
    if (algo == GDN_ALGO_TC_SINGLE && (ex || norm)) return GDN_ERR_UNSUPPORTED;
    if (ex && algo == GDN_ALGO_SIMT && ex->A_beta) return GDN_ERR_UNSUPPORTED;
    const size_t need = kStatusBytes + body_bytes(p, resolve_algo(p));
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;

    Args a;
    a.B = p->B; a.T = p->T; a.H = p->H; a.K = p->K; a.V = p->V;
    a.NT = static_cast<int>(num_chunks(p->T));
    a.T_pad = a.NT * kChunk;
    a.dtype = static_cast<gdn_dtype>(p->dtype);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale; a.h0 = h0;
    a.o = o; a.h_final = h_final;
    a.status = static_cast<uint32_t *>(workspace);
    a.flags = p->flags;
    if (norm) {
        a.gate = norm->gate;
        a.norm_w = norm->weight;
        a.norm_eps = norm->eps;
    }
    char *front = static_cast<char *>(workspace) + kStatusBytes;
    a.g_cum = reinterpret_cast<float *>(front);
    a.rk = reinterpret_cast<float *>(front + g_cum_bytes(p));
    void *body = empty ? front : front + front_bytes(p);

    // the status word starts clear on every path; only bounded waits that
    // give up set it
    cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    if (empty) {
        e = marks.mark(0, stream);
        if (e == cudaSuccess) e = copy_state(a, stream);
        if (e == cudaSuccess) e = marks.mark(1, stream);
    } else if (algo == GDN_ALGO_TC && per_channel(p)) {
        e = kda_tc_forward(a, body, stream, marks);
        if (e == cudaSuccess && ex && ex->A_beta) e = tc_export_abeta(a, body, ex->A_beta, stream);
    } else if (algo == GDN_ALGO_TC || algo == GDN_ALGO_TC_SINGLE || algo == GDN_ALGO_TC_WIDE) {
        e = tc_forward(a, body, stream, marks, tc_form(algo));
        if (e == cudaSuccess && ex && ex->A_beta) e = tc_export_abeta(a, body, ex->A_beta, stream);
    } else {
        const SimtWorkspace ws = simt_carve(body, a.B, a.T, a.H, a.K, a.V);
        e = simt_forward(a, ws, stream, marks);
        if (e == cudaSuccess && ex) {
            const size_t rows = static_cast<size_t>(a.B) * a.T_pad * a.H;
            struct { float *dst; const float *src; size_t n; } cp[] = {
                {ex->A, ws.A, rows * kChunk},
                {ex->w, ws.w, rows * a.K},
                {ex->u, ws.u, rows * a.V},
                {ex->v_new, ws.v_new, rows * a.V},
                {ex->h, ws.h, static_cast<size_t>(a.B) * a.NT * a.H * a.K * a.V},
            };
            for (auto &c : cp)
                if (c.dst && e == cudaSuccess)
                    e = cudaMemcpyAsync(c.dst, c.src, c.n * sizeof(float), cudaMemcpyDeviceToDevice,
                                        stream);
        }
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Kernels of one call.
int launches(const gdn_problem *p, const char **names, int max_names) {
    if (check_problem(p) != GDN_OK) return 0;
    if (p->T == 0) {
        if (names && max_names > 0) names[0] = kCopyStateName;
        return 1;
    }
    const gdn_algo algo = resolve_algo(p);
    if (algo == GDN_ALGO_TC && per_channel(p)) {
        for (int i = 0; names && i < kKdaTcLaunches && i < max_names; ++i) names[i] = kKdaTcKernelNames[i];
        return kKdaTcLaunches;
    }
    if (algo == GDN_ALGO_TC || algo == GDN_ALGO_TC_SINGLE || algo == GDN_ALGO_TC_WIDE)
        return tc_launches(tc_form(algo), p->B, p->H, p->V, names, max_names);
    for (int i = 0; names && i < kSimtLaunches && i < max_names; ++i) names[i] = kSimtKernelNames[i];
    return kSimtLaunches;
}

}  // namespace
}  // namespace gdn

extern "C" {

GDN_API size_t gdn_chunk_fwd_workspace_bytes(const gdn_problem *p) {
    if (gdn::check_problem(p) != GDN_OK) return 0;
    return gdn::kStatusBytes + gdn::body_bytes(p, gdn::resolve_algo(p));
}

GDN_API gdn_status gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float scale, const float *h0,
                                 void *o, float *h_final, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    return gdn::run(p, q, k, v, g, beta, scale, h0, o, h_final, workspace, workspace_bytes,
                    nullptr, gdn::Marks{}, static_cast<cudaStream_t>(stream));
}

GDN_API int32_t gdn_chunk_fwd_launches(const gdn_problem *p, const char **names,
                                       int32_t max_names) {
    return gdn::launches(p, names, max_names);
}

GDN_API gdn_status gdn_chunk_fwd_profiled(const gdn_problem *p, const void *q, const void *k,
                                          const void *v, const float *g, const float *beta,
                                          float scale, const float *h0, void *o, float *h_final,
                                          void *workspace, size_t workspace_bytes,
                                          void *const *events, int32_t n_events, void *stream) {
    const int n = gdn::launches(p, nullptr, 0);
    if (n == 0) return GDN_ERR_INVALID_ARG;
    if (!events || n_events < n + 1) return GDN_ERR_INVALID_ARG;
    gdn::Marks m;
    m.ev = reinterpret_cast<cudaEvent_t const *>(events);
    m.n = n_events;
    return gdn::run(p, q, k, v, g, beta, scale, h0, o, h_final, workspace, workspace_bytes,
                    nullptr, m, static_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_chunk_fwd_ex(const gdn_problem *p, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta, float scale,
                                    const float *h0, const gdn_output_norm *norm, void *o,
                                    float *h_final, void *workspace, size_t workspace_bytes,
                                    void *const *events, int32_t n_events, void *stream) {
    gdn::Marks m;
    if (events) {
        const int n = gdn::launches(p, nullptr, 0);
        if (n == 0 || n_events < n + 1) return GDN_ERR_INVALID_ARG;
        m.ev = reinterpret_cast<cudaEvent_t const *>(events);
        m.n = n_events;
    }
    return gdn::run(p, q, k, v, g, beta, scale, h0, o, h_final, workspace, workspace_bytes,
                    nullptr, m, static_cast<cudaStream_t>(stream), norm);
}

GDN_API gdn_status gdn_chunk_fwd_stages(const gdn_problem *p, const void *q, const void *k,
                                        const void *v, const float *g, const float *beta,
                                        float scale, const float *h0, void *o, float *h_final,
                                        void *workspace, size_t workspace_bytes,
                                        const gdn_stage_exports *ex, void *stream) {
    if (!ex) return GDN_ERR_INVALID_ARG;
    return gdn::run(p, q, k, v, g, beta, scale, h0, o, h_final, workspace, workspace_bytes, ex,
                    gdn::Marks{}, static_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_check_device_status(void *workspace, void *stream) {
    if (!workspace) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    if (word == 0) return GDN_OK;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_ERR_DEVICE_TIMEOUT;
}

GDN_API void gdn_debug_arm_stall(uint64_t wait_ns) {
    gdn::g_armed_stall.store(wait_ns == 0 ? 1 : wait_ns);
}

GDN_API const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported shape, dtype or algorithm";
        case GDN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

GDN_API uint32_t gdn_version(void) { return (0u << 16) | (1u << 8) | 0u; }

}  // extern "C"
