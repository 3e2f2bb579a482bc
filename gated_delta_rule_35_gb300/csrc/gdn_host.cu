// gdn_chunk_fwd_host (include/gdn.h): the forward from and to host memory.
// The sequence is cut into spans of T (multiples of 64 tokens, every batch row
// and head at once); span i's host-to-device copies run on stream a while span
// i - 1's kernels and device-to-host copies run on stream b, and each span
// starts from the previous span's final state. The kernels are gdn_chunk_fwd's;
// this file only places copies and launches.
#include <algorithm>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kMaxSpans = 16;

struct HostPlan {
    int spans, span_t;        // number of spans, tokens per span (last one may be short)
    size_t tok_q, tok_v, tok_g, tok_b;   // bytes per token (all heads) of q/k, v/o, g, beta
    size_t h_bytes;           // one state [B, H, K, V] fp32
    size_t ws_bytes;          // one span's workspace
    size_t off_q, off_k, off_v, off_g, off_b, off_o, off_h0, off_h1, off_h2, off_ws, off_st, total;
};

// Spans picked for pieces == 0: the last span's kernels and output copy are
// not overlapped by any input copy, so they shrink with more spans, while every
// span adds fixed per-copy and per-launch costs. Measured on GB300 (host link
// about 210 GB/s in, 190 GB/s out): 102 MB of inputs ran best with 3 to 5
// spans, 816 MB with 16.
constexpr size_t kAutoSpanBytes = size_t{32} << 20;
constexpr int kAutoMinSpans = 3;

bool make_plan(const gdn_problem *p, int pieces, HostPlan *pl) {
    if (!p || pieces < 0 || pieces > kMaxSpans) return false;
    if (gdn_chunk_fwd_workspace_bytes(p) == 0) return false;   // validates the problem
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t gk = (p->flags & GDN_FLAG_PER_CHANNEL_DECAY) ? p->K : 1;
    pl->tok_q = static_cast<size_t>(p->H) * p->K * es;
    pl->tok_v = static_cast<size_t>(p->H) * p->V * es;
    pl->tok_g = static_cast<size_t>(p->H) * gk * sizeof(float);
    pl->tok_b = static_cast<size_t>(p->H) * sizeof(float);
    if (pieces == 0) {
        const size_t in = static_cast<size_t>(p->B) * p->T *
                          (2 * pl->tok_q + pl->tok_v + pl->tok_g + pl->tok_b);
        const size_t n = (in + kAutoSpanBytes / 2) / kAutoSpanBytes;
        pieces = static_cast<int>(std::min<size_t>(kMaxSpans, std::max<size_t>(kAutoMinSpans, n)));
    }
    pl->h_bytes = static_cast<size_t>(p->B) * p->H * p->K * p->V * sizeof(float);
    const int chunks = static_cast<int>(num_chunks(p->T));
    const int n = std::max(1, std::min(pieces, chunks));
    pl->span_t = std::max(1, (chunks + n - 1) / n) * kChunk;
    pl->spans = p->T == 0 ? 1 : static_cast<int>((p->T + pl->span_t - 1) / pl->span_t);
    gdn_problem span = *p;
    span.T = std::min(p->T, pl->span_t);
    pl->ws_bytes = align_up(gdn_chunk_fwd_workspace_bytes(&span));
    const size_t tokens = static_cast<size_t>(p->B) * p->T;
    size_t at = 0;
    auto take = [&](size_t bytes) { const size_t o = at; at += align_up(bytes); return o; };
    pl->off_q = take(tokens * pl->tok_q);
    pl->off_k = take(tokens * pl->tok_q);
    pl->off_v = take(tokens * pl->tok_v);
    pl->off_g = take(tokens * pl->tok_g);
    pl->off_b = take(tokens * pl->tok_b);
    pl->off_o = take(tokens * pl->tok_v);
    pl->off_h0 = take(pl->h_bytes);
    pl->off_h1 = take(pl->h_bytes);
    pl->off_h2 = take(pl->h_bytes);
    pl->off_ws = take(pl->ws_bytes);
    pl->off_st = take(kMaxSpans * sizeof(uint32_t));   // each span's device status word
    pl->total = at;
    return true;
}

// Rows b = 0..B-1 of a [B, T, ...] host tensor, tokens [t0, t0 + nt), into a
// contiguous [B, nt, ...] device block (or back).
cudaError_t copy_span(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
    if (!width || !rows) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

}  // namespace
}  // namespace gdn

extern "C" {

GDN_API size_t gdn_chunk_fwd_host_bytes(const gdn_problem *p, int32_t pieces) {
    gdn::HostPlan pl;
    return gdn::make_plan(p, pieces, &pl) ? pl.total : 0;
}

GDN_API gdn_status gdn_chunk_fwd_host(const gdn_problem *p, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta,
                                      float scale, const float *h0, void *o, float *h_final,
                                      void *device_buffer, size_t device_bytes, int32_t pieces,
                                      void *stream_a, void *stream_b) {
    gdn::HostPlan pl;
    if (!gdn::make_plan(p, pieces, &pl)) return GDN_ERR_INVALID_ARG;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if (!stream_a || !stream_b || stream_a == stream_b) return GDN_ERR_INVALID_ARG;
    if (!device_buffer || device_bytes < pl.total) return GDN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(device_buffer) & 255u) return GDN_ERR_ALIGNMENT;
    char *dev = static_cast<char *>(device_buffer);
    const cudaStream_t sa = static_cast<cudaStream_t>(stream_a);
    const cudaStream_t sb = static_cast<cudaStream_t>(stream_b);
    const size_t B = static_cast<size_t>(p->B), T = static_cast<size_t>(p->T);
    const struct { const void *host; size_t off, tok; } in[] = {
        {q, pl.off_q, pl.tok_q}, {k, pl.off_k, pl.tok_q}, {v, pl.off_v, pl.tok_v},
        {g, pl.off_g, pl.tok_g}, {beta, pl.off_b, pl.tok_b}};

    cudaEvent_t landed[gdn::kMaxSpans] = {};
    int made = 0;
    cudaError_t e = cudaSuccess;
    gdn_status st = GDN_OK;
    for (; made < pl.spans && e == cudaSuccess; ++made)
        e = cudaEventCreateWithFlags(&landed[made], cudaEventDisableTiming);
    float *state = nullptr;
    if (e == cudaSuccess && h0) {
        state = reinterpret_cast<float *>(dev + pl.off_h0);
        e = cudaMemcpyAsync(state, h0, pl.h_bytes, cudaMemcpyHostToDevice, sa);
    }
    // every span's inputs on stream a, in order, each followed by its event
    for (int i = 0; i < pl.spans && e == cudaSuccess; ++i) {
        const size_t t0 = static_cast<size_t>(i) * pl.span_t;
        const size_t nt = std::min<size_t>(pl.span_t, T - std::min(T, t0));
        for (const auto &a : in) {
            if (e != cudaSuccess) break;
            e = gdn::copy_span(dev + a.off + B * t0 * a.tok, nt * a.tok,
                               static_cast<const char *>(a.host) + t0 * a.tok, T * a.tok,
                               nt * a.tok, B, cudaMemcpyHostToDevice, sa);
        }
        if (e == cudaSuccess) e = cudaEventRecord(landed[i], sa);
    }
    // kernels and outputs on stream b; the state alternates between two buffers
    for (int i = 0; i < pl.spans && e == cudaSuccess && st == GDN_OK; ++i) {
        const size_t t0 = static_cast<size_t>(i) * pl.span_t;
        const size_t nt = std::min<size_t>(pl.span_t, T - std::min(T, t0));
        e = cudaStreamWaitEvent(sb, landed[i], 0);
        if (e != cudaSuccess) break;
        float *next = reinterpret_cast<float *>(dev + ((i & 1) ? pl.off_h2 : pl.off_h1));
        gdn_problem sp = *p;
        sp.T = static_cast<int>(nt);
        st = gdn_chunk_fwd(&sp, dev + pl.off_q + B * t0 * pl.tok_q,
                           dev + pl.off_k + B * t0 * pl.tok_q, dev + pl.off_v + B * t0 * pl.tok_v,
                           reinterpret_cast<const float *>(dev + pl.off_g + B * t0 * pl.tok_g),
                           reinterpret_cast<const float *>(dev + pl.off_b + B * t0 * pl.tok_b),
                           scale, state, dev + pl.off_o + B * t0 * pl.tok_v, next, dev + pl.off_ws,
                           pl.ws_bytes, sb);
        if (st != GDN_OK) break;
        // the span's status word (the next span's call clears it) is kept aside
        e = cudaMemcpyAsync(dev + pl.off_st + i * sizeof(uint32_t), dev + pl.off_ws, sizeof(uint32_t),
                            cudaMemcpyDeviceToDevice, sb);
        if (e != cudaSuccess) break;
        e = gdn::copy_span(static_cast<char *>(o) + t0 * pl.tok_v, T * pl.tok_v,
                           dev + pl.off_o + B * t0 * pl.tok_v, nt * pl.tok_v, nt * pl.tok_v, B,
                           cudaMemcpyDeviceToHost, sb);
        state = next;
    }
    if (e == cudaSuccess && st == GDN_OK && h_final)
        e = cudaMemcpyAsync(h_final, state, pl.h_bytes, cudaMemcpyDeviceToHost, sb);
    const cudaError_t ea = cudaStreamSynchronize(sa), eb = cudaStreamSynchronize(sb);
    for (int i = 0; i < made; ++i) cudaEventDestroy(landed[i]);
    if (st != GDN_OK) return st;
    if (e != cudaSuccess || ea != cudaSuccess || eb != cudaSuccess) return GDN_ERR_CUDA;
    // a span whose bounded device wait gave up has garbage outputs: report it
    uint32_t words[gdn::kMaxSpans] = {};
    if (p->T > 0) {
        if (cudaMemcpyAsync(words, dev + pl.off_st, pl.spans * sizeof(uint32_t),
                            cudaMemcpyDeviceToHost, sb) != cudaSuccess ||
            cudaStreamSynchronize(sb) != cudaSuccess)
            return GDN_ERR_CUDA;
        for (int i = 0; i < pl.spans; ++i)
            if (words[i]) return GDN_ERR_DEVICE_TIMEOUT;
    }
    return GDN_OK;
}

}  // extern "C"
