// Recurrent (decode) step of the gated delta rule: gdn_decode_step of include/gdn.h.
//
// Per token (the row update of the "KdaSplit" decode kernel page, `update`,
// with Gated DeltaNet's scalar decay alpha = exp(gamma)):
//   S <- alpha S;  delta = beta (v - S^T k);  S += k delta^T;  o = scale S^T q.
// Column j of S [K, V] evolves on its own: delta[j] needs only column j of S
// (through (S^T k)[j]) and v[j]. So the work splits over (b, h, slice of VS
// columns) with no exchange between CTAs (the page instead splits the state's
// rows over a cluster and reduces across it). A CTA holds its [K, VS] slice in
// registers for all of the call's tokens: the state is read once and written
// once per call, which is the whole HBM cost at decode batch sizes.
//
// o is formed from the pre-update reads: S'^T q = alpha S^T q + delta (k . q),
// so one pass over the state per token gives both S^T k and S^T q.
//
// With the front-end norm (GDN_FLAG_QK_L2NORM) the same pass also sums |k|^2
// and |q|^2; with rk, rq their factors 1 / sqrt(sum + eps), the normalised
// rows enter as S^T k^ = rk S^T k, k^ . q^ = rk rq (k . q) and
// S += k (rk delta)^T, so the rows themselves are never rescaled.
//
// With the output stage (gated RMSNorm over V) one CTA holds a head's whole
// state (VS = V), so the row's mean square is a sum inside the CTA.
//
// With per-channel decay (GDN_FLAG_PER_CHANNEL_DECAY, gamma [B,T,H,K]) row i
// of S decays by exp(gamma[i]); each thread scales its rows before the pass,
// so the reads below always see the decayed state.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kRows = 8;   // state rows per thread
constexpr int kCols = 4;   // state columns per thread (one float4)
constexpr const char *kDecodeName = "gdn_decode_step_kernel";

__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32.
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ float load1(const float *p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store1(float *p, float x) { *p = x; }
__device__ __forceinline__ void store1(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <typename E>
struct DecodeParams {
    const E *q, *k, *v;
    const float *gamma, *beta;
    float scale;
    const float *state_in;
    float *state_out;
    E *o;
    int T, H, V;
    int l2norm;               // GDN_FLAG_QK_L2NORM
    int per_channel;          // GDN_FLAG_PER_CHANNEL_DECAY
    const E *gate;            // output stage, or nullptr
    const float *norm_w;
    float norm_eps;
};

// Thread (cg, rg) owns rows rg*8 .. rg*8+7 and columns cg*4 .. cg*4+3 of the
// CTA's slice, cg = tid % (VS/4). With VS <= 128 a warp covers 32/(VS/4) whole
// rows of the slice (VS*4 contiguous bytes each) and sums its row groups with
// shuffles; with VS = 256 a row group spans two warps. Either way each
// (slot, column) of the partial-sum buffers has exactly one writer.
// Threads of a CTA, and CTAs per SM asked of the compiler: 1024 threads per SM
// at 64 registers each keeps 128 KB of state loads in flight on every SM (768
// threads at up to 85 registers for the per-channel mode's extra factors).
constexpr int decode_threads(int K, int VS) { return K * VS / (kRows * kCols); }
constexpr int decode_min_blocks(int K, int VS, int threads_per_sm = 1024) {
    return decode_threads(K, VS) >= threads_per_sm ? 1 : threads_per_sm / decode_threads(K, VS);
}

// MODE 0 (plain): no front-end norm, per-channel decay or output stage, all
// compiled out; MODE 1: per-channel decay only; MODE 2: every option as a
// runtime switch (more registers, fewer CTAs per SM).
template <typename E, int K, int VS, int MODE>
__global__ void __launch_bounds__(decode_threads(K, VS),
                                  MODE == 0 ? decode_min_blocks(K, VS)
                                            : MODE == 1 ? decode_min_blocks(K, VS, 768) : 1)
gdn_decode_step_kernel(const DecodeParams<E> p) {
    constexpr bool PLAIN = MODE == 0;
    constexpr int CG = VS / kCols;                    // column groups
    constexpr int NT = CG * (K / kRows);              // threads
    constexpr int NW = NT / 32;                       // warps
    constexpr int WPR = CG > 32 ? CG / 32 : 1;        // warps per row group
    constexpr int NS = NW / WPR;                      // partial-sum slots
    constexpr int CW = CG < 32 ? CG : 32;             // column groups per warp
    static_assert(NT % 32 == 0 && NT <= 1024, "thread layout");
    __shared__ float red_k[NS][VS], red_q[NS][VS], red_kq[NS], red_kk[NS], red_qq[NS];
    __shared__ float red_o[(VS + 31) / 32];
    __shared__ __align__(16) float delta_s[VS];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % CG, rg = tid / CG;
    const int slot = warp / WPR;
    const int h = blockIdx.y, b = blockIdx.z;
    const int V = p.V, H = p.H, T = p.T;
    const int col0 = blockIdx.x * VS;
    const size_t bh = static_cast<size_t>(b) * H + h;
    const size_t s_off = (bh * K + rg * kRows) * V + col0 + cg * kCols;
    const bool norm = MODE == 2 && p.l2norm != 0, gated = MODE == 2 && p.gate != nullptr;
    const bool per_channel = MODE == 1 || (MODE == 2 && p.per_channel != 0);

    float S[kRows][kCols];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        const float4 x = *reinterpret_cast<const float4 *>(p.state_in + s_off + size_t(i) * V);
        S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
    }

#pragma unroll 1
    for (int t = 0; t < T; ++t) {
        const size_t row = (static_cast<size_t>(b) * T + t) * H + h;   // token-head row
        float kk[kRows], qq[kRows];
        load8(p.k + row * K + rg * kRows, kk);
        load8(p.q + row * K + rg * kRows, qq);
        // The decay: a scalar alpha (mode 0) or one factor per row (mode 1,
        // ar[i]) enters the sums and the update as a factor; mode 2 decays the
        // rows first, S <- diag(alpha) S, and alpha below is 1.
        float alpha = 1.f;
        float ar[kRows];
        if (PLAIN) {
            alpha = expf(p.gamma[row]);
        } else if (MODE == 1) {
            load8(p.gamma + row * K + rg * kRows, ar);
#pragma unroll
            for (int i = 0; i < kRows; ++i) ar[i] = expf(ar[i]);
        } else if (per_channel) {
            float ga[kRows];
            load8(p.gamma + row * K + rg * kRows, ga);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const float a = expf(ga[i]);
#pragma unroll
                for (int c = 0; c < kCols; ++c) S[i][c] *= a;
            }
        } else {
            const float a = expf(p.gamma[row]);
#pragma unroll
            for (int i = 0; i < kRows; ++i)
#pragma unroll
                for (int c = 0; c < kCols; ++c) S[i][c] *= a;
        }

        // Partial S^T k, S^T q over this thread's rows, k . q (and |k|^2, |q|^2).
        float pk[kCols], pq[kCols], kq = 0.f, k2 = 0.f, q2 = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c) pk[c] = pq[c] = 0.f;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            kq = fmaf(kk[i], qq[i], kq);
            if (MODE == 2) {
                k2 = fmaf(kk[i], kk[i], k2);
                q2 = fmaf(qq[i], qq[i], q2);
            }
            const float ki = MODE == 1 ? ar[i] * kk[i] : kk[i];
            const float qi = MODE == 1 ? ar[i] * qq[i] : qq[i];
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                pk[c] = fmaf(S[i][c], ki, pk[c]);
                pq[c] = fmaf(S[i][c], qi, pq[c]);
            }
        }
        // Sum over the row groups of the warp (lanes that share cg).
#pragma unroll
        for (int off = CW; off < 32; off <<= 1) {
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], off);
                pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], off);
            }
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (MODE == 2) {
                k2 += __shfl_xor_sync(0xffffffffu, k2, off);
                q2 += __shfl_xor_sync(0xffffffffu, q2, off);
            }
        }
        if (lane < CW) {
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                red_k[slot][cg * kCols + c] = pk[c];
                red_q[slot][cg * kCols + c] = pq[c];
            }
        }
        if (lane == 0 && warp % WPR == 0) {
            red_kq[slot] = kq;
            red_kk[slot] = k2;
            red_qq[slot] = q2;
        }
        __syncthreads();

        // One thread per column: delta and o.
        float o_val = 0.f;
        if (tid < VS) {
            float dk = 0.f, dq = 0.f, kqs = 0.f, kks = 0.f, qqs = 0.f;
#pragma unroll
            for (int w = 0; w < NS; ++w) {
                dk += red_k[w][tid];
                dq += red_q[w][tid];
                kqs += red_kq[w];
                kks += red_kk[w];
                qqs += red_qq[w];
            }
            const size_t vo = row * V + col0 + tid;
            const float rk = norm ? rsqrtf(kks + kL2NormEps) : 1.f;
            const float rq = norm ? rsqrtf(qqs + kL2NormEps) : 1.f;
            const float d = p.beta[row] * (load1(p.v + vo) - alpha * rk * dk);
            delta_s[tid] = rk * d;
            o_val = p.scale * rq * fmaf(d, rk * kqs, alpha * dq);
            if (!gated) store1(p.o + vo, o_val);
        }
        if (gated && warp < (VS + 31) / 32) {
            // the row's sum of squares over the CTA's V = VS columns
            float o2 = o_val * o_val;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) o2 += __shfl_xor_sync(0xffffffffu, o2, off);
            if (lane == 0) red_o[warp] = o2;
        }
        __syncthreads();
        if (gated && tid < VS) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < (VS + 31) / 32; ++w) ss += red_o[w];
            const size_t vo = row * V + col0 + tid;
            const float z = load1(p.gate + vo);
            const float sg = 1.f / (1.f + expf(-z));
            store1(p.o + vo, o_val * rsqrtf(ss / VS + p.norm_eps) * p.norm_w[tid] * sg);
        }

        // S = alpha S + k (rk delta)^T on this thread's block.
        const float4 d4 = *reinterpret_cast<const float4 *>(&delta_s[cg * kCols]);
        const float dd[kCols] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int i = 0; i < kRows; ++i)
#pragma unroll
            for (int c = 0; c < kCols; ++c)
                S[i][c] = fmaf(kk[i], dd[c],
                               PLAIN ? alpha * S[i][c] : MODE == 1 ? ar[i] * S[i][c] : S[i][c]);
        // The next token's writes to red_* and delta_s follow this token's
        // second barrier and its own first barrier, after every read above.
    }

#pragma unroll
    for (int i = 0; i < kRows; ++i)
        *reinterpret_cast<float4 *>(p.state_out + s_off + size_t(i) * V) =
            make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_decode(const gdn_problem *p, const gdn_output_norm *norm) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->B <= 0 || p->H <= 0 || p->T < 0 || p->K <= 0 || p->V <= 0) return GDN_ERR_INVALID_ARG;
    if (p->dtype != GDN_F32 && p->dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (p->algo != GDN_ALGO_AUTO && p->algo != GDN_ALGO_SIMT && p->algo != GDN_ALGO_TC &&
        p->algo != GDN_ALGO_TC_SINGLE && p->algo != GDN_ALGO_TC_WIDE)
        return GDN_ERR_INVALID_ARG;
    if (p->flags & ~kKnownFlags) return GDN_ERR_INVALID_ARG;
    if (norm && (!norm->gate || !norm->weight || !(norm->eps >= 0.f))) return GDN_ERR_INVALID_ARG;
    if (p->algo == GDN_ALGO_TC || p->algo == GDN_ALGO_TC_SINGLE || p->algo == GDN_ALGO_TC_WIDE)
        return GDN_ERR_UNSUPPORTED;
    if (p->K % 64 != 0 || p->K > 256) return GDN_ERR_UNSUPPORTED;
    if (p->V % 16 != 0 || p->V > 4096) return GDN_ERR_UNSUPPORTED;
    if (p->H > 65535 || p->B > 65535) return GDN_ERR_UNSUPPORTED;
    if (norm) {
        // one CTA per head: V must be a built slice width and K V / 32 <= 1024 threads
        const bool v_ok = p->V == 16 || p->V == 32 || p->V == 64 || p->V == 128 || p->V == 256;
        if (!v_ok || p->K * p->V > 32768) return GDN_ERR_UNSUPPORTED;
    }
    return GDN_OK;
}

// Columns per CTA: with the output stage the whole V; otherwise the widest
// slice (fewest, largest loads per row) that still gives at least two CTAs
// per SM; narrower slices only add CTAs.
int pick_vs(const gdn_problem *p, bool gated, int sms) {
    if (gated) return p->V;
    const long long heads = static_cast<long long>(p->B) * p->H;
    for (int vs : {64, 32}) {
        if (p->V % vs == 0 && heads * (p->V / vs) >= 2LL * sms) return vs;
    }
    return 16;
}

template <typename E, int K, int VS>
cudaError_t launch(const gdn_problem *pr, const DecodeParams<E> &p, cudaStream_t s) {
    if constexpr (decode_threads(K, VS) > 1024) {
        return cudaErrorInvalidConfiguration;   // excluded by check_decode
    } else {
        constexpr int threads = decode_threads(K, VS);
        const dim3 grid(pr->V / VS, pr->H, pr->B);
        const bool other = p.l2norm || p.gate;
        if (other)
            gdn_decode_step_kernel<E, K, VS, 2><<<grid, threads, 0, s>>>(p);
        else if (p.per_channel)
            gdn_decode_step_kernel<E, K, VS, 1><<<grid, threads, 0, s>>>(p);
        else
            gdn_decode_step_kernel<E, K, VS, 0><<<grid, threads, 0, s>>>(p);
        return cudaGetLastError();
    }
}

template <typename E, int K>
cudaError_t dispatch_vs(int vs, const gdn_problem *pr, const DecodeParams<E> &p, cudaStream_t s) {
    switch (vs) {
        case 256: return launch<E, K, 256>(pr, p, s);
        case 128: return launch<E, K, 128>(pr, p, s);
        case 64: return launch<E, K, 64>(pr, p, s);
        case 32: return launch<E, K, 32>(pr, p, s);
        default: return launch<E, K, 16>(pr, p, s);
    }
}

template <typename E>
cudaError_t dispatch(int vs, const gdn_problem *pr, const void *q, const void *k, const void *v,
                     const float *gamma, const float *beta, float scale, const float *state_in,
                     float *state_out, const gdn_output_norm *norm, void *o, cudaStream_t s) {
    DecodeParams<E> p;
    p.q = static_cast<const E *>(q);
    p.k = static_cast<const E *>(k);
    p.v = static_cast<const E *>(v);
    p.gamma = gamma;
    p.beta = beta;
    p.scale = scale;
    p.state_in = state_in;
    p.state_out = state_out;
    p.o = static_cast<E *>(o);
    p.T = pr->T;
    p.H = pr->H;
    p.V = pr->V;
    p.l2norm = (pr->flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
    p.per_channel = (pr->flags & GDN_FLAG_PER_CHANNEL_DECAY) ? 1 : 0;
    p.gate = norm ? static_cast<const E *>(norm->gate) : nullptr;
    p.norm_w = norm ? norm->weight : nullptr;
    p.norm_eps = norm ? norm->eps : 0.f;
    switch (pr->K) {
        case 64: return dispatch_vs<E, 64>(vs, pr, p, s);
        case 128: return dispatch_vs<E, 128>(vs, pr, p, s);
        case 192: return dispatch_vs<E, 192>(vs, pr, p, s);
        default: return dispatch_vs<E, 256>(vs, pr, p, s);
    }
}

}  // namespace
}  // namespace gdn

extern "C" {

GDN_API gdn_status gdn_decode_step_ex(const gdn_problem *p, const void *q, const void *k,
                                      const void *v, const float *gamma, const float *beta,
                                      float scale, const float *state_in, float *state_out,
                                      const gdn_output_norm *norm, void *o, void *stream) {
    const gdn_status st = gdn::check_decode(p, norm);
    if (st != GDN_OK) return st;
    if (!state_in || !state_out) return GDN_ERR_INVALID_ARG;
    const bool empty = p->T == 0;
    if (!empty && (!q || !k || !v || !gamma || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, gamma, beta, state_in, state_out, o,
                          norm ? norm->gate : nullptr, norm ? norm->weight : nullptr};
    for (const void *ptr : ptrs)
        if (ptr && !gdn::aligned16(ptr)) return GDN_ERR_ALIGNMENT;
    const size_t state_bytes =
        static_cast<size_t>(p->B) * p->H * p->K * p->V * sizeof(float);
    const char *si = reinterpret_cast<const char *>(state_in);
    const char *so = reinterpret_cast<const char *>(state_out);
    if (si != so && si < so + state_bytes && so < si + state_bytes) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (empty) {
        if (si != so)
            e = cudaMemcpyAsync(state_out, state_in, state_bytes, cudaMemcpyDeviceToDevice, s);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int vs = gdn::pick_vs(p, norm != nullptr, sms);
    if (p->dtype == GDN_BF16)
        e = gdn::dispatch<__nv_bfloat16>(vs, p, q, k, v, gamma, beta, scale, state_in, state_out,
                                         norm, o, s);
    else
        e = gdn::dispatch<float>(vs, p, q, k, v, gamma, beta, scale, state_in, state_out, norm, o,
                                 s);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

GDN_API gdn_status gdn_decode_step(const gdn_problem *p, const void *q, const void *k,
                                   const void *v, const float *gamma, const float *beta,
                                   float scale, const float *state_in, float *state_out, void *o,
                                   void *stream) {
    return gdn_decode_step_ex(p, q, k, v, gamma, beta, scale, state_in, state_out, nullptr, o,
                              stream);
}

GDN_API int32_t gdn_decode_step_launches(const gdn_problem *p, const char **names,
                                         int32_t max_names) {
    if (gdn::check_decode(p, nullptr) != GDN_OK || p->T == 0) return 0;
    if (names && max_names > 0) names[0] = gdn::kDecodeName;
    return 1;
}

}  // extern "C"
