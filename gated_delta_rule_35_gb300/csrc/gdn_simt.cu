// CUDA-core (SIMT) pipeline of the chunked gated delta rule forward, fp32
// arithmetic throughout. It is the path for fp32 inputs (tensor-core TF32
// would not hold 1e-4 relative error) and the stage-by-stage reference path
// whose intermediates can be exported. Four kernels, as in the "WarpDrive"
// page's pipeline (kernels 3-5): WY build + recompute_w_u, chunk_fwd_h,
// chunk_fwd_o. Intermediates live in an fp32 workspace.
#include <cuda_bf16.h>

#include <algorithm>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kBV = 16;   // V columns of the state per chunk_fwd_h block
constexpr int kMaxK = 128;  // largest K of the chunked forward

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Row index of token t of sequence (b, h) in a [B,T,H,*] tensor.
__device__ __forceinline__ int64_t tok(int b, int t, int h, int T, int H) {
    return (static_cast<int64_t>(b) * T + t) * H + h;
}

// Front-end q/k normalisation in shared memory: rows 0..n-1 of xs (stride KP,
// K values) become x / sqrt(sum x^2 + eps), one warp per row; the factors go
// to rs[i] when rs is given. Call between barriers.
__device__ void l2norm_rows_smem(float *xs, int KP, int K, int n, float *rs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int i = warp; i < n; i += nw) {
        float ss = 0.f;
        for (int kk = lane; kk < K; kk += 32) ss = fmaf(xs[i * KP + kk], xs[i * KP + kk], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = rsqrtf(ss + kL2NormEps);
        for (int kk = lane; kk < K; kk += 32) xs[i * KP + kk] *= r;
        if (rs && lane == 0) rs[i] = r;
    }
}

// Per-channel decay, factored about r_d = g_last,d / 2: with
//   a_id = x_id exp(g_id - r_d),   b_jd = y_jd exp(r_d - g_jd)
// sum_d a_id b_jd = sum_d x_id y_jd exp(g_id - g_jd), one product per term.
// Valid while every |g_last,d| <= 160 (both factors within e^+-80; decays <= 0
// keep g_id between g_last,d and 0). xs becomes a and gk (holding g) becomes b;
// rows past n hold zeros in xs and ys, so they stay zero. r_d goes to rs.
// Returns false, changing nothing, when some channel is out of that range.
__device__ bool factor_per_channel(float *xs, const float *ys, float *gk, float *rs, int KP, int K,
                                   int n) {
    const int tid = threadIdx.x;
    if (__syncthreads_or(tid < K && fabsf(gk[(n - 1) * KP + tid]) > 160.f)) return false;
    if (tid < K) rs[tid] = 0.5f * gk[(n - 1) * KP + tid];
    __syncthreads();
    for (int idx = tid; idx < kChunk * K; idx += blockDim.x) {
        const int i = idx / K, kk = idx - i * K;
        const float gv = gk[i * KP + kk], r = rs[kk];
        const float yv = ys[i * KP + kk];
        xs[i * KP + kk] *= expf(gv - r);
        gk[i * KP + kk] = yv * expf(r - gv);
    }
    __syncthreads();
    return true;
}

// ---------------------------------------------------------------------------
// WY build + recompute_w_u ("WarpDrive" kernel 5). One block per (chunk, h, b).
//   L_ij = beta_i (k_i . k_j) exp(g_i - g_j), i > j;  A = (I + L)^-1
//   w = A (k * beta * exp(g)),  u = A (v * beta)
// The inverse is a forward substitution: thread c owns column c of A and
// walks rows i = c..63: A_ic = [i == c] - sum_{c <= j < i} L_ij A_jc.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
wy_prepare_kernel(const T *__restrict__ k, const T *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, int Tn, int H, int K, int V, int T_pad,
                  float *__restrict__ A_ws, float *__restrict__ w_ws, float *__restrict__ u_ws,
                  int flags, float *__restrict__ g_cum, float *__restrict__ rk_out) {
    extern __shared__ float smem[];
    __shared__ float gs[kChunk], bs[kChunk], rks[kChunk], rs[kMaxK];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int t0 = c * kChunk;
    const int n = min(kChunk, Tn - t0);
    const int KP = K + 1;
    float *ks = smem;                  // [64][K+1]
    float *Ls = ks + kChunk * KP;      // [64][65]
    float *As = Ls + kChunk * 65;      // [64][65]
    float *xs = As + kChunk * 65;      // [64][65] slice of v * beta
    // per-channel decay: g of the chunk's tokens, [64][K+1]
    const bool pc = flags & GDN_FLAG_PER_CHANNEL_DECAY;
    float *gk = xs + kChunk * 65;

    if (tid < kChunk) {
        gs[tid] = (!pc && tid < n) ? g[tok(b, t0 + tid, h, Tn, H)] : 0.f;
        bs[tid] = tid < n ? beta[tok(b, t0 + tid, h, Tn, H)] : 0.f;
    }
#pragma unroll 8
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
        const int i = idx / K, kk = idx - i * K;
        ks[i * KP + kk] = i < n ? to_f32(k[tok(b, t0 + i, h, Tn, H) * K + kk]) : 0.f;
        if (pc) gk[i * KP + kk] = i < n ? g[tok(b, t0 + i, h, Tn, H) * K + kk] : 0.f;
    }
    __syncthreads();
    // Front-end: g from raw per-token log decays (chunk-local inclusive sum,
    // per channel with per-channel decay), k rows normalised; both written out
    // for the later kernels.
    if (flags & GDN_FLAG_RAW_G) {
        if (!pc && tid == 0) {
            float acc = 0.f;
            for (int i = 0; i < n; ++i) gs[i] = acc += gs[i];
        }
        if (pc && tid < K) {
            float acc = 0.f;
            for (int i = 0; i < n; ++i) {
                acc += gk[i * KP + tid];
                gk[i * KP + tid] = acc;
                g_cum[tok(b, t0 + i, h, Tn, H) * K + tid] = acc;
            }
        }
        __syncthreads();
        if (!pc && tid < n) g_cum[tok(b, t0 + tid, h, Tn, H)] = gs[tid];
    }
    if (flags & GDN_FLAG_QK_L2NORM) {
        l2norm_rows_smem(ks, KP, K, n, rks);
        __syncthreads();
        if (tid < n) rk_out[tok(b, t0 + tid, h, Tn, H)] = rks[tid];
    }

    // per-channel decay: k_i . k_j exp(g_i - g_j) channel by channel, factored
    // (ks <- k exp(g - r), gk <- k exp(r - g)) when the chunk's decays allow
    const bool pc_fz = pc && factor_per_channel(ks, ks, gk, rs, KP, K, n);

    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        const int i = idx >> 6, j = idx & 63;
        float val = 0.f;
        if (i > j && i < n) {
            float dot = 0.f;
            if (pc_fz) {
                for (int kk = 0; kk < K; ++kk) dot = fmaf(ks[i * KP + kk], gk[j * KP + kk], dot);
                val = bs[i] * dot;
            } else if (pc) {
                // sum_d k_id k_jd exp(g_id - g_jd): each channel its own decay
                for (int kk = 0; kk < K; ++kk)
                    dot = fmaf(ks[i * KP + kk] * ks[j * KP + kk],
                               expf(gk[i * KP + kk] - gk[j * KP + kk]), dot);
                val = bs[i] * dot;
            } else {
                for (int kk = 0; kk < K; ++kk) dot = fmaf(ks[i * KP + kk], ks[j * KP + kk], dot);
                val = bs[i] * dot * expf(gs[i] - gs[j]);
            }
        }
        Ls[i * 65 + j] = val;
    }
    __syncthreads();

    if (tid < kChunk) {
        const int col = tid;
        for (int i = 0; i < col; ++i) As[i * 65 + col] = 0.f;
        for (int i = col; i < kChunk; ++i) {
            float acc = (i == col) ? 1.f : 0.f;
            for (int j = col; j < i; ++j) acc = fmaf(-Ls[i * 65 + j], As[j * 65 + col], acc);
            As[i * 65 + col] = acc;
        }
    }
    // k <- k * beta * exp(g) (the Gram above used the unscaled rows)
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
        const int i = idx / K, kk = idx - i * K;
        // factored: ks holds k exp(g - r), so k exp(g) = ks exp(r)
        const float e = pc_fz ? expf(rs[kk]) : expf(pc ? gk[i * KP + kk] : gs[i]);
        ks[i * KP + kk] *= (i < n) ? bs[i] * e : 0.f;
    }
    __syncthreads();

    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        const int i = idx >> 6, j = idx & 63;
        A_ws[tok(b, t0 + i, h, T_pad, H) * kChunk + j] = As[i * 65 + j];
    }
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
        const int i = idx / K, kk = idx - i * K;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(As[i * 65 + j], ks[j * KP + kk], acc);
        w_ws[tok(b, t0 + i, h, T_pad, H) * K + kk] = acc;
    }
    for (int vs = 0; vs < V; vs += 64) {
        __syncthreads();
#pragma unroll 8
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int j = idx >> 6, nn = idx & 63;
            xs[j * 65 + nn] = j < n ? bs[j] * to_f32(v[tok(b, t0 + j, h, Tn, H) * V + vs + nn]) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int i = idx >> 6, nn = idx & 63;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc = fmaf(As[i * 65 + j], xs[j * 65 + nn], acc);
            u_ws[tok(b, t0 + i, h, T_pad, H) * V + vs + nn] = acc;
        }
    }
}

// ---------------------------------------------------------------------------
// chunk_fwd_h ("WarpDrive" kernel 3). One block per (V tile of 16, h, b),
// sequential over the chunks: store h; v_new = u - w @ h;
// v_gated = v_new * exp(g_last - g_t); h = h * exp(g_last) + k^T @ v_gated.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
chunk_h_kernel(const T *__restrict__ k, const float *__restrict__ g, const float *__restrict__ w_ws,
               const float *__restrict__ u_ws, const float *__restrict__ h0, int Tn, int H, int K,
               int V, int NT, int T_pad, float *__restrict__ h_ws, float *__restrict__ vn_ws,
               float *__restrict__ h_final, const float *__restrict__ rk, int flags) {
    extern __shared__ float smem[];
    __shared__ float gs[kChunk];
    const int v0 = blockIdx.x * kBV, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int KP = K + 1;
    float *hs = smem;                   // [K][kBV]
    float *ws = hs + K * kBV;           // [64][K+1]
    float *ks = ws + kChunk * KP;       // [64][K+1]
    float *vs = ks + kChunk * KP;       // [64][kBV + 1]: u, then v_new, then v_gated
    constexpr int VP = kBV + 1;
    // per-channel decay: the chunk's g, [64][K+1]
    const bool pc = flags & GDN_FLAG_PER_CHANNEL_DECAY;
    float *gk = vs + kChunk * VP;
    const int64_t state = (static_cast<int64_t>(b) * H + h) * K * V;

#pragma unroll 8
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
        const int kk = idx / kBV, nn = idx - kk * kBV;
        hs[idx] = h0 ? h0[state + static_cast<int64_t>(kk) * V + v0 + nn] : 0.f;
    }
    for (int c = 0; c < NT; ++c) {
        const int t0 = c * kChunk;
        const int n = min(kChunk, Tn - t0);
        __syncthreads();
        const int64_t hslot = ((static_cast<int64_t>(b) * NT + c) * H + h) * K * V;
#pragma unroll 8
        for (int idx = tid; idx < K * kBV; idx += kThreads) {
            const int kk = idx / kBV, nn = idx - kk * kBV;
            h_ws[hslot + static_cast<int64_t>(kk) * V + v0 + nn] = hs[idx];
        }
        if (tid < kChunk) gs[tid] = (!pc && tid < n) ? g[tok(b, t0 + tid, h, Tn, H)] : 0.f;
#pragma unroll 8
        for (int idx = tid; idx < kChunk * K; idx += kThreads) {
            const int i = idx / K, kk = idx - i * K;
            ws[i * KP + kk] = w_ws[tok(b, t0 + i, h, T_pad, H) * K + kk];
            const int64_t r = tok(b, t0 + i, h, Tn, H);
            ks[i * KP + kk] = i < n ? to_f32(k[r * K + kk]) * (rk ? rk[r] : 1.f) : 0.f;
            if (pc) gk[i * KP + kk] = i < n ? g[r * K + kk] : 0.f;
        }
#pragma unroll 8
        for (int idx = tid; idx < kChunk * kBV; idx += kThreads) {
            const int i = idx / kBV, nn = idx - i * kBV;
            vs[i * VP + nn] = u_ws[tok(b, t0 + i, h, T_pad, H) * V + v0 + nn];
        }
        __syncthreads();
        // v_new = u - w @ h
        float vnew[kChunk * kBV / kThreads];
#pragma unroll
        for (int r = 0; r < kChunk * kBV / kThreads; ++r) {
            const int idx = tid + r * kThreads;
            const int i = idx / kBV, nn = idx - i * kBV;
            float acc = vs[i * VP + nn];
            for (int kk = 0; kk < K; ++kk) acc = fmaf(-ws[i * KP + kk], hs[kk * kBV + nn], acc);
            vnew[r] = acc;
            vn_ws[tok(b, t0 + i, h, T_pad, H) * V + v0 + nn] = acc;
        }
        __syncthreads();
        const float glast = gs[n - 1];
#pragma unroll
        for (int r = 0; r < kChunk * kBV / kThreads; ++r) {
            const int idx = tid + r * kThreads;
            const int i = idx / kBV, nn = idx - i * kBV;
            vs[i * VP + nn] = i < n ? (pc ? vnew[r] : vnew[r] * expf(glast - gs[i])) : 0.f;
        }
        if (pc) {
            // per channel the gate sits on k: k_id exp(g_last,d - g_id)
            for (int idx = tid; idx < n * K; idx += kThreads) {
                const int i = idx / K, kk = idx - i * K;
                ks[i * KP + kk] *= expf(gk[(n - 1) * KP + kk] - gk[i * KP + kk]);
            }
        }
        __syncthreads();
        // h = h * exp(g_last) + k^T @ v_gated (row d by exp(g_last,d) per channel)
        const float decay = expf(glast);
        for (int idx = tid; idx < K * kBV; idx += kThreads) {
            const int kk = idx / kBV, nn = idx - kk * kBV;
            float acc = hs[idx] * (pc ? expf(gk[(n - 1) * KP + kk]) : decay);
            for (int i = 0; i < n; ++i) acc = fmaf(ks[i * KP + kk], vs[i * VP + nn], acc);
            hs[idx] = acc;
        }
    }
    if (h_final) {
        __syncthreads();
#pragma unroll 8
        for (int idx = tid; idx < K * kBV; idx += kThreads) {
            const int kk = idx / kBV, nn = idx - kk * kBV;
            h_final[state + static_cast<int64_t>(kk) * V + v0 + nn] = hs[idx];
        }
    }
}

// ---------------------------------------------------------------------------
// chunk_fwd_o ("WarpDrive" kernel 4). One block per (chunk, h, b):
//   P_ij = (q_i . k_j) exp(g_i - g_j) for j <= i (diagonal included), else 0
//   o_i  = scale * (exp(g_i) q_i^T h_c + sum_j P_ij v_new_j)
// with h_c the state entering the chunk and v_new the ungated values.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
chunk_o_kernel(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ g,
               const float *__restrict__ h_ws, const float *__restrict__ vn_ws, int Tn, int H,
               int K, int V, int NT, int T_pad, float scale, T *__restrict__ o, int flags,
               const T *__restrict__ gate, const float *__restrict__ norm_w, float norm_eps) {
    extern __shared__ float smem[];
    __shared__ float gs[kChunk], rs[kMaxK];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int t0 = c * kChunk;
    const int n = min(kChunk, Tn - t0);
    const int KP = K + 1;
    float *qs = smem;                  // [64][K+1]
    float *ks = qs + kChunk * KP;      // [64][K+1]
    float *Ps = ks + kChunk * KP;      // [64][65]
    float *hs = Ps + kChunk * 65;      // [K][65]
    float *vs = hs + K * 65;           // [64][65]
    // [64][V + 1] fp32 o rows (output stage only), sharing its space with the
    // per-channel g [64][K + 1], which is not read once o rows are written
    float *os = vs + kChunk * 65;
    const int OP = V + 1;
    const bool pc = flags & GDN_FLAG_PER_CHANNEL_DECAY;
    float *gk = os;

    if (tid < kChunk) gs[tid] = (!pc && tid < n) ? g[tok(b, t0 + tid, h, Tn, H)] : 0.f;
#pragma unroll 8
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
        const int i = idx / K, kk = idx - i * K;
        const bool ok = i < n;
        qs[i * KP + kk] = ok ? to_f32(q[tok(b, t0 + i, h, Tn, H) * K + kk]) : 0.f;
        ks[i * KP + kk] = ok ? to_f32(k[tok(b, t0 + i, h, Tn, H) * K + kk]) : 0.f;
        if (pc) gk[i * KP + kk] = ok ? g[tok(b, t0 + i, h, Tn, H) * K + kk] : 0.f;
    }
    __syncthreads();
    if (flags & GDN_FLAG_QK_L2NORM) {
        l2norm_rows_smem(qs, KP, K, n, nullptr);
        l2norm_rows_smem(ks, KP, K, n, nullptr);
        __syncthreads();
    }
    // per-channel decay, factored (qs <- q exp(g - r), gk <- k exp(r - g)) when
    // the chunk's decays allow
    const bool pc_fz = pc && factor_per_channel(qs, ks, gk, rs, KP, K, n);
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        const int i = idx >> 6, j = idx & 63;
        float val = 0.f;
        if (j <= i && i < n) {
            float dot = 0.f;
            if (pc_fz) {
                for (int kk = 0; kk < K; ++kk) dot = fmaf(qs[i * KP + kk], gk[j * KP + kk], dot);
                val = dot;
            } else if (pc) {
                for (int kk = 0; kk < K; ++kk)
                    dot = fmaf(qs[i * KP + kk] * ks[j * KP + kk],
                               expf(gk[i * KP + kk] - gk[j * KP + kk]), dot);
                val = dot;
            } else {
                for (int kk = 0; kk < K; ++kk) dot = fmaf(qs[i * KP + kk], ks[j * KP + kk], dot);
                val = dot * expf(gs[i] - gs[j]);
            }
        }
        Ps[i * 65 + j] = val;
    }
    if (pc) {
        // inter term per channel: (q_i * exp(g_i)) . h; gs stays 0 so exp(gs) = 1
        __syncthreads();
        for (int idx = tid; idx < n * K; idx += kThreads) {
            const int i = idx / K, kk = idx - i * K;
            qs[i * KP + kk] *= pc_fz ? expf(rs[kk]) : expf(gk[i * KP + kk]);
        }
    }
    const int64_t hslot = ((static_cast<int64_t>(b) * NT + c) * H + h) * K * V;
    for (int v0 = 0; v0 < V; v0 += 64) {
        __syncthreads();
#pragma unroll 8
        for (int idx = tid; idx < K * 64; idx += kThreads) {
            const int kk = idx >> 6, nn = idx & 63;
            hs[kk * 65 + nn] = h_ws[hslot + static_cast<int64_t>(kk) * V + v0 + nn];
        }
#pragma unroll 8
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int j = idx >> 6, nn = idx & 63;
            vs[j * 65 + nn] = vn_ws[tok(b, t0 + j, h, T_pad, H) * V + v0 + nn];
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int i = idx >> 6, nn = idx & 63;
            if (i >= n) continue;
            float inter = 0.f;
            for (int kk = 0; kk < K; ++kk) inter = fmaf(qs[i * KP + kk], hs[kk * 65 + nn], inter);
            float intra = 0.f;
            for (int j = 0; j <= i; ++j) intra = fmaf(Ps[i * 65 + j], vs[j * 65 + nn], intra);
            const float oi = scale * (expf(gs[i]) * inter + intra);
            if (gate)
                os[i * OP + v0 + nn] = oi;
            else
                store_as(&o[tok(b, t0 + i, h, Tn, H) * V + v0 + nn], oi);
        }
    }
    if (gate) {
        // gated RMSNorm over the V values of each row, one warp per row
        __syncthreads();
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < n; i += kThreads / 32) {
            float ss = 0.f;
            for (int nn = lane; nn < V; nn += 32) ss = fmaf(os[i * OP + nn], os[i * OP + nn], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float rstd = rsqrtf(ss / V + norm_eps);
            const int64_t r = tok(b, t0 + i, h, Tn, H) * V;
            for (int nn = lane; nn < V; nn += 32) {
                const float z = to_f32(gate[r + nn]);
                const float sg = 1.f / (1.f + expf(-z));
                store_as(&o[r + nn], os[i * OP + nn] * rstd * norm_w[nn] * sg);
            }
        }
    }
}

__global__ void copy_state_kernel(const float *__restrict__ h0, float *__restrict__ h_final,
                                  int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        h_final[i] = h0 ? h0[i] : 0.f;
}

size_t prepare_smem(int K, bool pc) {
    return sizeof(float) * (kChunk * (K + 1) + 3 * kChunk * 65 + (pc ? kChunk * (K + 1) : 0));
}
size_t chunk_h_smem(int K, bool pc) {
    return sizeof(float) * (K * kBV + 2 * kChunk * (K + 1) + kChunk * (kBV + 1) +
                            (pc ? kChunk * (K + 1) : 0));
}
size_t chunk_o_smem(int K, int V, bool normed, bool pc) {
    const int tail = std::max(normed ? kChunk * (V + 1) : 0, pc ? kChunk * (K + 1) : 0);
    return sizeof(float) * (2 * kChunk * (K + 1) + kChunk * 65 + K * 65 + kChunk * 65 + tail);
}

template <typename T>
cudaError_t run(const Args &a, const SimtWorkspace &ws, cudaStream_t s, const Marks &m) {
    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k),
            *v = static_cast<const T *>(a.v);
    cudaError_t e;
    const bool pc = a.flags & GDN_FLAG_PER_CHANNEL_DECAY;
    const size_t s1 = prepare_smem(a.K, pc), s2 = chunk_h_smem(a.K, pc),
                 s3 = chunk_o_smem(a.K, a.V, a.gate != nullptr, pc);
    if ((e = cudaFuncSetAttribute(wy_prepare_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(s1))) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(chunk_h_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(s2))) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(chunk_o_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(s3))) != cudaSuccess)
        return e;
    const dim3 chunks(a.NT, a.H, a.B);
    if ((e = m.mark(0, s)) != cudaSuccess) return e;
    wy_prepare_kernel<T><<<chunks, kThreads, s1, s>>>(k, v, a.g, a.beta, a.T, a.H, a.K, a.V,
                                                     a.T_pad, ws.A, ws.w, ws.u, a.flags, a.g_cum,
                                                     a.rk);
    if ((e = m.mark(1, s)) != cudaSuccess) return e;
    const float *rk = (a.flags & GDN_FLAG_QK_L2NORM) ? a.rk : nullptr;
    chunk_h_kernel<T><<<dim3(a.V / kBV, a.H, a.B), kThreads, s2, s>>>(
        k, a.g_chunk(), ws.w, ws.u, a.h0, a.T, a.H, a.K, a.V, a.NT, a.T_pad, ws.h, ws.v_new,
        a.h_final, rk, a.flags);
    if ((e = m.mark(2, s)) != cudaSuccess) return e;
    chunk_o_kernel<T><<<chunks, kThreads, s3, s>>>(q, k, a.g_chunk(), ws.h, ws.v_new, a.T, a.H, a.K,
                                                  a.V, a.NT, a.T_pad, a.scale,
                                                  static_cast<T *>(a.o), a.flags,
                                                  static_cast<const T *>(a.gate), a.norm_w,
                                                  a.norm_eps);
    if ((e = m.mark(3, s)) != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t simt_workspace_bytes(int B, int T, int H, int K, int V) {
    const size_t NT = static_cast<size_t>(num_chunks(T));
    const size_t rows = static_cast<size_t>(B) * NT * kChunk * H;
    return align_up(rows * kChunk * 4) + align_up(rows * K * 4) + 2 * align_up(rows * V * 4) +
           align_up(static_cast<size_t>(B) * NT * H * K * V * 4);
}

SimtWorkspace simt_carve(void *base, int B, int T, int H, int K, int V) {
    const size_t NT = static_cast<size_t>(num_chunks(T));
    const size_t rows = static_cast<size_t>(B) * NT * kChunk * H;
    char *p = static_cast<char *>(base);
    SimtWorkspace w;
    w.A = reinterpret_cast<float *>(p);
    p += align_up(rows * kChunk * 4);
    w.w = reinterpret_cast<float *>(p);
    p += align_up(rows * K * 4);
    w.u = reinterpret_cast<float *>(p);
    p += align_up(rows * V * 4);
    w.v_new = reinterpret_cast<float *>(p);
    p += align_up(rows * V * 4);
    w.h = reinterpret_cast<float *>(p);
    return w;
}

const char *const kSimtKernelNames[kSimtLaunches] = {"wy_prepare_kernel", "chunk_h_kernel",
                                                     "chunk_o_kernel"};

cudaError_t simt_forward(const Args &a, const SimtWorkspace &ws, cudaStream_t s, const Marks &m) {
    if (a.dtype == GDN_BF16) return run<__nv_bfloat16>(a, ws, s, m);
    return run<float>(a, ws, s, m);
}

cudaError_t copy_state(const Args &a, cudaStream_t s) {
    if (!a.h_final) return cudaSuccess;
    const int64_t n = static_cast<int64_t>(a.B) * a.H * a.K * a.V;
    copy_state_kernel<<<152, 256, 0, s>>>(a.h0, a.h_final, n);
    return cudaGetLastError();
}

}  // namespace gdn
