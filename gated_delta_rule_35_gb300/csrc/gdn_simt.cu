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
    float *xs = As + kChunk * 65;      // [64][64] slice of v * beta (rows read as float4)
    // per-channel decay: g of the chunk's tokens, [64][K+1]
    const bool pc = flags & GDN_FLAG_PER_CHANNEL_DECAY;
    float *gk = xs + kChunk * 64;

    if (tid < kChunk) {
        gs[tid] = (!pc && tid < n) ? g[tok(b, t0 + tid, h, Tn, H)] : 0.f;
        bs[tid] = tid < n ? beta[tok(b, t0 + tid, h, Tn, H)] : 0.f;
    }
#pragma unroll 4
    for (int idx = tid; idx < kChunk * K / 4; idx += kThreads) {
        const int i = idx / (K / 4), kk = (idx - i * (K / 4)) * 4;
        const int64_t r = tok(b, t0 + i, h, Tn, H) * K + kk;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ks[i * KP + kk + e] = i < n ? to_f32(k[r + e]) : 0.f;
            if (pc) gk[i * KP + kk + e] = i < n ? g[r + e] : 0.f;
        }
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

    // L, 4 x 4 tiles per thread (rows 4 ti.., columns 4 tj..; tiles above the
    // diagonal stay 0)
    {
        const int i0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
        float acc[4][4] = {};
        if (c0 < i0 + 3 && i0 < n) {
            const float *kb = pc_fz ? gk : ks;
            for (int kk = 0; kk < K; ++kk) {
                float ki[4], kj[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    ki[r] = ks[(i0 + r) * KP + kk];
                    kj[r] = kb[(c0 + r) * KP + kk];
                }
                if (pc && !pc_fz) {
                    // sum_d k_id k_jd exp(g_id - g_jd): each channel its own decay
                    float gi[4], gj[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        gi[r] = gk[(i0 + r) * KP + kk];
                        gj[r] = gk[(c0 + r) * KP + kk];
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            acc[r][cc] = fmaf(ki[r] * kj[cc], expf(gi[r] - gj[cc]), acc[r][cc]);
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) acc[r][cc] = fmaf(ki[r], kj[cc], acc[r][cc]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int i = i0 + r, j = c0 + cc;
                float val = 0.f;
                if (i > j && i < n)
                    val = bs[i] * (pc ? acc[r][cc] : acc[r][cc] * expf(gs[i] - gs[j]));
                Ls[i * 65 + j] = val;
            }
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

#pragma unroll 4
    for (int idx = tid; idx < kChunk * 16; idx += kThreads) {
        const int i = idx >> 4, j4 = (idx & 15) * 4;
        *reinterpret_cast<float4 *>(&A_ws[tok(b, t0 + i, h, T_pad, H) * kChunk + j4]) =
            make_float4(As[i * 65 + j4], As[i * 65 + j4 + 1], As[i * 65 + j4 + 2], As[i * 65 + j4 + 3]);
    }
    // w = A (scaled k), 4 x 4 tiles; A is 0 above the diagonal, so a tile of
    // rows i0.. needs columns j < i0 + 4 only
    for (int t = tid; t < 16 * (K / 4); t += kThreads) {
        const int i0 = (t / (K / 4)) * 4, c0 = (t % (K / 4)) * 4;
        float acc[4][4] = {};
        for (int j = 0; j < i0 + 4; ++j) {
            float kv[4], av[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                kv[r] = ks[j * KP + c0 + r];
                av[r] = As[(i0 + r) * 65 + j];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) acc[r][cc] = fmaf(av[r], kv[cc], acc[r][cc]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4 *>(&w_ws[tok(b, t0 + i0 + r, h, T_pad, H) * K + c0]) =
                make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
    for (int vs = 0; vs < V; vs += 64) {
        __syncthreads();
#pragma unroll 4
        for (int idx = tid; idx < kChunk * 16; idx += kThreads) {
            const int j = idx >> 4, n4 = (idx & 15) * 4;
            const int64_t r = tok(b, t0 + j, h, Tn, H) * V + vs + n4;
            const float bj = j < n ? bs[j] : 0.f;
            float4 x;
            x.x = j < n ? bj * to_f32(v[r]) : 0.f;
            x.y = j < n ? bj * to_f32(v[r + 1]) : 0.f;
            x.z = j < n ? bj * to_f32(v[r + 2]) : 0.f;
            x.w = j < n ? bj * to_f32(v[r + 3]) : 0.f;
            *reinterpret_cast<float4 *>(&xs[j * 64 + n4]) = x;
        }
        __syncthreads();
        {
            // u = A (v * beta), one 4 x 4 tile per thread
            const int i0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
            float acc[4][4] = {};
            for (int j = 0; j < i0 + 4; ++j) {
                const float4 x4 = *reinterpret_cast<const float4 *>(&xs[j * 64 + c0]);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float av = As[(i0 + r) * 65 + j];
                    acc[r][0] = fmaf(av, x4.x, acc[r][0]);
                    acc[r][1] = fmaf(av, x4.y, acc[r][1]);
                    acc[r][2] = fmaf(av, x4.z, acc[r][2]);
                    acc[r][3] = fmaf(av, x4.w, acc[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
                *reinterpret_cast<float4 *>(&u_ws[tok(b, t0 + i0 + r, h, T_pad, H) * V + vs + c0]) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
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
    float *vs = ks + kChunk * KP;       // [64][kBV]: u, then v_new, then v_gated
    constexpr int VP = kBV;             // rows of 16 floats, read as float4
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
        // global traffic in 16-byte pieces: 4 consecutive floats (or k values)
#pragma unroll 4
        for (int idx = tid; idx < K * kBV / 4; idx += kThreads) {
            const int kk = idx / (kBV / 4), n4 = (idx - kk * (kBV / 4)) * 4;
            *reinterpret_cast<float4 *>(&h_ws[hslot + static_cast<int64_t>(kk) * V + v0 + n4]) =
                *reinterpret_cast<const float4 *>(&hs[kk * kBV + n4]);
        }
        if (tid < kChunk) gs[tid] = (!pc && tid < n) ? g[tok(b, t0 + tid, h, Tn, H)] : 0.f;
#pragma unroll 4
        for (int idx = tid; idx < kChunk * K / 4; idx += kThreads) {
            const int i = idx / (K / 4), kk = (idx - i * (K / 4)) * 4;
            const float4 wv = *reinterpret_cast<const float4 *>(&w_ws[tok(b, t0 + i, h, T_pad, H) * K + kk]);
            ws[i * KP + kk] = wv.x;
            ws[i * KP + kk + 1] = wv.y;
            ws[i * KP + kk + 2] = wv.z;
            ws[i * KP + kk + 3] = wv.w;
            const int64_t r = tok(b, t0 + i, h, Tn, H);
            const float sc = i < n ? (rk ? rk[r] : 1.f) : 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) ks[i * KP + kk + e] = i < n ? to_f32(k[r * K + kk + e]) * sc : 0.f;
            if (pc) {
#pragma unroll
                for (int e = 0; e < 4; ++e) gk[i * KP + kk + e] = i < n ? g[r * K + kk + e] : 0.f;
            }
        }
#pragma unroll 4
        for (int idx = tid; idx < kChunk * kBV / 4; idx += kThreads) {
            const int i = idx / (kBV / 4), n4 = (idx - i * (kBV / 4)) * 4;
            *reinterpret_cast<float4 *>(&vs[i * VP + n4]) =
                *reinterpret_cast<const float4 *>(&u_ws[tok(b, t0 + i, h, T_pad, H) * V + v0 + n4]);
        }
        __syncthreads();
        // v_new = u - w @ h: thread (i, 4 columns), one w and one float4 of h
        // per four products
        static_assert(kChunk * kBV == 4 * kThreads, "v_new tiling");
        const int vi = tid >> 2, vn0 = (tid & 3) * 4;
        float4 vnew = *reinterpret_cast<const float4 *>(&vs[vi * VP + vn0]);
#pragma unroll 4
        for (int kk = 0; kk < K; ++kk) {
            const float wv = ws[vi * KP + kk];
            const float4 h4 = *reinterpret_cast<const float4 *>(&hs[kk * kBV + vn0]);
            vnew.x = fmaf(-wv, h4.x, vnew.x);
            vnew.y = fmaf(-wv, h4.y, vnew.y);
            vnew.z = fmaf(-wv, h4.z, vnew.z);
            vnew.w = fmaf(-wv, h4.w, vnew.w);
        }
        *reinterpret_cast<float4 *>(&vn_ws[tok(b, t0 + vi, h, T_pad, H) * V + v0 + vn0]) = vnew;
        __syncthreads();
        const float glast = gs[n - 1];
        {
            const float gate = vi < n ? (pc ? 1.f : expf(glast - gs[vi])) : 0.f;
            *reinterpret_cast<float4 *>(&vs[vi * VP + vn0]) =
                make_float4(vnew.x * gate, vnew.y * gate, vnew.z * gate, vnew.w * gate);
        }
        if (pc) {
            // per channel the gate sits on k: k_id exp(g_last,d - g_id)
            for (int idx = tid; idx < n * K; idx += kThreads) {
                const int i = idx / K, kk = idx - i * K;
                ks[i * KP + kk] *= expf(gk[(n - 1) * KP + kk] - gk[i * KP + kk]);
            }
        }
        __syncthreads();
        // h = h * exp(g_last) + k^T @ v_gated (row d by exp(g_last,d) per channel):
        // thread (K / 128 row pairs, 4 columns), two k values and one float4 of
        // v_gated per eight products
        const float decay = expf(glast);
        for (int kb = 0; kb < K; kb += 128) {
            const int kk0 = kb + (tid >> 2) * 2, hn0 = (tid & 3) * 4;
            if (kk0 >= K) break;   // K = 64: half the threads have no rows
            float4 a0 = *reinterpret_cast<const float4 *>(&hs[kk0 * kBV + hn0]);
            float4 a1 = *reinterpret_cast<const float4 *>(&hs[(kk0 + 1) * kBV + hn0]);
            const float d0 = pc ? expf(gk[(n - 1) * KP + kk0]) : decay;
            const float d1 = pc ? expf(gk[(n - 1) * KP + kk0 + 1]) : decay;
            a0 = make_float4(a0.x * d0, a0.y * d0, a0.z * d0, a0.w * d0);
            a1 = make_float4(a1.x * d1, a1.y * d1, a1.z * d1, a1.w * d1);
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                const float k0 = ks[i * KP + kk0], k1 = ks[i * KP + kk0 + 1];
                const float4 v4 = *reinterpret_cast<const float4 *>(&vs[i * VP + hn0]);
                a0.x = fmaf(k0, v4.x, a0.x); a0.y = fmaf(k0, v4.y, a0.y);
                a0.z = fmaf(k0, v4.z, a0.z); a0.w = fmaf(k0, v4.w, a0.w);
                a1.x = fmaf(k1, v4.x, a1.x); a1.y = fmaf(k1, v4.y, a1.y);
                a1.z = fmaf(k1, v4.z, a1.z); a1.w = fmaf(k1, v4.w, a1.w);
            }
            // every thread read its own rows of hs above; all reads of hs in this
            // chunk (v_new) finished before the last barrier
            *reinterpret_cast<float4 *>(&hs[kk0 * kBV + hn0]) = a0;
            *reinterpret_cast<float4 *>(&hs[(kk0 + 1) * kBV + hn0]) = a1;
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
    float *hs = Ps + kChunk * 65;      // [K][64] (rows read as float4)
    float *vs = hs + K * 64;           // [64][64]
    // [64][V + 1] fp32 o rows (output stage only), sharing its space with the
    // per-channel g [64][K + 1], which is not read once o rows are written
    float *os = vs + kChunk * 64;
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
    // Thread (ti, tj) owns rows 4 ti .. 4 ti + 3 and columns 4 tj .. 4 tj + 3 of
    // each 64 x 64 product: eight shared loads (or five with a float4) per
    // sixteen products.
    const int i0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
    {
        float acc[4][4] = {};
        if (c0 <= i0 + 3 && i0 < n) {   // tiles wholly above the diagonal stay 0
            const float *kb = pc_fz ? gk : ks;
            for (int kk = 0; kk < K; ++kk) {
                float qv[4], kv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    qv[r] = qs[(i0 + r) * KP + kk];
                    kv[r] = kb[(c0 + r) * KP + kk];
                }
                if (pc && !pc_fz) {
                    float gq[4], gj[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        gq[r] = gk[(i0 + r) * KP + kk];
                        gj[r] = gk[(c0 + r) * KP + kk];
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            acc[r][cc] = fmaf(qv[r] * kv[cc], expf(gq[r] - gj[cc]), acc[r][cc]);
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) acc[r][cc] = fmaf(qv[r], kv[cc], acc[r][cc]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int i = i0 + r, j = c0 + cc;
                float val = 0.f;
                if (j <= i && i < n) val = pc ? acc[r][cc] : acc[r][cc] * expf(gs[i] - gs[j]);
                Ps[i * 65 + j] = val;
            }
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
        for (int idx = tid; idx < K * 16; idx += kThreads) {
            const int kk = idx >> 4, n4 = (idx & 15) * 4;
            *reinterpret_cast<float4 *>(&hs[kk * 64 + n4]) = *reinterpret_cast<const float4 *>(
                &h_ws[hslot + static_cast<int64_t>(kk) * V + v0 + n4]);
        }
#pragma unroll 8
        for (int idx = tid; idx < kChunk * 16; idx += kThreads) {
            const int j = idx >> 4, n4 = (idx & 15) * 4;
            *reinterpret_cast<float4 *>(&vs[j * 64 + n4]) = *reinterpret_cast<const float4 *>(
                &vn_ws[tok(b, t0 + j, h, T_pad, H) * V + v0 + n4]);
        }
        __syncthreads();
        if (i0 < n) {
            float inter[4][4] = {}, intra[4][4] = {};
            for (int kk = 0; kk < K; ++kk) {
                const float4 h4 = *reinterpret_cast<const float4 *>(&hs[kk * 64 + c0]);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float qv = qs[(i0 + r) * KP + kk];
                    inter[r][0] = fmaf(qv, h4.x, inter[r][0]);
                    inter[r][1] = fmaf(qv, h4.y, inter[r][1]);
                    inter[r][2] = fmaf(qv, h4.z, inter[r][2]);
                    inter[r][3] = fmaf(qv, h4.w, inter[r][3]);
                }
            }
            // P is 0 above the diagonal and past n, so the tile's last row bounds j
            const int jmax = min(n, i0 + 4);
            for (int j = 0; j < jmax; ++j) {
                const float4 v4 = *reinterpret_cast<const float4 *>(&vs[j * 64 + c0]);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float pv = Ps[(i0 + r) * 65 + j];
                    intra[r][0] = fmaf(pv, v4.x, intra[r][0]);
                    intra[r][1] = fmaf(pv, v4.y, intra[r][1]);
                    intra[r][2] = fmaf(pv, v4.z, intra[r][2]);
                    intra[r][3] = fmaf(pv, v4.w, intra[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                if (i >= n) break;
                const float e = expf(gs[i]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const float oi = scale * (e * inter[r][cc] + intra[r][cc]);
                    if (gate)
                        os[i * OP + v0 + c0 + cc] = oi;
                    else
                        store_as(&o[tok(b, t0 + i, h, Tn, H) * V + v0 + c0 + cc], oi);
                }
            }
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
    return sizeof(float) * (kChunk * (K + 1) + 2 * kChunk * 65 + kChunk * 64 +
                            (pc ? kChunk * (K + 1) : 0));
}
size_t chunk_h_smem(int K, bool pc) {
    return sizeof(float) * (K * kBV + 2 * kChunk * (K + 1) + kChunk * kBV +
                            (pc ? kChunk * (K + 1) : 0));
}
size_t chunk_o_smem(int K, int V, bool normed, bool pc) {
    const int tail = std::max(normed ? kChunk * (V + 1) : 0, pc ? kChunk * (K + 1) : 0);
    return sizeof(float) * (2 * kChunk * (K + 1) + kChunk * 65 + K * 64 + kChunk * 64 + tail);
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
