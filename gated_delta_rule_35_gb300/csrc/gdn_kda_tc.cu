// Per-channel (KDA) decay on the tensor cores: the chunked form of the
// "KdaSplit" page's recurrence, in which every token decays each state row d
// by its own factor exp(gamma_t,d) before the delta-rule read and write.
//
// With g the chunk-local cumulative log decay (a K-vector per token) a chunk
// of 64 tokens entered with state h gives
//   L_ij = beta_i sum_d k_id k_jd exp(g_id - g_jd)         (j < i)
//   A    = (I + L)^-1,  Ab = A diag(beta)
//   w    = Ab (k * exp(g)),  u = Ab v,  v_new = u - w h
//   P_ij = scale sum_d q_id k_jd exp(g_id - g_jd)           (j <= i)
//   o    = scale (q * exp(g)) h + P v_new
//   h'   = diag(exp(g_last)) h + (k * exp(g_last - g))^T v_new
// Substituting v_new into o gives o = PA v + Q' h with PA = P Ab and
// Q' = scale (q * exp(g)) - PA (k * exp(g)), so the forward kernel gets v_new
// and o of a chunk from one stacked M = 128 accumulator,
//   [v_new; o] = [Ab; PA] v + [-w; Q'] h,
// and its chain per chunk is that product, the v_new copy, the state-update
// product and the state update.
//
// gdn_kda_prep_tc_kernel (one CTA per chunk and head) builds from q, k, g and
// beta: X1 = [Ab | PA] (bf16 [B, T, H, 128]), X2 = [-w | Q'] (bf16
// [B, T, H, 2K]), KH = k * exp(g_last - g) (bf16 [B, T, H, K]) and the chunk's
// decay exp(g_last) (fp32 [B, NT, H, K]):
//   operands  kp = k exp(g - r), qp = q exp(g - r), km = k exp(r - g), r = g_last / 2
//   MMA 1     [G; S] = [kp; qp] km^T    (G_ij = sum_d k_id k_jd exp(g_id - g_jd), S with q_i)
//   epi       L = diag(beta) G (strictly lower, fp32), P = scale S (lower, bf16)
//   SIMT      A = (I + L)^-1 by forward substitution, one column per thread (fp32)
//   MMA 2     [. ; PA] = [Ab; P] Ab
//   MMA 3     [w; PA ke] = [Ab; PA] ke,  ke = k exp(g)
//   epi       -w and Q' = q_hat - PA ke, TMA stores
// With r = g_last / 2 and non-positive log decays every factor lies within
// exp(+-|g_last| / 2), so the factored products are exact up to rounding while
// every channel has |g_last| <= 160; a chunk with a stronger decay takes L and P
// from one exponential per term on the CUDA cores instead (the masked entries
// of the factored product may overflow; they are replaced, never multiplied).
//
// gdn_kda_fwd_tc_kernel (one CTA per 64 V columns of a head) runs the chunk
// loop: the fp32 state sits in registers, one K row per thread, and its bf16
// copy in shared memory is the B operand of the next chunk's product. With
// the gated RMSNorm output stage a head's V tiles run as one cluster that
// exchanges each o row's sum of squares.
#include "gdn_internal.h"
#include "tc_sync.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kKdaThreads = 128;
constexpr uint64_t kKdaWaitNs = 1000000000ull;
constexpr float kFactorLimit = 160.f;   // |g_last| up to which the products are factored


__device__ __forceinline__ void st_bf16(unsigned char *p, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float ld_bf16(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

// ================================================================= prep kernel
template <int K>
struct KdaPrepLayout {
    static constexpr int KB = K / 64;
    // Per 64-feature block (16 KB): rows 0-63 the k tile, rows 64-127 the q
    // tile, as loaded. With the factored products they become [kp; qp] in
    // place (MMA 1's A), then [ke; qp] (ke: MMA 3's B) and [ke; Q'] (Q' staged
    // for its store); otherwise [ke; q_hat], then [ke; Q'].
    static constexpr uint32_t kKQ = 0;
    // km (K-major, MMA 1's B), then KH in place (staged for its store), then -w
    static constexpr uint32_t kM = KB * 16384;
    static constexpr uint32_t kAP = kM + KB * 8192;        // [Ab; P], then [Ab; PA]
    static constexpr uint32_t kLStride = 68;               // L rows, 16-byte aligned (fp32)
    // g (fp32 [64][K]), then L (fp32 [64][kLStride])
    static constexpr uint32_t kG = kAP + 16384;
    static constexpr uint32_t kGBytes = (64 * K > 64 * kLStride) ? 64 * K * 4 : 64 * kLStride * 4;
    // beta, row factors of q and k (64 each), r and exp(r) (K each)
    static constexpr uint32_t kMisc = kG + kGBytes;
    static constexpr uint32_t kBar = kMisc + (3 * 64 + 2 * K) * 4;
    static constexpr uint32_t kBytes = kBar + 64;
};

// Helpers of the prep kernel's exact path (one exponential per term), kept out
// of line: it runs only for chunks whose decay is too strong for the factored
// products, and inline its code sat among the hot path's (the prep kernel
// 0.127 -> 0.123 ms on B4 H16 T2048 out of line).
template <int KB>
__device__ __forceinline__ void kda_item(int it, int &i, int &kb, int &j) {
    j = it & 7;
    kb = (it >> 3) % KB;
    i = it / (8 * KB);
}
__device__ __forceinline__ void kda_unpack8(const uint4 u, float f, float (&x)[8]) {
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 p = unpack_bf16(w4[e]);
        x[2 * e] = p.x * f;
        x[2 * e + 1] = p.y * f;
    }
}
__device__ __forceinline__ void kda_load8(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), bb = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = bb.x, x[5] = bb.y, x[6] = bb.z, x[7] = bb.w;
}
template <int K>
__device__ __noinline__ void kda_exact_lp(unsigned char *sm, int tid, float scale) {
    using Lay = KdaPrepLayout<K>;
    constexpr int KB = K / 64;
    float *g_s = reinterpret_cast<float *>(sm + Lay::kG);
    float *L_s = g_s;
    float *b_s = reinterpret_cast<float *>(sm + Lay::kMisc);
    float *fq_s = b_s + 64, *fk_s = b_s + 128, *r_s = b_s + 192;
    // one exponential per term (exponents <= 0 on the kept entries):
    // threads 0-63 row i of L, threads 64-127 row i of P
    const int i = tid & 63;
    const bool is_p = tid >= 64;
    const float fi = is_p ? fq_s[i] * scale : fk_s[i] * b_s[i];
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
#pragma unroll 1
    for (int d = 0; d < K; ++d) {
        const uint32_t col = Lay::kKQ + (d >> 6) * 16384, byte = 2 * (d & 63);
        const float xi = ld_bf16(sm + col + (is_p ? 8192 : 0) + sw128(i, byte));
        const float gi = g_s[i * K + d];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            const bool keep = is_p ? (j <= i) : (j < i);
            const float kj = ld_bf16(sm + col + sw128(j, byte)) * fk_s[j];
            const float t = xi * kj * __expf(gi - g_s[j * K + d]);
            acc[j] += keep ? t : 0.f;   // a dropped term may overflow; it is never used
        }
    }
    if (is_p) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = fi * acc[ch * 8 + e];
            st_bf16x8(sm + Lay::kAP + sw128(64 + i, ch * 16), v);
        }
    }
    __syncthreads();   // every read of the raw tiles done
    // ke = k exp(g) and q_hat = scale q exp(g) in place, KH beside them
    for (int it = tid; it < 64 * KB * 8; it += kKdaThreads) {
        int ii, kb, j;
        kda_item<KB>(it, ii, kb, j);
        const int d0 = kb * 64 + 8 * j;
        const uint32_t ck = Lay::kKQ + kb * 16384 + sw128(ii, 16 * j);
        float kv[8], qv[8], gv[8], rv[8];
        kda_unpack8(ld_shared_v4(sm + ck), fk_s[ii], kv);
        kda_unpack8(ld_shared_v4(sm + ck + 8192), fq_s[ii] * scale, qv);
        kda_load8(g_s + ii * K + d0, gv);
        kda_load8(r_s + d0, rv);
        float kh[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float eg = __expf(gv[e]);
            kh[e] = kv[e] * __expf(2.f * rv[e] - gv[e]);
            kv[e] *= eg;
            qv[e] *= eg;
        }
        st_bf16x8(sm + ck, kv);
        st_bf16x8(sm + ck + 8192, qv);
        st_bf16x8(sm + Lay::kM + kb * 8192 + sw128(ii, 16 * j), kh);
    }
    __syncthreads();   // every read of g done before L overwrites it
    if (!is_p) {
#pragma unroll
        for (int j = 0; j < 64; ++j) L_s[i * Lay::kLStride + j] = fi * acc[j];
    }
}

constexpr uint32_t kPrepColG = 0, kPrepColPA = 64, kPrepColW = 128, kPrepTmemCols = 256;

// FRONT: the instance that may take the front-end flags; calls without them
// run one with none of that code (fewer instructions to fetch: the prep
// kernel 0.133 -> 0.128 ms on B4 H16 T2048).
template <int K, bool FRONT>
// Two CTAs per SM (98.8 KB of shared memory and 256 TMEM columns each at K = 128).
__global__ void __launch_bounds__(kKdaThreads, 2)
gdn_kda_prep_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_x1, const __grid_constant__ CUtensorMap tm_x2,
                       const __grid_constant__ CUtensorMap tm_kh, const float *__restrict__ g,
                       const float *__restrict__ beta, float *__restrict__ dec_out, float scale, int T,
                       int H, int NT, uint32_t *status, int flags) {
    using Lay = KdaPrepLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *g_s = reinterpret_cast<float *>(sm + Lay::kG);
    float *L_s = g_s;
    float *b_s = reinterpret_cast<float *>(sm + Lay::kMisc);
    float *fq_s = b_s + 64, *fk_s = b_s + 128, *r_s = b_s + 192, *er_s = r_s + K;
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + Lay::kBar);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int t0 = c * 64, n = min(64, T - t0);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kPrepTmemCols);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    // the forward kernel may be scheduled as SMs free up
    griddep_launch_dependents();
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, 2 * KB * 8192);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load_4d(sm + Lay::kKQ + kb * 16384, &tm_k, bar_tma, kb * 64, h, t0, b);
            tma_load_4d(sm + Lay::kKQ + kb * 16384 + 8192, &tm_q, bar_tma, kb * 64, h, t0, b);
        }
    }
    const bool raw_g = FRONT && (flags & GDN_FLAG_RAW_G), l2norm = FRONT && (flags & GDN_FLAG_QK_L2NORM);
    const int64_t row0 = (static_cast<int64_t>(b) * T + t0) * H + h;   // (b, t0, h)
    {
        // g tile, every load issued before the first store; rows >= n read as 0
        // (their q and k rows are zero too, so they add nothing)
        constexpr int kPer = 64 * (K / 4) / kKdaThreads;
        float4 x[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = tid + u * kKdaThreads, i = e / (K / 4), d4 = e % (K / 4);
            x[u] = i < n ? *reinterpret_cast<const float4 *>(g + (row0 + static_cast<int64_t>(i) * H) * K + d4 * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = tid + u * kKdaThreads, i = e / (K / 4), d4 = e % (K / 4);
            *reinterpret_cast<float4 *>(g_s + i * K + d4 * 4) = x[u];
        }
    }
    if (tid < 64) b_s[tid] = tid < n ? beta[row0 + static_cast<int64_t>(tid) * H] : 0.f;
    __syncthreads();
    if (raw_g && tid < K) {
        // chunk-local inclusive sum, one channel per thread
        float acc = 0.f;
        for (int i = 0; i < 64; ++i) {
            acc += g_s[i * K + tid];
            g_s[i * K + tid] = acc;
        }
    }
    __syncthreads();
    bool fz = true;
    if (tid < K) {
        const float gl = g_s[(n - 1) * K + tid];
        r_s[tid] = 0.5f * gl;
        er_s[tid] = __expf(0.5f * gl);
        fz = fabsf(gl) <= kFactorLimit;
        dec_out[((static_cast<int64_t>(b) * NT + c) * H + h) * K + tid] = __expf(gl);
    }
    fz = __syncthreads_and(fz);
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t s_ap = smem_u32(sm + Lay::kAP);
    // (the barriers were initialised before the block-wide barriers above)
    bool fail = !mbar_wait(bar_tma, 0, kKdaWaitNs);
    uint32_t phase = 0;
    auto mma_wait = [&]() {
        fail |= !mbar_wait(bar_mma, phase, kKdaWaitNs);
        phase ^= 1;
        tc_fence_after_sync();
    };
    // item it of the 64 x K / 8 chunks of 8 features: row, block, chunk
    auto item = [](int it, int &i, int &kb, int &j) {
        j = it & 7;
        kb = (it >> 3) % KB;
        i = it / (8 * KB);
    };
    auto unpack8 = [](const uint4 u, float f, float (&x)[8]) {
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 p = unpack_bf16(w4[e]);
            x[2 * e] = p.x * f;
            x[2 * e + 1] = p.y * f;
        }
    };
    auto load8 = [](const float *p, float (&x)[8]) {
        const float4 a = *reinterpret_cast<const float4 *>(p), bb = *reinterpret_cast<const float4 *>(p + 4);
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = bb.x, x[5] = bb.y, x[6] = bb.z, x[7] = bb.w;
    };

    do {
        if (__syncthreads_or(fail)) break;
        {
            // row factors: 1, or 1 / sqrt(|x_i|^2 + eps) of the row as loaded
            const int i = tid & 63;
            const uint32_t base = Lay::kKQ + (tid < 64 ? 8192 : 0);
            float f = 1.f;
            if (l2norm) {
                float ss = 0.f;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float x[8];
                        unpack8(ld_shared_v4(sm + base + kb * 16384 + sw128(i, 16 * j)), 1.f, x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                    }
                f = rsqrtf(ss + kL2NormEps);
            }
            (tid < 64 ? fq_s : fk_s)[i] = f;
        }
        __syncthreads();
        if (fz) {
            // ---- kp, qp in place, km beside them
            for (int it = tid; it < 64 * KB * 8; it += kKdaThreads) {
                int i, kb, j;
                item(it, i, kb, j);
                const int d0 = kb * 64 + 8 * j;
                const uint32_t ck = Lay::kKQ + kb * 16384 + sw128(i, 16 * j);
                float kv[8], qv[8], gv[8], rv[8];
                unpack8(ld_shared_v4(sm + ck), fk_s[i], kv);
                unpack8(ld_shared_v4(sm + ck + 8192), fq_s[i], qv);
                load8(g_s + i * K + d0, gv);
                load8(r_s + d0, rv);
                float kp[8], qp[8], km[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = gv[e] - rv[e];
                    const float up = __expf(x), dn = __expf(-x);
                    kp[e] = kv[e] * up;
                    qp[e] = qv[e] * up;
                    km[e] = kv[e] * dn;
                }
                st_bf16x8(sm + ck, kp);
                st_bf16x8(sm + ck + 8192, qp);
                st_bf16x8(sm + Lay::kM + kb * 8192 + sw128(i, 16 * j), km);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                // [G; S] = [kp; qp] km^T
                tc_fence_after_sync();
                const uint32_t id = idesc_bf16(128, 64, false, false);
                const TileDesc da(smem_u32(sm + Lay::kKQ), 16, 1024), db(smem_u32(sm + Lay::kM), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    mma_bf16(tmem + kPrepColG, da.at((ks >> 2) * 16384 + (ks & 3) * 32),
                             db.at((ks >> 2) * 8192 + (ks & 3) * 32), id, ks > 0);
                mma_commit(bar_mma);
            }
            mma_wait();
            if (__syncthreads_or(fail)) break;
            // rows 0-63 of the accumulator (warps 0-1): G -> L; rows 64-127: S -> P
            const int i = tid & 63;
            if (tid < 64) {
                const float bi = b_s[i];
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    float v[16];
                    tmem_ld16f(tmem + lane_off + kPrepColG + blk * 16, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        L_s[i * Lay::kLStride + blk * 16 + e] = (blk * 16 + e < i) ? bi * v[e] : 0.f;
                }
            } else {
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    float v[16];
                    tmem_ld16f(tmem + lane_off + kPrepColG + blk * 16, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = (blk * 16 + e <= i) ? scale * v[e] : 0.f;
                    st_bf16x8(sm + Lay::kAP + sw128(64 + i, blk * 32), v);
                    st_bf16x8(sm + Lay::kAP + sw128(64 + i, blk * 32 + 16), v + 8);
                }
            }
            // MMA 1 has read kp and km: ke = kp exp(r) = k exp(g) and
            // KH = km exp(r) = k exp(g_last - g), both in place
            for (int it = tid; it < 64 * KB * 8; it += kKdaThreads) {
                int ii, kb, j;
                item(it, ii, kb, j);
                const int d0 = kb * 64 + 8 * j;
                float ev[8], x[8];
                load8(er_s + d0, ev);
                const uint32_t ck = Lay::kKQ + kb * 16384 + sw128(ii, 16 * j);
                const uint32_t cm = Lay::kM + kb * 8192 + sw128(ii, 16 * j);
                unpack8(ld_shared_v4(sm + ck), 1.f, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= ev[e];
                st_bf16x8(sm + ck, x);
                unpack8(ld_shared_v4(sm + cm), 1.f, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= ev[e];
                st_bf16x8(sm + cm, x);
            }
        } else {
            // one exponential per term, out of line (rare: some |g_last| > 160)
            kda_exact_lp<K>(sm, tid, scale);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_store_4d(&tm_kh, sm + Lay::kM + kb * 8192, kb * 64, h, t0, b);
            bulk_commit_group();
        }
        // ---- A = (I + L)^-1, column j per thread: (I + L) a = e_j top to bottom,
        // each row's sum in four interleaved partial sums
        if (tid < 64) {
            const int j = tid;
            float a[64];
            a[0] = j == 0 ? 1.f : 0.f;
#pragma unroll
            for (int i = 1; i < 64; ++i) {
                const float *Li = L_s + i * Lay::kLStride;
                float s0 = i == j ? 1.f : 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                for (int m = 0; m < (i & ~3); m += 4) {
                    const float4 l = *reinterpret_cast<const float4 *>(Li + m);
                    s0 = fmaf(-l.x, a[m], s0);
                    s1 = fmaf(-l.y, a[m + 1], s1);
                    s2 = fmaf(-l.z, a[m + 2], s2);
                    s3 = fmaf(-l.w, a[m + 3], s3);
                }
#pragma unroll
                for (int m = i & ~3; m < i; ++m) s0 = fmaf(-Li[m], a[m], s0);
                a[i] = (s0 + s1) + (s2 + s3);
            }
            // Ab = A diag(beta): column j, rows 0-63 of [Ab; P]
            const float bj = b_s[j];
#pragma unroll
            for (int i = 0; i < 64; ++i) st_bf16(sm + Lay::kAP + sw128(i, 2 * j), a[i] * bj);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        // ---- [. ; PA] = [Ab; P] Ab (Ab read again as the B operand, rows along N)
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, false, true);
            const TileDesc da(s_ap, 16, 1024), db(s_ap, 8192, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tmem + kPrepColPA, da.at(ks * 32), db.at(ks * 2048), id, ks > 0);
            mma_commit(bar_mma);
        }
        mma_wait();
        if (__syncthreads_or(fail)) break;
        if (tid >= 64) {
            const int i = tid - 64;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                tmem_ld16f(tmem + lane_off + kPrepColPA + blk * 16, v);
                st_bf16x8(sm + Lay::kAP + sw128(64 + i, blk * 32), v);
                st_bf16x8(sm + Lay::kAP + sw128(64 + i, blk * 32 + 16), v + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        // ---- X1 out; [w; PA ke] = [Ab; PA] ke (ke: rows 0-63 of each feature block)
        if (tid == 0) {
            tc_fence_after_sync();
            tma_store_4d(&tm_x1, sm + Lay::kAP, 0, h, t0, b);
            tma_store_4d(&tm_x1, sm + Lay::kAP + 8192, 64, h, t0, b);
            bulk_commit_group();
            const uint32_t id = idesc_bf16(128, K, false, true);
            const TileDesc da(s_ap, 16, 1024), db(smem_u32(sm + Lay::kKQ), 16384, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tmem + kPrepColW, da.at(ks * 32), db.at(ks * 2048), id, ks > 0);
            mma_commit(bar_mma);
        }
        mma_wait();
        if (tid == 0) bulk_wait_group_read0();   // KH's staging is read before -w replaces it
        if (__syncthreads_or(fail)) break;
        {
            // -w (rows 0-63) and Q' = q_hat - PA ke (rows 64-127; q_hat = scale
            // exp(r) qp with the factored operands)
            const int i = tid & 63;
#pragma unroll 1
            for (int blk = 0; blk < K / 16; ++blk) {
                float v[16];
                tmem_ld16f(tmem + lane_off + kPrepColW + blk * 16, v);
                const int kb = blk >> 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t byte = (blk & 3) * 32 + half * 16;
                    float x[8];
                    if (tid < 64) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = -v[half * 8 + e];
                        st_bf16x8(sm + Lay::kM + kb * 8192 + sw128(i, byte), x);
                    } else {
                        const uint32_t cq = Lay::kKQ + kb * 16384 + 8192 + sw128(i, byte);
                        float qf[8];
                        if (fz) {
                            load8(er_s + blk * 16 + half * 8, qf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) qf[e] *= scale;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) qf[e] = 1.f;
                        }
                        unpack8(ld_shared_v4(sm + cq), 1.f, x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = fmaf(qf[e], x[e], -v[half * 8 + e]);
                        st_bf16x8(sm + cq, x);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                tma_store_4d(&tm_x2, sm + Lay::kM + kb * 8192, kb * 64, h, t0, b);
                tma_store_4d(&tm_x2, sm + Lay::kKQ + kb * 16384 + 8192, K + kb * 64, h, t0, b);
            }
            bulk_commit_group();
        }
    } while (false);
    if (tid == 0) {
        bulk_wait_group_read0();   // only the shared sources must outlive the CTA
        if (fail) atomicOr(status, 2u);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ================================================================= forward kernel
template <int K>
struct KdaFwdLayout {
    static constexpr int KB = K / 64;
    static constexpr uint32_t kX1 = 0;                   // [Ab; PA] (16 KB)
    static constexpr uint32_t kX2 = 16384;               // [-w; Q'] per feature block, 16 KB each
    static constexpr uint32_t kKH = kX2 + KB * 16384;    // KH, rows = tokens, 8 KB per feature block
    static constexpr uint32_t kV = kKH + KB * 8192;      // v, 64 tokens x 64 columns
    static constexpr uint32_t kStage = kV + 8192;
    static constexpr uint32_t kHB = 2 * kStage;           // state, bf16, rows = features (K x 64)
    static constexpr uint32_t kVN = kHB + KB * 8192;      // v_new, bf16 (64 x 64)
    // barriers: full[2], mma, ht, norm[2] (output stage), vn_ready, o_taken,
    // h_ready, drain; then the TMEM address and the abort flag
    static constexpr uint32_t kBar = kVN + 8192;
    // output stage: row sums of squares, [2 chunk slots][4 ranks][64 rows]
    static constexpr uint32_t kRed = kBar + 128;
    static constexpr uint32_t kBytes = kRed;
    static constexpr uint32_t kBytesGated = kRed + 2 * 4 * 64 * 4;
};

constexpr uint32_t kFwdColD = 0, kFwdColH = 64, kFwdTmemCols = 128;

// sigmoid(z) = (1 + tanh(z / 2)) / 2 with the hardware tanh (one special-function
// instruction; absolute error below 3e-4, far inside the bf16 rounding of o).
__device__ __forceinline__ float kda_sigmoid(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}

// GATED: the output stage (gated RMSNorm over the head's V columns), the V
// tiles of a head running as one cluster of V / 64 CTAs that exchange each
// row's sum of squares.
template <int K, bool GATED>
__global__ void __launch_bounds__(kKdaThreads, 1)
gdn_kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_x1, const __grid_constant__ CUtensorMap tm_x2,
                      const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_v,
                      __nv_bfloat16 *__restrict__ o, const float *__restrict__ dec,
                      const float *__restrict__ h0, float *__restrict__ h_final, int T, int H, int V, int NT,
                      uint32_t *status, const __nv_bfloat16 *__restrict__ gate, const float *__restrict__ norm_w,
                      float norm_eps, uint64_t wlim, int stall) {
    using Lay = KdaFwdLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::kBar);   // [2]
    uint64_t *mma_bar = full + 2, *ht_bar = full + 3, *norm_bar = full + 4;   // norm_bar[2]
    // v_new rows in shared memory (warps 0-1), o rows out of the accumulator
    // (warps 2-3), the state's bf16 copy written (its K rows)
    uint64_t *vn_ready = full + 6, *o_taken = full + 7, *h_ready = full + 8;
    uint64_t *drain = full + 9;   // every MMA issued is done (before TMEM is freed)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full + 10);
    volatile uint32_t *abort = tmem_slot + 1;
    const int nrank = GATED ? V / 64 : 0;

    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(tmem_slot, kFwdTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mma_bar, 1);
        mbar_init(ht_bar, 1);
        // output stage: one local arrival (with the expected bytes) per chunk;
        // the row sums of every CTA of the cluster arrive as transactions
        if (GATED) {
            mbar_init(&norm_bar[0], 1);
            mbar_init(&norm_bar[1], 1);
        }
        mbar_init(vn_ready, 64);
        mbar_init(o_taken, 64);
        mbar_init(h_ready, K);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    // the state: row d = tid of the K x 64 block of columns [64 vt, 64 vt + 64)
    const int d = tid;
    const int64_t srow = ((static_cast<int64_t>(b) * H + h) * K + d) * V + vt * 64;
    float hr[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) hr[e] = 0.f;
    if (h0 && d < K) {
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(h0 + srow + e);
            hr[e] = x.x, hr[e + 1] = x.y, hr[e + 2] = x.z, hr[e + 3] = x.w;
        }
    }
    auto write_state = [&]() {
        if (d < K) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) st_bf16x8(sm + Lay::kHB + sw128(d, ch * 16), hr + ch * 8);
        }
    };
    write_state();
    // everything below reads the prep kernel's output
    griddep_wait();
    auto load_stage = [&](int c) {
        unsigned char *st = sm + (c & 1) * Lay::kStage;
        const int t0 = c * 64;
        mbar_arrive_expect_tx(&full[c & 1], Lay::kStage);
        tma_load_4d(st + Lay::kX1, &tm_x1, &full[c & 1], 0, h, t0, b);
        tma_load_4d(st + Lay::kX1 + 8192, &tm_x1, &full[c & 1], 64, h, t0, b);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load_4d(st + Lay::kX2 + kb * 16384, &tm_x2, &full[c & 1], kb * 64, h, t0, b);
            tma_load_4d(st + Lay::kX2 + kb * 16384 + 8192, &tm_x2, &full[c & 1], K + kb * 64, h, t0, b);
            tma_load_4d(st + Lay::kKH + kb * 8192, &tm_kh, &full[c & 1], kb * 64, h, t0, b);
        }
        tma_load_4d(st + Lay::kV, &tm_v, &full[c & 1], vt * 64, h, t0, b);
    };
    // thread 0: chunks whose loads were issued, and whose landing was waited for
    // (test hook: with `stall` chunk 0's loads are withheld, so the first wait
    // on them runs out after wlim and every role leaves its loop)
    int loaded = 0, landed = stall ? 1 : 0;
    if (tid == 0) {
        if (!stall) load_stage(0);
        if (NT > 1) load_stage(1);
        loaded = NT > 1 ? 2 : 1;
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    // the cluster's barriers are initialised before any CTA sends to them
    if (GATED) cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // [v_new; o] = [Ab; PA] v (first) + [-w; Q'] h
    constexpr uint32_t idD = idesc_bf16(128, 64, false, true);
    constexpr uint32_t idHT = idesc_bf16(128, 64, true, true);
    auto issue_a = [&](int s) {
        const uint32_t st = s_base + s * Lay::kStage;
        const TileDesc da(st + Lay::kX1, 16, 1024), db(st + Lay::kV, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tmem + kFwdColD, da.at(ks * 32), db.at(ks * 2048), idD, ks > 0);
    };
    auto issue_b = [&](int s) {
        const uint32_t st = s_base + s * Lay::kStage;
        const TileDesc da(st + Lay::kX2, 16, 1024), db(s_base + Lay::kHB, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks)
            mma_bf16_k<true>(tmem + kFwdColD, da.at((ks >> 2) * 16384 + (ks & 3) * 32), db.at(ks * 2048), idD);
    };
    // dH = KH^T v_new: KH read M-major (features along M; with K = 64 the upper
    // 64 rows repeat the lower ones and are not read)
    auto issue_ht = [&](int s) {
        const uint32_t st = s_base + s * Lay::kStage;
        const TileDesc da(st + Lay::kKH, K == 128 ? 8192 : 0, 1024), db(s_base + Lay::kVN, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tmem + kFwdColH, da.at(ks * 2048), db.at(ks * 2048), idHT, ks > 0);
    };

    // The chunk loop runs on barrier hand-offs rather than block-wide
    // barriers, so that the o rows (and the output stage) stay off the chain:
    //   thread 0   h_ready(c) -> [Ab; PA] v (unless issued already) + [-w; Q'] h
    //              -> commit mma; vn_ready(c) -> KH^T v_new -> commit ht;
    //              o_taken(c) -> the next chunk's [Ab; PA] v
    //   warps 0-1  mma(c) -> v_new rows to shared memory -> vn_ready
    //   warps 2-3  mma(c) -> o rows into registers -> o_taken
    //   rows < K   ht(c) -> state update -> bf16 copy -> h_ready(c + 1)
    //   warps 2-3  then the o rows' output stage and store
    // No waiter can fall two phases behind its barrier: each barrier's next
    // phase needs, through this chain, the waiter's own earlier arrival. Every
    // wait is bounded and gives up once any role has given up (abort flag).
    const uint64_t lim = wlim;
    if (d < K) {
        // the entering state's copy (written above) for the first product
        fence_proxy_async_smem();
        mbar_arrive(h_ready);
    }
    bool ok = true;
    bool a_issued = false;
    for (int c = 0; c < NT; ++c) {
        const int s = c & 1;
        if (tid == 0) {
            ok = wait_bar(h_ready, c & 1, abort, lim) &&
                 (a_issued || wait_bar(&full[s], (c >> 1) & 1, abort, lim));
            if (ok) landed = c + 1;
            if (ok) {
                tc_fence_after_sync();
                if (!a_issued) issue_a(s);
                issue_b(s);
                mma_commit(mma_bar);
            }
            a_issued = false;
        }
        const float dv = d < K ? dec[((static_cast<int64_t>(b) * NT + c) * H + h) * K + d] : 0.f;
        if (!warp_all(ok && wait_bar(mma_bar, c & 1, abort, lim))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        float ov[64];   // warps 2-3: this thread's o row
        if (tid < 64) {
            // v_new row (token) tid -> the B operand of the state update
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                tmem_ld16f(tmem + lane_off + kFwdColD + blk * 16, v);
                st_bf16x8(sm + Lay::kVN + sw128(tid, blk * 32), v);
                st_bf16x8(sm + Lay::kVN + sw128(tid, blk * 32 + 16), v + 8);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(vn_ready);
        } else {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                tmem_ld16f(tmem + lane_off + kFwdColD + blk * 16, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) ov[blk * 16 + e] = v[e];
            }
            tc_fence_before_sync();
            mbar_arrive(o_taken);
        }
        if (tid == 0) {
            ok = wait_bar(vn_ready, c & 1, abort, lim);
            if (ok) {
                tc_fence_after_sync();
                issue_ht(s);
                mma_commit(ht_bar);
            }
            // the next chunk's [Ab; PA] v once this chunk's o rows are out of
            // the accumulator
            if (ok && c + 1 < NT) {
                ok = wait_bar(o_taken, c & 1, abort, lim) &&
                     wait_bar(&full[s ^ 1], ((c + 1) >> 1) & 1, abort, lim);
                if (ok) landed = c + 2;
                if (ok) {
                    tc_fence_after_sync();
                    issue_a(s ^ 1);
                    a_issued = true;
                }
            }
        }
        if (d < K) {
            if (!warp_all(ok && wait_bar(ht_bar, c & 1, abort, lim))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            // the stage's last reader (the state update) is done
            if (tid == 0 && c + 2 < NT) {
                load_stage(c + 2);
                loaded = c + 3;
            }
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                tmem_ld16f(tmem + lane_off + kFwdColH + blk * 16, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) hr[blk * 16 + e] = fmaf(dv, hr[blk * 16 + e], v[e]);
            }
            write_state();
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(h_ready);
        }
        if (tid >= 64) {
            const int i = tid - 64;
            if (GATED) {
                // Output stage: the row's sum of squares goes to every CTA of
                // the cluster (slot c % 2, entry = rank) as asynchronous stores
                // that complete bytes of the receiver's norm_bar; with every
                // sum in, the row is normalised and gated. A slot is next
                // written for chunk c + 2, after the sender has waited for this
                // CTA's sums of chunk c + 1, which are sent only after this CTA
                // has read its slot for chunk c.
                const int slot = c & 1;
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 64; ++e) ss = fmaf(ov[e], ov[e], ss);
                const uint32_t red = s_base + Lay::kRed + ((slot * 4 + vt) * 64 + i) * 4;
                const uint32_t nb = smem_u32(&norm_bar[slot]);
                if (tid == 64) mbar_arrive_expect_tx(&norm_bar[slot], nrank * 64 * 4);
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (r < nrank) st_async_cluster_f32(mapa_shared(red, r), ss, mapa_shared(nb, r));
                if (!warp_all(wait_bar_cluster(&norm_bar[slot], (c >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                const float *sums = reinterpret_cast<const float *>(sm + Lay::kRed) + slot * 256;
                float tot = 0.f;
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (r < nrank) tot += sums[r * 64 + i];
                const float rstd = rsqrtf(tot / V + norm_eps);
                const float *wv = norm_w + vt * 64;
                const int t = c * 64 + i;
                const uint4 *zrow = reinterpret_cast<const uint4 *>(
                    gate + ((static_cast<int64_t>(b) * T + min(t, T - 1)) * H + h) * V + vt * 64);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 z4 = zrow[q];
                    const uint32_t w4[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 z = unpack_bf16(w4[e]);
                        const int j = q * 8 + 2 * e;
                        ov[j] *= rstd * wv[j] * kda_sigmoid(z.x);
                        ov[j + 1] *= rstd * wv[j + 1] * kda_sigmoid(z.y);
                    }
                }
            }
            // o row (token) i: the thread's own 128 bytes of the row
            if (c * 64 + i < T) {
                __nv_bfloat16 *dst = o + ((static_cast<int64_t>(b) * T + c * 64 + i) * H + h) * V + vt * 64;
#pragma unroll
                for (int q = 0; q < 8; ++q) store_bf16x8_global(dst + q * 8, ov + q * 8);
            }
        }
    }
    const bool fail = !ok || *abort;
    if (!fail && d < K) {
#pragma unroll
        for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4 *>(h_final + srow + e) = make_float4(hr[e], hr[e + 1], hr[e + 2], hr[e + 3]);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        if (!ok || *abort) atomicOr(status, 2u);
        // after a failure: the loads still in flight land and every MMA issued
        // completes (bounded) before the CTA's shared and tensor memory go
        for (int k = landed; k < loaded; ++k) mbar_wait(&full[k & 1], (k >> 1) & 1, kKdaWaitNs);
        mma_commit(drain);
        mbar_wait(drain, 0, kKdaWaitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    // no CTA of a cluster leaves while another may still write its shared memory
    if (GATED) cluster_sync();
    if (warp == 0) tmem_dealloc(tmem, kFwdTmemCols);
}

struct KdaWs {
    void *x1, *x2, *kh;
    float *dec;
};

size_t rows_of(int B, int T, int H) { return static_cast<size_t>(B) * T * H; }

KdaWs kda_carve(void *ws, int B, int T, int H, int K) {
    char *p = static_cast<char *>(ws);
    KdaWs w;
    const size_t rows = rows_of(B, T, H);
    w.x1 = p;
    p += align_up(rows * 128 * 2);
    w.x2 = p;
    p += align_up(rows * 2 * K * 2);
    w.kh = p;
    p += align_up(rows * K * 2);
    w.dec = reinterpret_cast<float *>(p);
    return w;
}

template <int K>
cudaError_t launch_kda(const Args &a, void *ws, cudaStream_t s, const Marks &m) {
    const KdaWs w = kda_carve(ws, a.B, a.T, a.H, K);
    CUtensorMap mq, mk, mx1, mx2, mkh, mv;
    if (!make_tmap_bthx(&mq, a.q, K, a.H, a.T, a.B) || !make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mx1, w.x1, 128, a.H, a.T, a.B) || !make_tmap_bthx(&mx2, w.x2, 2 * K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mkh, w.kh, K, a.H, a.T, a.B) || !make_tmap_bthx(&mv, a.v, a.V, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem_p = static_cast<int>(KdaPrepLayout<K>::kBytes + 1024);
    const bool gated = a.gate != nullptr;
    const auto fwd = gated ? gdn_kda_fwd_tc_kernel<K, true> : gdn_kda_fwd_tc_kernel<K, false>;
    const int smem_f =
        static_cast<int>((gated ? KdaFwdLayout<K>::kBytesGated : KdaFwdLayout<K>::kBytes) + 1024);
    const auto prep = (a.flags & (GDN_FLAG_RAW_G | GDN_FLAG_QK_L2NORM)) ? gdn_kda_prep_tc_kernel<K, true>
                                                                        : gdn_kda_prep_tc_kernel<K, false>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_f);
    if (e != cudaSuccess) return e;
    if ((e = m.mark(0, s)) != cudaSuccess) return e;
    prep<<<dim3(a.NT, a.H, a.B), kKdaThreads, smem_p, s>>>(
        mq, mk, mx1, mx2, mkh, a.g, a.beta, w.dec, a.scale, a.T, a.H, a.NT, a.status, a.flags);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = m.mark(1, s)) != cudaSuccess) return e;
    // The forward grid may start while the prep kernel's last CTAs run (its
    // setup and state load overlap them); it waits for their output before
    // its first load. Only with more than one wave: otherwise its CTAs would
    // hold SMs the prep kernel still needs.
    const long long ctas = static_cast<long long>(a.V / 64) * a.H * a.B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.V / 64, a.H, a.B);
    cfg.blockDim = dim3(kKdaThreads);
    cfg.dynamicSmemBytes = smem_f;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (ctas > tc_sm_count()) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (gated) {
        // a head's V tiles form one cluster for the output stage's exchange
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = a.V / 64;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr++].val.clusterDim.z = 1;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    const float *dec = w.dec;
    const float *h0 = a.h0;
    float *hf = a.h_final;
    int T = a.T, H = a.H, V = a.V, NT = a.NT;
    uint32_t *status = a.status;
    const __nv_bfloat16 *gate = static_cast<const __nv_bfloat16 *>(a.gate);
    const float *norm_w = a.norm_w;
    float norm_eps = a.norm_eps;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);
    uint64_t wlim = kKdaWaitNs;
    int stall = 0;
    if (const uint64_t armed = take_armed_stall()) {
        wlim = armed;
        stall = 1;
    }
    void *args[] = {&mx1, &mx2, &mkh, &mv, &o,       &dec,  &h0,       &hf,   &T,     &H, &V,
                    &NT,  &status, &gate, &norm_w, &norm_eps, &wlim, &stall};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fwd), args);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return m.mark(2, s);
}

}  // namespace

const char *const kKdaTcKernelNames[kKdaTcLaunches] = {"gdn_kda_prep_tc_kernel", "gdn_kda_fwd_tc_kernel"};

size_t kda_tc_workspace_bytes(int B, int T, int H, int K, int) {
    const size_t rows = rows_of(B, T, H);
    return align_up(rows * 128 * 2) + align_up(rows * 2 * K * 2) + align_up(rows * K * 2) +
           align_up(static_cast<size_t>(B) * num_chunks(T) * H * K * sizeof(float));
}

cudaError_t kda_tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m) {
    return a.K == 128 ? launch_kda<128>(a, ws, s, m) : launch_kda<64>(a, ws, s, m);
}

}  // namespace gdn
