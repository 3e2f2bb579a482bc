// Tensor-core path of the chunked gated delta rule forward for bf16 q, k, v.
//
// One kernel fuses the whole pipeline of the "WarpDrive" page (kernel 5
// recompute_w_u with its WY matrix, kernel 3 chunk_fwd_h, kernel 4
// chunk_fwd_o). One CTA owns one (b, h, 64-wide V tile) and walks the chunks in
// order with the [K, 64] slice of the state in registers (fp32) and in shared
// memory (bf16, the MMA operand), so neither h, A, w, u nor v_new ever reaches
// HBM: per token it reads q, k, v, g, beta and writes o.
//
// Per chunk (C = 64 tokens), with D_* accumulators in tensor memory:
//   TMA      q, k [64 x K] and the v tile [64 x 64] (rows past T read as 0)
//   MMA_G    D_G[128 x 64] = [k; q] k^T                      (Gram and q k^T)
//   epi G    L_ij = beta_i G_ij exp(g_i - g_j), i > j (fp32, smem)
//            P_ij = scale (q_i.k_j) exp(g_i - g_j), i >= j (bf16 operand)
//   inverse  A = (I + L)^-1: 16x16 diagonal blocks by forward substitution,
//            then two block-merge levels, fp32 on the CUDA cores
//            A' = A diag(beta exp(g)), A'' = A diag(beta) (bf16 operands)
//   MMA_W    D_W = A' k   (= w)       MMA_U  D_U = A'' v (= u)
//   MMA_QH   D_QH = q h
//   epi W    w -> bf16 operand
//   MMA_X    D_U += (-w) h            (= v_new, negated-A MMA)
//   epi X    v_new and v_new * exp(g_last - g_t) -> bf16 operands
//   MMA_PV   D_PV = P v_new           MMA_H  D_H = k^T (v_new * exp(g_last - g_t))
//   epi H    h = h * exp(g_last) + D_H (fp32 registers), bf16 copy for the next chunk
//   epi O    o = scale exp(g_t) D_QH + D_PV -> bf16 -> TMA store
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "gdn_internal.h"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kTcThreads = 128;
constexpr int kTcBV = 64;
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait

// Shared-memory map (bytes from a 1024-aligned base). Regions reused within a
// chunk are listed with every role they take, in order.
template <int K>
struct TcLayout {
    static constexpr int KB = K / 64;                        // 64-feature blocks
    static constexpr uint32_t kKQ = 0;                       // per block: k rows 0-63 | q rows 0-63
    static constexpr uint32_t kVT = kKQ + KB * 16384;        // v tile -> o staging
    static constexpr uint32_t kAP = kVT + 8192;              // inverse temps -> A' -> v_new
    static constexpr uint32_t kAU = kAP + 8192;              // A'' -> v_gated
    static constexpr uint32_t kPS = kAU + 8192;              // P
    static constexpr uint32_t kWS = kPS + 8192;              // L/A fp32 (16 KB) -> w bf16
    static constexpr uint32_t kHS = kWS + 16384;             // h bf16 [K rows x 64]
    static constexpr uint32_t kMisc = kHS + K * 128;         // g, beta exp(g), beta, barriers
    static constexpr uint32_t kBytes = kMisc + 1024;
};

// TMEM columns (one 256-column allocation).
constexpr uint32_t kColW = 0, kColPV = 0, kColH = 64, kColG = 128, kColU = 128, kColQH = 192;

// Strictly-lower fp32 64x64 matrix with an XOR swizzle on the column so that
// both row-parallel and column-parallel accesses are free of bank conflicts.
struct Tri64 {
    float *p;
    __device__ __forceinline__ float &operator()(int i, int j) const {
        return p[i * 64 + (j ^ (i & 31))];
    }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void st_shared_v4(unsigned char *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}
// Eight fp32 values -> one 16-byte chunk of bf16 at `dst`.
__device__ __forceinline__ void st_bf16x8(unsigned char *dst, const float *v) {
    st_shared_v4(dst, pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                 pack_bf16(v[6], v[7]));
}

// A = (I + L)^-1 in place in `L` (strictly lower on entry, unit lower on exit),
// 128 threads. `tmp` holds >= 32*33 floats.
__device__ __forceinline__ void invert_unit_lower64(const Tri64 &L, float *tmp, int tid) {
    // 1) the four 16x16 diagonal blocks: thread (blk, c) solves (I + L_bb) x = e_c
    float x[16];
    const int blk = tid >> 4, c = tid & 15, base = blk * 16;
    if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 15; ++j)
#pragma unroll
            for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-L(base + i, base + j), x[j], x[i]);
    }
    __syncthreads();
    if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) L(base + i, base + c) = x[i];
    }
    __syncthreads();
    // 2) blocks (1,0) and (3,2): X_21 = -X_22 L_21 X_11
    {
        const int p = tid >> 6, idx = tid & 63, i = idx >> 2, j0 = (idx & 3) * 4;
        const int rb = 16 * (2 * p + 1), cb = 32 * p;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float l = L(rb + i, cb + k);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(l, L(cb + k, cb + j0 + e), acc[e]);
        }
        float *T1 = tmp + p * 16 * 17;
#pragma unroll
        for (int e = 0; e < 4; ++e) T1[i * 17 + j0 + e] = acc[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float xh = L(rb + i, rb + k);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(xh, T1[k * 17 + j0 + e], acc[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) L(rb + i, cb + j0 + e) = -acc[e];
    }
    __syncthreads();
    // 3) bottom-left 32x32: X_BL = -X_BR L_BL X_TL
    {
        const int i = tid >> 2, j0 = (tid & 3) * 8;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float l = L(32 + i, k);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(l, L(k, j0 + e), acc[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) tmp[i * 33 + j0 + e] = acc[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float xb = L(32 + i, 32 + k);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(xb, tmp[k * 33 + j0 + e], acc[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) L(32 + i, j0 + e) = -acc[e];
    }
    __syncthreads();
}

template <int K>
__global__ void __launch_bounds__(kTcThreads, 1)
gdn_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const float *__restrict__ g, const float *__restrict__ beta,
                    const float *__restrict__ h0, float *__restrict__ h_final, int T, int H, int V,
                    float scale, uint32_t *status) {
    using Lay = TcLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *g_s = reinterpret_cast<float *>(sm + Lay::kMisc);   // g
    float *s1_s = g_s + 64;                                      // beta exp(g)
    float *s2_s = g_s + 128;                                     // beta
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + Lay::kMisc + 768);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = (T + 63) / 64;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

    const uint32_t s_kq = smem_u32(sm + Lay::kKQ), s_vt = smem_u32(sm + Lay::kVT);
    const uint32_t s_ap = smem_u32(sm + Lay::kAP), s_au = smem_u32(sm + Lay::kAU);
    const uint32_t s_ps = smem_u32(sm + Lay::kPS), s_ws = smem_u32(sm + Lay::kWS);
    const uint32_t s_hs = smem_u32(sm + Lay::kHS);
    const Tri64 L{reinterpret_cast<float *>(sm + Lay::kWS)};

    // Row of the state this thread owns: the M = 128 accumulator puts row i in
    // TMEM lane i; the M = 64 one puts row i in lane 32 (i / 16) + i % 16.
    const int feat = (K == 128) ? tid : (lane < 16 ? warp * 16 + lane : -1);
    const int row64 = lane < 16 ? warp * 16 + lane : -1;   // row of M = 64 accumulators
    const int64_t state_off = (static_cast<int64_t>(b) * H + h) * K * V + vt * kTcBV;
    float hreg[kTcBV];
#pragma unroll
    for (int j = 0; j < kTcBV; ++j)
        hreg[j] = (feat >= 0 && h0) ? h0[state_off + static_cast<int64_t>(feat) * V + j] : 0.f;
    if (feat >= 0) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) st_bf16x8(sm + Lay::kHS + sw128(feat, ch * 16), &hreg[ch * 8]);
    }
    fence_proxy_async_smem();

    uint32_t ph_tma = 0, ph_mma = 0;
    bool fail = false;
    for (int c = 0; c < NT; ++c) {
        const int t0 = c * 64, n = min(64, T - t0);
        if (tid == 0) {
            bulk_wait_group_read0();   // the previous o store has left the v-tile region
            mbar_arrive_expect_tx(bar_tma, KB * 16384 + 8192);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                tma_load_4d(sm + Lay::kKQ + kb * 16384, &tm_k, bar_tma, kb * 64, h, t0, b);
                tma_load_4d(sm + Lay::kKQ + kb * 16384 + 8192, &tm_q, bar_tma, kb * 64, h, t0, b);
            }
            tma_load_4d(sm + Lay::kVT, &tm_v, bar_tma, vt * kTcBV, h, t0, b);
        }
        if (tid < 64) {
            float gv = 0.f, bv = 0.f;
            if (tid < n) {
                const int64_t r = (static_cast<int64_t>(b) * T + t0 + tid) * H + h;
                gv = g[r];
                bv = beta[r];
            }
            g_s[tid] = gv;
            s1_s[tid] = bv * __expf(gv);
            s2_s[tid] = bv;
        }
        fail |= !mbar_wait(bar_tma, ph_tma, kWaitNs);
        ph_tma ^= 1;
        if (__syncthreads_or(fail)) break;

        // ---- MMA_G: [k; q] k^T
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks) {
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem + kColG, smem_desc(s_kq + off, 16, 1024, kLayoutSw128),
                         smem_desc(s_kq + off, 16, 1024, kLayoutSw128), id, ks > 0);
            }
            mma_commit(bar_mma);
        }
        fail |= !mbar_wait(bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (__syncthreads_or(fail)) break;
        tc_fence_after_sync();

        // ---- epilogue G: L (fp32) and P (bf16)
        {
            const int i = tid & 63;
            const float gi = g_s[i];
            const float bi = s2_s[i];
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t r[16];
                tmem_ld16(tmem + kColG + lane_off + blk * 16, r);
                tmem_wait_ld();
                float v[16];
                if (tid < 64) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = blk * 16 + e;
                        v[e] = (j < i) ? bi * __uint_as_float(r[e]) * __expf(gi - g_s[j]) : 0.f;
                        L(i, j) = v[e];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = blk * 16 + e;
                        v[e] = (j <= i) ? scale * __uint_as_float(r[e]) * __expf(gi - g_s[j]) : 0.f;
                    }
                    st_bf16x8(sm + Lay::kPS + sw128(i, blk * 32), v);
                    st_bf16x8(sm + Lay::kPS + sw128(i, blk * 32 + 16), v + 8);
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();

        // ---- A = (I + L)^-1, then A' = A diag(beta exp(g)), A'' = A diag(beta)
        invert_unit_lower64(L, reinterpret_cast<float *>(sm + Lay::kAP), tid);
        {
            const int i = tid >> 1, half = tid & 1;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int j0 = half * 32 + ch * 8;
                float a1[8], a2[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float a = L(i, j0 + e);
                    a1[e] = a * s1_s[j0 + e];
                    a2[e] = a * s2_s[j0 + e];
                }
                st_bf16x8(sm + Lay::kAP + sw128(i, j0 * 2), a1);
                st_bf16x8(sm + Lay::kAU + sw128(i, j0 * 2), a2);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();

        // ---- MMA_W, MMA_U, MMA_QH
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t idW = idesc_bf16(64, K, false, true);
            constexpr uint32_t id64 = idesc_bf16(64, 64, false, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColW, smem_desc(s_ap + ks * 32, 16, 1024, kLayoutSw128),
                         smem_desc(s_kq + ks * 2048, 16384, 1024, kLayoutSw128), idW, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColU, smem_desc(s_au + ks * 32, 16, 1024, kLayoutSw128),
                         smem_desc(s_vt + ks * 2048, 8192, 1024, kLayoutSw128), id64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                mma_bf16(tmem + kColQH,
                         smem_desc(s_kq + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32, 16, 1024,
                                   kLayoutSw128),
                         smem_desc(s_hs + ks * 2048, K * 128, 1024, kLayoutSw128), id64, ks > 0);
            mma_commit(bar_mma);
        }
        fail |= !mbar_wait(bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (__syncthreads_or(fail)) break;
        tc_fence_after_sync();

        // ---- epilogue W: w -> bf16 operand (K-major, K/64 blocks of 8 KB)
#pragma unroll
        for (int blk = 0; blk < K / 16; ++blk) {
            uint32_t r[16];
            tmem_ld16(tmem + kColW + lane_off + blk * 16, r);
            tmem_wait_ld();
            if (row64 >= 0) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
                const int f0 = blk * 16;
                unsigned char *base = sm + Lay::kWS + (f0 >> 6) * 8192;
                st_bf16x8(base + sw128(row64, (f0 & 63) * 2), v);
                st_bf16x8(base + sw128(row64, (f0 & 63) * 2 + 16), v + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---- MMA_X: D_U += (-w) h  ->  v_new
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t idX = idesc_bf16(64, 64, false, true, true);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                mma_bf16(tmem + kColU,
                         smem_desc(s_ws + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kLayoutSw128),
                         smem_desc(s_hs + ks * 2048, K * 128, 1024, kLayoutSw128), idX, 1);
            mma_commit(bar_mma);
        }
        fail |= !mbar_wait(bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (__syncthreads_or(fail)) break;
        tc_fence_after_sync();

        // ---- epilogue X: v_new and v_gated -> bf16 operands (token rows, V contiguous)
        const float g_last = g_s[n - 1];
        {
            const float gate = (row64 >= 0 && row64 < n) ? __expf(g_last - g_s[row64]) : 0.f;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t r[16];
                tmem_ld16(tmem + kColU + lane_off + blk * 16, r);
                tmem_wait_ld();
                if (row64 >= 0) {
                    float v[16], vg[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        v[e] = __uint_as_float(r[e]);
                        vg[e] = v[e] * gate;
                    }
                    st_bf16x8(sm + Lay::kAP + sw128(row64, blk * 32), v);
                    st_bf16x8(sm + Lay::kAP + sw128(row64, blk * 32 + 16), v + 8);
                    st_bf16x8(sm + Lay::kAU + sw128(row64, blk * 32), vg);
                    st_bf16x8(sm + Lay::kAU + sw128(row64, blk * 32 + 16), vg + 8);
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();

        // ---- MMA_PV: P v_new ; MMA_H: k^T v_gated
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t id64 = idesc_bf16(64, 64, false, true);
            constexpr uint32_t idH = idesc_bf16(K, 64, true, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColPV, smem_desc(s_ps + ks * 32, 16, 1024, kLayoutSw128),
                         smem_desc(s_ap + ks * 2048, 8192, 1024, kLayoutSw128), id64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColH, smem_desc(s_kq + ks * 2048, 16384, 1024, kLayoutSw128),
                         smem_desc(s_au + ks * 2048, 8192, 1024, kLayoutSw128), idH, ks > 0);
            mma_commit(bar_mma);
        }
        fail |= !mbar_wait(bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (__syncthreads_or(fail)) break;
        tc_fence_after_sync();

        // ---- epilogue H: h = h exp(g_last) + k^T v_gated; bf16 copy for the next chunk
        {
            const float decay = __expf(g_last);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t r[16];
                tmem_ld16(tmem + kColH + lane_off + blk * 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    hreg[blk * 16 + e] = fmaf(hreg[blk * 16 + e], decay, __uint_as_float(r[e]));
            }
            if (feat >= 0) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_bf16x8(sm + Lay::kHS + sw128(feat, ch * 16), &hreg[ch * 8]);
            }
        }
        // ---- epilogue O: o = scale exp(g_t) q h + P v_new -> bf16 staging -> TMA store
        {
            const float so = (row64 >= 0) ? scale * __expf(g_s[row64]) : 0.f;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t rq[16], rp[16];
                tmem_ld16(tmem + kColQH + lane_off + blk * 16, rq);
                tmem_ld16(tmem + kColPV + lane_off + blk * 16, rp);
                tmem_wait_ld();
                if (row64 >= 0) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[e] = fmaf(so, __uint_as_float(rq[e]), __uint_as_float(rp[e]));
                    st_bf16x8(sm + Lay::kVT + sw128(row64, blk * 32), v);
                    st_bf16x8(sm + Lay::kVT + sw128(row64, blk * 32 + 16), v + 8);
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tma_store_4d(&tm_o, sm + Lay::kVT, vt * kTcBV, h, t0, b);
            bulk_commit_group();
        }
    }

    if (!fail && feat >= 0 && h_final) {
#pragma unroll
        for (int j = 0; j < kTcBV; ++j) h_final[state_off + static_cast<int64_t>(feat) * V + j] = hreg[j];
    }
    if (tid == 0) {
        bulk_wait_group0();
        if (fail) atomicOr(status, 1u);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [B, T, H, inner] bf16 viewed as a 4-D tensor (inner, H, T, B); box 64 x 1 x 64 x 1,
// 128-byte swizzle. Rows t >= T fall outside the tensor: loads read zeros and
// stores skip them.
bool make_map(CUtensorMap *m, const void *ptr, int inner, int H, int T, int B) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(inner) * 2,
                                   static_cast<cuuint64_t>(H) * inner * 2,
                                   static_cast<cuuint64_t>(T) * H * inner * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K>
cudaError_t launch_tc(const Args &a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, K, a.H, a.T, a.B) || !make_map(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_map(&mv, a.v, a.V, a.H, a.T, a.B) || !make_map(&mo, a.o, a.V, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem = static_cast<int>(TcLayout<K>::kBytes + 1024);
    cudaError_t e = cudaFuncSetAttribute(gdn_fused_tc_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gdn_fused_tc_kernel<K><<<dim3(a.V / kTcBV, a.H, a.B), kTcThreads, smem, s>>>(
        mq, mk, mv, mo, a.g, a.beta, a.h0, a.h_final, a.T, a.H, a.V, a.scale, a.status);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int K, int V, gdn_dtype dtype) {
    return dtype == GDN_BF16 && (K == 64 || K == 128) && V % kTcBV == 0 && V >= kTcBV;
}

size_t tc_workspace_bytes(int, int, int, int, int) { return 0; }

int tc_launches(const char **names, int max_names) {
    if (names && max_names > 0) names[0] = "gdn_fused_tc_kernel";
    return 1;
}

cudaError_t tc_forward(const Args &a, void *, cudaStream_t s, const Marks &m) {
    cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    if ((e = m.mark(0, s)) != cudaSuccess) return e;
    e = (a.K == 128) ? launch_tc<128>(a, s) : launch_tc<64>(a, s);
    if (e != cudaSuccess) return e;
    return m.mark(1, s);
}

}  // namespace gdn
