// Tensor-core path of the chunked gated delta rule forward for bf16 q, k, v.
//
// Two kernels, following the "WarpDrive" page's pipeline (kernel 5
// recompute_w_u takes the chunk's WY matrix A as given; kernels 3 chunk_fwd_h
// and 4 chunk_fwd_o follow it):
//   1. gdn_wy_tc_kernel (gdn_tc_wy.cu): A diag(beta) for every chunk, in
//      parallel over all chunks, to a bf16 workspace [B, T, H, 64].
//   2. gdn_fused_tc_kernel (this file): recompute_w_u, chunk_fwd_h and
//      chunk_fwd_o fused. One CTA owns one (b, h, 64-wide V tile) and walks the
//      chunks in order with its [K, 64] slice of the state in registers (fp32)
//      and in shared memory (bf16, the MMA operand); h, w, u and v_new never
//      reach HBM.
//
// Per chunk (C = 64 tokens), D_* accumulators in tensor memory:
//   TMA      q, k [64 x K], the v tile [64 x 64], A diag(beta) [64 x 64] (rows past T read 0)
//   MMA_QK   D_QK = q k^T
//   epi P    P_ij = scale (q_i.k_j) exp(g_i - g_j), i >= j  -> bf16 operand
//            k_hat = exp(g) * k                             -> bf16 operand
//   MMA_W    D_W = A diag(beta) k_hat   (= w)    MMA_U  D_U = A diag(beta) v (= u)
//   MMA_QH   D_QH = q h
//   epi W    w -> bf16 operand
//   MMA_X    D_U += (-w) h            (= v_new, negated-A MMA)
//   epi X    v_new and v_new * exp(g_last - g_t) -> bf16 operands
//   MMA_PV   D_PV = P v_new           MMA_H  D_H = k^T (v_new * exp(g_last - g_t))
//   epi H    h = h * exp(g_last) + D_H (fp32 registers), bf16 copy for the next chunk
//   epi O    o = scale exp(g_t) D_QH + D_PV -> bf16 -> TMA store
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kTcThreads = 128;
constexpr int kTcBV = 64;
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait

// Shared-memory map (bytes from a 1024-aligned base). Regions reused within a
// chunk list every role they take, in order.
template <int K>
struct TcLayout {
    static constexpr int KB = K / 64;                        // 64-feature blocks
    static constexpr uint32_t kKQ = 0;                       // per block: k rows 0-63 | q rows 0-63
    static constexpr uint32_t kVT = kKQ + KB * 16384;        // v tile -> o staging
    static constexpr uint32_t kAP = kVT + 8192;              // A diag(beta) -> v_new
    static constexpr uint32_t kAU = kAP + 8192;              // v_gated
    static constexpr uint32_t kPS = kAU + 8192;              // P
    static constexpr uint32_t kWS = kPS + 8192;              // k_hat -> w (K/64 blocks of 8 KB)
    static constexpr uint32_t kHS = kWS + KB * 8192;         // h bf16 [K rows x 64]
    static constexpr uint32_t kMisc = kHS + K * 128;         // g, barriers
    static constexpr uint32_t kBytes = kMisc + 1024;
};

// TMEM columns (one 256-column allocation).
constexpr uint32_t kColW = 0, kColPV = 0, kColH = 64, kColQK = 128, kColU = 128, kColQH = 192;

template <int K>
__global__ void __launch_bounds__(kTcThreads, 1)
gdn_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ g,
                    const float *__restrict__ h0, float *__restrict__ h_final, int T, int H, int V,
                    float scale, uint32_t *status) {
    using Lay = TcLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *g_s = reinterpret_cast<float *>(sm + Lay::kMisc);   // g (0 past T)
    float *eg_s = g_s + 64;                                      // exp(g)
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
        prefetch_tmap(&tm_a);
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
            mbar_arrive_expect_tx(bar_tma, KB * 16384 + 8192 + 8192);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                tma_load_4d(sm + Lay::kKQ + kb * 16384, &tm_k, bar_tma, kb * 64, h, t0, b);
                tma_load_4d(sm + Lay::kKQ + kb * 16384 + 8192, &tm_q, bar_tma, kb * 64, h, t0, b);
            }
            tma_load_4d(sm + Lay::kVT, &tm_v, bar_tma, vt * kTcBV, h, t0, b);
            tma_load_4d(sm + Lay::kAP, &tm_a, bar_tma, 0, h, t0, b);
        }
        if (tid < 64) {
            float gv = 0.f;
            if (tid < n) gv = g[(static_cast<int64_t>(b) * T + t0 + tid) * H + h];
            g_s[tid] = gv;
            eg_s[tid] = tid < n ? __expf(gv) : 0.f;
        }
        fail |= !mbar_wait(bar_tma, ph_tma, kWaitNs);
        ph_tma ^= 1;
        if (__syncthreads_or(fail)) break;

        // ---- MMA_QK: q k^T (M = 64)
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks) {
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem + kColQK, smem_desc(s_kq + off + 8192, 16, 1024, kLayoutSw128),
                         smem_desc(s_kq + off, 16, 1024, kLayoutSw128), id, ks > 0);
            }
            mma_commit(bar_mma);
        }
        // ---- k_hat = exp(g) k while the MMA runs (same swizzled positions)
#pragma unroll
        for (int it = 0; it < KB * 4; ++it) {
            const int idx = tid + it * kTcThreads;           // 16-byte chunk of k
            const int kb = idx >> 9, rem = idx & 511, row = rem >> 3, ch = rem & 7;
            const uint32_t off = sw128(row, ch * 16);
            const uint4 raw = ld_shared_v4(sm + Lay::kKQ + kb * 16384 + off);
            const float s = eg_s[row];
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16(w4[e]);
                o4[e] = pack_bf16(f.x * s, f.y * s);
            }
            st_shared_v4(sm + Lay::kWS + kb * 8192 + off, o4[0], o4[1], o4[2], o4[3]);
        }
        fail |= !mbar_wait(bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (__syncthreads_or(fail)) break;
        tc_fence_after_sync();

        // ---- epilogue P (bf16, K-major rows)
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            uint32_t r[16];
            tmem_ld16(tmem + kColQK + lane_off + blk * 16, r);
            tmem_wait_ld();
            if (row64 >= 0) {
                const float gi = g_s[row64];
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = blk * 16 + e;
                    v[e] = (j <= row64) ? scale * __uint_as_float(r[e]) * __expf(gi - g_s[j]) : 0.f;
                }
                st_bf16x8(sm + Lay::kPS + sw128(row64, blk * 32), v);
                st_bf16x8(sm + Lay::kPS + sw128(row64, blk * 32 + 16), v + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---- MMA_W, MMA_U, MMA_QH
        if (tid == 0) {
            tc_fence_after_sync();
            constexpr uint32_t idW = idesc_bf16(64, K, false, true);
            constexpr uint32_t id64 = idesc_bf16(64, 64, false, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColW, smem_desc(s_ap + ks * 32, 16, 1024, kLayoutSw128),
                         smem_desc(s_ws + ks * 2048, 8192, 1024, kLayoutSw128), idW, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + kColU, smem_desc(s_ap + ks * 32, 16, 1024, kLayoutSw128),
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
            const float so = (row64 >= 0) ? scale * eg_s[row64] : 0.f;
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

// Stage export: A diag(beta) bf16 [B, T, H, 64] -> fp32 [B, T_pad, H, 64] (pad rows 0).
__global__ void export_abeta_kernel(const __nv_bfloat16 *__restrict__ src, float *__restrict__ dst,
                                    int B, int T, int T_pad, int H) {
    const int64_t n = static_cast<int64_t>(B) * T_pad * H * 64;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / 64;   // (b, t, h) in the padded layout
        const int hh = static_cast<int>(row % H);
        const int64_t bt = row / H;
        const int t = static_cast<int>(bt % T_pad), bb = static_cast<int>(bt / T_pad);
        dst[i] = t < T ? __bfloat162float(src[((static_cast<int64_t>(bb) * T + t) * H + hh) * 64 + i % 64])
                       : 0.f;
    }
}

template <int K>
cudaError_t launch_fused(const Args &a, const void *abeta, cudaStream_t s) {
    CUtensorMap mq, mk, mv, ma, mo;
    if (!make_tmap_bthx(&mq, a.q, K, a.H, a.T, a.B) || !make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mv, a.v, a.V, a.H, a.T, a.B) ||
        !make_tmap_bthx(&ma, abeta, 64, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mo, a.o, a.V, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem = static_cast<int>(TcLayout<K>::kBytes + 1024);
    cudaError_t e = cudaFuncSetAttribute(gdn_fused_tc_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gdn_fused_tc_kernel<K><<<dim3(a.V / kTcBV, a.H, a.B), kTcThreads, smem, s>>>(
        mq, mk, mv, ma, mo, a.g, a.h0, a.h_final, a.T, a.H, a.V, a.scale, a.status);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int K, int V, gdn_dtype dtype) {
    return dtype == GDN_BF16 && (K == 64 || K == 128) && V % kTcBV == 0 && V >= kTcBV;
}

size_t tc_workspace_bytes(int B, int T, int H, int, int) {
    return align_up(static_cast<size_t>(B) * T * H * 64 * sizeof(__nv_bfloat16));
}

int tc_launches(const char **names, int max_names) {
    static const char *const kNames[2] = {"gdn_wy_tc_kernel", "gdn_fused_tc_kernel"};
    for (int i = 0; names && i < 2 && i < max_names; ++i) names[i] = kNames[i];
    return 2;
}

cudaError_t tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m) {
    cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    if ((e = m.mark(0, s)) != cudaSuccess) return e;
    if ((e = wy_tc_forward(a, ws, s)) != cudaSuccess) return e;
    if ((e = m.mark(1, s)) != cudaSuccess) return e;
    e = (a.K == 128) ? launch_fused<128>(a, ws, s) : launch_fused<64>(a, ws, s);
    if (e != cudaSuccess) return e;
    return m.mark(2, s);
}

cudaError_t tc_export_abeta(const Args &a, const void *ws, float *dst, cudaStream_t s) {
    export_abeta_kernel<<<304, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(ws), dst, a.B, a.T,
                                           a.T_pad, a.H);
    return cudaGetLastError();
}

}  // namespace gdn
