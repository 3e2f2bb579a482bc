// WY build on the tensor cores: for every 64-token chunk, the matrix
// A = (I + L)^-1 of the "WarpDrive" page's recompute_w_u (kernel 5 takes it as
// given), with L_ij = beta_i (k_i . k_j) exp(g_i - g_j) for i > j, written out as
// A diag(beta) in bf16 [B, T, H, 64].
//
// One CTA per (chunk, h, b); the chunks are independent, so the grid is as
// wide as the problem and several CTAs share an SM. Per chunk:
//   TMA     k [64 x K]
//   MMA     G = k k^T (M = 64)
//   epi     L rows (fp32): the four 16x16 diagonal blocks to shared memory; the
//           off-diagonal blocks as two bf16 operands N1 (blocks (1,0), (3,2))
//           and N2 (rows 32-63, columns 0-31)
//   SIMT    X = blockdiag of the inverted 16x16 diagonal blocks (forward
//           substitution in fp32)
//   MMA x4  level 1: Y1 = N1 X, Z1 = X Y1, A0 = X - Z1   (32x32 diagonal blocks)
//           level 2: Y2 = N2 A0, Z2 = A0 Y2, A = A0 - Z2
//           which is (I + L)^-1 because each off-diagonal part is nilpotent of
//           order two against its block-diagonal: (D + N)^-1 = D^-1 - D^-1 N D^-1.
//   epi     A diag(beta) -> bf16 -> TMA store
// The correction products run with bf16 operands and fp32 accumulation; the
// block-diagonal part and the subtractions stay fp32.
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kWyThreads = 128;
constexpr uint64_t kWyWaitNs = 1000000000ull;

template <int K>
struct WyLayout {
    static constexpr int KB = K / 64;
    static constexpr uint32_t kK = 0;                                  // k tile -> N1 | N2 -> out
    static constexpr uint32_t kKBytes = (KB * 8192 > 16384) ? KB * 8192 : 16384;
    static constexpr uint32_t kN1 = 0, kN2 = 8192, kOut = 0;
    static constexpr uint32_t kX = kKBytes;                            // X -> A0 (bf16)
    static constexpr uint32_t kY = kX + 8192;                          // Y1 -> Y2 (bf16)
    static constexpr uint32_t kLd = kY + 8192;                         // diag blocks fp32 [4][16][17]
    static constexpr uint32_t kMisc = kLd + 4 * 16 * 17 * 4;           // g, beta, bars
    static constexpr uint32_t kBytes = kMisc + 768;
};

template <int K>
__global__ void __launch_bounds__(kWyThreads, 3)
gdn_wy_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_a,
                 const float *__restrict__ g, const float *__restrict__ beta, int T, int H,
                 uint32_t *status) {
    using Lay = WyLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *Ld = reinterpret_cast<float *>(sm + Lay::kLd);
    float *g_s = reinterpret_cast<float *>(sm + Lay::kMisc);
    float *b_s = g_s + 64;
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + Lay::kMisc + 512);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = c * 64, n = min(64, T - t0);
    // Row of the M = 64 accumulator this thread reads (TMEM lane 32 (r/16) + r%16).
    const int r = lane < 16 ? warp * 16 + lane : -1;
    const int rb = r >> 4;   // 16-row block of r
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, KB * 8192);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
            tma_load_4d(sm + Lay::kK + kb * 8192, &tm_k, bar_tma, kb * 64, h, t0, b);
    }
    if (tid < 64) {
        float gv = 0.f, bv = 0.f;
        if (tid < n) {
            const int64_t row = (static_cast<int64_t>(b) * T + t0 + tid) * H + h;
            gv = g[row];
            bv = beta[row];
        }
        g_s[tid] = gv;
        b_s[tid] = bv;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t s_k = smem_u32(sm + Lay::kK), s_x = smem_u32(sm + Lay::kX),
                   s_y = smem_u32(sm + Lay::kY);
    uint32_t phase = 0;
    bool fail = !mbar_wait(bar_tma, 0, kWyWaitNs);

    // D = A_op * B_op with M = N = 64, both operands 64x64 bf16 tiles (A K-major,
    // B stored row-by-row along N), issued by one thread; everyone waits.
    auto mma64 = [&](uint32_t a, uint32_t bop, bool b_mn, int ksteps, uint32_t b_kstep) {
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t id = idesc_bf16(64, 64, false, b_mn);
            for (int ks = 0; ks < ksteps; ++ks) {
                const uint32_t a_off = (ks >> 2) * 8192 + (ks & 3) * 32;
                mma_bf16(tmem, smem_desc(a + a_off, 16, 1024, kLayoutSw128),
                         smem_desc(bop + (b_mn ? ks * 2048 : a_off), 8192, 1024, kLayoutSw128), id,
                         ks > 0);
            }
            (void)b_kstep;
            mma_commit(bar_mma);
        }
        fail |= !mbar_wait(bar_mma, phase, kWyWaitNs);
        phase ^= 1;
        tc_fence_after_sync();
    };
    // Loads this thread's accumulator row (64 fp32; meaningful when r >= 0).
    auto load_row = [&](float *v) {
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            uint32_t t[16];
            tmem_ld16(tmem + lane_off + blk * 16, t);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[blk * 16 + e] = __uint_as_float(t[e]);
        }
    };
    auto store_row_bf16 = [&](uint32_t region, const float *v) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) st_bf16x8(sm + region + sw128(r, ch * 16), v + ch * 8);
    };

    // ---- G = k k^T
    if (__syncthreads_or(fail)) goto done;
    mma64(s_k, s_k, false, K / 16, 0);
    if (__syncthreads_or(fail)) goto done;
    {
        float v[64];
        load_row(v);
        __syncthreads();   // every k-tile read done before N1 | N2 overwrite it
        if (r >= 0) {
            const float gr = g_s[r], br = b_s[r];
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = (j < r) ? br * v[j] * __expf(gr - g_s[j]) : 0.f;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
                if (blk == rb) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) Ld[(rb * 16 + (r & 15)) * 17 + e] = v[blk * 16 + e];
                }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const int jb = ch >> 1;   // 16-column block of this 8-column chunk
                const bool in1 = (rb == 1 && jb == 0) || (rb == 3 && jb == 2);
                const bool in2 = rb >= 2 && jb < 2;
                float n1[8], n2[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    n1[e] = in1 ? v[ch * 8 + e] : 0.f;
                    n2[e] = in2 ? v[ch * 8 + e] : 0.f;
                }
                st_bf16x8(sm + Lay::kN1 + sw128(r, ch * 16), n1);
                st_bf16x8(sm + Lay::kN2 + sw128(r, ch * 16), n2);
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    // ---- X: inverse of each 16x16 unit-lower diagonal block, column per thread
    {
        float x[16];
        const int blk = tid >> 4, col = tid & 15;
        float *Lb = Ld + blk * 16 * 17;
        if (tid < 64) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < 15; ++j)
#pragma unroll
                for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-Lb[i * 17 + j], x[j], x[i]);
        }
        __syncthreads();
        if (tid < 64) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Lb[i * 17 + col] = x[i];
        }
        __syncthreads();
    }
    float a0[64];   // this thread's row of X, then of A0 (fp32)
    if (r >= 0) {
#pragma unroll
        for (int j = 0; j < 64; ++j) a0[j] = ((j >> 4) == rb) ? Ld[(rb * 16 + (r & 15)) * 17 + (j & 15)] : 0.f;
        store_row_bf16(Lay::kX, a0);
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---- level 1: A0 = X - X (N1 X)
    mma64(smem_u32(sm + Lay::kN1), s_x, true, 4, 0);
    if (__syncthreads_or(fail)) goto done;
    {
        float v[64];
        load_row(v);
        if (r >= 0) store_row_bf16(Lay::kY, v);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    mma64(s_x, s_y, true, 4, 0);
    if (__syncthreads_or(fail)) goto done;
    {
        float v[64];
        load_row(v);
        if (r >= 0) {
#pragma unroll
            for (int j = 0; j < 64; ++j) a0[j] -= v[j];
            store_row_bf16(Lay::kX, a0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    // ---- level 2: A = A0 - A0 (N2 A0)
    mma64(smem_u32(sm + Lay::kN2), s_x, true, 4, 0);
    if (__syncthreads_or(fail)) goto done;
    {
        float v[64];
        load_row(v);
        if (r >= 0) store_row_bf16(Lay::kY, v);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    mma64(s_x, s_y, true, 4, 0);
    if (__syncthreads_or(fail)) goto done;
    {
        float v[64];
        load_row(v);
        if (r >= 0) {
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = (a0[j] - v[j]) * b_s[j];
            store_row_bf16(Lay::kOut, v);
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        tma_store_4d(&tm_a, sm + Lay::kOut, 0, h, t0, b);
        bulk_commit_group();
        bulk_wait_group0();
    }
done:
    if (tid == 0 && fail) atomicOr(status, 2u);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

template <int K>
cudaError_t launch_wy(const Args &a, void *abeta, cudaStream_t s) {
    CUtensorMap mk, ma;
    if (!make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) || !make_tmap_bthx(&ma, abeta, 64, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem = static_cast<int>(WyLayout<K>::kBytes + 1024);
    cudaError_t e = cudaFuncSetAttribute(gdn_wy_tc_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gdn_wy_tc_kernel<K><<<dim3(a.NT, a.H, a.B), kWyThreads, smem, s>>>(mk, ma, a.g, a.beta, a.T,
                                                                       a.H, a.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t wy_tc_forward(const Args &a, void *abeta, cudaStream_t s) {
    return a.K == 128 ? launch_wy<128>(a, abeta, s) : launch_wy<64>(a, abeta, s);
}

}  // namespace gdn
