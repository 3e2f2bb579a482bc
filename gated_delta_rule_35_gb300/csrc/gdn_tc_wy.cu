// WY build on the tensor cores: for every 64-token chunk, the matrix
// A = (I + L)^-1 of the "WarpDrive" page's recompute_w_u (kernel 5 takes it as
// given), with L_ij = beta_i (k_i . k_j) exp(g_i - g_j) for i > j, written out as
// A diag(beta) and A diag(beta exp(g)) in bf16 [B, T, H, 128] (columns 0-63
// and 64-127).
//
// One CTA per (chunk, h, b); the chunks are independent, so the grid is as
// wide as the problem and several CTAs share an SM. With X the inverse of the
// block diagonal of I + L (four 16x16 blocks), N1 its off-diagonal blocks
// (1,0) and (3,2), N2 its bottom-left 32x32 block:
//   A0 = (I + L_32x32 blocks)^-1 = X - X N1 X            (level 1)
//   A  = A0 - A0 N2 A0                                    (level 2)
// because each off-diagonal part squares to zero against its block diagonal:
// (D + N)^-1 = D^-1 - D^-1 N D^-1. Expanding level 2 with Y1 = N1 X and
// U = N2 X gives N2 A0 = U - U Y1, so after the Gram matrix only three tensor-
// core round trips remain, each a stacked M = 128 product:
//   MMA 1   G = k k^T                                     (M = 64)
//   epi     L (fp32 16x16 diagonal blocks, bf16 N1 | N2 stacked)
//   SIMT    X: forward substitution on the diagonal blocks (fp32)
//   MMA 2   [Y1; U] = [N1; N2] X
//   MMA 3   [A0; Y2] = [X; U] + [X; U] (-Y1)   (accumulator preloaded with X, keeps U)
//   MMA 4   A = A0 + A0 (-Y2)                   (accumulator keeps A0)
//   epi     A diag(beta), A diag(beta exp(g)) -> bf16 -> TMA store
// The correction products run with bf16 operands and fp32 accumulation; the
// block-diagonal part and the subtractions stay fp32 (in the accumulator).
//
// Front-end (problem flags): with GDN_FLAG_RAW_G the chunk's g is the inclusive
// sum of the raw per-token log decays, taken here and written to g_cum for the
// fused kernel; with GDN_FLAG_QK_L2NORM each k row's factor
// r_i = 1 / sqrt(|k_i|^2 + eps) is taken from the k tile and written to rk. The
// normalised rows never exist: L_ij gains r_i r_j and the second output's
// column scale gains r_j (w = A diag(beta exp(g)) diag(r) k), while the Gram
// MMA still reads the k tile as loaded.
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
    // k tile twice, [k; k] per 64-feature block (16 KB each), so that the Gram
    // product's rows land in both TMEM lane halves and all four warps form L.
    // After the Gram MMA the first 16 KB hold the stacked operand [N1; N2],
    // read only by the first merge product, and the next 16 KB [X; U].
    static constexpr uint32_t kK = 0, kKBlk = 16384;
    static constexpr uint32_t kN = 0;
    static constexpr uint32_t kXU = 16384;                 // [X; U] stacked, then A0 (bf16)
    // The fp32 diagonal blocks live in the U half of [X; U] until X is built
    // from them (U is written after the first merge product): each block's L
    // transposed ([16 columns][16 rows], blocks 272 floats apart, so that a
    // thread reads four rows of one column with one 16-byte load and the two
    // blocks of a warp sit on different banks), then X in place, row-major
    // with a stride of 17.
    static constexpr uint32_t kLd = kXU + 8192;
    // One 8 KB region in the [N2] half of [N1; N2], free once the first merge
    // product has read it: Y1, Y2 (read by the last product), and finally the
    // A diag(beta) staging of the TMA store.
    static constexpr uint32_t kY = kN + 8192;
    static constexpr uint32_t kOut = kY;
    // g, beta, beta exp(g) r, cf, r (64 floats each), a scan total; barriers
    static constexpr uint32_t kMisc = (KB * kKBlk > kXU + 16384) ? KB * kKBlk : kXU + 16384;
    static constexpr uint32_t kBar = kMisc + 1344;
    static constexpr uint32_t kBytes = kBar + 256;
    static_assert(16 * 17 * 4 * 4 <= 8192, "diagonal blocks fit the U half");
};

// FRONT: the instance that may take the front-end flags; the one without them
// has none of that code (a smaller kernel fetches fewer instructions: 0.4% of
// the B8 H64 T8192 step).
template <int K, bool FRONT>
// Six CTAs per SM (35.4 KB of shared memory and 64 TMEM columns each).
__global__ void __launch_bounds__(kWyThreads, 6)
gdn_wy_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_a,
                 const float *__restrict__ g, const float *__restrict__ beta, int T, int H,
                 uint32_t *status, int flags, float *__restrict__ g_cum, float *__restrict__ rk_out) {
    using Lay = WyLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *Ld = reinterpret_cast<float *>(sm + Lay::kLd);
    float *g_s = reinterpret_cast<float *>(sm + Lay::kMisc);
    float *b_s = g_s + 64;
    float *eb_s = g_s + 128;   // beta exp(g): the column scale of A diag(beta exp(g))
    // exp(g_ref - g_j) with g_ref = g_last / 2: with the row factor
    // beta_i exp(g_i - g_ref) it gives beta_i exp(g_i - g_j) without an
    // exponential per element, while |g_last| keeps both factors finite
    float *cf_s = g_s + 192;
    float *rk_s = g_s + 256;    // the k rows' normalisation factors (1 without it)
    float *tot_s = g_s + 320;   // raw-g scan: total of tokens 0-31
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + Lay::kBar);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = c * 64, n = min(64, T - t0);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    // the fused kernel that follows may be scheduled as SMs free up
    griddep_launch_dependents();
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, KB * 16384);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            // the second copy is served from L2
            tma_load_4d(sm + Lay::kK + kb * Lay::kKBlk, &tm_k, bar_tma, kb * 64, h, t0, b);
            tma_load_4d(sm + Lay::kK + kb * Lay::kKBlk + 8192, &tm_k, bar_tma, kb * 64, h, t0, b);
        }
    }
    const bool raw_g = FRONT && (flags & GDN_FLAG_RAW_G), l2norm = FRONT && (flags & GDN_FLAG_QK_L2NORM);
    const int64_t my_row = (static_cast<int64_t>(b) * T + t0 + tid) * H + h;
    float gv = 0.f, bv = 0.f;
    if (tid < n) {
        gv = g[my_row];
        bv = beta[my_row];
    }
    if (raw_g) {
        // inclusive sum over the chunk: tokens 0-31 in warp 0, 32-63 in warp 1
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, gv, off);
            if (lane >= off) gv += y;
        }
        if (tid == 31) *tot_s = gv;
        __syncthreads();
        if (warp == 1) gv += *tot_s;
        if (tid >= n) gv = 0.f;
        else if (tid < 64) g_cum[my_row] = gv;
    }
    if (tid < 64) {
        g_s[tid] = gv;
        b_s[tid] = bv;
        rk_s[tid] = 1.f;
    }
    __syncthreads();
    const float g_last = g_s[n - 1];
    const float g_ref = 0.5f * g_last;
    const bool fz = fabsf(g_last) <= 160.f;   // |g_i - g_ref| <= |g_last| / 2 for decays <= 0
    if (tid < 64) {
        eb_s[tid] = bv * __expf(gv);
        cf_s[tid] = tid < n ? __expf(g_ref - gv) : 0.f;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t s_k = smem_u32(sm + Lay::kK), s_n = smem_u32(sm + Lay::kN);
    const uint32_t s_xu = smem_u32(sm + Lay::kXU), s_y = smem_u32(sm + Lay::kY);
    uint32_t phase = 0;
    bool fail = !mbar_wait(bar_tma, 0, kWyWaitNs);

    // One MMA group issued by thread 0 (A K-major, B K-major or rows-along-N),
    // then everyone waits for it.
    // acc: add to the accumulator's current contents from the first step on
    auto mma_issue = [&](int M, uint32_t a, uint32_t bop, bool b_mn, int ksteps, bool acc = false) {
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t id = idesc_bf16(M, 64, false, b_mn);
            for (int ks = 0; ks < ksteps; ++ks) {
                const uint32_t a_off = (ks >> 2) * 8192 + (ks & 3) * 32;
                mma_bf16(tmem, smem_desc(a + a_off, 16, 1024, kLayoutSw128),
                         smem_desc(bop + (b_mn ? ks * 2048 : a_off), 8192, 1024, kLayoutSw128), id,
                         acc || ks > 0);
            }
            mma_commit(bar_mma);
        }
    };
    auto mma_wait = [&]() {
        fail |= !mbar_wait(bar_mma, phase, kWyWaitNs);
        phase ^= 1;
        tc_fence_after_sync();
    };
    auto mma = [&](int M, uint32_t a, uint32_t bop, bool b_mn, int ksteps, bool acc = false) {
        mma_issue(M, a, bop, b_mn, ksteps, acc);
        mma_wait();
    };
    // This thread's accumulator row, 16 columns at a time.
    auto load16 = [&](int blk, float *v) {
        uint32_t t[16];
        tmem_ld16(tmem + lane_off + blk * 16, t);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(t[e]);
    };

    // ---- [G; G] = [k; k] k^T (M = 128): row r of G in TMEM lanes r and 64 + r,
    // so warps 0-1 form L's columns 0-31 and warps 2-3 its columns 32-63
    if (__syncthreads_or(fail)) goto done;
    if (tid == 0) {
        tc_fence_after_sync();
        const uint32_t id = idesc_bf16(128, 64, false, false);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint32_t off = (ks >> 2) * Lay::kKBlk + (ks & 3) * 32;
            mma_bf16(tmem, smem_desc(s_k + off, 16, 1024, kLayoutSw128), smem_desc(s_k + off, 16, 1024, kLayoutSw128),
                     id, ks > 0);
        }
        mma_commit(bar_mma);
    }
    if (l2norm && tid < 64) {
        // |k_i|^2 from the k tile while the Gram runs. The 128-byte swizzle
        // permutes the 16-byte chunks within a row, which a sum of squares does
        // not see; visiting chunk j ^ (row % 8) keeps 8 consecutive rows on
        // different banks.
        float ss = 0.f;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 u = *reinterpret_cast<const uint4 *>(sm + Lay::kK + kb * Lay::kKBlk + tid * 128 +
                                                                 ((j ^ (tid & 7)) * 16));
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
            }
        const float r = rsqrtf(ss + kL2NormEps);
        rk_s[tid] = r;
        cf_s[tid] *= r;
        eb_s[tid] *= r;
        if (tid < n) rk_out[my_row] = r;
    }
    mma_wait();
    if (__syncthreads_or(fail)) goto done;
    {
        // row r (lanes r and 64 + r), column blocks 2 ch and 2 ch + 1
        const int r = (warp & 1) * 32 + lane, rb = r >> 4, ch = warp >> 1;
        const float gr = g_s[r], br = b_s[r] * rk_s[r];
        const float rf = br * __expf(gr - g_ref);
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
            const int blk = 2 * ch + bi;
            float v[16];
            load16(blk, v);
            if (r >= 0) {
                if (fz) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float4 c4 = *reinterpret_cast<const float4 *>(cf_s + blk * 16 + 4 * m);
                        const float cf[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const int e = 4 * m + e4;
                            v[e] = (blk * 16 + e < r) ? v[e] * rf * cf[e4] : 0.f;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = blk * 16 + e;
                        const float d = (j < r) ? gr - g_s[j] : -INFINITY;
                        v[e] = br * v[e] * rk_s[j] * __expf(d);
                    }
                }
                if (blk == rb) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) Ld[rb * 272 + e * 16 + (r & 15)] = v[e];
                }
                // N1: blocks (1,0) and (3,2); N2: rows 32-63 x columns 0-31
                const bool in1 = (rb == 1 && blk == 0) || (rb == 3 && blk == 2);
                const bool in2 = rb >= 2 && blk < 2;
                float n1[16], n2[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    n1[e] = in1 ? v[e] : 0.f;
                    n2[e] = in2 ? v[e] : 0.f;
                }
                st_bf16x8(sm + Lay::kN + sw128(r, blk * 32), n1);
                st_bf16x8(sm + Lay::kN + sw128(r, blk * 32 + 16), n1 + 8);
                st_bf16x8(sm + Lay::kN + 8192 + sw128(r, blk * 32), n2);
                st_bf16x8(sm + Lay::kN + 8192 + sw128(r, blk * 32 + 16), n2 + 8);
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    // ---- X: inverse of each 16x16 unit-lower diagonal block, column per thread
    {
        float x[16];
        const int blk = tid >> 4, col = tid & 15;
        float *Lb = Ld + blk * 272;
        if (tid < 64) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < 15; ++j)
#pragma unroll
                for (int q = (j + 1) >> 2; q < 4; ++q) {
                    // rows 4q .. 4q + 3 of column j (L's upper triangle is zero)
                    const float4 l4 = *reinterpret_cast<const float4 *>(Lb + j * 16 + 4 * q);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * q + e > j) x[4 * q + e] = fmaf(-lv[e], x[j], x[4 * q + e]);
                }
        }
        __syncthreads();
        if (tid < 64) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Lb[i * 17 + col] = x[i];
        }
        __syncthreads();
    }
    // From here on thread t owns row t of the M = 128 accumulators: rows 0-63
    // belong to X / A0 / A, rows 64-127 to U / Y2. The subtractions happen in
    // the fp32 accumulator: it is loaded with X (rows 0-63) or keeps U (rows
    // 64-127) and the next product adds [X; U] (-Y1), then [A0; U] (-Y2).
    {
        const int r = tid & 63, rb = r >> 4;
        // row r of X (threads < 64): its diagonal block; the rest of the row is 0
        float xr[16];
        if (tid < 64) {
            const float z8[8] = {};
#pragma unroll
            for (int j = 0; j < 16; ++j) xr[j] = Ld[(rb * 16 + (r & 15)) * 17 + j];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                if ((ch >> 1) == rb)
                    st_bf16x8(sm + Lay::kXU + sw128(r, ch * 16), xr + (ch & 1) * 8);
                else
                    st_bf16x8(sm + Lay::kXU + sw128(r, ch * 16), z8);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- [Y1; U] = [N1; N2] X
        mma(128, s_n, s_xu, true, 4);
        if (__syncthreads_or(fail)) goto done;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            float v[16];
            load16(blk, v);
            if (tid < 64) {
                // -Y1, the B operand (rows along N) of the next product
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = -v[e];
                st_bf16x8(sm + Lay::kY + sw128(r, blk * 32), v);
                st_bf16x8(sm + Lay::kY + sw128(r, blk * 32 + 16), v + 8);
            } else {
                // U, the second half of the A operand [X; U]; its fp32 copy stays
                // in the accumulator
                st_bf16x8(sm + Lay::kXU + 8192 + sw128(r, blk * 32), v);
                st_bf16x8(sm + Lay::kXU + 8192 + sw128(r, blk * 32 + 16), v + 8);
            }
        }
        if (tid < 64) {
            // the accumulator's rows 0-63 start the next product from X
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t t[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) t[e] = blk == rb ? __float_as_uint(xr[e]) : 0u;
                tmem_st16(tmem + lane_off + blk * 16, t);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        // ---- [A0; Y2] = [X; U] + [X; U] (-Y1)
        mma(128, s_xu, s_y, true, 4, true);
        if (__syncthreads_or(fail)) goto done;
        tc_fence_before_sync();
        __syncthreads();   // every MMA operand read before A0 / -Y2 overwrite them
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            float v[16];
            load16(blk, v);
            if (tid < 64) {
                // A0 as the next A operand (its fp32 copy stays in the accumulator)
                st_bf16x8(sm + Lay::kXU + sw128(r, blk * 32), v);
                st_bf16x8(sm + Lay::kXU + sw128(r, blk * 32 + 16), v + 8);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = -v[e];
                st_bf16x8(sm + Lay::kY + sw128(r, blk * 32), v);
                st_bf16x8(sm + Lay::kY + sw128(r, blk * 32 + 16), v + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        // ---- A = A0 + A0 (-Y2) in rows 0-63 (rows 64-127 of the product are unused)
        mma(128, s_xu, s_y, true, 4, true);
        if (__syncthreads_or(fail)) goto done;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            if (tid < 64) {
                // A diag(beta) and A diag(beta exp(g)); the second goes to the
                // [N1; N2] tile, free since the first merge product (rows
                // 64-127 of the product are not needed: warps 2-3 skip them)
                float v[16], v2[16];
                load16(blk, v);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(b_s + blk * 16 + 4 * m);
                    const float4 e4 = *reinterpret_cast<const float4 *>(eb_s + blk * 16 + 4 * m);
                    const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, ee[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = v[4 * m + e];
                        v[4 * m + e] = a * bb[e];
                        v2[4 * m + e] = a * ee[e];
                    }
                }
                st_bf16x8(sm + Lay::kOut + sw128(r, blk * 32), v);
                st_bf16x8(sm + Lay::kOut + sw128(r, blk * 32 + 16), v + 8);
                st_bf16x8(sm + Lay::kN + sw128(r, blk * 32), v2);
                st_bf16x8(sm + Lay::kN + sw128(r, blk * 32 + 16), v2 + 8);
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        tma_store_4d(&tm_a, sm + Lay::kOut, 0, h, t0, b);
        tma_store_4d(&tm_a, sm + Lay::kN, 64, h, t0, b);
        bulk_commit_group();
        bulk_wait_group_read0();   // only the shared source must outlive the CTA
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
    if (!make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) || !make_tmap_bthx(&ma, abeta, 128, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem = static_cast<int>(WyLayout<K>::kBytes + 1024);
    const auto kernel = a.flags ? gdn_wy_tc_kernel<K, true> : gdn_wy_tc_kernel<K, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3(a.NT, a.H, a.B), kWyThreads, smem, s>>>(
        mk, ma, a.g, a.beta, a.T, a.H, a.status, a.flags, a.g_cum, a.rk);
    return cudaGetLastError();
}

}  // namespace

cudaError_t wy_tc_forward(const Args &a, void *abeta, cudaStream_t s) {
    return a.K == 128 ? launch_wy<128>(a, abeta, s) : launch_wy<64>(a, abeta, s);
}

}  // namespace gdn
