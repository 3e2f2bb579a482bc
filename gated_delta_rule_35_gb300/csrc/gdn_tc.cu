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

// 20 warps: 0 MMA issuer, 1 TMA producer, 2-3 scale group, 4-11 prep group, 12-19 chain group
constexpr int kTcThreads = 640;
constexpr int kScaleThreads = 64, kPrepThreads = 256, kChainThreads = 256;
constexpr int kTcBV = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait

// Shared-memory map (bytes from a 1024-aligned base).
template <int K>
struct TcLayout {
    static constexpr int KB = K / 64;                            // 64-feature blocks
    // Two input stages. Per 64-feature block: k rows | h^T rows | q rows (8 KB
    // each, K-major, 128-byte swizzle), then A diag(beta). k and h^T are
    // adjacent so that together they form one 128-row operand.
    static constexpr uint32_t kKb = 24576;                        // per-block stride
    static constexpr uint32_t kHT = 8192, kQ = 16384;             // offsets in a block
    static constexpr uint32_t kAb = KB * kKb;                     // offset in a stage
    static constexpr uint32_t kStage = kAb + 8192;
    static constexpr uint32_t kKHV = 2 * kStage;                  // exp(g) k (KB x 8 KB) | v tile
    static constexpr uint32_t kW = kKHV + (KB + 1) * 8192;        // -w operand, KB x 8 KB
    static constexpr uint32_t kP = kW + KB * 8192;                // P
    static constexpr uint32_t kVN = kP + 8192;                    // v_new
    static constexpr uint32_t kVG = kVN + 8192;                   // v_new exp(g_last - g)
    static constexpr uint32_t kOS = kVG + 8192;                   // o staging for the TMA store
    static constexpr uint32_t kG = kOS + 8192;                    // g[2][64], exp(g)[2][64]
    static constexpr uint32_t kBar = kG + 1024;                   // mbarriers, flags
    static constexpr uint32_t kBytes = kBar + 256;
};

// TMEM columns of the 512-column allocation: [w | u] (K + 64), [q k^T | q h]
// (128), (dh)^T (K), P v_new (64).
constexpr uint32_t kColWU = 0, kColQKH = 192, kColHT = 320, kColPV = 448;

struct Bars {
    uint64_t full[2], empty[2], v_full;             // TMA: stage / v tile filled, stage released
    uint64_t w_done, x_done, qkh_done, h_done, o_done;   // MMA completions (tcgen05.commit)
    uint64_t g_ready;                               // scale group: g of the chunk in place
    uint64_t kh_ready, p_ready, w_ready;            // prep group: operands written
    uint64_t hs_ready, vn_ready, o_free;            // chain group
    uint32_t abort, tmem;
};

// Bounded wait: false if another role aborted or the limit passed (then aborts).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// Polling variant for the latency-critical roles (MMA issuer, chain group): a
// suspended waiter can take hundreds of cycles to resume after the phase
// completes.
__device__ __forceinline__ bool spin_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int K>
__global__ void __launch_bounds__(kTcThreads, 1)
gdn_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ g,
                    const float *__restrict__ h0, float *__restrict__ h_final, int T, int H, int V,
                    float scale, uint32_t *status) {
    using Lay = TcLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so
    // that every access through it stays a shared-memory access.
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *g_s = reinterpret_cast<float *>(sm + Lay::kG);   // [2][64] g (0 past T)
    float *eg_s = g_s + 128;                                 // [2][64] exp(g) (0 past T)
    Bars *bs = reinterpret_cast<Bars *>(sm + Lay::kBar);
    volatile uint32_t *abort = &bs->abort;

    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = (T + 63) / 64;

    if (warp == 0) {
        tmem_alloc(&bs->tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&bs->full[0], 1);
        mbar_init(&bs->full[1], 1);
        mbar_init(&bs->empty[0], 1);
        mbar_init(&bs->empty[1], 1);
        mbar_init(&bs->v_full, 1);
        mbar_init(&bs->w_done, 1);
        mbar_init(&bs->x_done, 1);
        mbar_init(&bs->qkh_done, 1);
        mbar_init(&bs->h_done, 1);
        mbar_init(&bs->o_done, 1);
        mbar_init(&bs->g_ready, kScaleThreads);
        mbar_init(&bs->kh_ready, kPrepThreads);
        mbar_init(&bs->p_ready, kPrepThreads);
        mbar_init(&bs->w_ready, kPrepThreads);
        mbar_init(&bs->hs_ready, kChainThreads);
        mbar_init(&bs->vn_ready, kChainThreads);
        mbar_init(&bs->o_free, kChainThreads);
        bs->abort = 0;
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
    const uint32_t tmem = bs->tmem;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idWU = idesc_bf16(64, K + 64, false, true);
            constexpr uint32_t idX = idesc_bf16(64, 64, false, false, true);
            constexpr uint32_t idQKH = idesc_bf16(64, 128, false, false);
            constexpr uint32_t idHT = idesc_bf16(64, K, true, true);
            constexpr uint32_t idPV = idesc_bf16(64, 64, false, true);
            const uint32_t s_khv = s_base + Lay::kKHV, s_w = s_base + Lay::kW, s_p = s_base + Lay::kP;
            const uint32_t s_vn = s_base + Lay::kVN, s_vg = s_base + Lay::kVG;
            // [w | u] = A diag(beta) [exp(g) k | v]
            auto issue_wu = [&](int s) {
                const uint32_t ab = s_base + s * Lay::kStage + Lay::kAb;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColWU, smem_desc(ab + ks * 32, 16, 1024, kLayoutSw128),
                             smem_desc(s_khv + ks * 2048, 8192, 1024, kLayoutSw128), idWU, ks > 0);
                mma_commit(&bs->w_done);
            };
            bool ok = spin_bar(&bs->full[0], 0, abort) && spin_bar(&bs->v_full, 0, abort) &&
                      spin_bar(&bs->kh_ready, 0, abort);
            if (ok) {
                tc_fence_after_sync();
                issue_wu(0);
            }
            for (int c = 0; ok && c < NT; ++c) {
                const int s = c & 1;
                const uint32_t par = c & 1;
                const uint32_t st = s_base + s * Lay::kStage;
                // v_new = u - w h (accumulates onto u)
                if (!(ok = spin_bar(&bs->hs_ready, par, abort) && spin_bar(&bs->w_ready, par, abort)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    mma_bf16(tmem + kColWU + K,
                             smem_desc(s_w + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kLayoutSw128),
                             smem_desc(st + (ks >> 2) * Lay::kKb + Lay::kHT + (ks & 3) * 32, 16, 1024,
                                       kLayoutSw128),
                             idX, 1);
                mma_commit(&bs->x_done);
                // [q k^T | q h]: k and h^T rows stacked as one operand
                if (c >= 1 && !(ok = spin_bar(&bs->o_free, (c - 1) & 1, abort))) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * Lay::kKb + (ks & 3) * 32;
                    mma_bf16(tmem + kColQKH, smem_desc(st + off + Lay::kQ, 16, 1024, kLayoutSw128),
                             smem_desc(st + off, 16, 1024, kLayoutSw128), idQKH, ks > 0);
                }
                mma_commit(&bs->qkh_done);
                // (dh)^T = (v_new exp(g_last - g))^T k; the stage's last reader
                if (!(ok = spin_bar(&bs->vn_ready, par, abort))) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColHT, smem_desc(s_vg + ks * 2048, 8192, 1024, kLayoutSw128),
                             smem_desc(st + ks * 2048, Lay::kKb, 1024, kLayoutSw128), idHT, ks > 0);
                mma_commit(&bs->h_done);
                mma_commit(&bs->empty[s]);
                // next chunk's [w | u]
                if (c + 1 < NT) {
                    if (!(ok = spin_bar(&bs->full[s ^ 1], ((c + 1) >> 1) & 1, abort) &&
                               spin_bar(&bs->v_full, (c + 1) & 1, abort) &&
                               spin_bar(&bs->kh_ready, (c + 1) & 1, abort)))
                        break;
                    tc_fence_after_sync();
                    issue_wu(s ^ 1);
                }
                // P v_new
                if (!(ok = spin_bar(&bs->p_ready, par, abort))) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColPV, smem_desc(s_p + ks * 32, 16, 1024, kLayoutSw128),
                             smem_desc(s_vn + ks * 2048, 8192, 1024, kLayoutSw128), idPV, ks > 0);
                mma_commit(&bs->o_done);
            }
        }
    } else if (warp == 1) {
        // ================================================================ TMA producer
        if (lane == 0) {
            for (int c = 0; c < NT; ++c) {
                const int s = c & 1;
                if (c >= 2 && !wait_bar(&bs->empty[s], ((c >> 1) - 1) & 1, abort)) break;
                unsigned char *st = sm + s * Lay::kStage;
                const int t0 = c * 64;
                mbar_arrive_expect_tx(&bs->full[s], KB * 16384 + 8192);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(st + kb * Lay::kKb, &tm_k, &bs->full[s], kb * 64, h, t0, b);
                    tma_load_4d(st + kb * Lay::kKb + Lay::kQ, &tm_q, &bs->full[s], kb * 64, h, t0, b);
                }
                tma_load_4d(st + Lay::kAb, &tm_a, &bs->full[s], 0, h, t0, b);
                // the single v slot is free once the previous [w | u] product is done
                if (c >= 1 && !wait_bar(&bs->w_done, (c - 1) & 1, abort)) break;
                mbar_arrive_expect_tx(&bs->v_full, 8192);
                tma_load_4d(sm + Lay::kKHV + KB * 8192, &tm_v, &bs->v_full, vt * kTcBV, h, t0, b);
            }
        }
    } else if (warp < 4) {
        // ================================================================ scale group
        // g of each chunk, loaded one chunk ahead.
        const int stid = tid - 64;
        auto load_g = [&](int c) {
            const int t = c * 64 + stid;
            return (c < NT && t < T) ? g[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
        };
        float g_next = load_g(0);
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1;
            const int n = min(64, T - c * 64);
            const float g_cur = g_next;
            g_next = load_g(c + 1);
            if (!wait_bar(&bs->full[s], (c >> 1) & 1, abort)) break;
            g_s[s * 64 + stid] = g_cur;
            eg_s[s * 64 + stid] = stid < n ? __expf(g_cur) : 0.f;
            named_sync(3, kScaleThreads);
            mbar_arrive(&bs->g_ready);
        }
    } else if (warp < 12) {
        // ================================================================ prep group
        // Two warps per TMEM lane quarter, each owning half of the columns.
        const int ptid = tid - 128, q4 = warp & 3, phalf = (warp - 4) >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const int row64 = lane < 16 ? q4 * 16 + lane : -1;
        // k_hat = exp(g) k for chunk c (same swizzled positions as k)
        auto make_khat = [&](int c) -> bool {
            const int s = c & 1;
            if (!wait_bar(&bs->g_ready, c & 1, abort) || !wait_bar(&bs->full[s], (c >> 1) & 1, abort))
                return false;
            const unsigned char *st = sm + s * Lay::kStage;
#pragma unroll
            for (int it = 0; it < KB * 2; ++it) {
                const int idx = ptid + it * kPrepThreads;   // 16-byte chunk of k
                const int kb = idx >> 9, rem = idx & 511, row = rem >> 3, ch = rem & 7;
                const uint32_t off = sw128(row, ch * 16);
                const uint4 raw = ld_shared_v4(st + kb * Lay::kKb + off);
                const float sc = eg_s[s * 64 + row];
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack_bf16(w4[e]);
                    o4[e] = pack_bf16(f.x * sc, f.y * sc);
                }
                st_shared_v4(sm + Lay::kKHV + kb * 8192 + off, o4[0], o4[1], o4[2], o4[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bs->kh_ready);
            return true;
        };
        // w (rows 0-63 of [w | u]) -> bf16 operand, negated by the MMA
        auto epi_w = [&](int c) -> bool {
            if (!wait_bar(&bs->w_done, c & 1, abort)) return false;
            tc_fence_after_sync();
#pragma unroll
            for (int bb = 0; bb < K / 32; ++bb) {
                const int blk = phalf * (K / 32) + bb;
                uint32_t r[16];
                tmem_ld16(tmem + kColWU + lane_off + blk * 16, r);
                tmem_wait_ld();
                if (row64 >= 0) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
                    const int f0 = blk * 16;
                    unsigned char *base = sm + Lay::kW + (f0 >> 6) * 8192;
                    st_bf16x8(base + sw128(row64, (f0 & 63) * 2), v);
                    st_bf16x8(base + sw128(row64, (f0 & 63) * 2 + 16), v + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->w_ready);
            return true;
        };
        if (make_khat(0) && epi_w(0)) {
            for (int c = 0; c < NT; ++c) {
                const int s = c & 1;
                // the exp(g) k slot is free: its product for chunk c finished (w_done(c))
                if (c + 1 < NT && !make_khat(c + 1)) break;
                // P = scale (q k^T) exp(g_i - g_j), i >= j. Column blocks right of this
                // quarter's rows are all zero.
                if (!wait_bar(&bs->qkh_done, c & 1, abort)) break;
                tc_fence_after_sync();
                {
                    const float gi = row64 >= 0 ? g_s[s * 64 + row64] : 0.f;
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        const int blk = phalf * 2 + bb;
                        float v[16];
                        if (blk <= q4) {
                            uint32_t r[16];
                            tmem_ld16(tmem + kColQKH + lane_off + blk * 16, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int j = blk * 16 + e;
                                const float d = (j <= row64) ? gi - g_s[s * 64 + j] : -INFINITY;
                                v[e] = scale * __uint_as_float(r[e]) * __expf(d);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = 0.f;
                        }
                        if (row64 >= 0) {
                            st_bf16x8(sm + Lay::kP + sw128(row64, blk * 32), v);
                            st_bf16x8(sm + Lay::kP + sw128(row64, blk * 32 + 16), v + 8);
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->p_ready);
                if (c + 1 < NT && !epi_w(c + 1)) break;
            }
        }
    } else {
        // ================================================================ chain group
        // Two warps per TMEM lane quarter, each owning half of the columns. The
        // state is kept transposed: this thread owns row v = row64 of h^T (the
        // v tile's column), features [half K/2, half K/2 + K/2).
        constexpr int FH = K / 2;
        const int ctid = tid - 384, q4 = warp & 3, half = (warp - 12) >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const int row64 = lane < 16 ? q4 * 16 + lane : -1;
        const int col0 = half * 32;   // v-columns of this warp in the v_new / o epilogues
        const int f0 = half * FH;     // features of this warp in the state epilogue
        const uint32_t ht_off = (f0 >> 6) * Lay::kKb + Lay::kHT;   // h^T block inside a stage
        const uint32_t ht_byte = (f0 & 63) * 2;
        const int64_t state_off = (static_cast<int64_t>(b) * H + h) * K * V + vt * kTcBV;
        float hreg[FH];
#pragma unroll
        for (int j = 0; j < FH; ++j)
            hreg[j] = (row64 >= 0 && h0) ? h0[state_off + static_cast<int64_t>(f0 + j) * V + row64] : 0.f;
        if (row64 >= 0) {
#pragma unroll
            for (int ch = 0; ch < FH / 8; ++ch)
                st_bf16x8(sm + ht_off + sw128(row64, ht_byte + ch * 16), &hreg[ch * 8]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bs->hs_ready);
        bool ok = true;
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1;
            const uint32_t par = c & 1;
            const int t0 = c * 64, n = min(64, T - t0);
            if (!(ok = spin_bar(&bs->x_done, par, abort))) break;
            tc_fence_after_sync();
            const float g_last = g_s[s * 64 + n - 1];
            const float gate = (row64 >= 0 && row64 < n) ? __expf(g_last - g_s[s * 64 + row64]) : 0.f;
            const float so = row64 >= 0 ? scale * eg_s[s * 64 + row64] : 0.f;
            const float decay = __expf(g_last);
            // v_new and v_gated -> bf16 operands (token rows, V contiguous)
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint32_t r[16];
                tmem_ld16(tmem + kColWU + K + col0 + lane_off + blk * 16, r);
                tmem_wait_ld();
                if (row64 >= 0) {
                    float v[16], vg[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        v[e] = __uint_as_float(r[e]);
                        vg[e] = v[e] * gate;
                    }
                    const uint32_t byte = (col0 + blk * 16) * 2;
                    st_bf16x8(sm + Lay::kVN + sw128(row64, byte), v);
                    st_bf16x8(sm + Lay::kVN + sw128(row64, byte + 16), v + 8);
                    st_bf16x8(sm + Lay::kVG + sw128(row64, byte), vg);
                    st_bf16x8(sm + Lay::kVG + sw128(row64, byte + 16), vg + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->vn_ready);
            // h^T = h^T exp(g_last) + (dh)^T; bf16 copy into the next chunk's stage
            if (!(ok = spin_bar(&bs->h_done, par, abort))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int blk = 0; blk < FH / 16; ++blk) {
                uint32_t r[16];
                tmem_ld16(tmem + kColHT + f0 + lane_off + blk * 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    hreg[blk * 16 + e] = fmaf(hreg[blk * 16 + e], decay, __uint_as_float(r[e]));
            }
            if (row64 >= 0) {
                unsigned char *dst = sm + (s ^ 1) * Lay::kStage + ht_off;
#pragma unroll
                for (int ch = 0; ch < FH / 8; ++ch) st_bf16x8(dst + sw128(row64, ht_byte + ch * 16), &hreg[ch * 8]);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->hs_ready);
            // o = scale exp(g_t) q h + P v_new -> bf16 staging -> TMA store
            if (!(ok = wait_bar(&bs->o_done, par, abort))) break;
            tc_fence_after_sync();
            if (ctid == 0) bulk_wait_group_read0();
            named_sync(2, kChainThreads);
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint32_t rq[16], rp[16];
                tmem_ld16(tmem + kColQKH + 64 + col0 + lane_off + blk * 16, rq);
                tmem_ld16(tmem + kColPV + col0 + lane_off + blk * 16, rp);
                tmem_wait_ld();
                if (row64 >= 0) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = fmaf(so, __uint_as_float(rq[e]), __uint_as_float(rp[e]));
                    const uint32_t byte = (col0 + blk * 16) * 2;
                    st_bf16x8(sm + Lay::kOS + sw128(row64, byte), v);
                    st_bf16x8(sm + Lay::kOS + sw128(row64, byte + 16), v + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->o_free);
            named_sync(2, kChainThreads);
            if (ctid == 0) {
                tma_store_4d(&tm_o, sm + Lay::kOS, vt * kTcBV, h, t0, b);
                bulk_commit_group();
            }
        }
        if (ok && row64 >= 0 && h_final) {
#pragma unroll
            for (int j = 0; j < FH; ++j) h_final[state_off + static_cast<int64_t>(f0 + j) * V + row64] = hreg[j];
        }
        if (ctid == 0) bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort) atomicOr(status, 1u);
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
