// Tensor-core path of the chunked gated delta rule forward for bf16 q, k, v.
//
// Two kernels, following the "WarpDrive" page's pipeline (kernel 5
// recompute_w_u takes the chunk's WY matrix A as given; kernels 3 chunk_fwd_h
// and 4 chunk_fwd_o follow it):
//   1. gdn_wy_tc_kernel (gdn_tc_wy.cu): A diag(beta) and A diag(beta exp(g)) for
//      every chunk, in parallel over all chunks, to a bf16 workspace [B, T, H, 128].
//   2. gdn_fused_tc_kernel (this file): recompute_w_u, chunk_fwd_h and
//      chunk_fwd_o fused. One CTA owns one (b, h, 64-wide V tile) and walks the
//      chunks in order. The state lives in tensor memory in fp32, with a bf16
//      copy in shared memory as an MMA operand; h, w, u and v_new never reach HBM.
//
// Per chunk (C = 64 tokens), with A' = A diag(beta exp(g)) so that
// w = A diag(beta) (exp(g) k) = A' k. Accumulators live in tensor memory, one
// row per TMEM lane; "." marks operand rows whose products are never read:
//   W    [A'; .] k                      W rows 0-63 = w
//   U    [0; A diag(beta)] v            X rows 64-127 = u, X rows 0-63 = 0
//   BIG  [q; -w] [h^T | k]              X += [q h; -w h]  (rows 64-127: v_new)
//                                       QK rows 0-63 += q k^T (cleared after each read)
//   HT   [v_g; v_g]^T k                 h^T += v_g^T k, v_g = v_new exp(g_last - g)
//   PV   [P; .] v_new                   O += P v_new
// TMA writes q and k straight into the stacked operands' halves; the prep group
// builds the per-chunk decay tables; the w epilogue writes -w under q.
// The chain group turns QK into P = scale (q k^T) exp(g_i - g_j) (i >= j),
// normally as QK times a row and a column factor of exp(g_i - g_j) taken about
// g_last / 2 (per-element exponentials only for chunks whose decay could
// overflow those factors). It seeds O with scale exp(g) (q h), writes v_new and
// v_g, keeps the state (pre-decayed by the next chunk's exp(g_last), so that
// HT completes the update) and sends o to HBM. From one chunk to the next the
// dependency chain is BIG -> v_new -> HT -> bf16 h^T -> BIG; W, U and PV fill
// the tensor pipe around it.
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;

// 16 warps: 0 MMA issuer, 1 TMA producer, 2-3 and 6-7 prep group, 4-5 w
// epilogue, 8-15 chain group. A warp reaches the TMEM lanes of quarter warp % 4.
constexpr int kTcThreads = 512;
constexpr int kPrepThreads = 128, kWThreads = 64, kChainThreads = 256;
constexpr int kTcBV = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait

// Shared-memory map (bytes from a 1024-aligned base). Every tile is 64 rows of
// 128 bytes with the 128-byte swizzle, as TMA writes it.
template <int K>
struct TcLayout {
    static constexpr int KB = K / 64;                            // 64-feature blocks
    // Two stages, one per chunk parity. Per 64-feature block the stacked
    // operands [q; -w] and [h^T; k] (16 KB each: TMA writes q and k straight
    // into their halves), then v | zero tile | A diag(beta) | A', [0; A diag(beta)]
    // being U's A operand. W and HT read k N-major out of [h^T; k] (atoms 16 KB
    // apart); HT reads the one v_g tile as both halves of its A operand.
    static constexpr uint32_t kStAbig = 0, kStBbig = KB * 16384;
    static constexpr uint32_t kStV = 2 * KB * 16384, kStZ = kStV + 8192, kStA = kStZ + 8192;
    static constexpr uint32_t kStAp = kStA + 8192;               // A' (W's A operand rows 0-63)
    static constexpr uint32_t kStage = kStAp + 8192;
    static constexpr uint32_t kP = 2 * kStage;                   // P
    static constexpr uint32_t kVN = kP + 8192;                   // v_new
    static constexpr uint32_t kVG = kVN + 8192;                  // v_g
    static constexpr uint32_t kG = kVG + 8192;                   // decay tables, 4 chunk slots
    static constexpr uint32_t kBar = kG + 5 * 4 * 64 * 4 + 16;
    // output stage: row sums of squares, [2 chunk slots][4 ranks x 2 halves][64 rows]
    static constexpr uint32_t kRed = kBar + 256;
    static constexpr uint32_t kBytes = kRed + 2 * 8 * 64 * 4;
};

// TMEM columns: X-region [X (64) | QK (64)], O (64), W (K), HT (K).
constexpr uint32_t kColX = 0, kColQK = 64, kColO = 128, kColW = 192, kColHT = 320;
// With the output stage O is double-buffered (chunk parity), the second copy
// in the columns after HT, so that a chunk's normalisation can wait for the
// cluster's row sums while the next chunk runs.
constexpr uint32_t kColO2 = 448;

struct Bars {
    uint64_t full[2], empty[2];                     // TMA stages
    uint64_t big_done, w_done, h_done, o_done;      // MMA completions (tcgen05.commit)
    uint64_t g_ready[4];                            // prep group (one per table slot)
    uint64_t w_ready;                               // w epilogue
    uint64_t xo_ready, vn_ready, hs_ready;          // chain group
    uint64_t drain;                                 // every MMA issued is done
    uint64_t norm_bar[2];                           // output stage: row sums of the cluster
    uint32_t abort, tmem;
};

// Bounded wait: false if another role aborted or the limit passed (then aborts).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                         uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// wait_bar for a barrier completed by other CTAs of the cluster (acquire at
// cluster scope).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity,
                                                 volatile uint32_t *abort, uint64_t limit) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// Polling variant for the latency-critical roles: a suspended waiter can take
// hundreds of cycles to resume after the phase completes.
__device__ __forceinline__ bool spin_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                         uint64_t limit) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                *abort = 1;
                return false;
            }
        }
    }
}
// A warp leaves its loop together: the tcgen05 loads that follow a wait are
// warp-collective.
__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }
__device__ __forceinline__ void store_bf16x8_global(void *dst, const float *v) {
    uint4 u = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                         pack_bf16(v[6], v[7]));
    *reinterpret_cast<uint4 *>(dst) = u;
}
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}

// GATED: the output stage (gated RMSNorm over V) with the V tiles of a head as
// one cluster of nrank_arg CTAs; without it the cluster code is compiled out.
template <int K, bool GATED>
__global__ void __launch_bounds__(kTcThreads, 1)
gdn_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                    const float *__restrict__ g, const float *__restrict__ h0,
                    float *__restrict__ h_final, __nv_bfloat16 *__restrict__ o, int T, int H, int V,
                    float scale, int l2_prefetch, uint32_t *status, int l2norm,
                    const float *__restrict__ rk, const __nv_bfloat16 *__restrict__ gate,
                    const float *__restrict__ norm_w, float norm_eps, int nrank_arg,
                    uint64_t wlim, int stall) {
    using Lay = TcLayout<K>;
    const int nrank = GATED ? nrank_arg : 0;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so
    // that every access through it stays a shared-memory access.
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // Per chunk slot (c & 3), 0 past T where marked, with rq_i and rk_j the
    // q and k rows' normalisation factors (1 without the front-end norm):
    // exp(g) rq (0); exp(g_last - g) rk (0); and the row and column factors of
    // scale rq_i rk_j exp(g_i - g_j): about g_ref = g_last / 2, scale rq
    // exp(g_i - g_ref) (0) and rk exp(g_ref - g_j) (0), usable while |g_last|
    // stays small enough for both to be finite fp32 numbers (flag fz_s); else
    // the exponents g_i + ln rq_i and g_j - ln rk_j.
    float *tab = reinterpret_cast<float *>(sm + Lay::kG);   // first 256 floats unused
    float *eg_s = tab + 256;
    float *gate_s = tab + 512;
    float *rf_s = tab + 768;
    float *cf_s = tab + 1024;
    int *fz_s = reinterpret_cast<int *>(tab + 1280);
    Bars *bs = reinterpret_cast<Bars *>(sm + Lay::kBar);
    volatile uint32_t *abort = &bs->abort;

    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = (T + 63) / 64;

    // the zero tiles of both stages, read by U as the zero halves of its operands
    for (int i = tid; i < 1024; i += kTcThreads)
        st_shared_v4(sm + (i >> 9) * Lay::kStage + Lay::kStZ + (i & 511) * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&bs->tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bs->full[s], 1);
            mbar_init(&bs->empty[s], 1);
        }
        mbar_init(&bs->big_done, 1);
        mbar_init(&bs->w_done, 1);
        mbar_init(&bs->h_done, 1);
        mbar_init(&bs->o_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&bs->g_ready[i], kPrepThreads);
        mbar_init(&bs->w_ready, kWThreads);
        mbar_init(&bs->xo_ready, kChainThreads / 2);
        mbar_init(&bs->vn_ready, kChainThreads / 2);
        mbar_init(&bs->hs_ready, kChainThreads);
        mbar_init(&bs->drain, 1);
        // output stage: one local arrival (with the expected bytes) per chunk;
        // the row sums of every CTA of the cluster arrive as transactions
        if (nrank)
            for (int i = 0; i < 2; ++i) mbar_init(&bs->norm_bar[i], 1);
        bs->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_a);
    }
    tc_fence_before_sync();
    __syncthreads();
    // With the output stage the V tiles of one head run as a cluster (rank =
    // V tile); its barriers must be initialised before any CTA arrives on them.
    if (nrank) cluster_sync();
    // The setup above overlaps the WY kernel's last CTAs; everything below may
    // read its output.
    griddep_wait();
    tc_fence_after_sync();
    const uint32_t tmem = bs->tmem;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idW = idesc_bf16(128, K, false, true);
            constexpr uint32_t idU = idesc_bf16(128, 64, false, true);
            constexpr uint32_t idBIG = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idHT = idesc_bf16(128, K, true, true);
            constexpr uint32_t idPV = idesc_bf16(128, 64, false, true);
            const uint32_t s_p = s_base + Lay::kP;
            const uint32_t s_vn = s_base + Lay::kVN, s_vg = s_base + Lay::kVG;
            // W = [A'; .] k, k read N-major from the stage's [h^T; k]; the rows under A'
            // are whatever follows it (the next stage or P): their products are unused
            auto issue_w = [&](int s) {
                const uint32_t kt = s_base + s * Lay::kStage + Lay::kStBbig + 8192;
                const uint32_t ap = s_base + s * Lay::kStage + Lay::kStAp;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColW, smem_desc(ap + ks * 32, 16, 1024, kLayoutSw128),
                             smem_desc(kt + ks * 2048, 16384, 1024, kLayoutSw128), idW, ks > 0);
                mma_commit(&bs->w_done);
            };
            // X = [0; A diag(beta)] v
            auto issue_u = [&](int s) {
                const uint32_t st = s_base + s * Lay::kStage;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColX, smem_desc(st + Lay::kStZ + ks * 32, 16, 1024, kLayoutSw128),
                             smem_desc(st + Lay::kStV + ks * 2048, 8192, 1024, kLayoutSw128), idU,
                             ks > 0);
            };
            // O += [P; .] v_new of chunk cp
            auto issue_pv = [&](int cp) {
                const uint32_t vn = s_vn;
                const uint32_t ocol = (GATED && (cp & 1)) ? kColO2 : kColO;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + ocol, smem_desc(s_p + ks * 32, 16, 1024, kLayoutSw128),
                             smem_desc(vn + ks * 2048, 8192, 1024, kLayoutSw128), idPV, 1);
                mma_commit(&bs->o_done);
            };
            bool ok = spin_bar(&bs->full[0], 0, abort, wlim);
            if (ok) {
                tc_fence_after_sync();
                issue_w(0);
                issue_u(0);
            }
            for (int c = 0; ok && c < NT; ++c) {
                const int s = c & 1;
                const uint32_t par = c & 1;
                // X += [q; -w] [h^T | k] (q and k landed before W(c) was issued)
                if (!(ok = spin_bar(&bs->hs_ready, par, abort, wlim) && spin_bar(&bs->w_ready, par, abort, wlim)))
                    break;
                tc_fence_after_sync();
                const uint32_t st = s_base + s * Lay::kStage;
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + kColX, smem_desc(st + Lay::kStAbig + off, 16, 1024, kLayoutSw128),
                             smem_desc(st + Lay::kStBbig + off, 16, 1024, kLayoutSw128), idBIG, 1);
                }
                mma_commit(&bs->big_done);
                // Next chunk's w as soon as its inputs land, if that happens before
                // v_new is ready; otherwise after HT(c), which must not queue behind
                // it in the in-order tensor pipe. One loop polls both.
                bool w_next = c + 1 < NT;
                {
                    const uint64_t t0 = globaltimer_ns();
                    for (uint32_t i = 1;; ++i) {
                        if (w_next && mbar_test_wait(&bs->full[s ^ 1], ((c + 1) >> 1) & 1)) {
                            tc_fence_after_sync();
                            issue_w(s ^ 1);
                            w_next = false;
                        }
                        if (mbar_test_wait(&bs->vn_ready, par)) break;
                        if ((i & 255) == 0) {
                            if (*abort) { ok = false; break; }
                            if (globaltimer_ns() - t0 > wlim) { *abort = 1; ok = false; break; }
                        }
                    }
                    if (!ok) break;
                }
                // h^T += v_g^T k
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + kColHT, smem_desc(s_vg + ks * 2048, 0, 1024, kLayoutSw128),
                             smem_desc(st + Lay::kStBbig + 8192 + ks * 2048, 16384, 1024, kLayoutSw128),
                             idHT, 1);
                mma_commit(&bs->h_done);
                mma_commit(&bs->empty[s]);   // HT(c) is the stage's last reader
                if (w_next) {
                    if (!(ok = spin_bar(&bs->full[s ^ 1], ((c + 1) >> 1) & 1, abort, wlim))) break;
                    tc_fence_after_sync();
                    issue_w(s ^ 1);
                }
                // once P, q h and v_new are out of the X-region: next chunk's u, then o
                if (!(ok = spin_bar(&bs->xo_ready, par, abort, wlim))) break;
                tc_fence_after_sync();
                if (c + 1 < NT) issue_u(s ^ 1);
                issue_pv(c);
            }
            // nothing of ours may still run when the accumulators are released
            mma_commit(&bs->drain);
            mbar_wait(&bs->drain, 0, kWaitNs);
        }
    } else if (warp == 1) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int issued = 0;   // chunks whose loads were issued
            for (int c = 0; c < NT; ++c) {
                const int s = c & 1, t0 = c * 64;
                if (c >= 2 && !wait_bar(&bs->empty[s], ((c >> 1) - 1) & 1, abort, wlim)) break;
                // test hook: chunk 0's loads are withheld, so every role's first
                // wait on them runs out and the launch reports a device timeout
                if (stall && c == 0) continue;
                unsigned char *st = sm + s * Lay::kStage;
                mbar_arrive_expect_tx(&bs->full[s], KB * 16384 + 24576);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(st + Lay::kStAbig + kb * 16384, &tm_q, &bs->full[s], kb * 64, h, t0, b);
                    tma_load_4d(st + Lay::kStBbig + kb * 16384 + 8192, &tm_k, &bs->full[s], kb * 64, h,
                                t0, b);
                }
                tma_load_4d(st + Lay::kStV, &tm_v, &bs->full[s], vt * kTcBV, h, t0, b);
                tma_load_4d(st + Lay::kStA, &tm_a, &bs->full[s], 0, h, t0, b);
                tma_load_4d(st + Lay::kStAp, &tm_a, &bs->full[s], 64, h, t0, b);
                issued = c + 1;
                // chunk c + 2 into L2 now, so that its stage load, two chunks from
                // now, is served from L2 rather than HBM. Only when the grid leaves
                // SMs idle: with every SM busy it costs more than the latency it hides.
                if (l2_prefetch && c + 2 < NT) {
                    const int tp = t0 + 128;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) {
                        tma_prefetch_4d(&tm_q, kb * 64, h, tp, b);
                        tma_prefetch_4d(&tm_k, kb * 64, h, tp, b);
                    }
                    tma_prefetch_4d(&tm_v, vt * kTcBV, h, tp, b);
                    tma_prefetch_4d(&tm_a, 0, h, tp, b);
                    tma_prefetch_4d(&tm_a, 64, h, tp, b);
                }
            }
            // no copy may still be landing in shared memory when the CTA exits
            // (after an abort the last loads may have no consumer)
            for (int c = max(stall ? 1 : 0, issued - 2); c < issued; ++c)
                mbar_wait(&bs->full[c & 1], (c >> 1) & 1, kWaitNs);
        }
    } else if (warp == 2 || warp == 3 || warp == 6 || warp == 7) {
        // ================================================================ prep group
        // Per-chunk decay tables (A' = A diag(beta exp(g)) comes with A diag(beta)
        // from the WY kernel).
        const int ptid = warp < 4 ? tid - 64 : tid - 128;
        // g of chunk c and of its last valid token, loaded one chunk ahead
        auto load_g = [&](int c) {
            const int t = c * 64 + ptid;
            return (ptid < 64 && c < NT && t < T) ? g[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
        };
        auto load_gl = [&](int c) {
            return (ptid < 64 && c < NT) ? g[(static_cast<int64_t>(b) * T + min(T, c * 64 + 64) - 1) * H + h]
                                         : 0.f;
        };
        // k rows' normalisation factors, from the WY kernel
        auto load_rk = [&](int c) {
            const int t = c * 64 + ptid;
            return (l2norm && ptid < 64 && c < NT && t < T) ? rk[(static_cast<int64_t>(b) * T + t) * H + h]
                                                           : 1.f;
        };
        float g_next = load_g(0), gl_next = load_gl(0), rk_next = load_rk(0);
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1, gs = c & 3;
            const int n = min(64, T - c * 64);
            const float g_cur = g_next, gl = gl_next, rk_cur = rk_next;
            g_next = load_g(c + 1);
            gl_next = load_gl(c + 1);
            rk_next = load_rk(c + 1);
            // Decay tables of chunk c in slot c % 4. Their previous reader, chunk
            // c - 4, finished before U(c - 3) was issued, and stage s landing for
            // chunk c needs HT(c - 2). For the same reason the next phase of
            // g_ready[c % 4] (chunk c + 4) cannot complete before every waiter of
            // this one has passed.
            if (!wait_bar(&bs->full[s], (c >> 1) & 1, abort, wlim)) break;
            if (ptid < 64) {
                float rq = 1.f;
                if (l2norm) {
                    // |q_i|^2 from the stage's q tile (rows 0-63 of the stacked
                    // operand; the swizzle only permutes 16-byte chunks in a
                    // row, and chunk j ^ (row % 8) keeps 8 rows on distinct banks)
                    const unsigned char *qrow = sm + s * Lay::kStage + Lay::kStAbig + ptid * 128;
                    float ss = 0.f;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(qrow + kb * 16384 +
                                                                             ((j ^ (ptid & 7)) * 16));
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(w4[e] << 16);
                                const float hi = __uint_as_float(w4[e] & 0xffff0000u);
                                ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                            }
                        }
                    rq = rsqrtf(ss + kL2NormEps);
                }
                const float gref = 0.5f * gl;
                // |g_i - g_ref| <= |g_last| / 2 for cumulative log decays in [g_last, 0]
                const bool fzc = fabsf(gl) <= 160.f;
                const bool ok = ptid < n;
                eg_s[gs * 64 + ptid] = ok ? __expf(g_cur) * rq : 0.f;
                gate_s[gs * 64 + ptid] = ok ? __expf(gl - g_cur) * rk_cur : 0.f;
                if (fzc) {
                    rf_s[gs * 64 + ptid] = ok ? scale * __expf(g_cur - gref) * rq : 0.f;
                    cf_s[gs * 64 + ptid] = ok ? __expf(gref - g_cur) * rk_cur : 0.f;
                } else {
                    rf_s[gs * 64 + ptid] = l2norm ? g_cur + __logf(rq) : g_cur;
                    cf_s[gs * 64 + ptid] = l2norm ? g_cur - __logf(rk_cur) : g_cur;
                }
                if (ptid == 0) fz_s[gs] = fzc;
            }
            mbar_arrive(&bs->g_ready[gs]);
        }
    } else if (warp < 6) {
        // ================================================================ w epilogue
        // Rows 0-63 of W (lane quarters 0-1) -> -w, bf16, under q in the stage's
        // stacked operand (that half was last read by BIG(c - 2)).
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int row = (warp & 3) * 32 + lane;
        for (int c = 0; c < NT; ++c) {
            if (!warp_all(wait_bar(&bs->w_done, c & 1, abort, wlim))) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int bb = 0; bb < K / 32; ++bb) {
                const int f0 = bb * 32;
                uint32_t r[32];
                tmem_ld32(tmem + kColW + lane_off + f0, r);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = -__uint_as_float(r[e]);
                unsigned char *base = sm + (c & 1) * Lay::kStage + Lay::kStAbig + (f0 >> 6) * 16384;
#pragma unroll
                for (int q = 0; q < 4; ++q) st_bf16x8(base + sw128(64 + row, (f0 & 63) * 2 + q * 16), v + q * 8);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->w_ready);
        }
    } else {
        // ================================================================ chain group
        // Warps on lane quarters 0-1 own token rows 0-63 (P, the O seed, o);
        // warps on quarters 2-3 own rows 64-127 (v_new). Each handles 32 of the
        // 64 columns. The state h^T (rows v) sits twice in HT, lanes 0-63 and
        // 64-127; copy q4 / 2 keeps features [q4 / 2 * K / 2, + K / 2) current,
        // and each warp owns K / 4 of them.
        constexpr int NF = K / 4;
        const int q4 = warp & 3, hf = (warp - 8) >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const bool upper = q4 < 2;
        const int row = (q4 & 1) * 32 + lane;
        const int col0 = hf * 32;
        const int f0 = (q4 >> 1) * (K / 2) + hf * NF;
        const int64_t state_off = (static_cast<int64_t>(b) * H + h) * K * V + vt * kTcBV;
        auto g_last_of = [&](int c) {
            return g[(static_cast<int64_t>(b) * T + min(T, c * 64 + 64) - 1) * H + h];
        };
        // initial state: bf16 h^T under k in the stacked operand; fp32 in TMEM,
        // pre-decayed by exp(g_last) of chunk 0
        {
            const float d0 = __expf(g_last_of(0));
#pragma unroll 1
            for (int blk = 0; blk < NF / 16; ++blk) {
                const int f = f0 + blk * 16;
                float v[16];
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    v[e] = h0 ? h0[state_off + static_cast<int64_t>(f + e) * V + row] : 0.f;
                    r[e] = __float_as_uint(v[e] * d0);
                }
                tmem_st16(tmem + kColHT + lane_off + f, r);
                unsigned char *dst = sm + Lay::kStBbig + (f >> 6) * 16384;
                st_bf16x8(dst + sw128(row, (f & 63) * 2), v);
                st_bf16x8(dst + sw128(row, (f & 63) * 2 + 16), v + 8);
            }
            if (upper) {   // QK starts at zero (U writes X only)
                const uint32_t z[16] = {};
                tmem_st16(tmem + kColQK + lane_off + col0, z);
                tmem_st16(tmem + kColQK + lane_off + col0 + 16, z);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(&bs->hs_ready);
        bool ok = true;
        // Output stage (gated RMSNorm over the head's V columns), in two parts
        // per chunk so that the cluster exchange overlaps the next chunk:
        // part 1, after o_done(c), sends this thread's sum of squares over its
        // 32 columns to every CTA of the cluster (slot c % 2, entry rank * 2 +
        // half) and prefetches the gate; part 2, after the next chunk's O seed,
        // waits for all sums, reads O(c) again and writes the output. A slot is
        // next written for chunk c + 2, which needs every thread of the
        // cluster to have arrived for chunk c + 1, i.e. to have finished part 2
        // of chunk c: neither the sums nor the barrier phase can be overtaken.
        // The sums travel as asynchronous stores that complete bytes of the
        // receiving CTA's barrier, so the sender needs no memory fence.
        auto gated_send = [&](int c) {
            const uint32_t ob = (c & 1) ? kColO2 : kColO;
            float v0[16], v1[16];
            tmem_ld16f(tmem + ob + lane_off + col0, v0);
            tmem_ld16f(tmem + ob + lane_off + col0 + 16, v1);
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) ss = fmaf(v0[e], v0[e], fmaf(v1[e], v1[e], ss));
            const int tc0 = c * 64;
            if (row < min(64, T - tc0))
                prefetch_l2(gate + ((static_cast<int64_t>(b) * T + tc0 + row) * H + h) * V +
                            vt * kTcBV + col0);
            const int slot = c & 1;
            const uint32_t red = s_base + Lay::kRed + ((slot * 8 + vt * 2 + hf) * 64 + row) * 4;
            const uint32_t nb = smem_u32(&bs->norm_bar[slot]);
            // this CTA expects one sum from each of the cluster's o-epilogue threads
            if (warp == 8 && lane == 0) mbar_arrive_expect_tx(&bs->norm_bar[slot], nrank * 128 * 4);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (r < nrank) st_async_cluster_f32(mapa_shared(red, r), ss, mapa_shared(nb, r));
        };
        auto gated_finish = [&](int c) -> bool {
            const int slot = c & 1;
            if (!warp_all(wait_bar_cluster(&bs->norm_bar[slot], (c >> 1) & 1, abort, wlim))) return false;
            const float *sums = reinterpret_cast<const float *>(sm + Lay::kRed) + slot * 512;
            float tot = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < 2 * nrank) tot += sums[i * 64 + row];
            const float rstd = rsqrtf(tot / V + norm_eps);
            const uint32_t ob = (c & 1) ? kColO2 : kColO;
            float v0[16], v1[16];
            tmem_ld16f(tmem + ob + lane_off + col0, v0);
            tmem_ld16f(tmem + ob + lane_off + col0 + 16, v1);
            const int tc0 = c * 64;
            if (row < min(64, T - tc0)) {
                const int64_t oi = ((static_cast<int64_t>(b) * T + tc0 + row) * H + h) * V +
                                   vt * kTcBV + col0;
                const float *wv = norm_w + vt * kTcBV + col0;
                float y[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 zr = reinterpret_cast<const uint4 *>(gate + oi)[i];
                    const uint32_t w4[4] = {zr.x, zr.y, zr.z, zr.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = i * 8 + 2 * e;
                        const float z0 = __uint_as_float(w4[e] << 16);
                        const float z1 = __uint_as_float(w4[e] & 0xffff0000u);
                        const float o0 = j < 16 ? v0[j] : v1[j - 16];
                        const float o1 = j + 1 < 16 ? v0[j + 1] : v1[j - 15];
                        y[j] = o0 * rstd * wv[j] * __fdividef(1.f, 1.f + __expf(-z0));
                        y[j + 1] = o1 * rstd * wv[j + 1] * __fdividef(1.f, 1.f + __expf(-z1));
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) store_bf16x8_global(o + oi + i * 8, y + i * 8);
            }
            return true;
        };
        float g_last_next = NT > 1 ? g_last_of(1) : 0.f;
        for (int c = 0; c < NT; ++c) {
            const int t0 = c * 64, n = min(64, T - t0), gs = c & 3;
            const float d_next = (c + 1 < NT) ? __expf(g_last_next) : 1.f;
            if (c + 2 < NT) g_last_next = g_last_of(c + 2);   // one chunk ahead
            if (!(ok = warp_all(wait_bar(&bs->g_ready[gs], (c >> 2) & 1, abort, wlim) &&
                                spin_bar(&bs->big_done, c & 1, abort, wlim))))
                break;
            tc_fence_after_sync();
            if (upper) {
                const bool fz = fz_s[gs];
                const float ri = rf_s[gs * 64 + row];
                const float *cfc = cf_s + gs * 64;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int j0 = col0 + half * 16;
                    float v[16];
                    if (j0 <= (q4 & 1) * 32 + 31) {
                        float fj[16];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 f4 = *reinterpret_cast<const float4 *>(cfc + j0 + 4 * m);
                            fj[4 * m] = f4.x;
                            fj[4 * m + 1] = f4.y;
                            fj[4 * m + 2] = f4.z;
                            fj[4 * m + 3] = f4.w;
                        }
                        tmem_ld16f(tmem + kColQK + lane_off + j0, v);
                        if (fz) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = (j0 + e <= row) ? v[e] * ri * fj[e] : 0.f;
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float d = (j0 + e <= row) ? ri - fj[e] : -INFINITY;
                                v[e] = scale * v[e] * __expf(d);
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = 0.f;
                    }
                    st_bf16x8(sm + Lay::kP + sw128(row, j0 * 2), v);
                    st_bf16x8(sm + Lay::kP + sw128(row, j0 * 2 + 16), v + 8);
                }
                {
                    const uint32_t z[16] = {};
                    tmem_st16(tmem + kColQK + lane_off + col0, z);
                    tmem_st16(tmem + kColQK + lane_off + col0 + 16, z);
                }
                const float so = scale * eg_s[gs * 64 + row];
                const uint32_t ocol = (GATED && (c & 1)) ? kColO2 : kColO;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[16];
                    tmem_ld16(tmem + kColX + lane_off + col0 + half * 16, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(so * __uint_as_float(r[e]));
                    tmem_st16(tmem + ocol + lane_off + col0 + half * 16, r);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->xo_ready);
                // previous chunk's output stage, part 2, while this chunk's MMAs run
                if (GATED && c >= 1 && !(ok = gated_finish(c - 1))) break;
            } else {
                if (c >= 1 && !(ok = warp_all(wait_bar(&bs->o_done, (c - 1) & 1, abort, wlim)))) break;
                const float gate = gate_s[gs * 64 + row];
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int cc = col0 + half * 16;
                    float v[16], vg[16];
                    tmem_ld16f(tmem + kColX + lane_off + cc, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) vg[e] = v[e] * gate;
                    st_bf16x8(sm + Lay::kVN + sw128(row, cc * 2), v);
                    st_bf16x8(sm + Lay::kVN + sw128(row, cc * 2 + 16), v + 8);
                    st_bf16x8(sm + Lay::kVG + sw128(row, cc * 2), vg);
                    st_bf16x8(sm + Lay::kVG + sw128(row, cc * 2 + 16), vg + 8);
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->vn_ready);
            }
            if (!(ok = warp_all(spin_bar(&bs->h_done, c & 1, abort, wlim)))) break;
            tc_fence_after_sync();
            if (c + 1 < NT) {
#pragma unroll 1
                for (int blk = 0; blk < NF / 16; ++blk) {
                    const int f = f0 + blk * 16;
                    uint32_t r[16];
                    tmem_ld16(tmem + kColHT + lane_off + f, r);
                    tmem_wait_ld();
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        v[e] = __uint_as_float(r[e]);
                        r[e] = __float_as_uint(v[e] * d_next);
                    }
                    tmem_st16(tmem + kColHT + lane_off + f, r);
                    unsigned char *dst = sm + ((c + 1) & 1) * Lay::kStage + Lay::kStBbig + (f >> 6) * 16384;
                    st_bf16x8(dst + sw128(row, (f & 63) * 2), v);
                    st_bf16x8(dst + sw128(row, (f & 63) * 2 + 16), v + 8);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            mbar_arrive(&bs->hs_ready);
            if (upper) {
                if (!(ok = warp_all(wait_bar(&bs->o_done, c & 1, abort, wlim)))) break;
                tc_fence_after_sync();
                const int64_t oi = ((static_cast<int64_t>(b) * T + t0 + row) * H + h) * V +
                                   vt * kTcBV + col0;
                if (!nrank) {
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float v[16];
                        tmem_ld16f(tmem + kColO + lane_off + col0 + half * 16, v);
                        if (row < n) {
                            store_bf16x8_global(o + oi + half * 16, v);
                            store_bf16x8_global(o + oi + half * 16 + 8, v + 8);
                        }
                    }
                } else {
                    gated_send(c);   // output stage, part 1
                }
            }
        }
        // output stage, part 2 of the last chunk
        if (GATED && upper && warp_all(ok)) ok = gated_finish(NT - 1);
        // final state straight from tensor memory
        if (warp_all(ok) && h_final) {
            tc_fence_after_sync();
#pragma unroll 1
            for (int blk = 0; blk < NF / 16; ++blk) {
                float v[16];
                tmem_ld16f(tmem + kColHT + lane_off + f0 + blk * 16, v);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    h_final[state_off + static_cast<int64_t>(f0 + blk * 16 + e) * V + row] = v[e];
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // no CTA of a cluster leaves while another may still write its shared memory
    if (nrank) cluster_sync();
    if (tid == 0 && *abort) atomicOr(status, 1u);
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Stage export: A diag(beta), columns 0-63 of the bf16 workspace [B, T, H, 128],
// -> fp32 [B, T_pad, H, 64] (pad rows 0).
__global__ void export_abeta_kernel(const __nv_bfloat16 *__restrict__ src, float *__restrict__ dst,
                                    int B, int T, int T_pad, int H) {
    const int64_t n = static_cast<int64_t>(B) * T_pad * H * 64;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / 64;   // (b, t, h) in the padded layout
        const int hh = static_cast<int>(row % H);
        const int64_t bt = row / H;
        const int t = static_cast<int>(bt % T_pad), bb = static_cast<int>(bt / T_pad);
        dst[i] = t < T ? __bfloat162float(src[((static_cast<int64_t>(bb) * T + t) * H + hh) * 128 + i % 64])
                       : 0.f;
    }
}

template <int K>
cudaError_t launch_fused(const Args &a, const void *abeta, cudaStream_t s) {
    CUtensorMap mq, mk, mv, ma;
    if (!make_tmap_bthx(&mq, a.q, K, a.H, a.T, a.B) || !make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mv, a.v, a.V, a.H, a.T, a.B) ||
        !make_tmap_bthx(&ma, abeta, 128, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    // the row-sum region at the end is only used (and only allocated) with the output stage
    const int smem = static_cast<int>((a.gate ? TcLayout<K>::kBytes : TcLayout<K>::kRed) + 1024);
    const auto kernel = a.gate ? gdn_fused_tc_kernel<K, true> : gdn_fused_tc_kernel<K, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(a.V / kTcBV) * a.H * a.B;
    const int nrank = a.gate ? a.V / kTcBV : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.V / kTcBV, a.H, a.B);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    // With more CTAs than SMs the kernel may start while the WY kernel before
    // it in the stream finishes (it waits for that kernel's output after its
    // own setup), which saves about 5 us on B8 H64 T8192. With one wave or
    // less the early start gains nothing and cost 20 us (1.7%) on
    // B1 H32 T32768, so those grids launch after the WY kernel ends.
    if (ctas > sms) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (nrank) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = nrank;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr++].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    // kernel arguments, in order, for the untyped launch call
    const float *g_arg = a.g_chunk(), *h0_arg = a.h0, *rk_arg = a.rk, *nw_arg = a.norm_w;
    float *hf_arg = a.h_final;
    __nv_bfloat16 *o_arg = static_cast<__nv_bfloat16 *>(a.o);
    const __nv_bfloat16 *gate_arg = static_cast<const __nv_bfloat16 *>(a.gate);
    int T_arg = a.T, H_arg = a.H, V_arg = a.V, pf_arg = ctas <= sms ? 1 : 0;
    int norm_arg = (a.flags & GDN_FLAG_QK_L2NORM) ? 1 : 0, nrank_arg = nrank;
    float scale_arg = a.scale, eps_arg = a.norm_eps;
    uint32_t *status_arg = a.status;
    uint64_t wlim_arg = kWaitNs;
    int stall_arg = 0;
    if (const uint64_t armed = take_armed_stall()) {
        wlim_arg = armed;
        stall_arg = 1;
    }
    void *args[] = {&mq, &mk, &mv, &ma, &g_arg, &h0_arg, &hf_arg, &o_arg, &T_arg, &H_arg, &V_arg,
                    &scale_arg, &pf_arg, &status_arg, &norm_arg, &rk_arg, &gate_arg, &nw_arg,
                    &eps_arg, &nrank_arg, &wlim_arg, &stall_arg};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kernel), args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int K, int V, gdn_dtype dtype) {
    return dtype == GDN_BF16 && (K == 64 || K == 128) && V % kTcBV == 0 && V >= kTcBV;
}

size_t tc_workspace_bytes(int B, int T, int H, int, int) {
    return align_up(static_cast<size_t>(B) * T * H * 128 * sizeof(__nv_bfloat16));
}

int tc_launches(const char **names, int max_names) {
    static const char *const kNames[2] = {"gdn_wy_tc_kernel", "gdn_fused_tc_kernel"};
    for (int i = 0; names && i < 2 && i < max_names; ++i) names[i] = kNames[i];
    return 2;
}

cudaError_t tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m) {
    cudaError_t e = m.mark(0, s);
    if (e != cudaSuccess) return e;
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
