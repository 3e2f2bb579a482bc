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
//   W    [A diag(beta); A'] k           W rows 64-127 = w
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
#include "tc_sync.cuh"

namespace gdn {
namespace {

using namespace ptx;

// Two-kernel form (the WY kernel writes A to the workspace): 16 warps, 0 MMA
// issuer, 1 TMA producer, 2-5 prep group, 6-7 w epilogue, 8-15 chain group.
// Single-kernel form (FA: the A build runs in this kernel): 18 warps, 0 MMA
// issuer, 1 TMA producer, 2-3 prep group, 4-7 WY group, 8-15 chain group,
// 16-17 w epilogue. A warp reaches the TMEM lanes of quarter warp % 4 and runs
// on sub-partition warp % 4: the two-kernel form's w epilogue reads W from
// lanes 64-127, so that its work shares no sub-partition with the MMA issuer
// or with the chain warps that turn QK into P (lanes 0-63); on GB300 that
// placement ran 2.5-3% faster than w in lanes 0-63 with warps 4-5.
template <bool FA> constexpr int tc_threads() { return FA ? 576 : 512; }
template <bool FA> constexpr int prep_threads() { return FA ? 64 : 128; }
constexpr int kWThreads = 64, kChainThreads = 256, kWyThreads = 128;
constexpr int kTcBV = 64;
constexpr uint32_t kTmemCols = 512;

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
    static constexpr uint32_t kStAp = kStA + 8192;               // A': [A diag(beta); A'] is W's A operand
    static constexpr uint32_t kStage = kStAp + 8192;
    static constexpr uint32_t kP = 2 * kStage;                   // P
    static constexpr uint32_t kVN = kP + 8192;                   // v_new
    static constexpr uint32_t kVG = kVN + 8192;                  // v_g
    static constexpr uint32_t kG = kVG + 8192;                   // decay tables, 4 chunk slots
    static constexpr uint32_t kBar = kG + 5 * 4 * 64 * 4 + 16;
    // output stage: row sums of squares, [2 chunk slots][4 ranks][64 rows]
    static constexpr uint32_t kRed = kBar + 256;
    static constexpr uint32_t kBytes = kRed + 2 * 8 * 64 * 4;
};

// Single-kernel form: the WY matrix of every chunk is built in the kernel (the
// WY group, one chunk ahead of its use), so A never reaches HBM. Per stage
// [q; -w], [h^T; k] and v as above; once BIG has read a stage's q and -w, P
// takes the q half and v_new the -w half of its first 64-feature block, and v_g
// replaces v (read only by U). The A tiles are single-buffered, Z | A diag(beta)
// | A', written by the WY group after the previous chunk's W and U completed.
// The WY group keeps its own k tile (loaded a chunk ahead), [N1; N2] (Y in its
// second half after the first merge product), [X; U] (the fp32 diagonal blocks
// in its U half until X is built) and per-chunk tables for the prep group.
template <int K>
struct FaLayout {
    static constexpr int KB = K / 64;
    static constexpr uint32_t kStV = 2 * KB * 16384;             // [q; -w] and [h^T; k] first
    static constexpr uint32_t kStage = kStV + 8192;
    static constexpr uint32_t kZ = 2 * kStage, kA = kZ + 8192, kAp = kA + 8192;
    static constexpr uint32_t kWk = kAp + 8192;                  // WY k tile, KB x 8 KB
    static constexpr uint32_t kWn = kWk + KB * 8192;             // [N1; N2]
    static constexpr uint32_t kWxu = kWn + 16384;                // [X; U]
    // g, beta, beta exp(g) r, cf, r (64 floats each) and the scan total
    static constexpr uint32_t kWmisc = kWxu + 16384;
    // to the prep group, 4 chunk slots: the chunk's g (cumulative) and k-row factors
    static constexpr uint32_t kWtab = kWmisc + 1536;
    static constexpr uint32_t kG = kWtab + 2 * 4 * 64 * 4;
    static constexpr uint32_t kBar = kG + 5 * 4 * 64 * 4 + 16;
    static constexpr uint32_t kBytes = kBar + 256;
    static_assert(kBytes + 1024 <= 232448, "fits the 227 KB of shared memory a CTA may use");
};

// Per-chunk operand tiles of both forms, by stage s.
template <int K, bool FA>
struct Tiles {
    using L = TcLayout<K>;
    using F = FaLayout<K>;
    static constexpr uint32_t stage = FA ? F::kStage : L::kStage;
    static constexpr uint32_t bar = FA ? F::kBar : L::kBar;
    static constexpr uint32_t g = FA ? F::kG : L::kG;
    __host__ __device__ static constexpr uint32_t p(int s) { return FA ? s * F::kStage : L::kP; }
    __host__ __device__ static constexpr uint32_t vn(int s) { return FA ? s * F::kStage + 8192 : L::kVN; }
    __host__ __device__ static constexpr uint32_t vg(int s) { return FA ? s * F::kStage + F::kStV : L::kVG; }
    __host__ __device__ static constexpr uint32_t z(int s) { return FA ? F::kZ : s * L::kStage + L::kStZ; }
    __host__ __device__ static constexpr uint32_t ap(int s) { return FA ? F::kAp : s * L::kStage + L::kStAp; }
};

// TMEM columns: X-region [X (64) | QK (64)], O (64), W (K), HT (K).
constexpr uint32_t kColX = 0, kColQK = 64, kColO = 128, kColW = 192, kColHT = 320;
// Single-kernel form: the WY group's accumulator (Gram, merge products).
constexpr uint32_t kColWY = 448;
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
    uint64_t o_done2[2];                            // output stage: PV of chunk slot c % 2 done
    uint64_t o_free[2];                             // output stage: O of chunk slot c % 2 read
    // single-kernel form
    uint64_t a_ready;                               // WY group: A tiles of the next chunk
    uint64_t wu_done;                               // W and U of a chunk are done (A tiles free)
    uint64_t wy_mma, wyk_full;                      // WY group's MMAs and k tile
    uint64_t wy_tab[4];                             // WY group: tables of chunk slot c % 4
    uint32_t abort, tmem;
};
static_assert(sizeof(Bars) <= 256, "the barrier block has 256 bytes in both layouts");

// Named barrier 1 over the WY group's four warps (128 threads), and the same
// barrier reducing a predicate with OR over them.
__device__ __forceinline__ void wy_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool wy_any(bool x) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(x))
        : "memory");
    return r != 0;
}
// sigmoid(z) = (1 + tanh(z / 2)) / 2 with the hardware tanh: one special-function
// instruction instead of an exponential and a reciprocal. Those units are shared
// with the chain warps of the same sub-partitions, and with two per element they
// set the output stage's pace. Absolute error below 3e-4, far inside the bf16
// rounding of o.
__device__ __forceinline__ float sigmoid_tanh(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}
// GATED: the output stage (gated RMSNorm over V) with the V tiles of a head as
// one cluster of nrank_arg CTAs; without it the cluster code is compiled out.
// FA: the single-kernel form (A built here by the WY group; tm_a unused, g
// holds raw per-token log decays when raw_g is set, else the chunk-local
// cumulative sums; beta read here). Without FA, A diag(beta) and A' come from
// the WY kernel through tm_a, and g (and rk) from its workspace.
template <int K, bool GATED, bool FA>
__global__ void __launch_bounds__(tc_threads<FA>(), 1)
gdn_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                    const float *__restrict__ g, const float *__restrict__ h0,
                    float *__restrict__ h_final, __nv_bfloat16 *__restrict__ o, int T, int H, int V,
                    float scale, int l2_prefetch, uint32_t *status, int l2norm,
                    const float *__restrict__ rk, const __nv_bfloat16 *__restrict__ gate,
                    const float *__restrict__ norm_w, float norm_eps, int nrank_arg,
                    uint64_t wlim, int stall, const float *__restrict__ beta, int raw_g, int head0,
                    int dep_wait) {
    static_assert(!(GATED && FA), "the output stage runs on the two-kernel form");
    using Lay = TcLayout<K>;
    using FLay = FaLayout<K>;
    using Tl = Tiles<K, FA>;
    constexpr int kThreads = tc_threads<FA>();
    // with the output stage, the prep group's warps 4-5 run it instead
    constexpr int kPrepThreads = GATED ? 64 : prep_threads<FA>();
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
    float *tab = reinterpret_cast<float *>(sm + Tl::g);     // first 4 floats: g_last per slot (FA)
    float *eg_s = tab + 256;
    float *gate_s = tab + 512;
    float *rf_s = tab + 768;
    float *cf_s = tab + 1024;
    int *fz_s = reinterpret_cast<int *>(tab + 1280);
    Bars *bs = reinterpret_cast<Bars *>(sm + Tl::bar);
    volatile uint32_t *abort = &bs->abort;

    // one-dimensional grid over (head, V tile), heads from head0 on (b * H + h)
    const int nvt = V / kTcBV;
    const long long head = head0 + static_cast<long long>(blockIdx.x / nvt);
    const int vt = static_cast<int>(blockIdx.x % nvt), h = static_cast<int>(head % H),
              b = static_cast<int>(head / H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = (T + 63) / 64;

    // the zero tile(s), read by U as the zero half of its operand
    for (int i = tid; i < (FA ? 512 : 1024); i += kThreads)
        st_shared_v4(sm + Tl::z(i >> 9) + (i & 511) * 16, 0u, 0u, 0u, 0u);
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
            for (int i = 0; i < 2; ++i) {
                mbar_init(&bs->norm_bar[i], 1);
                mbar_init(&bs->o_done2[i], 1);
                mbar_init(&bs->o_free[i], 64);
            }
        if (FA) {
            mbar_init(&bs->a_ready, kWyThreads);
            mbar_init(&bs->wu_done, 1);
            mbar_init(&bs->wy_mma, 1);
            mbar_init(&bs->wyk_full, 1);
            for (int i = 0; i < 4; ++i) mbar_init(&bs->wy_tab[i], kWyThreads);
        }
        bs->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (!FA) prefetch_tmap(&tm_a);
    }
    tc_fence_before_sync();
    __syncthreads();
    // With the output stage the V tiles of one head run as a cluster (rank =
    // V tile); its barriers must be initialised before any CTA arrives on them.
    if (nrank) cluster_sync();
    // The setup above overlaps the WY kernel's last CTAs; everything below may
    // read its output. Launched behind the wide kernel (dep_wait = 0), the WY
    // kernel had completed before that one let this grid start.
    if (dep_wait) griddep_wait();
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
            // W = [A diag(beta); A'] k (w in rows 64-127), k read N-major from the
            // stage's [h^T; k]; single-kernel form: [A'; .] k (w in rows 0-63, the
            // rows under A' being whatever follows it). The other half's products
            // are unused.
            auto issue_w = [&](int s) {
                const TileDesc da(s_base + (FA ? Tl::ap(s) : s * Tl::stage + Lay::kStA), 16, 1024);
                const TileDesc db(s_base + s * Tl::stage + Lay::kStBbig + 8192, 16384, 1024);
                mma_bf16_k<false>(tmem + kColW, da.at(0), db.at(0), idW);
#pragma unroll
                for (int ks = 1; ks < 4; ++ks) mma_bf16_k<true>(tmem + kColW, da.at(ks * 32), db.at(ks * 2048), idW);
                mma_commit(&bs->w_done);
            };
            // X = [0; A diag(beta)] v
            auto issue_u = [&](int s) {
                const TileDesc da(s_base + Tl::z(s), 16, 1024);
                const TileDesc db(s_base + s * Tl::stage + Lay::kStV, 8192, 1024);
                mma_bf16_k<false>(tmem + kColX, da.at(0), db.at(0), idU);
#pragma unroll
                for (int ks = 1; ks < 4; ++ks) mma_bf16_k<true>(tmem + kColX, da.at(ks * 32), db.at(ks * 2048), idU);
            };
            // O += [P; .] v_new of chunk cp
            auto issue_pv = [&](int cp) {
                const TileDesc da(s_base + Tl::p(cp & 1), 16, 1024);
                const TileDesc db(s_base + Tl::vn(cp & 1), 8192, 1024);
                const uint32_t ocol = (GATED && (cp & 1)) ? kColO2 : kColO;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_k<true>(tmem + ocol, da.at(ks * 32), db.at(ks * 2048), idPV);
                mma_commit(&bs->o_done);
                if (GATED) mma_commit(&bs->o_done2[cp & 1]);
            };
            // single-kernel form: chunk c's A tiles are in (WY group) once a_ready
            // completes its phase c
            auto a_in = [&](int c) { return !FA || mbar_test_wait(&bs->a_ready, c & 1); };
            bool ok = spin_bar(&bs->full[0], 0, abort, wlim) && (!FA || spin_bar(&bs->a_ready, 0, abort, wlim));
            if (ok) {
                tc_fence_after_sync();
                issue_w(0);
                issue_u(0);
                if (FA) mma_commit(&bs->wu_done);   // chunk 0's A tiles are free again
            }
            for (int c = 0; ok && c < NT; ++c) {
                const int s = c & 1;
                const uint32_t par = c & 1;
                // X += [q; -w] [h^T | k] (q and k landed before W(c) was issued)
                if (!(ok = spin_bar(&bs->hs_ready, par, abort, wlim) && spin_bar(&bs->w_ready, par, abort, wlim)))
                    break;
                tc_fence_after_sync();
                const uint32_t st = s_base + s * Tl::stage;
                {
                    const TileDesc da(st + Lay::kStAbig, 16, 1024), db(st + Lay::kStBbig, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16_k<true>(tmem + kColX, da.at(off), db.at(off), idBIG);
                    }
                }
                mma_commit(&bs->big_done);
                // Next chunk's w as soon as its inputs land, if that happens before
                // v_new is ready; otherwise after HT(c), which must not queue behind
                // it in the in-order tensor pipe. One loop polls both.
                bool w_next = c + 1 < NT;
                {
                    const uint64_t t0 = globaltimer_ns();
                    for (uint32_t i = 1;; ++i) {
                        if (w_next && mbar_test_wait(&bs->full[s ^ 1], ((c + 1) >> 1) & 1) && a_in(c + 1)) {
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
                {
                    const TileDesc da(s_base + Tl::vg(s), 0, 1024), db(st + Lay::kStBbig + 8192, 16384, 1024);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_k<true>(tmem + kColHT, da.at(ks * 2048), db.at(ks * 2048), idHT);
                }
                mma_commit(&bs->h_done);
                // HT(c) is the stage's last reader; in the single-kernel form P and
                // v_new sit in the stage too, so PV(c) is
                if (!FA) mma_commit(&bs->empty[s]);
                if (w_next) {
                    if (!(ok = spin_bar(&bs->full[s ^ 1], ((c + 1) >> 1) & 1, abort, wlim) &&
                               (!FA || spin_bar(&bs->a_ready, (c + 1) & 1, abort, wlim))))
                        break;
                    tc_fence_after_sync();
                    issue_w(s ^ 1);
                }
                // once P, q h and v_new are out of the X-region: next chunk's u, then o
                if (!(ok = spin_bar(&bs->xo_ready, par, abort, wlim))) break;
                tc_fence_after_sync();
                if (c + 1 < NT) issue_u(s ^ 1);
                issue_pv(c);
                if (FA) {
                    mma_commit(&bs->wu_done);   // W(c + 1) and U(c + 1): the A tiles are free
                    mma_commit(&bs->empty[s]);
                }
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
                unsigned char *st = sm + s * Tl::stage;
                mbar_arrive_expect_tx(&bs->full[s], KB * 16384 + (FA ? 8192 : 24576));
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(st + Lay::kStAbig + kb * 16384, &tm_q, &bs->full[s], kb * 64, h, t0, b);
                    tma_load_4d(st + Lay::kStBbig + kb * 16384 + 8192, &tm_k, &bs->full[s], kb * 64, h,
                                t0, b);
                }
                tma_load_4d(st + Lay::kStV, &tm_v, &bs->full[s], vt * kTcBV, h, t0, b);
                if (!FA) {
                    tma_load_4d(st + Lay::kStA, &tm_a, &bs->full[s], 0, h, t0, b);
                    tma_load_4d(st + Lay::kStAp, &tm_a, &bs->full[s], 64, h, t0, b);
                }
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
                    if (!FA) {
                        tma_prefetch_4d(&tm_a, 0, h, tp, b);
                        tma_prefetch_4d(&tm_a, 64, h, tp, b);
                    }
                }
            }
            // no copy may still be landing in shared memory when the CTA exits
            // (after an abort the last loads may have no consumer)
            for (int c = max(stall ? 1 : 0, issued - 2); c < issued; ++c)
                mbar_wait(&bs->full[c & 1], (c >> 1) & 1, kWaitNs);
        }
    } else if (GATED && (warp == 4 || warp == 5)) {
        // ================================================================ output stage
        // Gated RMSNorm over the head's V columns, off the chunk chain. Warps
        // 4-5 sit on TMEM lane quarters 0-1, where O lives: one token row per
        // thread, all 64 of this CTA's columns. Per chunk c:
        //  - load the row's gate (in flight while O(c) is produced);
        //  - once PV(c) is done, send the row's sum of squares to every CTA of
        //    the cluster (slot c % 2, entry = rank) as asynchronous stores that
        //    complete bytes of the receiver's norm_bar;
        //  - with every sum in, normalise, gate and store the row, and hand
        //    O(c)'s columns back (o_free) for the O seed of chunk c + 2.
        // A slot is next written for chunk c + 2. That send follows the
        // sender's own finish of chunk c + 1, which waits for this CTA's sums
        // of chunk c + 1, which are sent only after this CTA has read its slot
        // for chunk c: neither the sums nor the barrier phase can be overtaken.
        const int orow = tid - 128;
        const uint32_t olane = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float *wv = norm_w + vt * kTcBV;
        for (int c = 0; c < NT; ++c) {
            const int slot = c & 1, t0 = c * 64;
            const bool valid = orow < min(64, T - t0);
            const int64_t oi = ((static_cast<int64_t>(b) * T + t0 + orow) * H + h) * V + vt * kTcBV;
            uint4 zr[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                zr[i] = valid ? reinterpret_cast<const uint4 *>(gate + oi)[i] : make_uint4(0u, 0u, 0u, 0u);
            // and the next chunk's row into L2
            if (orow < min(64, T - t0 - 64)) prefetch_l2(gate + oi + static_cast<int64_t>(64) * H * V);
            if (!warp_all(wait_bar(&bs->o_done2[slot], (c >> 1) & 1, abort, wlim))) break;
            tc_fence_after_sync();
            const uint32_t ob = slot ? kColO2 : kColO;
            float ss = 0.f;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                tmem_ld16f(tmem + ob + olane + blk * 16, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) ss = fmaf(v[e], v[e], ss);
            }
            const uint32_t red = s_base + Lay::kRed + ((slot * 4 + vt) * 64 + orow) * 4;
            const uint32_t nb = smem_u32(&bs->norm_bar[slot]);
            // this CTA expects one sum per row from each CTA of the cluster
            if (warp == 4 && lane == 0) mbar_arrive_expect_tx(&bs->norm_bar[slot], nrank * 64 * 4);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (r < nrank) st_async_cluster_f32(mapa_shared(red, r), ss, mapa_shared(nb, r));
            if (!warp_all(wait_bar_cluster(&bs->norm_bar[slot], (c >> 1) & 1, abort, wlim))) break;
            const float *sums = reinterpret_cast<const float *>(sm + Lay::kRed) + slot * 256;
            float tot = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (r < nrank) tot += sums[r * 64 + orow];
            const float rstd = rsqrtf(tot / V + norm_eps);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16], y[16];
                tmem_ld16f(tmem + ob + olane + blk * 16, v);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint4 z4 = zr[blk * 2 + i];
                    const uint32_t w4[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = i * 8 + 2 * e;
                        const float z0 = __uint_as_float(w4[e] << 16);
                        const float z1 = __uint_as_float(w4[e] & 0xffff0000u);
                        y[j] = v[j] * rstd * wv[blk * 16 + j] * sigmoid_tanh(z0);
                        y[j + 1] = v[j + 1] * rstd * wv[blk * 16 + j + 1] * sigmoid_tanh(z1);
                    }
                }
                if (valid) {
                    store_bf16x8_global(o + oi + blk * 16, y);
                    store_bf16x8_global(o + oi + blk * 16 + 8, y + 8);
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&bs->o_free[slot]);
        }
    } else if (FA ? (warp == 2 || warp == 3) : (warp >= 2 && warp < 6)) {
        // ================================================================ prep group
        // Per-chunk decay tables (A' = A diag(beta exp(g)) comes with A diag(beta)
        // from the WY kernel or, in the single-kernel form, from the WY group,
        // which also hands over the chunk's cumulative g and k-row factors).
        const int ptid = tid - 64;
        const float *gcum_t = reinterpret_cast<const float *>(sm + FLay::kWtab);
        const float *rk_t = gcum_t + 256;
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
        float g_next = FA ? 0.f : load_g(0), gl_next = FA ? 0.f : load_gl(0);
        float rk_next = FA ? 1.f : load_rk(0);
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1, gs = c & 3;
            const int n = min(64, T - c * 64);
            float g_cur = g_next, gl = gl_next, rk_cur = rk_next;
            if (FA) {
                // the WY group's tables of this chunk (slot c % 4; their next
                // writer, chunk c + 4, needs U(c + 3), which needs these tables)
                if (!wait_bar(&bs->wy_tab[gs], (c >> 2) & 1, abort, wlim)) break;
                g_cur = gcum_t[gs * 64 + ptid];
                gl = gcum_t[gs * 64 + n - 1];
                rk_cur = rk_t[gs * 64 + ptid];
                if (ptid == 0) tab[gs] = gl;   // the chain group's g_last of this chunk
            } else {
                g_next = load_g(c + 1);
                gl_next = load_gl(c + 1);
                rk_next = load_rk(c + 1);
            }
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
                    const unsigned char *qrow = sm + s * Tl::stage + Lay::kStAbig + ptid * 128;
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
    } else if (FA ? warp >= 16 : (warp == 6 || warp == 7)) {
        // ================================================================ w epilogue
        // The w rows of W (lanes 64-127, quarters 2-3; single-kernel form lanes
        // 0-63, quarters 0-1) -> -w, bf16, under q in the stage's stacked
        // operand (that half was last read by BIG(c - 2)).
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
                unsigned char *base = sm + (c & 1) * Tl::stage + Lay::kStAbig + (f0 >> 6) * 16384;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_bf16x8(base + sw128(64 + (row & 63), (f0 & 63) * 2 + q * 16), v + q * 8);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->w_ready);
        }
    } else if (FA && warp < 8) {
        // ================================================================ WY group
        // Single-kernel form: A = (I + L)^-1 of every chunk, in order, with
        // L_ij = beta_i (k_i . k_j) exp(g_i - g_j) for i > j; written as
        // A diag(beta) (U's operand) and A' = A diag(beta exp(g)) (W's). With X
        // the inverse of the four 16x16 diagonal blocks of I + L (forward
        // substitution in fp32), N1 its off-diagonal blocks (1,0) and (3,2) and
        // N2 its bottom-left 32x32 block:
        //   A0 = X - X N1 X,  A = A0 - A0 N2 A0
        // ((D + N)^-1 = D^-1 - D^-1 N D^-1 when N D^-1 N = 0), formed from the
        // Gram matrix in three stacked M = 128 products, each subtraction in the
        // fp32 accumulator:
        //   G = k k^T;  [Y1; U] = [N1; N2] X;  [A0; Y2] = [X; U] + [X; U](-Y1);
        //   A = A0 + A0 (-Y2).
        // The group loads its own copy of each chunk's k (a chunk ahead), takes
        // the chunk-local sum of raw decays and the k-row norms when the flags
        // ask, and hands g, the norms and the A tiles to the other roles.
        const int wtid = tid - 128, ww = warp - 4;     // ww = this warp's lane quarter
        const uint32_t lane_off = static_cast<uint32_t>(ww * 32) << 16;
        const uint32_t tw = tmem + kColWY;
        float *Ld = reinterpret_cast<float *>(sm + FLay::kWxu + 8192);
        float *g_s = reinterpret_cast<float *>(sm + FLay::kWmisc);
        float *b_s = g_s + 64, *eb_s = g_s + 128, *wcf_s = g_s + 192, *rk_s = g_s + 256;
        float *tot_s = g_s + 320;
        float *gcum_t = reinterpret_cast<float *>(sm + FLay::kWtab), *rk_t = gcum_t + 256;
        const uint32_t s_k = s_base + FLay::kWk, s_n = s_base + FLay::kWn;
        const uint32_t s_xu = s_base + FLay::kWxu, s_y = s_n + 8192;
        unsigned char *n_t = sm + FLay::kWn, *xu_t = sm + FLay::kWxu, *y_t = n_t + 8192;
        uint32_t mph = 0;            // next phase of wy_mma
        int k_loaded = 0;            // chunks whose k tile was requested
        bool mma_out = false;        // an MMA whose completion was not seen
        bool ok = true;
        auto load_k = [&](int j) {   // one thread
            mbar_arrive_expect_tx(&bs->wyk_full, KB * 8192);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                tma_load_4d(sm + FLay::kWk + kb * 8192, &tm_k, &bs->wyk_full, kb * 64, h, j * 64, b);
        };
        // one MMA group (A K-major; B K-major or rows along N) issued by one thread
        // (M = 128, N = 64; the first product overwrites, the merges accumulate)
        auto mma_issue = [&](uint32_t a, uint32_t bop, bool b_mn, int ksteps, bool acc) {
            if (wtid == 0) {
                tc_fence_after_sync();
                const uint32_t id = idesc_bf16(128, 64, false, b_mn);
                const TileDesc da(a, 16, 1024), db(bop, 8192, 1024);
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint32_t a_off = (ks >> 2) * 8192 + (ks & 3) * 32;
                    const uint64_t bd = db.at(b_mn ? ks * 2048 : a_off);
                    if (acc || ks > 0)
                        mma_bf16_k<true>(tw, da.at(a_off), bd, id);
                    else
                        mma_bf16_k<false>(tw, da.at(a_off), bd, id);
                }
                mma_commit(&bs->wy_mma);
            }
            mma_out = true;
        };
        // every thread of the group waits for it; false: give up (abort)
        // one warp polls, the others wait at the group barrier
        auto mma_wait = [&]() -> bool {
            const bool got = ww != 0 || warp_all(spin_bar(&bs->wy_mma, mph, abort, wlim));
            const bool all = !wy_any(!got);
            if (all) {
                mph ^= 1;
                mma_out = false;
            }
            tc_fence_after_sync();
            return all;
        };
        auto load16 = [&](int blk, float *v) {
            uint32_t t[16];
            tmem_ld16(tw + lane_off + blk * 16, t);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(t[e]);
        };
        if (wtid == 0 && NT > 0) {
            load_k(0);
            k_loaded = 1;
        }
        for (int j = 0; j < NT && ok; ++j) {
            const int t0 = j * 64, n = min(64, T - t0), slot = j & 3;
            const int64_t my_row = (static_cast<int64_t>(b) * T + t0 + wtid) * H + h;
            float gv = 0.f, bv = 0.f;
            if (wtid < n) {
                gv = g[my_row];
                bv = beta[my_row];
            }
            if (raw_g) {
                // inclusive sum over the chunk: tokens 0-31 in the first warp,
                // 32-63 in the second, one shared total between them
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gv, off);
                    if (lane >= off) gv += y;
                }
                if (wtid == 31) *tot_s = gv;
                wy_sync();
                if (ww == 1) gv += *tot_s;
                if (wtid >= n) gv = 0.f;
            }
            // the previous chunk's readers of these tables are past the barrier
            // that ended its A tiles
            if (wtid < 64) {
                g_s[wtid] = gv;
                b_s[wtid] = bv;
                rk_s[wtid] = 1.f;
            }
            wy_sync();
            const float g_last = g_s[n - 1];
            const float g_ref = 0.5f * g_last;
            const bool fz = fabsf(g_last) <= 160.f;   // |g_i - g_ref| <= |g_last| / 2 for decays <= 0
            if (wtid < 64) {
                eb_s[wtid] = bv * __expf(gv);
                wcf_s[wtid] = wtid < n ? __expf(g_ref - gv) : 0.f;
            }
            // ---- this chunk's k tile, then G = k k^T issued as M = 128 (rows
            // past the k tile are whatever follows it; their products are unused)
            if (!(ok = !wy_any(ww == 0 && !warp_all(spin_bar(&bs->wyk_full, j & 1, abort, wlim))))) break;
            mma_issue(s_k, s_k, false, K / 16, false);
            if (l2norm && wtid < 64) {
                // |k_i|^2 from the k tile while the Gram runs (the swizzle only
                // permutes 16-byte chunks within a row)
                float ss = 0.f;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(sm + FLay::kWk + kb * 8192 + wtid * 128 +
                                                                         ((jj ^ (wtid & 7)) * 16));
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                        }
                    }
                const float r = rsqrtf(ss + kL2NormEps);
                rk_s[wtid] = r;
                wcf_s[wtid] *= r;
                eb_s[wtid] *= r;
            }
            if (!(ok = mma_wait())) break;
            // the Gram and the norms have read the k tile: the next chunk's may land
            if (wtid == 0 && j + 1 < NT) {
                load_k(j + 1);
                k_loaded = j + 2;
            }
            if (ww < 2) {
                const int r = ww * 32 + lane, rb = r >> 4;
                const float gr = g_s[r], br = b_s[r] * rk_s[r];
                const float rf = br * __expf(gr - g_ref);
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    float v[16];
                    load16(blk, v);
                    if (fz) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 c4 = *reinterpret_cast<const float4 *>(wcf_s + blk * 16 + 4 * m);
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
                            const int jj = blk * 16 + e;
                            const float d = (jj < r) ? gr - g_s[jj] : -INFINITY;
                            v[e] = br * v[e] * rk_s[jj] * __expf(d);
                        }
                    }
                    if (blk == rb) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) Ld[(rb * 16 + (r & 15)) * 17 + e] = v[e];
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
                    st_bf16x8(n_t + sw128(r, blk * 32), n1);
                    st_bf16x8(n_t + sw128(r, blk * 32 + 16), n1 + 8);
                    st_bf16x8(n_t + 8192 + sw128(r, blk * 32), n2);
                    st_bf16x8(n_t + 8192 + sw128(r, blk * 32 + 16), n2 + 8);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            wy_sync();
            // ---- X: inverse of each 16x16 unit-lower diagonal block, column per thread
            {
                float x[16];
                const int blk = wtid >> 4, col = wtid & 15;
                float *Lb = Ld + blk * 16 * 17;
                if (wtid < 64) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
                    for (int jj = 0; jj < 15; ++jj)
#pragma unroll
                        for (int i = jj + 1; i < 16; ++i) x[i] = fmaf(-Lb[i * 17 + jj], x[jj], x[i]);
                }
                wy_sync();
                if (wtid < 64) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) Lb[i * 17 + col] = x[i];
                }
                wy_sync();
            }
            // From here on thread t owns row t of the M = 128 accumulators: rows
            // 0-63 belong to X / A0 / A, rows 64-127 to U / Y2.
            const int r = wtid & 63, rb = r >> 4;
            float xr[16];   // row r of X (threads < 64): its diagonal block
            if (wtid < 64) {
                const float z8[8] = {};
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) xr[jj] = Ld[(rb * 16 + (r & 15)) * 17 + jj];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    if ((ch >> 1) == rb)
                        st_bf16x8(xu_t + sw128(r, ch * 16), xr + (ch & 1) * 8);
                    else
                        st_bf16x8(xu_t + sw128(r, ch * 16), z8);
                }
            }
            fence_proxy_async_smem();
            wy_sync();
            // ---- [Y1; U] = [N1; N2] X
            mma_issue(s_n, s_xu, true, 4, false);
            if (!(ok = mma_wait())) break;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                load16(blk, v);
                if (wtid < 64) {
                    // -Y1, the B operand (rows along N) of the next product
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = -v[e];
                    st_bf16x8(y_t + sw128(r, blk * 32), v);
                    st_bf16x8(y_t + sw128(r, blk * 32 + 16), v + 8);
                } else {
                    // U, the second half of the A operand [X; U]; its fp32 copy
                    // stays in the accumulator
                    st_bf16x8(xu_t + 8192 + sw128(r, blk * 32), v);
                    st_bf16x8(xu_t + 8192 + sw128(r, blk * 32 + 16), v + 8);
                }
            }
            if (wtid < 64) {
                // the accumulator's rows 0-63 start the next product from X
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t t[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) t[e] = blk == rb ? __float_as_uint(xr[e]) : 0u;
                    tmem_st16(tw + lane_off + blk * 16, t);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            wy_sync();
            // ---- [A0; Y2] = [X; U] + [X; U] (-Y1)
            mma_issue(s_xu, s_y, true, 4, true);
            if (!(ok = mma_wait())) break;
            tc_fence_before_sync();
            wy_sync();   // every MMA operand read before A0 / -Y2 overwrite them
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                load16(blk, v);
                if (wtid < 64) {
                    // A0 as the next A operand (its fp32 copy stays in the accumulator)
                    st_bf16x8(xu_t + sw128(r, blk * 32), v);
                    st_bf16x8(xu_t + sw128(r, blk * 32 + 16), v + 8);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = -v[e];
                    st_bf16x8(y_t + sw128(r, blk * 32), v);
                    st_bf16x8(y_t + sw128(r, blk * 32 + 16), v + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            wy_sync();
            // ---- A = A0 + A0 (-Y2) in rows 0-63 (rows 64-127 of the product are unused)
            mma_issue(s_xu, s_y, true, 4, true);
            if (!(ok = mma_wait())) break;
            // the A tiles are free once W and U of the previous chunk are done
            if (j >= 1 && !(ok = !wy_any(ww == 0 && !warp_all(spin_bar(&bs->wu_done, (j - 1) & 1, abort, wlim)))))
                break;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float v[16];
                load16(blk, v);
                if (wtid < 64) {
                    float v2[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float a = v[e];
                        v[e] = a * b_s[blk * 16 + e];
                        v2[e] = a * eb_s[blk * 16 + e];
                    }
                    st_bf16x8(sm + FLay::kA + sw128(r, blk * 32), v);
                    st_bf16x8(sm + FLay::kA + sw128(r, blk * 32 + 16), v + 8);
                    st_bf16x8(sm + FLay::kAp + sw128(r, blk * 32), v2);
                    st_bf16x8(sm + FLay::kAp + sw128(r, blk * 32 + 16), v2 + 8);
                }
            }
            // tables of this chunk for the prep group: g (summed), k-row factors
            if (wtid < 64) {
                gcum_t[slot * 64 + wtid] = g_s[wtid];
                rk_t[slot * 64 + wtid] = wtid < n ? rk_s[wtid] : 1.f;
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->wy_tab[slot]);
            mbar_arrive(&bs->a_ready);
            wy_sync();   // every thread is done with this chunk's tables and accumulator
        }
        // nothing of the group may still land in shared memory or write tensor
        // memory when the CTA exits (after an abort)
        if (wtid == 0) {
            if (mma_out) mbar_wait(&bs->wy_mma, mph, kWaitNs);
            // a requested k tile whose wait did not complete: its phase is the
            // one of chunk k_loaded - 1
            if (!ok && k_loaded > 0) mbar_wait(&bs->wyk_full, (k_loaded - 1) & 1, kWaitNs);
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
        // pre-decayed by exp(g_last) of chunk 0 (in the single-kernel form the
        // prep group has it, once the WY group summed the chunk)
        {
            float d0 = 1.f;
            if (!FA)
                d0 = __expf(g_last_of(0));
            else if (warp_all(wait_bar(&bs->g_ready[0], 0, abort, wlim)))
                d0 = __expf(tab[0]);   // else the run is aborting and the loop below leaves
#pragma unroll 1
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
        float g_last_next = (!FA && NT > 1) ? g_last_of(1) : 0.f;
        for (int c = 0; c < NT; ++c) {
            const int t0 = c * 64, n = min(64, T - t0), gs = c & 3;
            float d_next = (!FA && c + 1 < NT) ? __expf(g_last_next) : 1.f;
            if (!FA && c + 2 < NT) g_last_next = g_last_of(c + 2);   // one chunk ahead
            if (!(ok = warp_all(wait_bar(&bs->g_ready[gs], (c >> 2) & 1, abort, wlim) &&
                                nap_bar(&bs->big_done, c & 1, abort, wlim, kNapNs))))
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
                    st_bf16x8(sm + Tl::p(c & 1) + sw128(row, j0 * 2), v);
                    st_bf16x8(sm + Tl::p(c & 1) + sw128(row, j0 * 2 + 16), v + 8);
                }
                {
                    const uint32_t z[16] = {};
                    tmem_st16(tmem + kColQK + lane_off + col0, z);
                    tmem_st16(tmem + kColQK + lane_off + col0 + 16, z);
                }
                // with the output stage, O(c - 2) (same columns) must have been read
                if (GATED && c >= 2 &&
                    !(ok = warp_all(wait_bar(&bs->o_free[c & 1], ((c >> 1) + 1) & 1, abort, wlim))))
                    break;
                tc_fence_after_sync();
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
                    st_bf16x8(sm + Tl::vn(c & 1) + sw128(row, cc * 2), v);
                    st_bf16x8(sm + Tl::vn(c & 1) + sw128(row, cc * 2 + 16), v + 8);
                    st_bf16x8(sm + Tl::vg(c & 1) + sw128(row, cc * 2), vg);
                    st_bf16x8(sm + Tl::vg(c & 1) + sw128(row, cc * 2 + 16), vg + 8);
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->vn_ready);
            }
            if (FA && c + 1 < NT) {
                // the next chunk's g_last, from the prep group's table of it
                if (!(ok = warp_all(wait_bar(&bs->g_ready[(c + 1) & 3], ((c + 1) >> 2) & 1, abort, wlim))))
                    break;
                d_next = __expf(tab[(c + 1) & 3]);
            }
            if (!(ok = warp_all(nap_bar(&bs->h_done, c & 1, abort, wlim, kNapNs)))) break;
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
                    unsigned char *dst = sm + ((c + 1) & 1) * Tl::stage + Lay::kStBbig + (f >> 6) * 16384;
                    st_bf16x8(dst + sw128(row, (f & 63) * 2), v);
                    st_bf16x8(dst + sw128(row, (f & 63) * 2 + 16), v + 8);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            mbar_arrive(&bs->hs_ready);
            if (upper && !GATED) {
                if (!(ok = warp_all(wait_bar(&bs->o_done, c & 1, abort, wlim)))) break;
                tc_fence_after_sync();
                const int64_t oi = ((static_cast<int64_t>(b) * T + t0 + row) * H + h) * V +
                                   vt * kTcBV + col0;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float v[16];
                    tmem_ld16f(tmem + kColO + lane_off + col0 + half * 16, v);
                    if (row < n) {
                        store_bf16x8_global(o + oi + half * 16, v);
                        store_bf16x8_global(o + oi + half * 16 + 8, v + 8);
                    }
                }
            }
        }
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
    // Launched behind the wide kernel without waiting on it: this grid ends no
    // sooner than that one, so whatever follows in the stream sees both done.
    if (!dep_wait) griddep_wait();
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

// fa: the single-kernel form (abeta unused); else the second kernel of the
// two-kernel form, reading A from abeta.
// heads [head0, head0 + nheads) of the B * H; after_wide: launched right behind
// gdn_wide_tc_kernel, which covered the other heads (early start, no wait on it)
template <int K>
cudaError_t launch_fused(const Args &a, const void *abeta, cudaStream_t s, bool fa, long long head0,
                         long long nheads, bool after_wide) {
    CUtensorMap mq, mk, mv, ma;
    if (!make_tmap_bthx(&mq, a.q, K, a.H, a.T, a.B) || !make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mv, a.v, a.V, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    if (fa)
        ma = mk;   // a valid map the kernel never reads
    else if (!make_tmap_bthx(&ma, abeta, 128, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    // the row-sum region at the end is only used (and only allocated) with the output stage
    const int smem = static_cast<int>(
        (fa ? FaLayout<K>::kBytes : a.gate ? TcLayout<K>::kBytes : TcLayout<K>::kRed) + 1024);
    const auto kernel = fa ? gdn_fused_tc_kernel<K, false, true>
                           : a.gate ? gdn_fused_tc_kernel<K, true, false> : gdn_fused_tc_kernel<K, false, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(a.V / kTcBV) * nheads;
    const int nrank = a.gate ? a.V / kTcBV : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(fa ? tc_threads<true>() : tc_threads<false>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    // With more CTAs than SMs the kernel may start while the WY kernel before
    // it in the stream finishes (it waits for that kernel's output after its
    // own setup), which saves about 5 us on B8 H64 T8192. With one wave or
    // less the early start gains nothing and cost 20 us (1.7%) on
    // B1 H32 T32768, so those grids launch after the WY kernel ends.
    if (!fa && (ctas > sms || after_wide)) {
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
    // the single-kernel form sums raw decays itself
    const float *g_arg = fa ? a.g : a.g_chunk(), *h0_arg = a.h0, *rk_arg = a.rk, *nw_arg = a.norm_w;
    const float *beta_arg = a.beta;
    int rawg_arg = (fa && (a.flags & GDN_FLAG_RAW_G)) ? 1 : 0;
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
    int head0_arg = static_cast<int>(head0), dep_arg = after_wide ? 0 : 1;
    void *args[] = {&mq, &mk, &mv, &ma, &g_arg, &h0_arg, &hf_arg, &o_arg, &T_arg, &H_arg, &V_arg,
                    &scale_arg, &pf_arg, &status_arg, &norm_arg, &rk_arg, &gate_arg, &nw_arg,
                    &eps_arg, &nrank_arg, &wlim_arg, &stall_arg, &beta_arg, &rawg_arg, &head0_arg, &dep_arg};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kernel), args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int K, int V, gdn_dtype dtype) {
    return dtype == GDN_BF16 && (K == 64 || K == 128) && V % kTcBV == 0 && V >= kTcBV;
}

// A diag(beta) | A' (bf16 [B, T, H, 128]).
size_t tc_abeta_bytes(int B, int T, int H) {
    return align_up(static_cast<size_t>(B) * T * H * 128 * sizeof(__nv_bfloat16));
}
size_t tc_workspace_bytes(int B, int T, int H, int, int) { return tc_abeta_bytes(B, T, H); }

// Heads of the two-kernel form's plain call that the wide kernel takes: all
// of them, or (form kTwo) only whole waves of its CTAs when the rest fit one
// wave of 64-column CTAs, which finish their chains sooner than a partial
// wave of wide CTAs would.
long long tc_wide_heads(TcForm form, int B, int H, int V) {
    const long long heads = static_cast<long long>(B) * H;
    if (form != TcForm::kTwo) return heads;
    const int nvt = V / 128, sms = tc_sm_count();
    const long long ctas = heads * nvt;
    if (ctas <= sms) return heads;
    const long long wide_heads = (ctas / sms) * sms / nvt;
    return (heads - wide_heads) * (V / 64) <= sms ? wide_heads : heads;
}

// Kernel names of the call, with or without the output stage.
int tc_launches(TcForm form, int B, int H, int V, const char **names, int max_names) {
    if (form == TcForm::kSingle) {
        if (names && max_names > 0) names[0] = "gdn_fused_tc_kernel";
        return 1;
    }
    const bool wide = form == TcForm::kWide || tc_wide(B, H, V);
    const bool split = wide && tc_wide_heads(form, B, H, V) < static_cast<long long>(B) * H;
    const char *const all[3] = {"gdn_wy_tc_kernel", wide ? "gdn_wide_tc_kernel" : "gdn_fused_tc_kernel",
                                "gdn_fused_tc_kernel"};
    const int n = split ? 3 : 2;
    for (int i = 0; names && i < n && i < max_names; ++i) names[i] = all[i];
    return n;
}

cudaError_t tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m, TcForm form) {
    cudaError_t e = m.mark(0, s);
    if (e != cudaSuccess) return e;
    if (form == TcForm::kSingle) {
        // single kernel: the WY matrix is built in the forward kernel itself
        const long long heads = static_cast<long long>(a.B) * a.H;
        e = (a.K == 128) ? launch_fused<128>(a, nullptr, s, true, 0, heads, false)
                         : launch_fused<64>(a, nullptr, s, true, 0, heads, false);
        if (e != cudaSuccess) return e;
        return m.mark(1, s);
    }
    if ((e = wy_tc_forward(a, ws, s)) != cudaSuccess) return e;
    if ((e = m.mark(1, s)) != cudaSuccess) return e;
    const long long heads = static_cast<long long>(a.B) * a.H;
    if (form == TcForm::kWide || tc_wide(a.B, a.H, a.V)) {
        // whole waves on the wide kernel, the last partial one on the 64-column
        // one; the output stage runs inside either (the head's CTAs of either
        // as a cluster when a row spans several)
        const long long wh = tc_wide_heads(form, a.B, a.H, a.V);
        if ((e = wide_tc_forward(a, ws, s, wh)) != cudaSuccess) return e;
        if (wh == heads) return m.mark(2, s);
        if ((e = m.mark(2, s)) != cudaSuccess) return e;
        e = (a.K == 128) ? launch_fused<128>(a, ws, s, false, wh, heads - wh, m.ev == nullptr)
                         : launch_fused<64>(a, ws, s, false, wh, heads - wh, m.ev == nullptr);
        if (e != cudaSuccess) return e;
        return m.mark(3, s);
    }
    e = (a.K == 128) ? launch_fused<128>(a, ws, s, false, 0, heads, false)
                     : launch_fused<64>(a, ws, s, false, 0, heads, false);
    if (e != cudaSuccess) return e;
    return m.mark(2, s);
}

cudaError_t tc_export_abeta(const Args &a, const void *ws, float *dst, cudaStream_t s) {
    export_abeta_kernel<<<304, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(ws), dst, a.B, a.T,
                                           a.T_pad, a.H);
    return cudaGetLastError();
}

}  // namespace gdn
