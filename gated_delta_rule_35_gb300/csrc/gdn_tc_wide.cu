// Forward kernel of the two-kernel tensor-core form with both 64-column V tiles
// of a 128-wide V block in one CTA (recompute_w_u, chunk_fwd_h and chunk_fwd_o
// of the "WarpDrive" page, its kernels 5, 3 and 4, fused as in gdn_tc.cu).
//
// gdn_fused_tc_kernel runs one (b, h, 64-wide V tile) per CTA and one CTA per
// SM, so every chunk of a head computes W = A' k, q k^T, P and loads q, k and A
// once per V tile. Here one CTA owns a 128-wide V block: those are computed
// once, and every MMA of the chain covers 128 (or 192) columns, so each
// instruction does twice the work. Per chunk c (accumulators in TMEM, one row
// per lane; "." rows are never read):
//   W    [A'; 0] k or [0; A'] k          w in the lane half that O(c) does not use
//   U    [0; A diag(beta)] v or [A diag(beta); 0] v   u in the lanes of v_new
//   BIG  [q; -w] [k; h^T] or [-w; q] [h^T; k]   X = [q h; u - w h], QK = q k^T
//   HT   v_g^T k                         h^T += v_g^T k (fp32, pre-decayed)
//   PV   [P; 0] v_new or [0; P] v_new    O += P v_new
// The shared-memory budget (two q / k stages, 128 rows of h^T, 128-wide v,
// v_new and v_g tiles) only fits with -w and h^T single-buffered. They sit
// between the two stages' q (k) tiles, [q0 | -w | q1] and [k0 | h^T | k1],
// so that BIG's operands are [q0; -w] and [k0; h^T] for even chunks and
// [-w; q1] and [h^T; k1] for odd ones. Which TMEM lane half holds q's rows, and
// which columns hold X and QK, therefore alternate with the chunk's parity, and
// so do the chain warps' roles. The A operands of W, U and PV take their zero
// half from a row of tiles [0 | A' | 0 | P | 0 | A diag(beta) | 0], so that W
// and O share 128 TMEM columns by lane halves: an MMA whose A rows are zero
// adds exact zeros to the other half. It still reads and rewrites that half,
// so no thread may store into it meanwhile: W(c + 1) waits until O(c) is
// seeded, and the readers of O clear it before the W that follows is issued.
#include "gdn_internal.h"
#include "tc_common.cuh"
#include "tc_sync.cuh"

namespace gdn {
namespace {

using namespace ptx;

// 22 warps: 0 MMA issuer, 1 TMA producer, 2-5 aux group (decay tables, and the
// w epilogue on the lane quarter of the chunk's W), 6-21 chain group (four
// warps per lane quarter). A warp reaches the TMEM lanes of quarter warp % 4.
constexpr int kWideThreads = 704;
constexpr int kWideBV = 128;
constexpr int kAuxThreads = 128, kChainWarps = 16;
constexpr uint32_t kWideTmemCols = 512;
// TMEM columns: BIG's accumulator [X | QK] or [QK | X] (192), HT (K), W / O (128).
constexpr uint32_t kCBig = 0, kCHT = 192, kCWO = 320;
// With the output stage in the kernel (V = 128): a lane's o row, rounded to
// bf16 and packed in pairs, between its write and its normalisation.
constexpr uint32_t kCStash = 448;
// The stage's rows span at most two CTAs (V <= 256), a thread-block cluster of
// V / 128.
constexpr int kWideMaxRanks = 2;
static_assert(kCWO + kWideBV <= kCStash && kCStash + kWideBV / 2 <= kWideTmemCols, "the stash fits");

// Shared-memory map (bytes from a 1024-aligned base); every tile is 64 rows of
// 128 bytes (h^T: 128 rows) with the 128-byte swizzle, as TMA writes it.
template <int K>
struct WideLayout {
    static constexpr int KB = K / 64;                     // 64-feature blocks
    static constexpr uint32_t kQWBlk = 24576, kKHBlk = 32768;
    static constexpr uint32_t kQW = 0;                    // per block: q0 | -w | q1
    static constexpr uint32_t kKH = KB * kQWBlk;          // per block: k0 | h^T (128 rows) | k1
    static constexpr uint32_t kZx = kKH + KB * kKHBlk;
    static constexpr uint32_t kAp = kZx + 8192, kZy = kAp + 8192, kP = kZy + 8192, kZz = kP + 8192;
    static constexpr uint32_t kAb = kZz + 8192, kZw = kAb + 8192;
    static constexpr uint32_t kV = kZw + 8192;            // v, two 64-column atoms (single)
    static constexpr uint32_t kVN = kV + 16384;           // v_new
    static constexpr uint32_t kVG = kVN + 16384;          // v_g
    static constexpr uint32_t kG = kVG + 16384;           // decay tables, 4 chunk slots
    static constexpr uint32_t kBar = kG + 5 * 4 * 64 * 4 + 16;
    static constexpr uint32_t kNw = kBar + 256;           // output stage: norm weight (128 floats)
    // output stage with a row over a cluster: each row's partial sums of
    // squares from every CTA of the cluster, [chunk slot (4)][rank][64 rows]
    static constexpr uint32_t kSums = kNw + kWideBV * 4;
    static constexpr uint32_t kBytes = kSums + 4 * kWideMaxRanks * 64 * 4;
    static_assert(kBytes + 1024 <= 232448, "fits the 227 KB of shared memory a CTA may use");
    // q / k tile of chunk parity p within a block; -w and h^T sit between them
    __host__ __device__ static constexpr uint32_t qslot(int p) { return p ? 16384 : 0; }
    __host__ __device__ static constexpr uint32_t kslot(int p) { return p ? 24576 : 0; }
    static constexpr uint32_t kWslot = 8192, kHslot = 8192;
};

struct WideBars {
    uint64_t full[2], empty[2];                 // q and k, by chunk parity
    uint64_t ap_full, abv_full;                 // A'; A diag(beta) and v (one buffer each)
    uint64_t big_done, h_done, u_done;          // MMA completions
    uint64_t o_done[2];                         // PV(c), by chunk parity (its readers alternate)
    // W(c) and its epilogue, one barrier per lane half (chunk parity): the aux
    // warps of a half see every phase of their own barrier in order, where
    // one shared barrier's parity would let a half run a chunk ahead
    uint64_t w_done[2], w_ready[2];
    uint64_t g_ready[4];                        // decay tables (4 chunk slots)
    uint64_t o_seeded, xo_ready, vn_ready, hs_ready, o_free;
    uint64_t drain;
    // output stage over a cluster: the rows' partial sums of a chunk slot
    // (c % 4) arrive as transactions from every CTA of the cluster
    uint64_t norm_bar[4];
    uint32_t abort, tmem;
};
static_assert(sizeof(WideBars) <= 256, "the barriers fit their region");

// Output stage (gated RMSNorm over V), by instance (kOsNorm with it, kOsNormX
// with it over a cluster, kOsNone without; the plain instance has none of its
// code, and only kOsNormX has the cluster's). The aux warp takes its
// row's sum of squares over the CTA's 128 columns from the fp32 accumulator
// O(c), parks the row rounded to bf16 in spare TMEM columns and frees O; one
// chunk later, in the chunk whose W and O lie in the other lane half (its idle
// turn), it applies norm, weight and gate and stores o. The chain never waits
// for the stage's element work. With V = 256 (kOsNormX) the head's two CTAs
// form a cluster and every CTA sends each row's partial sum to both (st.async
// into a slot of chunk c % 4), and both add them in rank order.
constexpr int kOsNone = 0, kOsNorm = 1, kOsNormX = 2;

__device__ __forceinline__ float sigmoid_tanh_w(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}

template <int K, int OS>
__global__ void __launch_bounds__(kWideThreads, 1)
gdn_wide_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                   const float *__restrict__ g, const float *__restrict__ h0,
                   float *__restrict__ h_final, __nv_bfloat16 *__restrict__ o, int T, int H, int V,
                   float scale, uint32_t *status, int l2norm, const float *__restrict__ rk,
                   uint64_t wlim, int stall, const __nv_bfloat16 *__restrict__ gate, const float *__restrict__ norm_w, float norm_eps) {
    using Lay = WideLayout<K>;
    constexpr int KB = K / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // Per chunk slot (c & 3): exp(g) rq; exp(g_last - g) rk; the row and column
    // factors scale rq exp(g_i - g_ref) and rk exp(g_ref - g_j) about g_ref =
    // g_last / 2 while |g_last| <= 160 (flag fz_s), else the exponents.
    float *tab = reinterpret_cast<float *>(sm + Lay::kG);
    float *eg_s = tab, *gate_s = tab + 256, *rf_s = tab + 512, *cf_s = tab + 768;
    int *fz_s = reinterpret_cast<int *>(tab + 1024);
    WideBars *bs = reinterpret_cast<WideBars *>(sm + Lay::kBar);
    volatile uint32_t *abort = &bs->abort;

    // one-dimensional grid over (head, 128-column V block), head = b * H + h
    const int nvt = V / kWideBV;
    const long long head = static_cast<long long>(blockIdx.x / nvt);
    const int vt = static_cast<int>(blockIdx.x % nvt), h = static_cast<int>(head % H),
              b = static_cast<int>(head / H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = (T + 63) / 64;

    // the four zero tiles of the operand row [0 | A' | 0 | P | 0 | A diag(beta) | 0]
    static_assert(Lay::kZy == Lay::kZx + 16384 && Lay::kZz == Lay::kZx + 32768 && Lay::kZw == Lay::kZx + 49152,
                  "the zero tiles are every other tile of the row");
    for (int i = tid; i < 4 * 512; i += kWideThreads)
        st_shared_v4(sm + Lay::kZx + (i >> 9) * 16384 + (i & 511) * 16, 0u, 0u, 0u, 0u);
    // the stage's first column: a row spans the CTAs of a cluster only in kOsNormX
    const int scol0 = OS == kOsNormX ? vt * kWideBV : 0;
    if (OS != kOsNone && tid < kWideBV) reinterpret_cast<float *>(sm + Lay::kNw)[tid] = norm_w[scol0 + tid];
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&bs->tmem, kWideTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bs->full[s], 1);
            mbar_init(&bs->empty[s], 1);
        }
        mbar_init(&bs->ap_full, 1);
        mbar_init(&bs->abv_full, 1);
        mbar_init(&bs->big_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bs->w_done[i], 1);
            mbar_init(&bs->w_ready[i], 64);               // the two aux warps on that half
        }
        mbar_init(&bs->h_done, 1);
        mbar_init(&bs->o_done[0], 1);
        mbar_init(&bs->o_done[1], 1);
        mbar_init(&bs->u_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&bs->g_ready[i], kAuxThreads);
        mbar_init(&bs->o_seeded, kChainWarps * 16);       // the eight warps on q's lanes
        mbar_init(&bs->xo_ready, kChainWarps * 16);
        mbar_init(&bs->vn_ready, kChainWarps * 16);       // the eight on v_new's
        mbar_init(&bs->hs_ready, kChainWarps * 32);
        mbar_init(&bs->o_free, 64);                       // the two aux warps on O's lanes
        mbar_init(&bs->drain, 1);
        // one local arrival (with the expected bytes) per chunk of the slot
        if (OS == kOsNormX)
            for (int i = 0; i < 4; ++i) mbar_init(&bs->norm_bar[i], 1);
        bs->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_a);
    }
    tc_fence_before_sync();
    __syncthreads();
    // output stage over a cluster: its barriers are initialised before any CTA
    // of the cluster sends to them
    const int nrank = OS == kOsNormX ? nvt : 1;
    if (nrank > 1) cluster_sync();
    // the setup above overlaps the WY kernel's last CTAs; everything below may
    // read its output. A 64-column kernel for the remaining heads may start
    // behind this grid from here on (it reads only the WY kernel's output).
    griddep_wait();
    griddep_launch_dependents();
    tc_fence_after_sync();
    const uint32_t tmem = bs->tmem;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idW = idesc_bf16(128, K, false, true);
            constexpr uint32_t idU = idesc_bf16(128, kWideBV, false, true);
            constexpr uint32_t idBIG = idesc_bf16(128, 192, false, false);
            constexpr uint32_t idHT = idesc_bf16(128, K, true, true);
            constexpr uint32_t idPV = idesc_bf16(128, kWideBV, false, true);
            // chunk c's k, read N-major (feature atoms one block apart)
            auto k_desc = [&](int c) {
                return TileDesc(s_base + Lay::kKH + Lay::kslot(c & 1), Lay::kKHBlk, 1024);
            };
            // W(c) = [A'; 0] k (w in lanes 0-63) for even c, [0; A'] k (lanes
            // 64-127) for odd c: the lanes where q's rows, and then O(c), go.
            // Accumulating onto zeros that the last reader of O left there.
            auto issue_w = [&](int c) {
                const TileDesc da(s_base + ((c & 1) ? Lay::kZx : Lay::kAp), 16, 1024);
                const TileDesc db = k_desc(c);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_k<true>(tmem + kCWO, da.at(ks * 32), db.at(ks * 2048), idW);
                mma_commit(&bs->w_done[c & 1]);
            };
            // X(c) = [0; A diag(beta)] v (u in lanes 64-127) for even c,
            // [A diag(beta); 0] v (lanes 0-63) for odd c
            auto issue_u = [&](int c) {
                const TileDesc da(s_base + ((c & 1) ? Lay::kAb : Lay::kZz), 16, 1024);
                const TileDesc db(s_base + Lay::kV, 8192, 1024);
                const uint32_t xc = (c & 1) ? 0 : 64;
                mma_bf16_k<false>(tmem + kCBig + xc, da.at(0), db.at(0), idU);
#pragma unroll
                for (int ks = 1; ks < 4; ++ks) mma_bf16_k<true>(tmem + kCBig + xc, da.at(ks * 32), db.at(ks * 2048), idU);
                mma_commit(&bs->u_done);
            };
            // O(c) += [P; 0] v_new (even c) or [0; P] v_new (odd c)
            auto issue_pv = [&](int c) {
                const TileDesc da(s_base + ((c & 1) ? Lay::kZy : Lay::kP), 16, 1024);
                const TileDesc db(s_base + Lay::kVN, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_k<true>(tmem + kCWO, da.at(ks * 32), db.at(ks * 2048), idPV);
                mma_commit(&bs->o_done[c & 1]);
            };
            // W(c) may go once its k and A' landed, O(c - 1) (the other lane
            // half, which W(c) rewrites unchanged) is seeded, and O(c - 2) (its
            // own lanes) is read and cleared
            auto w_inputs = [&](int c) {
                return mbar_test_wait(&bs->full[c & 1], (c >> 1) & 1) && mbar_test_wait(&bs->ap_full, c & 1) &&
                       mbar_test_wait(&bs->o_seeded, (c - 1) & 1) &&
                       (c < 2 || mbar_test_wait(&bs->o_free, c & 1));
            };
            // the chain group zeroes the W / O columns before its first hs_ready
            bool ok = spin_bar(&bs->full[0], 0, abort, wlim) && spin_bar(&bs->ap_full, 0, abort, wlim) &&
                      spin_bar(&bs->hs_ready, 0, abort, wlim);
            if (ok) {
                tc_fence_after_sync();
                issue_w(0);
                ok = spin_bar(&bs->abv_full, 0, abort, wlim);
                if (ok) {
                    tc_fence_after_sync();
                    issue_u(0);
                }
            }
            for (int c = 0; ok && c < NT; ++c) {
                const int s = c & 1;
                const uint32_t par = c & 1;
                if (!(ok = spin_bar(&bs->hs_ready, par, abort, wlim) &&
                           spin_bar(&bs->w_ready[s], (c >> 1) & 1, abort, wlim)))
                    break;
                tc_fence_after_sync();
                {
                    // [q0; -w] [k0; h^T] (even) or [-w; q1] [h^T; k1] (odd), K-steps of 16
                    const TileDesc da(s_base + Lay::kQW + s * 8192, 16, 1024);
                    const TileDesc db(s_base + Lay::kKH + s * 8192, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks)
                        mma_bf16_k<true>(tmem + kCBig, da.at((ks >> 2) * Lay::kQWBlk + (ks & 3) * 32),
                                         db.at((ks >> 2) * Lay::kKHBlk + (ks & 3) * 32), idBIG);
                }
                mma_commit(&bs->big_done);
                // the next chunk's W as soon as its inputs are in, if before v_new
                bool w_next = c + 1 < NT;
                {
                    const uint64_t t0 = globaltimer_ns();
                    for (uint32_t i = 1;; ++i) {
                        if (w_next && w_inputs(c + 1)) {
                            tc_fence_after_sync();
                            issue_w(c + 1);
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
                    const TileDesc da(s_base + Lay::kVG, 8192, 1024);
                    const TileDesc db = k_desc(c);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_k<true>(tmem + kCHT, da.at(ks * 2048), db.at(ks * 2048), idHT);
                }
                mma_commit(&bs->h_done);
                mma_commit(&bs->empty[s]);   // HT(c) is the last reader of chunk c's q and k
                if (w_next) {
                    if (!(ok = spin_bar(&bs->full[s ^ 1], ((c + 1) >> 1) & 1, abort, wlim) &&
                               spin_bar(&bs->ap_full, (c + 1) & 1, abort, wlim) &&
                               spin_bar(&bs->o_seeded, c & 1, abort, wlim) &&
                               (c + 1 < 2 || spin_bar(&bs->o_free, (c + 1) & 1, abort, wlim))))
                        break;
                    tc_fence_after_sync();
                    issue_w(c + 1);
                }
                // once P, q h and v_new are out of X(c): the next chunk's u, then o
                if (!(ok = spin_bar(&bs->xo_ready, par, abort, wlim))) break;
                if (c + 1 < NT) {
                    if (!(ok = spin_bar(&bs->abv_full, (c + 1) & 1, abort, wlim))) break;
                    tc_fence_after_sync();
                    issue_u(c + 1);
                }
                // PV(c) rewrites the other lane half too: O(c - 1) must be out and cleared
                if (c >= 1 && !(ok = spin_bar(&bs->o_free, (c - 1) & 1, abort, wlim))) break;
                tc_fence_after_sync();
                issue_pv(c);
            }
            // nothing of ours may still run when the accumulators are released
            mma_commit(&bs->drain);
            mbar_wait(&bs->drain, 0, kWaitNs);
        }
    } else if (warp == 1) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int issued = 0, a_issued = 0, v_issued = 0;   // chunks whose loads were issued
            for (int c = 0; c < NT; ++c) {
                const int s = c & 1, t0 = c * 64;
                if (c >= 2 && !wait_bar(&bs->empty[s], ((c >> 1) - 1) & 1, abort, wlim)) break;
                // test hook: chunk 0's loads are withheld, so every role's first
                // wait on them runs out and the launch reports a device timeout
                if (stall && c == 0) continue;
                mbar_arrive_expect_tx(&bs->full[s], KB * 16384);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(sm + Lay::kQW + kb * Lay::kQWBlk + Lay::qslot(s), &tm_q, &bs->full[s], kb * 64,
                                h, t0, b);
                    tma_load_4d(sm + Lay::kKH + kb * Lay::kKHBlk + Lay::kslot(s), &tm_k, &bs->full[s], kb * 64,
                                h, t0, b);
                }
                issued = c + 1;
                // A'(c) once W(c - 1) read A'(c - 1)
                if (c >= 1 && !wait_bar(&bs->w_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort, wlim)) break;
                mbar_arrive_expect_tx(&bs->ap_full, 8192);
                tma_load_4d(sm + Lay::kAp, &tm_a, &bs->ap_full, 64, h, t0, b);
                a_issued = c + 1;
                // A diag(beta)(c) and v(c) once U(c - 1) read theirs
                if (c >= 1 && !wait_bar(&bs->u_done, (c - 1) & 1, abort, wlim)) break;
                mbar_arrive_expect_tx(&bs->abv_full, 8192 + 16384);
                tma_load_4d(sm + Lay::kAb, &tm_a, &bs->abv_full, 0, h, t0, b);
                tma_load_4d(sm + Lay::kV, &tm_v, &bs->abv_full, vt * kWideBV, h, t0, b);
                tma_load_4d(sm + Lay::kV + 8192, &tm_v, &bs->abv_full, vt * kWideBV + 64, h, t0, b);
                v_issued = c + 1;
            }
            // no copy may still be landing in shared memory when the CTA exits
            // (after an abort the last loads may have no consumer)
            for (int c = max(stall ? 1 : 0, issued - 2); c < issued; ++c)
                mbar_wait(&bs->full[c & 1], (c >> 1) & 1, kWaitNs);
            if (a_issued > (stall ? 1 : 0)) mbar_wait(&bs->ap_full, (a_issued - 1) & 1, kWaitNs);
            if (v_issued > (stall ? 1 : 0)) mbar_wait(&bs->abv_full, (v_issued - 1) & 1, kWaitNs);
        }
    } else if (warp < 6) {
        // ================================================================ aux group
        // Decay tables of every chunk (threads 0-63, one token each), and on the
        // two warps whose lane quarters hold chunk c's W and O (lane half c % 2):
        // o(c - 2) out of TMEM, those lanes cleared for W(c), then the w
        // epilogue, W(c) rows -> -w, bf16, into the one -w tile (last read by
        // BIG(c - 1), done before W(c) was). The chain warps stay on the chunk
        // chain.
        const int ptid = tid - 64;
        const int q4 = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const int wrow = (q4 & 1) * 32 + lane;
        // kOsNorm: the row's 1 / rms, kept from write_o(cc) to finish_o(cc)
        float rstd_pend = 0.f;
        // o(cc) from O (these 32 lanes, all 128 columns), then the lanes cleared
        auto write_o = [&](int cc) -> bool {
            if (!warp_all(wait_bar(&bs->o_done[cc & 1], (cc >> 1) & 1, abort, wlim))) return false;
            tc_fence_after_sync();
            const int64_t row = (static_cast<int64_t>(b) * T + cc * 64 + wrow) * H + h;
            const int64_t oi = row * V + vt * kWideBV;
            const bool in = wrow < min(64, T - cc * 64);
            // with the output stage: the row's sum of squares over these columns,
            // before rounding (four partial sums; none without the stage)
            float ss[4] = {0.f, 0.f, 0.f, 0.f};
            if (OS != kOsNone && in) {
                // the gate row (256 B) is read in this warp's next idle turn
                const __nv_bfloat16 *zr = gate + row * V + scol0;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(zr));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(zr + 64));
            }
#pragma unroll 1
            for (int bb = 0; bb < kWideBV / 32; ++bb) {
                uint32_t r[32];
                tmem_ld32(tmem + kCWO + lane_off + bb * 32, r);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                if constexpr (OS != kOsNone) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss[e & 3] = fmaf(v[e], v[e], ss[e & 3]);
                }
                if constexpr (OS != kOsNone) {
                    // the same rounding as the plain store
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                    tmem_st16(tmem + kCStash + lane_off + bb * 16, pk);
                } else if (in) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) store_bf16x8_global(o + oi + bb * 32 + q * 8, v + q * 8);
                }
            }
            if (OS != kOsNone && nrank == 1) rstd_pend = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) / V + norm_eps);
            if (OS != kOsNone && nrank > 1) {
                // every row (in range or not) to every CTA of the cluster, this
                // CTA's entry (its rank, vt) of the slot; one thread of the
                // half posts the bytes its own barrier expects
                const int slot = cc & 3;
                if ((q4 & 1) == 0 && lane == 0) mbar_arrive_expect_tx(&bs->norm_bar[slot], nrank * 64 * 4);
                const uint32_t dst = s_base + Lay::kSums + ((slot * kWideMaxRanks + vt) * 64 + wrow) * 4;
                const uint32_t nb = smem_u32(&bs->norm_bar[slot]);
                const float part = (ss[0] + ss[1]) + (ss[2] + ss[3]);
#pragma unroll
                for (int r = 0; r < kWideMaxRanks; ++r)
                    if (r < nrank) st_async_cluster_f32(mapa_shared(dst, r), part, mapa_shared(nb, r));
            }
            const uint32_t z[16] = {};
#pragma unroll
            for (int bb = 0; bb < kWideBV / 16; ++bb) tmem_st16(tmem + kCWO + lane_off + bb * 16, z);
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(&bs->o_free);   // W(cc + 2) and PV(cc + 1) may rewrite these lanes
            return true;
        };
        // kOsNorm: o(cc) <- o * rstd * weight * sigmoid(gate) for this lane's row,
        // 32 columns a step from the TMEM stash (the tcgen05.ld is warp-wide, so
        // every lane takes part), with the gate's next 64 bytes loaded while the
        // current ones are used.
        auto finish_o = [&](int cc) -> bool {
            if (nrank > 1) {
                // every CTA's partial sums of chunk cc's rows, added in rank order
                const int slot = cc & 3;
                if (!warp_all(wait_bar_cluster(&bs->norm_bar[slot], (cc >> 2) & 1, abort, wlim))) return false;
                const float *sums = reinterpret_cast<const float *>(sm + Lay::kSums) + slot * kWideMaxRanks * 64;
                float tot = 0.f;
#pragma unroll
                for (int r = 0; r < kWideMaxRanks; ++r)
                    if (r < nrank) tot += sums[r * 64 + wrow];
                rstd_pend = rsqrtf(tot / V + norm_eps);
            }
            const bool in = wrow < min(64, T - cc * 64);
            const int64_t row = in ? (static_cast<int64_t>(b) * T + cc * 64 + wrow) * H + h : 0;
            const uint4 *zp = reinterpret_cast<const uint4 *>(gate + row * V + scol0);
            uint4 *op = reinterpret_cast<uint4 *>(o + row * V + scol0);
            const float4 *nw4 = reinterpret_cast<const float4 *>(sm + Lay::kNw);
            const float rs = rstd_pend;
            uint4 zn[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) zn[q] = in ? __ldg(zp + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
            for (int p = 0; p < kWideBV / 32; ++p) {
                uint4 z[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) z[q] = zn[q];
                if (p + 1 < kWideBV / 32) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) zn[q] = in ? __ldg(zp + 4 * (p + 1) + q) : make_uint4(0u, 0u, 0u, 0u);
                }
                uint32_t pk[16];
                tmem_ld16(tmem + kCStash + lane_off + p * 16, pk);
                tmem_wait_ld();
                if (!in) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 w0 = nw4[8 * p + 2 * q], w1 = nw4[8 * p + 2 * q + 1];   // this CTA's columns
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                    const uint32_t z4[4] = {z[q].x, z[q].y, z[q].z, z[q].w};
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 a = unpack_bf16(pk[4 * q + e]), zz = unpack_bf16(z4[e]);
                        y[2 * e] = a.x * rs * wv[2 * e] * sigmoid_tanh_w(zz.x);
                        y[2 * e + 1] = a.y * rs * wv[2 * e + 1] * sigmoid_tanh_w(zz.y);
                    }
                    op[4 * p + q] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                                               pack_bf16(y[6], y[7]));
                }
            }
            return true;
        };
        auto load_g = [&](int c) {
            const int t = c * 64 + ptid;
            return (ptid < 64 && c < NT && t < T) ? g[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
        };
        auto load_gl = [&](int c) {
            return (ptid < 64 && c < NT) ? g[(static_cast<int64_t>(b) * T + min(T, c * 64 + 64) - 1) * H + h]
                                         : 0.f;
        };
        auto load_rk = [&](int c) {
            const int t = c * 64 + ptid;
            return (l2norm && ptid < 64 && c < NT && t < T) ? rk[(static_cast<int64_t>(b) * T + t) * H + h]
                                                           : 1.f;
        };
        float g_next = load_g(0), gl_next = load_gl(0), rk_next = load_rk(0);
        bool ok = true;
        int pend = -1;   // kOsNorm: the chunk whose rows wait for finish_o
        for (int c = 0; c < NT; ++c) {
            const int s = c & 1, gs = c & 3;
            const int n = min(64, T - c * 64);
            const bool mine = (q4 >> 1) == (c & 1);   // W(c) and O(c) lie in these lanes
            if (mine && c >= 2) {
                if (!(ok = write_o(c - 2))) break;
                if (OS != kOsNone) pend = c - 2;
            }
            const float g_cur = g_next, gl = gl_next, rk_cur = rk_next;
            g_next = load_g(c + 1);
            gl_next = load_gl(c + 1);
            rk_next = load_rk(c + 1);
            // Slot c % 4's previous reader, chunk c - 4, finished before U(c - 3)
            // was issued, and chunk c's stage landing needs HT(c - 2).
            if (!(ok = wait_bar(&bs->full[s], (c >> 1) & 1, abort, wlim))) break;
            if (ptid < 64) {
                float rq = 1.f;
                if (l2norm) {
                    // |q_i|^2 from the chunk's q tile (the swizzle only permutes
                    // 16-byte chunks in a row; chunk j ^ (row % 8) keeps 8 rows on
                    // distinct banks)
                    const unsigned char *qrow = sm + Lay::kQW + Lay::qslot(s) + ptid * 128;
                    float ss = 0.f;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(qrow + kb * Lay::kQWBlk +
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
                const bool fzc = fabsf(gl) <= 160.f;
                const bool okt = ptid < n;
                eg_s[gs * 64 + ptid] = okt ? __expf(g_cur) * rq : 0.f;
                gate_s[gs * 64 + ptid] = okt ? __expf(gl - g_cur) * rk_cur : 0.f;
                if (fzc) {
                    rf_s[gs * 64 + ptid] = okt ? scale * __expf(g_cur - gref) * rq : 0.f;
                    cf_s[gs * 64 + ptid] = okt ? __expf(gref - g_cur) * rk_cur : 0.f;
                } else {
                    rf_s[gs * 64 + ptid] = l2norm ? g_cur + __logf(rq) : g_cur;
                    cf_s[gs * 64 + ptid] = l2norm ? g_cur - __logf(rk_cur) : g_cur;
                }
                if (ptid == 0) fz_s[gs] = fzc;
            }
            mbar_arrive(&bs->g_ready[gs]);
            if (!mine) {
                // W(c) lies in the other lane half: this warp's idle turn
                if (OS != kOsNone && pend >= 0) {
                    if (!(ok = finish_o(pend))) break;
                    pend = -1;
                }
                continue;
            }
            if (!(ok = warp_all(wait_bar(&bs->w_done[c & 1], (c >> 1) & 1, abort, wlim)))) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int bb = 0; bb < K / 32; ++bb) {
                const int f0 = bb * 32;
                uint32_t r[32];
                tmem_ld32(tmem + kCWO + lane_off + f0, r);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = -__uint_as_float(r[e]);
                unsigned char *base = sm + Lay::kQW + (f0 >> 6) * Lay::kQWBlk + Lay::kWslot;
#pragma unroll
                for (int q = 0; q < 4; ++q) st_bf16x8(base + sw128(wrow, (f0 & 63) * 2 + q * 16), v + q * 8);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bs->w_ready[c & 1]);
        }
        // the last two chunks' o
        if (OS != kOsNone && ok && pend >= 0) ok = finish_o(pend);
        for (int cc = max(0, NT - 2); ok && cc < NT; ++cc)
            if ((q4 >> 1) == (cc & 1)) {
                ok = write_o(cc);
                if (OS != kOsNone && ok) ok = finish_o(cc);
            }
    } else {
        // ================================================================ chain group
        // Chunk c's q rows sit in lane half c % 2: the eight warps there turn QK
        // into P, seed O with scale exp(g) (q h) and write o; the eight on the
        // other half write v_new and v_g and clear the next chunk's QK columns.
        // All sixteen copy the state: HT holds h^T with V row = lane, and
        // warp j of a quarter owns features [j K / 4, (j + 1) K / 4).
        constexpr int NF = K / 4;
        const int q4 = warp & 3, j = (warp - 6) >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const int row = (q4 & 1) * 32 + lane;    // token row in the chunk
        const int vrow = q4 * 32 + lane;         // V row of the state
        const int col0 = j * 32;                 // this warp's 32 of the 128 V columns
        const int f0 = j * NF;
        const int64_t state_off = (static_cast<int64_t>(b) * H + h) * K * V + vt * kWideBV;
        auto g_last_of = [&](int c) {
            return g[(static_cast<int64_t>(b) * T + min(T, c * 64 + 64) - 1) * H + h];
        };
        // the state's bf16 copy: row vrow of h^T, features f .. f + 15
        auto store_ht = [&](int f, const float *v) {
            unsigned char *dst = sm + Lay::kKH + (f >> 6) * Lay::kKHBlk + Lay::kHslot;
            st_bf16x8(dst + sw128(vrow, (f & 63) * 2), v);
            st_bf16x8(dst + sw128(vrow, (f & 63) * 2 + 16), v + 8);
        };
        {
            // initial state (fp32 in TMEM pre-decayed by chunk 0's exp(g_last));
            // chunk 0's QK columns and the W / O columns start at zero
            const float d0 = __expf(g_last_of(0));
#pragma unroll 1
            for (int blk = 0; blk < NF / 16; ++blk) {
                const int f = f0 + blk * 16;
                float v[16];
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    v[e] = h0 ? h0[state_off + static_cast<int64_t>(f + e) * V + vrow] : 0.f;
                    r[e] = __float_as_uint(v[e] * d0);
                }
                tmem_st16(tmem + kCHT + lane_off + f, r);
                store_ht(f, v);
            }
            const uint32_t z[16] = {};
            tmem_st16(tmem + kCBig + lane_off + j * 16, z);
            tmem_st16(tmem + kCWO + lane_off + col0, z);
            tmem_st16(tmem + kCWO + lane_off + col0 + 16, z);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(&bs->hs_ready);
        bool ok = true;
        float g_last_next = NT > 1 ? g_last_of(1) : 0.f;
        for (int c = 0; c < NT; ++c) {
            const int t0 = c * 64, n = min(64, T - t0), gs = c & 3;
            const bool qside = (q4 >> 1) == (c & 1);
            const uint32_t xcol = kCBig + ((c & 1) ? 0 : 64), qkcol = kCBig + ((c & 1) ? 128 : 0);
            const float d_next = c + 1 < NT ? __expf(g_last_next) : 1.f;
            if (c + 2 < NT) g_last_next = g_last_of(c + 2);   // one chunk ahead
            if (!(ok = warp_all(wait_bar(&bs->g_ready[gs], (c >> 2) & 1, abort, wlim) &&
                                nap_bar(&bs->big_done, c & 1, abort, wlim, kNapNs))))
                break;
            tc_fence_after_sync();
            if (qside) {
                // O(c) = scale exp(g) (q h), into the W / O columns of these lanes
                const float so = scale * eg_s[gs * 64 + row];
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[16];
                    tmem_ld16(tmem + xcol + lane_off + col0 + half * 16, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(so * __uint_as_float(r[e]));
                    tmem_st16(tmem + kCWO + lane_off + col0 + half * 16, r);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&bs->o_seeded);   // W(c + 1) may rewrite these lanes now
                // P = QK masked and scaled, 16 of its 64 columns per warp
                {
                    const bool fz = fz_s[gs];
                    const float ri = rf_s[gs * 64 + row];
                    const int j0 = j * 16;
                    float v[16];
                    if (j0 <= (q4 & 1) * 32 + 31) {
                        float fj[16];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 f4 = *reinterpret_cast<const float4 *>(cf_s + gs * 64 + j0 + 4 * m);
                            fj[4 * m] = f4.x;
                            fj[4 * m + 1] = f4.y;
                            fj[4 * m + 2] = f4.z;
                            fj[4 * m + 3] = f4.w;
                        }
                        tmem_ld16f(tmem + qkcol + lane_off + j0, v);
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
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->xo_ready);
            } else {
                // v_new and v_g (v_new tile last read by PV(c - 1))
                if (c >= 1 && !(ok = warp_all(wait_bar(&bs->o_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort, wlim))))
                    break;
                const float gate = gate_s[gs * 64 + row];
                const int atom = col0 >> 6, cb = (col0 & 63) * 2;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float v[16], vg[16];
                    tmem_ld16f(tmem + xcol + lane_off + col0 + half * 16, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) vg[e] = v[e] * gate;
                    unsigned char *vn = sm + Lay::kVN + atom * 8192, *vgp = sm + Lay::kVG + atom * 8192;
                    st_bf16x8(vn + sw128(row, cb + half * 32), v);
                    st_bf16x8(vn + sw128(row, cb + half * 32 + 16), v + 8);
                    st_bf16x8(vgp + sw128(row, cb + half * 32), vg);
                    st_bf16x8(vgp + sw128(row, cb + half * 32 + 16), vg + 8);
                }
                // the next chunk's QK columns in these lanes (its q rows) start at
                // zero: the half of X(c) that becomes them, once read above
                if ((j >> 1) != (c & 1)) {
                    const uint32_t z[16] = {};
                    tmem_st16(tmem + xcol + lane_off + col0, z);
                    tmem_st16(tmem + xcol + lane_off + col0 + 16, z);
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bs->vn_ready);
            }
            if (!(ok = warp_all(nap_bar(&bs->h_done, c & 1, abort, wlim, kNapNs)))) break;
            tc_fence_after_sync();
            if (c + 1 < NT) {
                // the state, pre-decayed by the next chunk's exp(g_last), and its
                // bf16 copy for BIG(c + 1)
#pragma unroll 1
                for (int blk = 0; blk < NF / 16; ++blk) {
                    const int f = f0 + blk * 16;
                    uint32_t r[16];
                    tmem_ld16(tmem + kCHT + lane_off + f, r);
                    tmem_wait_ld();
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        v[e] = __uint_as_float(r[e]);
                        r[e] = __float_as_uint(v[e] * d_next);
                    }
                    tmem_st16(tmem + kCHT + lane_off + f, r);
                    store_ht(f, v);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            mbar_arrive(&bs->hs_ready);
        }
        // final state straight from tensor memory
        if (warp_all(ok) && h_final) {
            tc_fence_after_sync();
#pragma unroll 1
            for (int blk = 0; blk < NF / 16; ++blk) {
                float v[16];
                tmem_ld16f(tmem + kCHT + lane_off + f0 + blk * 16, v);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    h_final[state_off + static_cast<int64_t>(f0 + blk * 16 + e) * V + vrow] = v[e];
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // no CTA of a cluster leaves while another may still write its shared memory
    if (nrank > 1) cluster_sync();
    if (tid == 0 && *abort) atomicOr(status, 1u);
    if (warp == 0) tmem_dealloc(tmem, kWideTmemCols);
}

int sm_count_of_device() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();   // no device visible: GB300's SM count
        return 152;
    }
    return sms;
}

template <int K>
cudaError_t launch_wide(const Args &a, const void *abeta, cudaStream_t s, long long heads) {
    // the output stage: in the kernel when a row is one CTA's, else row sums
    const int nvt = a.V / kWideBV;
    if (a.gate && nvt > kWideMaxRanks) return cudaErrorInvalidValue;
    const int os = !a.gate ? kOsNone : nvt > 1 ? kOsNormX : kOsNorm;
    CUtensorMap mq, mk, mv, ma;
    if (!make_tmap_bthx(&mq, a.q, K, a.H, a.T, a.B) || !make_tmap_bthx(&mk, a.k, K, a.H, a.T, a.B) ||
        !make_tmap_bthx(&mv, a.v, a.V, a.H, a.T, a.B) || !make_tmap_bthx(&ma, abeta, 128, a.H, a.T, a.B))
        return cudaErrorInvalidValue;
    const int smem = static_cast<int>(WideLayout<K>::kBytes + 1024);
    const auto kernel = os == kOsNormX  ? gdn_wide_tc_kernel<K, kOsNormX>
                        : os == kOsNorm ? gdn_wide_tc_kernel<K, kOsNorm>
                                        : gdn_wide_tc_kernel<K, kOsNone>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(a.V / kWideBV) * heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kWideThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    // as for gdn_fused_tc_kernel: an early start only pays with more than one wave
    if (ctas > sm_count_of_device()) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (os == kOsNormX) {
        // the head's V / 128 CTAs share the rows' sums of squares
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = nvt;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr++].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    const float *g_arg = a.g_chunk(), *h0_arg = a.h0, *rk_arg = a.rk;
    float *hf_arg = a.h_final;
    __nv_bfloat16 *o_arg = static_cast<__nv_bfloat16 *>(a.o);
    int T_arg = a.T, H_arg = a.H, V_arg = a.V, norm_arg = (a.flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
    float scale_arg = a.scale;
    uint32_t *status_arg = a.status;
    uint64_t wlim_arg = kWaitNs;
    int stall_arg = 0;
    if (const uint64_t armed = take_armed_stall()) {
        wlim_arg = armed;
        stall_arg = 1;
    }
    const __nv_bfloat16 *gate_arg = static_cast<const __nv_bfloat16 *>(a.gate);
    const float *nw_arg = a.norm_w;
    float eps_arg = a.norm_eps;
    void *args[] = {&mq, &mk, &mv, &ma, &g_arg, &h0_arg, &hf_arg, &o_arg, &T_arg, &H_arg, &V_arg,
                    &scale_arg, &status_arg, &norm_arg, &rk_arg, &wlim_arg, &stall_arg, &gate_arg, &nw_arg, &eps_arg};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kernel), args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_wide(int B, int H, int V) {
    // with 64-wide tiles the grid would need more than one wave of SMs; with
    // fewer heads the narrow form keeps more SMs busy
    return V % kWideBV == 0 && static_cast<long long>(B) * H * (V / 64) > sm_count_of_device();
}

int tc_sm_count() { return sm_count_of_device(); }

cudaError_t wide_tc_forward(const Args &a, const void *abeta, cudaStream_t s, long long heads) {
    return a.K == 128 ? launch_wide<128>(a, abeta, s, heads) : launch_wide<64>(a, abeta, s, heads);
}

}  // namespace gdn
