// Internal declarations shared by the host launcher and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;

inline int64_t num_chunks(int T) { return (static_cast<int64_t>(T) + kChunk - 1) / kChunk; }

// Pointers of one call, already validated by the launcher.
struct Args {
    int B, T, H, K, V;
    int NT;          // ceil(T / 64)
    int T_pad;       // NT * 64
    gdn_dtype dtype;
    const void *q, *k, *v;
    const float *g, *beta;
    float scale;
    const float *h0;
    void *o;
    float *h_final;
    uint32_t *status;   // device status word (first bytes of the workspace)
    // Input front-end (GDN_FLAG_*). With GDN_FLAG_RAW_G, g holds raw per-token
    // log decays and the first kernel writes their chunk-local cumulative sum
    // to g_cum, which the later kernels read; with GDN_FLAG_QK_L2NORM the first
    // kernel writes each k row's factor 1 / sqrt(|k|^2 + eps) to rk.
    int flags;
    float *g_cum;   // [B, T, H] fp32 workspace ([B, T, H, K] with per-channel decay)
    float *rk;      // [B, T, H] fp32 workspace
    // g as the kernels after the first one read it: g_cum or g
    const float *g_chunk() const { return (flags & GDN_FLAG_RAW_G) ? g_cum : g; }
    // Output stage (gated RMSNorm over V); gate == nullptr: plain o.
    const void *gate = nullptr;
    const float *norm_w = nullptr;
    float norm_eps = 0.f;
};

constexpr float kL2NormEps = 1e-6f;
constexpr int kKnownFlags = GDN_FLAG_RAW_G | GDN_FLAG_QK_L2NORM | GDN_FLAG_PER_CHANNEL_DECAY;

// Workspace of the SIMT pipeline: fp32 intermediates, every region 256-byte aligned.
struct SimtWorkspace {
    float *A, *w, *u, *v_new, *h;
};

// Optional timing markers: ev[0] before the first kernel, ev[i + 1] after kernel i.
struct Marks {
    cudaEvent_t const *ev = nullptr;
    int n = 0;
    cudaError_t mark(int i, cudaStream_t s) const {
        return (ev && i < n) ? cudaEventRecord(ev[i], s) : cudaSuccess;
    }
};

size_t simt_workspace_bytes(int B, int T, int H, int K, int V);
SimtWorkspace simt_carve(void *base, int B, int T, int H, int K, int V);
cudaError_t simt_forward(const Args &a, const SimtWorkspace &ws, cudaStream_t s, const Marks &m);
constexpr int kSimtLaunches = 3;
extern const char *const kSimtKernelNames[kSimtLaunches];

// Tensor-core path: the WY kernel writing A to the workspace followed by the
// forward kernel reading it, or (single) one kernel that builds A itself.
bool tc_supported(int K, int V, gdn_dtype dtype);
size_t tc_workspace_bytes(int B, int T, int H, int K, int V);
// Tensor-core forms: two kernels (the forward kernel 64 or 128 V columns per CTA,
// by grid size), one kernel, or two kernels with the 128-column forward kernel.
enum class TcForm { kTwo, kSingle, kWide };
cudaError_t tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m, TcForm form);
int tc_launches(TcForm form, int B, int H, int V, const char **names, int max_names);
// The 128-column forward kernel (gdn_tc_wide.cu), reading A from abeta, for the
// first `heads` of the B * H (b * H + h order); whether the two-kernel form picks
// it for this shape; the device's SM count (152 when no device is visible).
// With the output stage (a.gate) it applies the stage itself (V = 256: the
// head's two CTAs as a cluster).
cudaError_t wide_tc_forward(const Args &a, const void *abeta, cudaStream_t s, long long heads);
bool tc_wide(int B, int H, int V);
int tc_sm_count();
// WY kernel: A diag(beta) per chunk, bf16 [B, T, H, 64], into `abeta`.
cudaError_t wy_tc_forward(const Args &a, void *abeta, cudaStream_t s);
// Converts the workspace's A diag(beta) to fp32 [B, T_pad, H, 64].
cudaError_t tc_export_abeta(const Args &a, const void *ws, float *dst, cudaStream_t s);

// Per-channel decay on the tensor cores (gdn_kda_tc.cu): a prep kernel per
// chunk, then the forward kernel over the chunks; workspace [A diag(beta) | P A
// diag(beta)] bf16 [B, T, H, 128] first, as the plain path's.
size_t kda_tc_workspace_bytes(int B, int T, int H, int K, int V);
cudaError_t kda_tc_forward(const Args &a, void *ws, cudaStream_t s, const Marks &m);
constexpr int kKdaTcLaunches = 2;
extern const char *const kKdaTcKernelNames[kKdaTcLaunches];

// h_final = h0 (or 0) for T == 0.
cudaError_t copy_state(const Args &a, cudaStream_t s);
constexpr const char *kCopyStateName = "copy_state_kernel";

constexpr size_t kStatusBytes = 256;

// Test hook (gdn_debug_arm_stall): the wait limit in nanoseconds for the next
// tensor-core launch, which then withholds its first chunk's loads; 0 when
// nothing is armed. Taking it disarms it.
uint64_t take_armed_stall();

inline size_t align_up(size_t x, size_t a = 256) { return (x + a - 1) / a * a; }

}  // namespace gdn
