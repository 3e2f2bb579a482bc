// gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
// device memory (see include/gdn.h). Its scratch is a fixed array in the
// library's own device image instead of a caller-provided workspace.
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

// Largest workspace the no-allocation entry point can serve: 64 MiB, held on
// every device that loads the library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device. The first call on
// a device asks the runtime for it (once, under a lock) and caches it.
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gdn

extern "C" GDN_API gdn_status gdn_chunk_fwd_noalloc(const gdn_problem *p, const void *q,
                                                    const void *k, const void *v, const float *g,
                                                    const float *beta, float scale,
                                                    const float *h0, void *o, float *h_final,
                                                    void *stream) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->algo != GDN_ALGO_AUTO && p->algo != GDN_ALGO_SIMT) return GDN_ERR_UNSUPPORTED;
    gdn_problem simt = *p;
    simt.algo = GDN_ALGO_SIMT;
    const size_t need = gdn_chunk_fwd_workspace_bytes(&simt);
    if (need > gdn::kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;   // beyond the fixed maximum
    void *scratch = nullptr;
    if (gdn::scratch_address(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
    // The SIMT pipeline writes every scratch region before reading it, so the
    // previous call's contents never need clearing.
    return gdn_chunk_fwd(&simt, q, k, v, g, beta, scale, h0, o, h_final, scratch,
                         gdn::kNoAllocScratchBytes, stream);
}
