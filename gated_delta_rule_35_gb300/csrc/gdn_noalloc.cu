// gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
// device memory (see include/gdn.h). Its scratch is a fixed array in the
// library's own device image instead of a caller-provided workspace.
#include "gdn_internal.h"

namespace gdn {
namespace {

// Largest workspace the no-allocation entry point can serve: 64 MiB, held on
// every device that loads the library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up on
// every call: the lookup is a host-side table read once the library's device
// code is loaded on the device (the first call on a device loads it), and a
// fresh lookup stays valid across a cudaDeviceReset or a re-created primary
// context, where a cached address would dangle.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    *out = p;
    return cudaSuccess;
}

// The stream's work must run on the current device, whose scratch array is
// the one handed to the kernels (NULL, the legacy default stream, always
// belongs to the current device).
bool stream_on_current_device(cudaStream_t s) {
    if (!s) return true;
    int cur = -1, dev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    if (cudaStreamGetDevice(s, &dev) != cudaSuccess) return false;
    return cur == dev;
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
    if (!gdn::stream_on_current_device(static_cast<cudaStream_t>(stream))) return GDN_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (gdn::scratch_address(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
    // The SIMT pipeline writes every scratch region before reading it, so the
    // previous call's contents never need clearing.
    return gdn_chunk_fwd(&simt, q, k, v, g, beta, scale, h0, o, h_final, scratch,
                         gdn::kNoAllocScratchBytes, stream);
}
