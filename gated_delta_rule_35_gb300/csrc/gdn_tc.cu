// Tensor-core path (tcgen05/TMEM, TMA) of the chunked gated delta rule forward.
#include "gdn_internal.h"

namespace gdn {

bool tc_supported(int, int, gdn_dtype) { return false; }
size_t tc_workspace_bytes(int, int, int, int, int) { return 0; }
cudaError_t tc_forward(const Args &, void *, cudaStream_t, const Marks &) { return cudaErrorNotSupported; }
int tc_launches(const char **, int) { return 0; }

}  // namespace gdn
