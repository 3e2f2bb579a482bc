"""fp64 CPU oracle of the chunked gated delta rule forward.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA path and never imports it.

  recurrence  token-by-token fp64 recurrence in plain C (``gdn_ref.c``)
  chunked     fp64 NumPy chunked form exporting every intermediate stage
  frontend    fp64 input steps: chunk-local cumsum of raw log decays, q/k L2 norm
  epilogue    fp64 gated RMSNorm of the output rows
"""
