"""gdn_chunk_fwd_noalloc, the entry point for callers that cannot allocate device
memory (for instance a plugin whose host framework owns every allocation and
hands it only input and output buffers).

It is called straight through the C ABI and must give the same outputs as
gdn_chunk_fwd with a caller workspace (bit for bit: the same CUDA-core kernels
run) and match the fp64 oracle within the parity tolerance, on two calls in a
row: the second call reuses the fixed scratch array left dirty by the first,
with a different shape and dtype. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_35_gb300 import native
from gated_delta_rule_35_gb300.inputs import make_inputs, to_f64
from oracle import recurrence
from tests.pins import rel

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _entry():
    f = native.lib().gdn_chunk_fwd_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(native.Problem), vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
    return f


def _call_noalloc(d, B, T, H, K, V, dtype):
    o = torch.full((B, T, H, V), float("nan"), dtype=dtype, device="cuda")
    hf = torch.full((B, H, K, V), float("nan"), dtype=torch.float32, device="cuda")
    p = native.problem(B, T, H, K, V, dtype, "auto")
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = _entry()(ctypes.byref(p), ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]),
                  ptr(d["beta"]), 1.0, ptr(d["h0"]), ptr(o), ptr(hf),
                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == native.GDN_OK, native.status_string(st)
    return o, hf


CASES = [  # (B, T, H, K, V, dtype, seed): two different problems, run back to back
    (2, 200, 3, 128, 128, "bf16", 31),
    (1, 130, 2, 64, 64, "f32", 32),
]


def test_noalloc_matches_workspace_entry_twice():
    """Both entries run the same deterministic CUDA-core kernels, so the
    outputs must be bit-identical; both are also checked against the fp64
    oracle at the parity tolerance."""
    for B, T, H, K, V, dt, seed in CASES:
        x = make_inputs(B, T, H, K, V, dtype=dt, seed=seed, h0_std=0.1)
        d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        tdt = d["q"].dtype
        o_ref, hf_ref = native.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"],
                                         algo="simt")
        o, hf = _call_noalloc(d, B, T, H, K, V, tdt)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(hf, hf_ref)
        o_or, hf_or = recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                         to_f64(x["g"]), to_f64(x["beta"]), 1.0, to_f64(x["h0"]))
        o_np = o.float().cpu().numpy()
        assert np.isfinite(o_np).all() and np.isfinite(hf.cpu().numpy()).all()
        assert rel(o_np, o_or) < TOL[dt]
        assert rel(hf.cpu().numpy(), hf_or) < TOL[dt]


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    # B*T*H = 2M token-heads needs far more than 64 MiB of SIMT workspace;
    # the call must fail before touching any pointer.
    p = native.problem(8, 8192, 32, 128, 128, torch.bfloat16, "auto")
    fake = ctypes.c_void_p(0x10000)
    st = _entry()(ctypes.byref(p), fake, fake, fake, fake, fake, 1.0, None, fake, None,
                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == native.GDN_ERR_WORKSPACE
    p = native.problem(1, 64, 1, 64, 64, torch.bfloat16, "tc")
    st = _entry()(ctypes.byref(p), fake, fake, fake, fake, fake, 1.0, None, fake, None, None)
    assert st == native.GDN_ERR_UNSUPPORTED
