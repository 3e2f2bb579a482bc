"""Decode step (gdn_decode_step) on the GPU against the fp64 token recurrence.

The oracle's recurrence with chunk = 1 takes the per-token log-decay gamma
directly (g restarted at every token). Tolerances, relative Frobenius error:
the inputs widen exactly and the state stays fp32 on both sides, so only fp32
rounding of the K-term sums separates them: 1e-5 for the state and for fp32 o;
a bf16 o is also rounded once to bf16 (at most 2^-9 relative per element),
so 2.5e-3 there."""
import numpy as np
import pytest
import torch

from oracle import recurrence
from tests.pins import rel
from tests.whole_tensor import whole_errors
from gated_delta_rule_35_gb300 import chunk_fwd, decode_step, native
from gated_delta_rule_35_gb300.inputs import (DECODE_WORKLOADS, chunk_local_cumsum, make_inputs,
                                              make_workload, to_f64)

pytestmark = pytest.mark.gpu

TOL_O = {"f32": 1e-5, "bf16": 2.5e-3}
TOL_S = 1e-5


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def oracle(x, state, scale=1.0):
    return recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]),
                              to_f64(x["beta"]), scale, to_f64(state), chunk=1)


def decode_inputs(B, T, H, K, V, dtype, seed, **kw):
    """Inputs with g = gamma (the per-token log-decay) and a non-zero state."""
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=seed, h0_std=0.1, chunk=1, **kw)
    return x, x.pop("h0")


# (B, T, H, K, V): covers the 64-, 32- and 16-column slices, every K, ragged V.
SHAPES = [(1, 1, 1, 128, 128), (8, 2, 16, 128, 128), (20, 1, 16, 64, 128), (2, 3, 3, 256, 48),
          (1, 2, 2, 192, 64), (3, 5, 2, 64, 96)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("inplace", [True, False])
def test_decode_against_oracle(shape, dtype, inplace):
    B, T, H, K, V = shape
    x, s0 = decode_inputs(B, T, H, K, V, dtype, seed=B * 1000 + T * 100 + K + V)
    d = gpu(x)
    state = s0.cuda()
    out = None if inplace else torch.full_like(state, float("nan"))
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, 0.7, state_out=out)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle(x, s0, 0.7)
    o_np, s_np = o.float().cpu().numpy(), s1.cpu().numpy()
    assert np.isfinite(o_np).all() and np.isfinite(s_np).all()
    assert rel(o_np, o_ref) < TOL_O[dtype], rel(o_np, o_ref)
    assert rel(s_np, s_ref) < TOL_S, rel(s_np, s_ref)
    if inplace:
        assert s1.data_ptr() == state.data_ptr()
    else:
        assert torch.equal(state.cpu(), s0)   # state_in untouched


def test_multi_token_call_equals_single_token_calls():
    """T tokens in one call run the same fp32 arithmetic as T calls of one token."""
    B, T, H, K, V = 4, 6, 8, 128, 128
    x, s0 = decode_inputs(B, T, H, K, V, "bf16", seed=3)
    d = gpu(x)
    s_all = s0.cuda()
    o_all, _ = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], s_all)
    s_one = s0.cuda()
    outs = []
    for t in range(T):
        sl = {n: d[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        o_t, _ = decode_step(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], s_one)
        outs.append(o_t)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), o_all)
    assert torch.equal(s_one, s_all)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode_equals_one_prefill(dtype):
    """chunk_fwd over the first 100 tokens, then 30 decode calls of one token
    from its h_final, give the outputs and final state of one chunk_fwd over
    all 130 tokens (the decode step consumes the chunked path's state layout)."""
    B, T, H, K, V = 2, 130, 3, 128, 128
    T1 = 100
    x, s0 = decode_inputs(B, T, H, K, V, dtype, seed=17)
    gam = x["g"]
    g_cum = chunk_local_cumsum(gam)
    d = gpu(x)
    gc = g_cum.cuda()
    o_full, h_full = chunk_fwd(d["q"], d["k"], d["v"], gc, d["beta"], 1.0, s0.cuda(), algo="simt")
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o_pre, h_pre = chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1),
                             sl(gc, 0, T1), sl(d["beta"], 0, T1), 1.0, s0.cuda(), algo="simt")
    outs = [o_pre]
    for t in range(T1, T):
        o_t, _ = decode_step(*(sl(d[n], t, t + 1) for n in ("q", "k", "v", "g", "beta")), h_pre)
        outs.append(o_t)
    torch.cuda.synchronize()
    o_cat = torch.cat(outs, 1).float().cpu().numpy()
    tol = 1e-4 if dtype == "f32" else 2.5e-3
    assert rel(o_cat, o_full.float().cpu().numpy()) < tol
    assert rel(h_pre.cpu().numpy(), h_full.cpu().numpy()) < 1e-4
    o_ref, h_ref = oracle(x, s0)   # the same 130 tokens, token by token in fp64
    assert rel(o_cat, o_ref) < tol and rel(h_pre.cpu().numpy(), h_ref) < 1e-4


def test_strong_decay_and_zero_state():
    """gamma down to about -60 (alpha near 1e-27) and a zero state."""
    x, _ = decode_inputs(4, 3, 4, 128, 128, "bf16", seed=8, g_div=0.03)
    assert float(x["g"].min()) < -40
    s0 = torch.zeros(4, 4, 128, 128)
    d = gpu(x)
    state = s0.cuda()
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle(x, s0)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL_O["bf16"]
    assert rel(s1.cpu().numpy(), s_ref) < TOL_S


def test_empty_call():
    """T = 0: state_out receives state_in; in place nothing changes."""
    s0 = torch.randn(2, 3, 128, 64, device="cuda")
    e = torch.empty(2, 0, 3, 128, dtype=torch.bfloat16, device="cuda")
    ev = torch.empty(2, 0, 3, 64, dtype=torch.bfloat16, device="cuda")
    ef = torch.empty(2, 0, 3, dtype=torch.float32, device="cuda")
    out = torch.full_like(s0, float("nan"))
    o, s1 = decode_step(e, e, ev, ef, ef, s0, state_out=out)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 3, 64) and torch.equal(s1, s0)
    keep = s0.clone()
    decode_step(e, e, ev, ef, ef, s0)
    torch.cuda.synchronize()
    assert torch.equal(s0, keep)


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_workload_whole(name):
    """The full decode workload, in the launch configuration the benchmark
    times, against the oracle over the whole of o and the new state."""
    w = DECODE_WORKLOADS[name]
    x = make_workload(name)
    s0 = x["h0"]
    d = gpu({n: t for n, t in x.items() if n != "h0"})
    state = s0.cuda()
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state)
    torch.cuda.synchronize()
    eo, es = whole_errors(x, o, s1, lambda sub: oracle(sub, sub["h0"]))
    assert eo < TOL_O["bf16"], eo
    assert es < TOL_S, es
    assert native.decode_launches(native.problem(w.B, w.T, w.H, w.K, w.V, torch.bfloat16)) == \
        ["gdn_decode_step_kernel"]
