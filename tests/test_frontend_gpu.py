"""The in-kernel input front-end (problem flags GDN_FLAG_RAW_G and
GDN_FLAG_QK_L2NORM) against the fp64 oracle, element by element.

The oracle applies ``oracle.frontend.prepare`` (chunk-local cumsum, row
normalisation) and then the token recurrence. Tolerances are those of the plain
path: relative Frobenius 1e-4 for fp32 inputs, 2e-2 for bf16 inputs; the
SIMT stages 1e-5 against the fp64 chunked form."""
import numpy as np
import pytest
import torch

from oracle import chunked, frontend, recurrence
from tests.pins import rel
from tests.whole_tensor import whole_errors
from gated_delta_rule_35_gb300 import chunk_fwd, chunk_fwd_stages, decode_step, native
from gated_delta_rule_35_gb300.inputs import chunk_local_cumsum, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}
MODES = {"raw_g": (True, False), "l2norm": (False, True), "both": (True, True)}


def have_algo(algo, K, V, dtype):
    return native.workspace_bytes(native.problem(1, 64, 1, K, V, TORCH[dtype], algo)) > 0


def inputs(B, T, H, K, V, dtype, seed, raw_g, l2norm, **kw):
    """q, k unnormalised when the kernels normalise them; g raw when the kernels sum it."""
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=seed, h0_std=0.1, raw=l2norm, chunk=1, **kw)
    if not raw_g:
        x["g"] = chunk_local_cumsum(x["g"])
    return x


def oracle(x, scale, raw_g, l2norm):
    q, k, g = frontend.prepare(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["g"]), raw_g=raw_g,
                               qk_l2norm=l2norm)
    return recurrence.forward(q, k, to_f64(x["v"]), g, to_f64(x["beta"]), scale, to_f64(x["h0"]))


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


@pytest.mark.parametrize("algo", ["simt", "tc", "tc1", "tcw"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_frontend_parity(algo, dtype, mode, K, V, T):
    if not have_algo(algo, K, V, dtype):
        pytest.skip(f"{algo} not built for K={K} V={V} {dtype}")
    raw_g, l2norm = MODES[mode]
    x = inputs(2, T, 3, K, V, dtype, 300 + T + K + V, raw_g, l2norm)
    scale = K ** -0.5 if l2norm else 1.0
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale, d["h0"], algo=algo,
                      raw_g=raw_g, qk_l2norm=l2norm)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, scale, raw_g, l2norm)
    o, hf = o.float().cpu().numpy(), hf.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(hf).all()
    assert rel(o, o_ref) < TOL[dtype], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL[dtype], rel(hf, hf_ref)


@pytest.mark.parametrize("algo", ["simt", "tc", "tc1", "tcw"])
@pytest.mark.parametrize("g_div", [1.0, 0.25])
def test_frontend_strong_decay(algo, g_div):
    """Chunk sums of the raw decays near -45 and -180: the second takes the
    tensor-core path's per-element exponential form, with the norm factors
    entering as exponent offsets."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    x = inputs(2, 200, 2, 128, 128, "bf16", 41, True, True, g_div=g_div)
    assert float(chunk_local_cumsum(x["g"]).min()) < (-30 if g_div == 1.0 else -150)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 128 ** -0.5, d["h0"], algo=algo,
                      raw_g=True, qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, 128 ** -0.5, True, True)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_frontend_simt_stages(dtype):
    """Every SIMT intermediate with both front-end steps, against the fp64
    chunked form run on the oracle's prepared inputs."""
    T = 150
    x = inputs(2, T, 2, 128, 128, dtype, 43, True, True)
    d = gpu(x)
    st = chunk_fwd_stages(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.5, d["h0"], algo="simt",
                          raw_g=True, qk_l2norm=True)
    torch.cuda.synchronize()
    q, k, g = frontend.prepare(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["g"]), raw_g=True,
                               qk_l2norm=True)
    ref = chunked.forward(q, k, to_f64(x["v"]), g, to_f64(x["beta"]), 0.5, to_f64(x["h0"]),
                          stages=True)
    for name in ("A", "w", "u", "v_new"):
        got = st[name][:, :T].cpu().numpy()
        assert rel(got, ref[name]) < 1e-5, (name, rel(got, ref[name]))
    assert rel(st["h"].cpu().numpy(), ref["h"]) < 1e-5


def test_frontend_full_size_whole():
    """The default workload's shape (B4 H16 T2048, K = V = 128, bf16) with raw
    inputs and both steps through 'auto', against the oracle over the whole
    of o and h_final."""
    B, T, H, K, V = 4, 2048, 16, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=1, raw=True)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], K ** -0.5, None, raw_g=True,
                      qk_l2norm=True)
    torch.cuda.synchronize()
    eo, eh = whole_errors(x, o, hf, lambda sub: oracle(sub, K ** -0.5, True, True))
    assert eo < TOL["bf16"], eo
    assert eh < TOL["bf16"], eh


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 2, 4, 128, 128), (20, 1, 16, 64, 128), (1, 3, 2, 256, 48)])
def test_decode_l2norm(dtype, shape):
    """The decode step with the norm: unnormalised q, k against the oracle on
    normalised rows (state 1e-5; o 1e-5 fp32, 2.5e-3 bf16)."""
    B, T, H, K, V = shape
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=B + T + K, h0_std=0.1, raw=True)
    s0 = x.pop("h0")
    d = gpu(x)
    state = s0.cuda()
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, K ** -0.5,
                        qk_l2norm=True)
    torch.cuda.synchronize()
    q, k, _ = frontend.prepare(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["g"]), raw_g=False,
                               qk_l2norm=True)
    o_ref, s_ref = recurrence.forward(q, k, to_f64(x["v"]), to_f64(x["g"]), to_f64(x["beta"]),
                                      K ** -0.5, to_f64(s0), chunk=1)
    assert rel(o.float().cpu().numpy(), o_ref) < (1e-5 if dtype == "f32" else 2.5e-3)
    assert rel(s1.cpu().numpy(), s_ref) < 1e-5
