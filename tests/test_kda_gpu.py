"""Per-channel (KDA) decay, problem flag GDN_FLAG_PER_CHANNEL_DECAY, against the
fp64 oracle's per-channel recurrence, element by element.

The chunked forward runs it on the CUDA-core pipeline (fp32 arithmetic) or,
for bf16, on the tensor-core form of its own (gdn_kda_prep_tc_kernel and
gdn_kda_fwd_tc_kernel), the decode step in its own kernel. Tolerances: relative Frobenius 1e-4 for fp32
inputs and 2e-2 for bf16 inputs (the plain path's); the exported stages 1e-5;
decode 1e-5 (state, fp32 o) and 2.5e-3 (bf16 o)."""
import numpy as np
import pytest
import torch

from oracle import epilogue, frontend, recurrence
from tests.pins import rel
from tests.whole_tensor import whole_errors
from gated_delta_rule_35_gb300 import GdnError, chunk_fwd, chunk_fwd_stages, decode_step, native
from gated_delta_rule_35_gb300.inputs import make_inputs, make_output_norm, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def oracle(x, scale=1.0, raw_g=False, l2norm=False, chunk=64, stages=False):
    q, k, g = frontend.prepare(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["g"]), raw_g=raw_g,
                               qk_l2norm=l2norm)
    return recurrence.forward(q, k, to_f64(x["v"]), g, to_f64(x["beta"]), scale,
                              to_f64(x["h0"]), chunk=chunk, stages=stages)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_kda_chunked_parity(dtype, K, V, T):
    x = make_inputs(2, T, 3, K, V, dtype=dtype, seed=700 + T + K + V, h0_std=0.1,
                    per_channel=True)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"],
                      per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x)
    o, hf = o.float().cpu().numpy(), hf.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(hf).all()
    assert rel(o, o_ref) < TOL[dtype], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL[dtype], rel(hf, hf_ref)


@pytest.mark.parametrize("g_div", [1.0, 0.2])
def test_kda_strong_and_uneven_decay(g_div):
    """Channels decaying at very different rates, some near exp(-300) over a chunk."""
    x = make_inputs(2, 150, 2, 128, 128, dtype="f32", seed=71, h0_std=0.1, per_channel=True,
                    g_div=g_div)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"],
                      per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x)
    assert rel(o.cpu().numpy(), o_ref) < TOL["f32"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["f32"]


def test_kda_stages_against_recurrence():
    """The state entering each chunk and the per-token correction d_t (v_new)
    of the CUDA-core pipeline against the recurrence's exports."""
    T = 150
    x = make_inputs(2, T, 2, 64, 64, dtype="f32", seed=72, h0_std=0.1, per_channel=True)
    d = gpu(x)
    st = chunk_fwd_stages(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="simt",
                          stages=("v_new", "h"), per_channel_decay=True)
    torch.cuda.synchronize()
    _, _, hc, dl = oracle(x, stages=True)
    assert rel(st["h"].cpu().numpy(), hc) < 1e-5
    assert rel(st["v_new"][:, :T].cpu().numpy(), dl) < 1e-5


def test_kda_with_front_end_and_output_stage():
    B, T, H, K, V = 2, 130, 2, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=73, h0_std=0.1, raw=True, per_channel=True)
    gate, weight = make_output_norm(B, T, H, V, seed=73)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], K ** -0.5, d["h0"], raw_g=True,
                      qk_l2norm=True, gate=gate.cuda(), norm_weight=weight.cuda(),
                      per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, K ** -0.5, raw_g=True, l2norm=True)
    o_ref = epilogue.gated_rmsnorm(o_ref, to_f64(gate), to_f64(weight), 1e-6)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256), (64, 192)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 200])
def test_kda_tensor_core_parity(K, V, T):
    """The tensor-core form requested by name, every (b, h) against the oracle."""
    x = make_inputs(2, T, 3, K, V, dtype="bf16", seed=900 + T + K + V, h0_std=0.1, per_channel=True)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.7, d["h0"], algo="tc",
                      per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, 0.7)
    o, hf = o.float().cpu().numpy(), hf.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(hf).all()
    assert rel(o, o_ref) < TOL["bf16"], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL["bf16"], rel(hf, hf_ref)


@pytest.mark.parametrize("g_div", [1.0, 0.2])
def test_kda_tensor_core_strong_decay(g_div):
    """Decays reaching exp(-300) over a chunk: chunks with a channel beyond
    |g_last| = 160 take the one-exponential-per-term products, the others the
    factored ones; both against the oracle."""
    x = make_inputs(2, 150, 2, 128, 128, dtype="bf16", seed=75, h0_std=0.1, per_channel=True, g_div=g_div)
    gl = x["g"][:, 63::64].abs().amax().item()
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tc",
                      per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"], (gl, rel(o.float().cpu().numpy(), o_ref))
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


@pytest.mark.parametrize("raw_g,l2norm", [(True, False), (False, True), (True, True)])
def test_kda_tensor_core_front_end(raw_g, l2norm):
    B, T, H, K, V = 2, 130, 2, 128, 128
    # the same draws raw (q, k unnormalised, g per token) and prepared; q, k
    # raw only where the kernels normalise them
    xr = make_inputs(B, T, H, K, V, dtype="bf16", seed=76, h0_std=0.1, raw=True, per_channel=True)
    xp = make_inputs(B, T, H, K, V, dtype="bf16", seed=76, h0_std=0.1, per_channel=True)
    x = dict(xp)
    if l2norm:
        x["q"], x["k"] = xr["q"], xr["k"]
    if raw_g:
        x["g"] = xr["g"]
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], K ** -0.5, d["h0"], algo="tc", raw_g=raw_g,
                      qk_l2norm=l2norm, per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, K ** -0.5, raw_g=raw_g, l2norm=l2norm)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


def test_kda_tensor_core_a_export():
    """The exported A diag(beta) of the tensor-core form: per chunk lower
    triangular with diagonal beta_i (A is unit lower triangular), zero past T."""
    B, T, H, K, V = 1, 100, 2, 64, 64
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=77, per_channel=True)
    d = gpu(x)
    st = chunk_fwd_stages(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None, algo="tc",
                          stages=("A_beta",), per_channel_decay=True)
    torch.cuda.synchronize()
    a = st["A_beta"].cpu().numpy()
    beta = x["beta"].numpy()
    for t in range(T):
        r = t % 64
        assert np.all(a[:, t, :, r + 1:] == 0)
        np.testing.assert_allclose(a[:, t, :, r], beta[:, t, :], rtol=1e-2, atol=1e-3)
    assert np.all(a[:, T:] == 0)


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256), (64, 192)])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_kda_tensor_core_output_stage(K, V, T):
    """The per-channel tensor-core form with the gated RMSNorm output stage
    (a head's V tiles as one cluster), against the oracle's recurrence and
    epilogue."""
    B, H = 2, 3
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=950 + T + V, h0_std=0.1, per_channel=True)
    gate, weight = make_output_norm(B, T, H, V, seed=950 + T + V)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.5, d["h0"], algo="tc", gate=gate.cuda(),
                      norm_weight=weight.cuda(), per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, 0.5)
    o_ref = epilogue.gated_rmsnorm(o_ref, to_f64(gate), to_f64(weight), 1e-6)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"], rel(o.float().cpu().numpy(), o_ref)
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


def test_kda_tensor_core_limits():
    x = gpu(make_inputs(1, 64, 1, 64, 64, dtype="bf16", seed=74, per_channel=True))
    for algo in ("tc1", "tcw"):
        with pytest.raises(GdnError) as e:
            chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, None, algo=algo,
                      per_channel_decay=True)
        assert e.value.status == native.GDN_ERR_UNSUPPORTED
    with pytest.raises(GdnError) as e:
        chunk_fwd_stages(x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, None, algo="tc",
                         stages=("A", "w"), per_channel_decay=True)
    assert e.value.status == native.GDN_ERR_UNSUPPORTED
    p = native.problem(4, 2048, 16, 128, 128, torch.bfloat16, "auto",
                       native.flags_of(per_channel=True))
    assert native.launches(p) == ["gdn_kda_prep_tc_kernel", "gdn_kda_fwd_tc_kernel"]


def test_kda_full_size_whole():
    """The default workload's shape with per-channel decay through 'auto',
    against the oracle over the whole of o and h_final."""
    B, T, H, K, V = 4, 2048, 16, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=1, per_channel=True)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None,
                      per_channel_decay=True)
    torch.cuda.synchronize()
    eo, eh = whole_errors(x, o, hf, oracle)
    assert eo < TOL["bf16"], eo
    assert eh < TOL["bf16"], eh


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 2, 4, 128, 128), (20, 1, 16, 64, 128), (1, 3, 2, 256, 48)])
@pytest.mark.parametrize("l2norm", [False, True])
def test_kda_decode(dtype, shape, l2norm):
    B, T, H, K, V = shape
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=B + T + K, h0_std=0.1, raw=l2norm, chunk=1,
                    per_channel=True)
    d = gpu(x)
    state = x["h0"].cuda()
    scale = K ** -0.5 if l2norm else 1.0
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, scale,
                        qk_l2norm=l2norm, per_channel_decay=True)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle(x, scale, l2norm=l2norm, chunk=1)
    assert rel(o.float().cpu().numpy(), o_ref) < (1e-5 if dtype == "f32" else 2.5e-3)
    assert rel(s1.cpu().numpy(), s_ref) < 1e-5
