"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerance: relative Frobenius error ||x - x_ref||_F / ||x_ref||_F over the whole
tensor, separately for o and h_final: 1e-4 for fp32 inputs, 2e-2 for bf16
inputs (the bf16 tensor-core path rounds its MMA operands to bf16)."""
import numpy as np
import pytest
import torch

from oracle import chunked, recurrence
from tests.pins import rel
from tests.whole_tensor import whole_errors
from gated_delta_rule_35_gb300 import chunk_fwd, chunk_fwd_stages, check_device_status, native
from gated_delta_rule_35_gb300.inputs import WORKLOADS, make_inputs, make_workload, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def have_algo(algo, K, V, dtype):
    p = native.problem(1, 64, 1, K, V, TORCH[dtype], algo)
    return native.workspace_bytes(p) > 0


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def run_gpu(x, algo, scale=1.0):
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale, d["h0"], algo=algo)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), hf.cpu().numpy()


def run_oracle(x, scale=1.0):
    return recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]),
                              to_f64(x["beta"]), scale, to_f64(x["h0"]))


ALGOS = ["simt", "tc", "tc1", "tcw"]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256), (64, 192)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 100, 200])
def test_small_parity(algo, dtype, K, V, T):
    if not have_algo(algo, K, V, dtype):
        pytest.skip(f"{algo} not built for K={K} V={V} {dtype}")
    x = make_inputs(2, T, 3, K, V, dtype=dtype, seed=1000 + T + K + V, h0_std=0.1)
    o, hf = run_gpu(x, algo)
    o_ref, hf_ref = run_oracle(x)
    assert np.isfinite(o).all() and np.isfinite(hf).all()
    assert rel(o, o_ref) < TOL[dtype], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL[dtype], rel(hf, hf_ref)


@pytest.mark.parametrize("algo", ALGOS)
def test_scale_and_zero_state(algo):
    """scale = K^-0.5 with unnormalised-scale q, and h0 = None (zero state)."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    x = make_inputs(1, 300, 4, 128, 128, dtype="bf16", seed=77)
    x["q"] = (x["q"].float() * 128 ** 0.5).to(torch.bfloat16)
    o, hf = run_gpu(x, algo, scale=128 ** -0.5)
    o_ref, hf_ref = run_oracle(x, scale=128 ** -0.5)
    assert rel(o, o_ref) < TOL["bf16"] and rel(hf, hf_ref) < TOL["bf16"]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("g_div", [1.0, 0.25])
def test_strong_decay(algo, g_div):
    """Forget gates far below 1: a chunk's cumulative log decay reaches about -45
    (g_div = 1) or about -180 (g_div = 0.25), where the inverse decay factors
    leave the fp32 range and the exact exp(g_i - g_j) form must be used."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    x = make_inputs(2, 200, 2, 128, 128, dtype="bf16", seed=21, h0_std=0.1, g_div=g_div)
    assert float(x["g"].min()) < (-30 if g_div == 1.0 else -150)
    o, hf = run_gpu(x, algo)
    o_ref, hf_ref = run_oracle(x)
    assert np.isfinite(o).all() and np.isfinite(hf).all()
    assert rel(o, o_ref) < TOL["bf16"], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL["bf16"], rel(hf, hf_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_simt_stages_against_chunked_form(dtype):
    """Every SIMT intermediate (A, w, u, v_new, h) against the fp64 chunked form.
    The SIMT path computes in fp32 from the same inputs, so 1e-5 holds for both dtypes."""
    x = make_inputs(2, 150, 2, 128, 128, dtype=dtype, seed=5, h0_std=0.1)
    d = gpu(x)
    st = chunk_fwd_stages(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="simt")
    torch.cuda.synchronize()
    ref = chunked.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]),
                          to_f64(x["beta"]), 1.0, to_f64(x["h0"]), stages=True)
    T = 150
    for name in ("A", "w", "u", "v_new"):
        got = st[name][:, :T].cpu().numpy()
        assert rel(got, ref[name]) < 1e-5, (name, rel(got, ref[name]))
    assert rel(st["h"].cpu().numpy(), ref["h"]) < 1e-5
    assert rel(st["o"].float().cpu().numpy(), ref["o"]) < TOL[dtype]


@pytest.mark.parametrize("K", [64, 128])
def test_tc_wy_stage_against_chunked_form(K):
    """The tensor-core WY stage, A diag(beta) per chunk (bf16 in the workspace),
    against the fp64 chunked form's A with its columns scaled by beta."""
    if not have_algo("tc", K, 128, "bf16"):
        pytest.skip("not built")
    T = 150
    x = make_inputs(2, T, 2, K, 128, dtype="bf16", seed=6)
    d = gpu(x)
    st = chunk_fwd_stages(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None, algo="tc",
                          stages=("A_beta",))
    torch.cuda.synchronize()
    ref = chunked.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]),
                          to_f64(x["beta"]), 1.0, None, stages=True)
    beta = to_f64(x["beta"])
    B, _, H = beta.shape
    cols = np.zeros((B, T, H, 64))
    for t in range(T):
        s = (t // 64) * 64
        e = min(T, s + 64)
        cols[:, t, :, : e - s] = beta[:, s:e, :].transpose(0, 2, 1)
    want = ref["A"] * cols
    got = st["A_beta"][:, :T].cpu().numpy()
    assert rel(got, want) < 1e-2, rel(got, want)
    assert np.all(st["A_beta"][:, T:].cpu().numpy() == 0)


@pytest.mark.parametrize("algo", ALGOS)
def test_empty_sequence(algo):
    """T = 0: no output rows; h_final = h0, or zeros without h0."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    h0 = torch.randn(2, 3, 128, 128, device="cuda")
    e = torch.empty(2, 0, 3, 128, dtype=torch.bfloat16, device="cuda")
    ef = torch.empty(2, 0, 3, dtype=torch.float32, device="cuda")
    o, hf = chunk_fwd(e, e, e, ef, ef, 1.0, h0, algo=algo)
    assert o.shape == (2, 0, 3, 128) and torch.equal(hf, h0)
    o, hf = chunk_fwd(e, e, e, ef, ef, 1.0, None, algo=algo)
    assert torch.count_nonzero(hf) == 0


@pytest.mark.parametrize("algo", ALGOS)
def test_split_resume(algo):
    """fwd(T1) then fwd(T2, h0 = h_final) matches fwd(T1 + T2) when 64 | T1."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    x = gpu(make_inputs(2, 320, 2, 128, 128, dtype="bf16", seed=9, h0_std=0.1))
    a = {n: t for n, t in x.items()}
    o, hf = chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], 1.0, a["h0"], algo=algo)
    T1 = 192
    sl = lambda t, s: t[:, s].contiguous()
    o1, h1 = chunk_fwd(*(sl(a[n], slice(0, T1)) for n in ("q", "k", "v", "g", "beta")), 1.0,
                       a["h0"], algo=algo)
    o2, h2 = chunk_fwd(*(sl(a[n], slice(T1, None)) for n in ("q", "k", "v", "g", "beta")), 1.0,
                       h1, algo=algo)
    torch.cuda.synchronize()
    oc = torch.cat([o1, o2], 1).float().cpu().numpy()
    assert rel(oc, o.float().cpu().numpy()) < 1e-3
    assert rel(h2.cpu().numpy(), hf.cpu().numpy()) < 1e-3


@pytest.mark.parametrize("V", [128, 256])
def test_wide_kernel_matches_narrow(V):
    """The 128-column forward kernel against the 64-column one on the same
    inputs: the same products in the same precision, only grouped differently
    per CTA, so the two agree far inside the oracle tolerance."""
    if not have_algo("tcw", 128, V, "bf16"):
        pytest.skip("not built")
    x = make_inputs(2, 300, 3, 128, V, dtype="bf16", seed=61 + V, h0_std=0.1)
    o_w, hf_w = run_gpu(x, "tcw")
    o_n, hf_n = run_gpu(x, "tc")
    assert rel(o_w, o_n) < 1e-3, rel(o_w, o_n)
    assert rel(hf_w, hf_n) < 1e-3, rel(hf_w, hf_n)


def test_wide_waves_then_narrow_remainder():
    """B1 H160: 160 wide CTAs on 152 SMs, so 152 heads run on the wide kernel
    and the other 8 on the 64-column kernel launched right behind it; every
    head against the oracle."""
    if not have_algo("tc", 128, 128, "bf16"):
        pytest.skip("not built")
    p = native.problem(1, 130, 160, 128, 128, torch.bfloat16, "tc")
    names = native.launches(p)
    x = make_inputs(1, 130, 160, 128, 128, dtype="bf16", seed=71, h0_std=0.1)
    o, hf = run_gpu(x, "tc")
    o_ref, hf_ref = run_oracle(x)
    assert rel(o, o_ref) < TOL["bf16"], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL["bf16"], rel(hf, hf_ref)
    # the last heads specifically (the 64-column kernel's share when split)
    assert rel(o[:, :, 150:], o_ref[:, :, 150:]) < TOL["bf16"]
    assert rel(hf[:, 150:], hf_ref[:, 150:]) < TOL["bf16"]
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert names == ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel", "gdn_fused_tc_kernel"]


def test_small_workload_fp32():
    """The fp32 workload (B1 H1 T256 K=V=64) in full, tolerance 1e-4."""
    x = make_workload("f32_b1_h1_t256_k64_v64")
    o, hf = run_gpu(x, "auto")
    o_ref, hf_ref = run_oracle(x)
    assert rel(o, o_ref) < 1e-4 and rel(hf, hf_ref) < 1e-4


@pytest.mark.parametrize("name", [n for n in WORKLOADS if WORKLOADS[n].dtype == "bf16"])
def test_full_workload_whole(name):
    """Full-size bf16 workloads, in the launch configuration the benchmark
    times (algo 'auto'), against the oracle over the whole of o and h_final:
    every (b, h) sequence, relative Frobenius error over the whole tensor."""
    x = make_workload(name)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"])
    torch.cuda.synchronize()
    eo, eh = whole_errors(x, o, hf, run_oracle)
    assert eo < TOL["bf16"], (name, eo)
    assert eh < TOL["bf16"], (name, eh)


def test_device_status_clear():
    x = gpu(make_inputs(1, 64, 1, 64, 64, dtype="bf16", seed=1))
    ws = torch.zeros(native.workspace_bytes(native.problem(1, 64, 1, 64, 64, torch.bfloat16)),
                     dtype=torch.uint8, device="cuda")
    chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, None, workspace=ws)
    assert check_device_status(ws) == native.GDN_OK
