"""The gated RMSNorm output stage against the fp64 oracle (recurrence, then
``oracle.epilogue.gated_rmsnorm``), element by element, on both chunked paths
and the decode step. Tolerances are the plain path's (relative Frobenius 1e-4
fp32, 2e-2 bf16; decode 1e-5 fp32 and 2.5e-3 bf16, its state 1e-5): the stage
is formed in fp32 from the same o before its one rounding."""
import numpy as np
import pytest
import torch

from oracle import epilogue, frontend, recurrence
from tests.pins import rel
from tests.whole_tensor import whole_errors
from gated_delta_rule_35_gb300 import chunk_fwd, decode_step, native
from gated_delta_rule_35_gb300.inputs import make_inputs, make_output_norm, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}
EPS = 1e-6


def have_algo(algo, K, V, dtype):
    return native.workspace_bytes(native.problem(1, 64, 1, K, V, TORCH[dtype], algo)) > 0


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def oracle(x, gate, weight, scale=1.0, raw_g=False, l2norm=False, chunk=64):
    q, k, g = frontend.prepare(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["g"]), raw_g=raw_g,
                               qk_l2norm=l2norm)
    o, hf = recurrence.forward(q, k, to_f64(x["v"]), g, to_f64(x["beta"]), scale,
                               to_f64(x["h0"]), chunk=chunk)
    return epilogue.gated_rmsnorm(o, to_f64(gate), to_f64(weight), EPS), hf


@pytest.mark.parametrize("algo", ["simt", "tc", "tcw"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 256), (64, 192)])
@pytest.mark.parametrize("T", [1, 64, 65, 200])
def test_chunked_output_norm(algo, dtype, K, V, T):
    if not have_algo(algo, K, V, dtype):
        pytest.skip(f"{algo} not built for K={K} V={V} {dtype}")
    B, H = 2, 3
    seed = 500 + T + K + V
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=seed, h0_std=0.1)
    gate, weight = make_output_norm(B, T, H, V, dtype=dtype, seed=seed)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo,
                      gate=gate.cuda(), norm_weight=weight.cuda(), norm_eps=EPS)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, gate, weight)
    o, hf = o.float().cpu().numpy(), hf.cpu().numpy()
    assert np.isfinite(o).all()
    assert rel(o, o_ref) < TOL[dtype], rel(o, o_ref)
    assert rel(hf, hf_ref) < TOL[dtype], rel(hf, hf_ref)


@pytest.mark.parametrize("algo", ["simt", "tc", "tcw"])
def test_front_end_and_output_stage_together(algo):
    """Raw g, unnormalised q and k, and the gated RMSNorm in one call (tcw: the
    128-column kernel, which applies the stage itself)."""
    if not have_algo(algo, 128, 128, "bf16"):
        pytest.skip("not built")
    B, T, H, K, V = 2, 150, 2, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=61, h0_std=0.1, raw=True)
    gate, weight = make_output_norm(B, T, H, V, seed=61)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], K ** -0.5, d["h0"], algo=algo,
                      raw_g=True, qk_l2norm=True, gate=gate.cuda(), norm_weight=weight.cuda(),
                      norm_eps=EPS)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, gate, weight, K ** -0.5, raw_g=True, l2norm=True)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


@pytest.mark.parametrize("H,V,kernel", [(27, 192, "gdn_fused_tc_kernel"), (20, 256, "gdn_wide_tc_kernel")])
def test_output_norm_clusters_over_several_waves(H, V, kernel):
    """Clusters over more than one wave, 16 chunks with a ragged last one, so
    every slot of the output stage's hand-offs cycles several times: V = 192
    on the 64-column kernel (three-CTA clusters, 162 CTAs on 152 SMs, some
    clusters starting only as others finish) and V = 256 on the 128-column
    kernel (two-CTA clusters, 80 CTAs)."""
    B, T, K = 2, 1000, 128
    assert native.launches(native.problem(B, T, H, K, V, torch.bfloat16, "tc"))[1] == kernel
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=17, h0_std=0.1)
    gate, weight = make_output_norm(B, T, H, V, seed=17)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.5, d["h0"], algo="tc", gate=gate.cuda(),
                      norm_weight=weight.cuda(), norm_eps=EPS)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, gate, weight, scale=0.5)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]


def test_output_norm_on_the_wide_kernel_grid():
    """A grid that takes the 128-column kernel (B3 H64: 384 64-column tiles on
    152 SMs) with the output stage through 'auto': one whole wave of the wide
    kernel (152 heads), which applies the stage itself one chunk behind its
    o, and the other 40 heads on the 64-column kernel's cluster form; four
    chunks, the last ragged. Against the oracle, and the wide heads bit for bit
    against the wide-only form, which takes every head."""
    B, T, H, K, V = 3, 200, 64, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=19, h0_std=0.1)
    gate, weight = make_output_norm(B, T, H, V, seed=19)
    d = gpu(x)
    kw = dict(gate=gate.cuda(), norm_weight=weight.cuda(), norm_eps=EPS)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], **kw)
    ow, hw = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tcw", **kw)
    torch.cuda.synchronize()
    o_ref, hf_ref = oracle(x, gate, weight)
    assert rel(o.float().cpu().numpy(), o_ref) < TOL["bf16"]
    assert rel(hf.cpu().numpy(), hf_ref) < TOL["bf16"]
    assert rel(ow.float().cpu().numpy(), o_ref) < TOL["bf16"]
    p = native.problem(B, T, H, K, V, torch.bfloat16, "tc")
    assert native.launches(p) == ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel", "gdn_fused_tc_kernel"]
    # heads b * H + h < 152 are the wide kernel's in both calls
    wide = torch.arange(B * H).reshape(B, H) < 152
    assert torch.equal(o.permute(0, 2, 1, 3)[wide], ow.permute(0, 2, 1, 3)[wide])
    assert torch.equal(hf[wide], hw[wide])


@pytest.mark.parametrize("shape", [(8, 8192, 64, 128, 128, 3), (2, 16384, 32, 128, 256, 4)])
def test_output_norm_wide_shapes_whole(shape):
    """Full-size shapes that take the 128-column kernel, with the output stage
    through 'auto': B8 H64 T8192 (three whole waves with the stage inside the
    kernel, the other 56 heads on the 64-column kernel's cluster form, 128
    chunks each) and B2 H32 T16384 V256 (two-CTA clusters of the 128-column
    kernel sharing the row sums, 256 chunks); against the oracle over the
    whole of o and h_final."""
    B, T, H, K, V, seed = shape
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=seed)
    gate, weight = make_output_norm(B, T, H, V, seed=seed)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None, gate=gate.cuda(),
                      norm_weight=weight.cuda(), norm_eps=EPS)
    torch.cuda.synchronize()
    del d
    eo, eh = whole_errors(x, o, hf, lambda sub: oracle(sub, sub["gate"], weight),
                          extra={"gate": gate})
    assert eo < TOL["bf16"], eo
    assert eh < TOL["bf16"], eh


def test_output_norm_full_size_whole():
    """The default workload's shape with the output stage through 'auto' (the
    tensor-core path with two-CTA clusters), against the oracle over the whole
    of o and h_final."""
    B, T, H, K, V = 4, 2048, 16, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=1)
    gate, weight = make_output_norm(B, T, H, V, seed=1)
    d = gpu(x)
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None, gate=gate.cuda(),
                      norm_weight=weight.cuda(), norm_eps=EPS)
    torch.cuda.synchronize()
    eo, eh = whole_errors(x, o, hf, lambda sub: oracle(sub, sub["gate"], weight),
                          extra={"gate": gate})
    assert eo < TOL["bf16"], eo
    assert eh < TOL["bf16"], eh


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 2, 4, 128, 128), (2, 1, 5, 64, 64), (1, 3, 2, 128, 256),
                                   (4, 1, 2, 64, 16)])
@pytest.mark.parametrize("l2norm", [False, True])
def test_decode_output_norm(dtype, shape, l2norm):
    B, T, H, K, V = shape
    x = make_inputs(B, T, H, K, V, dtype=dtype, seed=B * 7 + T + V, h0_std=0.1, raw=l2norm,
                    chunk=1)
    gate, weight = make_output_norm(B, T, H, V, dtype=dtype, seed=B + V)
    s0 = x["h0"]
    d = gpu(x)
    state = s0.cuda()
    scale = K ** -0.5 if l2norm else 1.0
    o, s1 = decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, scale,
                        qk_l2norm=l2norm, gate=gate.cuda(), norm_weight=weight.cuda(),
                        norm_eps=EPS)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle(x, gate, weight, scale, l2norm=l2norm, chunk=1)
    assert rel(o.float().cpu().numpy(), o_ref) < (1e-5 if dtype == "f32" else 2.5e-3)
    assert rel(s1.cpu().numpy(), s_ref) < 1e-5
