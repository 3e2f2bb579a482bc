"""The device-timeout path of the tensor-core forward, made to run out on
purpose without faulting or hanging anything.

gdn_debug_arm_stall makes the next tensor-core launch withhold its first
chunk's loads: every role's first wait on them is a wait on a barrier that
nothing completes, so each gives up after the armed limit, the roles leave
their loops, what was issued drains, and the launch records the timeout in the
workspace's status word. The test checks that gdn_check_device_status reports
GDN_ERR_DEVICE_TIMEOUT, that the host-memory entry returns it, and that the
next call on the same context is correct again."""
import numpy as np
import pytest
import torch

from oracle import recurrence
from tests.pins import rel
from gated_delta_rule_35_gb300 import GdnError, chunk_fwd, chunk_fwd_host, check_device_status, native
from gated_delta_rule_35_gb300.inputs import make_inputs, to_f64

pytestmark = pytest.mark.gpu

LIMIT_NS = 5_000_000   # 5 ms: each waiting role gives up after this long


def _inputs():
    x = make_inputs(2, 300, 3, 128, 128, dtype="bf16", seed=88, h0_std=0.1)
    return x, {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


@pytest.mark.parametrize("algo", ["tc", "tc1", "tcw"])
def test_withheld_loads_report_a_device_timeout_then_recover(algo):
    """Both tensor-core forms; in the single-kernel form the WY group's own
    waits (on the next chunk's W and U) run out as well."""
    x, d = _inputs()
    p = native.problem(2, 300, 3, 128, 128, torch.bfloat16, algo)
    ws = torch.zeros(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    native.debug_arm_stall(LIMIT_NS)
    chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo, workspace=ws)
    assert check_device_status(ws) == native.GDN_ERR_DEVICE_TIMEOUT
    # the status word was cleared by the read; the context is still usable
    assert check_device_status(ws) == native.GDN_OK
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo,
                      workspace=ws)
    torch.cuda.synchronize()
    assert check_device_status(ws) == native.GDN_OK
    o_ref, hf_ref = recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                       to_f64(x["g"]), to_f64(x["beta"]), 1.0, to_f64(x["h0"]))
    assert rel(o.float().cpu().numpy(), o_ref) < 2e-2
    assert rel(hf.cpu().numpy(), hf_ref) < 2e-2


@pytest.mark.parametrize("V", [128, 256])
def test_wide_kernel_output_stage_reports_a_device_timeout_then_recovers(V):
    """The 128-column kernel with the output stage inside it (V = 256: two-CTA
    clusters sharing the row sums): withheld loads end every role's wait, both
    CTAs of a cluster meet at its closing barrier, and the next call is right."""
    from oracle import epilogue
    from gated_delta_rule_35_gb300.inputs import make_output_norm
    B, T, H, K = 2, 300, 3, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=90, h0_std=0.1)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    gate, weight = make_output_norm(B, T, H, V, seed=90)
    kw = dict(gate=gate.cuda(), norm_weight=weight.cuda(), norm_eps=1e-6)
    p = native.problem(B, T, H, K, V, torch.bfloat16, "tcw")
    ws = torch.zeros(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    native.debug_arm_stall(LIMIT_NS)
    chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tcw", workspace=ws, **kw)
    assert check_device_status(ws) == native.GDN_ERR_DEVICE_TIMEOUT
    assert check_device_status(ws) == native.GDN_OK
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tcw", workspace=ws, **kw)
    torch.cuda.synchronize()
    assert check_device_status(ws) == native.GDN_OK
    o_ref, hf_ref = recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                       to_f64(x["g"]), to_f64(x["beta"]), 1.0, to_f64(x["h0"]))
    o_ref = epilogue.gated_rmsnorm(o_ref, to_f64(gate), to_f64(weight), 1e-6)
    assert rel(o.float().cpu().numpy(), o_ref) < 2e-2
    assert rel(hf.cpu().numpy(), hf_ref) < 2e-2


@pytest.mark.parametrize("gated", [False, True])
def test_per_channel_form_reports_a_device_timeout_then_recovers(gated):
    """The per-channel tensor-core form's forward kernel: its first load
    withheld, every role's bounded wait runs out (with the output stage, in
    every CTA of each cluster), the status word records it, and the next call
    on the same context is correct."""
    from oracle import epilogue
    from gated_delta_rule_35_gb300.inputs import make_output_norm
    B, T, H, K, V = 2, 200, 3, 128, 128
    x = make_inputs(B, T, H, K, V, dtype="bf16", seed=89, h0_std=0.1, per_channel=True)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    kw = {}
    if gated:
        gate, weight = make_output_norm(B, T, H, V, seed=89)
        kw = dict(gate=gate.cuda(), norm_weight=weight.cuda(), norm_eps=1e-6)
    p = native.problem(B, T, H, K, V, torch.bfloat16, "tc", native.flags_of(per_channel=True))
    ws = torch.zeros(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    native.debug_arm_stall(LIMIT_NS)
    chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tc", workspace=ws,
              per_channel_decay=True, **kw)
    assert check_device_status(ws) == native.GDN_ERR_DEVICE_TIMEOUT
    assert check_device_status(ws) == native.GDN_OK
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="tc", workspace=ws,
                      per_channel_decay=True, **kw)
    torch.cuda.synchronize()
    assert check_device_status(ws) == native.GDN_OK
    o_ref, hf_ref = recurrence.forward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]),
                                       to_f64(x["beta"]), 1.0, to_f64(x["h0"]))
    if gated:
        o_ref = epilogue.gated_rmsnorm(o_ref, to_f64(gate), to_f64(weight), 1e-6)
    assert rel(o.float().cpu().numpy(), o_ref) < 2e-2
    assert rel(hf.cpu().numpy(), hf_ref) < 2e-2


def test_host_entry_returns_a_device_timeout():
    x, _ = _inputs()
    hx = {n: (t.pin_memory() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    native.debug_arm_stall(LIMIT_NS)
    with pytest.raises(GdnError) as e:
        chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], 1.0, hx["h0"], algo="tc")
    assert e.value.status == native.GDN_ERR_DEVICE_TIMEOUT
    o, hf = chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], 1.0, hx["h0"], algo="tc")
    assert np.isfinite(o.float().numpy()).all() and np.isfinite(hf.numpy()).all()
