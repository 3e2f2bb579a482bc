"""Both product calls are capturable in a CUDA graph: neither allocates, syncs
or reads device memory on the host, so a serving loop can replay them without
launch overhead. The replayed graph must give exactly what eager calls give."""
import pytest
import torch

from gated_delta_rule_35_gb300 import chunk_fwd, decode_step, native
from gated_delta_rule_35_gb300.inputs import make_inputs, make_output_norm

pytestmark = pytest.mark.gpu


def gpu(x):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def test_decode_steps_replay_from_a_graph():
    B, T, H, K, V = 8, 4, 16, 128, 128
    x = gpu(make_inputs(B, T, H, K, V, dtype="bf16", seed=51, h0_std=0.1, chunk=1))
    tok = [{n: x[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
           for t in range(T)]
    outs = [torch.empty(B, 1, H, V, dtype=torch.bfloat16, device="cuda") for _ in range(T)]

    eager_state = x["h0"].clone()
    eager = []
    for t in range(T):
        o, _ = decode_step(tok[t]["q"], tok[t]["k"], tok[t]["v"], tok[t]["g"], tok[t]["beta"],
                           eager_state)
        eager.append(o)

    state = x["h0"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside capture
        decode_step(tok[0]["q"], tok[0]["k"], tok[0]["v"], tok[0]["g"], tok[0]["beta"],
                    state.clone(), out=outs[0])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for t in range(T):
            decode_step(tok[t]["q"], tok[t]["k"], tok[t]["v"], tok[t]["g"], tok[t]["beta"],
                        state, out=outs[t])
    g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(outs[t], eager[t]), t
    assert torch.equal(state, eager_state)


@pytest.mark.parametrize("algo", ["simt", "tc"])
@pytest.mark.parametrize("gated", [False, True])
def test_chunk_fwd_replays_from_a_graph(algo, gated):
    """With the output stage the tensor-core path is a cluster launch."""
    B, T, H, K, V = 2, 200, 4, 128, 128
    p = native.problem(B, T, H, K, V, torch.bfloat16, algo)
    if native.workspace_bytes(p) == 0:
        pytest.skip(f"{algo} not built")
    x = gpu(make_inputs(B, T, H, K, V, dtype="bf16", seed=52, h0_std=0.1))
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, x["h0"])
    kw = {}
    if gated:
        gate, weight = make_output_norm(B, T, H, V, seed=52)
        kw = dict(gate=gate.cuda(), norm_weight=weight.cuda())
    o_e, hf_e = chunk_fwd(*args, algo=algo, **kw)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o_e)
    hf = torch.empty_like(hf_e)
    chunk_fwd(*args, algo=algo, workspace=ws, out=o, final_state=hf, **kw)   # warm-up
    torch.cuda.synchronize()
    o.fill_(float("nan"))
    hf.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chunk_fwd(*args, algo=algo, workspace=ws, out=o, final_state=hf, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(hf, hf_e)


@pytest.mark.parametrize("shape,per_channel", [((1, 130, 160, 128, 128), False), ((2, 200, 3, 128, 128), True)])
def test_split_forward_and_per_channel_form_replay_from_a_graph(shape, per_channel):
    """The split forward (the wide kernel on a whole wave of heads, the
    64-column kernel started right behind it for the rest: B1 H160 gives 152 +
    8 heads on 152 SMs) and the per-channel tensor-core form, captured and
    replayed: bit for bit the eager result."""
    B, T, H, K, V = shape
    x = gpu(make_inputs(B, T, H, K, V, dtype="bf16", seed=53, h0_std=0.1, per_channel=per_channel))
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, x["h0"])
    kw = dict(algo="tc", per_channel_decay=per_channel)
    p = native.problem(B, T, H, K, V, torch.bfloat16, "tc", native.flags_of(per_channel=per_channel))
    o_e, hf_e = chunk_fwd(*args, **kw)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o_e)
    hf = torch.empty_like(hf_e)
    chunk_fwd(*args, workspace=ws, out=o, final_state=hf, **kw)   # warm-up
    torch.cuda.synchronize()
    o.fill_(float("nan"))
    hf.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chunk_fwd(*args, workspace=ws, out=o, final_state=hf, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(hf, hf_e)
    assert native.check_device_status(ws) == native.GDN_OK


@pytest.mark.parametrize("shape,algo", [((1, 130, 160, 128, 128), "tc"), ((1, 130, 3, 128, 256), "tcw")])
def test_output_stage_on_the_wide_kernel_replays_from_a_graph(shape, algo):
    """The output stage inside the 128-column kernel, captured and replayed:
    the split forward (152 heads on that kernel, 8 on the 64-column kernel's
    cluster form) and V = 256 (two-CTA clusters of the wide kernel); bit for
    bit the eager result."""
    B, T, H, K, V = shape
    x = gpu(make_inputs(B, T, H, K, V, dtype="bf16", seed=54, h0_std=0.1))
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, x["h0"])
    gate, weight = make_output_norm(B, T, H, V, seed=54)
    kw = dict(algo=algo, gate=gate.cuda(), norm_weight=weight.cuda())
    p = native.problem(B, T, H, K, V, torch.bfloat16, algo)
    o_e, hf_e = chunk_fwd(*args, **kw)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o_e)
    hf = torch.empty_like(hf_e)
    chunk_fwd(*args, workspace=ws, out=o, final_state=hf, **kw)   # warm-up
    torch.cuda.synchronize()
    o.fill_(float("nan"))
    hf.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chunk_fwd(*args, workspace=ws, out=o, final_state=hf, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(hf, hf_e)
    assert native.check_device_status(ws) == native.GDN_OK
