"""The host-tensor entry (chunk_fwd_host, gdn_chunk_fwd_host): pinned host
inputs in, host outputs out, with the copies of one span of T overlapping the
kernels of the previous one. It must give what the device entry gives: bit for
bit with one span, within 1e-3 with several (the state crosses a span boundary
through h_final -> h0, as in the split/resume test)."""
import pytest
import torch

from tests.pins import rel
from gated_delta_rule_35_gb300 import chunk_fwd, chunk_fwd_host
from gated_delta_rule_35_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def pinned(x):
    return {n: (t.pin_memory() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


@pytest.mark.parametrize("algo", ["simt", "tc"])
@pytest.mark.parametrize("B,T", [(4, 200), (3, 201), (1, 130)])
def test_host_entry_one_span_bitwise(algo, B, T):
    x = make_inputs(B, T, 3, 128, 128, dtype="bf16", seed=80 + B, h0_std=0.1)
    h = pinned(x)
    ho, hhf = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], 1.0, h["h0"], algo=algo,
                             pieces=1)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo)
    torch.cuda.synchronize()
    assert ho.is_pinned() and torch.equal(ho, o.cpu()) and torch.equal(hhf, hf.cpu())


@pytest.mark.parametrize("algo", ["simt", "tc"])
@pytest.mark.parametrize("B,T,pieces", [(1, 300, 4), (1, 64, 4), (1, 1000, 8), (4, 2048, 8),
                                        (3, 201, 3)])
def test_host_entry_spans(algo, B, T, pieces):
    x = make_inputs(B, T, 4, 128, 128, dtype="bf16", seed=90 + T, h0_std=0.1)
    h = pinned(x)
    ho, hhf = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], 1.0, h["h0"], algo=algo,
                             pieces=pieces)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo)
    torch.cuda.synchronize()
    assert rel(ho.float().numpy(), o.float().cpu().numpy()) < 1e-3
    assert rel(hhf.numpy(), hf.cpu().numpy()) < 1e-3


@pytest.mark.parametrize("algo", ["simt", "tc"])
@pytest.mark.parametrize("pieces", [1, 4])
def test_host_entry_per_channel_decay(algo, pieces):
    """Per-channel decay through the host entry (g [B,T,H,K] cut into the same
    spans): bit for bit with one span, within 1e-3 with several."""
    x = make_inputs(2, 300, 3, 128, 128, dtype="bf16", seed=97, h0_std=0.1, per_channel=True)
    h = pinned(x)
    ho, hhf = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], 1.0, h["h0"], algo=algo,
                             pieces=pieces, per_channel_decay=True)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=algo,
                      per_channel_decay=True)
    torch.cuda.synchronize()
    if pieces == 1:
        assert torch.equal(ho, o.cpu()) and torch.equal(hhf, hf.cpu())
    else:
        assert rel(ho.float().numpy(), o.float().cpu().numpy()) < 1e-3
        assert rel(hhf.numpy(), hf.cpu().numpy()) < 1e-3


def test_host_entry_without_final_state_and_empty():
    x = pinned(make_inputs(2, 100, 2, 64, 64, dtype="bf16", seed=95))
    ho, hhf = chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, None,
                             output_final_state=False)
    assert hhf is None and ho.shape == (2, 100, 2, 64)
    e = torch.empty(2, 0, 3, 64, dtype=torch.bfloat16)
    ef = torch.empty(2, 0, 3)
    h0 = torch.randn(2, 3, 64, 64)
    ho, hhf = chunk_fwd_host(e, e, e, ef, ef, 1.0, h0)
    assert ho.shape == (2, 0, 3, 64) and torch.equal(hhf, h0)


def test_host_entry_into_given_outputs_and_growing_buffer():
    """Caller-owned outputs are written in place; a larger problem after a
    smaller one grows the kept device buffer, and a smaller one after it
    reuses it, each matching the device entry."""
    for B, T, H in [(1, 130, 2), (2, 700, 4), (1, 64, 1)]:
        x = make_inputs(B, T, H, 128, 128, dtype="bf16", seed=97 + T, h0_std=0.1)
        h = pinned(x)
        out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
        fs = torch.full((B, H, 128, 128), float("nan")).pin_memory()
        ho, hhf = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], 1.0, h["h0"],
                                 pieces=1, out=out, final_state=fs)
        assert ho.data_ptr() == out.data_ptr() and hhf.data_ptr() == fs.data_ptr()
        d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        o, hf = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"])
        torch.cuda.synchronize()
        assert torch.equal(out, o.cpu()) and torch.equal(fs, hf.cpu()), (B, T, H)


def test_host_entry_rejects_bad_outputs():
    x = pinned(make_inputs(1, 64, 1, 64, 64, dtype="bf16", seed=98))
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], 1.0, None)
    with pytest.raises(ValueError):
        chunk_fwd_host(*args, out=torch.empty(1, 64, 1, 64, dtype=torch.float32))
    with pytest.raises(ValueError):
        chunk_fwd_host(*args, final_state=torch.empty(1, 1, 64, 32))
    with pytest.raises(ValueError):
        chunk_fwd_host(*args, out=torch.empty(1, 64, 1, 64, dtype=torch.bfloat16, device="cuda"))
