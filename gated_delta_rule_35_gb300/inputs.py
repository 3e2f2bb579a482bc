"""Seeded synthetic inputs for the chunked gated delta rule forward.

This module only draws and shapes random inputs; it contains none of the
forward pass's arithmetic, so the CUDA path and the fp64 oracle can both take
their inputs from it without sharing any of the method.

Recipe (one ``torch.Generator('cpu')`` per workload, drawn in this order):
  q, k ~ N(0,1) [B,T,H,K]; v ~ N(0,1) [B,T,H,V]; beta_raw ~ N(0,1) [B,T,H];
  g_raw ~ N(0,1) [B,T,H]; h0 ~ N(0,1) [B,H,K,V] (only when h0_std > 0).
  q, k are L2-normalised over K per (b,t,h) in fp32 (no epsilon); q is then
  multiplied by K**-0.5; beta = sigmoid(beta_raw + beta_mean);
  per-token log-decay = logsigmoid(g_raw + g_mean) / g_div;
  g = cumulative sum of the per-token log-decay *within each 64-token chunk*
  (``chunk=1`` leaves the per-token log-decay itself, the decode step's gamma);
  with ``raw=True`` q and k are left unnormalised (and q unscaled) and g is
  the per-token log-decay itself: the inputs of the in-kernel front-end;
  with ``per_channel=True`` g_raw is [B,T,H,K], one decay per key channel;
  h0 = h0_std * h0_raw. q, k, v are then cast to the compute dtype; g, beta and
  h0 stay fp32.

Five named workloads: a small fp32 case (one 256-token head, K=V=64), and
four bf16 cases with K=128: a short batch, a long prefill with a non-zero
initial state, a wide batch, and a V=256 case with near-zero decay and large
beta. The chunk size is C=64 throughout ("WarpDrive" page, section "Pipeline").

One decode workload (``DECODE_WORKLOADS``): 256 sequences x 16 heads advanced by
one token each, K = V = 128, bf16, from a state of std 0.1 (a prefill's h_final
stands there in use); its gamma is the per-token log-decay (``chunk=1``).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch
import torch.nn.functional as F

CHUNK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str          # "f32" or "bf16": dtype of q, k, v and o
    seed: int
    h0_std: float = 0.0
    g_mean: float = 0.0
    g_div: float = 16.0
    beta_mean: float = 0.0

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H

    def as_dict(self) -> dict:
        return asdict(self)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_b1_h1_t256_k64_v64", 1, 256, 1, 64, 64, "f32", seed=0),
        Workload("bf16_b4_h16_t2048_k128_v128", 4, 2048, 16, 128, 128, "bf16", seed=1),
        Workload("bf16_b1_h32_t32768_k128_v128_h0", 1, 32768, 32, 128, 128, "bf16", seed=2,
                 h0_std=0.1),
        Workload("bf16_b8_h64_t8192_k128_v128", 8, 8192, 64, 128, 128, "bf16", seed=3),
        Workload("bf16_b2_h32_t16384_k128_v256_weakdecay", 2, 16384, 32, 128, 256, "bf16",
                 seed=4, g_mean=4.0, g_div=64.0, beta_mean=2.0),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)
DECODE_WORKLOADS = {
    w.name: w
    for w in [
        Workload("bf16_b256_h16_t1_k128_v128_decode", 256, 1, 16, 128, 128, "bf16", seed=11,
                 h0_std=0.1),
    ]
}
# the largest single-GPU workload is the benchmark's headline; the feature
# measurements (front-end, output stage, per-channel decay) run on the short batch
BENCH_WORKLOAD = "bf16_b8_h64_t8192_k128_v128"
FEATURE_WORKLOAD = "bf16_b4_h16_t2048_k128_v128"

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def chunk_local_cumsum(x: torch.Tensor, chunk: int = CHUNK) -> torch.Tensor:
    """Cumulative sum over dim 1 (time) restarted at every ``chunk`` tokens."""
    B, T = x.shape[:2]
    NT = (T + chunk - 1) // chunk
    pad = torch.zeros((B, NT * chunk - T) + tuple(x.shape[2:]), dtype=x.dtype)
    xp = torch.cat([x, pad], dim=1).reshape((B, NT, chunk) + tuple(x.shape[2:]))
    return torch.cumsum(xp, dim=2).reshape((B, NT * chunk) + tuple(x.shape[2:]))[:, :T].contiguous()


def make_inputs(B: int, T: int, H: int, K: int, V: int, *, dtype: str = "bf16", seed: int = 0,
                h0_std: float = 0.0, g_mean: float = 0.0, g_div: float = 16.0,
                beta_mean: float = 0.0, chunk: int = CHUNK, raw: bool = False,
                per_channel: bool = False) -> dict:
    """Return CPU tensors q,k,v (dtype), g, beta (fp32) and h0 (fp32 or None).
    g is the per-token log-decay summed within chunks of ``chunk`` tokens;
    ``raw`` skips the q/k normalisation and the sum (same draws);
    ``per_channel`` draws one decay per key channel (g [B,T,H,K])."""
    gen = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, T, H, K, generator=gen)
    k = torch.randn(B, T, H, K, generator=gen)
    v = torch.randn(B, T, H, V, generator=gen)
    beta_raw = torch.randn(B, T, H, generator=gen)
    g_raw = torch.randn((B, T, H, K) if per_channel else (B, T, H), generator=gen)
    h0 = None
    if h0_std > 0:
        h0 = torch.randn(B, H, K, V, generator=gen) * h0_std
    if not raw:
        q = q / q.norm(dim=-1, keepdim=True) * (K ** -0.5)
        k = k / k.norm(dim=-1, keepdim=True)
    beta = torch.sigmoid(beta_raw + beta_mean)
    g = F.logsigmoid(g_raw + g_mean) / g_div
    if not raw:
        g = chunk_local_cumsum(g, chunk)
    td = TORCH_DTYPE[dtype]
    return {
        "q": q.to(td).contiguous(),
        "k": k.to(td).contiguous(),
        "v": v.to(td).contiguous(),
        "g": g.contiguous(),
        "beta": beta.contiguous(),
        "h0": None if h0 is None else h0.contiguous(),
        "scale": 1.0,
    }


def make_output_norm(B: int, T: int, H: int, V: int, *, dtype: str = "bf16", seed: int = 0):
    """Gate [B,T,H,V] ~ N(0,1) in the I/O dtype and norm weight [V] ~ 1 + 0.1 N(0,1)
    fp32, the extra inputs of the gated RMSNorm output stage (own generator)."""
    gen = torch.Generator("cpu").manual_seed(seed + 7919)
    gate = torch.randn(B, T, H, V, generator=gen).to(TORCH_DTYPE[dtype]).contiguous()
    weight = (1.0 + 0.1 * torch.randn(V, generator=gen)).contiguous()
    return gate, weight


def make_workload(name, **overrides) -> dict:
    """Inputs of a workload (a name, or a Workload such as a slice of a named
    one); ``overrides`` may change B/T/H (e.g. a sample)."""
    if isinstance(name, Workload):
        w, name = name, name.name
    else:
        w = WORKLOADS[name] if name in WORKLOADS else DECODE_WORKLOADS[name]
    p = w.as_dict()
    p.update(overrides)
    return make_inputs(p["B"], p["T"], p["H"], p["K"], p["V"], dtype=p["dtype"], seed=p["seed"],
                       h0_std=p["h0_std"], g_mean=p["g_mean"], g_div=p["g_div"],
                       beta_mean=p["beta_mean"], chunk=1 if name in DECODE_WORKLOADS else CHUNK)


def to_f64(t):
    """Exact fp64 numpy copy of a CPU tensor (bf16/fp32 widen exactly), or None."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
