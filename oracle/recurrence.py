"""ctypes front of the fp64 token-recurrence oracle (``gdn_ref.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline leg, never by the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "gdn_ref.c"
LIB_DIR = HERE / "lib"
LIB = LIB_DIR / "libgdn_oracle.so"

_lib = None


def build(force: bool = False, src: Path = SRC, out: Path = LIB) -> Path:
    """Compile the oracle with the host C compiler (portable flags only)."""
    if out.exists() and not force and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    subprocess.run(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-pthread",
                    str(src), "-o", str(tmp), "-lm"], check=True)
    os.replace(tmp, out)
    return out


def load(path: Path | None = None):
    """Load (building first if needed) and return the oracle's ctypes handle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(build())))
    return _lib


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gdn_oracle_forward_pc.restype = ctypes.c_int
    lib.gdn_oracle_forward_pc.argtypes = [ctypes.c_int] * 7 + [dp] * 5 + [ctypes.c_double] + \
        [dp] * 5 + [ctypes.c_int]
    return lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def default_threads() -> int:
    return os.cpu_count() or 1


def forward(q, k, v, g, beta, scale=1.0, h0=None, *, chunk: int = 64, nthreads: int | None = None,
            lib=None, stages: bool = False):
    """Token-by-token fp64 recurrence. Arrays in [B,T,H,*] layout; returns (o, h_final),
    or with ``stages`` (o, h_final, h_chunks [B,NT,H,K,V], delta [B,T,H,V]).
    g [B,T,H] is the scalar decay; g [B,T,H,K] is the per-channel (KDA) decay."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, K = q.shape
    V = v.shape[-1]
    per_channel = g.ndim == 4
    assert k.shape == (B, T, H, K) and v.shape == (B, T, H, V)
    assert g.shape == ((B, T, H, K) if per_channel else (B, T, H)) and beta.shape == (B, T, H)
    assert h0 is None or h0.shape == (B, H, K, V)
    o = np.zeros((B, T, H, V))
    hf = np.zeros((B, H, K, V))
    hc = dl = None
    if stages:
        hc = np.zeros((B, (T + chunk - 1) // chunk, H, K, V))
        dl = np.zeros((B, T, H, V))
    lib = lib or load()
    rc = lib.gdn_oracle_forward_pc(B, T, H, K, V, chunk, int(per_channel), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g),
                                   _ptr(beta), float(scale), _ptr(h0), _ptr(o), _ptr(hf),
                                   _ptr(hc), _ptr(dl), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_forward failed with code {rc}")
    if stages:
        return o, hf, hc, dl
    return o, hf
