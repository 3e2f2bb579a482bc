"""ctypes binding of ``libgdn.so`` (include/gdn.h): argument marshalling only.

Every step of the forward runs in the library's CUDA kernels; PyTorch only
allocates device memory and supplies the current stream. There is no CPU or
PyTorch fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "lib" / "libgdn.so"

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_ALIGNMENT = 0, 1, 2, 3
GDN_ERR_WORKSPACE, GDN_ERR_CUDA, GDN_ERR_DEVICE_TIMEOUT = 4, 5, 6
GDN_F32, GDN_BF16 = 0, 1
GDN_FLAG_RAW_G, GDN_FLAG_QK_L2NORM, GDN_FLAG_PER_CHANNEL_DECAY = 1, 2, 4
ALGOS = {"auto": 0, "simt": 1, "tc": 2, "tc1": 3, "tcw": 4}
DTYPES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}
CHUNK = 64

# Every function include/gdn.h declares.
EXPORTS = ("gdn_chunk_fwd_workspace_bytes", "gdn_chunk_fwd", "gdn_chunk_fwd_stages",
           "gdn_chunk_fwd_launches", "gdn_chunk_fwd_profiled", "gdn_check_device_status",
           "gdn_chunk_fwd_noalloc", "gdn_decode_step", "gdn_decode_step_launches",
           "gdn_chunk_fwd_ex", "gdn_decode_step_ex", "gdn_chunk_fwd_host_bytes",
           "gdn_chunk_fwd_host", "gdn_debug_arm_stall", "gdn_status_string", "gdn_version")


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("K", ctypes.c_int32), ("V", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("algo", ctypes.c_int32), ("flags", ctypes.c_int32)]


class OutputNorm(ctypes.Structure):
    """gdn_output_norm: gated RMSNorm of the output rows."""
    _fields_ = [("gate", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("eps", ctypes.c_float)]


class StageExports(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("w", ctypes.c_void_p), ("u", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("h", ctypes.c_void_p), ("A_beta", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(str(LIB_PATH))
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        pp = ctypes.POINTER(Problem)
        L.gdn_chunk_fwd_workspace_bytes.restype = sz
        L.gdn_chunk_fwd_workspace_bytes.argtypes = [pp]
        fwd_args = [pp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, sz]
        L.gdn_chunk_fwd.restype = ctypes.c_int
        L.gdn_chunk_fwd.argtypes = fwd_args + [vp]
        L.gdn_chunk_fwd_stages.restype = ctypes.c_int
        L.gdn_chunk_fwd_stages.argtypes = fwd_args + [ctypes.POINTER(StageExports), vp]
        L.gdn_chunk_fwd_launches.restype = ctypes.c_int32
        L.gdn_chunk_fwd_launches.argtypes = [pp, ctypes.POINTER(ctypes.c_char_p), ctypes.c_int32]
        L.gdn_chunk_fwd_profiled.restype = ctypes.c_int
        L.gdn_chunk_fwd_profiled.argtypes = fwd_args + [ctypes.POINTER(ctypes.c_void_p),
                                                        ctypes.c_int32, vp]
        L.gdn_check_device_status.restype = ctypes.c_int
        L.gdn_check_device_status.argtypes = [vp, vp]
        L.gdn_chunk_fwd_ex.restype = ctypes.c_int
        L.gdn_chunk_fwd_ex.argtypes = [pp, vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                       ctypes.POINTER(OutputNorm), vp, vp, vp, sz,
                                       ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32, vp]
        L.gdn_decode_step_ex.restype = ctypes.c_int
        L.gdn_decode_step_ex.argtypes = [pp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                         ctypes.POINTER(OutputNorm), vp, vp]
        L.gdn_chunk_fwd_host_bytes.restype = sz
        L.gdn_chunk_fwd_host_bytes.argtypes = [pp, ctypes.c_int32]
        L.gdn_chunk_fwd_host.restype = ctypes.c_int
        L.gdn_chunk_fwd_host.argtypes = [pp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, sz,
                                         ctypes.c_int32, vp, vp]
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [pp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
        L.gdn_decode_step_launches.restype = ctypes.c_int32
        L.gdn_decode_step_launches.argtypes = [pp, ctypes.POINTER(ctypes.c_char_p),
                                               ctypes.c_int32]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_version.restype = ctypes.c_uint32
        L.gdn_version.argtypes = []
        L.gdn_debug_arm_stall.restype = None
        L.gdn_debug_arm_stall.argtypes = [ctypes.c_uint64]
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().gdn_status_string(int(s)).decode()


def flags_of(raw_g: bool = False, qk_l2norm: bool = False, per_channel: bool = False) -> int:
    return ((GDN_FLAG_RAW_G if raw_g else 0) | (GDN_FLAG_QK_L2NORM if qk_l2norm else 0)
            | (GDN_FLAG_PER_CHANNEL_DECAY if per_channel else 0))


def problem(B, T, H, K, V, dtype, algo="auto", flags: int = 0) -> Problem:
    d = DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return Problem(int(B), int(T), int(H), int(K), int(V), d,
                   ALGOS[algo] if isinstance(algo, str) else int(algo), int(flags))


def workspace_bytes(p: Problem) -> int:
    return int(lib().gdn_chunk_fwd_workspace_bytes(ctypes.byref(p)))


def launches(p: Problem) -> list[str]:
    """Names of the kernels one call launches, in order."""
    n = int(lib().gdn_chunk_fwd_launches(ctypes.byref(p), None, 0))
    names = (ctypes.c_char_p * max(n, 1))()
    lib().gdn_chunk_fwd_launches(ctypes.byref(p), names, n)
    return [names[i].decode() for i in range(n)]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_inputs(q, k, v, g, beta, h0, per_channel: bool = False):
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors (use chunk_fwd_host for host tensors)")
    if q.dtype not in DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float32 or bfloat16")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    g_shape = (B, T, H, K) if per_channel else (B, T, H)
    if k.shape != (B, T, H, K) or v.shape[:3] != (B, T, H) or g.shape != g_shape \
            or beta.shape != (B, T, H):
        raise ValueError("shapes must be q,k [B,T,H,K], v [B,T,H,V], beta [B,T,H], g [B,T,H] "
                         "([B,T,H,K] with per-channel decay)")
    if h0 is not None and (h0.shape != (B, H, K, V) or h0.dtype != torch.float32):
        raise ValueError("h0 must be float32 [B,H,K,V]")
    for t in (q, k, v, g, beta, h0):
        if t is not None and (not t.is_contiguous() or t.device != dev):
            raise ValueError("all tensors must be contiguous and on the same device")
    return B, T, H, K, V


def _given(t, shape, dtype, dev, name):
    """A caller-supplied output buffer, checked against what the kernels write
    into it: the library knows only the problem's sizes, so a smaller or
    strided buffer would be written past its end."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != dev or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor {tuple(shape)} on {dev}")
    return t


def _workspace(ws, need: int, dev):
    """A caller-supplied workspace must be a contiguous uint8 tensor on the
    inputs' device holding at least ``need`` bytes: the kernels and a later
    check_device_status read the status word in that very buffer, so a
    too-small one is an error rather than silently replaced. None: a fresh
    one is allocated."""
    if ws is None:
        return torch.empty(need, dtype=torch.uint8, device=dev)
    if ws.dtype != torch.uint8 or ws.device != dev or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    if ws.numel() < need:
        raise ValueError(f"workspace holds {ws.numel()} bytes; this problem needs {need}")
    return ws


def _output_norm(gate, weight, eps, shape, like):
    if gate is None and weight is None:
        return None
    if gate is None or weight is None:
        raise ValueError("the output stage needs both gate and norm_weight")
    if gate.shape != shape or gate.dtype != like.dtype or not gate.is_contiguous() \
            or gate.device != like.device:
        raise ValueError(f"gate must be contiguous {tuple(shape)} in the input dtype")
    if weight.shape != (shape[-1],) or weight.dtype != torch.float32 or not weight.is_contiguous() \
            or weight.device != like.device:
        raise ValueError("norm_weight must be contiguous float32 [V]")
    return OutputNorm(ctypes.c_void_p(gate.data_ptr()), ctypes.c_void_p(weight.data_ptr()),
                      float(eps))


def chunk_fwd(q, k, v, g, beta, scale: float = 1.0, h0=None, output_final_state: bool = True,
              algo: str = "auto", workspace=None, out=None, final_state=None, stream=None,
              events=None, raw_g: bool = False, qk_l2norm: bool = False, gate=None,
              norm_weight=None, norm_eps: float = 1e-6, per_channel_decay: bool = False):
    """Chunked gated-delta-rule forward on CUDA tensors. Returns (o, h_final or None).

    q, k [B,T,H,K] and v [B,T,H,V] (float32 or bfloat16), g and beta [B,T,H]
    float32 (g: chunk-local cumulative log-decay), h0 [B,H,K,V] float32 or None.
    ``workspace``/``out``/``final_state`` may be passed to reuse buffers.
    ``raw_g``: g holds per-token log decays, summed per chunk in the kernels;
    ``qk_l2norm``: q and k rows are L2-normalised in the kernels (eps 1e-6).
    ``gate`` [B,T,H,V] (q's dtype) with ``norm_weight`` [V] float32: the output
    rows pass through the gated RMSNorm o * rsqrt(mean o^2 + norm_eps) *
    norm_weight * sigmoid(gate) before their rounding.
    ``per_channel_decay``: g is [B,T,H,K], one decay per key channel (the KDA
    variant; bf16 runs on its own tensor-core form, fp32 on the CUDA-core
    pipeline)."""
    B, T, H, K, V = _check_inputs(q, k, v, g, beta, h0, per_channel_decay)
    norm = _output_norm(gate, norm_weight, norm_eps, (B, T, H, V), q)
    p = problem(B, T, H, K, V, q.dtype, algo, flags_of(raw_g, qk_l2norm, per_channel_decay))
    need = workspace_bytes(p)
    if need == 0:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_chunk_fwd_workspace_bytes")
    workspace = _workspace(workspace, need, q.device)
    o = _given(out, (B, T, H, V), q.dtype, q.device, "out") if out is not None else \
        torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    hf = None
    if output_final_state:
        hf = _given(final_state, (B, H, K, V), torch.float32, q.device, "final_state") \
            if final_state is not None else \
            torch.empty((B, H, K, V), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    args = (ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
            _ptr(h0), _ptr(o), _ptr(hf), _ptr(workspace), workspace.numel())
    if norm is not None:
        arr = None if events is None else (ctypes.c_void_p * len(events))(*events)
        st = lib().gdn_chunk_fwd_ex(*args[:8], ctypes.byref(norm), *args[8:], arr,
                                    0 if events is None else len(events),
                                    ctypes.c_void_p(s.cuda_stream))
    elif events is None:
        st = lib().gdn_chunk_fwd(*args, ctypes.c_void_p(s.cuda_stream))
    else:
        # events: raw cudaEvent_t handles (ints); markers between the kernels
        arr = (ctypes.c_void_p * len(events))(*events)
        st = lib().gdn_chunk_fwd_profiled(*args, arr, len(events), ctypes.c_void_p(s.cuda_stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd")
    return o, hf


STAGES = ("A", "w", "u", "v_new", "h", "A_beta")


def chunk_fwd_stages(q, k, v, g, beta, scale: float = 1.0, h0=None, algo: str = "simt",
                     stages=("A", "w", "u", "v_new", "h"), raw_g: bool = False,
                     qk_l2norm: bool = False, per_channel_decay: bool = False):
    """Forward plus the requested exported intermediates (fp32 tensors): A, w, u,
    v_new, h (SIMT path) or A_beta = A diag(beta) (tensor-core path)."""
    B, T, H, K, V = _check_inputs(q, k, v, g, beta, h0, per_channel_decay)
    p = problem(B, T, H, K, V, q.dtype, algo, flags_of(raw_g, qk_l2norm, per_channel_decay))
    NT = (T + CHUNK - 1) // CHUNK
    Tp = NT * CHUNK
    f32 = dict(dtype=torch.float32, device=q.device)
    shapes = {"A": (B, Tp, H, CHUNK), "w": (B, Tp, H, K), "u": (B, Tp, H, V),
              "v_new": (B, Tp, H, V), "h": (B, NT, H, K, V), "A_beta": (B, Tp, H, CHUNK)}
    st_bufs = {n: torch.empty(shapes[n], **f32) for n in stages}
    ex = StageExports(*(ctypes.c_void_p(st_bufs[n].data_ptr()) if n in st_bufs else None
                        for n in STAGES))
    need = workspace_bytes(p)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    o = torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    hf = torch.empty((B, H, K, V), **f32)
    s = torch.cuda.current_stream(q.device)
    st = lib().gdn_chunk_fwd_stages(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(beta), float(scale), _ptr(h0), _ptr(o), _ptr(hf),
                                    _ptr(ws), ws.numel(), ctypes.byref(ex),
                                    ctypes.c_void_p(s.cuda_stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd_stages")
    st_bufs.update(o=o, h_final=hf)
    return st_bufs


def decode_step(q, k, v, gamma, beta, state, scale: float = 1.0, state_out=None, out=None,
                stream=None, qk_l2norm: bool = False, gate=None, norm_weight=None,
                norm_eps: float = 1e-6, per_channel_decay: bool = False):
    """Recurrent step(s) of the rule on CUDA tensors: advances every sequence by
    its T tokens and returns (o, state_out).

    q, k [B,T,H,K] and v [B,T,H,V] (float32 or bfloat16); gamma, beta [B,T,H]
    float32, gamma the per-token log decay itself (not a cumulative sum);
    state [B,H,K,V] float32 (an h_final of chunk_fwd). ``state_out=None``
    updates ``state`` in place; pass ``state_out=state`` for the same, or
    another buffer to keep ``state``. ``qk_l2norm`` normalises the q and k
    rows in the kernel (eps 1e-6); ``gate``/``norm_weight`` add the output
    stage as in chunk_fwd."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float32 or bfloat16")
    if gamma.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("gamma and beta must be float32")
    g_shape = (B, T, H, K) if per_channel_decay else (B, T, H)
    if k.shape != (B, T, H, K) or v.shape[:3] != (B, T, H) or gamma.shape != g_shape \
            or beta.shape != (B, T, H):
        raise ValueError("shapes must be q,k [B,T,H,K], v [B,T,H,V], beta [B,T,H], gamma "
                         "[B,T,H] ([B,T,H,K] with per-channel decay)")
    so = state if state_out is None else state_out
    for st in (state, so):
        if st.shape != (B, H, K, V) or st.dtype != torch.float32:
            raise ValueError("state must be float32 [B,H,K,V]")
    for t in (q, k, v, gamma, beta, state, so):
        if not t.is_contiguous() or t.device != dev:
            raise ValueError("all tensors must be contiguous and on the same device")
    o = _given(out, (B, T, H, V), q.dtype, dev, "out") if out is not None else \
        torch.empty((B, T, H, V), dtype=q.dtype, device=dev)
    p = problem(B, T, H, K, V, q.dtype, "auto", flags_of(False, qk_l2norm, per_channel_decay))
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    norm = _output_norm(gate, norm_weight, norm_eps, (B, T, H, V), q)
    st = lib().gdn_decode_step_ex(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                  _ptr(beta), float(scale), _ptr(state), _ptr(so),
                                  None if norm is None else ctypes.byref(norm), _ptr(o),
                                  ctypes.c_void_p(s.cuda_stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_step")
    return o, so


def decode_launches(p: Problem) -> list[str]:
    """Names of the kernels one decode_step call launches."""
    names = (ctypes.c_char_p * 1)()
    n = int(lib().gdn_decode_step_launches(ctypes.byref(p), names, 1))
    return [names[i].decode() for i in range(n)]


def debug_arm_stall(wait_ns: int) -> None:
    """Test hook: the next tensor-core launch withholds its first chunk's loads,
    so its bounded waits give up after ``wait_ns`` and it reports a device
    timeout through check_device_status (gdn_debug_arm_stall)."""
    lib().gdn_debug_arm_stall(int(wait_ns))


def check_device_status(workspace, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    return int(lib().gdn_check_device_status(_ptr(workspace), ctypes.c_void_p(s.cuda_stream)))


_host_streams: dict = {}
_host_buffers: dict = {}
_host_plans: dict = {}
_host_events: dict = {}
_host_lock = threading.Lock()


def _pipeline_streams(dev, n: int):
    """n side streams of ``dev``, created once and reused by every host call."""
    key = (dev.index, n)
    if key not in _host_streams:
        _host_streams[key] = [torch.cuda.Stream(dev) for _ in range(n)]
    return _host_streams[key]


def _host_plan(B, T, H, K, V, dtype, algo, flags, pieces):
    """(problem, device bytes) of one host call, computed once per shape."""
    key = (B, T, H, K, V, dtype, algo, flags, pieces)
    plan = _host_plans.get(key)
    if plan is None:
        p = problem(B, T, H, K, V, dtype, algo, flags)
        need = int(lib().gdn_chunk_fwd_host_bytes(ctypes.byref(p), int(pieces)))
        if need == 0:
            raise GdnError(GDN_ERR_INVALID_ARG, "gdn_chunk_fwd_host_bytes")
        if len(_host_plans) > 64:
            _host_plans.clear()
        plan = _host_plans[key] = (p, need)
    return plan


def _host_buffer(dev, need: int):
    """The device buffer of the host calls on ``dev``, grown on demand and kept:
    every call has finished with it when it returns."""
    buf = _host_buffers.get(dev.index)
    if buf is None or buf.numel() < need:
        _host_buffers[dev.index] = None
        buf = _host_buffers[dev.index] = torch.empty(need, dtype=torch.uint8, device=dev)
    return buf


def _host_out(t, shape, dtype, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    if t.device.type != "cpu" or not t.is_contiguous() or tuple(t.shape) != shape or t.dtype != dtype:
        raise ValueError(f"{name} must be a contiguous host tensor {shape} of {dtype}")
    return t


def chunk_fwd_host(q, k, v, g, beta, scale: float = 1.0, h0=None, output_final_state: bool = True,
                   algo: str = "auto", device=None, raw_g: bool = False, qk_l2norm: bool = False,
                   pieces: int = 0, out=None, final_state=None, per_channel_decay: bool = False):
    """Host-tensor front end (gdn_chunk_fwd_host): host inputs in, host outputs
    out; returns when o (and h_final) are in host tensors. Pinned inputs let the
    library overlap the copies of one span of T (up to ``pieces`` 64-aligned
    spans; 0: the library's choice) with the kernels of the previous one.
    ``out`` / ``final_state``:
    host tensors [B, T, H, V] / [B, H, K, V] fp32 to write into (pinned ones
    allocated when None). torch supplies the device buffer and the two side
    streams, both kept per device for later calls; a lock serialises callers,
    and the work waits for what the caller's current stream has queued.
    ``per_channel_decay``: g is [B,T,H,K] (as for chunk_fwd)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    B, T, H, K = q.shape
    V = v.shape[-1]
    for t in (q, k, v, g, beta, h0):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError("chunk_fwd_host takes contiguous host tensors")
    if q.dtype not in DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float32 or bfloat16")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    g_shape = (B, T, H, K) if per_channel_decay else (B, T, H)
    if tuple(g.shape) != g_shape or tuple(beta.shape) != (B, T, H):
        raise ValueError(f"g must be {g_shape} and beta {(B, T, H)}")
    p, need = _host_plan(B, T, H, K, V, q.dtype, algo, flags_of(raw_g, qk_l2norm, per_channel_decay), pieces)
    ho = _host_out(out, (B, T, H, V), q.dtype, "out")
    hhf = _host_out(final_state, (B, H, K, V), torch.float32, "final_state") \
        if output_final_state else None
    with _host_lock, torch.cuda.device(dev):
        buf = _host_buffer(dev, need)
        sa, sb = _pipeline_streams(dev, 2)
        ready = _host_events.get(dev.index)
        if ready is None:
            ready = _host_events[dev.index] = torch.cuda.Event()
        ready.record(torch.cuda.current_stream(dev))
        sa.wait_event(ready)
        sb.wait_event(ready)
        st = lib().gdn_chunk_fwd_host(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      _ptr(beta), float(scale), _ptr(h0), _ptr(ho), _ptr(hhf),
                                      _ptr(buf), need, int(pieces),
                                      ctypes.c_void_p(sa.cuda_stream),
                                      ctypes.c_void_p(sb.cuda_stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd_host")
    return ho, hhf


def chunk_fwd_noalloc(q, k, v, g, beta, scale: float = 1.0, h0=None, out=None, final_state=None,
                      stream=None):
    """gdn_chunk_fwd_noalloc: the forward with the library's fixed device scratch
    instead of a workspace, for callers that cannot allocate device memory. The
    caller passes preallocated ``out`` [B,T,H,V] and ``final_state`` [B,H,K,V]
    (or None to skip h_final); without ``out`` this wrapper allocates it."""
    B, T, H, K, V = _check_inputs(q, k, v, g, beta, h0)
    L = lib()
    f = L.gdn_chunk_fwd_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
    p = problem(B, T, H, K, V, q.dtype, "simt")
    o = _given(out, (B, T, H, V), q.dtype, q.device, "out") if out is not None else \
        torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    if final_state is not None:
        _given(final_state, (B, H, K, V), torch.float32, q.device, "final_state")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    # the library finds its scratch on the current device: make it the inputs'
    with torch.cuda.device(q.device):
        st = f(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
               _ptr(h0), _ptr(o), _ptr(final_state), ctypes.c_void_p(s.cuda_stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd_noalloc")
    return o, final_state
