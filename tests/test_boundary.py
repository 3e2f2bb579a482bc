"""The C-ABI library on the CPU: it loads, exports every function include/gdn.h
declares, sizes its workspace and rejects bad arguments before touching CUDA."""
import ctypes
import re
from pathlib import Path

import pytest

from gated_delta_rule_35_gb300 import native

HEADER = Path(__file__).resolve().parents[1] / "include" / "gdn.h"
FAKE = 0x10000   # an aligned non-NULL address; never dereferenced by validation


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and len(names) >= 5
    lib = native.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(native.EXPORTS) >= set(names)


def test_version_and_status_strings():
    assert native.lib().gdn_version() > 0
    for s in range(7):
        assert native.status_string(s)
    assert native.status_string(99) == "unknown status"


def _call(p, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, o=FAKE, hf=None, ws=FAKE,
          ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = 0
    vp = ctypes.c_void_p
    return native.lib().gdn_chunk_fwd(ctypes.byref(p) if p is not None else None, vp(q), vp(k),
                                      vp(v), vp(g), vp(beta), 1.0, vp(h0), vp(o), vp(hf), vp(ws),
                                      ws_bytes, None)


def test_workspace_bytes():
    p = native.problem(4, 2048, 16, 128, 128, native.GDN_BF16, "simt")
    n = native.workspace_bytes(p)
    # fp32 A, w, u, v_new, per-chunk h, plus the status word
    rows = 4 * 2048 * 16
    assert n >= rows * (64 + 128 + 128 + 128) * 4 + 4 * 32 * 16 * 128 * 128 * 4
    assert native.workspace_bytes(native.problem(4, 2048, 16, 96, 128, 1)) == 0   # K unsupported
    assert native.workspace_bytes(native.problem(1, 0, 1, 64, 64, 0)) > 0          # T = 0 valid



def test_host_entry_span_count():
    """gdn_chunk_fwd_host_bytes: 1..16 spans, or 0 for the library's choice of
    about one span per 32 MiB of inputs (3 to 16). The buffer holds one span's
    workspace, so its size tells the span count apart."""
    L = native.lib()

    def host_bytes(p, pieces):
        return int(L.gdn_chunk_fwd_host_bytes(ctypes.byref(p), pieces))

    short = native.problem(4, 2048, 16, 128, 128, native.GDN_BF16)    # 102 MB of inputs
    long = native.problem(1, 32768, 32, 128, 128, native.GDN_BF16)    # 814 MB
    tiny = native.problem(1, 640, 1, 64, 64, native.GDN_BF16)         # 0.2 MB
    assert host_bytes(short, 0) == host_bytes(short, 3) != host_bytes(short, 4)
    assert host_bytes(long, 0) == host_bytes(long, 16) != host_bytes(long, 8)
    assert host_bytes(tiny, 0) == host_bytes(tiny, 3) != host_bytes(tiny, 1)
    for bad in (-1, 17):
        assert host_bytes(short, bad) == 0
    # one span's workspace at most: the buffer shrinks as the span count grows
    assert host_bytes(long, 1) > host_bytes(long, 4) > host_bytes(long, 16)

@pytest.mark.parametrize("shape,status", [
    ((0, 64, 1, 64, 64), native.GDN_ERR_INVALID_ARG),
    ((1, -1, 1, 64, 64), native.GDN_ERR_INVALID_ARG),
    ((1, 64, 0, 64, 64), native.GDN_ERR_INVALID_ARG),
    ((1, 64, 1, 32, 64), native.GDN_ERR_UNSUPPORTED),
    ((1, 64, 1, 64, 96), native.GDN_ERR_UNSUPPORTED),
    ((1, 64, 1, 64, 320), native.GDN_ERR_UNSUPPORTED),
])
def test_rejects_bad_shapes(shape, status):
    assert _call(native.problem(*shape, native.GDN_F32, "simt")) == status


def test_rejects_bad_enums_and_null():
    assert _call(None) == native.GDN_ERR_INVALID_ARG
    p = native.Problem(1, 64, 1, 64, 64, 7, 0)
    assert _call(p) == native.GDN_ERR_INVALID_ARG
    p = native.Problem(1, 64, 1, 64, 64, 0, 9)
    assert _call(p) == native.GDN_ERR_INVALID_ARG
    p = native.problem(1, 64, 1, 64, 64, native.GDN_F32, "simt")
    for field in ("q", "k", "v", "g", "beta", "o"):
        assert _call(p, **{field: None}) == native.GDN_ERR_INVALID_ARG, field


def test_rejects_misaligned_pointers():
    p = native.problem(1, 64, 1, 64, 64, native.GDN_F32, "simt")
    for field in ("q", "k", "v", "g", "beta", "o", "h0", "hf", "ws"):
        assert _call(p, **{field: FAKE + 4}) == native.GDN_ERR_ALIGNMENT, field


def test_rejects_small_workspace():
    p = native.problem(2, 100, 3, 64, 64, native.GDN_BF16, "simt")
    need = native.workspace_bytes(p)
    assert _call(p, ws_bytes=need - 1) == native.GDN_ERR_WORKSPACE
    assert _call(p, ws=None, ws_bytes=need) == native.GDN_ERR_WORKSPACE


def test_stage_export_needs_exports():
    p = native.problem(1, 64, 1, 64, 64, native.GDN_F32, "simt")
    vp = ctypes.c_void_p
    st = native.lib().gdn_chunk_fwd_stages(ctypes.byref(p), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                           vp(FAKE), 1.0, None, vp(FAKE), None, vp(FAKE), 1 << 30,
                                           None, None)
    assert st == native.GDN_ERR_INVALID_ARG
    assert native.lib().gdn_check_device_status(None, None) == native.GDN_ERR_INVALID_ARG


def _decode(p, q=FAKE, k=FAKE, v=FAKE, gamma=FAKE, beta=FAKE, s_in=FAKE, s_out=FAKE, o=FAKE):
    vp = ctypes.c_void_p
    return native.lib().gdn_decode_step(ctypes.byref(p) if p is not None else None, vp(q),
                                        vp(k), vp(v), vp(gamma), vp(beta), 1.0, vp(s_in),
                                        vp(s_out), vp(o), None)


@pytest.mark.parametrize("shape,algo,status", [
    ((0, 1, 1, 64, 64), "auto", native.GDN_ERR_INVALID_ARG),
    ((1, -1, 1, 64, 64), "auto", native.GDN_ERR_INVALID_ARG),
    ((1, 1, 1, 96, 64), "auto", native.GDN_ERR_UNSUPPORTED),    # K not a multiple of 64
    ((1, 1, 1, 320, 64), "auto", native.GDN_ERR_UNSUPPORTED),   # K > 256
    ((1, 1, 1, 64, 24), "auto", native.GDN_ERR_UNSUPPORTED),    # V not a multiple of 16
    ((1, 1, 1, 64, 8192), "auto", native.GDN_ERR_UNSUPPORTED),  # V > 4096
    ((1, 1, 1, 64, 64), "tc", native.GDN_ERR_UNSUPPORTED),      # no tensor-core decode
    ((1, 1, 1, 64, 64), "tc1", native.GDN_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_problems(shape, algo, status):
    assert _decode(native.problem(*shape, native.GDN_BF16, algo)) == status


def test_decode_rejects_null_misaligned_and_overlapping():
    p = native.problem(2, 1, 3, 128, 128, native.GDN_BF16, "auto")
    assert _decode(None) == native.GDN_ERR_INVALID_ARG
    for field in ("q", "k", "v", "gamma", "beta", "s_in", "s_out", "o"):
        assert _decode(p, **{field: None}) == native.GDN_ERR_INVALID_ARG, field
        assert _decode(p, **{field: FAKE + 4}) == native.GDN_ERR_ALIGNMENT, field
    # the state is 2*3*128*128*4 bytes; an output starting inside it overlaps
    assert _decode(p, s_out=FAKE + 4096) == native.GDN_ERR_INVALID_ARG
    assert _decode(p, s_in=FAKE + 4096) == native.GDN_ERR_INVALID_ARG


def test_decode_launches():
    assert native.decode_launches(native.problem(4, 1, 16, 128, 128, native.GDN_BF16)) == \
        ["gdn_decode_step_kernel"]
    assert native.decode_launches(native.problem(4, 0, 16, 128, 128, native.GDN_BF16)) == []
    assert native.decode_launches(native.problem(4, 1, 16, 96, 128, native.GDN_BF16)) == []


def test_single_kernel_form_sizes_and_limits():
    """GDN_ALGO_TC_SINGLE keeps A on chip: its workspace holds only the status
    word and the front-end tables; it launches one kernel; per-channel decay,
    an output stage and the A export are refused before anything runs."""
    two = native.problem(4, 2048, 16, 128, 128, native.GDN_BF16, "tc")
    one = native.problem(4, 2048, 16, 128, 128, native.GDN_BF16, "tc1")
    rows = 4 * 2048 * 16
    assert native.workspace_bytes(two) >= rows * 128 * 2
    assert 0 < native.workspace_bytes(one) < rows * 16
    assert native.launches(one) == ["gdn_fused_tc_kernel"]
    assert native.launches(two) == ["gdn_wy_tc_kernel", "gdn_fused_tc_kernel"]
    assert native.launches(native.problem(4, 2048, 16, 128, 128, native.GDN_BF16)) == native.launches(two)
    # more 64-column tiles than SMs: the 128-column forward kernel (without a
    # visible device the SM count is GB300's 152); B8 H64: three whole waves of
    # it (456 heads), the other 56 heads on the 64-column kernel (112 CTAs)
    wide = native.problem(2, 8192, 32, 128, 256, native.GDN_BF16)
    assert native.launches(wide) == ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel"]
    split = native.problem(8, 8192, 64, 128, 128, native.GDN_BF16)
    assert native.launches(split) == ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel", "gdn_fused_tc_kernel"]
    assert native.launches(native.problem(8, 8192, 64, 128, 128, native.GDN_BF16, "tcw")) == native.launches(wide)
    assert native.launches(native.problem(1, 64, 1, 128, 256, native.GDN_BF16, "tcw")) == native.launches(wide)
    assert native.workspace_bytes(native.problem(1, 64, 1, 128, 256, native.GDN_BF16, "tcw")) == \
        native.workspace_bytes(native.problem(1, 64, 1, 128, 256, native.GDN_BF16, "tc"))
    assert native.workspace_bytes(native.problem(1, 64, 1, 128, 192, native.GDN_BF16, "tcw")) == 0
    kda = native.problem(1, 64, 1, 128, 128, native.GDN_BF16, "tc1", native.GDN_FLAG_PER_CHANNEL_DECAY)
    assert native.workspace_bytes(kda) == 0
    assert native.workspace_bytes(native.problem(1, 64, 1, 128, 128, native.GDN_F32, "tc1")) == 0
    p = native.problem(1, 64, 1, 64, 64, native.GDN_BF16, "tc1")
    norm = native.OutputNorm(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1e-6)
    vp = ctypes.c_void_p
    st = native.lib().gdn_chunk_fwd_ex(ctypes.byref(p), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                       1.0, None, ctypes.byref(norm), vp(FAKE), None, vp(FAKE),
                                       native.workspace_bytes(p), None, 0, None)
    assert st == native.GDN_ERR_UNSUPPORTED
    ex = native.StageExports(None, None, None, None, None, vp(FAKE))
    st = native.lib().gdn_chunk_fwd_stages(ctypes.byref(p), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                           vp(FAKE), 1.0, None, vp(FAKE), None, vp(FAKE),
                                           native.workspace_bytes(p), ctypes.byref(ex), None)
    assert st == native.GDN_ERR_UNSUPPORTED
    # the forward kernels apply the output stage themselves: no workspace
    # beyond A diag(beta) | A'
    for V in (128, 256):
        assert native.workspace_bytes(native.problem(2, 100, 3, 128, V, native.GDN_BF16, "tcw")) == \
            native.workspace_bytes(native.problem(2, 100, 3, 128, 64, native.GDN_BF16, "tc"))


def test_flags_validated():
    """Known front-end bits are accepted by every path; unknown bits are rejected."""
    for algo in ("simt", "tc", "tc1", "tcw"):
        for flags in (1, 2, 3):
            p = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, algo, flags)
            assert native.workspace_bytes(p) > native.workspace_bytes(
                native.problem(2, 100, 3, 128, 128, native.GDN_BF16, algo)) - 1
    bad = native.problem(1, 64, 1, 64, 64, native.GDN_BF16, "auto", 8)
    assert native.workspace_bytes(bad) == 0
    assert _call(bad) == native.GDN_ERR_INVALID_ARG
    assert _decode(native.problem(1, 1, 1, 64, 64, native.GDN_BF16, "auto", 16)) == \
        native.GDN_ERR_INVALID_ARG


def test_output_norm_validated():
    p = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, "auto")
    vp = ctypes.c_void_p
    lib = native.lib()

    def fwd(norm):
        return lib.gdn_chunk_fwd_ex(ctypes.byref(p), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                    vp(FAKE), 1.0, None, ctypes.byref(norm), vp(FAKE), None,
                                    vp(FAKE), 1 << 40, None, 0, None)

    assert fwd(native.OutputNorm(None, FAKE, 1e-6)) == native.GDN_ERR_INVALID_ARG
    assert fwd(native.OutputNorm(FAKE, None, 1e-6)) == native.GDN_ERR_INVALID_ARG
    assert fwd(native.OutputNorm(FAKE, FAKE, -1.0)) == native.GDN_ERR_INVALID_ARG
    assert fwd(native.OutputNorm(FAKE + 8, FAKE, 1e-6)) == native.GDN_ERR_ALIGNMENT

    def dec(K, V, norm):
        q = native.problem(2, 1, 3, K, V, native.GDN_BF16, "auto")
        return lib.gdn_decode_step_ex(ctypes.byref(q), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                      vp(FAKE), 1.0, vp(FAKE), vp(FAKE), ctypes.byref(norm),
                                      vp(FAKE), None)

    ok = native.OutputNorm(FAKE, FAKE, 1e-6)
    assert dec(128, 48, ok) == native.GDN_ERR_UNSUPPORTED     # V not a slice width
    assert dec(256, 256, ok) == native.GDN_ERR_UNSUPPORTED    # K V > 32768
    assert dec(128, 128, native.OutputNorm(None, FAKE, 1e-6)) == native.GDN_ERR_INVALID_ARG


def test_per_channel_flag_routes():
    """Per-channel decay: bf16 on the tensor-core form of its own (two kernels),
    fp32 on the CUDA-core pipeline; 'auto' reserves room for both, since a call
    with the output stage or the stage exports runs on the CUDA-core pipeline."""
    flags = native.GDN_FLAG_PER_CHANNEL_DECAY
    p_tc = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, "tc", flags)
    p_auto = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, "auto", flags)
    p_simt = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, "simt", flags)
    assert 0 < native.workspace_bytes(p_tc) <= native.workspace_bytes(p_auto)
    assert native.workspace_bytes(p_auto) == max(native.workspace_bytes(p_tc), native.workspace_bytes(p_simt))
    kda = ["gdn_kda_prep_tc_kernel", "gdn_kda_fwd_tc_kernel"]
    assert native.launches(p_tc) == kda and native.launches(p_auto) == kda
    for form in ("tc1", "tcw"):
        assert native.workspace_bytes(native.problem(2, 100, 3, 128, 128, native.GDN_BF16, form, flags)) == 0
    p32 = native.problem(2, 100, 3, 128, 128, native.GDN_F32, "auto", flags)
    assert native.launches(p32) == ["wy_prepare_kernel", "chunk_h_kernel", "chunk_o_kernel"]
    # the front-end's g region holds one value per channel with this flag
    plain = native.problem(2, 100, 3, 128, 128, native.GDN_BF16, "simt")
    assert native.workspace_bytes(p_simt) - native.workspace_bytes(plain) >= 2 * 100 * 3 * 127 * 4 - 256
    # tensor-core workspace: [A diag(beta) | P A diag(beta)], [-w | Q'], KH (bf16), decays
    rows = 2 * 100 * 3
    body = native.workspace_bytes(p_tc) - native.workspace_bytes(native.problem(2, 0, 3, 128, 128, native.GDN_BF16, "tc", flags))
    assert body >= rows * (128 + 256 + 128) * 2 + 2 * 2 * 3 * 128 * 4


def test_host_binding_output_validation():
    """chunk_fwd_host's caller-owned outputs are checked on the host before any
    device work: shape, dtype, contiguity and host residency."""
    import torch
    good = torch.empty(2, 64, 3, 64, dtype=torch.bfloat16)
    assert native._host_out(good, (2, 64, 3, 64), torch.bfloat16, "out") is good
    for bad in (torch.empty(2, 64, 3, 32, dtype=torch.bfloat16),
                torch.empty(2, 64, 3, 64, dtype=torch.float32),
                torch.empty(2, 3, 64, 64, dtype=torch.bfloat16).transpose(1, 2)):
        with pytest.raises(ValueError):
            native._host_out(bad, (2, 64, 3, 64), torch.bfloat16, "out")


def test_device_output_buffers_are_checked():
    """chunk_fwd / decode_step accept caller-owned o, h_final and workspace only
    when the kernels cannot write past them: exact shape, dtype, device and a
    contiguous layout."""
    import torch
    cpu = torch.device("cpu")
    good = torch.empty(2, 64, 3, 64, dtype=torch.bfloat16)
    assert native._given(good, (2, 64, 3, 64), torch.bfloat16, cpu, "out") is good
    for bad in (torch.empty(2, 63, 3, 64, dtype=torch.bfloat16),
                torch.empty(2, 64, 3, 64, dtype=torch.float32),
                torch.empty(2, 3, 64, 64, dtype=torch.bfloat16).transpose(1, 2)):
        with pytest.raises(ValueError):
            native._given(bad, (2, 64, 3, 64), torch.bfloat16, cpu, "out")
    with pytest.raises(ValueError):
        native._given(good, (2, 64, 3, 64), torch.bfloat16, torch.device("meta"), "out")


def test_caller_workspace_is_checked_not_replaced():
    """A caller workspace that is too small (or of the wrong kind) raises: the
    kernels would otherwise use a fresh buffer while the caller later reads the
    status word of its own, stale one."""
    import torch
    cpu = torch.device("cpu")
    ws = torch.zeros(1024, dtype=torch.uint8)
    assert native._workspace(ws, 1024, cpu) is ws
    assert native._workspace(None, 512, cpu).numel() == 512
    with pytest.raises(ValueError):
        native._workspace(ws, 1025, cpu)
    for bad in (torch.zeros(1024, dtype=torch.int8), torch.zeros(2048, dtype=torch.uint8)[::2]):
        with pytest.raises(ValueError):
            native._workspace(bad, 16, cpu)
    with pytest.raises(ValueError):
        native._workspace(ws, 16, torch.device("meta"))
