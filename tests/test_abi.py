"""The C-ABI library loads and exports every symbol include/dts.h declares.

Runs without a GPU: only host-side entry points are called (version, status
text, workspace size, argument validation that fails before any launch).
"""
import ctypes
import os
import re

import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dts.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dts_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        B.build()
    return dts.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    assert set(names) == set(dts.EXPORTED)
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_host_only_calls(lib):
    assert dts.version() >= 100
    assert dts.status_string(0) == "ok"
    assert "workspace" in dts.status_string(dts.ERR_WORKSPACE)
    assert dts.device_error_string(dts.DEV_BAD_PARENT) == "bad parent index"
    # workspace: n_splits * B*N*Hq * (d + 1) fp32 words (each part 256-byte aligned)
    ws = dts.tree_verify_attention_workspace(32, 64, 32, 8, 128, 8192)
    rows = 32 * 64 * 32
    assert ws % 256 == 0 and ws >= rows * 129 * 4
    assert dts.tree_verify_attention_workspace(1, 5, 4, 1, 64, 0) > 0
    assert dts.tree_verify_attention_workspace(1, 5, 4, 3, 64, 10) == 0     # Hq % Hkv != 0


def test_validation_before_launch(lib):
    L = dts.lib()
    # N > 64 is unsupported; B = 0 launches nothing
    assert L.dts_build_tree_mask(None, None, None, 1, 65, None, None, None, None, None, None) == dts.ERR_UNSUPPORTED
    assert L.dts_build_tree_mask(None, None, None, 0, 8, None, None, None, None, None, None) == dts.OK
    assert L.dts_build_tree_mask(None, None, None, 2, 8, None, None, None, None, None, None) == dts.ERR_INVALID
    assert L.dts_verify_tree_greedy(None, None, None, None, None, 3, 8, None, None, None, None, None) == dts.ERR_INVALID
    assert L.dts_compact_rows(4096, 6, None, None, None, None, 2, 8, None, None) == dts.ERR_INVALID  # row_bytes % 4
    assert L.dts_compact_rows(None, 0, None, None, None, None, 2, 8, None, None) == dts.OK       # nothing to do
    assert L.dts_compact_window_rows(None, 1, None, None, None, 1, 65, None, None) == dts.ERR_UNSUPPORTED
    assert L.dts_write_window_kv(None, None, None, None, 4, 64, None, 1, 8, 8, 96, 100, 5e5, None, None, None,
                                 None, None) == dts.ERR_UNSUPPORTED
    assert L.dts_tree_verify_attention(None, None, None, 100, None, 4, 48, None, 0, None, None, 5e5, 1, 8, 32, 8,
                                       128, 0.0, None, None, None, 0, None, None) == dts.ERR_UNSUPPORTED
    assert L.dts_tree_verify_attention(None, None, None, 100, None, 4, 64, None, 0, None, None, 5e5, 1, 8, 30, 8,
                                       128, 0.0, None, None, None, 0, None, None) == dts.ERR_INVALID


def test_argmax_host_checks(lib):
    L = dts.lib()
    # 8 bytes per row and 16384-logit chunk
    assert dts.target_argmax_workspace(2048, 128256) == 2048 * 8 * 8
    assert dts.target_argmax_workspace(5, 1000) == 5 * 8
    assert dts.target_argmax_workspace(3, 16385) == 3 * 2 * 8
    assert dts.target_argmax_workspace(-1, 10) == 0 and dts.target_argmax_workspace(4, 0) == 0
    # bad shapes and pointers fail before any launch; zero rows launch nothing
    assert L.dts_target_argmax(None, 0, 10, 10, None, None, 0, None) == dts.OK
    assert L.dts_target_argmax(None, 4, 10, 9, None, None, 0, None) == dts.ERR_INVALID      # row_stride < vocab
    assert L.dts_target_argmax(None, 4, 10, 10, None, None, 0, None) == dts.ERR_INVALID     # null logits
    assert L.dts_target_argmax(4096, 4, 10, 10, 8192, None, 0, None) == dts.ERR_WORKSPACE   # no workspace
    assert L.dts_target_argmax(4098, 4, 10, 10, 8192, 65536, 4096, None) == dts.ERR_INVALID  # logits not 4-byte aligned
    assert L.dts_target_argmax(4096, 4, 10, 10, 8192, 65537, 4096, None) == dts.ERR_INVALID  # workspace not 8-byte aligned
    assert L.dts_verify_tree_greedy_logits(None, None, 10, 10, None, None, None, 2, 65, None, None, None, None, None,
                                           0, None, None) == dts.ERR_UNSUPPORTED
    assert L.dts_verify_tree_greedy_logits(None, None, 10, 10, None, None, None, 2, 8, None, None, None, None, None,
                                           0, None, None) == dts.ERR_INVALID


def test_fp8_host_checks(lib):
    """The E4M3-cache calls take d = 128 only and otherwise validate like the
    bf16 calls, all before any launch."""
    L = dts.lib()
    wkv = lambda d, B=1, ps=64, ptr=None: L.dts_write_window_kv_fp8(ptr, ptr, ptr, ptr, 4, ps, ptr, B, 8, 8, d, 100,
                                                                    5e5, ptr, ptr, None, None, None)
    assert wkv(64) == dts.ERR_UNSUPPORTED            # the bf16 call takes d = 64; the E4M3 one does not
    assert wkv(96) == dts.ERR_UNSUPPORTED
    assert wkv(128, ps=48) == dts.ERR_UNSUPPORTED
    assert wkv(128, B=0) == dts.OK
    assert wkv(128) == dts.ERR_INVALID               # null pointers
    att = lambda d, B=1, ps=64, hq=32: L.dts_tree_verify_attention_fp8(None, None, None, 100, None, 4, ps, None, 0,
                                                                      None, None, 5e5, B, 8, hq, 8, d, 0.0, None,
                                                                      None, None, 0, None, None)
    assert att(64) == dts.ERR_UNSUPPORTED
    assert att(128, ps=48) == dts.ERR_UNSUPPORTED
    assert att(128, hq=30) == dts.ERR_INVALID        # Hq % Hkv != 0
    assert att(128, B=0) == dts.OK
    assert att(128) == dts.ERR_INVALID               # null pointers
    win = lambda d, R=8, W=48: L.dts_tree_window_attention_fp8(None, None, None, 100, None, 4, 64, None, 0, None,
                                                              None, 5e5, 1, R, W, 32, 8, d, 0.0, None, None, None,
                                                              0, None, None)
    assert win(64) == dts.ERR_UNSUPPORTED
    assert win(128, W=65) == dts.ERR_UNSUPPORTED
    assert win(128) == dts.ERR_INVALID


def test_static_workspace_validates_like_the_regular_call(lib):
    """The allocation-free attention answers every argument error exactly as
    dts_tree_verify_attention does (same checks, same order), B = 0 included,
    without touching the device: nothing is looked up or launched."""
    L = dts.lib()

    def both(B=1, N=8, Hq=32, Hkv=8, d=128, ps=64, theta=5e5, ptr=None):
        reg = L.dts_tree_verify_attention(ptr, ptr, ptr, 100, ptr, 4, ps, ptr, 0, ptr, ptr, theta, B, N, Hq, Hkv, d,
                                          0.0, ptr, ptr, None, 0, None, None)
        sta = L.dts_tree_verify_attention_static_ws(ptr, ptr, ptr, 100, ptr, 4, ps, ptr, 0, ptr, ptr, theta, B, N,
                                                    Hq, Hkv, d, 0.0, ptr, ptr, None, None)
        return reg, sta

    for kw, want in [(dict(B=0), dts.OK), (dict(B=0, N=65), dts.ERR_UNSUPPORTED), (dict(N=65), dts.ERR_UNSUPPORTED),
                     (dict(d=96), dts.ERR_UNSUPPORTED), (dict(ps=48), dts.ERR_UNSUPPORTED),
                     (dict(Hq=30), dts.ERR_INVALID), (dict(theta=0.0, ptr=4096), dts.ERR_INVALID),
                     (dict(B=-1), dts.ERR_INVALID), (dict(), dts.ERR_INVALID)]:
        reg, sta = both(**kw)
        assert reg == sta == want, (kw, reg, sta)
    # a shape beyond the static array is refused as a workspace error once the
    # arguments are valid (aligned non-null pointers; nothing is launched)
    big = dict(B=64, N=64, ptr=4096)
    assert dts.tree_verify_attention_workspace(64, 64, 32, 8, 128, 0) > (64 << 20)
    assert both(**big) == (dts.ERR_WORKSPACE, dts.ERR_WORKSPACE)


def test_stall_hook_validates(lib):
    """The test hook takes stall 0 or 1 and a budget of 2^16 .. 2^31 cycles;
    anything else is refused, and stall = 0 leaves normal operation."""
    L = dts.lib()
    assert L.dts_test_stall_attention(2, 1 << 20) == dts.ERR_INVALID
    assert L.dts_test_stall_attention(1, 100) == dts.ERR_INVALID
    assert L.dts_test_stall_attention(1, 1 << 40) == dts.ERR_INVALID
    assert L.dts_test_stall_attention(0, 1 << 31) == dts.OK


def test_fused_step_calls_validate(lib):
    """The fused prologue and epilogue refuse what the separate calls refuse,
    before any launch; B = 0 launches nothing."""
    L = dts.lib()
    pro = lambda B=1, N=8, d=128, ps=64, theta=5e5, ptr=None: L.dts_verify_prologue(
        ptr, ptr, ptr, ptr, ptr, ptr, 4, ps, ptr, B, N, 8, d, 100, theta, ptr, ptr, ptr, ptr, ptr, ptr, None, None,
        None)
    assert pro(N=65) == dts.ERR_UNSUPPORTED
    assert pro(d=96) == dts.ERR_UNSUPPORTED
    assert pro(ps=48) == dts.ERR_UNSUPPORTED
    assert pro(theta=0.0) == dts.ERR_INVALID
    assert pro(B=0) == dts.OK
    assert pro() == dts.ERR_INVALID                      # null pointers
    assert pro(ptr=4100) == dts.ERR_INVALID              # K/V not 8-byte aligned
    epi = lambda B=1, N=8, nb=0, links=True, ptr=None: L.dts_verify_epilogue(
        ptr, ptr, None, ptr if links else None, ptr if links else None, B, N, ptr, ptr, ptr, ptr, nb, ptr, None, 0,
        None, None, None, None)
    assert epi(N=65) == dts.ERR_UNSUPPORTED
    assert epi(B=0) == dts.OK
    assert epi() == dts.ERR_INVALID                      # null pointers
    assert epi(ptr=4096, links=False) == dts.ERR_INVALID  # neither links nor parents
    assert epi(ptr=4096, nb=-1) == dts.ERR_INVALID
