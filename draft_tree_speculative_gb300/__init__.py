"""Python binding of libdts.so, the GB300 library for the target-verify step
of draft-tree speculative decoding.

The functions here have the names of the C entry points (without the ``dts_``
prefix) and only marshal arguments: they check dtypes, shapes and devices of
torch tensors, pass raw device pointers and sizes to the C ABI on the current
CUDA stream, and raise ``DtsError`` on a non-zero status. Every step of the
verify path runs in the library's CUDA kernels; there is no other code path.
If the library has not been built, loading it fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdts.so")

# status codes (include/dts.h)
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = 0, -1, -2, -3, -4
DEV_OK, DEV_BAD_PARENT, DEV_BAD_DEPTH, DEV_BAD_LINK, DEV_BAD_SLOT, DEV_BAD_PATH, DEV_BAD_BUFFER, DEV_TIMEOUT = range(8)

EXPORTED = (
    "dts_version", "dts_status_string", "dts_device_error_string", "dts_build_tree_mask",
    "dts_write_window_kv", "dts_tree_verify_attention_workspace", "dts_tree_verify_attention",
    "dts_verify_tree_greedy", "dts_compact_window_rows", "dts_compact_rows",
    "dts_tree_verify_attention_static_ws", "dts_target_argmax_workspace", "dts_target_argmax",
    "dts_verify_tree_greedy_logits", "dts_tree_window_attention_workspace", "dts_tree_window_attention",
    "dts_sample_draws", "dts_verify_tree_sampled", "dts_write_window_kv_fp8", "dts_tree_window_attention_fp8",
    "dts_tree_verify_attention_fp8", "dts_test_stall_attention", "dts_verify_prologue", "dts_verify_epilogue",
)


class DtsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "dts_version": (_I, []),
    "dts_status_string": (ctypes.c_char_p, [_I]),
    "dts_device_error_string": (ctypes.c_char_p, [_I]),
    "dts_build_tree_mask": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "dts_write_window_kv": (_I, [_P, _P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _L, _F, _P, _P, _P, _P, _P]),
    "dts_tree_verify_attention_workspace": (_SZ, [_I, _I, _I, _I, _I, _L]),
    "dts_tree_verify_attention": (_I, [_P, _P, _P, _L, _P, _I, _I, _P, _L, _P, _P, _F, _I, _I, _I, _I, _I, _F,
                                       _P, _P, _P, _SZ, _P, _P]),
    "dts_tree_window_attention_workspace": (_SZ, [_I, _I, _I, _I, _I, _I, _L]),
    "dts_tree_window_attention": (_I, [_P, _P, _P, _L, _P, _I, _I, _P, _L, _P, _P, _F, _I, _I, _I, _I, _I, _I, _F,
                                       _P, _P, _P, _SZ, _P, _P]),
    "dts_write_window_kv_fp8": (_I, [_P, _P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _L, _F, _P, _P, _P, _P, _P]),
    "dts_tree_window_attention_fp8": (_I, [_P, _P, _P, _L, _P, _I, _I, _P, _L, _P, _P, _F, _I, _I, _I, _I, _I, _I,
                                           _F, _P, _P, _P, _SZ, _P, _P]),
    "dts_tree_verify_attention_fp8": (_I, [_P, _P, _P, _L, _P, _I, _I, _P, _L, _P, _P, _F, _I, _I, _I, _I, _I, _F,
                                           _P, _P, _P, _SZ, _P, _P]),
    "dts_tree_verify_attention_static_ws": (_I, [_P, _P, _P, _L, _P, _I, _I, _P, _L, _P, _P, _F, _I, _I, _I, _I, _I,
                                                 _F, _P, _P, _P, _P]),
    "dts_verify_tree_greedy": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "dts_target_argmax_workspace": (_SZ, [_L, _I]),
    "dts_sample_draws": (_I, [_P, _I, _L, _P, _P, _P, _P, _I, _I, _P, _P, _SZ, _P]),
    "dts_verify_tree_sampled": (_I, [_P, _P, _I, _L, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _SZ, _P,
                                     _P]),
    "dts_target_argmax": (_I, [_P, _L, _I, _L, _P, _P, _SZ, _P]),
    "dts_verify_tree_greedy_logits": (_I, [_P, _P, _I, _L, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "dts_compact_window_rows": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _P]),
    "dts_compact_rows": (_I, [_P, _L, _P, _P, _P, _P, _I, _I, _P, _P]),
    "dts_test_stall_attention": (_I, [_I, ctypes.c_longlong]),
    "dts_verify_prologue": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _L, _F, _P, _P, _P, _P, _P, _P,
                                 _P, _P, _P]),
    "dts_verify_epilogue": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _P, _P, _L, _P, _P, _P, _P]),
}


def lib():
    """Load libdts.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m draft_tree_speculative_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dts_status_string(status).decode()


def device_error_string(code: int) -> str:
    return lib().dts_device_error_string(code).decode()


def version() -> int:
    return lib().dts_version()


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _check(t, dtypes, shape=None, name="tensor"):
    torch = _torch()
    if t is None:
        return
    if isinstance(dtypes, torch.dtype):
        dtypes = (dtypes,)
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _raise(status: int, where: str):
    if status != OK:
        raise DtsError(status, where)


def _i32():
    return _torch().int32


def _u64():
    torch = _torch()
    return (torch.int64, getattr(torch, "uint64", torch.int64))


# ----------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------

def build_tree_mask(parents, depth, vc, mask, positions, next_token, next_sibling, err=None, stream=None):
    B, N = parents.shape
    i32 = _i32()
    _check(parents, i32, (B, N), "parents")
    _check(depth, i32, (B, N), "depth")
    _check(vc, i32, (B,), "vc")
    _check(mask, _u64(), (B, N), "mask")
    _check(positions, i32, (B, N), "positions")
    _check(next_token, i32, (B, N), "next_token")
    _check(next_sibling, i32, (B, N), "next_sibling")
    _check(err, i32, None, "err")
    st = lib().dts_build_tree_mask(_ptr(parents), _ptr(depth), _ptr(vc), B, N, _ptr(mask), _ptr(positions),
                                   _ptr(next_token), _ptr(next_sibling), _ptr(err), _stream(stream))
    _raise(st, "build_tree_mask")


def write_window_kv(k_new, v_new, positions, page_table, page_size, prefix_len, k_cache, v_cache,
                    rope_theta, write_locations=None, err=None, stream=None, N=None):
    torch = _torch()
    BN, Hkv, d = k_new.shape
    B = prefix_len.shape[0]
    N = BN // B if N is None else N
    _check(k_new, torch.bfloat16, (BN, Hkv, d), "k_new")
    _check(v_new, torch.bfloat16, (BN, Hkv, d), "v_new")
    _check(positions, _i32(), None, "positions")
    _check(page_table, _i32(), None, "page_table")
    _check(k_cache, torch.bfloat16, None, "k_cache")
    _check(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    _check(write_locations, torch.int64, (BN,), "write_locations")
    st = lib().dts_write_window_kv(_ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(page_table),
                                   page_table.shape[1], page_size, _ptr(prefix_len), B, N, Hkv, d,
                                   k_cache.shape[0], float(rope_theta), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(write_locations), _ptr(err), _stream(stream))
    _raise(st, "write_window_kv")


def tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_prefix) -> int:
    return int(lib().dts_tree_verify_attention_workspace(B, N, Hq, Hkv, d, int(max_prefix)))


def tree_verify_attention(q, k_cache, v_cache, page_table, page_size, prefix_len, max_prefix, mask, positions,
                          rope_theta, out, lse2, workspace, softmax_scale=0.0, err=None, stream=None, N=None):
    torch = _torch()
    BN, Hq, d = q.shape
    B = prefix_len.shape[0]
    N = BN // B if N is None else N
    Hkv = k_cache.shape[1]
    _check(q, torch.bfloat16, (BN, Hq, d), "q")
    _check(k_cache, torch.bfloat16, None, "k_cache")
    _check(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), None, "mask")
    _check(out, torch.bfloat16, (BN, Hq, d), "out")
    _check(lse2, torch.float32, (BN, Hq), "lse2")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_tree_verify_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(page_table), page_table.shape[1], page_size,
        _ptr(prefix_len), int(max_prefix), _ptr(mask), _ptr(positions), float(rope_theta), B, N, Hq, Hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse2), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _raise(st, "tree_verify_attention")


def tree_window_attention_workspace(B, R, W, Hq, Hkv, d, max_prefix) -> int:
    return int(lib().dts_tree_window_attention_workspace(B, R, W, Hq, Hkv, d, int(max_prefix)))


def tree_window_attention(q, k_cache, v_cache, page_table, page_size, prefix_len, max_prefix, mask, positions,
                          rope_theta, out, lse2, workspace, W, softmax_scale=0.0, err=None, stream=None):
    """R = q rows / B query rows per request over the prefix plus a W-key
    masked window (draft lanes: R = K, W = (S - 1) * K)."""
    torch = _torch()
    BR, Hq, d = q.shape
    B = prefix_len.shape[0]
    if BR % B:
        raise ValueError("q rows must be a multiple of B")
    R = BR // B
    Hkv = k_cache.shape[1]
    _check(q, torch.bfloat16, (BR, Hq, d), "q")
    _check(k_cache, torch.bfloat16, None, "k_cache")
    _check(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), (B, R), "mask")
    _check(positions, _i32(), (B, R), "positions")
    _check(out, torch.bfloat16, (BR, Hq, d), "out")
    _check(lse2, torch.float32, (BR, Hq), "lse2")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_tree_window_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(page_table), page_table.shape[1], page_size,
        _ptr(prefix_len), int(max_prefix), _ptr(mask), _ptr(positions), float(rope_theta), B, R, int(W), Hq, Hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse2), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _raise(st, "tree_window_attention")


def _fp8_cache(torch):
    """An E4M3 cache is passed as torch.float8_e4m3fn or as its raw bytes (uint8)."""
    return (torch.float8_e4m3fn, torch.uint8)


def write_window_kv_fp8(k_new, v_new, positions, page_table, page_size, prefix_len, k_cache, v_cache,
                        rope_theta, write_locations=None, err=None, stream=None, N=None):
    """write_window_kv into E4M3 caches (include/dts.h, dts_write_window_kv_fp8)."""
    torch = _torch()
    BN, Hkv, d = k_new.shape
    B = prefix_len.shape[0]
    N = BN // B if N is None else N
    _check(k_new, torch.bfloat16, (BN, Hkv, d), "k_new")
    _check(v_new, torch.bfloat16, (BN, Hkv, d), "v_new")
    _check(positions, _i32(), None, "positions")
    _check(page_table, _i32(), None, "page_table")
    _check(k_cache, _fp8_cache(torch), None, "k_cache")
    _check(v_cache, _fp8_cache(torch), tuple(k_cache.shape), "v_cache")
    _check(write_locations, torch.int64, (BN,), "write_locations")
    st = lib().dts_write_window_kv_fp8(_ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(page_table),
                                       page_table.shape[1], page_size, _ptr(prefix_len), B, N, Hkv, d,
                                       k_cache.shape[0], float(rope_theta), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(write_locations), _ptr(err), _stream(stream))
    _raise(st, "write_window_kv_fp8")


def tree_window_attention_fp8(q, k_cache, v_cache, page_table, page_size, prefix_len, max_prefix, mask, positions,
                              rope_theta, out, lse2, workspace, W, softmax_scale=0.0, err=None, stream=None):
    """tree_window_attention over E4M3 caches (include/dts.h, dts_tree_window_attention_fp8)."""
    torch = _torch()
    BR, Hq, d = q.shape
    B = prefix_len.shape[0]
    if BR % B:
        raise ValueError("q rows must be a multiple of B")
    R = BR // B
    Hkv = k_cache.shape[1]
    _check(q, torch.bfloat16, (BR, Hq, d), "q")
    _check(k_cache, _fp8_cache(torch), None, "k_cache")
    _check(v_cache, _fp8_cache(torch), tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), (B, R), "mask")
    _check(positions, _i32(), (B, R), "positions")
    _check(out, torch.bfloat16, (BR, Hq, d), "out")
    _check(lse2, torch.float32, (BR, Hq), "lse2")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_tree_window_attention_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(page_table), page_table.shape[1], page_size,
        _ptr(prefix_len), int(max_prefix), _ptr(mask), _ptr(positions), float(rope_theta), B, R, int(W), Hq, Hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse2), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _raise(st, "tree_window_attention_fp8")


def tree_verify_attention_fp8(q, k_cache, v_cache, page_table, page_size, prefix_len, max_prefix, mask, positions,
                              rope_theta, out, lse2, workspace, softmax_scale=0.0, err=None, stream=None, N=None):
    """tree_verify_attention over E4M3 caches (include/dts.h, dts_tree_verify_attention_fp8)."""
    torch = _torch()
    BN, Hq, d = q.shape
    B = prefix_len.shape[0]
    N = BN // B if N is None else N
    Hkv = k_cache.shape[1]
    _check(q, torch.bfloat16, (BN, Hq, d), "q")
    _check(k_cache, _fp8_cache(torch), None, "k_cache")
    _check(v_cache, _fp8_cache(torch), tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), None, "mask")
    _check(out, torch.bfloat16, (BN, Hq, d), "out")
    _check(lse2, torch.float32, (BN, Hq), "lse2")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_tree_verify_attention_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(page_table), page_table.shape[1], page_size,
        _ptr(prefix_len), int(max_prefix), _ptr(mask), _ptr(positions), float(rope_theta), B, N, Hq, Hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse2), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _raise(st, "tree_verify_attention_fp8")


def tree_verify_attention_static_ws(q, k_cache, v_cache, page_table, page_size, prefix_len, max_prefix, mask,
                                    positions, rope_theta, out, lse2, softmax_scale=0.0, err=None, stream=None,
                                    N=None):
    """tree_verify_attention with the library's own fixed device workspace, for
    callers that cannot allocate device memory (see include/dts.h)."""
    torch = _torch()
    BN, Hq, d = q.shape
    B = prefix_len.shape[0]
    N = BN // B if N is None else N
    Hkv = k_cache.shape[1]
    _check(q, torch.bfloat16, (BN, Hq, d), "q")
    _check(k_cache, torch.bfloat16, None, "k_cache")
    _check(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), None, "mask")
    _check(out, torch.bfloat16, (BN, Hq, d), "out")
    _check(lse2, torch.float32, (BN, Hq), "lse2")
    st = lib().dts_tree_verify_attention_static_ws(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(page_table), page_table.shape[1], page_size,
        _ptr(prefix_len), int(max_prefix), _ptr(mask), _ptr(positions), float(rope_theta), B, N, Hq, Hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse2), _ptr(err), _stream(stream))
    _raise(st, "tree_verify_attention_static_ws")


def verify_tree_greedy(draft_tokens, target_argmax, accept_len, accepted_path, accepted_tokens, parents=None,
                       next_token=None, next_sibling=None, err=None, stream=None):
    B, N = draft_tokens.shape
    i32 = _i32()
    for name, t in (("draft_tokens", draft_tokens), ("target_argmax", target_argmax), ("parents", parents),
                    ("next_token", next_token), ("next_sibling", next_sibling),
                    ("accepted_path", accepted_path), ("accepted_tokens", accepted_tokens)):
        _check(t, i32, (B, N), name)
    _check(accept_len, i32, (B,), "accept_len")
    st = lib().dts_verify_tree_greedy(_ptr(draft_tokens), _ptr(target_argmax), _ptr(parents), _ptr(next_token),
                                      _ptr(next_sibling), B, N, _ptr(accept_len), _ptr(accepted_path),
                                      _ptr(accepted_tokens), _ptr(err), _stream(stream))
    _raise(st, "verify_tree_greedy")


def _logits(logits):
    """(pointer, rows, vocab, row stride) of fp32 logits [rows][vocab] whose
    rows may be strided (each row's vocab entries contiguous)."""
    torch = _torch()
    if logits.dtype != torch.float32 or logits.dim() != 2:
        raise TypeError("logits: expected a 2-D float32 tensor")
    if not logits.is_cuda:
        raise ValueError("logits: expected a CUDA tensor")
    if logits.shape[1] > 1 and logits.stride(1) != 1:
        raise ValueError("logits: each row must be contiguous")
    return logits.data_ptr(), logits.shape[0], logits.shape[1], logits.stride(0)


def target_argmax_workspace(rows, vocab) -> int:
    return int(lib().dts_target_argmax_workspace(int(rows), int(vocab)))


def target_argmax(logits, argmax, workspace, stream=None):
    """argmax [rows] int32 <- the index of each row's largest logit."""
    p, rows, vocab, stride = _logits(logits)
    _check(argmax, _i32(), (rows,), "argmax")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_target_argmax(p, rows, vocab, stride, _ptr(argmax), _ptr(workspace), ws_bytes, _stream(stream))
    _raise(st, "target_argmax")


def verify_tree_greedy_logits(draft_tokens, logits, target_argmax, accept_len, accepted_path, accepted_tokens,
                              workspace, parents=None, next_token=None, next_sibling=None, err=None, stream=None):
    """The argmax of logits [B*N][vocab] into target_argmax [B][N], then the greedy walk."""
    B, N = draft_tokens.shape
    p, rows, vocab, stride = _logits(logits)
    if rows != B * N:
        raise ValueError("logits must have B*N rows")
    i32 = _i32()
    for name, t in (("draft_tokens", draft_tokens), ("target_argmax", target_argmax), ("parents", parents),
                    ("next_token", next_token), ("next_sibling", next_sibling),
                    ("accepted_path", accepted_path), ("accepted_tokens", accepted_tokens)):
        _check(t, i32, (B, N), name)
    _check(accept_len, i32, (B,), "accept_len")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_verify_tree_greedy_logits(_ptr(draft_tokens), p, vocab, stride, _ptr(parents), _ptr(next_token),
                                             _ptr(next_sibling), B, N, _ptr(target_argmax), _ptr(accept_len),
                                             _ptr(accepted_path), _ptr(accepted_tokens), _ptr(workspace), ws_bytes,
                                             _ptr(err), _stream(stream))
    _raise(st, "verify_tree_greedy_logits")


def sample_draws(logits, vc, depth, temperature, seed, draws, workspace, stream=None):
    """draws [B][N] <- Gumbel-max draws of logits [B*N][vocab] keyed by
    (seed[b], vc[b] + depth[b][i] + 1); temperature float32 [B], seed int64/uint64 [B]."""
    torch = _torch()
    B, N = depth.shape
    p, rows, vocab, stride = _logits(logits)
    if rows != B * N:
        raise ValueError("logits must have B*N rows")
    _check(vc, _i32(), (B,), "vc")
    _check(depth, _i32(), (B, N), "depth")
    _check(temperature, torch.float32, (B,), "temperature")
    _check(seed, _u64(), (B,), "seed")
    _check(draws, _i32(), (B, N), "draws")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_sample_draws(p, vocab, stride, _ptr(vc), _ptr(depth), _ptr(temperature), _ptr(seed), B, N,
                                _ptr(draws), _ptr(workspace), ws_bytes, _stream(stream))
    _raise(st, "sample_draws")


def verify_tree_sampled(draft_tokens, logits, vc, depth, temperature, seed, draws, accept_len, accepted_path,
                        accepted_tokens, workspace, parents=None, next_token=None, next_sibling=None, err=None,
                        stream=None):
    """Sampled draws (sample_draws), then the greedy walk over them."""
    torch = _torch()
    B, N = draft_tokens.shape
    p, rows, vocab, stride = _logits(logits)
    if rows != B * N:
        raise ValueError("logits must have B*N rows")
    i32 = _i32()
    for name, t in (("draft_tokens", draft_tokens), ("depth", depth), ("draws", draws), ("parents", parents),
                    ("next_token", next_token), ("next_sibling", next_sibling),
                    ("accepted_path", accepted_path), ("accepted_tokens", accepted_tokens)):
        _check(t, i32, (B, N), name)
    _check(vc, i32, (B,), "vc")
    _check(accept_len, i32, (B,), "accept_len")
    _check(temperature, torch.float32, (B,), "temperature")
    _check(seed, _u64(), (B,), "seed")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().dts_verify_tree_sampled(_ptr(draft_tokens), p, vocab, stride, _ptr(vc), _ptr(depth), _ptr(temperature),
                                       _ptr(seed), _ptr(parents), _ptr(next_token), _ptr(next_sibling), B, N,
                                       _ptr(draws), _ptr(accept_len), _ptr(accepted_path), _ptr(accepted_tokens),
                                       _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    _raise(st, "verify_tree_sampled")


def make_kv_table(entries: Sequence, device="cuda"):
    """Device copy of a dts_kv_buffer table. entries: (base pointer or tensor,
    slot_stride_bytes, num_slots, row_bytes) tuples. Returns an int64 [L][4]
    tensor laid out as the C struct (the last word holds row_bytes | reserved<<32)."""
    torch = _torch()
    rows = []
    for base, stride, nslots, row_bytes in entries:
        p = base if isinstance(base, int) else base.data_ptr()
        rows.append([p, int(stride), int(nslots), int(row_bytes) & 0xFFFFFFFF])
    return torch.tensor(rows, dtype=torch.int64).to(device)


def compact_window_rows(table, write_locations, accepted_path, accept_len, err=None, stream=None):
    B, N = accepted_path.shape
    _check(write_locations, _torch().int64, (B * N,), "write_locations")
    _check(accepted_path, _i32(), (B, N), "accepted_path")
    _check(accept_len, _i32(), (B,), "accept_len")
    st = lib().dts_compact_window_rows(_ptr(table), table.shape[0], _ptr(write_locations), _ptr(accepted_path),
                                       _ptr(accept_len), B, N, _ptr(err), _stream(stream))
    _raise(st, "compact_window_rows")


def compact_rows(hidden, positions, vc, accepted_path, accept_len, err=None, stream=None):
    B, N = accepted_path.shape
    row_bytes = 0
    if hidden is not None:
        row_bytes = hidden[0].numel() * hidden.element_size()
        if hidden.shape[0] != B * N:
            raise ValueError("hidden must have B*N rows")
    _check(positions, _i32(), (B, N), "positions")
    st = lib().dts_compact_rows(_ptr(hidden), row_bytes, _ptr(positions), _ptr(vc), _ptr(accepted_path),
                                _ptr(accept_len), B, N, _ptr(err), _stream(stream))
    _raise(st, "compact_rows")


def verify_prologue(parents, depth, vc, k_new, v_new, page_table, page_size, prefix_len, k_cache, v_cache, rope_theta,
                    mask, positions, next_token, next_sibling, write_locations=None, err=None, stream=None):
    """build_tree_mask and write_window_kv (bf16 cache) in one launch."""
    torch = _torch()
    B, N = parents.shape
    BN, Hkv, d = k_new.shape
    if BN != B * N:
        raise ValueError("k_new must have B*N rows")
    i32 = _i32()
    _check(parents, i32, (B, N), "parents")
    _check(depth, i32, (B, N), "depth")
    _check(vc, i32, (B,), "vc")
    _check(prefix_len, i32, (B,), "prefix_len")
    _check(k_new, torch.bfloat16, (BN, Hkv, d), "k_new")
    _check(v_new, torch.bfloat16, (BN, Hkv, d), "v_new")
    _check(page_table, i32, None, "page_table")
    _check(k_cache, torch.bfloat16, None, "k_cache")
    _check(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    _check(mask, _u64(), (B, N), "mask")
    for name, t in (("positions", positions), ("next_token", next_token), ("next_sibling", next_sibling)):
        _check(t, i32, (B, N), name)
    _check(write_locations, torch.int64, (BN,), "write_locations")
    st = lib().dts_verify_prologue(_ptr(parents), _ptr(depth), _ptr(vc), _ptr(k_new), _ptr(v_new), _ptr(page_table),
                                   page_table.shape[1], page_size, _ptr(prefix_len), B, N, Hkv, d, k_cache.shape[0],
                                   float(rope_theta), _ptr(mask), _ptr(positions), _ptr(next_token),
                                   _ptr(next_sibling), _ptr(k_cache), _ptr(v_cache), _ptr(write_locations), _ptr(err),
                                   _stream(stream))
    _raise(st, "verify_prologue")


def verify_epilogue(draft_tokens, target_argmax, accept_len, accepted_path, accepted_tokens, table=None,
                    write_locations=None, hidden=None, positions=None, vc=None, parents=None, next_token=None,
                    next_sibling=None, err=None, stream=None):
    """verify_tree_greedy, compact_window_rows and compact_rows in one launch."""
    B, N = draft_tokens.shape
    i32 = _i32()
    for name, t in (("draft_tokens", draft_tokens), ("target_argmax", target_argmax), ("parents", parents),
                    ("next_token", next_token), ("next_sibling", next_sibling),
                    ("accepted_path", accepted_path), ("accepted_tokens", accepted_tokens), ("positions", positions)):
        _check(t, i32, (B, N), name)
    _check(accept_len, i32, (B,), "accept_len")
    _check(vc, i32, (B,), "vc")
    _check(write_locations, _torch().int64, (B * N,), "write_locations")
    row_bytes = 0
    if hidden is not None:
        row_bytes = hidden[0].numel() * hidden.element_size()
        if hidden.shape[0] != B * N:
            raise ValueError("hidden must have B*N rows")
    n_buffers = 0 if table is None else table.shape[0]
    st = lib().dts_verify_epilogue(_ptr(draft_tokens), _ptr(target_argmax), _ptr(parents), _ptr(next_token),
                                   _ptr(next_sibling), B, N, _ptr(accept_len), _ptr(accepted_path),
                                   _ptr(accepted_tokens), _ptr(table), n_buffers, _ptr(write_locations),
                                   _ptr(hidden), row_bytes, _ptr(positions), _ptr(vc), _ptr(err), _stream(stream))
    _raise(st, "verify_epilogue")
