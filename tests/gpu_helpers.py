"""Helpers shared by the GPU parity tests (the oracle side and the CUDA side
meet only here, on the same seeded inputs)."""
import dataclasses

import numpy as np

from draft_tree_speculative_gb300 import synth

OUT_ATOL = 1e-2   # bf16 attention output: |gpu - oracle| <= OUT_ATOL + OUT_RTOL * |oracle|
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3   # fp32 base-2 log-sum-exp: |gpu - oracle| <= LSE_ATOL


def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    return torch


def random_tree(rng, n):
    parents = np.zeros(n, np.int32)
    parents[0] = -1
    for i in range(1, n):
        parents[i] = rng.integers(0, i)
    return parents, synth.depth_of(parents)


def custom_workload(base: str, index: int, **kw) -> synth.Workload:
    return dataclasses.replace(synth.WORKLOADS[base], name=f"{base}_custom{index}", index=100 + index, **kw)


def bf16_bits_of(t) -> np.ndarray:
    """uint16 bits of a bf16 torch tensor (host copy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t) -> np.ndarray:
    return synth.bf16_bits_to_f64(bf16_bits_of(t))


def assert_attention_close(out_gpu, lse_gpu, out_ref, lse_ref, rows):
    """rows: list of flat row indices b*N+v to compare (all heads)."""
    for r in rows:
        o, l = out_gpu[r], lse_gpu[r]
        ro, rl = out_ref[r], lse_ref[r]
        assert np.isfinite(ro).all(), f"oracle row {r} not finite"
        err_o = np.abs(o - ro)
        bad = err_o > OUT_ATOL + OUT_RTOL * np.abs(ro)
        assert not bad.any(), (f"row {r}: out mismatch at {np.argwhere(bad)[:5].tolist()}, "
                               f"max err {err_o.max():.3e}")
        err_l = np.abs(l - rl)
        assert (err_l <= LSE_ATOL).all(), f"row {r}: lse2 max err {err_l.max():.3e}"


# ----------------------------------------------------------------------------
# the oracle on every row of a full-size workload, in spawned host processes
# ----------------------------------------------------------------------------

_WORKER_INPUTS = {}


def _worker_inputs(kind, name):
    key = (kind, name)
    if key not in _WORKER_INPUTS:
        w = synth.WORKLOADS[name]
        if kind == "bf16":
            _WORKER_INPUTS[key] = (synth.make_inputs(w, with_hidden=False),)
        else:
            inp = synth.make_inputs(w, with_cache=False, with_hidden=False)
            _WORKER_INPUTS[key] = (inp, *synth.fp8_kv_cache(w.index, inp.layout.num_slots, w.Hkv, w.d))
    return _WORKER_INPUTS[key]


def _oracle_task(kind, name, requests, rotate):
    """Oracle rows of `requests` (every node, all heads) of a named workload:
    the bf16 path-driven oracle, or the mask-driven one over the E4M3 cache."""
    from oracle import attention as OA
    from oracle import tree as OT
    got = _worker_inputs(kind, name)
    inp = got[0]
    w, lay = inp.w, inp.layout
    N = w.N
    rows = np.concatenate([np.arange(b * N, (b + 1) * N) for b in requests])
    if kind == "bf16":
        o, l = OA.verify_attention(inp.q, inp.k_new, inp.v_new, inp.k_cache, inp.v_cache, lay.page_table, inp.vc,
                                   inp.parents, w.Hkv, w.rope_theta, page_size=w.page_size,
                                   rows=[(b, v) for b in requests for v in range(N)])
        return rows, o[rows], l[rows]
    k8, v8 = got[1], got[2]
    req = list(requests)
    mask = [[int(x) for x in OT.ancestor_mask(inp.parents[b])] for b in req]
    pos = [[int(x) for x in OT.positions(int(lay.prefix_len[b]), inp.depth[b])] for b in req]
    o, l = OA.window_attention(inp.q[rows], k8, v8, lay.page_table[req], lay.prefix_len[req], mask, pos, N, w.Hkv,
                               w.rope_theta, page_size=w.page_size, q_rotated=not rotate, kv_fp8=True, q_fp8=True)
    return rows, o, l


def oracle_every_row(kind, name, rotate=True, max_workers=16):
    """(out [B*N][Hq][d], lse2 [B*N][Hq]) of the oracle for every row of the
    named workload. Requests are spread over spawned worker processes, one
    BLAS thread each (each worker draws the seeded inputs itself, so nothing
    large crosses a process boundary); spawn keeps a CUDA context out of the
    workers."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    w = synth.WORKLOADS[name]
    n = max(1, min(max_workers, os.cpu_count() or 1, w.B))
    chunks = [list(range(w.B))[i::n] for i in range(n)]
    keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in keep:
        os.environ[k] = "1"
    try:
        with cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            parts = list(ex.map(_oracle_task, [kind] * n, [name] * n, chunks, [rotate] * n))
    finally:
        for k, v in keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    out = np.full((w.B * w.N, w.Hq, w.d), np.nan)
    lse = np.full((w.B * w.N, w.Hq), np.nan)
    for rows, o, l in parts:
        out[rows], lse[rows] = o, l
    return out, lse
