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
