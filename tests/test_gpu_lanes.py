"""GPU parity: tree_window_attention (R query rows over the prefix plus a
W-key masked window: draft lanes) against the oracle, through the C ABI.

Tolerances as for the verify attention: output within atol 1e-2 / rtol 1e-2
(bf16), base-2 LSE within 1e-3 absolute."""
import dataclasses

import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch
from oracle import attention as OA
from tests.gpu_helpers import assert_attention_close, bf16_to_f64, torch_cuda

pytestmark = pytest.mark.gpu


def _run_lanes(li, mask=None):
    torch = torch_cuda()
    lw = li.lw
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to("cuda")
    B, R, W = lw.B, lw.R, lw.W
    m = li.mask if mask is None else mask
    q = bf(li.q)
    kc, vc = bf(li.k_cache), bf(li.v_cache)
    out = torch.full((B * R, lw.Hq, lw.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B * R, lw.Hq), float("nan"), dtype=torch.float32, device="cuda")
    max_prefix = int(max(lw.prefix))
    ws = torch.empty(dts.tree_window_attention_workspace(B, R, W, lw.Hq, lw.Hkv, lw.d, max_prefix),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.tree_window_attention(q, kc, vc, t(li.layout.page_table), lw.page_size, t(li.prefix_len), max_prefix,
                              t(np.asarray(m, np.uint64).view(np.int64)), t(li.positions), lw.rope_theta, out, lse,
                              ws, W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def _oracle(li, mask=None):
    lw = li.lw
    return OA.window_attention(li.q, li.k_cache, li.v_cache, li.layout.page_table, li.prefix_len,
                               li.mask if mask is None else mask, li.positions, lw.W, lw.Hkv, lw.rope_theta,
                               page_size=lw.page_size)


def _lane(name="lanes_eagle2_p8192_k8_s7", **kw):
    base = synth.LANE_WORKLOADS[name]
    return dataclasses.replace(base, name=f"{name}_t", index=200 + len(kw), **kw) if kw else base


def test_lane_workload_full_size():
    """The EAGLE-2 batch's last drafting step: 32 requests x 8 lane rows over
    the 48-key lane window and an 8192-token frontier; every row compared."""
    li = synth.make_lane_inputs(_lane())
    out, lse = _run_lanes(li)
    ref_o, ref_l = _oracle(li)
    assert_attention_close(out, lse, ref_o, ref_l, range(li.lw.B * li.lw.R))


@pytest.mark.parametrize("kw", [
    dict(B=3, K=4, S=5, prefix=[0, 129, 1000]),                           # empty and ragged prefixes
    dict(B=2, K=8, S=9, prefix=[300, 64]),                                 # W = 64
    dict(B=2, K=5, S=3, step=1, prefix=[77, 200]),                         # the first drafting step
    dict(B=2, K=8, S=7, Hq=64, Hkv=8, prefix=[1023, 2048]),               # g = 8: M = 64
    dict(B=2, K=4, S=4, Hq=16, Hkv=1, d=64, prefix=[500, 31]),             # g = 16, d = 64
    dict(B=2, K=6, S=4, Hq=8, Hkv=8, page_size=16, prefix=[90, 400]),     # g = 1, small pages
    dict(B=1, K=32, S=3, Hq=32, Hkv=2, prefix=[700]),                      # R = 32, M = 512: two units
])
def test_lane_shapes(kw):
    li = synth.make_lane_inputs(_lane(**kw))
    out, lse = _run_lanes(li)
    ref_o, ref_l = _oracle(li)
    assert_attention_close(out, lse, ref_o, ref_l, range(li.lw.B * li.lw.R))


def test_arbitrary_window_masks():
    """Any bit pattern over the window, including rows that see no window key
    (prefix only) and rows that see every window key."""
    li = synth.make_lane_inputs(_lane(B=2, K=8, S=5, prefix=[333, 12]))
    rng = np.random.default_rng(70)
    W = li.lw.W
    mask = rng.integers(0, 1 << W, size=(2, 8), dtype=np.uint64)
    mask[0, 0] = 0
    mask[1, 1] = (1 << W) - 1
    out, lse = _run_lanes(li, mask)
    ref_o, ref_l = _oracle(li, mask)
    assert_attention_close(out, lse, ref_o, ref_l, range(16))


def test_verify_is_window_attention_with_r_equal_w():
    """dts_tree_verify_attention is the window call with R = W = N: the two
    give bit-identical outputs on a verify batch."""
    torch = torch_cuda()
    inp = synth.make_inputs(synth.WORKLOADS["llama8b_p4096_n8"])
    w = inp.w
    db = DeviceBatch(inp, compact_attention_kv=False, fp8_layers=0)
    db.mask_step()
    db.window_kv_step()
    db.attention_step()
    torch.cuda.synchronize()
    out_v, lse_v = db.out.clone(), db.lse2.clone()
    out = torch.empty_like(out_v)
    lse = torch.empty_like(lse_v)
    ws = torch.empty(dts.tree_window_attention_workspace(w.B, w.N, w.N, w.Hq, w.Hkv, w.d, db.max_prefix),
                     dtype=torch.uint8, device="cuda")
    dts.tree_window_attention(db.q, db.k_cache, db.v_cache, db.page_table, w.page_size, db.prefix_len,
                              db.max_prefix, db.mask, db.positions, w.rope_theta, out, lse, ws, w.N, err=db.err)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    assert torch.equal(out.view(torch.int16), out_v.view(torch.int16)) and torch.equal(lse, lse_v)
