"""GPU parity of the fused step launches, through the C ABI.

verify_prologue (build_tree_mask + write_window_kv) and verify_epilogue
(verify_tree_greedy + compact_window_rows + compact_rows) must leave every
output byte for byte as the separate calls do, on the workloads' seeded
inputs (the high-concurrency one with its 64 fp8 buffers and hidden rows) and
on bad trees and links, where the device-side error codes must agree too. The
fused path's mask, links and walk are also compared with the oracle directly.
"""
import numpy as np
import pytest

from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch, run_step
from oracle import tree as OT
from oracle import walk as OW
from tests.gpu_helpers import torch_cuda

pytestmark = pytest.mark.gpu

OUTPUTS = ("mask", "positions", "next_token", "next_sibling", "write_locations", "accept_len", "accepted_path",
           "accepted_tokens", "k_cache", "v_cache", "out", "lse2", "err")


def _state(db):
    torch = torch_cuda()
    torch.cuda.synchronize()
    st = {k: getattr(db, k).detach().clone().view(torch.uint8).cpu().numpy() if getattr(db, k).dtype in
          (torch.bfloat16, torch.float32) else getattr(db, k).cpu().numpy() for k in OUTPUTS}
    if db.hidden is not None:
        st["hidden"] = db.hidden.view(torch.int16).cpu().numpy()
    # the fp8 buffers: their window rows, and a checksum of every byte (the
    # whole buffers are too large to bring back)
    wl = db.write_locations.clamp(min=0)
    for i, buf in enumerate(db.fp8_buffers):
        st[f"fp8_{i}_window"] = buf[wl].cpu().numpy()
        st[f"fp8_{i}_sum"] = int(buf.view(torch.int32).to(torch.int64).sum().item())
    return st


def _both(inp, fp8_layers=None):
    a = DeviceBatch(inp, fp8_layers=fp8_layers)
    run_step(a, fused=False)
    sa = _state(a)
    del a
    b = DeviceBatch(inp, fp8_layers=fp8_layers)
    run_step(b, fused=True)
    sb = _state(b)
    return sa, sb, b


def _assert_same(sa, sb):
    assert sa.keys() == sb.keys()
    for k in sa:
        assert np.array_equal(sa[k], sb[k]), k


@pytest.mark.parametrize("name", ["tiny_p128_n5", "llama8b_p4096_n8", "eagle2_p8192_n64", "highconc_b128_n16"])
def test_fused_launches_equal_separate_calls(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    sa, sb, db = _both(inp)
    _assert_same(sa, sb)
    assert int(sb["err"][0]) == 0
    # the fused path against the oracle: mask, links, the walk
    w = inp.w
    for b in range(min(w.B, 8)):
        m, p, nt, ns = OT.build_tree_mask(inp.parents[b], inp.depth[b], int(inp.vc[b]))
        assert (sb["mask"][b].view(np.uint64) == m).all()
        assert (sb["next_token"][b] == nt).all() and (sb["next_sibling"][b] == ns).all()
    alen, path, tok = OW.greedy_walk_batch(inp.parents, inp.draft, inp.target_argmax)
    assert (sb["accept_len"] == alen).all() and (sb["accepted_path"] == path).all()
    assert (sb["accepted_tokens"] == tok).all()


def _bad(inp, kind):
    inp.parents = inp.parents.copy()
    inp.depth = inp.depth.copy()
    if kind == "parent":
        inp.parents[1, 3] = 5            # a parent after its child
    elif kind == "depth":
        inp.depth[0, 2] += 1             # depth not parent's + 1
    return inp


@pytest.mark.parametrize("kind", ["parent", "depth"])
def test_fused_launches_report_bad_trees_alike(kind):
    inp = _bad(synth.make_inputs(synth.WORKLOADS["llama8b_p4096_n8"]), kind)
    sa, sb, _ = _both(inp)
    _assert_same(sa, sb)
    assert int(sb["err"][0]) != 0
