"""GPU parity over an FP8-E4M3 KV cache: write_window_kv_fp8,
tree_verify_attention_fp8 and tree_window_attention_fp8 against the oracle,
through the C ABI.

Attention tolerances are those of the bf16 cache: output within atol 1e-2 /
rtol 1e-2 (bf16), base-2 LSE within 1e-3 absolute. Both sides read the same
E4M3 bytes and cast the query to E4M3 by the same rule, so neither adds a
rounding to compare, and the kernel's f16 softmax weights are finer than the
bf16 ones those bounds were set for. Where the query is rotated on both sides
(fp32 on the device, exact in the oracle), a rare element rounds to
neighbouring bf16 values and then to neighbouring E4M3 values; the full-size
cases pass the query as already rotated, so that the cast sees identical
inputs. The window write is compared byte for byte."""
import dataclasses

import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from oracle import attention as OA
from oracle import fp8 as F8
from oracle import tree as OT
from tests.gpu_helpers import (assert_attention_close, bf16_to_f64, custom_workload, oracle_every_row, random_tree,
                               torch_cuda)

pytestmark = pytest.mark.gpu


def _dev(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _bf(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to("cuda")


def _outputs(rows, Hq, d):
    torch = torch_cuda()
    out = torch.full((rows, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((rows, Hq), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


# ---------------------------------------------------------------------------- verify (R = W = N, tree masks)

def _verify_case(w, trees=None):
    inp = synth.make_inputs(w, with_cache=False, with_hidden=False, trees=trees)
    k8, v8 = synth.fp8_kv_cache(w.index, inp.layout.num_slots, w.Hkv, w.d)
    return inp, k8, v8


def _run_verify_fp8(inp, k8, v8, rotate=True, page_table=None, expect_err=0):
    """GPU: the tree's masks and positions (build_tree_mask), then the
    attention with the query rotated at each node's position (or taken as
    already rotated); the device error code must read `expect_err`."""
    torch = torch_cuda()
    w, lay = inp.w, inp.layout
    B, N = w.B, w.N
    mask = torch.zeros((B, N), dtype=torch.int64, device="cuda")
    pos = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    nt = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    ns = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.build_tree_mask(_dev(inp.parents), _dev(inp.depth), _dev(lay.prefix_len), mask, pos, nt, ns, err=err)
    out, lse = _outputs(B * N, w.Hq, w.d)
    max_prefix = int(lay.prefix_len.max())
    ws = torch.empty(dts.tree_verify_attention_workspace(B, N, w.Hq, w.Hkv, w.d, max_prefix), dtype=torch.uint8,
                     device="cuda")
    pt = lay.page_table if page_table is None else page_table
    dts.tree_verify_attention_fp8(_bf(inp.q), _dev(k8), _dev(v8), _dev(pt), w.page_size,
                                  _dev(lay.prefix_len), max_prefix, mask, pos if rotate else None, w.rope_theta, out,
                                  lse, ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def _oracle_verify_fp8(inp, k8, v8, requests, rotate=True):
    """The oracle on the given requests: ancestor masks and positions vc +
    depth of its own, the window's keys read from the cache as stored."""
    w, lay = inp.w, inp.layout
    N = w.N
    req = list(requests)
    rows = np.concatenate([np.arange(b * N, (b + 1) * N) for b in req])
    mask = [[int(x) for x in OT.ancestor_mask(inp.parents[b])] for b in req]
    pos = [[int(x) for x in OT.positions(int(lay.prefix_len[b]), inp.depth[b])] for b in req]
    o, l = OA.window_attention(inp.q[rows], k8, v8, lay.page_table[req], lay.prefix_len[req], mask, pos, N, w.Hkv,
                               w.rope_theta, page_size=w.page_size, q_rotated=not rotate, kv_fp8=True, q_fp8=True)
    return rows, o, l


def _check_verify(inp, k8, v8, requests, out, lse, rotate=True):
    rows, ro, rl = _oracle_verify_fp8(inp, k8, v8, requests, rotate)
    assert_attention_close(out[rows], lse[rows], ro, rl, range(len(rows)))


def test_verify_fp8_llama8b_all_rows():
    """8 requests x 8 nodes over 4096-key prefixes: 33 key tiles per unit, the
    last one ragged; every row compared."""
    inp, k8, v8 = _verify_case(synth.WORKLOADS["llama8b_p4096_n8"])
    out, lse = _run_verify_fp8(inp, k8, v8)
    _check_verify(inp, k8, v8, range(inp.w.B), out, lse)


def test_verify_fp8_eagle2_full_size_every_row():
    """The EAGLE-2 batch at full size (32 requests x 64 nodes, P = 8192) in
    the launch the bench times; every row compared (the oracle spread over
    host processes)."""
    w = synth.WORKLOADS["eagle2_p8192_n64"]
    inp, k8, v8 = _verify_case(w)
    out, lse = _run_verify_fp8(inp, k8, v8, rotate=False)
    ro, rl = oracle_every_row("fp8", w.name, rotate=False)
    assert_attention_close(out, lse, ro, rl, range(w.B * w.N))


@pytest.mark.parametrize("i, over, kind", [
    (0, dict(B=3, prefix=[0, 129, 1000]), "random"),     # empty and ragged prefixes
    (1, dict(B=2, prefix=[127, 128]), "chain"),          # a 64-deep chain; tile edges
    (2, dict(B=2, prefix=[64, 4000], Hq=64), "star"),    # g = 8; a star
    (3, dict(B=2, prefix=[300, 77], Hq=8, page_size=16), "random"),  # g = 1, small pages
])
def test_verify_fp8_edge_cases(i, over, kind):
    w = custom_workload("eagle2_p8192_n64", 60 + i, **over)
    rng = np.random.default_rng(600 + i)
    par = np.zeros((w.B, w.N), np.int32)
    for b in range(w.B):
        if kind == "chain":
            par[b] = np.arange(-1, w.N - 1)
        elif kind == "star":
            par[b] = [-1] + [0] * (w.N - 1)
        else:
            par[b] = random_tree(rng, w.N)[0]
    dep = np.stack([synth.depth_of(p) for p in par]).astype(np.int32)
    inp, k8, v8 = _verify_case(w, trees=(par, dep))
    out, lse = _run_verify_fp8(inp, k8, v8)
    _check_verify(inp, k8, v8, range(w.B), out, lse)


def test_verify_fp8_every_finite_code():
    """Caches drawn uniformly from every E4M3 code of magnitude <= 8, the
    subnormals (S.0000.MMM) and both zeros included: the widening is exact for
    each code, whatever its binade."""
    w = custom_workload("llama8b_p4096_n8", 62, B=2, prefix=[500, 130])
    inp, _, _ = _verify_case(w)
    codes = np.array([c for c in range(256) if (c & 0x7F) <= 0x50], np.uint8)   # 0x50 = 8.0
    rng = np.random.default_rng(62)
    shape = (inp.layout.num_slots, w.Hkv, w.d)
    k8, v8 = rng.choice(codes, size=shape), rng.choice(codes, size=shape)
    assert (F8.decode_e4m3(codes) != 0).sum() > 150 and ((codes & 0x78) == 0).sum() == 16
    out, lse = _run_verify_fp8(inp, k8, v8, rotate=False)
    _check_verify(inp, k8, v8, range(w.B), out, lse, rotate=False)


def test_verify_fp8_nan_bytes_reach_only_the_rows_that_see_them():
    """NaN bytes in slots no row may read (the reserved page, slots past each
    window: K and V) and one NaN byte in a leaf's V row: only the leaf's own
    rows change, and they turn non-finite."""
    w = custom_workload("llama8b_p4096_n8", 61, B=3, prefix=[100, 191, 4096])
    inp, k8, v8 = _verify_case(w)
    lay, N, ps = inp.layout, w.N, w.page_size
    out_ref, lse_ref = _run_verify_fp8(inp, k8, v8)
    k8p, v8p = k8.copy(), v8.copy()
    k8p[:ps] = 0x7F
    v8p[:ps] = 0xFF
    leaf = N - 1                        # depth-first numbering: the last node is a leaf
    for b in range(w.B):
        end = int(lay.prefix_len[b]) + N
        for p in range(end, (end + ps - 1) // ps * ps):
            k8p[lay.slot(b, p)] = 0x7F
            v8p[lay.slot(b, p)] = 0x7F
        v8p[lay.slot(b, int(lay.prefix_len[b]) + leaf), :, 5] = 0x7F
    out, lse = _run_verify_fp8(inp, k8p, v8p)
    keep = [r for r in range(w.B * N) if r % N != leaf]
    rows, ro, rl = _oracle_verify_fp8(inp, k8, v8, range(w.B))
    assert_attention_close(out[keep], lse[keep], ro[keep], rl[keep], range(len(keep)))
    for b in range(w.B):
        assert not np.isfinite(out[b * N + leaf]).all()
    assert np.array_equal(out[keep], out_ref[keep])


def test_verify_fp8_bad_window_page_reaches_only_the_rows_that_see_it():
    """A window page id that points outside the cache (-1 for request 0's
    last window page, past the cache for request 1's) is reported as a bad
    slot and turns exactly the rows that see one of its keys NaN: with pages
    of 16 keys and depth-first numbering those are nodes 48..63. Every other
    row still matches the oracle. The prefixes end on a key-tile edge, so no
    prefix tile reaches the broken pages."""
    w = custom_workload("eagle2_p8192_n64", 64, B=2, prefix=[1024, 640], Hq=8, page_size=16)
    rng = np.random.default_rng(640)
    par = np.stack([random_tree(rng, w.N)[0] for _ in range(w.B)]).astype(np.int32)
    dep = np.stack([synth.depth_of(p) for p in par]).astype(np.int32)
    inp, k8, v8 = _verify_case(w, trees=(par, dep))
    lay, N, ps = inp.layout, w.N, w.page_size
    pt = lay.page_table.copy()
    num_pages = lay.num_slots // ps
    for b, bad in ((0, -1), (1, num_pages + 5)):
        last = (int(lay.prefix_len[b]) + N - 1) // ps
        assert last == (int(lay.prefix_len[b]) + 48) // ps          # keys 48..63 share the last page
        pt[b, last] = bad
    out, lse = _run_verify_fp8(inp, k8, v8, page_table=pt, expect_err=dts.DEV_BAD_SLOT)
    hit = [b * N + i for b in range(w.B) for i in range(48, N)]
    keep = [r for r in range(w.B * N) if r not in hit]
    rows, ro, rl = _oracle_verify_fp8(inp, k8, v8, range(w.B))
    assert_attention_close(out[keep], lse[keep], ro[keep], rl[keep], range(len(keep)))
    assert np.isnan(out[hit]).all() and np.isnan(lse[hit]).all()


# ---------------------------------------------------------------------------- draft lanes (R = K, W = (S-1) K)

def _lane(**kw):
    base = synth.LANE_WORKLOADS["lanes_eagle2_p8192_k8_s7"]
    return dataclasses.replace(base, name="lanes_fp8_t", index=300 + len(kw), **kw) if kw else base


def _run_lanes_fp8(li, rotate=True):
    torch = torch_cuda()
    lw = li.lw
    B, R, W = lw.B, lw.R, lw.W
    out, lse = _outputs(B * R, lw.Hq, lw.d)
    max_prefix = int(max(lw.prefix))
    ws = torch.empty(dts.tree_window_attention_workspace(B, R, W, lw.Hq, lw.Hkv, lw.d, max_prefix),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.tree_window_attention_fp8(_bf(li.q), _dev(li.k_cache), _dev(li.v_cache), _dev(li.layout.page_table),
                                  lw.page_size, _dev(li.prefix_len), max_prefix,
                                  _dev(np.asarray(li.mask, np.uint64).view(np.int64)),
                                  _dev(li.positions) if rotate else None, lw.rope_theta, out, lse, ws, W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def _oracle_lanes_fp8(li, rotate=True):
    lw = li.lw
    return OA.window_attention(li.q, li.k_cache, li.v_cache, li.layout.page_table, li.prefix_len, li.mask,
                               li.positions, lw.W, lw.Hkv, lw.rope_theta, page_size=lw.page_size,
                               q_rotated=not rotate, kv_fp8=True, q_fp8=True)


@pytest.mark.parametrize("kw", [
    dict(),                                                    # the EAGLE-2 batch's last drafting step, full size
    dict(B=3, K=4, S=5, prefix=[0, 129, 1000]),                # empty and ragged prefixes
    dict(B=2, K=8, S=9, prefix=[300, 64]),                     # W = 64
    dict(B=1, K=32, S=3, Hq=32, Hkv=2, prefix=[700]),          # R = 32, M = 512: two units
])
def test_lanes_fp8(kw):
    li = synth.make_lane_inputs(_lane(**kw), kv_fp8=True)
    rotate = bool(kw)                                          # full size: the query as already rotated
    out, lse = _run_lanes_fp8(li, rotate)
    ref_o, ref_l = _oracle_lanes_fp8(li, rotate)
    assert_attention_close(out, lse, ref_o, ref_l, range(li.lw.B * li.lw.R))


# ---------------------------------------------------------------------------- window write

def test_write_window_kv_fp8_matches_the_oracle():
    """V bytes equal the oracle's; a K byte equals it or, where the device's
    fp32 rotation and the oracle's exact one round to neighbouring bf16
    values across an E4M3 midpoint, is the neighbouring code (rare); no other
    slot changes."""
    torch = torch_cuda()
    w = synth.WORKLOADS["eagle2_p8192_n64"]
    inp = synth.make_inputs(w, with_cache=False, with_hidden=False)
    lay = inp.layout
    fill = 0x3C
    kc = torch.full((lay.num_slots, w.Hkv, w.d), fill, dtype=torch.uint8, device="cuda")
    vc = torch.full((lay.num_slots, w.Hkv, w.d), fill, dtype=torch.uint8, device="cuda")
    pos = (lay.prefix_len[:, None].astype(np.int64) + inp.depth).astype(np.int32)
    wl = torch.zeros(w.B * w.N, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.write_window_kv_fp8(_bf(inp.k_new), _bf(inp.v_new), _dev(pos), _dev(lay.page_table), w.page_size,
                            _dev(lay.prefix_len), kc, vc, w.rope_theta, write_locations=wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slots = wl.cpu().numpy()
    assert (slots == lay.write_locations).all()
    k_ref, v_ref = F8.window_kv_fp8(inp.k_new, inp.v_new, pos.reshape(-1), w.rope_theta)
    k_all, v_all = kc.cpu().numpy(), vc.cpu().numpy()
    assert (v_all[slots] == v_ref).all()
    kg = k_all[slots]
    diff = kg != k_ref
    assert diff.mean() < 1e-4, diff.mean()
    same_sign = (kg[diff] & 0x80) == (k_ref[diff] & 0x80)
    step = np.abs((kg[diff] & 0x7F).astype(int) - (k_ref[diff] & 0x7F).astype(int))
    assert same_sign.all() and (step == 1).all()
    untouched = np.ones(lay.num_slots, bool)
    untouched[slots] = False
    assert (k_all[untouched] == fill).all() and (v_all[untouched] == fill).all()


# ---------------------------------------------------------------------------- statuses

def test_fp8_calls_refuse_d64_and_small_workspaces():
    torch = torch_cuda()
    q = torch.zeros((4, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((128, 1, 64), dtype=torch.uint8, device="cuda")
    pt = torch.ones((1, 2), dtype=torch.int32, device="cuda")
    pl = torch.tensor([10], dtype=torch.int32, device="cuda")
    m = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    pos = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    out, lse = _outputs(4, 4, 64)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(dts.DtsError) as e:
        dts.tree_verify_attention_fp8(q, k, k, pt, 64, pl, 10, m, pos, 5e5, out, lse, ws)
    assert e.value.status == dts.ERR_UNSUPPORTED
    kn = torch.zeros((4, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dts.DtsError) as e:
        dts.write_window_kv_fp8(kn, kn, pos, pt, 64, pl, k, k, 5e5)
    assert e.value.status == dts.ERR_UNSUPPORTED
    q = torch.zeros((4, 4, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((128, 1, 128), dtype=torch.uint8, device="cuda")
    out, lse = _outputs(4, 4, 128)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dts.DtsError) as e:
        dts.tree_verify_attention_fp8(q, k, k, pt, 64, pl, 10, m, pos, 5e5, out, lse, small)
    assert e.value.status == dts.ERR_WORKSPACE
