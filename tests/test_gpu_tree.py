"""GPU parity: build_tree_mask and verify_tree_greedy against the oracle,
bit-exact, through the C ABI."""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from oracle import tree as OT
from oracle import walk as OW
from tests.gpu_helpers import random_tree, torch_cuda

pytestmark = pytest.mark.gpu


def _mask_on_gpu(parents, depth, vc):
    torch = torch_cuda()
    B, N = parents.shape
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    mask = torch.full((B, N), -7, dtype=torch.int64, device=dev)
    pos = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    nt = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    ns = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dts.build_tree_mask(t(parents), t(depth), t(vc), mask, pos, nt, ns, err=err)
    torch.cuda.synchronize()
    return (mask.cpu().numpy().view(np.uint64), pos.cpu().numpy(), nt.cpu().numpy(), ns.cpu().numpy(),
            int(err.item()))


def _check_trees(parents, depth, vc):
    mask, pos, nt, ns, err = _mask_on_gpu(parents, depth, vc)
    assert err == 0
    for b in range(parents.shape[0]):
        m, p, t, s = OT.build_tree_mask(parents[b], depth[b], int(vc[b]))
        assert (mask[b] == m).all()
        assert (pos[b] == p).all()
        assert (nt[b] == t).all() and (ns[b] == s).all()


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_mask_workload_trees(name):
    w = synth.WORKLOADS[name]
    parents, depth = synth.make_trees(w, synth.streams(w.index)["tree"])
    vc = np.arange(w.B, dtype=np.int32) * 37 + 5
    _check_trees(parents, depth, vc)


@pytest.mark.parametrize("n", [1, 2, 5, 8, 16, 17, 31, 32, 33, 63, 64])
def test_mask_random_trees(n):
    rng = np.random.default_rng(1000 + n)
    B = 37
    ps, ds = zip(*[random_tree(rng, n) for _ in range(B)])
    _check_trees(np.array(ps), np.array(ds), rng.integers(0, 1 << 20, B).astype(np.int32))


def test_mask_chain_star_and_bit63():
    chain_p, chain_d = synth.chain_tree(64)
    star_p, star_d = synth.star_tree(64)
    parents = np.stack([chain_p, star_p])
    depth = np.stack([chain_d, star_d])
    mask, *_ = _mask_on_gpu(parents, depth, np.array([0, 9], np.int32))
    assert int(mask[0, 63]) == (1 << 64) - 1
    assert int(mask[1, 63]) == (1 << 63) | 1
    _check_trees(parents, depth, np.array([0, 9], np.int32))


def test_mask_invalid_trees_report():
    parents = np.array([[-1, 0, 0, 1], [-1, 0, 2, 1], [0, 0, 0, 0], [-1, 0, 1, 1]], np.int32)
    depth = np.array([[0, 1, 1, 2], [0, 1, 2, 2], [0, 1, 1, 1], [0, 1, 2, 3]], np.int32)
    for b, code in [(1, dts.DEV_BAD_PARENT), (2, dts.DEV_BAD_PARENT), (3, dts.DEV_BAD_DEPTH)]:
        mask, pos, nt, ns, err = _mask_on_gpu(parents[[0, b]], depth[[0, b]], np.array([3, 4], np.int32))
        assert err == code
        assert (mask[1] == 0).all() and (pos[1] == 4).all() and (nt[1] == -1).all() and (ns[1] == -1).all()
        m, p, t, s = OT.build_tree_mask(parents[0], depth[0], 3)      # the valid request is unaffected
        assert (mask[0] == m).all() and (nt[0] == t).all()


def _walk_on_gpu(parents, draft, argmax, use_links):
    torch = torch_cuda()
    B, N = parents.shape
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)).to(dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    path = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    tok = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if use_links:
        links = [OT.links(parents[b]) for b in range(B)]
        nt = np.stack([l[0] for l in links])
        ns = np.stack([l[1] for l in links])
        dts.verify_tree_greedy(t(draft), t(argmax), alen, path, tok, next_token=t(nt), next_sibling=t(ns), err=err)
    else:
        dts.verify_tree_greedy(t(draft), t(argmax), alen, path, tok, parents=t(parents), err=err)
    torch.cuda.synchronize()
    return alen.cpu().numpy(), path.cpu().numpy(), tok.cpu().numpy(), int(err.item())


def _check_walk(parents, draft, argmax):
    ref = OW.greedy_walk_batch(parents, draft, argmax)
    for use_links in (True, False):
        alen, path, tok, err = _walk_on_gpu(parents, draft, argmax, use_links)
        assert err == 0
        assert (alen == ref[0]).all()
        assert (path == ref[1]).all()
        assert (tok == ref[2]).all()


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_walk_workloads(name):
    w = synth.WORKLOADS[name]
    s = synth.streams(w.index)
    parents, depth = synth.make_trees(w, s["tree"])
    draft, argmax = synth.make_tokens(w, parents, s["tokens"])
    _check_walk(parents, draft, argmax)


@pytest.mark.parametrize("n", [1, 5, 8, 16, 17, 64])
def test_walk_random_with_duplicate_tokens(n):
    rng = np.random.default_rng(2000 + n)
    B = 64
    ps = np.array([random_tree(rng, n)[0] for _ in range(B)])
    draft = rng.integers(0, 3, (B, n)).astype(np.int32)     # tiny vocab: repeated sibling tokens
    argmax = rng.integers(0, 3, (B, n)).astype(np.int32)
    _check_walk(ps, draft, argmax)


def test_walk_chain_accepts_everything_and_examples(golden):
    for name in ("accept_0_2_5_6.txt", "chain_walk.txt"):
        g = golden(name)
        _check_walk(np.array([g["parents"]]), np.array([g["draft"]]), np.array([g["target_argmax"]]))
    p, _ = synth.chain_tree(64)
    argmax = np.arange(64, dtype=np.int32)
    draft = np.concatenate([[7], np.arange(63)]).astype(np.int32)
    alen, path, tok, err = _walk_on_gpu(p[None], draft[None], argmax[None], True)
    assert alen[0] == 64 and (path[0] == np.arange(64)).all()


def test_walk_bad_links_report():
    torch = torch_cuda()
    dev = "cuda"
    N = 4
    nt = torch.tensor([[1, -1, -1, -1]], dtype=torch.int32, device=dev)
    ns = torch.tensor([[-1, 2, 1, -1]], dtype=torch.int32, device=dev)   # 1 -> 2 -> 1: a cycle
    z = torch.zeros((1, N), dtype=torch.int32, device=dev)
    alen = torch.zeros(1, dtype=torch.int32, device=dev)
    path = torch.zeros((1, N), dtype=torch.int32, device=dev)
    tok = torch.zeros((1, N), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dts.verify_tree_greedy(z, z, alen, path, tok, next_token=nt, next_sibling=ns, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dts.DEV_BAD_LINK
    assert int(alen.item()) == 1 and path.cpu().tolist()[0] == [0, -1, -1, -1]
