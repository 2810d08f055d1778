"""GPU parity: sampled draws (Gumbel-max keyed by position) and the walk over
them, against the oracle, bit-exact, through the C ABI."""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from oracle import sampling as OS
from tests.gpu_helpers import torch_cuda

pytestmark = pytest.mark.gpu


def _dev(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _draws_gpu(logits, vc, depth, temp, seed, pad=0, offset=0):
    torch = torch_cuda()
    B, N = depth.shape
    rows, vocab = logits.shape
    stride = vocab + pad
    buf = torch.full((offset + rows * stride + 4,), float("nan"), dtype=torch.float32, device="cuda")
    view = buf[offset: offset + rows * stride].view(rows, stride)[:, :vocab]
    view.copy_(torch.from_numpy(logits))
    draws = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(8, dts.target_argmax_workspace(rows, vocab)), dtype=torch.uint8, device="cuda")
    dts.sample_draws(view, _dev(np.asarray(vc, np.int32)), _dev(depth.astype(np.int32)),
                     _dev(np.asarray(temp, np.float32)), _dev(np.asarray(seed, np.uint64).view(np.int64)), draws, ws)
    torch.cuda.synchronize()
    return draws.cpu().numpy()


@pytest.mark.parametrize("vocab", [7, 1000, 16385, 40001])
def test_draws_bit_exact(vocab):
    rng = np.random.default_rng(400 + vocab)
    B, N = 3, 5
    logits = rng.standard_normal((B * N, vocab)).astype(np.float32)
    logits[4, vocab // 2] = np.nan                        # a NaN wins its row
    depth = rng.integers(0, 4, size=(B, N))
    vc = [0, 1234, 2 ** 30]
    temp = [1.0, 0.35, 4.0]
    seed = [0, 2 ** 64 - 1, 0x0123456789ABCDEF]
    got = _draws_gpu(logits, vc, depth, temp, seed)
    ref = OS.sampled_draws(logits, vc, depth, temp, seed)
    assert (got == ref).all()


@pytest.mark.parametrize("pad, offset", [(3, 0), (0, 1), (5, 2)])
def test_draws_on_unaligned_rows(pad, offset):
    rng = np.random.default_rng(410 + pad + offset)
    B, N, vocab = 2, 4, 20001
    logits = rng.standard_normal((B * N, vocab)).astype(np.float32)
    depth = rng.integers(0, 3, size=(B, N))
    args = ([5, 77], depth, [0.8, 1.3], [99, 2 ** 40 + 3])
    got = _draws_gpu(logits, *args, pad=pad, offset=offset)
    assert (got == OS.sampled_draws(logits, *args)).all()


def test_non_positive_temperature_is_argmax():
    rng = np.random.default_rng(420)
    B, N, vocab = 3, 4, 3000
    logits = rng.standard_normal((B * N, vocab)).astype(np.float32)
    depth = np.tile(np.arange(N), (B, 1))
    temp = [0.0, -1.0, np.nan]
    got = _draws_gpu(logits, [1, 2, 3], depth, temp, [1, 2, 3])
    assert got.reshape(-1).tolist() == np.argmax(logits, axis=1).tolist()
    assert (got == OS.sampled_draws(logits, [1, 2, 3], depth, temp, [1, 2, 3])).all()


def test_sampled_walk_on_workload_shape():
    """The EAGLE-2 batch's trees over the full vocabulary (128256): the draws of
    two requests (128 rows) and their walks equal the oracle's; every request's
    draws are computed in the same call."""
    torch = torch_cuda()
    w = synth.WORKLOADS["eagle2_p8192_n64"]
    inp = synth.make_inputs(w, with_cache=False, with_hidden=False)
    logits = synth.target_logits(w, inp.target_argmax)
    B, N = w.B, w.N
    temp = np.full(B, 0.9, np.float32)
    seed = (np.arange(B, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15)) + np.uint64(7)
    draws = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    alen = torch.zeros(B, dtype=torch.int32, device="cuda")
    path = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(dts.target_argmax_workspace(B * N, w.vocab), dtype=torch.uint8, device="cuda")
    dts.verify_tree_sampled(_dev(inp.draft), _dev(logits), _dev(inp.vc), _dev(inp.depth), _dev(temp),
                            _dev(seed.view(np.int64)), draws, alen, path, tok, ws, parents=_dev(inp.parents), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    d, a, p, t = draws.cpu().numpy(), alen.cpu().numpy(), path.cpu().numpy(), tok.cpu().numpy()
    for b in (0, 17):
        rows = slice(b * N, (b + 1) * N)
        ref = OS.sampled_walk(inp.parents[b: b + 1], inp.draft[b: b + 1], logits[rows], inp.vc[b: b + 1],
                              inp.depth[b: b + 1], temp[b: b + 1], seed[b: b + 1])
        assert (d[b] == ref[0][0]).all()
        assert a[b] == ref[1][0] and (p[b] == ref[2][0]).all() and (t[b] == ref[3][0]).all()
