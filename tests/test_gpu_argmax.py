"""GPU parity: the target's row argmax and the walk fed by it, against the
oracle, bit-exact, through the C ABI."""
import math

import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from oracle import argmax as OA
from oracle import walk as OW
from tests.gpu_helpers import torch_cuda

pytestmark = pytest.mark.gpu


def _argmax_gpu(x_host, stride_pad=0, offset=0):
    """Row argmax of x_host [rows][vocab] on the GPU, the rows laid out with
    row stride vocab + stride_pad, starting `offset` floats into the buffer."""
    torch = torch_cuda()
    rows, vocab = x_host.shape
    stride = vocab + stride_pad
    buf = torch.full((offset + rows * stride + 4,), float("nan"), dtype=torch.float32, device="cuda")
    view = buf[offset: offset + rows * stride].view(rows, stride)[:, :vocab]
    view.copy_(torch.from_numpy(x_host))
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(8, dts.target_argmax_workspace(rows, vocab)), dtype=torch.uint8, device="cuda")
    dts.target_argmax(view, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _rows_with_specials(rng, rows, vocab):
    x = rng.integers(-3, 4, size=(rows, vocab)).astype(np.float32)       # many ties
    x[rng.random((rows, vocab)) < 0.3] = rng.standard_normal(1)[0]
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 3.0], np.float32)
    k = max(1, vocab // 50)
    for r in range(rows):
        if rng.random() < 0.5:
            idx = rng.integers(0, vocab, k)
            x[r, idx] = rng.choice(specials, k)
    return x


@pytest.mark.parametrize("vocab", [1, 3, 4, 5, 97, 1000, 16383, 16384, 16385, 40001])
def test_argmax_ties_and_specials(vocab):
    rng = np.random.default_rng(300 + vocab)
    x = _rows_with_specials(rng, 9, vocab)
    assert (_argmax_gpu(x) == OA.row_argmax(x)).all()


@pytest.mark.parametrize("pad, offset", [(0, 0), (4, 0), (3, 0), (0, 1), (7, 2)])
def test_argmax_strided_and_unaligned_rows(pad, offset):
    """Aligned rows take the float4 path; a row stride or start off the 16-byte
    grid takes the scalar path: both agree with the oracle."""
    rng = np.random.default_rng(310 + pad * 10 + offset)
    x = _rows_with_specials(rng, 13, 20000)
    assert (_argmax_gpu(x, pad, offset) == OA.row_argmax(x)).all()


def test_argmax_all_nan_and_all_equal_rows():
    x = np.zeros((4, 3000), np.float32)
    x[1] = np.nan
    x[2] = -np.inf
    x[3, 2999] = np.nan
    assert _argmax_gpu(x).tolist() == OA.row_argmax(x).tolist() == [0, 0, 0, 2999]


def test_argmax_normal_rows_and_signed_zero_ties():
    rng = np.random.default_rng(320)
    x = rng.standard_normal((64, 128256), dtype=np.float32)
    x[5, :] = -1.0
    x[5, 77] = -0.0
    x[5, 70] = 0.0                         # -0 == +0: the lower index wins
    assert (_argmax_gpu(x) == OA.row_argmax(x)).all()


def _fused(inp, logits_host):
    torch = torch_cuda()
    w = inp.w
    B, N = w.B, w.N
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    logits = t(logits_host)
    arg = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    alen = torch.zeros(B, dtype=torch.int32, device="cuda")
    path = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(dts.target_argmax_workspace(B * N, w.vocab), dtype=torch.uint8, device="cuda")
    dts.verify_tree_greedy_logits(t(inp.draft), logits, arg, alen, path, tok, ws, parents=t(inp.parents), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return arg.cpu().numpy(), alen.cpu().numpy(), path.cpu().numpy(), tok.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny_p128_n5", "eagle2_p8192_n64", "highconc_b128_n16"])
def test_fused_walk_on_workload_logits(name):
    """The workload's full-size logits (vocab 128256 for the large ones): the
    argmax is the planted target, and the fused walk equals the oracle's."""
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, with_cache=False, with_hidden=False)
    logits = synth.target_logits(w, inp.target_argmax)
    arg, alen, path, tok = _fused(inp, logits)
    ref_arg, ref_alen, ref_path, ref_tok = OA.greedy_walk_from_logits(inp.parents, inp.draft, logits)
    assert (ref_arg == inp.target_argmax).all()
    assert (arg == ref_arg).all()
    assert (alen == ref_alen).all() and (path == ref_path).all() and (tok == ref_tok).all()


def test_fused_walk_with_ties_between_siblings():
    """Rows whose argmax needs the tie rule feed the walk: the fused call
    matches the oracle's argmax-then-walk on every request."""
    rng = np.random.default_rng(330)
    w = synth.WORKLOADS["llama8b_p4096_n8"]
    inp = synth.make_inputs(w, with_cache=False, with_hidden=False)
    vocab = w.vocab
    logits = rng.integers(-2, 3, size=(w.B * w.N, vocab)).astype(np.float32)
    logits[:, :6] = 5.0                          # the maximum ties at tokens 0..5: token 0 wins
    draft = inp.draft.copy()
    draft[:, 1:] = rng.integers(0, 2, size=(w.B, w.N - 1))
    inp.draft = draft
    arg, alen, path, tok = _fused(inp, logits)
    ref_arg, ref_alen, ref_path, ref_tok = OA.greedy_walk_from_logits(inp.parents, draft, logits)
    assert (ref_arg == 0).all() and (arg == ref_arg).all()
    assert (alen == ref_alen).all() and (path == ref_path).all() and (tok == ref_tok).all()
    assert ref_alen.max() > 1
