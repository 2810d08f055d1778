"""GPU parity: compact_window_rows and compact_rows against the oracle, bit-exact."""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch
from oracle import compact as OC
from oracle import walk as OW
from tests.gpu_helpers import torch_cuda

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().cpu().numpy()


def test_highconc_full_compaction_64_fp8_buffers_and_hidden():
    """The high-concurrency workload: 32 layers x {K, V} fp8 buffers, the
    attention layer's bf16 K/V and bf16 hidden rows, after a real walk."""
    torch = torch_cuda()
    w = synth.WORKLOADS["highconc_b128_n16"]
    inp = synth.make_inputs(w)
    db = DeviceBatch(inp)
    db.mask_step()
    db.window_kv_step()
    db.walk_step()
    torch.cuda.synchronize()
    alen, path = _np(db.accept_len), _np(db.accepted_path)
    ref = OW.greedy_walk_batch(inp.parents, inp.draft, inp.target_argmax)
    assert (alen == ref[0]).all() and (path == ref[1]).all()
    assert alen.max() > 1
    wl = inp.layout.write_locations
    before = [_np(b)[wl] for b in db.fp8_buffers]
    kv_before = [_np(db.k_cache.view(torch.int16)), _np(db.v_cache.view(torch.int16))]
    hid_before = _np(db.hidden.view(torch.int16))
    db.compact_step()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    # oracle on the window rows: re-index the window slots as 0..B*N-1
    local_wl = np.arange(w.B * w.N)
    want = OC.compact_window_rows(before, local_wl, path, alen)
    for k, buf in enumerate(db.fp8_buffers):
        got = _np(buf)
        assert (got[wl] == want[k]).all()
        mask = np.ones(got.shape[0], bool)
        mask[wl] = False
        assert not got[mask].any()          # nothing outside the window was touched
    for t_before, t in zip(kv_before, (db.k_cache, db.v_cache)):
        want_kv, = OC.compact_window_rows([t_before], wl, path, alen)
        assert (_np(t.view(torch.int16)) == want_kv).all()
    want_h = OC.compact_hidden_rows(hid_before, path, alen)
    assert (_np(db.hidden.view(torch.int16)) == want_h).all()
    assert (_np(db.positions) == OC.compact_positions(inp.vc, w.N)).all()


def _run_compact(table_entries, wl, path, alen, B, N):
    torch = torch_cuda()
    table = dts.make_kv_table(table_entries)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.compact_window_rows(table, torch.from_numpy(wl).cuda(), torch.from_numpy(path).cuda(),
                            torch.from_numpy(alen).cuda(), err=err)
    torch.cuda.synchronize()
    return int(err.item())


@pytest.mark.parametrize("row_bytes", [4, 8, 12, 16, 1024, 2052])
def test_overlapping_path_and_row_widths(row_bytes):
    """path [0, 2, 3]: slot 2 is read for t=1 before it is written for t=2."""
    torch = torch_cuda()
    rng = np.random.default_rng(row_bytes)
    B, N = 2, 4
    slots = 16
    host = rng.integers(0, 256, (slots, row_bytes), dtype=np.uint8)
    buf = torch.from_numpy(host.copy()).cuda()
    wl = np.array([4, 5, 6, 7, 9, 10, 11, 12], np.int64)
    path = np.array([[0, 2, 3, -1], [0, 1, 3, -1]], np.int32)
    alen = np.array([3, 3], np.int32)
    err = _run_compact([(buf, row_bytes, slots, row_bytes)], wl, path, alen, B, N)
    assert err == 0
    want, = OC.compact_window_rows([host], wl, path, alen)
    assert (_np(buf) == want).all()


def test_aliased_buffers_move_once():
    """A buffer listed twice, and a value view inside a key row (same stride,
    leading bytes), are moved once; a partial overlap is refused."""
    torch = torch_cuda()
    rng = np.random.default_rng(3)
    slots, row = 12, 64
    host = rng.integers(0, 256, (slots, row), dtype=np.uint8)
    buf = torch.from_numpy(host.copy()).cuda()
    wl = np.array([3, 4, 5, 6], np.int64)
    path = np.array([[0, 2, 3, -1]], np.int32)
    alen = np.array([3], np.int32)
    entries = [(buf, row, slots, row), (buf, row, slots, row), (buf.data_ptr(), row, slots, 32)]
    assert _run_compact(entries, wl, path, alen, 1, 4) == 0
    want, = OC.compact_window_rows([host], wl, path, alen)
    assert (_np(buf) == want).all()
    # partial overlap: [0, 64) and [32, 96) with the same stride
    big = torch.zeros((slots, 128), dtype=torch.uint8, device="cuda")
    entries = [(big, 128, slots, 64), (big.data_ptr() + 32, 128, slots, 64)]
    assert _run_compact(entries, wl, path, alen, 1, 4) == dts.DEV_BAD_BUFFER


def test_bad_path_and_slot_are_reported():
    torch = torch_cuda()
    slots, row = 8, 16
    buf = torch.zeros((slots, row), dtype=torch.uint8, device="cuda")
    wl = np.array([0, 1, 2, 3], np.int64)
    assert _run_compact([(buf, row, slots, row)], wl, np.array([[0, 2, 1, -1]], np.int32),
                        np.array([3], np.int32), 1, 4) == dts.DEV_BAD_PATH
    wl_bad = np.array([0, 1, 2, 99], np.int64)
    assert _run_compact([(buf, row, slots, row)], wl_bad, np.array([[0, 3, -1, -1]], np.int32),
                        np.array([2], np.int32), 1, 4) == dts.DEV_BAD_SLOT


def test_compact_rows_hidden_and_positions():
    torch = torch_cuda()
    rng = np.random.default_rng(9)
    B, N, H = 5, 16, 4096
    hid = rng.integers(-30000, 30000, (B * N, H), dtype=np.int16)
    paths, alens = [], []
    for b in range(B):
        k = int(rng.integers(1, 6))
        p = np.sort(rng.choice(np.arange(1, N), k - 1, replace=False))
        row = np.full(N, -1, np.int32)
        row[:k] = np.concatenate([[0], p])
        paths.append(row)
        alens.append(k)
    path = np.array(paths, np.int32)
    alen = np.array(alens, np.int32)
    vc = rng.integers(0, 10000, B).astype(np.int32)
    h = torch.from_numpy(hid.copy()).cuda()
    pos = torch.full((B, N), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dts.compact_rows(h, pos, torch.from_numpy(vc).cuda(), torch.from_numpy(path).cuda(),
                     torch.from_numpy(alen).cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert (_np(h) == OC.compact_hidden_rows(hid, path, alen)).all()
    assert (_np(pos) == OC.compact_positions(vc, N)).all()
