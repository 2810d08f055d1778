"""The tree pass's bounded waits run out, and the kernel leaves cleanly.

With the test hook dts_test_stall_attention(1, budget) the pass's producer
issues no copy at all, so nothing in flight can touch shared or tensor memory
while the other roles wait on barriers that nothing will complete. Each such
wait gives up after the (shortened) budget, the roles leave in their abort
order (named-barrier arrivals, the drain of issued MMAs, the release of tensor
memory) and the call reports DTS_DEV_TIMEOUT in err_dev. The same process then
runs the normal call, whose every row must match the oracle: the context is
still usable and nothing of the stalled call stays behind.
"""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch
from oracle import attention as OA
from tests.gpu_helpers import assert_attention_close, bf16_to_f64, torch_cuda

pytestmark = pytest.mark.gpu


def _oracle(inp, rows=None):
    w = inp.w
    return OA.verify_attention(inp.q, inp.k_new, inp.v_new, inp.k_cache, inp.v_cache, inp.layout.page_table, inp.vc,
                               inp.parents, w.Hkv, w.rope_theta, page_size=w.page_size, rows=rows)


# llama8b and tiny: units merged by the merge pass; highconc: units of 64 rows
# merged inside the tree pass, whose merge a timed-out CTA skips
@pytest.mark.parametrize("name", ["llama8b_p4096_n8", "tiny_p128_n5", "highconc_b128_n16"])
def test_stalled_attention_reports_timeout_then_runs_normally(name):
    torch = torch_cuda()
    L = dts.lib()
    inp = synth.make_inputs(synth.WORKLOADS[name], with_hidden=False)
    db = DeviceBatch(inp, compact_attention_kv=False, fp8_layers=0)
    db.mask_step()
    db.window_kv_step()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    assert L.dts_test_stall_attention(1, 1 << 22) == dts.OK   # about 2 ms per wait
    try:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        db.attention_step()
        end.record()
        torch.cuda.synchronize()
        assert int(db.err.item()) == dts.DEV_TIMEOUT
        assert start.elapsed_time(end) < 1000.0                 # the waits gave up, well within a second
    finally:
        assert L.dts_test_stall_attention(0, 1 << 31) == dts.OK
    db.err.zero_()
    db.out.fill_(float("nan"))
    db.attention_step()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    w = inp.w
    # every row of up to 8 requests (the first, the last and six between)
    reqs = sorted(set(np.linspace(0, w.B - 1, min(w.B, 8)).astype(int).tolist()))
    rows = [(b, v) for b in reqs for v in range(w.N)]
    ref_o, ref_l = _oracle(inp, rows)
    out, lse = bf16_to_f64(db.out), db.lse2.cpu().numpy().astype(np.float64)
    assert_attention_close(out, lse, ref_o, ref_l, [b * w.N + v for b, v in rows])
