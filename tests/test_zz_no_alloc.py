"""The allocation-free attention entry point.

dts_tree_verify_attention_static_ws serves callers that cannot allocate device
memory (a process whose own pool holds the whole GPU, a plugin without its
host's allocator, code that must not call cudaMalloc while it runs): it uses a
fixed 64 MiB array inside the library instead of a caller workspace. Here it
is called through the C ABI twice in a row and must agree with the regular
entry point (which takes a caller workspace) and with the oracle within the
attention tolerances; shapes whose workspace exceeds the array are refused.
This file is collected last so that a failure here stops a -x run only after
every other test ran.
"""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch
from oracle import attention as OA
from tests.gpu_helpers import LSE_ATOL, OUT_ATOL, OUT_RTOL, assert_attention_close, bf16_to_f64, torch_cuda

pytestmark = pytest.mark.gpu


def _static_call(db, out, lse2):
    dts.tree_verify_attention_static_ws(db.q, db.k_cache, db.v_cache, db.page_table, db.page_size, db.prefix_len,
                                        db.max_prefix, db.mask, db.positions, db.w.rope_theta, out, lse2,
                                        err=db.err, N=db.N)


@pytest.mark.parametrize("name", ["llama8b_p4096_n8", "eagle2_p8192_n64", "highconc_b128_n16"])
def test_static_workspace_matches_caller_workspace(name):
    torch = torch_cuda()
    inp = synth.make_inputs(synth.WORKLOADS[name], with_hidden=False)
    db = DeviceBatch(inp, compact_attention_kv=False, fp8_layers=0)
    db.mask_step()
    db.window_kv_step()
    db.attention_step()                       # the regular entry point, caller workspace
    torch.cuda.synchronize()
    ref_o, ref_l = bf16_to_f64(db.out), db.lse2.cpu().numpy().astype(np.float64)
    # the oracle on every row of a few requests (all of them for the small batch)
    w = inp.w
    reqs = range(w.B) if w.B <= 8 else (0, w.B // 2, w.B - 1)
    rows = [(b, v) for b in reqs for v in range(w.N)]
    or_o, or_l = OA.verify_attention(inp.q, inp.k_new, inp.v_new, inp.k_cache, inp.v_cache, inp.layout.page_table,
                                     inp.vc, inp.parents, w.Hkv, w.rope_theta, page_size=w.page_size, rows=rows)
    flat = [b * w.N + v for b, v in rows]
    for _ in range(2):                        # two calls in a row share the static array
        out = torch.full_like(db.out, float("nan"))
        lse2 = torch.full_like(db.lse2, float("nan"))
        _static_call(db, out, lse2)
        torch.cuda.synchronize()
        assert int(db.err.item()) == 0
        o, l = bf16_to_f64(out), lse2.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(o - ref_o) <= OUT_ATOL + OUT_RTOL * np.abs(ref_o))
        assert np.all(np.abs(l - ref_l) <= LSE_ATOL)
        assert_attention_close(o, l, or_o, or_l, flat)


def test_static_workspace_refuses_shapes_beyond_its_size():
    torch = torch_cuda()
    w = synth.WORKLOADS["eagle2_p8192_n64"]
    B = 2 * w.B                                   # twice eagle2's batch needs more than 64 MiB
    assert dts.tree_verify_attention_workspace(B, w.N, w.Hq, w.Hkv, w.d, 8192) > (64 << 20)
    L = dts.lib()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")   # valid pointers; nothing is launched
    p = buf.data_ptr()
    st = L.dts_tree_verify_attention_static_ws(p, p, p, 1 << 20, p, 200, 64, p, 8192, p, p, 5e5, B, w.N, w.Hq,
                                               w.Hkv, w.d, 0.0, p, p, None, torch.cuda.current_stream().cuda_stream)
    assert st == dts.ERR_WORKSPACE
