"""The allocation-free attention entry point.

dts_tree_verify_attention_static_ws serves callers that cannot allocate device
memory (a process whose own pool holds the whole GPU, a plugin without its
host's allocator, code that must not call cudaMalloc while it runs): it uses a
fixed 64 MiB array inside the library instead of a caller workspace. Here it
is called through the C ABI twice in a row and must agree with the regular
entry point (which takes a caller workspace) within the attention tolerances;
shapes whose workspace exceeds the array are refused. This file is collected
last so that a failure here stops a -x run only after every other test ran.
"""
import numpy as np
import pytest

import draft_tree_speculative_gb300 as dts
from draft_tree_speculative_gb300 import synth
from draft_tree_speculative_gb300.step import DeviceBatch
from tests.gpu_helpers import LSE_ATOL, OUT_ATOL, OUT_RTOL, bf16_to_f64, torch_cuda

pytestmark = pytest.mark.gpu


def _static_call(db, out, lse2):
    dts.tree_verify_attention_static_ws(db.q, db.k_cache, db.v_cache, db.page_table, db.page_size, db.prefix_len,
                                        db.max_prefix, db.mask, db.positions, db.w.rope_theta, out, lse2,
                                        err=db.err, N=db.N)


@pytest.mark.parametrize("name", ["llama8b_p4096_n8", "highconc_b128_n16"])
def test_static_workspace_matches_caller_workspace(name):
    torch = torch_cuda()
    inp = synth.make_inputs(synth.WORKLOADS[name], with_hidden=False)
    db = DeviceBatch(inp, compact_attention_kv=False, fp8_layers=0)
    db.mask_step()
    db.window_kv_step()
    db.attention_step()                       # the regular entry point, caller workspace
    torch.cuda.synchronize()
    ref_o, ref_l = bf16_to_f64(db.out), db.lse2.cpu().numpy().astype(np.float64)
    for _ in range(2):                        # two calls in a row share the static array
        out = torch.full_like(db.out, float("nan"))
        lse2 = torch.full_like(db.lse2, float("nan"))
        _static_call(db, out, lse2)
        torch.cuda.synchronize()
        assert int(db.err.item()) == 0
        o, l = bf16_to_f64(out), lse2.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(o - ref_o) <= OUT_ATOL + OUT_RTOL * np.abs(ref_o))
        assert np.all(np.abs(l - ref_l) <= LSE_ATOL)


def test_static_workspace_refuses_shapes_beyond_its_size():
    torch = torch_cuda()
    w = synth.WORKLOADS["eagle2_p8192_n64"]       # needs more than 64 MiB of workspace
    assert dts.tree_verify_attention_workspace(w.B, w.N, w.Hq, w.Hkv, w.d, 8192) > (64 << 20)
    L = dts.lib()
    st = L.dts_tree_verify_attention_static_ws(None, None, None, 1 << 20, None, 200, 64, None, 8192, None, None,
                                               5e5, w.B, w.N, w.Hq, w.Hkv, w.d, 0.0, None, None, None,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == dts.ERR_WORKSPACE
