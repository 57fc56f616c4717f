"""rf_attn_decode_splitkv_noalloc: the split-KV decode for callers that cannot
give the library device memory (its partial states live in a scratch array
built into the library).  Through the C ABI, on consecutive calls (whatever
the previous call left in the shared scratch), its output must equal the
workspace-taking rf_attn_decode_splitkv bit for bit (same kernels, same
segments, only the scratch memory differs) and match the fp64 oracle within
the decode tolerance; requests whose partial states do not fit the scratch
are refused with RF_ERR_WORKSPACE.

This file is collected last on purpose, and it sets up everything it needs
itself, so it passes both alone in a fresh process and after the others."""
import pytest
import torch

import workloads as I
from oracle import attention as A
from tests.helpers import Guarded, assert_bf16_close

pytestmark = pytest.mark.gpu


def _reference(rf, q, k, v, scale, splits):
    B, Hq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    o = torch.full_like(q, float("nan"))
    ws = torch.empty(rf.rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, d, splits),
                     dtype=torch.uint8, device="cuda")
    rf.rf_attn_decode_splitkv(q, k, v, o, scale, ws, splits)
    return o


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import cascaded_reductions_loop_gb300 as rf

    cases = [(I.AttnShape(4, 32, 8, 1, 3000, 128, "bf16", seed=501), 0),
             (I.AttnShape(2, 16, 2, 1, 777, 128, "bf16", seed=502), 5),
             (I.AttnShape(3, 8, 8, 1, 1, 128, "bf16", seed=504), 0),
             (I.AttnShape(4, 32, 8, 1, 3000, 128, "bf16", seed=503), 0)]
    for sh, splits in cases:          # consecutive calls share (and overwrite) the scratch
        q_h, k_h, v_h = I.decode_inputs(sh)
        q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
        o = Guarded(tuple(q.shape), torch.bfloat16)
        rf.rf_attn_decode_splitkv_noalloc(q, k, v, o.t, sh.scale, splits)
        ref = _reference(rf, q, k, v, sh.scale, splits)
        assert rf.rf_get_device_status() == rf.RF_OK
        o.check("noalloc output")
        what = f"noalloc {sh.B}x{sh.Hq}x{sh.Lk} splits={splits}"
        assert torch.equal(o.t, ref), f"{what}: differs from the workspace entry point"
        assert_bf16_close(o.t.cpu(), A.decode_attention(q_h, k_h, v_h, sh.scale), what)


def test_noalloc_refuses_requests_beyond_its_scratch():
    import cascaded_reductions_loop_gb300 as rf

    B, Hq, Hkv, Lk, d = 32, 32, 8, 32768, 128
    splits = 1024                     # partial states of 32*32*1024*(128+2)*4 B > 16 MiB
    assert rf.rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, d, splits) > \
        rf.RF_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Hkv, 16, d, dtype=torch.bfloat16, device="cuda")   # never read
    o = torch.empty_like(q)
    status = rf.lib.rf_attn_decode_splitkv_noalloc(
        q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), B, Hq, Hkv, Lk, d, 0.088,
        splits, None)
    assert status == rf.RF_ERR_WORKSPACE
