"""Every fused path is deterministic: the same inputs give the same bits on
every call, also when the calls are interleaved with the other paths (which
changes what sits in L2 and how the CTAs race).  A lost ordering between
cooperating CTAs or kernels -- the MoE gate's cluster exchange of partial
scores, the split-KV merge by the last CTA to finish a sequence, the FP8
GEMM reading a block of codes before its quantiser warps published it -- would show up as
a call whose bits differ."""
import pytest
import torch

import workloads as I
from tests.helpers import fp8_weight_gpu

pytestmark = pytest.mark.gpu

REPEATS = 12


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _calls(rf):
    """(name, call returning a fresh output) for each path on a mid-size input."""
    calls = []
    s = I.AttnShape(2, 32, 8, 1, 3000, 128, "bf16", seed=71)
    q, k, v = (t.cuda() for t in I.decode_inputs(s))
    ws = torch.empty(rf.rf_attn_decode_splitkv_workspace_size(2, 32, 8, 3000, 128, 0),
                     dtype=torch.uint8, device="cuda")

    def decode():
        o = torch.empty_like(q)
        rf.rf_attn_decode_splitkv(q, k, v, o, s.scale, ws, 0)
        return [o]
    calls.append(("decode", decode))

    b = I.AttnShape(2, 8, 8, 640, 640, 64, "bf16", seed=72)
    qb, kb, vb = (t.cuda() for t in I.attention_inputs(b))

    def prefill():
        o = torch.empty_like(qb)
        rf.rf_attn_fwd(qb, kb, vb, o, b.scale)
        oc = torch.empty_like(qb)
        rf.rf_attn_fwd(qb, kb, vb, oc, b.scale, 1)
        return [o, oc]
    calls.append(("prefill", prefill))

    m = I.MoEShape(T=4000, D=4096, E=64, k=2, seed=73)
    x, w = (t.cuda() for t in I.moe_inputs(m))

    def moe():
        idx = torch.empty(m.T, m.k, dtype=torch.int32, device="cuda")
        wt = torch.empty(m.T, m.k, dtype=torch.float32, device="cuda")
        rf.rf_moe_gate_topk_softmax(x, w, m.k, idx, wt)
        return [idx, wt]
    calls.append(("moe", moe))

    f = I.FP8Shape(M=1024, N=2048, K=4096, seed=74)
    X, W = (t.cuda() for t in I.fp8_inputs(f))
    Wq, sw = fp8_weight_gpu(rf, W)
    wsf = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(f.M, f.N, f.K), dtype=torch.uint8,
                      device="cuda")

    def fp8():
        y = torch.empty(f.M, f.N, dtype=torch.bfloat16, device="cuda")
        rf.rf_absmax_fp8_gemm(X, Wq, sw, y, wsf)
        return [y]
    calls.append(("fp8", fp8))
    return calls


def test_repeated_and_interleaved_calls_give_identical_bits(rf):
    calls = _calls(rf)
    first = {name: call() for name, call in calls}
    for r in range(REPEATS):
        order = calls if r % 2 == 0 else calls[::-1]
        for name, call in order:
            outs = call()
            for a, b in zip(first[name], outs):
                assert torch.equal(a, b), f"{name}: call {r + 1} differs from the first"
    assert rf.rf_get_device_status() == rf.RF_OK
