"""Every entry point only enqueues work on the caller's stream, so a call can
be captured into a CUDA graph and replayed: the replay must reproduce the
eager call's bits.  (The programmatic dependent launches of the split-KV
merge, of the FP8 GEMM and of the latent-KV merge, and the cluster launches,
become graph nodes and edges.)"""
import pytest
import torch

import workloads as I
from tests.helpers import fp8_weight_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _paths(rf):
    """(name, outputs, call writing into outputs) for each path."""
    paths = []
    s = I.AttnShape(2, 32, 8, 1, 3000, 128, "bf16", seed=81)
    q, k, v = (t.cuda() for t in I.decode_inputs(s))
    ws = torch.empty(rf.rf_attn_decode_splitkv_workspace_size(2, 32, 8, 3000, 128, 0),
                     dtype=torch.uint8, device="cuda")
    od = torch.empty_like(q)
    paths.append(("decode", [od], lambda: rf.rf_attn_decode_splitkv(q, k, v, od, s.scale, ws, 0)))
    on = torch.empty_like(q)
    paths.append(("decode_noalloc", [on],
                  lambda: rf.rf_attn_decode_splitkv_noalloc(q, k, v, on, s.scale, 0)))

    b = I.AttnShape(2, 8, 8, 300, 300, 64, "bf16", seed=82)
    qb, kb, vb = (t.cuda() for t in I.attention_inputs(b))
    ob, oc = torch.empty_like(qb), torch.empty_like(qb)

    def prefill():
        rf.rf_attn_fwd(qb, kb, vb, ob, b.scale)
        rf.rf_attn_fwd(qb, kb, vb, oc, b.scale, 1)
    paths.append(("prefill", [ob, oc], prefill))

    f32 = I.AttnShape(1, 2, 2, 64, 256, 64, "f32", seed=83)
    qf, kf, vf = (t.cuda() for t in I.attention_inputs(f32))
    of = torch.empty_like(qf)
    paths.append(("prefill_f32", [of], lambda: rf.rf_attn_fwd(qf, kf, vf, of, f32.scale)))

    vs = I.VarlenShape(B=3, H=2, d=64, len_lo=1, len_hi=300, dtype="bf16", seed=84)
    qv, kv_, vv, cu = I.varlen_inputs(vs)
    qv, kv_, vv, cu = qv.cuda(), kv_.cuda(), vv.cuda(), cu.cuda()
    ov = torch.empty_like(qv)
    maxlen = int((cu[1:] - cu[:-1]).max().item())
    paths.append(("varlen", [ov],
                  lambda: rf.rf_attn_fwd_varlen(qv, kv_, vv, ov, cu, cu, maxlen, vs.scale, 1)))

    m = I.MoEShape(T=1000, D=2048, E=64, k=2, seed=85)
    x, w = (t.cuda() for t in I.moe_inputs(m))
    idx = torch.empty(m.T, m.k, dtype=torch.int32, device="cuda")
    wt = torch.empty(m.T, m.k, dtype=torch.float32, device="cuda")
    paths.append(("moe", [idx, wt], lambda: rf.rf_moe_gate_topk_softmax(x, w, m.k, idx, wt)))

    fs = I.FP8Shape(M=512, N=1024, K=2048, seed=86)
    X, W = (t.cuda() for t in I.fp8_inputs(fs))
    Wq, sw = fp8_weight_gpu(rf, W)
    wsf = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(fs.M, fs.N, fs.K), dtype=torch.uint8,
                      device="cuda")
    y = torch.empty(fs.M, fs.N, dtype=torch.bfloat16, device="cuda")
    paths.append(("fp8", [y], lambda: rf.rf_absmax_fp8_gemm(X, Wq, sw, y, wsf)))

    ml = I.MLAShape(B=2, Hq=128, Lk=700, seed=87)
    qm, cm = (t.cuda() for t in I.mla_inputs(ml))
    om1 = torch.empty(ml.B, ml.Hq, ml.d_v, dtype=torch.bfloat16, device="cuda")
    om3 = torch.empty_like(om1)
    wsm = torch.empty(rf.rf_mla_decode_workspace_size(ml.B, ml.Hq, ml.Lk, 576, 512, 3),
                      dtype=torch.uint8, device="cuda")

    def mla():
        rf.rf_mla_decode(qm, cm, om1, ml.scale, None, 1)       # one segment (cluster kernel)
        rf.rf_mla_decode(qm, cm, om3, ml.scale, wsm, 3)        # three segments + merge
    paths.append(("mla", [om1, om3], mla))
    return paths


def test_each_path_replays_from_a_cuda_graph(rf):
    for name, outs, call in _paths(rf):
        call()                                    # eager call (also does first-call set-up)
        torch.cuda.synchronize()
        ref = [o.clone() for o in outs]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        for o in outs:
            o.fill_(0)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        for a, r in zip(outs, ref):
            assert torch.equal(a, r), f"{name}: graph replay differs from the eager call"
    assert rf.rf_get_device_status() == rf.RF_OK
