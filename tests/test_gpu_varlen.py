"""GPU parity: fused attention over packed variable-length sequences
(rf_attn_fwd_varlen, fp32 SIMT and bf16 tcgen05 paths, with and without the
causal mask) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as I
from oracle import attention as A
from tests.helpers import Guarded, assert_bf16_close, assert_f32_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _cu(lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return torch.from_numpy(cu)


def _inputs(lens_q, lens_k, H, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    cast = (lambda t: t) if dtype == "f32" else (lambda t: t.to(torch.bfloat16))
    q = cast(torch.randn(tq, H, d, generator=g))
    k = cast(torch.randn(tk, H, d, generator=g))
    v = cast(torch.randn(tk, H, d, generator=g))
    return q, k, v, _cu(lens_q), _cu(lens_k)


def _run(rf, q, k, v, cu_q, cu_k, max_q, scale, causal):
    o = Guarded(tuple(q.shape), q.dtype)
    rf.rf_attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o.t, cu_q.cuda(), cu_k.cuda(), max_q, scale,
                          causal)
    assert rf.rf_get_device_status() == rf.RF_OK
    o.check("varlen output")
    return o.t.cpu()


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("lens", [[1, 127, 128, 129, 300, 0, 513], [640], [64, 64, 64]])
def test_bf16_self_attention(rf, lens, causal):
    q, k, v, cu, _ = _inputs(lens, lens, 4, 64, "bf16", seed=sum(lens) + causal)
    o = _run(rf, q, k, v, cu, cu, max(lens), 0.125, causal)
    ref = A.attention_varlen(q, k, v, cu, cu, 0.125, causal=bool(causal))
    assert_bf16_close(o, ref, f"bf16 varlen {lens} causal={causal}")


@pytest.mark.parametrize("causal", [0, 1])
def test_bf16_different_query_and_key_lengths(rf, causal):
    """Per sequence Lq != Lk (a prefill continuing a cache, or the reverse),
    including a sequence with no keys (zero rows) and one with no queries."""
    lq, lk = [10, 200, 7, 0, 130], [300, 50, 0, 40, 129]
    q, k, v, cu_q, cu_k = _inputs(lq, lk, 3, 64, "bf16", seed=11 + causal)
    o = _run(rf, q, k, v, cu_q, cu_k, max(lq), 0.125, causal)
    ref = A.attention_varlen(q, k, v, cu_q, cu_k, 0.125, causal=bool(causal))
    assert_bf16_close(o, ref, f"bf16 varlen cross causal={causal}")
    assert (o[210:217].float() == 0).all()      # the sequence without keys


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [0, 1])
def test_fp32(rf, d, causal):
    lq, lk = [3, 64, 65, 0, 100], [3, 70, 65, 5, 90]
    q, k, v, cu_q, cu_k = _inputs(lq, lk, 2, d, "f32", seed=d + causal)
    o = _run(rf, q, k, v, cu_q, cu_k, max(lq), d ** -0.5, causal)
    ref = A.attention_varlen(q, k, v, cu_q, cu_k, d ** -0.5, causal=bool(causal))
    assert_f32_close(o, ref, f"fp32 varlen d={d} causal={causal}")


def test_prefill_varlen_workload(rf):
    s = I.PREFILL_VARLEN
    q, k, v, cu = I.varlen_inputs(s)
    lens = (cu[1:] - cu[:-1]).tolist()
    o = _run(rf, q, k, v, cu, cu, max(lens), s.scale, 0)
    assert_bf16_close(o, A.attention_varlen(q, k, v, cu, cu, s.scale), "prefill varlen")


@pytest.mark.parametrize("causal", [0, 1])
def test_fixed_and_varlen_entry_points_agree(rf, causal):
    """Equal lengths: the packed call and rf_attn_fwd on the [B,H,L,d] layout
    give the same attention.  They run different kernels (the fixed layout's
    single-pass bf16 calls go to the prefill kernel, whose rescaling and
    summation order differ), so they agree within the bf16 tolerance, and
    each matches the oracle."""
    B, H, L = 3, 4, 300
    sh = I.AttnShape(B, H, H, L, L, 64, "bf16", seed=21)
    q4, k4, v4 = I.attention_inputs(sh)
    o4 = torch.empty_like(q4, device="cuda")
    rf.rf_attn_fwd(q4.cuda(), k4.cuda(), v4.cuda(), o4, sh.scale, causal)
    pack = lambda t: t.transpose(1, 2).reshape(B * L, H, 64).contiguous()
    cu = _cu([L] * B)
    o = _run(rf, pack(q4), pack(k4), pack(v4), cu, cu, L, sh.scale, causal)
    ref = pack(torch.from_numpy(A.attention(q4, k4, v4, sh.scale, causal=bool(causal))))
    assert_bf16_close(o, pack(o4.cpu()), "packed vs fixed layout")
    assert_bf16_close(o, ref, "packed vs oracle")
    assert_bf16_close(pack(o4.cpu()), ref, "fixed layout vs oracle")


def test_inconsistent_lengths_are_reported_not_followed(rf):
    """cu_seqlens that contradict total_q are caught by the kernel: the
    sequence is skipped, nothing outside O is written, and the status says
    so.  The host-side sizes are valid, so the call itself is accepted."""
    H, d = 2, 64
    q = torch.randn(20, H, d).to(torch.bfloat16).cuda()
    buf = torch.full((40, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[:20]
    cu_q = torch.tensor([0, 10, 30], dtype=torch.int32, device="cuda")   # 30 > total_q = 20
    cu_k = torch.tensor([0, 10, 20], dtype=torch.int32, device="cuda")
    rf.rf_attn_fwd_varlen(q, q, q, o, cu_q, cu_k, 20, 0.125, 0)
    assert rf.rf_get_device_status() == rf.RF_ERR_DEVICE_INPUT
    assert (buf[20:].float() == 7.0).all()
    assert rf.rf_get_device_status() == rf.RF_OK          # reading the status cleared it
