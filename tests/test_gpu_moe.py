"""GPU parity: fused MoE gate (tcgen05 scores, top-k, softmax) against the
fp64 oracle, through the C ABI.  Indices must match bit for bit."""
import numpy as np
import pytest
import torch

import workloads as I
from oracle import moe_gate as G
from tests.helpers import Guarded, MOE_W_ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(rf, x, w, k):
    T = x.shape[0]
    idx = Guarded((T, k), torch.int32, fill=-1)
    wts = Guarded((T, k), torch.float32)
    rf.rf_moe_gate_topk_softmax(x.cuda(), w.cuda(), k, idx.t, wts.t)
    assert rf.rf_get_device_status() == rf.RF_OK
    idx.check("expert indices")
    wts.check("expert weights")
    return idx.t.cpu().numpy(), wts.t.cpu().numpy()


def _check(x, w, k, idx, wts, what):
    ref_idx, ref_w, scores = G.moe_gate(x, w, k)
    mism = np.nonzero((idx != ref_idx).any(axis=1))[0]
    assert mism.size == 0, f"{what}: {mism.size} tokens with different experts, e.g. {mism[:5]}"
    assert np.abs(wts - ref_w).max() <= MOE_W_ABS, f"{what}: weights"
    return scores


def test_moe_gate_full(rf):
    s = I.MOE_GATE
    x, w = I.moe_inputs(s)
    idx, wts = _run(rf, x, w, s.k)
    scores = _check(x, w, s.k, idx, wts, "MoE 8192x4096x64")
    # the tie-break is exercised at this size
    sel2 = np.take_along_axis(scores, idx[:, 1:2].astype(np.int64), axis=1)
    assert ((scores == sel2).sum(axis=1) > 1).sum() > 10


@pytest.mark.parametrize("T,D,k", [(300, 256, 2), (1, 64, 1), (129, 1024, 4), (64, 4096, 8),
                                   (513, 200, 2), (256, 2048, 3), (100, 8, 2), (4000, 4096, 2),
                                   (777, 65536, 2)])
def test_moe_gate_small(rf, T, D, k):
    x, w = I.moe_inputs(I.MoEShape(T=T, D=D, E=64, k=k, seed=T + D + k))
    idx, wts = _run(rf, x, w, k)
    _check(x, w, k, idx, wts, f"MoE {T}x{D} k={k}")


def _run_de(rf, x, w, k):
    """The same call with W_gate given dim-major, [D][E]."""
    T = x.shape[0]
    idx = Guarded((T, k), torch.int32, fill=-1)
    wts = Guarded((T, k), torch.float32)
    w_de = Guarded(tuple(w.t().shape), torch.bfloat16)
    w_de.t.copy_(w.t())
    rf.rf_moe_gate_topk_softmax_ex(x.cuda(), w_de.t, k, rf.RF_GATE_W_DE, idx.t, wts.t)
    assert rf.rf_get_device_status() == rf.RF_OK
    idx.check("expert indices")
    wts.check("expert weights")
    w_de.check("W_gate (read only)")
    return idx.t.cpu().numpy(), wts.t.cpu().numpy()


def test_moe_gate_full_dim_major(rf):
    """The full workload with W_gate in the [D][E] layout of the problem
    statement (x @ W_gate): indices bit-exact, as with [E][D]."""
    s = I.MOE_GATE
    x, w = I.moe_inputs(s)
    idx, wts = _run_de(rf, x, w, s.k)
    _check(x, w, s.k, idx, wts, "MoE 8192x4096x64 [D][E]")


@pytest.mark.parametrize("T,D,E,k", [(300, 256, 64, 2), (129, 1024, 128, 4), (64, 4096, 192, 8),
                                     (513, 200, 256, 2), (1, 64, 64, 1), (1000, 2048, 256, 8),
                                     (777, 8, 128, 3)])
def test_moe_gate_dim_major(rf, T, D, E, k):
    x, w = I.moe_inputs(I.MoEShape(T=T, D=D, E=E, k=k, seed=7 * T + D + E + k))
    idx, wts = _run_de(rf, x, w, k)
    _check(x, w, k, idx, wts, f"MoE {T}x{D}x{E} k={k} [D][E]")


def test_moe_gate_all_equal_scores(rf):
    """All scores equal: the first k experts, uniform weights."""
    x = torch.ones(130, 128, dtype=torch.bfloat16)
    w = torch.ones(64, 128, dtype=torch.bfloat16)
    idx, wts = _run(rf, x, w, 4)
    assert (idx == np.arange(4)[None, :]).all()
    assert np.abs(wts - 0.25).max() <= MOE_W_ABS


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_moe_gate_dense_ties(rf, k):
    """Scores drawn from {-2..2}: nearly every token has ties across the top-k
    boundary and inside it, including an equal score pushed down past a
    higher-index twin by a larger one."""
    T, D = 512, 8
    g = torch.Generator().manual_seed(77 + k)
    x = torch.zeros(T, D, dtype=torch.bfloat16)
    x[torch.arange(T), torch.arange(T) % D] = 1
    w = torch.randint(-2, 3, (64, D), generator=g).to(torch.bfloat16)
    idx, wts = _run(rf, x, w, k)
    _check(x, w, k, idx, wts, f"dense ties k={k}")


# ------------------------------------------------ other expert counts
# The MMA width is E rounded up to 32, 64, 128 or 256; columns past E are
# never read.  Small D keeps scores in a narrow range so ties are common.


@pytest.mark.parametrize("T,D,E,k", [(300, 256, 8, 2), (257, 1024, 8, 8), (129, 512, 20, 4),
                                     (1000, 2048, 32, 1), (200, 4096, 100, 8), (513, 1024, 128, 4),
                                     (300, 2048, 256, 8), (129, 64, 256, 1), (64, 8192, 250, 2),
                                     (100, 128, 1, 1), (4096, 4096, 256, 8)])
def test_moe_gate_expert_counts(rf, T, D, E, k):
    x, w = I.moe_inputs(I.MoEShape(T=T, D=D, E=E, k=k, seed=5 * T + D + E + k))
    idx, wts = _run(rf, x, w, k)
    _check(x, w, k, idx, wts, f"MoE {T}x{D} E={E} k={k}")


@pytest.mark.parametrize("E,k", [(8, 8), (128, 4), (256, 8)])
def test_moe_gate_dense_ties_expert_counts(rf, E, k):
    T, D = 512, 8
    g = torch.Generator().manual_seed(91 + E + k)
    x = torch.zeros(T, D, dtype=torch.bfloat16)
    x[torch.arange(T), torch.arange(T) % D] = 1
    w = torch.randint(-2, 3, (E, D), generator=g).to(torch.bfloat16)
    idx, wts = _run(rf, x, w, k)
    _check(x, w, k, idx, wts, f"dense ties E={E} k={k}")
