#!/usr/bin/env python3
"""Benchmark of the fused cascaded-reduction hot path on GB300.

One step = one pass of every fused kernel over its workload, on inputs
resident in HBM:
  decode split-KV, Lk = 2048 (B 32, Hq 32, Hkv 8, d 128, bf16)
  MoE gate (8192 x 4096 x 64 experts, top-2)
  row absmax -> E4M3 -> FP8 GEMM (4096^3)
  BERT-style prefill attention (B 8, H 16, L 512, d 64, bf16)
  decode split-KV, Lk = 32768
Each kernel's inputs were last touched one step earlier with >= 4.3 GB
streamed in between, far more than the 129 MB L2, so every launch starts
from a cold L2 without an explicit flush.  The order puts the prefill (whose
pace is set by the tensor pipe and latency, not HBM) right after the FP8
GEMM: the GEMM leaves its output and codes as dirty L2 lines, and the next
kernel that streams from HBM pays for their write-back.

Metric: the step's roofline time (sum over the kernels of
max(algorithmic bytes / HBM peak, algorithmic FLOPs / tensor peak)) divided
by the measured step time, in percent.  Peaks come from MEASURED_PEAKS.json
when present, else the fallback figures (6.8 TB/s, 1.9 PFLOP/s bf16; FP8 =
2x bf16).  The tensor peak is the burst figure: every kernel is timed in a
region far shorter than a second.  One JSON line is printed by rank 0.

Before timing, the first call of every op is checked against the fp64 CPU
oracle on the same seeded inputs (bit-exact indices, codes and scales; the
stated tolerances for floats); the run exits non-zero if any check fails.

--only times a subset of the step, or calls outside it (the causal and
variable-length prefill, short prefill in both evaluation orders, other
expert counts of the gate, the latent-KV decode), with the same metric, in
the order given.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--only CALL,...]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as I  # noqa: E402

METRIC = "fused cascaded-reduction TFLOP/s or HBM GB/s, % of GB300 roofline (1 GPU)"
UNIT = "% of roofline (step roofline time / measured step time)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFS = 1900.0
FALLBACK_BF16_TFS_SUSTAINED = 1700.0


# ------------------------------------------------------------------ peaks


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = float(d.get("hbm_gbs") or d.get("hbm_GBps") or 0)
            bf16 = float(d.get("bf16_tflops") or 0)
            bf16s = float(d.get("bf16_tflops_sustained") or bf16)
            if hbm > 0 and bf16 > 0:
                return {"hbm_gbs": hbm, "bf16_tfs": bf16, "bf16_tfs_sustained": bf16s,
                        "source": "measured"}
        except (ValueError, OSError):
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tfs": FALLBACK_BF16_TFS,
            "bf16_tfs_sustained": FALLBACK_BF16_TFS_SUSTAINED, "source": "fallback"}


# ------------------------------------------------------------------ workload


class Op:
    """One fused call of the step: its algorithmic bytes/FLOPs and a launcher."""

    def __init__(self, name, bytes_, flops, tc_dtype, n_kernels):
        self.name, self.bytes, self.flops, self.tc_dtype = name, bytes_, flops, tc_dtype
        self.n_kernels = n_kernels

    def tensor_peak(self, peaks):
        """Dense tensor peak of this op's dtype (TFLOP/s): the measured bf16
        burst figure, x2 for FP8 (the nominal ratio)."""
        return peaks["bf16_tfs"] * (2.0 if self.tc_dtype == "fp8" else 1.0)

    def roofline_s(self, peaks):
        t_mem = self.bytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = self.flops / (self.tensor_peak(peaks) * 1e12) if self.flops else 0.0
        return max(t_mem, t_tc)

    def bound(self, peaks):
        t_mem = self.bytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = self.flops / (self.tensor_peak(peaks) * 1e12) if self.flops else 0.0
        return "hbm" if t_mem >= t_tc else "tensor"


def decode_op(name, s):
    kv = 2 * s.B * s.Hkv * s.Lk * s.d * 2
    qo = 2 * s.B * s.Hq * s.d * 2
    return Op(name, kv + qo, 4 * s.B * s.Hq * s.Lk * s.d, "bf16", 1)


def make_ops():
    b = I.BERT_PREFILL
    m = I.MOE_GATE
    f = I.FP8_GEMM
    return [
        decode_op("decode_2k", I.DECODE_2K),
        Op("moe_gate", m.T * m.D * 2 + m.E * m.D * 2 + m.T * m.k * 8, 2 * m.T * m.D * m.E, "bf16", 1),
        Op("fp8_gemm", f.M * f.K * 2 + f.N * f.K + f.N * 4 + f.M * f.N * 2, 2 * f.M * f.N * f.K,
           "fp8", 1),
        Op("bert_prefill", 4 * b.B * b.Hq * b.Lq * b.d * 2, 4 * b.B * b.Hq * b.Lq * b.Lk * b.d,
           "bf16", 1),
        decode_op("decode_32k", I.DECODE_32K),
    ]


def make_extra_ops():
    """Calls measured on request (--only) but not part of the step: the
    causal-mask variant of the prefill workload (FLOPs count only the
    (query, key) pairs the mask lets through)."""
    b = I.BERT_PREFILL
    pairs = sum(min(b.Lk, i + (b.Lk - b.Lq) + 1) for i in range(b.Lq))
    ops = [Op("bert_prefill_causal", 4 * b.B * b.Hq * b.Lq * b.d * 2,
              4 * b.B * b.Hq * pairs * b.d, "bf16", 1)]
    for name, m in MOE_EXTRA.items():
        ops.append(Op(name, m.T * m.D * 2 + m.E * m.D * 2 + m.T * m.k * 8, 2 * m.T * m.D * m.E,
                      "bf16", 1))
    for name, (sh, _mode) in SHORT_EXTRA.items():
        ops.append(Op(name, 4 * sh.B * sh.Hq * sh.Lq * sh.d * 2,
                      4 * sh.B * sh.Hq * sh.Lq * sh.Lk * sh.d, "bf16", 1))
    v = I.PREFILL_VARLEN
    lens = varlen_lengths()
    ops.append(Op("prefill_varlen", 4 * sum(lens) * v.H * v.d * 2,
                  4 * v.H * v.d * sum(n * n for n in lens), "bf16", 1))
    ops.append(mla_op())
    return ops


def mla_op():
    """Latent-KV decode: the cache is read once (B * Lk rows of d_qk bf16),
    plus Q and O; FLOPs count the scores over d_qk dims and P.V over d_v.
    Its kernel count (1, or 2 with a merge) is filled in by run_ours from the
    library's choice of segments."""
    s = I.MLA_DECODE
    cache = s.B * s.Lk * s.d_qk * 2
    qo = s.B * s.Hq * (s.d_qk + s.d_v) * 2
    return Op("mla_decode", cache + qo, 2 * s.B * s.Hq * s.Lk * (s.d_qk + s.d_v), "bf16", 1)


def varlen_lengths():
    cu = I.varlen_inputs(I.PREFILL_VARLEN)[3]
    return (cu[1:] - cu[:-1]).tolist()


# Short prefill under both evaluation orders of the cascade (mode 1 =
# incremental, 2 = two-pass).
SHORT_EXTRA = {
    "short256_incremental": (I.SHORT_PREFILL_256, 1),
    "short256_two_pass": (I.SHORT_PREFILL_256, 2),
    "short128_incremental": (I.SHORT_PREFILL_128, 1),
    "short128_two_pass": (I.SHORT_PREFILL_128, 2),
}

# Gate shapes outside the step: the step's token count and width with 8
# experts / top-2 and 256 experts / top-8.
MOE_EXTRA = {
    "moe_gate_e8_k2": I.MoEShape(T=8192, D=4096, E=8, k=2, seed=41),
    "moe_gate_e256_k8": I.MoEShape(T=8192, D=4096, E=256, k=8, seed=42),
}


GENERATORS = {
    "decode_32k": lambda: list(I.decode_inputs(I.DECODE_32K)),
    "decode_2k": lambda: list(I.decode_inputs(I.DECODE_2K)),
    "bert_prefill": lambda: list(I.attention_inputs(I.BERT_PREFILL)),
    "bert_prefill_causal": lambda: list(I.attention_inputs(I.BERT_PREFILL)),
    "prefill_varlen": lambda: list(I.varlen_inputs(I.PREFILL_VARLEN)),
    **{name: (lambda sh=sh: list(I.attention_inputs(sh))) for name, (sh, _m) in SHORT_EXTRA.items()},
    "moe_gate_e8_k2": lambda: list(I.moe_inputs(MOE_EXTRA["moe_gate_e8_k2"])),
    "moe_gate_e256_k8": lambda: list(I.moe_inputs(MOE_EXTRA["moe_gate_e256_k8"])),
    "moe_gate": lambda: list(I.moe_inputs(I.MOE_GATE)),
    "mla_decode": lambda: list(I.mla_inputs(I.MLA_DECODE)),
    "fp8_gemm": lambda: list(I.fp8_inputs(I.FP8_GEMM)),
}


def host_inputs(names):
    """Step inputs as CPU tensors (seeded), keyed by op name."""
    return {n: GENERATORS[n]() for n in names}


SPLITS = {}


def args_splits(lk):
    """Explicit split count for a decode length (0 = the library's automatic choice)."""
    return SPLITS.get(lk, 0)


class Step:
    """Device buffers and the calls of one step, through the public binding."""

    def __init__(self, rf, dev_inputs):
        self.rf = rf
        d = dev_inputs
        self.inp = d
        s32, s2, sb, sm, sf = I.DECODE_32K, I.DECODE_2K, I.BERT_PREFILL, I.MOE_GATE, I.FP8_GEMM
        cuda = torch.device("cuda")
        self.o32 = torch.empty(s32.B, s32.Hq, s32.d, dtype=torch.bfloat16, device=cuda)
        self.o2 = torch.empty(s2.B, s2.Hq, s2.d, dtype=torch.bfloat16, device=cuda)
        self.ws32 = torch.empty(rf.rf_attn_decode_splitkv_workspace_size(
            s32.B, s32.Hq, s32.Hkv, s32.Lk, s32.d, args_splits(32768)), dtype=torch.uint8,
            device=cuda)
        self.ws2 = torch.empty(rf.rf_attn_decode_splitkv_workspace_size(
            s2.B, s2.Hq, s2.Hkv, s2.Lk, s2.d, args_splits(2048)), dtype=torch.uint8, device=cuda)
        self.ob = torch.empty(sb.B, sb.Hq, sb.Lq, sb.d, dtype=torch.bfloat16, device=cuda)
        self.idx = torch.empty(sm.T, sm.k, dtype=torch.int32, device=cuda)
        self.wts = torch.empty(sm.T, sm.k, dtype=torch.float32, device=cuda)
        self.y = torch.empty(sf.M, sf.N, dtype=torch.bfloat16, device=cuda)
        self.wsf = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(sf.M, sf.N, sf.K),
                               dtype=torch.uint8, device=cuda)
        if "fp8_gemm" in d:
            # the fused call takes W pre-quantised: made once here by the
            # library's own per-row quantiser (not part of the timed step)
            x_d, w_d = d["fp8_gemm"]
            self.wq = torch.empty(sf.N, sf.K, dtype=torch.uint8, device=cuda)
            self.sw = torch.empty(sf.N, dtype=torch.float32, device=cuda)
            rf.rf_absmax_quant_fp8(w_d, self.sw, self.wq)
            d["fp8_gemm"] = [x_d, self.wq, self.sw]
            self.sx = torch.empty(sf.M, dtype=torch.float32, device=cuda)
            self.xq = torch.empty(sf.M, sf.K, dtype=torch.uint8, device=cuda)
        if "moe_gate" in d:
            # W_gate in the [D][E] layout of the problem statement (x @ W_gate);
            # the generator (and the oracle) hold it as [E][D]
            x_m, w_m = d["moe_gate"]
            d["moe_gate"] = [x_m, w_m.t().contiguous()]
        self.calls = {
            "decode_32k": lambda: rf.rf_attn_decode_splitkv(*d["decode_32k"], self.o32, s32.scale,
                                                            self.ws32, args_splits(32768)),
            "bert_prefill": lambda: rf.rf_attn_fwd(*d["bert_prefill"], self.ob, sb.scale),
            "bert_prefill_causal": lambda: rf.rf_attn_fwd(*d["bert_prefill_causal"], self.ob,
                                                          sb.scale, 1),
            "moe_gate": lambda: rf.rf_moe_gate_topk_softmax_ex(*d["moe_gate"], sm.k, rf.RF_GATE_W_DE,
                                                               self.idx, self.wts),
            "fp8_gemm": lambda: rf.rf_absmax_fp8_gemm(*d["fp8_gemm"], self.y, self.wsf),
            "decode_2k": lambda: rf.rf_attn_decode_splitkv(*d["decode_2k"], self.o2, s2.scale,
                                                           self.ws2, args_splits(2048)),
        }
        if "prefill_varlen" in d:
            qv, kv_, vv, cuv = d["prefill_varlen"]
            self.ov = torch.empty_like(qv)
            maxlen = int((cuv[1:] - cuv[:-1]).max().item())
            self.calls["prefill_varlen"] = lambda: rf.rf_attn_fwd_varlen(
                qv, kv_, vv, self.ov, cuv, cuv, maxlen, I.PREFILL_VARLEN.scale)
        for name, (sh, mode) in SHORT_EXTRA.items():
            if name in d:
                ob = torch.empty_like(d[name][0])
                self.calls[name] = (lambda name=name, sh=sh, mode=mode, ob=ob:
                                    rf.rf_attn_fwd_ex(*d[name], ob, sh.scale, 0, mode))
                setattr(self, "out_" + name, [ob])
        if "mla_decode" in d:
            sl = I.MLA_DECODE
            self.oml = torch.empty(sl.B, sl.Hq, sl.d_v, dtype=torch.bfloat16, device=cuda)
            nb = rf.rf_mla_decode_workspace_size(sl.B, sl.Hq, sl.Lk, sl.d_qk, sl.d_v, 0)
            self.wsml = torch.empty(nb, dtype=torch.uint8, device=cuda) if nb else None
            self.calls["mla_decode"] = lambda: rf.rf_mla_decode(*d["mla_decode"], self.oml,
                                                                sl.scale, self.wsml)
        for name, m in MOE_EXTRA.items():
            ix = torch.empty(m.T, m.k, dtype=torch.int32, device=cuda)
            wt = torch.empty(m.T, m.k, dtype=torch.float32, device=cuda)
            self.calls[name] = (lambda name=name, m=m, ix=ix, wt=wt:
                                rf.rf_moe_gate_topk_softmax(*d[name], m.k, ix, wt))
            setattr(self, "out_" + name, [ix, wt])
        # the un-timed first call of the FP8 op also writes its codes and row
        # scales out, for the parity check; timed calls keep them in the workspace
        self.parity_calls = {
            "fp8_gemm": lambda: rf.rf_absmax_fp8_gemm(*d["fp8_gemm"], self.y, self.wsf,
                                                      sx_out=self.sx, xq_out=self.xq),
        }
        self.outputs = {"decode_32k": [self.o32], "decode_2k": [self.o2],
                        "bert_prefill": [self.ob], "bert_prefill_causal": [self.ob],
                        "moe_gate": [self.idx, self.wts],
                        "fp8_gemm": [self.y]}
        for name in MOE_EXTRA:
            self.outputs[name] = getattr(self, "out_" + name)
        if "prefill_varlen" in d:
            self.outputs["prefill_varlen"] = [self.ov]
        if "mla_decode" in d:
            self.outputs["mla_decode"] = [self.oml]
        for name in SHORT_EXTRA:
            if name in d:
                self.outputs[name] = getattr(self, "out_" + name)


# ------------------------------------------------------------------ parity

# Tolerances of the parity check: the ones the GPU parity tests use.
TOL_BF16_MAX_ABS = 2e-2        # attention outputs, elementwise
TOL_BF16_REL_L2 = 5e-3
TOL_FP8_Y_REL = 2e-2           # FP8 Y: |Y - Y_ref| <= 2e-2 * max(1, |Y_ref|)
TOL_FP8_Y_REL_L2 = 5e-3
TOL_MOE_W_ABS = 1e-6           # MoE weights (scores are exact integers)


def oracle_fp8_weight(w):
    """The pre-quantised FP8 weight as the oracle makes it (row_scale, then
    quantise, per row of W [N][K])."""
    from oracle import fp8_quant_gemm as F
    _, sw = F.row_scale(w)
    return F.quantise(w, sw), sw


def oracle_view(host):
    """The ops' inputs as the oracle takes them: the FP8 weight quantised by
    the oracle's own quantiser."""
    out = dict(host)
    if "fp8_gemm" in host:
        x, w = host["fp8_gemm"]
        wq, sw = oracle_fp8_weight(w)
        out["fp8_gemm"] = [x, wq, sw]
    return out


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _close(got, ref, max_abs, rel_l2, relative):
    got, ref = _f64(got).reshape(ref.shape), np.asarray(ref, np.float64)
    if not np.isfinite(got).all():
        return f"FAIL: {int((~np.isfinite(got)).sum())} non-finite elements"
    bound = max_abs * (np.maximum(1.0, np.abs(ref)) if relative else 1.0)
    nbad = int((np.abs(got - ref) > bound).sum())
    r = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    if nbad or r > rel_l2:
        return f"FAIL: {nbad} elements outside tolerance, rel-L2 {r:.2e}"
    return "ok"


def check_op(name, outs, ov):
    """Compares one op's outputs (host tensors) with the full fp64 oracle."""
    from oracle import attention as A
    from oracle import fp8_quant_gemm as F
    from oracle import moe_gate as G

    if name in ("decode_32k", "decode_2k"):
        s = I.DECODE_32K if name == "decode_32k" else I.DECODE_2K
        ref = A.decode_attention(*ov[name], s.scale)
        return _close(outs[0], ref, TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, False)
    if name in ("bert_prefill", "bert_prefill_causal"):
        s = I.BERT_PREFILL
        ref = A.attention(*ov[name], s.scale, causal=name.endswith("causal"))
        return _close(outs[0], ref, TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, False)
    if name in SHORT_EXTRA:
        sh = SHORT_EXTRA[name][0]
        ref = A.attention(*ov[name], sh.scale)
        return _close(outs[0], ref, TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, False)
    if name == "prefill_varlen":
        q, k, v, cu = ov[name]
        ref = A.attention_varlen(q, k, v, cu, cu, I.PREFILL_VARLEN.scale)
        return _close(outs[0], ref, TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, False)
    if name == "mla_decode":
        s = I.MLA_DECODE
        ref = A.mla_decode(*ov[name], s.scale, s.d_v)
        return _close(outs[0], ref, TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, False)
    if name == "moe_gate" or name in MOE_EXTRA:
        m = I.MOE_GATE if name == "moe_gate" else MOE_EXTRA[name]
        ref_idx, ref_w, _ = G.moe_gate(*ov[name], m.k)
        nbad = int((outs[0].numpy() != ref_idx).sum())
        if nbad:
            return f"FAIL: {nbad} expert indices differ"
        err = float(np.abs(_f64(outs[1]) - ref_w).max())
        return "ok" if err <= TOL_MOE_W_ABS else f"FAIL: weights differ by {err:.2e}"
    if name == "fp8_gemm":
        y, sx, xq = outs
        ref_sx, ref_xq, ref_y = F.absmax_fp8_gemm(*ov[name])
        if not np.array_equal(sx.numpy().view(np.uint32), ref_sx.view(np.uint32)):
            return "FAIL: row scales differ"
        nbad = int((xq.numpy() != ref_xq).sum())
        if nbad:
            return f"FAIL: {nbad} E4M3 codes differ"
        return _close(y, ref_y, TOL_FP8_Y_REL, TOL_FP8_Y_REL_L2, True)
    raise KeyError(name)


def parity_gate(rf, step, ops, host):
    """The first, un-timed call of every op, checked against the full oracle
    on the same seeded inputs; returns {op: "ok" | "FAIL: ..."}."""
    ov = oracle_view(host)
    res = {}
    if "fp8_gemm" in host:
        wq_o, sw_o = ov["fp8_gemm"][1:]
        same = (np.array_equal(step.wq.cpu().numpy(), wq_o)
                and np.array_equal(step.sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32)))
        res["fp8_weight"] = "ok" if same else "FAIL: weight codes or scales differ"
    for op in ops:
        (step.parity_calls.get(op.name) or step.calls[op.name])()
        torch.cuda.synchronize()
        outs = [t.cpu() for t in step.outputs[op.name]]
        if op.name == "fp8_gemm":
            outs += [step.sx.cpu(), step.xq.cpu()]
        res[op.name] = check_op(op.name, outs, ov)
    st = rf.rf_get_device_status()
    if st != rf.RF_OK:
        res["device_status"] = "FAIL: " + rf.rf_status_string(st)
    return res


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ timing


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def traffic_for(kernel_key):
    """Per-launch DRAM bytes from a committed ncu capture, if the kernel source
    has not changed since (matched by hash); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(kernel_key)
    except (ValueError, OSError):
        return None
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src):
        return None
    sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    return d["bytes_per_launch"] if sha == d["source_sha1"] else None


def run_ours(args, world, rank, local):
    import cascaded_reductions_loop_gb300 as rf

    torch.cuda.set_device(local)
    peaks = load_peaks()
    ops = select_ops(args)
    host = host_inputs([op.name for op in ops])
    dev = {k: [t.cuda() for t in v] for k, v in host.items()}
    step = Step(rf, dev)
    stream = torch.cuda.current_stream()
    for op in ops:
        if op.name == "mla_decode":
            s = I.MLA_DECODE
            op.n_kernels = 1 + (rf.rf_mla_decode_num_splits(s.B, s.Hq, s.Lk, s.d_qk, s.d_v, 0) > 1)
    # what a caller holds on the host for each call (the e2e copies): the FP8
    # call takes the quantised weight the set-up made
    call_host = dict(host)
    if "fp8_gemm" in host:
        call_host["fp8_gemm"] = [host["fp8_gemm"][0], step.wq.cpu(), step.sw.cpu()]
    if "moe_gate" in host:
        call_host["moe_gate"] = [host["moe_gate"][0], host["moe_gate"][1].t().contiguous()]

    # parity: the first call of every op against the oracle (rank 0)
    parity = None
    if args.parity == "full" and rank == 0:
        parity = parity_gate(rf, step, ops, host)
        if any(v != "ok" for v in parity.values()):
            print(json.dumps({"metric": METRIC, "value": None, "parity": parity,
                              "error": "GPU outputs differ from the oracle"}), flush=True)
            raise SystemExit(3)

    # warm-up
    for _ in range(args.warmup):
        for op in ops:
            step.calls[op.name]()
    torch.cuda.synchronize()
    st = rf.rf_get_device_status()
    if st != rf.RF_OK:
        raise RuntimeError(f"device status after warm-up: {rf.rf_status_string(st)}")

    # timed region: K steps, one event pair per fused call
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    n = len(ops)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    # a sleep kernel ahead of the timed region keeps the GPU busy while the
    # host enqueues the timed calls, so that calls shorter than their host-side
    # issue time (about 15-20 us per call through the binding) run back to
    # back and are timed as the GPU runs them, not at the host's issue rate
    torch.cuda._sleep(int(min(0.2, max(0.005, args.steps * n * 25e-6)) * 2.0e9))
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        evs[s][0].record(stream)
        for i, op in enumerate(ops):
            step.calls[op.name]()
            evs[s][i + 1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    st = rf.rf_get_device_status()
    if st != rf.RF_OK:
        raise RuntimeError(f"device status after timing: {rf.rf_status_string(st)}")

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_per_step = total_ms / args.steps
    # per call: mean of the middle 90 % of the K event intervals (a single
    # interval is quantised to about a microsecond; the mean over many is not)
    per_op_ms = {op.name: trimmed_mean([evs[s][i].elapsed_time(evs[s][i + 1])
                                        for s in range(args.steps)])
                 for i, op in enumerate(ops)}
    roof_s = sum(op.roofline_s(peaks) for op in ops)
    value = 100.0 * world * roof_s / (ms_per_step * 1e-3)

    rows = {}
    for op in ops:
        t = per_op_ms[op.name] * 1e-3
        r = {"ms": round(per_op_ms[op.name], 5), "bound": op.bound(peaks),
             "roofline_frac": round(op.roofline_s(peaks) / t, 4)}
        if op.bound(peaks) == "hbm":
            r["GBps"] = round(op.bytes / t / 1e9, 1)
        else:
            r["TFLOPs"] = round(op.flops / t / 1e12, 1)
        rows[op.name] = r

    dom = max(ops, key=lambda op: per_op_ms[op.name])
    dom_t = per_op_ms[dom.name] * 1e-3
    if dom.bound(peaks) == "hbm":
        achieved = dom.bytes / dom_t / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = dom.flops / dom_t / 1e12
        pk = dom.tensor_peak(peaks)
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk,
                    "unit": "TFLOP/s", "frac": round(achieved / pk, 4)}
    roofline.update({"traffic": traffic_for(dom.name), "kernel": dom.name,
                     "launches_per_call": dom.n_kernels,
                     "peak_source": peaks["source"]})

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the five named workloads)",
        "config": workload_config(ops, world),
        "peaks": {**{k: peaks[k] for k in ("hbm_gbs", "bf16_tfs", "bf16_tfs_sustained", "source")},
                  "tensor_basis": "bf16_tfs (burst; x2 for FP8): each kernel runs well under 1 s"},
        "rows": rows,
        "roofline": roofline,
        "gpu_launches": args.steps * sum(op.n_kernels for op in ops),
        "clocks": clk,
        "parity": parity if parity is not None else "not checked (--parity off or rank > 0)",
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(rf, ops, peaks, call_host, step, world, args)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(ops, peaks, oracle_view(host),
                                              budget_s=args.cpu_budget)
    return result


def trimmed_mean(xs, cut=0.05):
    xs = sorted(xs)
    k = int(len(xs) * cut)
    core = xs[k:len(xs) - k] or xs
    return sum(core) / len(core)


def select_ops(args):
    ops = make_ops()
    if args.only:
        names = args.only.split(",")
        known = ops + make_extra_ops()
        unknown = set(names) - {op.name for op in known}
        if unknown:
            raise SystemExit(f"unknown op(s) {sorted(unknown)}")
        by_name = {op.name: op for op in known}
        ops = [by_name[n] for n in dict.fromkeys(names)]     # in the order given
    return ops


def workload_name(ops):
    if [op.name for op in ops] == [op.name for op in make_ops()]:
        return "decode2k+moe_gate+fp8_gemm+bert_prefill+decode32k"
    return "+".join(op.name for op in ops)


def workload_config(ops, world):
    """The shapes of the calls a run times (the whole step, or the --only
    calls) and how L2 reuse between steps is avoided."""
    names = {op.name for op in ops}
    cfg = {"workload": workload_name(ops)}
    if names & {"decode_32k", "decode_2k"}:
        cfg["decode"] = "B32 Hq32 Hkv8 d128 Lk {32768, 2048} bf16"
    if names & {"bert_prefill", "bert_prefill_causal"}:
        cfg["prefill"] = "B8 H16 L512 d64 bf16"
    if "moe_gate" in names:
        cfg["moe"] = "T8192 D4096 E64 top2 bf16, W_gate [D][E]"
    if "fp8_gemm" in names:
        cfg["fp8"] = "M=N=K=4096 e4m3 (bf16 X in, bf16 Y out)"
    if "mla_decode" in names:
        s = I.MLA_DECODE
        cfg["mla"] = (f"B{s.B} Hq{s.Hq} Lk{s.Lk} d_qk{s.d_qk} d_v{s.d_v} bf16, one latent head, "
                      f"scale 1/sqrt(192)")
    total = sum(op.bytes for op in ops)
    cfg["l2"] = (f"no flush: inputs of {total / 1e6:.0f} MB per step streamed "
                 + ("(> 129 MB L2) between reuses" if total > 129e6 else
                    "(under the 129 MB L2: later steps may hit L2)"))
    cfg["parallelism"] = f"replicas x{world}"
    return cfg


def run_e2e(rf, ops, peaks, host, step, world, args):
    """Same metric through the public binding with host buffers: every step
    copies every call's inputs from pinned host memory and its results back.
    The input copies run on a stream of their own, ahead of the calls, and the
    result copies on a third stream, so copies and kernels overlap; events
    keep each buffer's writes after the previous step's reads of it."""
    pinned = {}
    for op in ops:
        dev, src = step.inp[op.name], host[op.name]
        if len(dev) == len(src) and all(s.shape == d.shape and s.dtype == d.dtype
                                        for s, d in zip(src, dev)):
            pinned[op.name] = [t.pin_memory() for t in src]
        else:
            # inputs made on the device at set-up (the FP8 weight's codes and
            # scales, quantised by the library): the host holds the same ones
            pinned[op.name] = [t.cpu().pin_memory() for t in dev]
        for s_, d_ in zip(pinned[op.name], dev):
            if s_.shape != d_.shape or s_.dtype != d_.dtype:
                raise SystemExit(f"e2e: host input of {op.name} does not match its device buffer")
    out_host = {op.name: [torch.empty(o.shape, dtype=o.dtype).pin_memory()
                          for o in step.outputs[op.name]] for op in ops}
    h2d = sum(t.numel() * t.element_size() for v in pinned.values() for t in v)
    d2h = sum(t.numel() * t.element_size() for v in out_host.values() for t in v)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    called = {}        # op -> event after its call (its inputs have been read)
    fetched = {}       # op -> event after its results were copied back

    def one():
        for op in ops:
            n = op.name
            with torch.cuda.stream(s_in):
                if n in called:
                    s_in.wait_event(called[n])
                for dst, src in zip(step.inp[n], pinned[n]):
                    dst.copy_(src, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            comp.wait_event(ready)
            if n in fetched:
                comp.wait_event(fetched[n])
            step.calls[n]()
            called[n] = torch.cuda.Event()
            called[n].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(called[n])
                for dst, src in zip(out_host[n], step.outputs[n]):
                    dst.copy_(src, non_blocking=True)
                fetched[n] = torch.cuda.Event()
                fetched[n].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    one()
    torch.cuda.synchronize()
    k = max(2, min(args.steps, 5))
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(k):
        one()
    b.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world) / k
    roof_s = sum(op.roofline_s(peaks) for op in ops)
    return {"value": round(100.0 * world * roof_s / (ms * 1e-3), 4), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": k, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "streams": "inputs, calls, results on three streams"}


# ------------------------------------------------------------------ CPU oracle


def oracle_sample_seconds(host, frac, only=None):
    """Times the fp64 oracle on a bounded sample of every op present in
    ``host`` (or of the ops in ``only``); returns {op: (seconds, fraction of
    the op's full work covered)}."""
    if only is not None:
        host = {k: v for k, v in host.items() if k in only}
    from oracle import attention as A
    from oracle import fp8_quant_gemm as F
    from oracle import moe_gate as G

    out = {}
    rng = np.random.default_rng(0)

    for name, s in (("decode_32k", I.DECODE_32K), ("decode_2k", I.DECODE_2K)):
        if name not in host:
            continue
        q, k, v = host[name]
        scale_rows = 1 if name == "decode_32k" else 4
        nrows = min(s.B * s.Hq, max(1, int(round(frac * scale_rows * s.B * s.Hq))))
        rows = [(int(b), int(h)) for b, h in
                zip(rng.integers(0, s.B, nrows), rng.integers(0, s.Hq, nrows))]
        t = time.perf_counter()
        A.decode_attention(q, k, v, s.scale, rows=rows)
        out[name] = (time.perf_counter() - t, nrows / (s.B * s.Hq))

    if "bert_prefill" in host:
        s = I.BERT_PREFILL
        q, k, v = host["bert_prefill"]
        nh = min(s.B * s.Hq, max(1, int(round(frac * 4 * s.B * s.Hq))))
        t = time.perf_counter()
        for i in range(nh):
            b, h = divmod(i % (s.B * s.Hq), s.Hq)
            A.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], s.scale)
        out["bert_prefill"] = (time.perf_counter() - t, nh / (s.B * s.Hq))

    if "bert_prefill_causal" in host:
        s = I.BERT_PREFILL
        q, k, v = host["bert_prefill_causal"]
        nh = min(s.B * s.Hq, max(1, int(round(frac * 4 * s.B * s.Hq))))
        t = time.perf_counter()
        for i in range(nh):
            b, h = divmod(i % (s.B * s.Hq), s.Hq)
            A.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], s.scale,
                        causal=True)
        out["bert_prefill_causal"] = (time.perf_counter() - t, nh / (s.B * s.Hq))

    if "moe_gate" in host:
        s = I.MOE_GATE
        x, w = host["moe_gate"]
        nt = min(s.T, max(1, int(round(frac * 4 * s.T))))
        t = time.perf_counter()
        G.moe_gate(x, w, s.k, rows=range(nt))
        out["moe_gate"] = (time.perf_counter() - t, nt / s.T)

    for name, (sh, _mode) in SHORT_EXTRA.items():
        if name not in host:
            continue
        q, k, v = host[name]
        nh = min(sh.B * sh.Hq, max(1, int(round(frac * 4 * sh.B * sh.Hq))))
        t = time.perf_counter()
        for i in range(nh):
            b, h = divmod(i % (sh.B * sh.Hq), sh.Hq)
            A.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], sh.scale)
        out[name] = (time.perf_counter() - t, nh / (sh.B * sh.Hq))

    if "prefill_varlen" in host:
        q, k, v, cu = host["prefill_varlen"]
        nseq = len(cu) - 1
        tot = sum(int(cu[b + 1] - cu[b]) ** 2 for b in range(nseq))
        done, b = 0, 0
        t = time.perf_counter()
        while done < frac * 4 * tot and b < nseq:   # whole sequences until the sample is covered
            sl = slice(int(cu[b]), int(cu[b + 1]))
            one = cu[b:b + 2] - cu[b]                   # [0, length]
            A.attention_varlen(q[sl], k[sl], v[sl], one, one, I.PREFILL_VARLEN.scale)
            done += int(cu[b + 1] - cu[b]) ** 2
            b += 1
        out["prefill_varlen"] = (time.perf_counter() - t, done / tot)

    for name, m in MOE_EXTRA.items():
        if name not in host:
            continue
        x, w = host[name]
        nt = min(m.T, max(1, int(round(frac * 4 * m.T))))
        t = time.perf_counter()
        G.moe_gate(x, w, m.k, rows=range(nt))
        out[name] = (time.perf_counter() - t, nt / m.T)

    if "mla_decode" in host:
        s = I.MLA_DECODE
        q, c = host["mla_decode"]
        nrows = min(s.B * s.Hq, max(1, int(round(frac * 4 * s.B * s.Hq))))
        rows = [divmod(i, s.Hq) for i in range(nrows)]     # whole batches first
        t = time.perf_counter()
        A.mla_decode(q, c, s.scale, s.d_v, rows=rows)
        out["mla_decode"] = (time.perf_counter() - t, nrows / (s.B * s.Hq))

    if "fp8_gemm" in host:
        s = I.FP8_GEMM
        x, wq, sw = host["fp8_gemm"]
        nr = min(s.M, max(1, int(round(frac * s.M))))
        t = time.perf_counter()
        F.absmax_fp8_gemm(x, wq, sw, rows=range(nr))
        out["fp8_gemm"] = (time.perf_counter() - t, nr / s.M)
    return out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def calibrated_fraction(host, budget_s, lo=1.0 / 1024, hi=1.0 / 64, cap=1.0):
    """Fraction of every op's rows whose oracle run takes about budget_s.
    The sample time is a fixed part (conversions of whole operands) plus a
    part proportional to the fraction, so both are fitted from two samples."""
    def run(frac):
        t0 = time.perf_counter()
        oracle_sample_seconds(host, frac)
        return time.perf_counter() - t0
    t_lo, t_hi = run(lo), run(hi)
    slope = max((t_hi - t_lo) / (hi - lo), 1e-6)
    fixed = max(t_lo - slope * lo, 0.0)
    frac = (budget_s - fixed) / slope
    return min(cap, max(lo, frac))


def oracle_cost_fits(host, lo, hi):
    """Per op: (fixed seconds, seconds per unit of the op's own fraction,
    the op's fraction per unit of the sampling fraction), from two samples.
    The fixed part (whole-operand conversions and decodes the oracle does on
    every call) must not be scaled up with the sample."""
    r_lo, r_hi = oracle_sample_seconds(host, lo), oracle_sample_seconds(host, hi)
    fits = {}
    for k in r_lo:
        (t1, f1), (t2, f2) = r_lo[k], r_hi[k]
        slope = (t2 - t1) / (f2 - f1) if f2 > f1 else t2 / max(f2, 1e-9)
        slope = max(slope, 1e-9)
        fits[k] = (max(0.0, t1 - slope * f1), slope, f1 / lo)
    return fits


def full_op_seconds(sample_s, f, fixed):
    """Oracle time for a whole op from a sample covering fraction f."""
    return fixed + max(sample_s - fixed, 0.0) / f


def cpu_baseline(ops, peaks, host, budget_s=15.0):
    # size the sample so that the timed oracle run takes about budget_s; the
    # per-op fixed parts come from two small samples
    fits = oracle_cost_fits(host, 1.0 / 1024, 1.0 / 64)
    frac = calibrated_fraction(host, budget_s)
    res = oracle_sample_seconds(host, frac)
    full_s = sum(full_op_seconds(sec, f, fits[k][0]) for k, (sec, f) in res.items())
    roof_s = sum(op.roofline_s(peaks) for op in ops)
    return {"value": 100.0 * roof_s / full_s, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "seconds_per_full_step": round(full_s, 2),
            "sample": ("fraction of each op's rows/heads/tokens run by the fp64 numpy oracle "
                       "(BLAS threads up to the core count): "
                       + ", ".join(f"{k} {f:.3f}" for k, (_, f) in res.items())
                       + "; full step = per op, the fixed per-call part plus the rest scaled "
                         "to the whole op"),
            "sample_seconds": round(sum(sec for sec, _ in res.values()), 2)}


def run_reference(args, world, rank):
    """The reference arm: the CPU fp64 oracle as it stands, on the same
    workload and metric.  Each warm-up and timed step samples one op (in
    turn), sized so that the whole run takes about args.ref_budget seconds;
    a step's time is the sum over ops of each op's latest whole-op estimate."""
    if rank != 0:
        return None
    peaks = load_peaks()
    ops = select_ops(args)
    host = oracle_view(host_inputs([op.name for op in ops]))
    fits = oracle_cost_fits(host, 1.0 / 8192, 1.0 / 1024)
    names = list(fits)
    est = {k: fixed + slope for k, (fixed, slope, _) in fits.items()}
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    t_full, fracs = [], {}
    for s in range(args.warmup + args.steps):
        k = names[s % len(names)]
        fixed, slope, mult = fits[k]
        f_op = min(1.0, max(1.0 / 8192, (per_step - fixed) / slope))
        frac = f_op / max(mult, 1e-9)
        sec, f = oracle_sample_seconds(host, frac, only={k})[k]
        est[k] = full_op_seconds(sec, f, fixed)
        fracs[k] = f
        if s >= args.warmup:
            t_full.append(sum(est.values()))
    full_s = statistics.median(t_full) if t_full else sum(est.values())
    roof_s = sum(op.roofline_s(peaks) for op in ops)
    value = 100.0 * roof_s / full_s
    sample = ("one op per step, in turn, by the fp64 numpy oracle; fraction of the op's "
              "rows/heads/tokens: " + ", ".join(f"{k} {f:.4f}" for k, f in fracs.items())
              + "; full step = sum of each op's latest estimate (fixed per-call part plus the "
                "rest scaled to the whole op); no full step is run: steps and ms_per_step are "
                "estimates")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(full_s * 1e3, 1),
        "estimated": True,
        "ops_sampled": {"per_step": 1, "total": args.steps + args.warmup,
                        "distinct": len(fracs)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the five named workloads)",
        "config": {"workload": workload_name(ops),
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--only", default="",
                    help="comma-separated subset of ops (decode_32k, bert_prefill, moe_gate, "
                         "fp8_gemm, decode_2k) or calls outside the step (bert_prefill_causal, prefill_varlen, "
                         "moe_gate_e8_k2, moe_gate_e256_k8, mla_decode, short256_incremental, short256_two_pass, "
                         "short128_incremental, short128_two_pass); "
                         "default: the whole step")
    ap.add_argument("--splits", default="",
                    help="explicit decode split counts, e.g. 32768:64,2048:8 (default: automatic)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--parity", choices=["full", "off"], default="full",
                    help="check the first call of every op against the full fp64 oracle "
                         "before timing (default full)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds of CPU oracle work for a whole --impl reference run")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: raising --warmup to 3 (minimum)", file=sys.stderr)
        args.warmup = 3

    for item in filter(None, args.splits.split(",")):
        lk, n = item.split(":")
        SPLITS[int(lk)] = int(n)

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            res = run_reference(args, world, rank)
        else:
            res = run_ours(args, world, rank, local)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
