"""Oracle: the safe-softmax attention cascade, computed pass by pass in fp64.

Test infrastructure only (see the package docstring for who may import it).

The cascade ([E] §2.2; [S] "Probleemstelling"): for one query row q and keys
k_i with values v_i,

    s_i = scale * (q . k_i)
    m   = max_i s_i                       reduction 1
    l   = sum_i exp(s_i - m)              reduction 2 (depends on m)
    o   = sum_i exp(s_i - m) / l * v_i    reduction 3 (depends on m and l)

``attention`` evaluates the three reductions as three separate full passes.
``attention_incremental`` and ``attention_segments`` are the method's own
single-loop and multi-segment forms, kept here only so that the tests can
show they equal the three-pass definition on small inputs.

Causal masking (an option of the fused loop the explainer presents for
prefill, [E] §4.1): the pages do not define it, so the usual autoregressive
reading is taken, aligned so that the last query row sees every key: with
off = Lk - Lq, query row i reads keys j <= i + off only.  A row that reads no
key at all (i + off < 0, possible only when Lq > Lk) is defined as zero.
"""
from __future__ import annotations

import numpy as np


def _f64(t) -> np.ndarray:
    """Exact conversion of a torch tensor or array (fp32/bf16/...) to fp64."""
    if hasattr(t, "detach"):
        import torch

        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """Grouped-query attention: query heads form Hkv contiguous groups of
    Hq/Hkv heads; group g reads K/V head g."""
    assert Hq % Hkv == 0
    return hq // (Hq // Hkv)


def causal_limit(iq: int, Lq: int, Lk: int) -> int:
    """Number of leading keys query row iq may read under the causal mask
    (clamped to 0..Lk)."""
    return max(0, min(Lk, iq + (Lk - Lq) + 1))


def three_pass_row(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One query row q [d] against K [Lk,d], V [Lk,d]; returns o [d] (fp64).
    With no keys (Lk = 0, a fully masked causal row) the result is zero."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    s = scale * (K @ q)            # scores
    m = s.max()                    # pass 1: max
    l = np.exp(s - m).sum()        # pass 2: sum of exp(s - m)
    p = np.exp(s - m) / l          # pass 3: weights, then contraction with V
    return p @ V


def probabilities(q, k, v, scale: float, b: int, hq: int) -> np.ndarray:
    """Softmax weights P [Lq, Lk] of one (batch, query head), fp64."""
    q64, k64 = _f64(q), _f64(k)
    Hq, Hkv = q64.shape[1], k64.shape[1]
    K = k64[b, kv_head_of(hq, Hq, Hkv)]
    s = scale * (q64[b, hq] @ K.T)
    m = s.max(axis=1, keepdims=True)
    l = np.exp(s - m).sum(axis=1, keepdims=True)
    return np.exp(s - m) / l


def attention(q, k, v, scale: float, rows=None, causal: bool = False) -> np.ndarray:
    """Three-pass attention.

    q: [B, Hq, Lq, d]; k, v: [B, Hkv, Lk, d] (any float dtype; converted to
    fp64 exactly).  Returns fp64 O [B, Hq, Lq, d], or, when ``rows`` is a
    list of (b, hq, iq) triples, O for those rows only as [len(rows), d].
    ``causal``: row iq reads only the first causal_limit(iq, Lq, Lk) keys.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    Lq, Lk = q.shape[2], k.shape[2]
    if rows is None:
        B, _, Lq, d = q.shape
        out = np.empty((B, Hq, Lq, d), dtype=np.float64)
        for b in range(B):
            for hq in range(Hq):
                kvh = kv_head_of(hq, Hq, Hkv)
                Q = _f64(q[b, hq])
                K = _f64(k[b, kvh])
                V = _f64(v[b, kvh])
                if causal:
                    for iq in range(Lq):
                        n = causal_limit(iq, Lq, Lk)
                        out[b, hq, iq] = three_pass_row(Q[iq], K[:n], V[:n], scale)
                    continue
                s = scale * (Q @ K.T)                        # [Lq, Lk]
                m = s.max(axis=1, keepdims=True)             # pass 1
                l = np.exp(s - m).sum(axis=1, keepdims=True)  # pass 2
                out[b, hq] = (np.exp(s - m) / l) @ V          # pass 3
        return out
    res = np.empty((len(rows), q.shape[-1]), dtype=np.float64)
    cache = {}
    for i, (b, hq, iq) in enumerate(rows):
        kvh = kv_head_of(hq, Hq, Hkv)
        if (b, kvh) not in cache:
            cache.clear()
            cache[(b, kvh)] = (_f64(k[b, kvh]), _f64(v[b, kvh]))
        K, V = cache[(b, kvh)]
        n = causal_limit(iq, Lq, Lk) if causal else Lk
        res[i] = three_pass_row(_f64(q[b, hq, iq]), K[:n], V[:n], scale)
    return res


def attention_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool = False) -> np.ndarray:
    """Packed variable-length batch: q [total_q, H, d], k/v [total_k, H, d];
    sequence b owns query tokens cu_q[b]..cu_q[b+1]-1 and key tokens
    cu_k[b]..cu_k[b+1]-1.  Each sequence is the three-pass attention of its
    own tokens (with the causal option); a sequence without keys gives zero
    rows.  Returns fp64 [total_q, H, d]."""
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    cq = [int(x) for x in _f64(cu_q)]
    ck = [int(x) for x in _f64(cu_k)]
    out = np.zeros_like(q64)
    for b in range(len(cq) - 1):
        if cq[b + 1] == cq[b]:
            continue
        Qb = q64[cq[b]:cq[b + 1]].transpose(1, 0, 2)[None]      # [1, H, Lq, d]
        Kb = k64[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None]
        Vb = v64[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None]
        Lq = Qb.shape[2]
        rows = [(0, h, i) for h in range(Qb.shape[1]) for i in range(Lq)]
        ob = attention(Qb, Kb, Vb, scale, rows=rows, causal=causal)   # [H*Lq, d]
        out[cq[b]:cq[b + 1]] = ob.reshape(Qb.shape[1], Lq, -1).transpose(1, 0, 2)
    return out


def decode_attention(q, k, v, scale: float, rows=None) -> np.ndarray:
    """Decode layout: q [B, Hq, d] (one query token), k/v [B, Hkv, Lk, d].
    Returns [B, Hq, d], or [len(rows), d] for a list of (b, hq) pairs."""
    B, Hq, d = q.shape
    if rows is None:
        rows_ = [(b, h) for b in range(B) for h in range(Hq)]
    else:
        rows_ = list(rows)
    q4 = q.reshape(B, Hq, 1, d)
    out = attention(q4, k, v, scale, rows=[(b, h, 0) for (b, h) in rows_])
    return out.reshape(B, Hq, d) if rows is None else out


def mla_decode(q, ckv, scale: float, dv: int, rows=None) -> np.ndarray:
    """Latent-KV (multi-latent) attention decode, absorbed form.

    The technical summary reports the fused kernels on multi-latent
    attention against a hand-written latent-attention decode library ([S]
    "Resultaten") but does not define the operation; its public definition
    is taken: every query head of batch b attends to the one
    latent cache of b, ckv[b] [Lk, Dqk].  Scores use all Dqk dims (latent
    part and positional part); the values are the first dv dims of the same
    rows.  The cascade is the three-pass one of ``attention``.

    q: [B, Hq, Dqk]; ckv: [B, Lk, Dqk].  Returns fp64 [B, Hq, dv], or
    [len(rows), dv] for a list of (b, hq) pairs.
    """
    B, Hq, _ = q.shape
    pairs = [(b, h) for b in range(B) for h in range(Hq)] if rows is None else list(rows)
    res = np.empty((len(pairs), dv), dtype=np.float64)
    cache_b, C = -1, None
    for i, (b, h) in enumerate(pairs):
        if b != cache_b:
            C = _f64(ckv[b])
            cache_b = b
        res[i] = three_pass_row(_f64(q[b, h]), C, C[:, :dv], scale)
    return res.reshape(B, Hq, dv) if rows is None else res


# ------------------------------------------------- the method's own forms


def attention_incremental(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                          tile: int) -> np.ndarray:
    """Single-loop incremental form ([E] §2.3 and §4.1; [S] Methodologie 2).

    Running state (m, l, o) is updated tile by tile.  When the running max
    grows from m to m', earlier terms were taken relative to m, so l and o
    are multiplied by exp(m - m') (the invertible dependent factor of the
    decomposition in [S] Methodologie 1).  The explainer's printed loop
    divides by the running sum inside the loop and adds the tile's sum
    without rescaling it; that does not reproduce the cascade, so the
    standard rescaled form is used and o is divided by l once at the end.
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    m = -np.inf
    l = 0.0
    o = np.zeros(V.shape[1])
    for a in range(0, K.shape[0], tile):
        s = scale * (K[a:a + tile] @ q)
        m_new = max(m, s.max())
        alpha = np.exp(m - m_new)      # 0 on the first tile (m = -inf)
        p = np.exp(s - m_new)
        l = l * alpha + p.sum()
        o = o * alpha + p @ V[a:a + tile]
        m = m_new
    return o / l


def segment_partial(q, K, V, scale: float, lo: int, hi: int):
    """Partial state of keys [lo, hi): (m, l, o) with o left unnormalised,
    i.e. o = sum_i exp(s_i - m) v_i.  An empty segment gives (-inf, 0, 0)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    if hi <= lo:
        return -np.inf, 0.0, np.zeros(V.shape[1])
    s = scale * (K[lo:hi] @ q)
    m = s.max()
    e = np.exp(s - m)
    return m, e.sum(), e @ V[lo:hi]


def merge_partials(parts) -> np.ndarray:
    """Merge of per-segment states ([S] Methodologie 3, multi-segment; [E]
    §3.3 inter-block): M = max_j m_j, w_j = exp(m_j - M),
    L = sum_j w_j l_j, O = sum_j w_j o_j / L."""
    M = max(p[0] for p in parts)
    L = 0.0
    O = np.zeros_like(parts[0][2])
    for m, l, o in parts:
        w = 0.0 if m == -np.inf else np.exp(m - M)
        L += w * l
        O += w * o
    return O / L


def attention_segments(q, K, V, scale: float, bounds) -> np.ndarray:
    """Multi-segment form: ``bounds`` = [b0=0, b1, ..., bS=Lk]; segment j
    holds keys [b_j, b_{j+1})."""
    parts = [segment_partial(q, K, V, scale, bounds[j], bounds[j + 1])
             for j in range(len(bounds) - 1)]
    return merge_partials(parts)
