"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  It shares no code
with the CUDA library in ``io_aware_exact_gb300``.  The dense functions'
arithmetic lives in ``attn_oracle.c`` (plain C, fp64), built by :func:`build`
with the host compiler, and this module only marshals numpy arrays into it.
Written here with numpy fp64 instead: the functions with an explicit
visibility mask (block-sparse layouts, a shifted causal mask for unequal
lengths), the exact merge of partial results and the backward with given
row statistics (chunked / ring attention), and dropout (Philox4x32-10, the
keep mask and dropout attention); grouped heads and packed batches compose
the single-head functions.

The functions follow, one head at a time:

* sj-techlog "FlashAttention 원 논문 해부", section "원 논문의 정의":
  S = tau Q K^T, P = softmax(S), O = P V, causal s_ij = -inf for j > i;
* wonbeomjang.kr FlashAttention-2 review, "개선 2: m과 l 대신 L만 저장":
  lse_i = m_i + log l_i (natural log, tau inside S);
* same review, "Backward Pass": dV = P^T dO, dP = dO V^T,
  dS_ij = P_ij (dP_ij - D_i), D_i = sum_j P_ij dP_ij, and (with tau inside S)
  dQ = tau dS K, dK = tau dS^T Q.

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` (page-printed worked examples, closed forms,
invariants and finite differences); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` (OpenMP if available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64, ci, cd = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, i64, i64, i64, i64, ci, cd,
                                                 ip, i64, dp, dp]
            lib.oracle_attn_bwd_rows.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, ci, cd,
                                                 ip, i64, dp, dp, dp]
            lib.oracle_attn_bwd_cols.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                                 ci, cd, ip, i64, dp, dp]
            for f in (lib.oracle_attn_fwd_rows, lib.oracle_attn_bwd_rows,
                      lib.oracle_attn_bwd_cols):
                f.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _idx(sel, n) -> np.ndarray:
    if sel is None:
        return np.arange(n, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1))


def _p(a):
    if a.dtype == np.int64:
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attention_forward(q, k, v, causal: bool, scale: float, rows=None):
    """O and lse of one head for the selected query rows (all by default).

    q [nq, d], k [nk, d], v [nk, dv] (any float dtype; upcast exactly to fp64).
    Returns (o [len(rows), dv], lse [len(rows)]), fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, d = q.shape
    nk, dv = v.shape
    assert k.shape == (nk, d)
    r = _idx(rows, nq)
    o = np.empty((r.size, dv), np.float64)
    lse = np.empty((r.size,), np.float64)
    rc = _load().oracle_attn_fwd_rows(_p(q), _p(k), _p(v), nq, nk, d, dv, int(bool(causal)),
                                      float(scale), _p(r), r.size, _p(o), _p(lse))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_rows rejected its arguments")
    return o, lse


def attention_backward_rows(q, k, v, dO, causal: bool, scale: float, rows=None,
                            with_dq: bool = True):
    """(lse, D, dQ) of one head for the selected query rows (all by default).

    With ``with_dq=False`` only lse and D are computed and dQ is None.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    nq, d = q.shape
    nk, dv = v.shape
    assert k.shape == (nk, d) and dO.shape == (nq, dv)
    r = _idx(rows, nq)
    lse = np.empty((r.size,), np.float64)
    D = np.empty((r.size,), np.float64)
    dq = np.empty((r.size, d), np.float64) if with_dq else None
    dq_p = _p(dq) if with_dq else ctypes.POINTER(ctypes.c_double)()
    rc = _load().oracle_attn_bwd_rows(_p(q), _p(k), _p(v), _p(dO), nq, nk, d, dv,
                                      int(bool(causal)), float(scale), _p(r), r.size,
                                      _p(lse), _p(D), dq_p)
    if rc != 0:
        raise ValueError("oracle_attn_bwd_rows rejected its arguments")
    return lse, D, dq


def attention_backward_cols(q, k, v, dO, lse_all, D_all, causal: bool, scale: float,
                            cols=None):
    """(dK, dV) of one head for the selected key columns (all by default).

    ``lse_all`` and ``D_all`` must be the oracle's own values for every row.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    lse_all, D_all = _f64(lse_all), _f64(D_all)
    nq, d = q.shape
    nk, dv = v.shape
    assert lse_all.shape == (nq,) and D_all.shape == (nq,)
    c = _idx(cols, nk)
    dk = np.empty((c.size, d), np.float64)
    dvo = np.empty((c.size, dv), np.float64)
    rc = _load().oracle_attn_bwd_cols(_p(q), _p(k), _p(v), _p(dO), _p(lse_all), _p(D_all),
                                      nq, nk, d, dv, int(bool(causal)), float(scale),
                                      _p(c), c.size, _p(dk), _p(dvo))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_cols rejected its arguments")
    return dk, dvo


def attention_backward(q, k, v, dO, causal: bool, scale: float):
    """Full backward of one head: (dQ, dK, dV, lse, D), fp64."""
    lse, D, dq = attention_backward_rows(q, k, v, dO, causal, scale)
    dk, dv = attention_backward_cols(q, k, v, dO, lse, D, causal, scale)
    return dq, dk, dv, lse, D


def kv_head_of(h: int, H: int, Hkv: int) -> int:
    """K / V head read by query head h when contiguous groups of H / Hkv query
    heads share one K / V head (grouped-query attention; Hkv = 1 is
    multi-query).  The paldyn.com survey lists GQA support among
    FlashAttention-2's additions ("v1에서 v3까지") without defining it; this
    is its plain reading."""
    assert Hkv >= 1 and H % Hkv == 0
    return h // (H // Hkv)


def attention_forward_grouped(q, k, v, causal: bool, scale: float):
    """O [H, nq, dv], lse [H, nq] for q [H, nq, d] and k, v [Hkv, nk, *]: each
    query head is single-head attention with its group's K / V head."""
    H, Hkv = len(q), len(k)
    outs = [attention_forward(q[h], k[kv_head_of(h, H, Hkv)], v[kv_head_of(h, H, Hkv)],
                              causal, scale) for h in range(H)]
    return np.stack([o for o, _ in outs]), np.stack([l for _, l in outs])


def attention_backward_grouped(q, k, v, dO, causal: bool, scale: float):
    """(dQ [H], dK [Hkv], dV [Hkv], lse [H], D [H]) for grouped K / V heads.

    dQ of a query head is the single-head dQ with its group's K / V.  K and V
    of a group enter every query head of the group, so by the chain rule
    their gradients are the sums of the single-head dK, dV over the group.
    """
    H, Hkv = len(q), len(k)
    dq = np.zeros(np.shape(q), np.float64)
    dk = np.zeros(np.shape(k), np.float64)
    dv = np.zeros(np.shape(v), np.float64)
    lse = np.zeros(np.shape(q)[:2], np.float64)
    D = np.zeros(np.shape(q)[:2], np.float64)
    for h in range(H):
        g = kv_head_of(h, H, Hkv)
        dq[h], dk_h, dv_h, lse[h], D[h] = attention_backward(q[h], k[g], v[g], dO[h], causal, scale)
        dk[g] += dk_h
        dv[g] += dv_h
    return dq, dk, dv, lse, D


def _seq_bounds(cu_seqlens):
    cu = [int(c) for c in cu_seqlens]
    assert cu[0] == 0 and all(a <= b for a, b in zip(cu, cu[1:]))
    return cu


def attention_forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool, scale: float):
    """Variable-length batch in the packed layout of the sj-techlog page
    ("2. module 경계는 ..."): the valid tokens of all sequences concatenated,
    q [total, H, d], k, v [total, Hkv, *], sequence b at tokens
    [cu_seqlens[b], cu_seqlens[b+1]).  Each sequence attends only to itself;
    the causal mask is per sequence.  Returns O [total, H, dv] and lse
    [B, H, max_seqlen] (lse of the page's {batch, heads, seq_len} shape; NaN
    past each sequence's length)."""
    cu = _seq_bounds(cu_seqlens)
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, H, _ = q.shape
    Hkv = k.shape[1]
    B = len(cu) - 1
    o = np.zeros((total, H, v.shape[2]), np.float64)
    lse = np.full((B, H, max_seqlen), np.nan, np.float64)
    for b in range(B):
        s0, s1 = cu[b], cu[b + 1]
        if s1 == s0:
            continue
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            ob, lb = attention_forward(q[s0:s1, h], k[s0:s1, g], v[s0:s1, g], causal, scale)
            o[s0:s1, h] = ob
            lse[b, h, :s1 - s0] = lb
    return o, lse


def attention_backward_varlen(q, k, v, dO, cu_seqlens, causal: bool, scale: float):
    """(dQ [total, H, d], dK [total, Hkv, d], dV [total, Hkv, dv]) of the
    packed variable-length batch above: each sequence and head is the
    single-head backward; dK, dV of a K / V head sum over its group."""
    cu = _seq_bounds(cu_seqlens)
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    total, H, _ = q.shape
    Hkv = k.shape[1]
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(v.shape, np.float64)
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        if s1 == s0:
            continue
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            dqb, dkb, dvb, _, _ = attention_backward(q[s0:s1, h], k[s0:s1, g], v[s0:s1, g],
                                                     dO[s0:s1, h], causal, scale)
            dq[s0:s1, h] = dqb
            dk[s0:s1, g] += dkb
            dv[s0:s1, g] += dvb
    return dq, dk, dv


def attention_forward_varlen_qk(q, k, v, cu_q, cu_k, max_seqlen_q: int, causal: bool,
                                scale: float):
    """Packed batch whose keys have lengths of their own: q [total_q, H, d]
    with sequence b at rows [cu_q[b], cu_q[b+1]), k, v [total_k, Hkv, *] with
    its keys at rows [cu_k[b], cu_k[b+1]).  Each sequence attends only to its
    own keys; with ``causal`` the mask is aligned bottom-right (key j visible
    to query i iff j <= i + Lk - Lq, attention_forward_offset).  Returns O
    [total_q, H, dv] and lse [B, H, max_seqlen_q] (NaN past each length)."""
    cq, ck = _seq_bounds(cu_q), _seq_bounds(cu_k)
    assert len(cq) == len(ck)
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, H, _ = q.shape
    Hkv = k.shape[1]
    B = len(cq) - 1
    o = np.zeros((total, H, v.shape[2]), np.float64)
    lse = np.full((B, H, max_seqlen_q), np.nan, np.float64)
    for b in range(B):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            ob, lb = attention_forward_offset(q[q0:q1, h], k[k0:k1, g], v[k0:k1, g], causal, scale,
                                              (k1 - k0) - (q1 - q0))
            o[q0:q1, h] = ob
            lse[b, h, :q1 - q0] = lb
    return o, lse


def attention_backward_varlen_qk(q, k, v, dO, cu_q, cu_k, causal: bool, scale: float):
    """(dQ [total_q, H, d], dK [total_k, Hkv, d], dV [total_k, Hkv, dv]) of
    attention_forward_varlen_qk: per sequence and head the single-head
    backward with the shifted causal mask; dK, dV sum over each group."""
    cq, ck = _seq_bounds(cu_q), _seq_bounds(cu_k)
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    H, Hkv = q.shape[1], k.shape[1]
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(v.shape, np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            dqb, dkb, dvb, _, _ = attention_backward_offset(q[q0:q1, h], k[k0:k1, g], v[k0:k1, g],
                                                            dO[q0:q1, h], causal, scale,
                                                            (k1 - k0) - (q1 - q0))
            dq[q0:q1, h] = dqb
            dk[k0:k1, g] += dkb
            dv[k0:k1, g] += dvb
    return dq, dk, dv


def expand_block_mask(block_mask, nq: int, nk: int, block: int, causal: bool) -> np.ndarray:
    """Element visibility [nq, nk] (True = key j enters row i's softmax) of a
    block-sparse layout: block_mask [ceil(nq / block), ceil(nk / block)], a
    nonzero entry keeps the block x block tile of scores, a zero entry drops
    it (sj-techlog "FlashAttention 원 논문 해부", section "대안, 비교와 선택
    기준": block-sparse FlashAttention skips the zero blocks of a block mask
    fixed in advance).  With ``causal`` the top-left causal mask applies on
    top (j <= i)."""
    bm = np.asarray(block_mask) != 0
    assert bm.shape == ((nq + block - 1) // block, (nk + block - 1) // block)
    vis = np.repeat(np.repeat(bm, block, axis=0), block, axis=1)[:nq, :nk]
    if causal:
        vis = vis & (np.arange(nk)[None, :] <= np.arange(nq)[:, None])
    return vis


def attention_forward_masked(q, k, v, visible, scale: float):
    """O [nq, dv] and lse [nq] of one head with an explicit visibility mask.

    S = tau Q K^T with invisible scores excluded, P the row softmax over the
    visible keys (row maximum subtracted), O = P V, lse_i = m_i + ln sum_j
    exp(s_ij - m_i) (same definitions as the rest of this module).  A row with
    no visible key has an empty softmax (the sj-techlog page's all-masked-row
    case, "값을 하나 바꾸는 경계 실험"); the reading taken is O = 0 and
    lse = -inf, the limit of a row whose keys all contribute nothing."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    vis = np.asarray(visible, dtype=bool)
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    has = vis.any(axis=1)
    m = np.where(has, s.max(axis=1, initial=-np.inf), 0.0)     # (no keys at all: every row empty)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    z = e.sum(axis=1)
    p = np.where(has[:, None], e / np.where(has, z, 1.0)[:, None], 0.0)
    lse = np.where(has, m + np.log(np.where(has, z, 1.0)), -np.inf)
    return p @ v, lse


def attention_backward_masked(q, k, v, dO, visible, scale: float):
    """(dQ, dK, dV, lse, D) of one head with an explicit visibility mask:
    the analytic backward of the FlashAttention-2 review ("Backward Pass"),
    dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P o (dP - D),
    dQ = tau dS K, dK = tau dS^T Q, with P = 0 on invisible entries.  Rows
    with no visible key contribute nothing."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    vis = np.asarray(visible, dtype=bool)
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    has = vis.any(axis=1)
    m = np.where(has, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    z = np.where(has, e.sum(axis=1), 1.0)
    p = e / z[:, None]
    lse = np.where(has, m + np.log(z), -np.inf)
    dv = p.T @ dO
    dp = dO @ v.T
    D = (p * dp).sum(axis=1)
    ds = p * (dp - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv, lse, D


def attention_forward_block_sparse(q, k, v, block_mask, causal: bool, scale: float,
                                   block: int = 128):
    """O, lse of one head under a block-sparse layout (see expand_block_mask)."""
    vis = expand_block_mask(block_mask, len(q), len(k), block, causal)
    return attention_forward_masked(q, k, v, vis, scale)


def attention_backward_block_sparse(q, k, v, dO, block_mask, causal: bool, scale: float,
                                    block: int = 128):
    """(dQ, dK, dV, lse, D) of one head under a block-sparse layout."""
    vis = expand_block_mask(block_mask, len(q), len(k), block, causal)
    return attention_backward_masked(q, k, v, dO, vis, scale)


def merge_partials(o1, lse1, o2, lse2):
    """Exact merge of two partial results of the same query rows over
    disjoint key sets (sj-techlog "FlashAttention 원 논문 해부", section "두
    tile을 한 row로 합치는 식": both states are rescaled by exp of their
    statistic minus the new maximum and the normaliser is renormalised).
    With normalised outputs o and natural-log logsumexps lse:
    lse = m + ln(e^{lse1-m} + e^{lse2-m}), m = max(lse1, lse2), and
    o = e^{lse1-lse} o1 + e^{lse2-lse} o2.  A side with lse = -inf (no
    visible key) has weight 0; two such sides give o = 0, lse = -inf."""
    o1, o2 = _f64(o1), _f64(o2)
    lse1, lse2 = _f64(lse1), _f64(lse2)
    m = np.maximum(lse1, lse2)
    fin = np.isfinite(m)
    ms = np.where(fin, m, 0.0)
    e1 = np.where(fin, np.exp(lse1 - ms), 0.0)
    e2 = np.where(fin, np.exp(lse2 - ms), 0.0)
    z = np.where(fin, e1 + e2, 1.0)
    lse = np.where(fin, ms + np.log(z), -np.inf)
    w1, w2 = e1 / z, e2 / z
    return w1[..., None] * o1 + w2[..., None] * o2, lse


def attention_backward_given_stats(q, k, v, dO, lse, D, causal: bool, scale: float,
                                   q_offset: int = 0):
    """(dQ, dK, dV) of one head's queries against one key / value chunk, with
    the rows' logsumexp and D taken as given (those of the whole key set the
    rows attend to): P_ij = exp(tau q_i.k_j - lse_i) on visible pairs, then
    the FlashAttention-2 review's backward ("Backward Pass"): dV = P^T dO,
    dP = dO V^T, dS = P o (dP - D), dQ = tau dS K, dK = tau dS^T Q.  Summed
    over the chunks of a split key set these are the gradients of the whole.
    With ``causal`` query i (row i + q_offset of the sequence, keys numbered
    from 0 in this chunk) sees key j iff j <= i + q_offset."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    lse, D = _f64(lse), _f64(D)
    nq, nk = len(q), len(k)
    vis = np.ones((nq, nk), bool)
    if causal:
        vis = np.arange(nk)[None, :] <= (np.arange(nq)[:, None] + q_offset)
    p = np.where(vis, np.exp(np.where(vis, scale * (q @ k.T), 0.0) - lse[:, None]), 0.0)
    dp = dO @ v.T
    ds = p * (dp - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), p.T @ dO


# --------------------------------------------------------------------------
# Dropout (the sj-techlog page, backward section: the forward keeps the
# pseudo-random generator's state and the backward regenerates the same
# dropout mask from it instead of storing it).  The generator is Philox4x32-10
# (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
# SC'11), written here from that definition.
# --------------------------------------------------------------------------

_PHILOX_M0, _PHILOX_M1 = 0xD2511F53, 0xCD9E8D57      # round multipliers
_PHILOX_W0, _PHILOX_W1 = 0x9E3779B9, 0xBB67AE85      # Weyl key increments
_MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds.  counter: uint array [..., 4], key: uint
    array [..., 2] (broadcast); returns uint32 [..., 4].  One round maps
    (c0, c1, c2, c3) with key (k0, k1) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
    hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key gains (W0, W1) between rounds."""
    c = [np.asarray(counter, dtype=np.uint64)[..., i] & _MASK32 for i in range(4)]
    k0 = np.asarray(key, dtype=np.uint64)[..., 0] & _MASK32
    k1 = np.asarray(key, dtype=np.uint64)[..., 1] & _MASK32
    for _ in range(10):
        p0 = np.uint64(_PHILOX_M0) * c[0]
        p1 = np.uint64(_PHILOX_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK32)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(_PHILOX_W0)) & np.uint64(_MASK32)
        k1 = (k1 + np.uint64(_PHILOX_W1)) & np.uint64(_MASK32)
    return np.stack(c, axis=-1).astype(np.uint32)


def dropout_threshold(p_drop: float) -> int:
    """Keep threshold t on a random byte: keep iff byte < t, with
    t = round(256 (1 - p_drop)) clamped to [1, 256]; the kept weights are
    scaled by 256 / t, so the expected output is the undropped one."""
    return int(min(256, max(1, round(256.0 * (1.0 - p_drop)))))


def dropout_keep(bh: int, nq: int, nk: int, p_drop: float, seed: int, offset: int):
    """Keep mask [nq, nk] of one (batch, head) index bh.  Element (i, j) takes
    byte j % 4 (bits 8 (j % 4) .. 8 (j % 4) + 7) of output word i % 4 of
    Philox4x32-10 with counter (j // 4, i // 4, bh, offset) and key
    (seed mod 2^32, seed div 2^32): one call covers a 4 x 4 patch."""
    qi, kj = np.meshgrid(np.arange(nq), np.arange(nk), indexing="ij")
    ctr = np.stack([kj // 4, qi // 4, np.full_like(qi, bh), np.full_like(qi, offset)], axis=-1)
    key = np.array([seed & _MASK32, (seed >> 32) & _MASK32], dtype=np.uint64)
    words = philox4x32_10(ctr.astype(np.uint64), key)
    w = np.take_along_axis(words, (qi % 4)[..., None], axis=-1)[..., 0].astype(np.uint64)
    byte = (w >> (8 * (kj % 4)).astype(np.uint64)) & np.uint64(0xFF)
    return byte < np.uint64(dropout_threshold(p_drop))


def attention_forward_dropout(q, k, v, causal: bool, scale: float, keep, p_drop: float):
    """O and lse of one head with dropout applied to P (sj-techlog page,
    backward section; FlashAttention's dropout on the softmax output):
    O = (P o Z) V * 256 / t with Z the keep mask and t the keep threshold;
    lse is that of the undropped softmax."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, nk = len(q), len(k)
    vis = np.ones((nq, nk), bool)
    if causal:
        vis = np.arange(nk)[None, :] <= np.arange(nq)[:, None]
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    m = s.max(axis=1)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    z = e.sum(axis=1)
    p = e / z[:, None]
    w = 256.0 / dropout_threshold(p_drop)
    return (p * np.asarray(keep)) @ v * w, m + np.log(z)


def attention_backward_dropout(q, k, v, dO, causal: bool, scale: float, keep, p_drop: float):
    """(dQ, dK, dV) of attention_forward_dropout: with P~ = P o Z * w
    (w = 256 / t), dV = P~^T dO, dP = Z o (dO V^T) * w, D_i = sum_j P_ij dP_ij
    (= rowsum(dO o O)), dS = P o (dP - D), dQ = tau dS K, dK = tau dS^T Q."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    nq, nk = len(q), len(k)
    vis = np.ones((nq, nk), bool)
    if causal:
        vis = np.arange(nk)[None, :] <= np.arange(nq)[:, None]
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    m = s.max(axis=1)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    p = e / e.sum(axis=1)[:, None]
    zw = np.asarray(keep) * (256.0 / dropout_threshold(p_drop))
    dv = (p * zw).T @ dO
    dp = (dO @ v.T) * zw
    D = (p * dp).sum(axis=1)
    ds = p * (dp - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv


def attention_forward_offset(q, k, v, causal: bool, scale: float, offset: int):
    """O, lse of one head whose nq queries attend to nk keys with the causal
    mask shifted by ``offset``: key j is visible to query i iff
    j <= i + offset.  offset = nk - nq aligns the last query with the last
    key (bottom-right, e.g. a query chunk after nk - nq cached keys);
    offset = 0 is the top-left mask of the rest of this module.  Rows with no
    visible key give O = 0, lse = -inf (the block-sparse reading)."""
    nq, nk = len(q), len(k)
    vis = np.ones((nq, nk), bool)
    if causal:
        vis = np.arange(nk)[None, :] <= (np.arange(nq)[:, None] + offset)
    return attention_forward_masked(q, k, v, vis, scale)


def attention_backward_offset(q, k, v, dO, causal: bool, scale: float, offset: int):
    """(dQ, dK, dV, lse, D) of attention_forward_offset."""
    nq, nk = len(q), len(k)
    vis = np.ones((nq, nk), bool)
    if causal:
        vis = np.arange(nk)[None, :] <= (np.arange(nq)[:, None] + offset)
    return attention_backward_masked(q, k, v, dO, vis, scale)
