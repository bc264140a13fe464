"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself.  Each test ties it to something
independent: values a page prints for a worked example (fixtures under
``tests/golden/``), closed forms, invariants of softmax attention, an
independently written online-softmax recurrence, and central finite
differences of the forward for the backward.  The mistakes these are meant to
catch include a dropped softmax scale, a transposed operand, a wrong causal
boundary (j < i instead of j <= i), a missing max-subtraction, a wrong sign in
dS and a wrong D.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Page-printed worked examples
# --------------------------------------------------------------------------

def test_merge_worked_example():
    """sj-techlog page, section "12살 숫자 예": fold new scores [3,1] (values
    [10,20]) into the state m=2, l=1.5, u=6.  Two earlier keys with scores 2 and
    2+ln(1/2) and values 6 and 0 produce exactly that state, so the whole row
    is the four keys together and the oracle's O, lse must give the printed
    l', u', o'."""
    g = _golden("page1_merge_example.json")
    st, new, pr, rnd = g["state_before"], g["new_tile"], g["printed"], g["printed_rounding"]
    prev_scores = [st["m"], st["m"] + math.log(0.5)]
    prev_values = [st["u"], 0.0]
    # the constructed earlier keys reproduce the printed state exactly
    o_prev, lse_prev = oracle.attention_forward([[1.0]], [[s] for s in prev_scores],
                                                [[x] for x in prev_values], False, 1.0)
    assert abs(lse_prev[0] - (st["m"] + math.log(st["l"]))) < 1e-14
    assert abs(o_prev[0, 0] - st["u"] / st["l"]) < 1e-14

    # the new tile alone: printed tilde_l, tilde_u
    o_t, lse_t = oracle.attention_forward([[1.0]], [[s] for s in new["scores"]],
                                          [[x] for x in new["values"]], False, 1.0)
    l_t = math.exp(lse_t[0] - max(new["scores"]))
    assert abs(l_t - pr["tilde_l"]) < 1e-4
    assert abs(o_t[0, 0] * l_t - pr["tilde_u"]) < 1e-4

    scores = prev_scores + new["scores"]
    values = prev_values + new["values"]
    o, lse = oracle.attention_forward([[1.0]], [[s] for s in scores], [[x] for x in values],
                                      False, 1.0)
    l_new = math.exp(lse[0] - pr["m_new"])
    assert abs(l_new - pr["l_new"]) <= rnd["l_new"]
    assert abs(o[0, 0] * l_new - pr["u_new"]) <= rnd["u_new"]
    assert abs(o[0, 0] - pr["o_new"]) <= rnd["o_new"]


def test_n5_example_printed_values():
    """sj-techlog page, section "직접 검증과 재현": causal row 0 is [1, 0], and
    row 4's running (m, l) after key blocks [0,2), [0,4), [0,5) are printed;
    m + ln l is the log-normaliser over those keys."""
    g = _golden("page1_n5_example.json")
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    tau = 1.0 / math.sqrt(q.shape[1])
    o, _ = oracle.attention_forward(q, k, v, True, tau)
    assert np.array_equal(o[0], np.array(g["printed"]["causal_row0_output"]))
    for st in g["printed"]["row4_block2_states"]:
        end = st["keys"][1]
        _, lse = oracle.attention_forward(q, k[:end], v[:end], False, tau, rows=[4])
        want = st["m"] + math.log(st["l"])
        assert abs(lse[0] - want) < 2e-6, (end, lse[0], want)
        # row 4 sees every key, so causal and non-causal agree on it
        _, lse_c = oracle.attention_forward(q, k, v, True, tau, rows=[4])
        if end == 5:
            assert abs(lse_c[0] - want) < 2e-6


def _online_recurrence(q, k, v, tau, causal, block):
    """Independent restatement of the tile-by-tile recurrence (sj-techlog page,
    section "두 tile을 한 row로 합치는 식"), used only as a second algorithm."""
    nq, nk = q.shape[0], k.shape[0]
    out = np.zeros((nq, v.shape[1]))
    lse = np.zeros(nq)
    for i in range(nq):
        m, l, u = -np.inf, 0.0, np.zeros(v.shape[1])
        for start in range(0, nk, block):
            idx = [j for j in range(start, min(start + block, nk)) if not causal or j <= i]
            if not idx:
                continue
            s = np.array([tau * float(np.dot(q[i], k[j])) for j in idx])
            mt = s.max()
            lt = np.exp(s - mt).sum()
            ut = (np.exp(s - mt)[:, None] * v[idx]).sum(axis=0)
            mn = max(m, mt)
            a = 0.0 if m == -np.inf else math.exp(m - mn)
            b = math.exp(mt - mn)
            l, u, m = a * l + b * lt, a * u + b * ut, mn
        out[i] = u / l
        lse[i] = m + math.log(l)
    return out, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 2, 3])
def test_n5_example_tiled_equals_standard(causal, block):
    """The page reports tiled == standard within 1e-12 for block sizes 1, 2, 3
    on its N=5 inputs, causal and not."""
    g = _golden("page1_n5_example.json")
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    tau = 1.0 / math.sqrt(3.0)
    o, lse = oracle.attention_forward(q, k, v, causal, tau)
    o2, lse2 = _online_recurrence(q, k, v, tau, causal, block)
    assert np.max(np.abs(o - o2)) <= g["printed"]["tiled_equals_standard_tol"]
    assert np.max(np.abs(lse - lse2)) <= 1e-12


def test_random_tiled_equals_standard():
    r = _rng(1)
    q, k, v = r.normal(size=(9, 4)), r.normal(size=(11, 4)), r.normal(size=(11, 3))
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, causal, 0.8)
        o2, lse2 = _online_recurrence(q, k, v, 0.8, causal, 4)
        assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(lse - lse2)) < 1e-12


# --------------------------------------------------------------------------
# Closed forms and invariants of the forward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    """With V = 1 every output entry equals the row sum of P, which is 1."""
    r = _rng(2)
    q, k = 3 * r.normal(size=(13, 6)), 3 * r.normal(size=(13, 6))
    o, _ = oracle.attention_forward(q, k, np.ones((13, 2)), causal, 1 / math.sqrt(6))
    assert np.max(np.abs(o - 1.0)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding w to every key adds tau q_i.w to all of row i's scores: O is
    unchanged (softmax shift invariance) and lse shifts by exactly tau q_i.w."""
    r = _rng(3)
    q, k, v = r.normal(size=(10, 5)), r.normal(size=(10, 5)), r.normal(size=(10, 4))
    w = r.normal(size=5)
    tau = 0.6
    o, lse = oracle.attention_forward(q, k, v, causal, tau)
    o2, lse2 = oracle.attention_forward(q, k + w, v, causal, tau)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse2 - lse - tau * q @ w)) < 1e-12


def test_key_value_permutation_equivariance():
    r = _rng(4)
    q, k, v = r.normal(size=(7, 4)), r.normal(size=(12, 4)), r.normal(size=(12, 3))
    perm = r.permutation(12)
    o, lse = oracle.attention_forward(q, k, v, False, 0.5)
    o2, lse2 = oracle.attention_forward(q, k[perm], v[perm], False, 0.5)
    assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(lse - lse2)) < 1e-12


def test_zero_query_gives_mean_and_log_count():
    """Q = 0 makes all visible scores equal: O is the (prefix) mean of V and
    lse is ln of the number of visible keys."""
    r = _rng(5)
    n = 9
    k, v = r.normal(size=(n, 4)), r.normal(size=(n, 3))
    q = np.zeros((n, 4))
    o, lse = oracle.attention_forward(q, k, v, False, 0.5)
    assert np.max(np.abs(o - v.mean(axis=0))) < 1e-12
    assert np.max(np.abs(lse - math.log(n))) < 1e-12
    o, lse = oracle.attention_forward(q, k, v, True, 0.5)
    for i in range(n):
        assert np.max(np.abs(o[i] - v[: i + 1].mean(axis=0))) < 1e-12
        assert abs(lse[i] - math.log(i + 1)) < 1e-12


def test_large_margin_key_selects_one_value_row():
    d = 8
    k = np.eye(d)
    r = _rng(6)
    v = r.normal(size=(d, 5))
    sel = [3, 0, 7, 5]
    q = np.stack([1000.0 * np.eye(d)[j] for j in sel])
    o, _ = oracle.attention_forward(q, k, v, False, 1 / math.sqrt(d))
    assert np.max(np.abs(o - v[sel])) < 1e-12


def test_causal_first_row_is_first_value():
    r = _rng(7)
    q, k, v = 5 * r.normal(size=(6, 4)), 5 * r.normal(size=(6, 4)), r.normal(size=(6, 4))
    o, lse = oracle.attention_forward(q, k, v, True, 0.5)
    assert np.array_equal(o[0], v[0])
    assert abs(lse[0] - 0.5 * float(q[0] @ k[0])) < 1e-12


def test_huge_scores_do_not_overflow():
    """Scores around 1e4 overflow exp() unless the row max is subtracted."""
    r = _rng(8)
    q, k, v = 100 * r.normal(size=(6, 4)), 100 * r.normal(size=(6, 4)), r.normal(size=(6, 2))
    o, lse = oracle.attention_forward(q, k, v, False, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.max(np.abs(o - oracle.attention_forward(q, k + 3.0, v, False, 1.0)[0])) < 1e-9


def test_row_subset_matches_full():
    r = _rng(9)
    q, k, v = r.normal(size=(20, 4)), r.normal(size=(20, 4)), r.normal(size=(20, 4))
    o, lse = oracle.attention_forward(q, k, v, True, 0.5)
    rows = [19, 0, 7, 7]
    o2, lse2 = oracle.attention_forward(q, k, v, True, 0.5, rows=rows)
    assert np.array_equal(o2, o[rows]) and np.array_equal(lse2, lse[rows])


def test_bad_rows_rejected():
    z = np.zeros((3, 2))
    with pytest.raises(ValueError):
        oracle.attention_forward(z, z, z, False, 1.0, rows=[3])


# --------------------------------------------------------------------------
# Backward
# --------------------------------------------------------------------------

def _loss(q, k, v, dO, causal, tau):
    o, _ = oracle.attention_forward(q, k, v, causal, tau)
    return float(np.sum(o * dO))


def _fd_grad(x, f, h=1e-6):
    g = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("causal,nq,nk", [(False, 5, 5), (True, 5, 5), (False, 4, 6),
                                          (True, 6, 4)])
def test_backward_matches_finite_differences(causal, nq, nk):
    """Central differences of L = sum(dO * O) w.r.t. every entry of Q, K, V.
    tau = 0.7 is neither 1 nor 1/sqrt(d), so a dropped scale shows; d != dv
    and nq != nk catch transposed operands."""
    r = _rng(10 + nq + nk + int(causal))
    d, dv, tau = 3, 2, 0.7
    q, k, v = r.normal(size=(nq, d)), r.normal(size=(nk, d)), r.normal(size=(nk, dv))
    dO = r.normal(size=(nq, dv))
    dq, dk, dvv, _, _ = oracle.attention_backward(q, k, v, dO, causal, tau)
    gq = _fd_grad(q, lambda x: _loss(x, k, v, dO, causal, tau))
    gk = _fd_grad(k, lambda x: _loss(q, x, v, dO, causal, tau))
    gv = _fd_grad(v, lambda x: _loss(q, k, x, dO, causal, tau))
    for got, want in ((dq, gq), (dk, gk), (dvv, gv)):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_backward_identities(causal):
    """D_i = rowsum(dO o O); sum_j dS_ij = 0 makes the column sums of dK vanish
    and dQ invariant to a shift of all keys; sum_j P_ij = 1 makes the column
    sums of dV equal those of dO."""
    r = _rng(20 + int(causal))
    n, d, tau = 16, 8, 1 / math.sqrt(8)
    q, k, v, dO = (2 * r.normal(size=(n, d)) for _ in range(4))
    dq, dk, dvv, lse, D = oracle.attention_backward(q, k, v, dO, causal, tau)
    o, lse_f = oracle.attention_forward(q, k, v, causal, tau)
    assert np.max(np.abs(D - np.sum(dO * o, axis=1))) < 1e-12
    assert np.max(np.abs(lse - lse_f)) < 1e-12
    assert np.max(np.abs(dk.sum(axis=0))) < 1e-12
    assert np.max(np.abs(dvv.sum(axis=0) - dO.sum(axis=0))) < 1e-12
    w = r.normal(size=d)
    dq2, _, _, _, _ = oracle.attention_backward(q, k + w, v, dO, causal, tau)
    assert np.max(np.abs(dq2 - dq)) < 1e-11


def test_backward_zero_upstream_gradient():
    r = _rng(30)
    q, k, v = r.normal(size=(7, 4)), r.normal(size=(7, 4)), r.normal(size=(7, 4))
    dq, dk, dvv, _, D = oracle.attention_backward(q, k, v, np.zeros((7, 4)), True, 0.5)
    assert not np.any(dq) and not np.any(dk) and not np.any(dvv) and not np.any(D)


def test_backward_column_subset_matches_full():
    r = _rng(31)
    n = 12
    q, k, v, dO = (r.normal(size=(n, 4)) for _ in range(4))
    dq, dk, dvv, lse, D = oracle.attention_backward(q, k, v, dO, True, 0.5)
    cols = [11, 2, 5]
    dk2, dv2 = oracle.attention_backward_cols(q, k, v, dO, lse, D, True, 0.5, cols=cols)
    assert np.array_equal(dk2, dk[cols]) and np.array_equal(dv2, dvv[cols])
    lse3, D3, dq3 = oracle.attention_backward_rows(q, k, v, dO, True, 0.5, rows=[4, 9])
    assert np.array_equal(dq3, dq[[4, 9]]) and np.array_equal(D3, D[[4, 9]])


# --------------------------------------------------------------------------
# Grouped K / V heads
# --------------------------------------------------------------------------

def test_grouped_head_mapping_is_contiguous():
    """Query heads 0..3 share K / V head 0 and 4..7 head 1 (H=8, Hkv=2); one
    K / V head serves all (multi-query); Hkv = H is plain multi-head."""
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 3, 1) for h in range(3)] == [0, 0, 0]
    assert [oracle.kv_head_of(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]


@pytest.mark.parametrize("H,Hkv,causal", [(4, 2, False), (4, 2, True), (3, 1, True)])
def test_grouped_backward_matches_finite_differences(H, Hkv, causal):
    """Central differences of L = sum over query heads of sum(dO_h * O_h)
    w.r.t. every entry of the shared K and V (and of Q): a dK / dV that is
    not summed over the group, or summed over the wrong heads, fails."""
    r = _rng(40 + H + Hkv + int(causal))
    n, d, dv, tau = 4, 3, 2, 0.7
    q, dO = r.normal(size=(H, n, d)), r.normal(size=(H, n, dv))
    k, v = r.normal(size=(Hkv, n, d)), r.normal(size=(Hkv, n, dv))

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward_grouped(qq, kk, vv, causal, tau)
        return float(np.sum(o * dO))

    dq, dk, dvv, _, _ = oracle.attention_backward_grouped(q, k, v, dO, causal, tau)
    gq = _fd_grad(q, lambda x: loss(x, k, v))
    gk = _fd_grad(k, lambda x: loss(q, x, v))
    gv = _fd_grad(v, lambda x: loss(q, k, x))
    for got, want in ((dq, gq), (dk, gk), (dvv, gv)):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6


# --------------------------------------------------------------------------
# Variable-length (packed) batches
# --------------------------------------------------------------------------

def _block_diag_attention(q, k, v, cu, causal, tau):
    """Brute force over the concatenated tokens: score -inf between tokens of
    different sequences (and above the diagonal within one if causal),
    softmax over every key of the whole batch, one head at a time."""
    total, H, _ = q.shape
    Hkv = k.shape[1]
    seq = np.zeros(total, np.int64)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    pos = np.arange(total) - np.asarray(cu)[seq]
    o = np.zeros((total, H, v.shape[2]))
    for h in range(H):
        g = h // (H // Hkv)
        s = tau * q[:, h] @ k[:, g].T
        allowed = seq[:, None] == seq[None, :]
        if causal:
            allowed &= pos[None, :] <= pos[:, None]
        s = np.where(allowed, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        o[:, h] = (p / p.sum(axis=1, keepdims=True)) @ v[:, g]
    return o


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_forward_matches_block_diagonal_mask(causal):
    r = _rng(60 + int(causal))
    cu = [0, 3, 4, 4, 9]                 # lengths 3, 1, 0, 5
    q, k, v = r.normal(size=(9, 4, 3)), r.normal(size=(9, 2, 3)), r.normal(size=(9, 2, 2))
    o, lse = oracle.attention_forward_varlen(q, k, v, cu, 6, causal, 0.7)
    want = _block_diag_attention(q, k, v, cu, causal, 0.7)
    assert np.max(np.abs(o - want)) < 1e-12
    assert np.all(np.isnan(lse[2])) and np.all(np.isnan(lse[1, :, 1:]))
    assert np.all(np.isfinite(lse[3, :, :5]))


def test_varlen_backward_matches_finite_differences():
    r = _rng(70)
    cu = [0, 2, 2, 5]
    q, dO = r.normal(size=(5, 2, 3)), r.normal(size=(5, 2, 2))
    k, v = r.normal(size=(5, 1, 3)), r.normal(size=(5, 1, 2))

    def loss(qq, kk, vv):
        return float(np.sum(_block_diag_attention(qq, kk, vv, cu, True, 0.7) * dO))

    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, dO, cu, True, 0.7)
    for got, want in ((dq, _fd_grad(q, lambda x: loss(x, k, v))),
                      (dk, _fd_grad(k, lambda x: loss(q, x, v))),
                      (dv, _fd_grad(v, lambda x: loss(q, k, x)))):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6


def _packed_qk_attention(q, k, v, cu_q, cu_k, causal, tau):
    """Brute force over the whole packed batch: one softmax per packed query
    row over every packed key row, with a mask that allows only the row's own
    sequence and, when causal, keys at position <= query position + Lk - Lq."""
    nq, nk = len(q), len(k)
    sq = np.searchsorted(cu_q, np.arange(nq), side="right") - 1
    sk = np.searchsorted(cu_k, np.arange(nk), side="right") - 1
    pq = np.arange(nq) - np.asarray(cu_q)[sq]
    pk = np.arange(nk) - np.asarray(cu_k)[sk]
    lq = np.diff(cu_q)[sq]
    lk = np.diff(cu_k)[sk]
    H, Hkv = q.shape[1], k.shape[1]
    o = np.zeros((nq, H, v.shape[2]))
    for h in range(H):
        g = h // (H // Hkv)
        allowed = sq[:, None] == sk[None, :]
        if causal:
            allowed &= pk[None, :] <= pq[:, None] + lk[None, :] - lq[:, None]
        s = np.where(allowed, tau * q[:, h] @ k[:, g].T, -np.inf)
        has = allowed.any(axis=1)
        m = np.where(has, s.max(axis=1), 0.0)
        p = np.where(allowed, np.exp(s - m[:, None]), 0.0)
        z = np.where(has, p.sum(axis=1), 1.0)
        o[:, h] = (p / z[:, None]) @ v[:, g]
    return o


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_qk_forward_matches_packed_mask(causal):
    """Keys of their own lengths: 5 queries against 8 keys (a query chunk
    after 3 earlier keys), 6 against 2 (the first 4 queries see no key under
    the bottom-right mask: O = 0, lse = -inf), an empty query set with 3 keys,
    1 against 1, and 2 queries without keys; every row equals brute-force
    attention over the whole packed batch with the sequence and shifted
    causal mask written out."""
    r = _rng(75 + int(causal))
    cu_q, cu_k = [0, 5, 11, 11, 12, 14], [0, 8, 10, 13, 14, 14]
    q, k, v = r.normal(size=(14, 4, 3)), r.normal(size=(14, 2, 3)), r.normal(size=(14, 2, 2))
    o, lse = oracle.attention_forward_varlen_qk(q, k, v, cu_q, cu_k, 6, causal, 0.7)
    want = _packed_qk_attention(q, k, v, np.array(cu_q), np.array(cu_k), causal, 0.7)
    assert np.max(np.abs(o - want)) < 1e-12
    if causal:
        assert np.all(o[5:9] == 0.0) and np.all(lse[1, :, :4] == -np.inf)
        assert np.all(np.isfinite(lse[1, :, 4:6]))
    assert np.all(np.isnan(lse[2]))
    # the last sequence has 2 queries and no keys: empty rows, causal or not
    assert np.all(o[12:14] == 0.0) and np.all(lse[4, :, :2] == -np.inf)
    # equal lengths: the packed function of one cu_seqlens
    cu = [0, 3, 7]
    q2, k2, v2 = r.normal(size=(7, 2, 3)), r.normal(size=(7, 1, 3)), r.normal(size=(7, 1, 2))
    a, la = oracle.attention_forward_varlen_qk(q2, k2, v2, cu, cu, 4, causal, 0.7)
    b, lb = oracle.attention_forward_varlen(q2, k2, v2, cu, 4, causal, 0.7)
    assert np.max(np.abs(a - b)) < 1e-13 and np.allclose(la, lb, equal_nan=True)


def test_varlen_qk_backward_matches_finite_differences():
    r = _rng(80)
    cu_q, cu_k = [0, 3, 7], [0, 5, 7]      # 3 queries on 5 keys; 4 queries on 2 keys
    q, dO = r.normal(size=(7, 2, 3)), r.normal(size=(7, 2, 2))
    k, v = r.normal(size=(7, 1, 3)), r.normal(size=(7, 1, 2))

    def loss(qq, kk, vv):
        return float(np.sum(_packed_qk_attention(qq, kk, vv, np.array(cu_q), np.array(cu_k),
                                                 True, 0.7) * dO))

    dq, dk, dv = oracle.attention_backward_varlen_qk(q, k, v, dO, cu_q, cu_k, True, 0.7)
    assert np.all(dq[3:5] == 0.0)          # rows that see no key
    for got, want in ((dq, _fd_grad(q, lambda x: loss(x, k, v))),
                      (dk, _fd_grad(k, lambda x: loss(q, x, v))),
                      (dv, _fd_grad(v, lambda x: loss(q, k, x)))):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6


# --------------------------------------------------------------------------
# Block-sparse layouts (numpy fp64 functions of the oracle)
# --------------------------------------------------------------------------

def _visible_keys_by_hand(bm, i, nk, block, causal):
    return [j for j in range(nk) if bm[i // block][j // block] and (not causal or j <= i)]


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_rows_match_attention_over_their_keys(causal):
    """Every row of the block-sparse forward equals plain attention (the C
    oracle) of that query over exactly the keys its blocks keep, listed by
    hand; a row whose blocks are all dropped gives O = 0 and lse = -inf.  An
    asymmetric mask with a ragged last block catches a transposed mask, an
    off-by-one block index and a lost causal mask."""
    r = _rng(80 + int(causal))
    nq = nk = 11
    block, d, dv, tau = 3, 3, 2, 0.7
    bm = np.array([[1, 0, 0, 1], [1, 1, 0, 0], [0, 0, 0, 0], [0, 1, 1, 1]], np.uint8)
    q, k, v = r.normal(size=(nq, d)), r.normal(size=(nk, d)), r.normal(size=(nk, dv))
    o, lse = oracle.attention_forward_block_sparse(q, k, v, bm, causal, tau, block=block)
    for i in range(nq):
        sel = _visible_keys_by_hand(bm, i, nk, block, causal)
        if not sel:
            assert np.all(o[i] == 0.0) and lse[i] == -np.inf
            continue
        oi, li = oracle.attention_forward(q[i:i + 1], k[sel], v[sel], False, tau)
        assert np.max(np.abs(o[i] - oi[0])) < 1e-13
        assert abs(lse[i] - li[0]) < 1e-13
    assert np.all(o[6:9] == 0.0)                 # query block 2 keeps no key block


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_full_mask_is_dense_attention(causal):
    """An all-ones block mask leaves plain (causal) attention, forward and
    backward, as the C oracle computes it."""
    r = _rng(82 + int(causal))
    n, block, tau = 10, 4, 0.6
    q, k, v, dO = (r.normal(size=(n, 3)) for _ in range(4))
    bm = np.ones((3, 3), np.uint8)
    o, lse = oracle.attention_forward_block_sparse(q, k, v, bm, causal, tau, block=block)
    o2, lse2 = oracle.attention_forward(q, k, v, causal, tau)
    assert np.max(np.abs(o - o2)) < 1e-13 and np.max(np.abs(lse - lse2)) < 1e-13
    got = oracle.attention_backward_block_sparse(q, k, v, dO, bm, causal, tau, block=block)
    want = oracle.attention_backward(q, k, v, dO, causal, tau)
    for a, b in zip(got, want):
        assert np.max(np.abs(a - b)) < 1e-12


def test_block_sparse_diagonal_mask_is_independent_blocks():
    """A block-diagonal mask is attention within each block: the C oracle
    run on each block's slice alone (the last block ragged), forward and
    backward."""
    r = _rng(84)
    n, block, tau = 10, 4, 0.8
    q, k, v, dO = (r.normal(size=(n, 2)) for _ in range(4))
    bm = np.eye(3, dtype=np.uint8)
    o, lse = oracle.attention_forward_block_sparse(q, k, v, bm, False, tau, block=block)
    dq, dk, dv, _, _ = oracle.attention_backward_block_sparse(q, k, v, dO, bm, False, tau,
                                                              block=block)
    for s0 in range(0, n, block):
        sl = slice(s0, min(n, s0 + block))
        ob, lb = oracle.attention_forward(q[sl], k[sl], v[sl], False, tau)
        gq, gk, gv, _, _ = oracle.attention_backward(q[sl], k[sl], v[sl], dO[sl], False, tau)
        for a, b in ((o[sl], ob), (lse[sl], lb), (dq[sl], gq), (dk[sl], gk), (dv[sl], gv)):
            assert np.max(np.abs(a - b)) < 1e-12


def test_block_sparse_dropped_keys_do_not_matter():
    """Keys and values in key blocks that no query block keeps can be
    anything: outputs unchanged, and their dK, dV are exactly zero."""
    r = _rng(86)
    n, block, tau = 9, 3, 0.7
    bm = np.array([[1, 0, 1], [1, 0, 0], [0, 0, 1]], np.uint8)  # key block 1 dropped
    q, k, v, dO = (r.normal(size=(n, 3)) for _ in range(4))
    k2, v2 = k.copy(), v.copy()
    k2[3:6] = 50 * r.normal(size=(3, 3))
    v2[3:6] = r.normal(size=(3, 3))
    a = oracle.attention_forward_block_sparse(q, k, v, bm, True, tau, block=block)
    b = oracle.attention_forward_block_sparse(q, k2, v2, bm, True, tau, block=block)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    _, dk, dv, _, _ = oracle.attention_backward_block_sparse(q, k, v, dO, bm, True, tau,
                                                             block=block)
    assert np.all(dk[3:6] == 0.0) and np.all(dv[3:6] == 0.0)


def test_block_sparse_backward_matches_finite_differences():
    """Central differences of L = sum(dO * O) for the block-sparse forward,
    causal, with an empty query block (its dQ must be zero); d != dv."""
    r = _rng(88)
    n, block, tau = 8, 3, 0.7
    bm = np.array([[1, 0, 1], [0, 0, 0], [1, 1, 1]], np.uint8)
    q, k = r.normal(size=(n, 3)), r.normal(size=(n, 3))
    v, dO = r.normal(size=(n, 2)), r.normal(size=(n, 2))

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward_block_sparse(qq, kk, vv, bm, True, tau, block=block)
        return float(np.sum(o * dO))

    dq, dk, dv, _, D = oracle.attention_backward_block_sparse(q, k, v, dO, bm, True, tau,
                                                              block=block)
    for got, want in ((dq, _fd_grad(q, lambda x: loss(x, k, v))),
                      (dk, _fd_grad(k, lambda x: loss(q, x, v))),
                      (dv, _fd_grad(v, lambda x: loss(q, k, x)))):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6
    assert np.all(dq[3:6] == 0.0) and np.all(D[3:6] == 0.0)


# --------------------------------------------------------------------------
# Combining partial results over a split key set
# --------------------------------------------------------------------------

def test_merge_partials_reproduces_printed_merge_example():
    """sj-techlog page, section "12살 숫자 예": the state m = 2, l = 1.5, u = 6
    merged with the new tile (scores [3, 1], values [10, 20]; printed
    tilde_l, tilde_u) gives the printed l', o'."""
    g = _golden("page1_merge_example.json")
    st, pr, rnd = g["state_before"], g["printed"], g["printed_rounding"]
    o1, lse1 = st["u"] / st["l"], st["m"] + math.log(st["l"])
    o2, lse2 = pr["tilde_u"] / pr["tilde_l"], pr["m_new"] + math.log(pr["tilde_l"])
    o, lse = oracle.merge_partials([[o1]], [lse1], [[o2]], [lse2])
    assert abs(o[0, 0] - pr["o_new"]) <= rnd["o_new"]
    assert abs(math.exp(lse[0] - pr["m_new"]) - pr["l_new"]) <= rnd["l_new"]


@pytest.mark.parametrize("split", [1, 3, 6])
def test_merge_of_key_chunks_is_full_attention(split):
    """Attention over keys [0, split) and [split, n) separately (C oracle),
    merged, equals attention over all keys; merging with an empty partial
    (lse = -inf) changes nothing."""
    r = _rng(90 + split)
    n, tau = 7, 0.9
    q, k, v = r.normal(size=(5, 3)), r.normal(size=(n, 3)), r.normal(size=(n, 2))
    o1, l1 = oracle.attention_forward(q, k[:split], v[:split], False, tau)
    o2, l2 = oracle.attention_forward(q, k[split:], v[split:], False, tau)
    o, lse = oracle.merge_partials(o1, l1, o2, l2)
    of, lf = oracle.attention_forward(q, k, v, False, tau)
    assert np.max(np.abs(o - of)) < 1e-13 and np.max(np.abs(lse - lf)) < 1e-13
    oe, le = oracle.merge_partials(o, lse, np.full_like(o, 7.0), np.full(len(o), -np.inf))
    assert np.array_equal(oe, o) and np.array_equal(le, lse)
    oz, lz = oracle.merge_partials(np.ones((2, 2)), [-np.inf] * 2, np.ones((2, 2)), [-np.inf] * 2)
    assert np.all(oz == 0.0) and np.all(np.isneginf(lz))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_given_stats_sums_to_full_backward(causal):
    """Gradients of one query chunk against each key chunk, with the whole
    row's lse and D given, sum to the full backward (C oracle): dQ is the sum
    over key chunks and dK, dV of a key chunk are its rows of the full
    result.  With the chunk's own statistics it is the plain backward."""
    r = _rng(95 + int(causal))
    n, nc, tau = 8, 4, 0.7
    q, k = r.normal(size=(n, 3)), r.normal(size=(n, 3))
    v, dO = r.normal(size=(n, 2)), r.normal(size=(n, 2))
    dq, dk, dv, lse, D = oracle.attention_backward(q, k, v, dO, causal, tau)
    for qc in range(0, n, nc):
        rows = slice(qc, qc + nc)
        dq_sum = np.zeros((nc, 3))
        for kc in range(0, n, nc):
            if causal and kc > qc:
                continue
            cols = slice(kc, kc + nc)
            gq, _, _ = oracle.attention_backward_given_stats(
                q[rows], k[cols], v[cols], dO[rows], lse[rows], D[rows], causal, tau,
                q_offset=qc - kc)
            dq_sum += gq
            # all query rows against this key chunk give its rows of dK, dV
            full_k = oracle.attention_backward_given_stats(q, k[cols], v[cols], dO, lse, D,
                                                           causal, tau, q_offset=-kc)
            assert np.max(np.abs(full_k[1] - dk[cols])) < 1e-12
            assert np.max(np.abs(full_k[2] - dv[cols])) < 1e-12
        assert np.max(np.abs(dq_sum - dq[rows])) < 1e-12
    own = oracle.attention_backward_given_stats(q, k, v, dO, lse, D, causal, tau)
    for a, b in zip(own, (dq, dk, dv)):
        assert np.max(np.abs(a - b)) < 1e-12


# --------------------------------------------------------------------------
# Dropout: the generator, the mask layout and dropout attention
# --------------------------------------------------------------------------

def test_philox_known_answers():
    g = _golden("philox4x32_10_kat.json")
    for vec in g["vectors"]:
        ctr = np.array([int(x, 16) for x in vec["counter"]], dtype=np.uint64)
        key = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint64)
        out = oracle.philox4x32_10(ctr, key)
        assert [int(x) for x in out] == [int(x, 16) for x in vec["output"]]


def test_dropout_mask_layout_and_rate():
    """Element (i, j) is byte j % 4 of word i % 4 of the call with counter
    (j // 4, i // 4, bh, offset); the keep rate matches t / 256; other
    offsets, heads and seeds give other masks."""
    p, seed, off = 0.3, 0x1234_5678_9ABC, 7
    keep = oracle.dropout_keep(5, 64, 96, p, seed, off)
    t = oracle.dropout_threshold(p)
    assert t == 179
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint64)
    # element by element, one generator call each, over a 16 x 12 corner
    # and the far corner (a swapped word / byte index fails both)
    for (i0, j0) in ((0, 0), (48, 84)):
        for i in range(i0, i0 + 16):
            for j in range(j0, j0 + 12):
                w = oracle.philox4x32_10(np.array([j // 4, i // 4, 5, off], dtype=np.uint64), key)
                byte = (int(w[i % 4]) >> (8 * (j % 4))) & 0xFF
                assert keep[i, j] == (byte < t), (i, j)
    big = oracle.dropout_keep(1, 512, 512, p, seed, off)
    n = big.size
    rate = big.mean()
    assert abs(rate - t / 256) < 5 * np.sqrt(t / 256 * (1 - t / 256) / n)
    for other in (oracle.dropout_keep(2, 512, 512, p, seed, off),
                  oracle.dropout_keep(1, 512, 512, p, seed, off + 1),
                  oracle.dropout_keep(1, 512, 512, p, seed + 1, off)):
        agree = (other == big).mean()
        expect = rate * rate + (1 - rate) * (1 - rate)
        assert abs(agree - expect) < 0.01
    assert oracle.dropout_threshold(0.0) == 256 and oracle.dropout_keep(0, 9, 9, 0.0, 1, 2).all()
    assert oracle.dropout_threshold(0.999) == 1


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_zero_is_plain_attention(causal):
    r = _rng(100 + int(causal))
    q, k, v, dO = (r.normal(size=(9, 3)) for _ in range(4))
    keep = np.ones((9, 9), bool)
    o, lse = oracle.attention_forward_dropout(q, k, v, causal, 0.7, keep, 0.0)
    o2, lse2 = oracle.attention_forward(q, k, v, causal, 0.7)
    assert np.max(np.abs(o - o2)) < 1e-13 and np.max(np.abs(lse - lse2)) < 1e-13
    got = oracle.attention_backward_dropout(q, k, v, dO, causal, 0.7, keep, 0.0)
    want = oracle.attention_backward(q, k, v, dO, causal, 0.7)[:3]
    for a, b in zip(got, want):
        assert np.max(np.abs(a - b)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_backward_matches_finite_differences(causal):
    """With the keep mask held fixed, central differences of L = sum(dO * O);
    p = 0.3 (scale 256 / 179), d != dv, and the kept set is a real mask."""
    r = _rng(110 + int(causal))
    n, tau, p = 7, 0.7, 0.3
    q, k = r.normal(size=(n, 3)), r.normal(size=(n, 3))
    v, dO = r.normal(size=(n, 2)), r.normal(size=(n, 2))
    keep = oracle.dropout_keep(3, n, n, p, 99, 1)
    assert 0 < keep.sum() < keep.size

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward_dropout(qq, kk, vv, causal, tau, keep, p)
        return float(np.sum(o * dO))

    dq, dk, dv = oracle.attention_backward_dropout(q, k, v, dO, causal, tau, keep, p)
    for got, want in ((dq, _fd_grad(q, lambda x: loss(x, k, v))),
                      (dk, _fd_grad(k, lambda x: loss(q, x, v))),
                      (dv, _fd_grad(v, lambda x: loss(q, k, x)))):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6


def _dropout_mask_average(p, n, d, masks, causal, seed_base):
    """Per-mask outputs of the dropout functions over `masks` generator seeds
    (same inputs), with the undropped results: returns (samples, plain),
    samples[name] of shape [masks, ...]."""
    r = _rng(140 + int(causal))
    tau = 0.5
    q, k = r.normal(size=(n, d)), r.normal(size=(n, d))
    v, dO = r.normal(size=(n, d)), r.normal(size=(n, d))
    ones = np.ones((n, 1))
    samples = {"O": [], "O1": [], "dQ": [], "dK": [], "dV": [], "dV1": []}
    for m in range(masks):
        keep = oracle.dropout_keep(m % 7, n, n, p, seed_base + m, 3)
        samples["O"].append(oracle.attention_forward_dropout(q, k, v, causal, tau, keep, p)[0])
        samples["O1"].append(oracle.attention_forward_dropout(q, k, ones, causal, tau, keep, p)[0])
        dq, dk, dv = oracle.attention_backward_dropout(q, k, v, dO, causal, tau, keep, p)
        samples["dQ"].append(dq)
        samples["dK"].append(dk)
        samples["dV"].append(dv)
        samples["dV1"].append(oracle.attention_backward_dropout(q, k, ones, ones, causal, tau, keep, p)[2])
    samples = {kk: np.stack(vv) for kk, vv in samples.items()}
    o, _ = oracle.attention_forward(q, k, v, causal, tau)
    dq, dk, dv, _, _ = oracle.attention_backward(q, k, v, dO, causal, tau)
    dv1 = oracle.attention_backward(q, k, ones, ones, causal, tau)[2]
    return samples, {"O": o, "O1": np.ones((n, 1)), "dQ": dq, "dK": dk, "dV": dv, "dV1": dv1}


@pytest.mark.parametrize("p,causal,masks", [(0.99, False, 480), (0.3, True, 240)])
def test_dropout_is_unbiased_over_masks(p, causal, masks):
    """Dropout leaves the output and the gradients unbiased: over the masks
    the generator draws (distinct seeds), O, dQ, dK and dV average to those
    of attention without dropout (O1 and dV1 are O and dV for V = 1 and
    dO = 1: the row and column sums of the kept weights, the outputs with the
    least sampling noise).  Each is projected on its undropped value,
    s = <x, ref> / <ref, ref> per mask, and the mean of s must be 1 within six
    standard errors (for p = 0.3 also element by element, which the rare
    kept entries at p = 0.99 make too heavy-tailed for).  This fixes the
    weight of the kept entries, 256 / t for a keep probability of t / 256 (t
    the byte threshold), in the forward and in the backward: at p = 0.99,
    t = 3 and 256 / t = 85.3, while the unquantised 1 / (1 - p) = 100 would
    bias every output by 17% and no weight at all by a factor of 3 / 256;
    both are shown to fall outside the bound on O1 (the forward's weight) and
    dV1 (the backward's).  The finite-difference test above then ties dQ and
    dK to the same weights."""
    t = oracle.dropout_threshold(p)
    samples, plain = _dropout_mask_average(p, 96, 8, masks, causal, seed_base=1000)
    for name, x in samples.items():
        ref = plain[name]
        s = np.tensordot(x, ref, axes=ref.ndim) / np.sum(ref * ref)
        mean, se = s.mean(), s.std(ddof=1) / np.sqrt(masks)
        assert abs(mean - 1.0) < 6 * se, (name, mean, se)
        if p > 0.9 and name in ("O1", "dV1"):
            for wrong in (1.0 / (1.0 - p), 1.0):
                ratio = wrong / (256.0 / t)
                assert abs(mean * ratio - 1.0) > 6 * se * ratio, (name, wrong)
        if p < 0.9:
            z = np.abs(x.mean(axis=0) - ref) / np.maximum(x.std(axis=0, ddof=1) / np.sqrt(masks), 1e-12)
            assert z.max() < 6.0, (name, float(z.max()))


# --------------------------------------------------------------------------
# Queries and keys of different lengths (shifted causal mask)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("nq,nk", [(3, 8), (8, 8), (8, 5)])
def test_offset_causal_rows_are_prefix_attention(nq, nk):
    """Bottom-right alignment (offset = nk - nq): query i attends to keys
    [0, i + nk - nq] exactly, each row equal to the C oracle over that key
    prefix; rows with no key (nq > nk) are O = 0, lse = -inf.  With
    offset = 0 and nq = nk it is the top-left causal mask."""
    r = _rng(120 + nq + nk)
    q, k, v = r.normal(size=(nq, 3)), r.normal(size=(nk, 3)), r.normal(size=(nk, 2))
    off = nk - nq
    o, lse = oracle.attention_forward_offset(q, k, v, True, 0.8, off)
    for i in range(nq):
        last = i + off
        if last < 0:
            assert np.all(o[i] == 0.0) and lse[i] == -np.inf
            continue
        oi, li = oracle.attention_forward(q[i:i + 1], k[:last + 1], v[:last + 1], False, 0.8)
        assert np.max(np.abs(o[i] - oi[0])) < 1e-13 and abs(lse[i] - li[0]) < 1e-13
    if nq <= nk:   # the last query sees every key
        assert abs(lse[-1] - oracle.attention_forward(q[-1:], k, v, False, 0.8)[1][0]) < 1e-13
    if nq == nk:
        o0, l0 = oracle.attention_forward_offset(q, k, v, True, 0.8, 0)
        o1, l1 = oracle.attention_forward(q, k, v, True, 0.8)
        assert np.max(np.abs(o0 - o1)) < 1e-13 and np.max(np.abs(l0 - l1)) < 1e-13


def test_offset_backward_matches_finite_differences():
    r = _rng(130)
    nq, nk, tau = 4, 7, 0.7
    q, k = r.normal(size=(nq, 3)), r.normal(size=(nk, 3))
    v, dO = r.normal(size=(nk, 2)), r.normal(size=(nq, 2))

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward_offset(qq, kk, vv, True, tau, nk - nq)
        return float(np.sum(o * dO))

    dq, dk, dv, _, _ = oracle.attention_backward_offset(q, k, v, dO, True, tau, nk - nq)
    for got, want in ((dq, _fd_grad(q, lambda x: loss(x, k, v))),
                      (dk, _fd_grad(k, lambda x: loss(q, x, v))),
                      (dv, _fd_grad(v, lambda x: loss(q, k, x)))):
        scale = max(1.0, np.max(np.abs(want)))
        assert np.max(np.abs(got - want)) / scale < 1e-6
