"""GPU parity for packed batches whose keys have lengths of their own.

Sequence b's queries are rows cu_q[b]:cu_q[b+1] of q [total_q, H, d] and its
keys rows cu_k[b]:cu_k[b+1] of k, v [total_k, Hkv, d]; with a causal mask key
j is visible to query i iff j <= i + Lk - Lq (aligned bottom-right, so the
last query sees every key).  The CUDA library's training path (fp32 O,
D = rowsum(dO o O), backward) is compared with the oracle's
attention_*_varlen_qk functions on the same bf16 / fp16 values, every token
and head.  The cases cover query chunks shorter than their key prefix, more
queries than keys (leading rows that see no key: O = 0, lse = -inf, dQ = 0),
a sequence with keys but no queries (dK = dV = 0), one with queries but no
keys, lengths straddling the 128-row tiles, grouped K / V heads and d = 64.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from parity import Parity, TOL_LSE, dtype_name

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _inputs(lq, lk, H, Hkv, d, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    tq, tk = int(sum(lq)), int(sum(lk))
    mk = lambda n, h: torch.randn((n, h, d), generator=g).to(dtype)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return {"q": mk(tq, H), "k": mk(tk, Hkv), "v": mk(tk, Hkv), "dO": mk(tq, H)}, cu_q, cu_k


def _run(x, cu_q, cu_k, max_q, max_k, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    cq, ck = torch.from_numpy(cu_q).to(dev), torch.from_numpy(cu_k).to(dev)
    B, H = len(cu_q) - 1, q.shape[1]
    lse = torch.full((B, H, max_q), SENTINEL, dtype=torch.float32, device=dev)
    # sentinels in the gradient outputs: every row must be written
    dq = torch.full_like(q, 7.0)
    dk, dv = torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    o, lse, o32 = attn.forward_varlen(q, k, v, cq, max_q, causal, scale, lse=lse, o32=True,
                                      cu_seqlens_k=ck, max_seqlen_k=max_k)
    assert torch.equal(o32.to(o.dtype), o)
    o_plain, lse_plain = attn.forward_varlen(q, k, v, cq, max_q, causal, scale,
                                             lse=torch.full_like(lse, SENTINEL),
                                             cu_seqlens_k=ck, max_seqlen_k=max_k)
    attn.backward_varlen(q, k, v, o32, lse, dO, cq, max_q, causal, scale, dq=dq, dk=dk, dv=dv,
                         cu_seqlens_k=ck, max_seqlen_k=max_k)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, o_plain=o_plain, lse_plain=lse_plain,
                                        dq=dq, dk=dk, dv=dv).items()}


def _compare(x, cu_q, cu_k, max_q, out, causal, scale):
    q, k, v, dO = (_f64(x[n]) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = oracle.attention_forward_varlen_qk(q, k, v, cu_q, cu_k, max_q, causal, scale)
    dq_ref, dk_ref, dv_ref = oracle.attention_backward_varlen_qk(q, k, v, dO, cu_q, cu_k, causal,
                                                                 scale)
    pc = Parity("varlen qk", dtype_name(x["q"]))
    H, Hkv = q.shape[1], k.shape[1]
    for name in ("lse", "lse_plain"):
        lse = out[name].numpy().astype(np.float64)
        for b in range(len(cu_q) - 1):
            n = int(cu_q[b + 1] - cu_q[b])
            assert np.all(lse[b, :, n:] == SENTINEL), "lse past the sequence was written"
            got, want = lse[b, :, :n], lse_ref[b, :, :n]
            # rows that see no key: exactly -inf
            assert np.array_equal(np.isneginf(got), np.isneginf(want)), (name, b)
            fin = np.isfinite(want)
            if fin.any():
                assert np.max(np.abs(got[fin] - want[fin])) <= TOL_LSE, (name, b)
    for h in range(H):
        pc.add("O", _f64(out["o"][:, h]), o_ref[:, h])
        pc.add("O plain", _f64(out["o_plain"][:, h]), o_ref[:, h])
        pc.add("dQ", _f64(out["dq"][:, h]), dq_ref[:, h])
    for g in range(Hkv):
        pc.add("dK", _f64(out["dk"][:, g]), dk_ref[:, g])
        pc.add("dV", _f64(out["dv"][:, g]), dv_ref[:, g])
    pc.check()
    # rows that see no key (lse = -inf) and keys of sequences without queries
    # are exactly 0
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = (int(c) for c in (cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]))
        empty = np.isneginf(lse_ref[b, :, :q1 - q0]).T          # [rows, H]
        for name in ("o", "dq"):
            assert np.all(_f64(out[name][q0:q1])[empty] == 0.0), (name, b)
        if q1 == q0:
            for name in ("dk", "dv"):
                assert np.all(_f64(out[name][k0:k1]) == 0.0), (name, b)


CASES = [
    # (query lengths, key lengths, H, Hkv, d, causal)
    ([5, 300, 129], [300, 130, 1000], 2, 2, 128, True),
    ([5, 300, 129], [300, 130, 1000], 2, 1, 128, False),
    ([0, 200, 257, 64], [200, 0, 3, 64], 2, 2, 64, True),    # keys, no queries / queries, no keys
    ([1, 640, 384], [1000, 256, 385], 4, 2, 64, True),
    ([700, 130], [130, 700], 2, 1, 128, True),
]


@pytest.mark.parametrize("lq,lk,H,Hkv,d,causal", CASES)
def test_varlen_qk(lq, lk, H, Hkv, d, causal):
    x, cu_q, cu_k = _inputs(lq, lk, H, Hkv, d, seed=41 + sum(lq) + 3 * sum(lk) + H)
    max_q, max_k = max(max(lq), 1), max(max(lk), 1)
    out = _run(x, cu_q, cu_k, max_q, max_k, causal, d ** -0.5)
    _compare(x, cu_q, cu_k, max_q, out, causal, d ** -0.5)


def test_varlen_qk_fp16_and_loose_maxima():
    """fp16, and maxima above every length (the extra CTAs exit at once)."""
    lq, lk = [300, 77], [128, 500]
    x, cu_q, cu_k = _inputs(lq, lk, 2, 2, 128, seed=44, dtype=torch.float16)
    out = _run(x, cu_q, cu_k, 700, 900, True, 128 ** -0.5)
    _compare(x, cu_q, cu_k, 700, out, True, 128 ** -0.5)


def test_varlen_qk_equal_lengths_match_packed_bits():
    """With cu_seqlens_k = cu_seqlens the results are the bits of the packed
    entry points of one cu_seqlens (bottom-right and top-left coincide)."""
    lengths = [300, 129, 1]
    x, cu, _ = _inputs(lengths, lengths, 2, 1, 128, seed=45)
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    c = torch.from_numpy(cu).to(dev)
    lse_a = torch.full((3, 2, 300), SENTINEL, dtype=torch.float32, device=dev)
    lse_b = torch.full_like(lse_a, SENTINEL)      # (entries past each length stay untouched)
    a = attn.forward_varlen(q, k, v, c, 300, True, lse=lse_a, o32=True, cu_seqlens_k=c,
                            max_seqlen_k=300)
    b = attn.forward_varlen(q, k, v, c, 300, True, lse=lse_b, o32=True)
    for ta, tb in zip(a, b):
        assert torch.equal(ta, tb)
    ga = attn.backward_varlen(q, k, v, a[2], a[1], dO, c, 300, True, cu_seqlens_k=c, max_seqlen_k=300)
    gb = attn.backward_varlen(q, k, v, b[2], b[1], dO, c, 300, True)
    torch.cuda.synchronize()
    assert torch.equal(ga[1], gb[1]) and torch.equal(ga[2], gb[2])
