"""GPU parity for packed variable-length batches.

Sequence b is tokens cu_seqlens[b]:cu_seqlens[b+1] of q, k, v ([total, heads,
d], heads interleaved per token); each attends only to itself.  The CUDA
library (training path: fp32 O, D = rowsum(dO o O)) is compared with the
oracle's packed functions on the same bf16 values: O, lse, dQ, dK, dV of
every token and head.  Lengths straddle the 128-row tiles (a sequence's last,
partial tile is stored row by row, not with a TMA box that would run into the
next sequence), include empty sequences, and K / V heads may be grouped.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from parity import Parity, check_tensor, dtype_name

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _inputs(lengths, H, Hkv, d, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    total = int(sum(lengths))
    mk = lambda h: torch.randn((total, h, d), generator=g).to(dtype)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return {"q": mk(H), "k": mk(Hkv), "v": mk(Hkv), "dO": mk(H)}, cu


def _run(x, cu, max_s, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    cu_d = torch.from_numpy(cu).to(dev)
    B, H = len(cu) - 1, q.shape[1]
    lse = torch.full((B, H, max_s), SENTINEL, dtype=torch.float32, device=dev)
    o, lse, o32 = attn.forward_varlen(q, k, v, cu_d, max_s, causal, scale, lse=lse, o32=True)
    assert torch.equal(o32.to(o.dtype), o)
    dq, dk, dv = attn.backward_varlen(q, k, v, o32, lse, dO, cu_d, max_s, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def _compare(x, cu, max_s, out, causal, scale):
    q, k, v, dO = (_f64(x[n]) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = oracle.attention_forward_varlen(q, k, v, cu, max_s, causal, scale)
    dq_ref, dk_ref, dv_ref = oracle.attention_backward_varlen(q, k, v, dO, cu, causal, scale)
    lse = out["lse"].numpy().astype(np.float64)
    pc = Parity("varlen", dtype_name(x["q"]))
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        assert np.all(lse[b, :, s1 - s0:] == SENTINEL), "lse past the sequence was written"
        if s1 == s0:
            continue
        for h in range(q.shape[1]):
            pc.add("O", _f64(out["o"][s0:s1, h]), o_ref[s0:s1, h])
            pc.add_lse(lse[b, h, :s1 - s0], lse_ref[b, h, :s1 - s0])
            pc.add("dQ", _f64(out["dq"][s0:s1, h]), dq_ref[s0:s1, h])
        for g in range(k.shape[1]):
            pc.add("dK", _f64(out["dk"][s0:s1, g]), dk_ref[s0:s1, g])
            pc.add("dV", _f64(out["dv"][s0:s1, g]), dv_ref[s0:s1, g])
    pc.check()


CASES = [
    # (lengths, H, Hkv, d, causal)
    ([1, 127, 128, 129, 300], 2, 2, 128, True),
    ([1, 127, 128, 129, 300], 2, 1, 128, False),
    ([0, 257, 5, 0], 2, 2, 64, True),
    ([513, 64], 4, 2, 64, False),
    ([1000, 3000, 65], 2, 1, 128, True),
]


@pytest.mark.parametrize("lengths,H,Hkv,d,causal", CASES)
def test_varlen(lengths, H, Hkv, d, causal):
    x, cu = _inputs(lengths, H, Hkv, d, seed=31 + sum(lengths) + H)
    max_s = max(max(lengths), 1)
    out = _run(x, cu, max_s, causal, d ** -0.5)
    _compare(x, cu, max_s, out, causal, d ** -0.5)


def test_varlen_max_seqlen_above_every_length():
    """A max_seqlen larger than needed only adds CTAs that exit at once."""
    lengths = [200, 90]
    x, cu = _inputs(lengths, 2, 2, 128, seed=8)
    out = _run(x, cu, 1000, True, 128 ** -0.5)
    _compare(x, cu, 1000, out, True, 128 ** -0.5)


def test_varlen_fp16():
    lengths = [300, 129]
    x, cu = _inputs(lengths, 2, 1, 128, seed=9, dtype=torch.float16)
    out = _run(x, cu, 300, True, 128 ** -0.5)
    _compare(x, cu, 300, out, True, 128 ** -0.5)


def test_one_sequence_equals_dense_layout():
    """One packed sequence gives the bits of the dense [1, H, N, d] call."""
    N, H, d = 700, 2, 128
    x, cu = _inputs([N], H, H, d, seed=10)
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    cu_d = torch.from_numpy(cu).to(dev)
    o, lse, o32 = attn.forward_varlen(q, k, v, cu_d, N, True, o32=True)
    dense = lambda t: t.transpose(0, 1).unsqueeze(0).contiguous()
    od, lsed, o32d = attn.forward(dense(q), dense(k), dense(v), True, o32=True)
    torch.cuda.synchronize()
    assert torch.equal(dense(o), od) and torch.equal(lse, lsed)
    dq, dk, dv = attn.backward_varlen(q, k, v, o32, lse, dO, cu_d, N, True)
    dqd, dkd, dvd = attn.backward(dense(q), dense(k), dense(v), od, lsed, dense(dO), True, o32=o32d)
    torch.cuda.synchronize()
    assert torch.equal(dense(dk), dkd) and torch.equal(dense(dv), dvd)
    check_tensor("dQ", _f64(dense(dq)[0]).reshape(-1, d), _f64(dqd[0]).reshape(-1, d))
