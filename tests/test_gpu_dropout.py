"""GPU parity for dropout on the attention probabilities.

The training forward and the backward regenerate the same keep mask from
(seed, offset) with Philox4x32-10; the oracle builds the mask from the same
definition (its own implementation of the generator, pinned by the
generator's published known answers) and evaluates dropout attention in fp64.
O, lse, dQ, dK, dV must match within the library's tolerances; p = 0 must
reproduce the plain training path; the same (seed, offset) reproduces the
same result and another offset gives another mask.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from io_aware_exact_gb300.inputs import make_inputs
from parity import Parity, dtype_name

pytestmark = pytest.mark.gpu

SEED = 0x5EED_0000_1234


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _run(x, p, seed, offset, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse, o32 = attn.forward_dropout(q, k, v, p, seed, offset, causal, scale)
    dq, dk, dv = attn.backward_dropout(q, k, v, o32, lse, dO, p, seed, offset, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return {n: t.cpu() for n, t in dict(o=o, o32=o32, lse=lse, dq=dq, dk=dk, dv=dv).items()}


@pytest.mark.parametrize("B,H,N,d,causal,p,dtype", [
    (1, 2, 256, 64, False, 0.1, torch.bfloat16),
    (1, 2, 1000, 128, True, 0.5, torch.bfloat16),
    (2, 1, 640, 128, False, 0.3, torch.float16),
    (1, 3, 384, 64, True, 0.2, torch.bfloat16),
    (1, 1, 1, 128, True, 0.4, torch.bfloat16),      # one row
    (1, 2, 129, 64, True, 0.05, torch.float16),     # ragged tail, fp16, d = 64
    (1, 1, 300, 128, False, 3 / 512, torch.bfloat16),   # 256 (1 - p) = 254.5: ties round to even
])
def test_dropout_matches_oracle(B, H, N, d, causal, p, dtype):
    scale = d ** -0.5
    x = make_inputs(B, H, N, d, seed=800 + N + d, dtype=dtype)
    offset = 17
    out = _run(x, p, SEED, offset, causal, scale)
    pc = Parity("dropout p=%g" % p, dtype_name(dtype))
    for b in range(B):
        for h in range(H):
            bh = b * H + h
            keep = oracle.dropout_keep(bh, N, N, p, SEED, offset)
            q, k, v, dO = (_f64(x[n][b, h]) for n in ("q", "k", "v", "dO"))
            o_ref, lse_ref = oracle.attention_forward_dropout(q, k, v, causal, scale, keep, p)
            dq_ref, dk_ref, dv_ref = oracle.attention_backward_dropout(q, k, v, dO, causal, scale,
                                                                       keep, p)
            pc.add_lse(out["lse"][b, h].numpy().astype(np.float64), lse_ref)
            for n, ref in (("o", o_ref), ("o32", o_ref), ("dq", dq_ref), ("dk", dk_ref),
                           ("dv", dv_ref)):
                pc.add(n, _f64(out[n][b, h]), ref, "f32" if n == "o32" else None)
    pc.check()


def test_dropout_zero_is_the_plain_training_path():
    B, H, N, d = 1, 2, 700, 128
    x = make_inputs(B, H, N, d, seed=811)
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    out = _run(x, 0.0, SEED, 3, True, d ** -0.5)
    o, lse, o32 = attn.forward(q, k, v, True, d ** -0.5, o32=True)
    dq, dk, dv = attn.backward(q, k, v, None, lse, dO, True, d ** -0.5, o32=o32)
    torch.cuda.synchronize()
    assert torch.equal(out["o"], o.cpu()) and torch.equal(out["lse"], lse.cpu())
    assert torch.equal(out["dk"], dk.cpu()) and torch.equal(out["dv"], dv.cpu())


def test_same_seed_reproduces_and_other_offset_differs():
    B, H, N, d = 1, 2, 512, 64
    x = make_inputs(B, H, N, d, seed=812)
    a = _run(x, 0.25, SEED, 5, False, d ** -0.5)
    b = _run(x, 0.25, SEED, 5, False, d ** -0.5)
    c = _run(x, 0.25, SEED, 6, False, d ** -0.5)
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["dk"], b["dk"]) and torch.equal(a["dv"], b["dv"])
    assert not torch.equal(a["o"], c["o"])
    assert torch.equal(a["lse"], c["lse"])      # lse is that of the undropped softmax
