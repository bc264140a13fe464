"""GPU parity for grouped K / V heads (GQA; MQA when Hkv = 1).

Query heads h share K / V head h / (H / Hkv).  The CUDA library (through the
C ABI, via the torch binding) is compared with the fp64 oracle's grouped
functions on the same bf16 values: O and lse of every query head, dQ of every
query head, and dK, dV of every K / V head (summed over its group), for the
training path (fp32 O, D = rowsum(dO o O)) and the exact-D path.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from io_aware_exact_gb300.inputs import make_inputs
from parity import Parity, check_tensor, dtype_name

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _grouped_inputs(B, H, Hkv, N, d, seed, dtype=torch.bfloat16):
    xq = make_inputs(B, H, N, d, seed, dtype=dtype)
    xkv = make_inputs(B, Hkv, N, d, seed + 1000, dtype=dtype)
    return {"q": xq["q"], "dO": xq["dO"], "k": xkv["k"], "v": xkv["v"]}


def _run(x, causal, scale, path, splits=None):
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    if path == "train":
        o, lse, o32 = attn.forward(q, k, v, causal, scale, o32=True)
        assert torch.equal(o32.to(o.dtype), o)
    else:
        o, lse = attn.forward(q, k, v, causal, scale)
        o32 = None
    dq, dk, dv = attn.backward(q, k, v, o, lse, dO, causal, scale, o32=o32, splits=splits)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def _compare(x, out, causal, scale):
    B = x["q"].shape[0]
    pc = Parity("grouped", dtype_name(x["q"]))
    for b in range(B):
        q, k, v, dO = (_f64(x[n][b]) for n in ("q", "k", "v", "dO"))
        o_ref, lse_ref = oracle.attention_forward_grouped(q, k, v, causal, scale)
        dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward_grouped(q, k, v, dO, causal, scale)
        for h in range(q.shape[0]):
            pc.add("O", _f64(out["o"][b, h]), o_ref[h])
            pc.add_lse(out["lse"][b, h].numpy().astype(np.float64), lse_ref[h])
            pc.add("dQ", _f64(out["dq"][b, h]), dq_ref[h])
        for g in range(k.shape[0]):
            pc.add("dK", _f64(out["dk"][b, g]), dk_ref[g])
            pc.add("dV", _f64(out["dv"][b, g]), dv_ref[g])
    pc.check()


CASES = [
    # (B, H, Hkv, N, d, causal)
    (1, 4, 2, 256, 128, True),
    (1, 4, 1, 300, 128, False),
    (2, 6, 3, 129, 64, True),
    (1, 8, 1, 640, 64, True),
    (1, 2, 1, 1, 128, True),
    (2, 4, 2, 1000, 128, False),
]


@pytest.mark.parametrize("path", ["train", "exact"])
@pytest.mark.parametrize("B,H,Hkv,N,d,causal", CASES)
def test_grouped_heads(B, H, Hkv, N, d, causal, path):
    x = _grouped_inputs(B, H, Hkv, N, d, seed=21 + N + H + Hkv)
    out = _run(x, causal, d ** -0.5, path)
    _compare(x, out, causal, d ** -0.5)


def test_grouped_heads_fp16():
    x = _grouped_inputs(1, 4, 2, 384, 128, seed=77, dtype=torch.float16)
    out = _run(x, True, 128 ** -0.5, "train")
    _compare(x, out, True, 128 ** -0.5)


def test_grouped_equals_repeated_kv():
    """GQA gives the same forward as plain multi-head attention with each K / V
    head repeated for its group (both through the CUDA library), and its dK, dV
    are the group sums of that multi-head result (to rounding)."""
    B, H, Hkv, N, d = 1, 4, 2, 512, 128
    x = _grouped_inputs(B, H, Hkv, N, d, seed=5)
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    kr, vr = (t.repeat_interleave(H // Hkv, dim=1).contiguous() for t in (k, v))
    o_g, lse_g = attn.forward(q, k, v, True)
    o_r, lse_r = attn.forward(q, kr, vr, True)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_r) and torch.equal(lse_g, lse_r)
    _, dk_g, dv_g = attn.backward(q, k, v, o_g, lse_g, dO, True)
    _, dk_r, dv_r = attn.backward(q, kr, vr, o_r, lse_r, dO, True)
    torch.cuda.synchronize()
    for got, rep in ((dk_g, dk_r), (dv_g, dv_r)):
        want = rep.float().reshape(B, Hkv, H // Hkv, N, d).sum(2)
        check_tensor("group sum", _f64(got[0]).reshape(-1, d), want[0].double().cpu().numpy().reshape(-1, d))


def test_grouped_argument_errors():
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 3, 128, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        attn.forward(q, k, k, True)
    # the C entry point itself rejects H not a multiple of Hkv
    o = torch.empty_like(q)
    lse = torch.empty(1, 3, 128, dtype=torch.float32, device=dev)
    rc = attn.lib().attn_fwd_gqa(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 1, 3, 2, 128, 64, 1, 0.125, None)
    assert rc == 1


@pytest.mark.parametrize("splits", [1, 2, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_group_split_over_ctas(splits, causal):
    """The group's query heads split over 1, 2 or 4 CTAs (fp32 shares of dK,
    dV summed at the end) give the oracle's gradients; the shares are summed
    in a fixed order, so dK, dV repeat bit for bit."""
    x = _grouped_inputs(1, 8, 2, 640, 128, seed=77)
    scale = 128 ** -0.5
    out = _run(x, causal, scale, "train", splits=splits)
    _compare(x, out, causal, scale)
    again = _run(x, causal, scale, "train", splits=splits)
    assert torch.equal(out["dk"], again["dk"]) and torch.equal(out["dv"], again["dv"])


def test_group_split_fp16_d64():
    x = _grouped_inputs(2, 6, 2, 257, 64, seed=78, dtype=torch.float16)
    out = _run(x, True, 64 ** -0.5, "train", splits=3)
    _compare(x, out, True, 64 ** -0.5)


def test_group_split_hint():
    L = attn.lib()
    assert L.attn_gqa_split_hint(2, 16, 16, 8192, 1) == 1        # no groups
    assert L.attn_gqa_split_hint(2, 16, 2, 8192, 1) == 2         # groups of 8 on 152 SMs
    assert L.attn_gqa_split_hint(2, 16, 1, 8192, 1) == 4         # MQA
    assert L.attn_gqa_split_hint(1, 4, 2, 256, 1) == 2           # tiny: all heads apart
