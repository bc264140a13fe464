"""GPU parity for ring attention emulated on one device, and for the kernels
that combine partial results.

io_aware_exact_gb300.ring runs the ring schedule of R ranks in one process
(run_local): each rank's query chunk is attended to every key / value chunk
with the library's kernels, partial results are merged with attn_merge, and
the backward kernel adds each pair's share of dK, dV into fp32 sums
(attn_bwd_acc) that travel with the chunk.  The gathered result must match the oracle's attention over the whole
sequence within the library's tolerances.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from io_aware_exact_gb300 import ring
from io_aware_exact_gb300.inputs import make_inputs
from parity import Parity, check_lse, check_tensor, dtype_name

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("R,N,d,causal,dtype", [
    (2, 1024, 128, True, torch.bfloat16),
    (4, 1024, 128, True, torch.bfloat16),
    (4, 1024, 128, False, torch.bfloat16),
    (3, 768, 64, True, torch.float16),
])
def test_ring_equals_whole_sequence(R, N, d, causal, dtype):
    B, H = 1, 2
    scale = d ** -0.5
    x = make_inputs(B, H, N, d, seed=700 + R + d, dtype=dtype)
    dev = torch.device("cuda:0")
    chunks = {n: [c.contiguous() for c in torch.chunk(t.to(dev), R, dim=2)] for n, t in x.items()}
    o, lse, o32 = ring.ring_forward(chunks["q"], chunks["k"], chunks["v"], causal, scale)
    dq, dk, dv = ring.ring_backward(chunks["q"], chunks["k"], chunks["v"], o32, lse, chunks["dO"],
                                    causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    got = {n: torch.cat(t, dim=2) for n, t in
           (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    pc = Parity("ring R=%d" % R, dtype_name(dtype))
    for h in range(H):
        q, k, v, dO = (_f64(x[n][0, h]) for n in ("q", "k", "v", "dO"))
        o_ref, lse_ref = oracle.attention_forward(q, k, v, causal, scale)
        dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward(q, k, v, dO, causal, scale)
        pc.add_lse(got["lse"][0, h].cpu().numpy().astype(np.float64), lse_ref)
        for n, ref in (("o", o_ref), ("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
            pc.add(n, _f64(got[n][0, h]), ref)
    pc.check()


@pytest.mark.parametrize("causal", [True, False])
def test_ring_with_grouped_heads(causal):
    """Grouped K / V heads (8 query heads, 2 K / V heads) through the CUDA ring:
    the forward takes the grouped path, attn_bwd_acc sums each group's dK, dV
    into the travelling fp32 sums."""
    B, H, Hkv, N, d, R = 1, 8, 2, 768, 128, 3
    scale = d ** -0.5
    xq = make_inputs(B, H, N, d, seed=720)
    xkv = make_inputs(B, Hkv, N, d, seed=721)
    x = {"q": xq["q"], "dO": xq["dO"], "k": xkv["k"], "v": xkv["v"]}
    dev = torch.device("cuda:0")
    ch = {n: [c.contiguous() for c in torch.chunk(t.to(dev), R, dim=2)] for n, t in x.items()}
    o, lse, o32 = ring.ring_forward(ch["q"], ch["k"], ch["v"], causal, scale)
    dq, dk, dv = ring.ring_backward(ch["q"], ch["k"], ch["v"], o32, lse, ch["dO"], causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    got = {n: torch.cat(t, dim=2)[0] for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    q, k, v, dO = (_f64(x[n][0]) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = oracle.attention_forward_grouped(q, k, v, causal, scale)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward_grouped(q, k, v, dO, causal, scale)
    check_lse(torch.cat(lse, dim=2)[0].cpu().numpy().astype(np.float64).reshape(-1),
              lse_ref.reshape(-1))
    for n, ref in (("o", o_ref), ("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
        check_tensor(n, _f64(got[n]).reshape(-1, d), ref.reshape(-1, d))


def test_merge_kernel_matches_oracle_and_handles_empty_partials():
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(5)
    rows, d = 1000, 128
    o1, o2 = (torch.randn((rows, d), generator=g) for _ in range(2))
    l1, l2 = (torch.randn((rows,), generator=g) * 5 for _ in range(2))
    l1[:10] = -float("inf")              # empty running state: take the partial
    l2[10:20] = -float("inf")            # empty partial: keep the running state
    l1[20:30] = -float("inf")
    l2[20:30] = -float("inf")            # both empty: O = 0, lse = -inf
    want_o, want_l = oracle.merge_partials(o1.numpy(), l1.numpy(), o2.numpy(), l2.numpy())
    acc_o, acc_l = o1.to(dev), l1.to(dev)
    out16 = torch.empty((rows, d), dtype=torch.bfloat16, device=dev)
    attn.merge(acc_o, acc_l, o2.to(dev), l2.to(dev), o_out=out16)
    torch.cuda.synchronize()
    got_o, got_l = acc_o.cpu().numpy().astype(np.float64), acc_l.cpu().numpy().astype(np.float64)
    fin = np.isfinite(want_l)
    assert np.array_equal(np.isneginf(got_l), ~fin)
    assert np.max(np.abs(got_l[fin] - want_l[fin])) < 1e-5
    assert np.max(np.abs(got_o - want_o)) < 1e-5
    assert np.all(got_o[20:30] == 0.0)
    assert torch.equal(acc_o[10:20], o1[10:20].to(dev))
    assert torch.equal(out16, acc_o.to(torch.bfloat16))


def test_convert():
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(6)
    x = torch.randn((4096,), generator=g).to(dev)
    y = attn.convert(x, torch.bfloat16, 0.5)
    assert torch.equal(y, (0.5 * x).to(torch.bfloat16))
    yh = attn.convert(x, torch.float16, 2.0)
    assert torch.equal(yh, (2.0 * x).to(torch.float16))


def test_backward_into_fp32_sums():
    """attn_bwd_acc writes fp32 dK, dV equal (within rounding) to attn_bwd's,
    and with accumulate adds to them; dQ is the same as attn_bwd's."""
    B, H, N, d = 1, 4, 640, 128
    dev = torch.device("cuda:0")
    x = {n: t.to(dev) for n, t in make_inputs(B, H, N, d, seed=710).items()}
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    scale = d ** -0.5
    o, lse, o32 = attn.forward(q, k, v, True, scale, o32=True)
    dq, dk, dv = attn.backward(q, k, v, None, lse, dO, True, scale, o32=o32)
    D = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dk32 = torch.full((B, H, N, d), 3.0, dtype=torch.float32, device=dev)
    dv32 = torch.full((B, H, N, d), 3.0, dtype=torch.float32, device=dev)
    dq2 = torch.empty_like(q)
    s = torch.cuda.current_stream().cuda_stream
    attn.attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), acc.data_ptr(),
                                 B, H, N, d, s)
    attn.attn_bwd_acc(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                      D.data_ptr(), acc.data_ptr(), dq2.data_ptr(), dk32.data_ptr(),
                      dv32.data_ptr(), False, B, H, H, N, d, True, scale, s)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert torch.equal(dk32.to(torch.bfloat16), dk) and torch.equal(dv32.to(torch.bfloat16), dv)
    check_tensor("dq", _f64(dq2).reshape(-1, d), _f64(dq).reshape(-1, d))
    first_k, first_v = dk32.clone(), dv32.clone()
    attn.attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), acc.data_ptr(),
                                 B, H, N, d, s)
    attn.attn_bwd_acc(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                      D.data_ptr(), acc.data_ptr(), dq2.data_ptr(), dk32.data_ptr(),
                      dv32.data_ptr(), True, B, H, H, N, d, True, scale, s)
    torch.cuda.synchronize()
    assert torch.equal(dk32, 2 * first_k) and torch.equal(dv32, 2 * first_v)
