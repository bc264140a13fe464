"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Every case draws seeded bf16 inputs, runs the library on the GPU over the
whole [B, H, N, d] problem (the same launch the benchmark times), and compares
O, lse, dQ, dK, dV with the oracle on the same bf16 values: every head for the
small shapes, sampled heads (and for N = 32768 sampled rows / key columns) for
the large workloads.  Tolerances are those of ``tests/parity.py``.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from io_aware_exact_gb300.inputs import WORKLOADS, make_inputs
from parity import Parity, check_tensor, dtype_name, sample_rows

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _run_gpu(x, causal, scale, backward, f16=False, path="train"):
    """path "train": attn_fwd_train + attn_bwd_preprocess_o32 + attn_bwd (the
    training path bench.py times); path "exact": attn_fwd +
    attn_bwd_preprocess (D from recomputed P and dP) + attn_bwd."""
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    if path == "train":
        o, lse, o32 = attn.forward(q, k, v, causal, scale, o32=True)
    else:
        o, lse = attn.forward(q, k, v, causal, scale)
        o32 = None
    out = {"o": o, "lse": lse}
    if o32 is not None:
        # the 16-bit O is the rounding of the fp32 O
        assert torch.equal(o32.to(o.dtype), o)
    if backward:
        dO = x["dO"].to(dev)
        dq, dk, dv = attn.backward(q, k, v, o, lse, dO, causal, scale, o32=o32)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return {kk: vv.cpu() for kk, vv in out.items()}


def _compare_head(x, out, b, h, causal, scale, backward, pc, rows=None, cols=None):
    """Add head (b, h)'s outputs and the oracle's to the collector pc."""
    q, k, v = (_f64(x[n][b, h]) for n in ("q", "k", "v"))
    o_ref, lse_ref = oracle.attention_forward(q, k, v, causal, scale, rows=rows)
    sel = slice(None) if rows is None else rows
    pc.add("O", _f64(out["o"][b, h])[sel], o_ref)
    pc.add_lse(out["lse"][b, h].numpy().astype(np.float64)[sel], lse_ref)
    if not backward:
        return
    dO = _f64(x["dO"][b, h])
    if rows is None and cols is None:
        dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward(q, k, v, dO, causal, scale)
        pc.add("dQ", _f64(out["dq"][b, h]), dq_ref)
        pc.add("dK", _f64(out["dk"][b, h]), dk_ref)
        pc.add("dV", _f64(out["dv"][b, h]), dv_ref)
        return
    _, _, dq_ref = oracle.attention_backward_rows(q, k, v, dO, causal, scale, rows=rows)
    pc.add("dQ", _f64(out["dq"][b, h])[rows], dq_ref)
    lse_all, D_all, _ = oracle.attention_backward_rows(q, k, v, dO, causal, scale,
                                                       with_dq=False)
    dk_ref, dv_ref = oracle.attention_backward_cols(q, k, v, dO, lse_all, D_all, causal, scale,
                                                    cols=cols)
    pc.add("dK", _f64(out["dk"][b, h])[cols], dk_ref)
    pc.add("dV", _f64(out["dv"][b, h])[cols], dv_ref)


def _compare_heads(x, out, heads, causal, scale, backward, label, rows=None, cols=None):
    """Compare the listed heads; each tensor is judged over all of them at once."""
    pc = Parity(label, dtype_name(x["q"]))
    for (b, h) in heads:
        _compare_head(x, out, b, h, causal, scale, backward, pc, rows=rows, cols=cols)
    pc.check()


def _all_heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


SMALL = [
    # (B, H, N, d, causal)
    (1, 1, 128, 64, False),
    (1, 1, 128, 128, True),
    (1, 2, 256, 128, False),
    (2, 1, 384, 64, True),
    (1, 1, 1, 64, False),
    (1, 1, 1, 128, True),
    (1, 1, 5, 64, True),
    (1, 1, 127, 128, False),
    (1, 1, 129, 64, True),
    (1, 2, 200, 128, True),
    (1, 1, 1000, 64, False),
    (1, 1, 1000, 128, True),
    (2, 2, 513, 128, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_forward_small(B, H, N, d, causal):
    x = make_inputs(B, H, N, d, seed=7 + N + d, with_grad=False)
    out = _run_gpu(x, causal, d ** -0.5, backward=False)
    _compare_heads(x, out, _all_heads(B, H), causal, d ** -0.5, False, "B%d H%d N%d d%d" % (B, H, N, d))


@pytest.mark.parametrize("path", ["train", "exact"])
@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_backward_small(B, H, N, d, causal, path):
    x = make_inputs(B, H, N, d, seed=11 + N + d)
    out = _run_gpu(x, causal, d ** -0.5, backward=True, path=path)
    _compare_heads(x, out, _all_heads(B, H), causal, d ** -0.5, True, "B%d H%d N%d d%d" % (B, H, N, d))


@pytest.mark.parametrize("causal", [False, True])
def test_scale_not_inverse_sqrt_d(causal):
    """A scale other than 1/sqrt(d) must enter both S and the gradients."""
    x = make_inputs(1, 2, 300, 64, seed=5)
    out = _run_gpu(x, causal, 0.3, backward=True)
    _compare_heads(x, out, _all_heads(1, 2), causal, 0.3, True, "scale 0.3")


def test_fp16_entry_points():
    x = make_inputs(1, 2, 320, 128, seed=9, dtype=torch.float16)
    out = _run_gpu(x, True, 128 ** -0.5, backward=True)
    _compare_heads(x, out, _all_heads(1, 2), True, 128 ** -0.5, True, "fp16")


@pytest.mark.parametrize("path", ["train", "exact"])
def test_peaked_rows(path):
    """Q, K scaled by 8: softmax rows close to one-hot stress the max/rescale
    and the cancellation in dS = P (dP - D)."""
    x = make_inputs(1, 2, 1024, 128, seed=13, qk_mult=8.0)
    out = _run_gpu(x, True, 128 ** -0.5, backward=True, path=path)
    _compare_heads(x, out, _all_heads(1, 2), True, 128 ** -0.5, True, "Q, K x8")


# ---------------------------------------------------------------------------
# The five named workloads at full size (sampled outputs for the large ones)
# ---------------------------------------------------------------------------

def _heads(w, n, seed):
    rng = np.random.default_rng(seed)
    all_h = [(b, h) for b in range(w.B) for h in range(w.H)]
    picks = {all_h[0], all_h[-1]}
    while len(picks) < min(n, len(all_h)):
        picks.add(all_h[int(rng.integers(len(all_h)))])
    return sorted(picks)


@pytest.mark.parametrize("name,nheads", [
    ("fwd_b1_h2_n256_d64", 2),
    ("fwdbwd_b8_h16_n1024_d64", 8),
    ("fwdbwd_causal_b4_h32_n4096_d128", 2),
    ("fwdbwd_causal_peaked_b2_h16_n8192_d128", 2),
])
def test_workload(name, nheads):
    w = WORKLOADS[name]
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_grad=w.backward)
    out = _run_gpu(x, w.causal, w.scale, backward=w.backward)
    _compare_heads(x, out, _heads(w, nheads, w.seed), w.causal, w.scale, w.backward, name)


def test_workload_peaked_exact_preprocess():
    """The headline workload through the exact-D preprocess (no fp32 O)."""
    w = WORKLOADS["fwdbwd_causal_peaked_b2_h16_n8192_d128"]
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    out = _run_gpu(x, w.causal, w.scale, backward=True, path="exact")
    _compare_heads(x, out, _heads(w, 2, w.seed + 1), w.causal, w.scale, True, "exact D")


def test_autograd_function():
    """attention() as a torch.autograd.Function: gradients through .backward()."""
    x = make_inputs(1, 2, 300, 64, seed=17)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev).requires_grad_(True) for n in ("q", "k", "v"))
    o = attn.attention(q, k, v, True)
    o.backward(x["dO"].to(dev))
    out = {"o": o.detach().cpu(), "dq": q.grad.cpu(), "dk": k.grad.cpu(), "dv": v.grad.cpu(),
           "lse": torch.zeros(1, 2, 300)}
    pc = Parity("autograd")
    for h in range(2):
        qh, kh, vh, dOh = (_f64(x[n][0, h]) for n in ("q", "k", "v", "dO"))
        o_ref, _ = oracle.attention_forward(qh, kh, vh, True, 64 ** -0.5)
        pc.add("O", _f64(out["o"][0, h]), o_ref)
        dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward(qh, kh, vh, dOh, True, 64 ** -0.5)
        pc.add("dQ", _f64(out["dq"][0, h]), dq_ref)
        pc.add("dK", _f64(out["dk"][0, h]), dk_ref)
        pc.add("dV", _f64(out["dv"][0, h]), dv_ref)
    pc.check()


def test_workload_long_sequence():
    """N = 32768: one head, sampled query rows (O, lse, dQ) and key columns (dK, dV)."""
    w = WORKLOADS["fwdbwd_causal_b1_h8_n32768_d128"]
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    out = _run_gpu(x, w.causal, w.scale, backward=True)
    rows = sample_rows(w.N, 96, seed=1)
    cols = sample_rows(w.N, 96, seed=2)
    _compare_heads(x, out, [(0, w.H - 1)], w.causal, w.scale, True, "N=32768 sampled",
                   rows=rows, cols=cols)


def test_no_nxn_buffer_long_sequence():
    """The library allocates nothing: device free memory is unchanged by the calls
    (an N x N fp32 score matrix for one head at N = 32768 would be 4 GiB)."""
    w = WORKLOADS["fwdbwd_causal_b1_h8_n32768_d128"]
    dev = torch.device("cuda:0")
    x = {k: v.to(dev) for k, v in make_inputs(w.B, w.H, w.N, w.d, w.seed).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    D = torch.empty_like(lse)
    acc = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    attn.forward(x["q"], x["k"], x["v"], True, None, o=o, lse=lse)
    attn.backward(x["q"], x["k"], x["v"], o, lse, x["dO"], True, None, dq=dq, dk=dk, dv=dv,
                  D=D, dq_accum=acc)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert attn.attn_get_device_status() == 0
    assert abs(free0 - free1) < (64 << 20)


def test_timeout_path_reports_and_context_survives():
    """A wait that nothing completes runs out, is reported, and the GPU keeps
    working (no trap, no hang)."""
    attn.attn_selftest_timeout(2000)
    assert attn.attn_get_device_status() == 6
    assert attn.attn_get_device_status() == 0
    x = make_inputs(1, 1, 128, 64, seed=3, with_grad=False)
    out = _run_gpu(x, False, 0.125, backward=False)
    _compare_heads(x, out, [(0, 0)], False, 0.125, False, "after timeout")


def test_repeated_calls_are_stable():
    """Every launch gives the same bits for O, lse, dK and dV (none of them is
    summed across CTAs) and finite dQ: catches intermittent launch-wide
    failures, which a single parity run can miss."""
    w = WORKLOADS["fwdbwd_causal_b1_h8_n32768_d128"]
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed)
    first = None
    for _ in range(6):
        out = _run_gpu(x, True, w.scale, backward=True)
        assert torch.isfinite(out["dq"].float()).all()
        if first is None:
            first = out
            assert torch.isfinite(out["o"].float()).all() and torch.isfinite(out["lse"]).all()
        for name in ("o", "lse", "dk", "dv"):
            assert torch.equal(out[name], first[name]), name


def test_many_ctas_no_barrier_overrun():
    """4096 CTAs with 1..32 query blocks each, run repeatedly with the device
    status checked after every call.  Guards the backward's barrier protocol:
    a barrier whose producer can complete two phases before its consumer
    looks makes the consumer's parity wait run out, which shows up here as a
    timeout status in a sizeable share of calls."""
    w = WORKLOADS["fwdbwd_causal_b4_h32_n4096_d128"]
    dev = torch.device("cuda:0")
    x = {k: v.to(dev) for k, v in make_inputs(w.B, w.H, w.N, w.d, w.seed).items()}
    o, lse, o32 = attn.forward(x["q"], x["k"], x["v"], True, w.scale, o32=True)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    bufs = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]))
    for rep in range(30):
        attn.backward(x["q"], x["k"], x["v"], o, lse, x["dO"], True, w.scale, o32=o32, **bufs)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0, "call %d" % rep


def test_results_do_not_depend_on_the_clock():
    """Calls spread over more than 2^32 ns (one wrap of the low word of the
    GPU's nanosecond timer) all return the same bits as the first, for the
    forward, the training forward and the backward.  A clock value kept live
    in a kernel once leaked into the forward's softmax, so that about a
    quarter of that cycle every row came out empty (lse = -inf, O = NaN)."""
    import time
    dev = torch.device("cuda:0")
    B, H, N, d, scale = 1, 4, 1000, 128, 128 ** -0.5
    x = {k: v.to(dev) for k, v in make_inputs(B, H, N, d, seed=300).items()}

    def run():
        o, lse = attn.forward(x["q"], x["k"], x["v"], True, scale)
        o_t, lse_t, o32 = attn.forward(x["q"], x["k"], x["v"], True, scale, o32=True)
        dq, dk, dv = attn.backward(x["q"], x["k"], x["v"], o_t, lse_t, x["dO"], True, scale, o32=o32)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        return dict(o=o, lse=lse, o_t=o_t, lse_t=lse_t, dk=dk, dv=dv, dq=dq)

    first = run()
    for name, t in first.items():
        assert torch.isfinite(t.float()).all(), name
    t_end = time.monotonic() + 4.6
    calls = 0
    while time.monotonic() < t_end:
        out = run()
        calls += 1
        for name in ("o", "lse", "o_t", "lse_t", "dk", "dv"):
            assert torch.equal(out[name], first[name]), "%s differs at call %d" % (name, calls)
        assert torch.isfinite(out["dq"].float()).all(), "dq at call %d" % calls
        time.sleep(0.01)
    assert calls > 100
