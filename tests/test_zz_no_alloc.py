"""attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Callers that run inside a host framework that owns all device allocations,
or in a real-time loop that allocates nothing after start-up, cannot hand
attn_bwd its D and dQ-accumulator workspaces.
attn_bwd_noalloc keeps those in a fixed 16 MiB device array inside the
library.  These tests call it through the C ABI and check it against the
regular attn_bwd_preprocess + attn_bwd path, twice in a row (the array is
shared between calls and keeps the previous call's contents), and, for a
problem that fills the array up to its last 256 floats, against the fp64
oracle as well.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import io_aware_exact_gb300 as attn
import oracle
from io_aware_exact_gb300.inputs import make_inputs
from parity import Parity, check_tensor


def _noalloc_fn():
    L = attn.lib()
    fn = L.attn_bwd_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
    fn.restype = I
    return fn


def test_noalloc_rejects_oversized_problem_without_gpu_work():
    fn = _noalloc_fn()
    A = 1 << 20
    # B*H*N = 32514 rows at d = 128 is one row above the limit
    assert fn(A, A, A, A, A, A, A, A, 1, 2, 16257, 128, 1, 0.08, None) == 8
    assert fn(A, A, A, A, A, A, A, A, 1, 1, 128, 96, 0, 0.1, None) == 2
    assert "scratch" in attn.status_string(8)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 4, 1000, 128, True), (2, 3, 700, 64, False)])
def test_noalloc_matches_regular_backward_twice(B, H, N, d, causal):
    fn = _noalloc_fn()
    dev = torch.device("cuda:0")
    scale = d ** -0.5
    stream = torch.cuda.current_stream()
    for call in range(2):
        x = {k: v.to(dev) for k, v in make_inputs(B, H, N, d, seed=300 + call).items()}
        o, lse = attn.forward(x["q"], x["k"], x["v"], causal, scale)
        ref = attn.backward(x["q"], x["k"], x["v"], o, lse, x["dO"], causal, scale)
        out = [torch.empty_like(x["q"]) for _ in range(3)]
        rc = fn(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["dO"].data_ptr(),
                lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
                B, H, N, d, int(causal), scale, stream.cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        for name, a, b in zip(("dQ", "dK", "dV"), out, ref):
            check_tensor(name, a.float().cpu().numpy().astype(np.float64),
                         b.float().cpu().numpy().astype(np.float64))


@pytest.mark.gpu
def test_noalloc_at_the_size_limit_matches_oracle():
    """B*H*N = 32512 rows at d = 128: D takes the first 32512 floats and the
    dQ accumulator the next 32512 * 128, ending 256 floats before the end of
    the 4,194,304-float array.  The last heads' rows sit at the array's end;
    their dQ, dK, dV are compared with the oracle, every head's with attn_bwd."""
    fn = _noalloc_fn()
    B, H, N, d, causal = 1, 8, 4064, 128, True
    assert B * H * N + B * H * N * d <= (1 << 22) - 256
    dev = torch.device("cuda:0")
    scale = d ** -0.5
    stream = torch.cuda.current_stream()
    x = make_inputs(B, H, N, d, seed=310)
    xd = {k: v.to(dev) for k, v in x.items()}
    o, lse = attn.forward(xd["q"], xd["k"], xd["v"], causal, scale)
    ref = attn.backward(xd["q"], xd["k"], xd["v"], o, lse, xd["dO"], causal, scale)
    out = [torch.empty_like(xd["q"]) for _ in range(3)]
    rc = fn(xd["q"].data_ptr(), xd["k"].data_ptr(), xd["v"].data_ptr(), xd["dO"].data_ptr(),
            lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
            B, H, N, d, int(causal), scale, stream.cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    for name, a, b in zip(("dQ", "dK", "dV"), out, ref):
        check_tensor(name, f(a), f(b))
    pc = Parity("noalloc at the limit")
    for h in (H - 2, H - 1):
        qh, kh, vh, dOh = (f(x[n][0, h]) for n in ("q", "k", "v", "dO"))
        dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward(qh, kh, vh, dOh, causal, scale)
        pc.add("dQ", f(out[0][0, h]), dq_ref)
        pc.add("dK", f(out[1][0, h]), dk_ref)
        pc.add("dV", f(out[2][0, h]), dv_ref)
    pc.check()
