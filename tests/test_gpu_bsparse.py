"""GPU parity for block-sparse layouts.

A block mask holds one byte per 128 x 128 tile (query block, key block);
zero drops the tile from the softmax.  The CUDA training path
(attn_fwd_train_bsparse, attn_bwd_preprocess_o32, attn_bwd_bsparse) is
compared with the oracle's block-sparse functions on the same bf16 / fp16
values: O, lse, dQ, dK, dV of every row.  Masks are random per head or shared,
with causal masking on top or not, ragged N, query blocks that keep nothing
(O = 0, lse = -inf) and key blocks that no query keeps (dK = dV = 0).  An
all-ones mask must reproduce the dense kernels.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import io_aware_exact_gb300 as attn
from io_aware_exact_gb300.inputs import make_inputs
from parity import check_lse, check_tensor, dtype_name

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _mask(B, H, N, density, seed, shared=False):
    nb = (N + 127) // 128
    rng = np.random.default_rng(seed)
    shape = (nb, nb) if shared else (B, H, nb, nb)
    return (rng.random(shape) < density).astype(np.uint8)


def _run(x, mask, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    m = torch.from_numpy(mask).to(dev)
    o, lse, o32 = attn.forward_bsparse(q, k, v, m, causal, scale, o32=True)
    o2, lse2 = attn.forward_bsparse(q, k, v, m, causal, scale)
    dq, dk, dv = attn.backward_bsparse(q, k, v, o32, lse, dO, m, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    # the plain and training variants share lse (O differs in its normaliser:
    # the exact sum of p, or the sum of p as rounded for the P V product)
    assert torch.equal(lse, lse2)
    return {n: t.cpu() for n, t in dict(o=o, o_plain=o2, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def _compare(x, mask, out, causal, scale):
    B, H, N, d = x["q"].shape
    ref = {n: [] for n in ("o", "lse", "dq", "dk", "dv")}
    for b in range(B):
        for h in range(H):
            mb = mask if mask.ndim == 2 else mask[b, h]
            q, k, v, dO = (_f64(x[n][b, h]) for n in ("q", "k", "v", "dO"))
            o, lse = oracle.attention_forward_block_sparse(q, k, v, mb, causal, scale)
            dq, dk, dv, _, _ = oracle.attention_backward_block_sparse(q, k, v, dO, mb, causal,
                                                                      scale)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
                ref[n].append(t)
    ref = {n: np.stack(t).reshape((B, H) + t[0].shape) for n, t in ref.items()}
    lse = out["lse"].numpy().astype(np.float64)
    empty = np.isneginf(ref["lse"])
    assert np.array_equal(np.isneginf(lse), empty), "rows with an empty softmax differ"
    assert np.all(out["o"].float().numpy()[empty] == 0.0)
    check_lse(lse[~empty], ref["lse"][~empty])
    assert np.all(out["o_plain"].float().numpy()[empty] == 0.0)
    for n in ("o", "o_plain", "dq", "dk", "dv"):
        check_tensor(n, _f64(out[n]).reshape(-1, d), ref[n[:1] if n == "o_plain" else n].reshape(-1, d),
                     dtype=dtype_name(x["q"]))
    return ref, empty


@pytest.mark.parametrize("B,H,N,d,causal,density,shared,dtype", [
    (1, 2, 1000, 64, False, 0.5, False, torch.bfloat16),
    (1, 2, 1000, 128, True, 0.5, False, torch.bfloat16),
    (2, 2, 640, 128, True, 0.6, True, torch.float16),
    (1, 3, 1536, 64, True, 0.3, False, torch.bfloat16),
    (1, 2, 2048, 128, False, 0.25, False, torch.bfloat16),
    (1, 1, 1, 64, False, 1.0, True, torch.bfloat16),          # one row, one tile
    (2, 2, 200, 64, True, 0.7, True, torch.float16),          # ragged, fp16, d = 64
])
def test_block_sparse_matches_oracle(B, H, N, d, causal, density, shared, dtype):
    x = make_inputs(B, H, N, d, seed=500 + N + d, dtype=dtype)
    mask = _mask(B, H, N, density, seed=N + H, shared=shared)
    scale = d ** -0.5
    out = _run(x, mask, causal, scale)
    _compare(x, mask, out, causal, scale)


def test_empty_query_and_key_blocks():
    """Query block 1 keeps nothing (O = 0, lse = -inf, dQ = 0) and key block 3
    is kept by no query (dK = dV = 0), with causal masking on top."""
    B, H, N, d = 1, 2, 900, 128
    x = make_inputs(B, H, N, d, seed=611)
    nb = (N + 127) // 128
    mask = np.tril(np.ones((nb, nb), np.uint8))
    mask[1, :] = 0
    mask[:, 3] = 0
    out = _run(x, mask, True, d ** -0.5)
    _, empty = _compare(x, mask, out, True, d ** -0.5)
    assert empty[:, :, 128:256].all() and not empty[:, :, :128].any()
    assert torch.all(out["dq"][:, :, 128:256] == 0)
    assert torch.all(out["dk"][:, :, 384:512] == 0) and torch.all(out["dv"][:, :, 384:512] == 0)


def test_all_dropped_mask():
    B, H, N, d = 1, 1, 700, 64
    x = make_inputs(B, H, N, d, seed=612)
    mask = np.zeros((6, 6), np.uint8)
    out = _run(x, mask, False, d ** -0.5)
    assert torch.all(out["o"] == 0) and torch.all(torch.isneginf(out["lse"]))
    for n in ("dq", "dk", "dv"):
        assert torch.all(out[n] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_reproduces_dense_kernels(causal):
    """With every tile kept the block-sparse kernels do the dense kernels' work
    in the same order: O, fp32 O, lse, dK and dV are bit-identical (dQ is
    summed with unordered reductions, so it is compared within tolerance)."""
    B, H, N, d = 2, 4, 1000, 128
    dev = torch.device("cuda:0")
    x = {n: t.to(dev) for n, t in make_inputs(B, H, N, d, seed=613).items()}
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    scale = d ** -0.5
    m = torch.ones((8, 8), dtype=torch.uint8, device=dev)
    o_s, lse_s, o32_s = attn.forward_bsparse(q, k, v, m, causal, scale, o32=True)
    o_d, lse_d, o32_d = attn.forward(q, k, v, causal, scale, o32=True)
    dq_s, dk_s, dv_s = attn.backward_bsparse(q, k, v, o32_s, lse_s, dO, m, causal, scale)
    dq_d, dk_d, dv_d = attn.backward(q, k, v, None, lse_d, dO, causal, scale, o32=o32_d)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert torch.equal(o_s, o_d) and torch.equal(lse_s, lse_d) and torch.equal(o32_s, o32_d)
    assert torch.equal(dk_s, dk_d) and torch.equal(dv_s, dv_d)
    check_tensor("dq", _f64(dq_s).reshape(-1, d), _f64(dq_d).reshape(-1, d))
