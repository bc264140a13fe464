"""The ring attention schedule on CPU ranks (gloo), with the oracle as the
arithmetic.

Each rank holds one chunk of the sequence and runs io_aware_exact_gb300.ring's
forward and backward schedules over torch.distributed point-to-point
transfers; the per-chunk arithmetic is the oracle's (fp64): attention of a
query chunk against a key chunk, the exact merge of partial results, and the
backward with the whole rows' lse and D.  The gathered result must equal the
oracle's attention over the whole sequence, so this checks the ring order,
the causal skipping of chunks, the transfers and the accumulation of dK, dV
as they travel.  The single-process driver (run_local) is checked against the
same reference.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleOps:
    """Per-chunk arithmetic of the ring from the fp64 oracle (CPU tensors).
    k, v may have fewer heads than q (grouped heads: query head h reads K / V
    head oracle.kv_head_of(h, H, Hkv), and dK, dV sum over the group)."""

    def fwd_chunk(self, q, k, v, causal, scale):
        import oracle
        B, H, N, _ = q.shape
        Hkv = k.shape[1]
        o = torch.empty((B, H, N, v.shape[-1]), dtype=torch.float64)
        lse = torch.empty((B, H, N), dtype=torch.float64)
        for b in range(B):
            for h in range(H):
                g = oracle.kv_head_of(h, H, Hkv)
                ob, lb = oracle.attention_forward(q[b, h].numpy(), k[b, g].numpy(),
                                                  v[b, g].numpy(), causal, scale)
                o[b, h], lse[b, h] = torch.from_numpy(ob), torch.from_numpy(lb)
        return o, lse

    def merge(self, o_acc, lse_acc, o_part, lse_part):
        import oracle
        o, lse = oracle.merge_partials(o_acc.numpy(), lse_acc.numpy(), o_part.numpy(),
                                       lse_part.numpy())
        o_acc.copy_(torch.from_numpy(o))
        lse_acc.copy_(torch.from_numpy(lse))

    def finish_output(self, o32, dtype):
        return o32.clone()

    def bwd_prepare(self, o32, dO):
        return (dO * o32).sum(-1), torch.zeros(dO.shape, dtype=torch.float64)

    def bwd_chunk(self, q, k, v, dO, lse, D, dq_acc, dk_acc, dv_acc, causal, scale):
        import oracle
        B, H = q.shape[:2]
        Hkv = k.shape[1]
        dk, dv = torch.zeros_like(k), torch.zeros_like(v)
        for b in range(B):
            for h in range(H):
                g = oracle.kv_head_of(h, H, Hkv)
                gq, gk, gv = oracle.attention_backward_given_stats(
                    q[b, h].numpy(), k[b, g].numpy(), v[b, g].numpy(), dO[b, h].numpy(),
                    lse[b, h].numpy(), D[b, h].numpy(), causal, scale)
                dq_acc[b, h] += torch.from_numpy(gq)
                dk[b, g] += torch.from_numpy(gk)
                dv[b, g] += torch.from_numpy(gv)
        if dk_acc is None:
            return dq_acc.clone(), dk, dv
        return dq_acc.clone(), dk_acc.add_(dk), dv_acc.add_(dv)

    def finish_grad(self, acc, dtype):
        return acc.clone()


def _data(R, Nc, seed=7):
    g = torch.Generator().manual_seed(seed)
    B, H, d = 1, 2, 4
    mk = lambda: torch.randn((B, H, R * Nc, d), generator=g, dtype=torch.float64)
    return mk(), mk(), mk(), mk()


def _reference(q, k, v, dO, causal, scale):
    import oracle
    B, H = q.shape[:2]
    out = {n: [] for n in ("o", "lse", "dq", "dk", "dv")}
    for b in range(B):
        for h in range(H):
            o, lse = oracle.attention_forward(q[b, h], k[b, h], v[b, h], causal, scale)
            dq, dk, dv, _, _ = oracle.attention_backward(q[b, h], k[b, h], v[b, h], dO[b, h],
                                                        causal, scale)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
                out[n].append(t)
    return {n: np.stack(t).reshape((B, H) + t[0].shape) for n, t in out.items()}


def _chunks(t, R):
    return [c.contiguous() for c in torch.chunk(t, R, dim=2)]


def _worker(rank, R, port, causal, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=R)
    from io_aware_exact_gb300 import ring
    q, k, v, dO = (_chunks(t, R)[rank] for t in _data(R, 3))
    scale = 0.6
    ops = OracleOps()
    o, lse, o32 = ring.run_distributed(ring.forward_schedule(rank, R, q, k, v, causal, scale, ops),
                                       rank, R)
    dq, dk, dv = ring.run_distributed(
        ring.backward_schedule(rank, R, q, k, v, o32, lse, dO, causal, scale, ops), rank, R)
    torch.save({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
               os.path.join(out_dir, "rank%d.pt" % rank))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _check(got, ref):
    for n in ("o", "lse", "dq", "dk", "dv"):
        err = np.max(np.abs(got[n] - ref[n]))
        assert err < 1e-11, "%s: max abs err %.3e" % (n, err)


@pytest.mark.parametrize("R,causal", [(2, False), (2, True), (3, True)])
def test_ring_over_gloo_ranks_equals_whole_sequence(R, causal, tmp_path):
    mp.start_processes(_worker, args=(R, _free_port(), causal, str(tmp_path)), nprocs=R,
                       join=True, start_method="spawn")
    parts = [torch.load(os.path.join(tmp_path, "rank%d.pt" % r)) for r in range(R)]
    got = {n: torch.cat([p[n] for p in parts], dim=2).numpy() for n in parts[0]}
    _check(got, _reference(*(t.numpy() for t in _data(R, 3)), causal, 0.6))


@pytest.mark.parametrize("R,causal", [(1, True), (3, False), (4, True)])
def test_ring_in_one_process_equals_whole_sequence(R, causal):
    from io_aware_exact_gb300 import ring
    q, k, v, dO = _data(R, 2, seed=11)
    qs, ks, vs, dOs = (_chunks(t, R) for t in (q, k, v, dO))
    o, lse, o32 = ring.ring_forward(qs, ks, vs, causal, 0.8, OracleOps)
    dq, dk, dv = ring.ring_backward(qs, ks, vs, o32, lse, dOs, causal, 0.8, OracleOps)
    got = {n: torch.cat(t, dim=2).numpy()
           for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    _check(got, _reference(q.numpy(), k.numpy(), v.numpy(), dO.numpy(), causal, 0.8))


@pytest.mark.parametrize("causal", [False, True])
def test_ring_with_grouped_heads_equals_whole_sequence(causal):
    """Grouped K / V heads (4 query heads, 2 K / V heads) through the ring in
    one process: K / V chunks of Hkv heads travel, dK, dV sum over each group."""
    import oracle
    from io_aware_exact_gb300 import ring
    R, Nc, d = 3, 3, 4
    g = torch.Generator().manual_seed(21)
    q = torch.randn((1, 4, R * Nc, d), generator=g, dtype=torch.float64)
    dO = torch.randn((1, 4, R * Nc, d), generator=g, dtype=torch.float64)
    k = torch.randn((1, 2, R * Nc, d), generator=g, dtype=torch.float64)
    v = torch.randn((1, 2, R * Nc, d), generator=g, dtype=torch.float64)
    qs, ks, vs, dOs = (_chunks(t, R) for t in (q, k, v, dO))
    o, lse, o32 = ring.ring_forward(qs, ks, vs, causal, 0.7, OracleOps)
    dq, dk, dv = ring.ring_backward(qs, ks, vs, o32, lse, dOs, causal, 0.7, OracleOps)
    o_ref, lse_ref = oracle.attention_forward_grouped(q[0].numpy(), k[0].numpy(), v[0].numpy(),
                                                      causal, 0.7)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.attention_backward_grouped(
        q[0].numpy(), k[0].numpy(), v[0].numpy(), dO[0].numpy(), causal, 0.7)
    for got, ref in ((o, o_ref), (lse, lse_ref), (dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        err = np.max(np.abs(torch.cat(got, dim=2)[0].numpy() - ref))
        assert err < 1e-11
