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
    """Per-chunk arithmetic of the ring from the fp64 oracle (CPU tensors)."""

    def fwd_chunk(self, q, k, v, causal, scale):
        import oracle
        B, H, N, _ = q.shape
        o = torch.empty((B, H, N, v.shape[-1]), dtype=torch.float64)
        lse = torch.empty((B, H, N), dtype=torch.float64)
        for b in range(B):
            for h in range(H):
                ob, lb = oracle.attention_forward(q[b, h].numpy(), k[b, h].numpy(),
                                                  v[b, h].numpy(), causal, scale)
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
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        for b in range(B):
            for h in range(H):
                gq, gk, gv = oracle.attention_backward_given_stats(
                    q[b, h].numpy(), k[b, h].numpy(), v[b, h].numpy(), dO[b, h].numpy(),
                    lse[b, h].numpy(), D[b, h].numpy(), causal, scale)
                dq_acc[b, h] += torch.from_numpy(gq)
                dk[b, h], dv[b, h] = torch.from_numpy(gk), torch.from_numpy(gv)
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
