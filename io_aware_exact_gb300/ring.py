"""Ring attention: exact attention over a sequence split into chunks.

The paldyn.com survey "어텐션 비용 줄이기" (section "다중 GPU 확장") describes
ring attention: each device keeps its share of the queries and the key /
value blocks travel around a ring of devices; inside each device the work is
the single-device attention kernel.  Partial results over different key
chunks combine exactly by their logsumexps (sj-techlog "FlashAttention 원 논문
해부", section "두 tile을 한 row로 합치는 식"), so the result is the attention
over the whole sequence.

Layout and masking.  The sequence of length R * Nc is split into R equal
chunks; chunk c is positions [c Nc, (c + 1) Nc).  Rank r holds q, k, v (and
dO) of chunk r as [B, H, Nc, d] tensors.  With ``causal`` (top-left over the
whole sequence) key chunk c is fully visible to the queries of chunk r when
c < r, causal within the chunk when c == r, and invisible (skipped) when
c > r.

Forward, rank r: for R steps, attend q to the key / value chunk in hand (the
training forward, giving an fp32 O normalised over that chunk and its lse),
merge it into the running (O, lse), and pass the chunk to rank r + 1 while
receiving the next one from rank r - 1.

Backward, rank r: D = rowsum(dO o O) from the merged fp32 O and the fp32 dQ
accumulator zeroed once; then for R steps the backward kernel of q against
the chunk in hand with the row statistics of the whole sequence (lse, D)
adds that chunk's share into dQ and adds the pair's share of dK, dV into fp32
sums that travel with the chunk (written by the backward kernel itself, so
no partial result is rounded to 16 bits).  After R passes the
accumulators are back with their owner and are rounded to 16 bits.

The schedule of one rank is a generator that yields ("send", payload) when
its payload should go to the next rank and ("recv",) when it needs the one
from the previous rank.  Two drivers run it: :func:`run_distributed`
(torch.distributed point-to-point, one process per device) and
:func:`run_local` (R ranks in one process, in lock step, passing the payloads
around a list: one device emulating the ring, with no kernel waiting on
another).  The arithmetic goes through an ``ops`` object; :class:`CudaOps`
(the library's kernels) is the default.
"""
from __future__ import annotations

from typing import Callable, List, Sequence


class CudaOps:
    """The library's kernels: training forward, merge, D preprocess, backward
    into fp32 dK / dV sums, and the final rounding.  Raises if the library is not
    available (there is no other implementation here)."""

    def __init__(self, stream=None):
        from io_aware_exact_gb300 import lib
        lib()
        self.stream = stream

    def fwd_chunk(self, q, k, v, causal, scale):
        import io_aware_exact_gb300 as attn
        _, lse, o32 = attn.forward(q, k, v, causal, scale, o32=True, stream=self.stream)
        return o32, lse

    def merge(self, o_acc, lse_acc, o_part, lse_part):
        import io_aware_exact_gb300 as attn
        attn.merge(o_acc, lse_acc, o_part, lse_part, stream=self.stream)

    def finish_output(self, o32, dtype):
        import io_aware_exact_gb300 as attn
        return attn.convert(o32, dtype, 1.0, stream=self.stream)

    def bwd_prepare(self, o32, dO):
        import torch
        import io_aware_exact_gb300 as attn
        B, H, N, d = dO.shape
        D = torch.empty((B, H, N), dtype=torch.float32, device=dO.device)
        acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dO.device)
        attn.attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), acc.data_ptr(),
                                     B, H, N, d, attn._stream_handle(self.stream),
                                     dO.dtype == torch.float16)
        return D, acc

    def bwd_chunk(self, q, k, v, dO, lse, D, dq_acc, dk_acc, dv_acc, causal, scale):
        """dQ so far (dq_acc gains this pair's share), and dk_acc, dv_acc (fp32,
        created on the first call) with this pair's share of dK, dV added."""
        import torch
        import io_aware_exact_gb300 as attn
        B, H, N, d = q.shape
        first = dk_acc is None
        if first:
            dk_acc = torch.empty(k.shape, dtype=torch.float32, device=k.device)
            dv_acc = torch.empty(v.shape, dtype=torch.float32, device=v.device)
        dq = torch.empty_like(q)
        attn.attn_bwd_acc(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                          D.data_ptr(), dq_acc.data_ptr(), dq.data_ptr(), dk_acc.data_ptr(),
                          dv_acc.data_ptr(), not first, B, H, k.shape[1], N, d, causal, scale,
                          attn._stream_handle(self.stream), q.dtype == torch.float16)
        return dq, dk_acc, dv_acc

    def finish_grad(self, acc, dtype):
        import io_aware_exact_gb300 as attn
        return attn.convert(acc, dtype, 1.0, stream=self.stream)


def forward_schedule(rank: int, R: int, q, k, v, causal: bool, scale: float, ops):
    """Rank ``rank``'s forward; returns (o, lse, o32) of its query chunk."""
    c, kv, acc = rank, [k, v], None
    for step in range(R):
        if step < R - 1:
            yield ("send", kv)
        if not causal or c <= rank:
            o32, lse = ops.fwd_chunk(q, kv[0], kv[1], causal and c == rank, scale)
            if acc is None:
                acc = [o32, lse]
            else:
                ops.merge(acc[0], acc[1], o32, lse)
        if step < R - 1:
            kv = yield ("recv",)
            c = (c - 1) % R
    # step 0 is the rank's own chunk, always visible: acc is set
    return ops.finish_output(acc[0], q.dtype), acc[1], acc[0]


def backward_schedule(rank: int, R: int, q, k, v, o32, lse, dO, causal: bool, scale: float, ops):
    """Rank ``rank``'s backward; returns (dq, dk, dv) of its chunk."""
    D, dq_acc = ops.bwd_prepare(o32, dO)
    c, payload, dq = rank, [k, v, None, None], None
    for step in range(R):
        if not causal or c <= rank:
            dq, payload[2], payload[3] = ops.bwd_chunk(q, payload[0], payload[1], dO, lse, D,
                                                       dq_acc, payload[2], payload[3],
                                                       causal and c == rank, scale)
        # every chunk is kept by its own rank at step 0, so its accumulators
        # exist from then on; after R passes they are back with their owner
        yield ("send", payload)
        payload = yield ("recv",)
        c = (c - 1) % R
    return dq, ops.finish_grad(payload[2], k.dtype), ops.finish_grad(payload[3], v.dtype)


def run_local(schedules: Sequence) -> List:
    """Run R rank schedules in one process, in lock step: at each exchange
    every rank's payload moves to the next rank.  Returns their results."""
    gens = list(schedules)
    R = len(gens)
    results: List = [None] * R
    pending = [None] * R          # what each generator yielded last
    for r, g in enumerate(gens):
        try:
            pending[r] = next(g)
        except StopIteration as e:  # a ring of one rank exchanges nothing
            results[r] = e.value
    while True:
        if all(p is None for p in pending):
            return results
        outgoing = [None] * R
        for r, g in enumerate(gens):
            # advance each rank until it waits for a payload (or finishes)
            while pending[r] is not None and pending[r][0] == "send":
                outgoing[r] = pending[r][1]
                try:
                    pending[r] = next(g)
                except StopIteration as e:
                    results[r], pending[r] = e.value, None
        if any(p is not None and p[0] != "recv" for p in pending):
            raise RuntimeError("ring schedule out of step")
        for r, g in enumerate(gens):
            if pending[r] is None:
                continue
            try:
                pending[r] = g.send(outgoing[(r - 1) % R])
            except StopIteration as e:
                results[r], pending[r] = e.value, None


def run_distributed(schedule, rank: int, R: int, group=None):
    """Run this process's rank schedule with torch.distributed point-to-point
    transfers to rank + 1 and from rank - 1 (NCCL between GPUs, gloo on CPU).
    Sends are posted as soon as the schedule yields them, so the transfer of
    the next chunk overlaps the work on the current one."""
    import torch
    import torch.distributed as dist
    nxt, prv = (rank + 1) % R, (rank - 1) % R
    reqs, recv_bufs = [], None     # transfers in flight (each waited on once)
    try:
        item = next(schedule)
        while True:
            if item[0] == "send":
                payload = item[1]
                recv_bufs = [None if t is None else torch.empty_like(t) for t in payload]
                p2p = [dist.P2POp(dist.isend, t, nxt, group) for t in payload if t is not None]
                p2p += [dist.P2POp(dist.irecv, b, prv, group) for b in recv_bufs if b is not None]
                reqs = dist.batch_isend_irecv(p2p) if p2p else []
                item = next(schedule)
            else:
                for rq in reqs:
                    rq.wait()
                reqs = []
                item = schedule.send(recv_bufs)
    except StopIteration as e:
        for rq in reqs:
            rq.wait()
        return e.value


def ring_forward(qs, ks, vs, causal: bool, scale: float, ops_factory: Callable = CudaOps):
    """Ring forward of R chunks emulated in one process (run_local).  qs, ks, vs
    are lists of [B, H, Nc, d] chunks; returns lists of o, lse, o32."""
    R = len(qs)
    res = run_local([forward_schedule(r, R, qs[r], ks[r], vs[r], causal, scale, ops_factory())
                     for r in range(R)])
    return [x[0] for x in res], [x[1] for x in res], [x[2] for x in res]


def ring_backward(qs, ks, vs, o32s, lses, dOs, causal: bool, scale: float,
                  ops_factory: Callable = CudaOps):
    """Ring backward of R chunks emulated in one process; lists of dq, dk, dv."""
    R = len(qs)
    res = run_local([backward_schedule(r, R, qs[r], ks[r], vs[r], o32s[r], lses[r], dOs[r],
                                       causal, scale, ops_factory()) for r in range(R)])
    return [x[0] for x in res], [x[1] for x in res], [x[2] for x in res]
