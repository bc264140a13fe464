"""Comparison helpers shared by the GPU parity tests, the smoke check and bench.

Tolerances (bf16/fp16 inputs, fp32 accumulation), for O, dQ, dK and dV, each
taken over the whole checked subset of one output tensor (all the heads,
rows or key columns that a test compares):

* mean criterion: mean |x - ref| / RMS(ref over the checked subset) <= 2e-3;
* max criterion: every element's error beyond the rounding of the stored
  output, |x - ref| - u |ref| (u the unit roundoff of the output type: 2^-8
  for bf16, 2^-11 for fp16, 2^-24 for fp32), divided by the larger of the
  RMS of its row (the d values of one query row for O and dQ, of one key row
  for dK and dV) and the RMS of the checked subset, is <= 2e-2;

and lse within 1e-3 absolute.  Why this form: with a causal mask the first
rows are up to ~20x the tensor's RMS, so storing the exact result rounded to
bf16 already costs 3.7e-2 to 8.8e-2 of the tensor-wide RMS (dQ, one head,
N=2048): against the tensor RMS alone the max criterion would reject a
correctly rounded result.  Against the row's RMS alone, single entries of
~10x their row's RMS (peaked softmax rows) lose up to 2^-8 x 10 = 3.9e-2 of
the row RMS to the same rounding.  An ideal implementation that rounds P and
dS to bf16 for the tensor cores and stores bf16 outputs (fp64 otherwise)
gives max errors of 2.11e-2 (dQ), 1.89e-2 (dK) and 2.02e-2 (dV) of the row
RMS on the Q, K x8 causal case of the GPU tests (B=1, H=2, N=1024, d=128) --
exactly what the kernels give -- and 1.8e-3 mean error on non-causal dV
(N=1000, d=64), again equal to the kernels'.  Taking the output's own
rounding out of the max criterion keeps it no looser than the numerics
need: a wrong row, mask or term still fails it by orders of magnitude, and
the mean criterion catches a systematic error of a few tenths of a percent.

Every comparison also computes the max error under three other rules: the
row rule without the rounding term, the tensor RMS alone, and the largest of
|ref|, the row RMS and the tensor RMS (a per-element relative rule), so that
a report shows how far each output is from each reading of "normalised by
output RMS".  With the environment
variable ``ATTN_PARITY_REPORT`` set to a file name, each check appends one
JSON line with all five figures; ``python tests/parity.py summarize FILE``
prints them as a table.
The oracle is the fp64 CPU implementation in ``oracle/``.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE = 1e-3

# unit roundoff of the stored output type (round to nearest)
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}


def dtype_name(t):
    """"bf16", "f16" or "f32" for a torch dtype (or a tensor)."""
    s = str(getattr(t, "dtype", t))
    return "bf16" if "bfloat16" in s else "f16" if "float16" in s else "f32"


def errors(x, ref, dtype="bf16"):
    """All figures of one comparison, for arrays of rows (last axis = row).

    max_store:  max (|x - ref| - u |ref|) / max(row RMS, tensor RMS), u the
                unit roundoff of `dtype`                   (the enforced rule)
    max_row:    max |x - ref| / max(row RMS, tensor RMS)
    max_tensor: max |x - ref| / tensor RMS
    max_elem:   max |x - ref| / max(|ref|, row RMS, tensor RMS)
    mean:       mean |x - ref| / tensor RMS                 (the enforced rule)
    The tensor RMS is that of ref over everything passed in."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if not np.all(np.isfinite(x)):
        inf = float("inf")
        return dict(max_store=inf, max_row=inf, max_tensor=inf, max_elem=inf, mean=inf)
    if ref.size == 0:
        return dict(max_store=0.0, max_row=0.0, max_tensor=0.0, max_elem=0.0, mean=0.0)
    if ref.ndim == 1:
        ref = ref[None, :]
        x = x[None, :]
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        rms = 1.0
    diff = np.abs(x - ref)
    row_rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    row_den = np.maximum(row_rms, rms)
    u = UNIT_ROUNDOFF[dtype]
    return dict(max_store=float(((diff - u * np.abs(ref)) / row_den).max()),
                max_row=float((diff / row_den).max()),
                max_tensor=float(diff.max() / rms),
                max_elem=float((diff / np.maximum(row_den, np.abs(ref))).max()),
                mean=float(diff.mean() / rms))


def rel_errors(x, ref, dtype="bf16"):
    """(max error under the enforced rule, mean error over the tensor RMS)."""
    e = errors(x, ref, dtype)
    return e["max_store"], e["mean"]


def _report(record):
    path = os.environ.get("ATTN_PARITY_REPORT")
    if not path:
        return
    record = dict(record)
    record["test"] = os.environ.get("PYTEST_CURRENT_TEST", "").split(" (")[0]
    with open(path, "a") as f:
        f.write(json.dumps(record) + "\n")


def check_tensor(name, x, ref, report=None, label="", dtype="bf16"):
    """Compare one output tensor (or the stacked rows of several heads) stored
    as `dtype` ("bf16", "f16" or "f32")."""
    e = errors(x, ref, dtype)
    if report is not None:
        report[name] = (e["max_store"], e["mean"])
    _report(dict(label=label, tensor=name, dtype=dtype,
                 rows=int(np.asarray(ref).size // max(1, np.asarray(ref).shape[-1])), **e))
    assert e["max_store"] <= TOL_MAX and e["mean"] <= TOL_MEAN, \
        "%s: max err beyond output rounding %.3e of row RMS (tol %.0e), mean err %.3e of RMS " \
        "(tol %.0e); without the rounding term %.3e, tensor-RMS max %.3e, per-element max %.3e" % (
            name, e["max_store"], TOL_MAX, e["mean"], TOL_MEAN, e["max_row"], e["max_tensor"],
            e["max_elem"])


def check_lse(x, ref, report=None, label=""):
    x = np.asarray(x, dtype=np.float64)
    err = float(np.max(np.abs(x - np.asarray(ref)))) if x.size else 0.0
    if not np.all(np.isfinite(x)):
        err = float("inf")
    if report is not None:
        report["lse"] = err
    _report(dict(label=label, tensor="lse", rows=int(x.size), max_abs=err))
    assert err <= TOL_LSE, "lse: max abs err %.3e (tol %.0e)" % (err, TOL_LSE)


class Parity:
    """Collects the compared pieces of each output over several heads (or
    row / column samples) and checks each tensor once, against the RMS of
    everything collected for it.  Pieces of one tensor must have the same
    row length."""

    def __init__(self, label="", dtype="bf16"):
        self.label = label
        self.dtype = dtype
        self.parts = {}
        self.lse = []

    def add(self, name, x, ref, dtype=None):
        """dtype: storage type of this output (default: the collector's)."""
        x = np.asarray(x, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert x.shape == ref.shape, (name, x.shape, ref.shape)
        if ref.ndim == 1:
            x, ref = x[None, :], ref[None, :]
        d = ref.shape[-1]
        self.parts.setdefault(name, []).append((x.reshape(-1, d), ref.reshape(-1, d),
                                                dtype or self.dtype))

    def add_lse(self, x, ref):
        self.lse.append((np.asarray(x, dtype=np.float64).ravel(),
                         np.asarray(ref, dtype=np.float64).ravel()))

    def check(self, report=None):
        failures = []
        for name, parts in self.parts.items():
            x = np.concatenate([p[0] for p in parts])
            ref = np.concatenate([p[1] for p in parts])
            try:
                check_tensor(name, x, ref, report, self.label, parts[0][2])
            except AssertionError as e:
                failures.append(str(e))
        if self.lse:
            x = np.concatenate([p[0] for p in self.lse])
            ref = np.concatenate([p[1] for p in self.lse])
            try:
                check_lse(x, ref, report, self.label)
            except AssertionError as e:
                failures.append(str(e))
        assert not failures, "; ".join(failures)


def sample_rows(N, n, seed=0):
    """A sorted sample of row indices that always includes both ends and the
    last partial 128-row tile, when there is one."""
    rng = np.random.default_rng(seed)
    fixed = {0, N - 1, min(N - 1, 127), min(N - 1, 128), (N // 128) * 128 if N % 128 else N - 1}
    k = max(0, min(N, n) - len(fixed))
    extra = rng.choice(N, size=k, replace=False) if k else []
    return np.array(sorted(fixed | set(int(e) for e in extra)), dtype=np.int64)


def summarize(path):
    """Markdown table of a report file: the largest figure per test and tensor."""
    worst = {}
    for line in open(path):
        r = json.loads(line)
        key = (r["test"], r["tensor"])
        w = worst.setdefault(key, {})
        for k in ("max_store", "max_row", "max_tensor", "max_elem", "mean", "max_abs"):
            if k in r:
                w[k] = max(w.get(k, -1.0), r[k])
    keys = ("max_store", "max_row", "max_tensor", "max_elem", "mean")
    out = ["| test | tensor | beyond rounding / row RMS (enforced, 2e-2) | max / row RMS | "
           "max / tensor RMS | max / max(|ref|, RMS) | mean / RMS (enforced, 2e-3) |",
           "|---|---|---|---|---|---|---|"]
    for (test, tensor), w in sorted(worst.items()):
        if tensor == "lse":
            out.append("| %s | lse | max abs %.2e (1e-3) | | | | |" % (test, w["max_abs"]))
        else:
            out.append("| %s | %s | %s |" % (test, tensor, " | ".join(
                "%.2e" % w.get(k, float("nan")) for k in keys)))
    overall = {}
    for (test, tensor), w in worst.items():
        if tensor == "lse":
            overall["lse"] = max(overall.get("lse", 0.0), w["max_abs"])
            continue
        for k in keys:
            overall[k] = max(overall.get(k, -1.0), w.get(k, -1.0))
    if overall:
        out.append("")
        out.append("Largest over all checks: beyond rounding / row RMS %.2e (enforced), "
                   "max / row RMS %.2e, max / tensor RMS %.2e, per-element %.2e, mean %.2e "
                   "(enforced), lse %.2e" % tuple(overall.get(k, float("nan")) for k in keys + ("lse",)))
    return "\n".join(out)


if __name__ == "__main__":
    if len(sys.argv) == 3 and sys.argv[1] == "summarize":
        print(summarize(sys.argv[2]))
    else:
        print("usage: python tests/parity.py summarize REPORT.jsonl")
