"""CPU checks of the comparison rule used by every GPU parity test."""
import numpy as np
import torch

from parity import TOL_MAX, TOL_MEAN, rel_errors, sample_rows


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def _causal_like(n=512, d=64, seed=0):
    """Rows shaped like causal attention outputs: row i averages i+1 values."""
    r = np.random.default_rng(seed)
    v = r.normal(size=(n, d))
    return np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]


def test_correctly_rounded_bf16_passes():
    ref = _causal_like()
    emax, emean = rel_errors(_bf16(ref), ref)
    assert emax <= TOL_MAX and emean <= TOL_MEAN


def test_tensor_wide_rms_alone_would_reject_correct_rounding():
    """Why the max criterion uses the row RMS: with the tensor-wide RMS only,
    the exact result rounded to bf16 already fails on the first rows."""
    ref = _causal_like()
    diff = np.abs(_bf16(ref) - ref)
    assert diff.max() / np.sqrt(np.mean(ref * ref)) > TOL_MAX


def test_planted_errors_are_caught():
    ref = _causal_like()
    bad = ref.copy()
    bad[100] *= 1.05                      # one row 5% off
    assert rel_errors(bad, ref)[0] > TOL_MAX
    bad = ref.copy()
    bad[:, 3] += 0.05 * np.sqrt(np.mean(ref * ref))   # a biased column
    assert rel_errors(bad, ref)[0] > TOL_MAX or rel_errors(bad, ref)[1] > TOL_MEAN
    bad = ref * (1 + 5e-3)                # a small global scale error
    assert rel_errors(bad, ref)[1] > TOL_MEAN
    nan = ref.copy()
    nan[5, 5] = np.nan
    assert rel_errors(nan, ref)[0] == float("inf")


def test_tiny_rows_use_tensor_rms():
    """A row whose reference is ~0 is judged against the tensor's RMS, not its own."""
    ref = _causal_like()
    ref[200] = 1e-12
    x = ref.copy()
    x[200] = 1e-4
    assert rel_errors(x, ref)[0] <= TOL_MAX


def test_sample_rows_covers_edges():
    s = sample_rows(1000, 20, seed=3)
    assert s[0] == 0 and s[-1] == 999 and 896 in s and 127 in s and 128 in s
    assert len(set(s.tolist())) == len(s)


def test_report_figures_order():
    """The per-element rule is the loosest and the tensor-RMS rule the
    strictest reading of the max criterion; the enforced row rule lies
    between them."""
    from parity import errors
    ref = _causal_like()
    e = errors(_bf16(ref), ref)
    assert e["max_elem"] <= e["max_row"] <= e["max_tensor"]
    assert e["max_row"] <= TOL_MAX < e["max_tensor"]


def test_collector_uses_one_rms_per_tensor():
    """Pieces collected from several heads are judged against the RMS of all
    of them: a head with tiny outputs cannot hide a large absolute error
    behind its own small RMS, and a 1% scale error on one of two heads still
    fails the mean criterion."""
    import pytest
    from parity import Parity
    ref_a = _causal_like(seed=1)
    ref_b = _causal_like(seed=2)
    pc = Parity("ok")
    pc.add("O", _bf16(ref_a), ref_a)
    pc.add("O", _bf16(ref_b), ref_b)
    pc.check()
    pc = Parity("bad")
    pc.add("O", ref_a * (1 + 1e-2), ref_a)
    pc.add("O", ref_b, ref_b)
    with pytest.raises(AssertionError):
        pc.check()
