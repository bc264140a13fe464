"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library is built with nvcc (cross-compiling for sm_103a) and loaded with
ctypes; these tests check that it exports every function include/attn.h
declares and that argument errors are reported synchronously with the
documented codes, before any device work.
"""
import ast
import ctypes
import re
import glob
import os

import pytest

import io_aware_exact_gb300 as attn
from io_aware_exact_gb300 import build as attn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    attn_build.build()
    return attn.lib()


def test_exports_every_declared_function(L):
    names = attn.header_functions()
    assert {"attn_fwd", "attn_bwd_preprocess", "attn_bwd"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(8):
        assert attn.status_string(code)
    assert "aligned" in attn.status_string(3)
    assert attn.version().startswith("io_aware_exact_gb300")


A = 1 << 20  # a 16-byte aligned fake address; never dereferenced by these tests


def _fwd(L, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return L.attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def _bwd(L, **kw):
    a = dict(q=A, k=A, v=A, dO=A, lse=A, D=A, acc=A, dq=A, dk=A, dv=A, B=1, H=1, N=128,
             d=64, causal=0, scale=0.125)
    a.update(kw)
    return L.attn_bwd(a["q"], a["k"], a["v"], a["dO"], a["lse"], a["D"], a["acc"],
                      a["dq"], a["dk"], a["dv"], a["B"], a["H"], a["N"], a["d"], a["causal"],
                      a["scale"], None)


def _pre(L, **kw):
    a = dict(q=A, k=A, v=A, dO=A, lse=A, D=A, acc=A, B=1, H=1, N=128, d=64, causal=0,
             scale=0.125)
    a.update(kw)
    return L.attn_bwd_preprocess(a["q"], a["k"], a["v"], a["dO"], a["lse"], a["D"], a["acc"],
                                 a["B"], a["H"], a["N"], a["d"], a["causal"], a["scale"], None)


def test_forward_argument_errors(L):
    assert _fwd(L, q=None) == 1
    assert _fwd(L, lse=None) == 1
    assert _fwd(L, B=0) == 1
    assert _fwd(L, N=0) == 1
    assert _fwd(L, N=(1 << 24) + 1) == 1
    assert _fwd(L, N=(1 << 24) - 255) == 1     # one 256-row block past the grid limit
    assert _fwd(L, d=32) == 2
    assert _fwd(L, d=96) == 2
    assert _fwd(L, d=256) == 2
    assert _fwd(L, scale=0.0) == 1
    assert _fwd(L, scale=-1.0) == 1
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, v=A + 8) == 3
    assert _fwd(L, lse=A + 4) == 3
    assert L.attn_fwd_f16(None, A, A, A, A, 1, 1, 1, 64, 0, 1.0, None) == 1


def test_training_entry_point_argument_errors(L):
    args = (A, A, A, A, A, A, 1, 1, 128, 64, 0, 0.125, None)
    assert L.attn_fwd_train(*args) in (4, 0)  # valid arguments: no device here
    bad = list(args); bad[4] = None
    assert L.attn_fwd_train(*bad) == 1          # o32 is required
    bad = list(args); bad[4] = A + 4
    assert L.attn_fwd_train(*bad) == 3
    assert L.attn_bwd_preprocess_o32(None, A, A, A, 1, 1, 128, 64, None) == 1
    assert L.attn_bwd_preprocess_o32(A, A, A, A, 1, 1, 128, 80, None) == 2
    assert L.attn_bwd_preprocess_o32(A + 8, A, A, A, 1, 1, 128, 64, None) == 3


def test_backward_argument_errors(L):
    assert _bwd(L, dq=None) == 1
    assert _bwd(L, acc=None) == 1
    assert _bwd(L, H=0) == 1
    assert _bwd(L, d=80) == 2
    assert _bwd(L, scale=0.0) == 1
    assert _bwd(L, dk=A + 2) == 3
    assert _bwd(L, D=A + 8) == 3
    assert _pre(L, lse=None) == 1
    assert _pre(L, d=48) == 2
    assert _pre(L, dO=A + 8) == 3
    assert _pre(L, scale=-2.0) == 1
    assert _pre(L, N=0) == 1
    assert L.attn_selftest_timeout(0, None) == 1
    assert L.attn_selftest_timeout(2000000, None) == 1


def test_no_device_is_reported_not_faked(L):
    """Without an sm_103 device a valid call reports UNSUPPORTED_DEVICE; there
    is no CPU fallback."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(L) == 4
    assert _bwd(L) == 4
    assert _pre(L) == 4
    with pytest.raises(attn.AttnError):
        attn.attn_fwd(A, A, A, A, A, 1, 1, 128, 64, False, 0.125, None)


def test_torch_wrapper_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.forward(q, q, q)
    with pytest.raises(ValueError):
        attn.forward(q.float(), q.float(), q.float())


def _imports(path):
    tree = ast.parse(open(path).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            mods.add(node.module.split(".")[0])
    return mods


def test_product_and_oracle_are_independent():
    for p in glob.glob(os.path.join(ROOT, "io_aware_exact_gb300", "*.py")):
        assert "oracle" not in _imports(p), p
    for p in glob.glob(os.path.join(ROOT, "io_aware_exact_gb300", "csrc", "*")):
        assert "oracle" not in open(p).read().lower(), p
    for p in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "io_aware_exact_gb300" not in _imports(p), p
    assert "attn" not in open(os.path.join(ROOT, "oracle", "attn_oracle.c")).read().split(
        "#include")[1].split("\n")[0]


def test_library_allocates_nothing():
    """The CUDA sources never call an allocator: every buffer is the caller's."""
    for p in glob.glob(os.path.join(ROOT, "io_aware_exact_gb300", "csrc", "*")):
        text = open(p).read()
        for bad in (r"\bcudaMalloc", r"\bcudaFree", r"\bcuMemAlloc", r"\bmalloc\s*\(",
                    r"=\s*new\b", r"\bcudaMallocAsync"):
            assert not re.search(bad, text), (p, bad)


def test_grouped_entry_point_argument_errors(L):
    """H must be a positive multiple of Hkv; checked before any device call."""
    fwd = lambda H, Hkv: L.attn_fwd_gqa(A, A, A, A, A, 1, H, Hkv, 128, 64, 1, 0.125, None)
    assert fwd(4, 2) in (4, 0)            # valid arguments: no device here
    assert fwd(3, 2) == 1
    assert fwd(4, 0) == 1
    assert fwd(2, 4) == 1
    assert L.attn_fwd_train_gqa(A, A, A, A, A, A, 1, 4, 3, 128, 64, 1, 0.125, None) == 1
    assert L.attn_fwd_train_gqa(A, A, A, A, None, A, 1, 4, 2, 128, 64, 1, 0.125, None) == 1
    assert L.attn_bwd_preprocess_gqa(A, A, A, A, A, A, A, 1, 6, 4, 128, 64, 1, 0.125, None) == 1
    assert L.attn_bwd_gqa(A, A, A, A, A, A, A, A, A, A, 1, 6, 4, 128, 64, 1, 0.125, None) == 1
    assert L.attn_bwd_gqa(A, A, A, A, A, A, A, A, A, A, 1, 6, 3, 128, 80, 1, 0.125, None) == 2


def test_block_sparse_argument_errors(L):
    """Mask arguments are checked on the host before anything is enqueued."""
    def fwd(mask=A, stride=0, N=1000, o32=None, **kw):
        a = dict(B=1, H=2, d=64, causal=1, scale=0.125)
        a.update(kw)
        if o32 is None:
            return L.attn_fwd_bsparse(A, A, A, A, A, mask, stride, a["B"], a["H"], N, a["d"],
                                      a["causal"], a["scale"], None)
        return L.attn_fwd_train_bsparse(A, A, A, A, o32, A, mask, stride, a["B"], a["H"], N,
                                        a["d"], a["causal"], a["scale"], None)

    def bwd(mask=A, stride=0, N=1000):
        return L.attn_bwd_bsparse(A, A, A, A, A, A, A, A, A, A, mask, stride, 1, 2, N, 64, 1,
                                  0.125, None)

    nb = (1000 + 127) // 128
    assert fwd() in (0, 4)                       # valid: no device here
    assert fwd(stride=nb * nb) in (0, 4)
    assert fwd(mask=None) == 1
    assert fwd(stride=-1) == 1
    assert fwd(stride=nb * nb - 1) == 1          # per-head masks would overlap
    assert fwd(N=384 * 128) in (0, 4)
    assert fwd(N=384 * 128 + 1) == 1             # beyond the shared-memory tile list
    assert fwd(d=96) == 2
    assert fwd(o32=None, scale=0.0) == 1
    assert fwd(o32=0) == 1                       # the training variant needs o32
    assert fwd(o32=A + 4) == 3
    assert bwd() in (0, 4)
    assert bwd(mask=None) == 1
    assert bwd(stride=5) == 1
    assert bwd(N=50000) == 1
    assert L.attn_bwd_bsparse_f16(A, A, A, A, A, A, A, A, A, None, A, 0, 1, 2, 1000, 64, 1,
                                  0.125, None) == 1


def test_combine_entry_points_argument_errors(L):
    """attn_merge / attn_convert / attn_bwd_acc check their arguments on the host."""
    assert L.attn_merge(A, A, A, A, None, 100, 128, None) in (0, 4)
    assert L.attn_merge(A, A, A, A, A, 100, 64, None) in (0, 4)
    assert L.attn_merge(None, A, A, A, None, 100, 128, None) == 1
    assert L.attn_merge(A, A, A, None, None, 100, 128, None) == 1
    assert L.attn_merge(A, A, A, A, None, -1, 128, None) == 1
    assert L.attn_merge(A, A, A, A, None, 100, 96, None) == 2
    assert L.attn_merge(A + 4, A, A, A, None, 100, 128, None) == 3
    assert L.attn_merge_f16(A, A, A, A, A + 8, 100, 128, None) == 3
    bwd = lambda **kw: L.attn_bwd_acc(*[kw.get(n, A) for n in ("q", "k", "v", "dO", "lse", "D",
                                                                 "acc", "dq", "dk32", "dv32")],
                                      kw.get("accumulate", 0), 1, 4, kw.get("Hkv", 2), 256, 128,
                                      1, 0.1, None)
    assert bwd() in (0, 4)
    assert bwd(accumulate=1, Hkv=4) in (0, 4)
    assert bwd(dk32=None) == 1
    assert bwd(dv32=None) == 1
    assert bwd(dv32=A + 4) == 3
    assert bwd(Hkv=3) == 1                                 # H not a multiple of Hkv
    assert bwd(dq=None) == 1
    assert L.attn_convert(A, A, 64, 1.0, None) in (0, 4)
    assert L.attn_convert(A, A, 12, 1.0, None) == 1       # not a multiple of 8
    assert L.attn_convert(A, A, 64, float("nan"), None) == 1
    assert L.attn_convert_f16(A, None, 64, 1.0, None) == 1


def test_dropout_argument_errors(L):
    def fwd(p=0.1, o32=A, **kw):
        return L.attn_fwd_train_dropout(A, A, A, A, o32, A, p, 123, 4, 1, 2, kw.get("N", 256),
                                        kw.get("d", 64), 1, 0.125, None)

    def bwd(p=0.1, dk=A):
        return L.attn_bwd_dropout(A, A, A, A, A, A, A, A, dk, A, p, 123, 4, 1, 2, 256, 64, 1,
                                  0.125, None)

    assert fwd() in (0, 4) and fwd(p=0.0) in (0, 4) and bwd() in (0, 4)
    for bad in (1.0, 1.5, -0.1, float("nan"), float("inf")):
        assert fwd(p=bad) == 1 and bwd(p=bad) == 1
    assert fwd(o32=None) == 1
    assert fwd(d=96) == 2
    assert bwd(dk=None) == 1
    assert bwd(dk=A + 2) == 3


def test_group_split_argument_errors(L):
    def split(part=A, splits=2, H=8, Hkv=2):
        return L.attn_bwd_gqa_split(A, A, A, A, A, A, A, A, A, A, part, splits, 1, H, Hkv, 256, 64,
                                    1, 0.125, None)

    assert split() in (0, 4) and split(splits=4) in (0, 4) and split(splits=1) in (0, 4)
    assert split(splits=3) == 1                 # 3 does not divide the group of 4
    assert split(splits=0) == 1
    assert split(part=None) == 1
    assert split(part=A + 4) == 3
    assert split(Hkv=3) == 1


def test_header_is_plain_c_and_the_library_links_from_c(L, tmp_path):
    """include/attn.h compiles as C99 with warnings as errors, and a C program
    links against the library and calls it (no device work: an argument error
    is reported on the host)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(
        '#include <stdio.h>\n#include "attn.h"\n'
        "int main(void) {\n"
        '    printf("%s|%s\\n", attn_version(), attn_status_string(ATTN_ERR_TIMEOUT));\n'
        "    return attn_fwd(0, 0, 0, 0, 0, 1, 1, 128, 64, 0, 0.125f, 0) == ATTN_ERR_INVALID_ARG"
        " ? 0 : 1;\n}\n")
    libdir = os.path.dirname(attn.LIB_PATH)
    exe = tmp_path / "abi"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lattn_gb300",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("io_aware_exact_gb300") and "bounded wait" in r.stdout


def test_binding_declares_every_entry_point(L):
    """Every function of include/attn.h has ctypes argument and result types in
    the binding, so no pointer or 64-bit argument is passed as a C int."""
    for n in attn.header_functions():
        f = getattr(L, n)
        assert f.argtypes is not None, n
        assert f.restype in (ctypes.c_int, ctypes.c_char_p), n
