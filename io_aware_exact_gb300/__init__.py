"""GB300-native exact IO-aware attention.

The compute lives in ``libattn_gb300.so`` (CUDA, sm_103a; C ABI declared in
``include/attn.h``).  This package is a thin ctypes binding:

* ``attn_fwd``, ``attn_bwd_preprocess``, ``attn_bwd`` (and ``*_f16``) take
  raw device pointers (ints), sizes and a ``cudaStream_t`` (int) exactly like
  the C functions, and raise :class:`AttnError` on a non-zero status;
* ``forward`` / ``backward`` / :class:`AttnFunction` marshal PyTorch CUDA
  tensors (which own all memory) into those calls.

There is no CPU or PyTorch fallback: if the library is missing or the device
is not an sm_103 GPU, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "attn.h")

_lib = None
_lock = threading.Lock()

STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED_HEAD_DIM",
    3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_UNSUPPORTED_DEVICE", 5: "ATTN_ERR_LAUNCH",
    6: "ATTN_ERR_TIMEOUT", 7: "ATTN_ERR_DEVICE_FAULT",
}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d: %s)" % (where, STATUS.get(status, "?"), status,
                                                     status_string(status) if _lib else ""))


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libattn_gb300.so is missing: build it with "
                                   "`python -m io_aware_exact_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            fwd = [P, P, P, P, P, I, I, I, I, I, F, P]
            pre = [P, P, P, P, P, P, P, I, I, I, I, I, F, P]
            bwd = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
            fwdt = [P, P, P, P, P, P, I, I, I, I, I, F, P]
            pre32 = [P, P, P, P, I, I, I, I, P]
            for name, at in (("attn_fwd", fwd), ("attn_fwd_f16", fwd),
                             ("attn_fwd_train", fwdt), ("attn_fwd_train_f16", fwdt),
                             ("attn_bwd_preprocess", pre), ("attn_bwd_preprocess_f16", pre),
                             ("attn_bwd_preprocess_o32", pre32),
                             ("attn_bwd_preprocess_o32_f16", pre32),
                             ("attn_bwd", bwd), ("attn_bwd_f16", bwd)):
                fn = getattr(L, name)
                fn.argtypes = at
                fn.restype = I
            # grouped K / V heads: one more int (Hkv) after H
            for name, at in (("attn_fwd_gqa", fwd), ("attn_fwd_gqa_f16", fwd),
                             ("attn_fwd_train_gqa", fwdt), ("attn_fwd_train_gqa_f16", fwdt),
                             ("attn_bwd_preprocess_gqa", pre),
                             ("attn_bwd_preprocess_gqa_f16", pre),
                             ("attn_bwd_gqa", bwd), ("attn_bwd_gqa_f16", bwd)):
                fn = getattr(L, name)
                h = at.index(I) + 2          # position of H is the second int (B, H, ...)
                fn.argtypes = at[:h] + [I] + at[h:]
                fn.restype = I
            # packed variable-length batches
            vfwd = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
            vfwdt = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
            vpre = [P, P, P, P, I, I, I, P]
            vbwd = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
            for name, at in (("attn_fwd_varlen", vfwd), ("attn_fwd_varlen_f16", vfwd),
                             ("attn_fwd_train_varlen", vfwdt), ("attn_fwd_train_varlen_f16", vfwdt),
                             ("attn_bwd_preprocess_o32_varlen", vpre),
                             ("attn_bwd_preprocess_o32_varlen_f16", vpre),
                             ("attn_bwd_varlen", vbwd), ("attn_bwd_varlen_f16", vbwd)):
                fn = getattr(L, name)
                fn.argtypes = at
                fn.restype = I
            # keys of their own lengths: (cu_seqlens_q, cu_seqlens_k, B, total_q, total_k,
            # max_seqlen_q, max_seqlen_k, H, Hkv, d, causal, scale, stream)
            kvt = [P, P, I, I, I, I, I, I, I, I, I, F, P]
            for name, at in (("attn_fwd_varlen_qk", [P] * 5 + kvt),
                             ("attn_fwd_varlen_qk_f16", [P] * 5 + kvt),
                             ("attn_fwd_train_varlen_qk", [P] * 6 + kvt),
                             ("attn_fwd_train_varlen_qk_f16", [P] * 6 + kvt),
                             ("attn_bwd_varlen_qk", [P] * 10 + kvt),
                             ("attn_bwd_varlen_qk_f16", [P] * 10 + kvt)):
                fn = getattr(L, name)
                fn.argtypes = at
                fn.restype = I
            # block-sparse layouts: (block_mask, mask_head_stride) before B
            LL = ctypes.c_longlong
            sfwd = [P, P, P, P, P, P, LL, I, I, I, I, I, F, P]
            sfwdt = [P, P, P, P, P, P, P, LL, I, I, I, I, I, F, P]
            sbwd = [P, P, P, P, P, P, P, P, P, P, P, LL, I, I, I, I, I, F, P]
            for name, at in (("attn_fwd_bsparse", sfwd), ("attn_fwd_bsparse_f16", sfwd),
                             ("attn_fwd_train_bsparse", sfwdt),
                             ("attn_fwd_train_bsparse_f16", sfwdt),
                             ("attn_bwd_bsparse", sbwd), ("attn_bwd_bsparse_f16", sbwd)):
                fn = getattr(L, name)
                fn.argtypes = at
                fn.restype = I
            # combining partial results
            for name in ("attn_merge", "attn_merge_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, P, P, LL, I, P]
                fn.restype = I
            for name in ("attn_bwd_acc", "attn_bwd_acc_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
                fn.restype = I
            for name in ("attn_convert", "attn_convert_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, LL, F, P]
                fn.restype = I
            # dropout: (p_drop, seed, offset) before B
            U64, U32 = ctypes.c_ulonglong, ctypes.c_uint
            for name in ("attn_fwd_train_dropout", "attn_fwd_train_dropout_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, P, P, P, F, U64, U32, I, I, I, I, I, F, P]
                fn.restype = I
            for name in ("attn_bwd_dropout", "attn_bwd_dropout_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, P, P, P, P, P, P, P, F, U64, U32, I, I, I, I, I, F, P]
                fn.restype = I
            for name in ("attn_bwd_gqa_split", "attn_bwd_gqa_split_f16"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
                fn.restype = I
            L.attn_gqa_split_hint.argtypes = [I, I, I, I, I]
            L.attn_gqa_split_hint.restype = I
            L.attn_status_string.argtypes = [I]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_get_device_status.argtypes = [P]
            L.attn_get_device_status.restype = I
            L.attn_selftest_timeout.argtypes = [I, P]
            L.attn_selftest_timeout.restype = I
            L.attn_version.argtypes = []
            L.attn_version.restype = ctypes.c_char_p
            L.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
            L.attn_bwd_noalloc.restype = I
            _lib = L
    return _lib


def header_functions():
    """Names of the functions declared in include/attn.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(attn_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def version() -> str:
    return lib().attn_version().decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise AttnError(rc, where)


# ---------------------------------------------------------------------------
# Raw C-ABI calls (pointers as ints)
# ---------------------------------------------------------------------------

def _heads(name, f16, H, Hkv):
    """The entry point for (dtype, grouping) and the head arguments it takes."""
    grouped = Hkv is not None and Hkv != H
    fn = getattr(lib(), name + ("_gqa" if grouped else "") + ("_f16" if f16 else ""))
    return fn, ((H, Hkv) if grouped else (H,))


def attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stream, f16=False, Hkv=None):
    fn, hs = _heads("attn_fwd", f16, H, Hkv)
    _check(fn(q, k, v, o, lse, B, *hs, N, d, int(bool(causal)), float(scale), stream),
           "attn_fwd")


def attn_fwd_train(q, k, v, o, o32, lse, B, H, N, d, causal, scale, stream, f16=False,
                   Hkv=None):
    fn, hs = _heads("attn_fwd_train", f16, H, Hkv)
    _check(fn(q, k, v, o, o32, lse, B, *hs, N, d, int(bool(causal)), float(scale), stream),
           "attn_fwd_train")


def attn_bwd_preprocess_o32(o32, dO, D, dq_accum, B, H, N, d, stream, f16=False):
    fn = lib().attn_bwd_preprocess_o32_f16 if f16 else lib().attn_bwd_preprocess_o32
    _check(fn(o32, dO, D, dq_accum, B, H, N, d, stream), "attn_bwd_preprocess_o32")


def attn_bwd_preprocess(q, k, v, dO, lse, D, dq_accum, B, H, N, d, causal, scale, stream,
                        f16=False, Hkv=None):
    fn, hs = _heads("attn_bwd_preprocess", f16, H, Hkv)
    _check(fn(q, k, v, dO, lse, D, dq_accum, B, *hs, N, d, int(bool(causal)), float(scale),
              stream), "attn_bwd_preprocess")


def attn_bwd(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, N, d, causal, scale, stream,
             f16=False, Hkv=None):
    fn, hs = _heads("attn_bwd", f16, H, Hkv)
    _check(fn(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, *hs, N, d, int(bool(causal)),
              float(scale), stream), "attn_bwd")


def attn_fwd_bsparse(q, k, v, o, lse, block_mask, mask_head_stride, B, H, N, d, causal, scale,
                     stream, f16=False, o32=None):
    """Block-sparse forward; with ``o32`` the training variant (also writes O in fp32)."""
    if o32 is None:
        fn = lib().attn_fwd_bsparse_f16 if f16 else lib().attn_fwd_bsparse
        _check(fn(q, k, v, o, lse, block_mask, int(mask_head_stride), B, H, N, d,
                  int(bool(causal)), float(scale), stream), "attn_fwd_bsparse")
    else:
        fn = lib().attn_fwd_train_bsparse_f16 if f16 else lib().attn_fwd_train_bsparse
        _check(fn(q, k, v, o, o32, lse, block_mask, int(mask_head_stride), B, H, N, d,
                  int(bool(causal)), float(scale), stream), "attn_fwd_train_bsparse")


def attn_bwd_bsparse(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, block_mask, mask_head_stride,
                     B, H, N, d, causal, scale, stream, f16=False):
    fn = lib().attn_bwd_bsparse_f16 if f16 else lib().attn_bwd_bsparse
    _check(fn(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, block_mask, int(mask_head_stride),
              B, H, N, d, int(bool(causal)), float(scale), stream), "attn_bwd_bsparse")


def attn_get_device_status(stream=None) -> int:
    return int(lib().attn_get_device_status(stream))


def attn_selftest_timeout(timeout_us: int, stream=None):
    _check(lib().attn_selftest_timeout(int(timeout_us), stream), "attn_selftest_timeout")


# ---------------------------------------------------------------------------
# PyTorch tensor marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_qkv(*ts):
    torch = _torch()
    t0 = ts[0]
    if t0.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    if t0.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("expected bfloat16 or float16 tensors")
    for t in ts:
        if t.shape != t0.shape or t.dtype != t0.dtype:
            raise ValueError("q, k, v (and o, dO) must share shape and dtype")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    return t0.shape, t0.dtype == torch.float16


def _check_grouped(q, k, v, *qlike):
    """Shapes for q (and dO) [B,H,N,d] with k, v [B,Hkv,N,d], H a multiple of Hkv."""
    (B, H, N, d), f16 = _check_qkv(q, *qlike)
    _check_qkv(k, v)
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, Nk, dk) != (B, N, d) or k.dtype != q.dtype or Hkv < 1 or H % Hkv != 0:
        raise ValueError("k, v must be [B, Hkv, N, d] like q with H a multiple of Hkv")
    return (B, H, Hkv, N, d), f16


def forward(q, k, v, causal: bool = False, scale=None, o=None, lse=None, stream=None,
            o32=None):
    """O, lse for [B,H,N,d] CUDA tensors (outputs allocated by torch if not given).

    k and v may have fewer heads than q ([B,Hkv,N,d], H a multiple of Hkv):
    groups of H / Hkv query heads then share one K / V head.  With ``o32``
    (an fp32 [B,H,N,d] tensor, or True to allocate one) the training forward
    also writes O in fp32 and returns (o, lse, o32).
    """
    torch = _torch()
    (B, H, Hkv, N, d), f16 = _check_grouped(q, k, v)
    scale = d ** -0.5 if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if o32 is None:
        attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                 B, H, N, d, causal, scale, _stream_handle(stream), f16, Hkv)
        return o, lse
    if o32 is True:
        o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    attn_fwd_train(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o32.data_ptr(),
                   lse.data_ptr(), B, H, N, d, causal, scale, _stream_handle(stream), f16, Hkv)
    return o, lse, o32


def backward(q, k, v, o, lse, dO, causal: bool = False, scale=None, dq=None, dk=None, dv=None,
             D=None, dq_accum=None, stream=None, o32=None, splits=None):
    """dQ, dK, dV for [B,H,N,d] CUDA tensors (workspace allocated by torch if not given).

    With ``o32`` (the fp32 O of the training forward) D comes from
    rowsum(dO o O); otherwise the preprocess recomputes it from q, k, v, dO
    and lse.  ``o`` (the 16-bit forward output) is not read and may be None.
    With grouped K / V heads, dk and dv are [B,Hkv,N,d], summed over each group;
    ``splits`` query-head shares per group run on separate CTAs (default: the
    library's hint for this device and shape).
    """
    torch = _torch()
    (B, H, Hkv, N, d), f16 = _check_grouped(q, k, v, dO)
    scale = d ** -0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    D = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if D is None else D
    if dq_accum is None:
        dq_accum = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    if o32 is not None:
        attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), dq_accum.data_ptr(),
                                B, H, N, d, s, f16)
    else:
        attn_bwd_preprocess(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(),
                            lse.data_ptr(), D.data_ptr(), dq_accum.data_ptr(), B, H, N, d,
                            causal, scale, s, f16, Hkv)
    if splits is None:
        splits = int(lib().attn_gqa_split_hint(B, H, Hkv, N, int(bool(causal)))) if Hkv != H else 1
    if splits > 1:
        # grouped heads split over CTAs: fp32 shares of dK, dV, summed at the end
        part = torch.empty((2, splits, B, Hkv, N, d), dtype=torch.float32, device=q.device)
        fn = lib().attn_bwd_gqa_split_f16 if f16 else lib().attn_bwd_gqa_split
        _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                  D.data_ptr(), dq_accum.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                  part.data_ptr(), splits, B, H, Hkv, N, d, int(bool(causal)), scale, s),
               "attn_bwd_gqa_split")
        return dq, dk, dv
    attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
             D.data_ptr(), dq_accum.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
             B, H, N, d, causal, scale, s, f16, Hkv)
    return dq, dk, dv


def _block_mask_arg(block_mask, B, H, N):
    """(pointer, per-head stride) of a uint8 CUDA block mask [Nb, Nb] (one mask
    for every head) or [B, H, Nb, Nb], Nb = ceil(N / 128)."""
    torch = _torch()
    nb = (N + 127) // 128
    if block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous():
        raise ValueError("block_mask must be a contiguous uint8 CUDA tensor")
    if tuple(block_mask.shape) == (nb, nb):
        return block_mask.data_ptr(), 0
    if tuple(block_mask.shape) == (B, H, nb, nb):
        return block_mask.data_ptr(), nb * nb
    raise ValueError("block_mask must be [Nb, Nb] or [B, H, Nb, Nb] with Nb = ceil(N / 128)")


def forward_bsparse(q, k, v, block_mask, causal: bool = False, scale=None, o=None, lse=None,
                    o32=None, stream=None):
    """Block-sparse forward over [B,H,N,d] tensors: 128 x 128 tiles whose
    block_mask byte is zero are dropped.  With ``o32`` (fp32 [B,H,N,d], or True)
    the training variant, returning (o, lse, o32); else (o, lse)."""
    torch = _torch()
    (B, H, N, d), f16 = _check_qkv(q, k, v)
    scale = d ** -0.5 if scale is None else float(scale)
    mp, ms = _block_mask_arg(block_mask, B, H, N)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if o32 is True:
        o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    attn_fwd_bsparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), mp,
                     ms, B, H, N, d, causal, scale, _stream_handle(stream), f16,
                     None if o32 is None else o32.data_ptr())
    return (o, lse) if o32 is None else (o, lse, o32)


def backward_bsparse(q, k, v, o32, lse, dO, block_mask, causal: bool = False, scale=None,
                     dq=None, dk=None, dv=None, D=None, dq_accum=None, stream=None):
    """dQ, dK, dV of the block-sparse forward: D from the fp32 O of
    forward_bsparse(..., o32=True), then the backward over the kept tiles."""
    torch = _torch()
    (B, H, N, d), f16 = _check_qkv(q, k, v, dO)
    scale = d ** -0.5 if scale is None else float(scale)
    mp, ms = _block_mask_arg(block_mask, B, H, N)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    D = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if D is None else D
    if dq_accum is None:
        dq_accum = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), dq_accum.data_ptr(),
                            B, H, N, d, s, f16)
    attn_bwd_bsparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                     D.data_ptr(), dq_accum.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                     dv.data_ptr(), mp, ms, B, H, N, d, causal, scale, s, f16)
    return dq, dk, dv


def merge(o_acc, lse_acc, o_part, lse_part, o_out=None, stream=None):
    """Merge a partial result (fp32 O [..., d] normalised over its keys, lse
    [...]) into a running one, in place; optionally also write the merged O
    rounded to o_out's 16-bit dtype."""
    torch = _torch()
    d = o_acc.shape[-1]
    rows = lse_acc.numel()
    for t in (o_acc, lse_acc, o_part, lse_part):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("merge takes contiguous fp32 CUDA tensors")
    if o_part.shape != o_acc.shape or lse_part.numel() != rows or o_acc.numel() != rows * d:
        raise ValueError("merge: shapes of the two partial results differ")
    f16 = o_out is not None and o_out.dtype == torch.float16
    fn = lib().attn_merge_f16 if f16 else lib().attn_merge
    _check(fn(o_acc.data_ptr(), lse_acc.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
              None if o_out is None else o_out.data_ptr(), rows, d, _stream_handle(stream)),
           "attn_merge")


def attn_bwd_acc(q, k, v, dO, lse, D, dq_accum, dq, dk32, dv32, accumulate, B, H, Hkv, N, d,
                 causal, scale, stream, f16=False):
    """Backward against one key / value chunk writing (or, with accumulate,
    adding to) fp32 dK, dV."""
    fn = lib().attn_bwd_acc_f16 if f16 else lib().attn_bwd_acc
    _check(fn(q, k, v, dO, lse, D, dq_accum, dq, dk32, dv32, int(bool(accumulate)), B, H, Hkv, N,
              d, int(bool(causal)), float(scale), stream), "attn_bwd_acc")


def convert(x, dtype, scale: float = 1.0, out=None, stream=None):
    """scale * x (fp32) rounded to a 16-bit dtype."""
    torch = _torch()
    out = torch.empty(x.shape, dtype=dtype, device=x.device) if out is None else out
    fn = lib().attn_convert_f16 if out.dtype == torch.float16 else lib().attn_convert
    _check(fn(x.data_ptr(), out.data_ptr(), x.numel(), float(scale), _stream_handle(stream)),
           "attn_convert")
    return out


def forward_dropout(q, k, v, p_drop: float, seed: int, offset: int = 0, causal: bool = False,
                    scale=None, o=None, lse=None, o32=None, stream=None):
    """Training forward with dropout on P (mask regenerated from seed, offset):
    returns (o, lse, o32) for [B,H,N,d] tensors."""
    torch = _torch()
    (B, H, N, d), f16 = _check_qkv(q, k, v)
    scale = d ** -0.5 if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device) if o32 is None else o32
    fn = lib().attn_fwd_train_dropout_f16 if f16 else lib().attn_fwd_train_dropout
    _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o32.data_ptr(),
              lse.data_ptr(), float(p_drop), int(seed), int(offset), B, H, N, d,
              int(bool(causal)), scale, _stream_handle(stream)), "attn_fwd_train_dropout")
    return o, lse, o32


def backward_dropout(q, k, v, o32, lse, dO, p_drop: float, seed: int, offset: int = 0,
                     causal: bool = False, scale=None, dq=None, dk=None, dv=None, D=None,
                     dq_accum=None, stream=None):
    """dQ, dK, dV of forward_dropout with the same p_drop, seed and offset."""
    torch = _torch()
    (B, H, N, d), f16 = _check_qkv(q, k, v, dO)
    scale = d ** -0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    D = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if D is None else D
    if dq_accum is None:
        dq_accum = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    attn_bwd_preprocess_o32(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), dq_accum.data_ptr(),
                            B, H, N, d, s, f16)
    fn = lib().attn_bwd_dropout_f16 if f16 else lib().attn_bwd_dropout
    _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
              D.data_ptr(), dq_accum.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
              float(p_drop), int(seed), int(offset), B, H, N, d, int(bool(causal)), scale, s),
           "attn_bwd_dropout")
    return dq, dk, dv


def _autograd_function():
    torch = _torch()

    class AttnFunction(torch.autograd.Function):
        """Exact attention with the library's forward and backward kernels.

        Saves q, k, v, lse and the fp32 O (O(N d) extra, no N x N buffer) and
        recomputes P in the backward, like the FlashAttention autograd
        function described on the sj-techlog page ("1. Python interface는
        scale·RNG state·작은 통계를 autograd에 넘긴다").
        """

        @staticmethod
        def forward(ctx, q, k, v, causal=False, scale=None):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            o, lse, o32 = forward(q, k, v, causal, scale, o32=True)
            ctx.save_for_backward(q, k, v, lse, o32)
            ctx.causal, ctx.scale = causal, scale
            return o

        @staticmethod
        def backward(ctx, dO):
            q, k, v, lse, o32 = ctx.saved_tensors
            dq, dk, dv = backward(q, k, v, None, lse, dO.contiguous(), ctx.causal, ctx.scale,
                                  o32=o32)
            return dq, dk, dv, None, None

    return AttnFunction


def attention(q, k, v, causal: bool = False, scale=None):
    """Differentiable exact attention over [B,H,N,d] bf16/fp16 CUDA tensors."""
    global AttnFunction
    if AttnFunction is None:
        AttnFunction = _autograd_function()
    return AttnFunction.apply(q, k, v, causal, scale)


AttnFunction = None


# ---------------------------------------------------------------------------
# Packed variable-length batches
# ---------------------------------------------------------------------------

def _check_cu(cu, B=None):
    torch = _torch()
    if cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_cuda or cu.numel() < 2:
        raise ValueError("cu_seqlens must be a CUDA int32 vector of B + 1 offsets")
    if B is not None and cu.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")


def _check_varlen(q, k, v, cu_seqlens, *qlike, own_keys=False):
    torch = _torch()
    for t in (q, k, v) + qlike:
        if t.dim() != 3 or not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("expected contiguous CUDA [total, heads, d] tensors of one dtype")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("expected bfloat16 or float16 tensors")
    total, H, d = q.shape
    if k.shape != v.shape or k.shape[2] != d or (not own_keys and k.shape[0] != total):
        raise ValueError("k, v must be [total, Hkv, d] like q (total_k rows with cu_seqlens_k)")
    for t in qlike:
        if t.shape != q.shape:
            raise ValueError("dO must be shaped like q")
    _check_cu(cu_seqlens)
    return (cu_seqlens.numel() - 1, total, H, k.shape[1], d), q.dtype == torch.float16


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale=None,
                   o=None, lse=None, o32=None, stream=None, cu_seqlens_k=None, max_seqlen_k=None):
    """O [total, H, d] and lse [B, H, max_seqlen] of a packed variable-length
    batch (sequence b is tokens cu_seqlens[b]:cu_seqlens[b+1] of q, k, v).
    With ``o32`` (True or an fp32 [total, H, d] tensor) the training forward
    also writes O in fp32 and returns (o, lse, o32).  With ``cu_seqlens_k``
    (and ``max_seqlen_k``) the keys have lengths of their own: k, v are
    [total_k, Hkv, d], sequence b's keys are rows cu_seqlens_k[b]:
    cu_seqlens_k[b+1], and the causal mask is aligned bottom-right."""
    torch = _torch()
    own = cu_seqlens_k is not None
    (B, total, H, Hkv, d), f16 = _check_varlen(q, k, v, cu_seqlens, own_keys=own)
    scale = d ** -0.5 if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, max_seqlen), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    if own:
        _check_cu(cu_seqlens_k, B)
        if max_seqlen_k is None:
            raise ValueError("max_seqlen_k is needed with cu_seqlens_k")
        args = (cu_seqlens.data_ptr(), cu_seqlens_k.data_ptr(), B, total, k.shape[0],
                int(max_seqlen), int(max_seqlen_k), H, Hkv, d, int(bool(causal)), scale, s)
        suffix = "_qk"
    else:
        args = (cu_seqlens.data_ptr(), B, total, int(max_seqlen), H, Hkv, d, int(bool(causal)),
                scale, s)
        suffix = ""
    L = lib()
    if o32 is None:
        name = "attn_fwd_varlen" + suffix
        fn = getattr(L, name + ("_f16" if f16 else ""))
        _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), *args),
               name)
        return o, lse
    if o32 is True:
        o32 = torch.empty((total, H, d), dtype=torch.float32, device=q.device)
    name = "attn_fwd_train_varlen" + suffix
    fn = getattr(L, name + ("_f16" if f16 else ""))
    _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o32.data_ptr(),
              lse.data_ptr(), *args), name)
    return o, lse, o32


def backward_varlen(q, k, v, o32, lse, dO, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale=None, dq=None, dk=None, dv=None, D=None, dq_accum=None, stream=None,
                    cu_seqlens_k=None, max_seqlen_k=None):
    """dQ, dK, dV of a packed variable-length batch, from the training
    forward's fp32 O and lse (D = rowsum(dO o O)); ``cu_seqlens_k`` and
    ``max_seqlen_k`` as for forward_varlen."""
    torch = _torch()
    own = cu_seqlens_k is not None
    (B, total, H, Hkv, d), f16 = _check_varlen(q, k, v, cu_seqlens, dO, own_keys=own)
    scale = d ** -0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    D = torch.empty((total, H), dtype=torch.float32, device=q.device) if D is None else D
    if dq_accum is None:
        dq_accum = torch.empty((total, H, d), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    L = lib()
    pre = L.attn_bwd_preprocess_o32_varlen_f16 if f16 else L.attn_bwd_preprocess_o32_varlen
    _check(pre(o32.data_ptr(), dO.data_ptr(), D.data_ptr(), dq_accum.data_ptr(), total, H, d, s),
           "attn_bwd_preprocess_o32_varlen")
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
            D.data_ptr(), dq_accum.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    if own:
        _check_cu(cu_seqlens_k, B)
        if max_seqlen_k is None:
            raise ValueError("max_seqlen_k is needed with cu_seqlens_k")
        fn = L.attn_bwd_varlen_qk_f16 if f16 else L.attn_bwd_varlen_qk
        _check(fn(*ptrs, cu_seqlens.data_ptr(), cu_seqlens_k.data_ptr(), B, total, k.shape[0],
                  int(max_seqlen), int(max_seqlen_k), H, Hkv, d, int(bool(causal)), scale, s),
               "attn_bwd_varlen_qk")
        return dq, dk, dv
    fn = L.attn_bwd_varlen_f16 if f16 else L.attn_bwd_varlen
    _check(fn(*ptrs, cu_seqlens.data_ptr(), B, total, int(max_seqlen), H, Hkv, d,
              int(bool(causal)), scale, s), "attn_bwd_varlen")
    return dq, dk, dv
