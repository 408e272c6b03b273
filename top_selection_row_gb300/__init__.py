"""Exact top-k / top-p candidate-set selection on GB300 (Python binding).

Thin wrappers over the C ABI of ``libqrita.so`` (include/qrita.h) with the
same names. They only marshal arguments: every step of the selection runs in
the library's CUDA kernel. PyTorch provides device memory and streams.
"""

from __future__ import annotations

import ctypes

import numpy as np

from ._lib import EXPORTED, lib  # noqa: F401

DTYPE_F32 = 0
DTYPE_BF16 = 1

OK, EINVAL, EUNSUPPORTED, ECUDA = 0, 1, 2, 3
ROW_OK, ROW_NONFINITE, ROW_SEARCH_CAP, ROW_TIMEOUT = 0, 1, 2, 3

FLAG_NO_TRUNCATION = 0x1
FLAG_FORCE_FALLBACK = 0x2
FLAG_KEY_PIVOTS = 0x4
FLAG_FORCE_RETRY = 0x8
FLAG_HIST_MISS = 0x10
FLAG_CLUSTER_SET = 0x800
FLAG_TEST_GIVE_UP = 0x1000
FLAG_NO_KEY_HIST = 0x2000
FLAG_SEARCH_QUATERNARY = 0x4000
FLAG_SEARCH_BINARY = 0x8000


def flag_cluster(n_ctas: int) -> int:
    """Flags that force ``n_ctas`` (1, 2, 4, 8 or 16) CTAs per row."""
    shift = {1: 0, 2: 1, 4: 2, 8: 3, 16: 4}[n_ctas]
    return FLAG_CLUSTER_SET | (shift << 8)


PATH_TOPK, PATH_TOPP, PATH_TRUNC, PATH_HIT = 0x1, 0x2, 0x4, 0x8
PATH_FALLBACK, PATH_OVERFLOW, PATH_KEEP_ALL, PATH_RETRY = 0x10, 0x20, 0x40, 0x80
PATH_HIST = 0x100
PATH_SAMPLE_T = 0x200
PATH_KEYHIST = 0x400

# Layout of qrita_row_info_t (64 bytes).
ROW_INFO_DTYPE = np.dtype(
    [
        ("mu", "<f4"),
        ("sigma", "<f4"),
        ("threshold", "<f4"),
        ("row_max", "<f4"),
        ("survivors", "<u4"),
        ("path", "<u4"),
        ("rounds_k", "<u4"),
        ("rounds_p", "<u4"),
        ("boundary", "<f4"),
        ("n_boundary", "<u4"),
        ("kept", "<u4"),
        ("status", "<u4"),
        ("z", "<f8"),
        ("passes", "<u4"),
        ("reserved", "<u4"),
    ]
)
assert ROW_INFO_DTYPE.itemsize == 64


class QritaError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"qrita error {code}: {strerror(code)}")


def strerror(code: int) -> str:
    return lib().qrita_strerror(int(code)).decode()


def version() -> int:
    return int(lib().qrita_version())


def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _check_rows(logits):
    if logits.dim() != 2:
        raise ValueError("logits must be [B, V]")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (use qrita_select_host for host buffers)")
    B, V = logits.shape
    if B > 0 and (logits.stride(1) != 1 or (B > 1 and logits.stride(0) != V)):
        raise ValueError("logits must be row-major with leading dimension V")
    return B, V


def _vec(t, n, dtype, name, device):
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(t)
    if t.dtype != dtype or t.device != device or not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of {n} elements on {device}")
    return t


def _stream_ptr(device, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def qrita_select(logits, k=None, p=None, out=None, stream=None):
    """Keep-mask of the exact top-k / top-p candidate set of every row.

    logits: CUDA tensor [B, V], float32 or bfloat16, row-major.
    k: CUDA int32 [B] or None (top-k off); p: CUDA float32 [B] or None.
    out: optional CUDA bool/uint8 tensor [B, V]. Returns the mask (bool).
    The kernel is enqueued on ``stream`` (default: the current stream).
    """
    return qrita_select_ex(logits, k, p, out=out, stream=stream)[0]


def qrita_select_ex(logits, k=None, p=None, out=None, stream=None, flags=0,
                    row_status=False, row_info=False):
    """qrita_select plus path flags, per-row status and per-row diagnostics.

    Returns (mask, status or None, info or None); ``status`` is a CUDA int32
    [B] tensor, ``info`` a CUDA uint8 [B, 64] tensor holding
    qrita_row_info_t records (decode with :func:`decode_row_info`).
    """
    torch = _torch()
    B, V = _check_rows(logits)
    dev = logits.device
    dt = _dtype_code(logits)
    kk = _vec(k, B, torch.int32, "k", dev)
    pp = _vec(p, B, torch.float32, "p", dev)
    if out is None:
        out = torch.empty((B, V), dtype=torch.bool, device=dev)
    elif out.shape != (B, V) or out.dtype not in (torch.bool, torch.uint8) or out.device != dev or not out.is_contiguous():
        raise ValueError("out must be a contiguous bool/uint8 [B, V] tensor on the logits' device")
    st = torch.empty(B, dtype=torch.int32, device=dev) if row_status else None
    info = torch.empty((B, 64), dtype=torch.uint8, device=dev) if row_info else None
    rc = lib().qrita_select_ex(
        ctypes.c_void_p(logits.data_ptr() if B else 0),
        dt,
        B,
        V,
        ctypes.c_void_p(kk.data_ptr() if kk is not None else 0),
        ctypes.c_void_p(pp.data_ptr() if pp is not None else 0),
        ctypes.c_void_p(out.data_ptr() if B else 0),
        _stream_ptr(dev, stream),
        ctypes.c_uint32(flags),
        ctypes.c_void_p(st.data_ptr() if st is not None else 0),
        ctypes.c_void_p(info.data_ptr() if info is not None else 0),
    )
    if rc != OK:
        raise QritaError(rc)
    return out, st, info


def decode_row_info(info) -> np.ndarray:
    """qrita_row_info_t records (CUDA uint8 [B, 64]) as a numpy structured array."""
    raw = info.detach().cpu().numpy()
    return np.ascontiguousarray(raw).view(ROW_INFO_DTYPE).reshape(-1)


def qrita_topk_ids(logits, k, kmax, out_mask=None, out_ids=None, stream=None):
    """Top-k ids of every row in stable order (logit descending, lower id
    first among equals) through qrita_topk_ids.

    logits: CUDA [B, V] float32 / bfloat16; k: CUDA int32 [B]; kmax: 1..8192.
    Returns (ids int32 [B, kmax], padded with -1; mask bool [B, V]).
    """
    torch = _torch()
    B, V = _check_rows(logits)
    dev = logits.device
    kk = _vec(k, B, torch.int32, "k", dev)
    if kk is None:
        raise ValueError("k is required")
    if out_mask is None:
        out_mask = torch.empty((B, V), dtype=torch.bool, device=dev)
    if out_ids is None:
        out_ids = torch.empty((B, int(kmax)), dtype=torch.int32, device=dev)
    elif out_ids.shape != (B, int(kmax)) or out_ids.dtype != torch.int32 or not out_ids.is_contiguous():
        raise ValueError("out_ids must be a contiguous int32 [B, kmax] tensor")
    rc = lib().qrita_topk_ids(
        ctypes.c_void_p(logits.data_ptr() if B else 0), _dtype_code(logits), B, V,
        ctypes.c_void_p(kk.data_ptr()), int(kmax), ctypes.c_void_p(out_mask.data_ptr() if B else 0),
        ctypes.c_void_p(out_ids.data_ptr() if B else 0), _stream_ptr(dev, stream))
    if rc != OK:
        raise QritaError(rc)
    return out_ids, out_mask


def qrita_candidates(logits, mask, cap, u=None, stream=None, out=None):
    """Kept ids in id order with probabilities renormalised over the kept set,
    the kept count, and (with u: CUDA float32 [B]) one token drawn per row,
    through qrita_candidates. Returns (ids [B, cap], probs [B, cap], count [B],
    sample [B] or None). Without ``out`` the entries past a row's count are
    -1 / 0; ``out`` = (ids, probs, count, sample) reuses the caller's buffers
    (contiguous int32 [B, cap], float32 [B, cap], int32 [B], int32 [B] or
    None exactly when u is), whose entries past a row's count are left as
    they were."""
    torch = _torch()
    B, V = _check_rows(logits)
    dev = logits.device
    if mask.shape != (B, V) or mask.dtype not in (torch.bool, torch.uint8) or not mask.is_contiguous():
        raise ValueError("mask must be a contiguous bool/uint8 [B, V] tensor")
    uu = _vec(u, B, torch.float32, "u", dev)
    if out is None:
        ids = torch.full((B, int(cap)), -1, dtype=torch.int32, device=dev)
        probs = torch.zeros((B, int(cap)), dtype=torch.float32, device=dev)
        count = torch.empty(B, dtype=torch.int32, device=dev)
        sample = torch.empty(B, dtype=torch.int32, device=dev) if uu is not None else None
    else:
        ids, probs, count, sample = out
        for t, shape, dt, name in ((ids, (B, int(cap)), torch.int32, "ids"), (probs, (B, int(cap)), torch.float32, "probs"),
                                   (count, (B,), torch.int32, "count")):
            if t.shape != shape or t.dtype != dt or not t.is_contiguous() or t.device != dev:
                raise ValueError(f"out {name} must be a contiguous {dt} {list(shape)} tensor on {dev}")
        if (sample is None) != (uu is None):
            raise ValueError("out sample must be given exactly when u is")
        if sample is not None and (sample.shape != (B,) or sample.dtype != torch.int32 or not sample.is_contiguous()
                                   or sample.device != dev):
            raise ValueError(f"out sample must be a contiguous int32 [{B}] tensor on {dev}")
    rc = lib().qrita_candidates(
        ctypes.c_void_p(logits.data_ptr() if B else 0), _dtype_code(logits), B, V,
        ctypes.c_void_p(mask.data_ptr() if B else 0), int(cap), ctypes.c_void_p(ids.data_ptr() if B else 0),
        ctypes.c_void_p(probs.data_ptr() if B else 0), ctypes.c_void_p(count.data_ptr() if B else 0),
        ctypes.c_void_p(uu.data_ptr() if uu is not None else 0),
        ctypes.c_void_p(sample.data_ptr() if sample is not None else 0), _stream_ptr(dev, stream))
    if rc != OK:
        raise QritaError(rc)
    return ids, probs, count, sample


def delta_table(which: int) -> np.ndarray:
    """The host-built truncation table the kernel receives: ``which`` 0 is the
    top-k table (entry i = Phi^-1(1 - 2^(-i/4))), 1 the top-p table (entry
    i = Phi^-1(2^(-i/4))). Returns float32 [length]."""
    n = int(lib().qrita_delta_table(int(which), None, 0))
    if n < 0:
        raise ValueError(f"unknown delta table {which}")
    out = np.zeros(n, np.float32)
    lib().qrita_delta_table(int(which), out.ctypes.data_as(ctypes.c_void_p), n)
    return out


def host_staging_bytes(dtype_code: int, B: int, V: int) -> int:
    return int(lib().qrita_host_staging_bytes(int(dtype_code), int(B), int(V)))


def qrita_select_host(logits, k=None, p=None, out=None, staging=None, stream=None):
    """End-to-end selection for HOST (CPU) tensors through qrita_select_host.

    logits: CPU tensor [B, V] float32 / bfloat16 (pinned for full-speed
    copies); k / p: CPU int32 / float32 [B] or None; out: CPU uint8/bool
    [B, V] or None; staging: CUDA uint8 tensor of at least
    host_staging_bytes(...) bytes (allocated here when None). Returns ``out``
    after the stream has finished.
    """
    torch = _torch()
    if logits.dim() != 2 or logits.is_cuda:
        raise ValueError("logits must be a host [B, V] tensor")
    B, V = logits.shape
    if B > 0 and (logits.stride(1) != 1 or (B > 1 and logits.stride(0) != V)):
        raise ValueError("logits must be row-major with leading dimension V")
    dt = _dtype_code(logits)
    cpu = torch.device("cpu")
    kk = _vec(k, B, torch.int32, "k", cpu)
    pp = _vec(p, B, torch.float32, "p", cpu)
    if out is None:
        out = torch.empty((B, V), dtype=torch.bool, pin_memory=logits.is_pinned())
    need = host_staging_bytes(dt, B, V)
    dev = torch.device("cuda", torch.cuda.current_device())
    if staging is None:
        staging = torch.empty(need, dtype=torch.uint8, device=dev)
    elif staging.numel() < need or not staging.is_cuda:
        raise ValueError(f"staging must be a CUDA tensor of at least {need} bytes")
    rc = lib().qrita_select_host(
        ctypes.c_void_p(logits.data_ptr() if B else 0),
        dt,
        B,
        V,
        ctypes.c_void_p(kk.data_ptr() if kk is not None else 0),
        ctypes.c_void_p(pp.data_ptr() if pp is not None else 0),
        ctypes.c_void_p(out.data_ptr() if B else 0),
        ctypes.c_void_p(staging.data_ptr()),
        ctypes.c_size_t(staging.numel()),
        _stream_ptr(staging.device, stream),
    )
    if rc != OK:
        raise QritaError(rc)
    return out
