"""Python front end of the CPU oracle (fp64, plain loops in C).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use it.  It never imports the product package's
compiled library and the product never imports this module.

``build()`` compiles ``lora_oracle.c`` with gcc (OpenMP when available) into
``oracle/_build/liboracle.so``.  The functions below marshal CPU torch tensors
into the C calls; every arithmetic step happens in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle; returns the path of the shared object."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_build_segments.restype = ctypes.c_int
        lib.oracle_build_segments.argtypes = [p, i64, i32, p, p, p, p, p, p, p, p]
        lib.oracle_lora_linear_rows.restype = None
        lib.oracle_lora_linear_rows.argtypes = [p, i64, i64, p, i64, p, p, i32, p, p, p, dbl,
                                                p, p, i64, p]
        lib.oracle_shrink_rows.restype = None
        lib.oracle_shrink_rows.argtypes = [p, i64, i64, p, i32, p, p, p, i64, i64, p]
        lib.oracle_lora_linear_elems.restype = None
        lib.oracle_lora_linear_elems.argtypes = [p, i64, p, i64, p, p, i32, p, p, p, dbl, p, p, p, i64, p]
        lib.oracle_lora_linear_slices_rows.restype = None
        lib.oracle_lora_linear_slices_rows.argtypes = [p, i64, i64, p, i64, p, p, i32, p, i32, p, p, p, dbl,
                                                       p, p, i64, p]
        lib.oracle_moe_rows.restype = None
        lib.oracle_moe_rows.argtypes = [p, i64, i64, p, i64, i32, i32, p, p, p, i64, p]
        lib.oracle_expand_rows.restype = None
        lib.oracle_expand_rows.argtypes = [p, i64, p, i64, p, i32, p, p, dbl, p, p, i64, p]
        lib.oracle_e4m3_to_f64.restype = dbl
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_lora_linear_rows_e4m3.restype = None
        lib.oracle_lora_linear_rows_e4m3.argtypes = [p, i64, i64, p, i64, p, p, i32, p, p, p, p, dbl, p, p, i64, p]
        lib.oracle_shrink_rows_e4m3.restype = None
        lib.oracle_shrink_rows_e4m3.argtypes = [p, i64, i64, p, i32, p, p, p, p, i64, i64, p]
        lib.oracle_expand_rows_e4m3.restype = None
        lib.oracle_expand_rows_e4m3.argtypes = [p, i64, p, i64, p, i32, p, p, p, dbl, p, p, i64, p]
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------------------
# marshalling helpers (no arithmetic)
# ---------------------------------------------------------------------------

def _bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """bf16 tensor -> contiguous uint16 numpy array of its raw bits."""
    if t is None:
        return None
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _adapter_scale(wl) -> Optional[np.ndarray]:
    """fp64 per-adapter factors of the LoRA term, or None (all 1)."""
    a = getattr(wl, "adapter_scale", None)
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    assert a.shape == (len(wl.ranks),)
    return a


def _codes(mats: List[torch.Tensor]) -> np.ndarray:
    """e4m3 codes (uint8 tensors) concatenated in the oracle's layout."""
    if not mats:
        return np.zeros(1, dtype=np.uint8)
    return np.ascontiguousarray(torch.cat([m.reshape(-1) for m in mats]).numpy().astype(np.uint8))


def _deq(wl) -> np.ndarray:
    """fp64 [num_adapters][2] dequant factors (A, B) of an e4m3 workload."""
    d = np.ascontiguousarray(np.asarray(wl.deq or [(1.0, 1.0)], dtype=np.float64).reshape(-1))
    return d


def e4m3_to_f64(code: int) -> float:
    """The oracle's decode of one e4m3 code."""
    return float(_load().oracle_e4m3_to_f64(int(code) & 0xFF))


def _concat(mats: List[torch.Tensor], K_or_N: int) -> np.ndarray:
    if not mats:
        return np.zeros(1, dtype=np.uint16)
    return _bits(torch.cat([m.reshape(-1) for m in mats]).contiguous())


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < M))
    return r, r.size


# ---------------------------------------------------------------------------
# public oracle calls
# ---------------------------------------------------------------------------

def build_segments(ids, num_adapters: int, true_ranks: Sequence[int]):
    """Segment table of "vLLM-Ascend dynamic LoRA" §2.3 (stable sort by id).

    Returns a dict of numpy int32 arrays: perm, bucket_offsets, seg_id,
    seg_start, seg_len, seg_rank (padded), plus num_segments and invalid.
    """
    lib = _load()
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    M = ids.size
    A = int(num_adapters)
    rk = np.ascontiguousarray(np.asarray(list(true_ranks) or [0], dtype=np.int32))
    perm = np.zeros(max(M, 1), np.int32)
    off = np.zeros(A + 2, np.int32)
    sid, sst, sln, srk = (np.zeros(max(A, 1), np.int32) for _ in range(4))
    ns = np.zeros(1, np.int32)
    invalid = lib.oracle_build_segments(_ptr(ids), M, A, _ptr(rk), _ptr(perm), _ptr(off),
                                        _ptr(sid), _ptr(sst), _ptr(sln), _ptr(srk), _ptr(ns))
    n = int(ns[0])
    return dict(perm=perm[:M], bucket_offsets=off, seg_id=sid[:n], seg_start=sst[:n],
                seg_len=sln[:n], seg_rank=srk[:n], num_segments=n, invalid=int(invalid))


def lora_linear(wl, rows=None, scale: Optional[float] = None) -> np.ndarray:
    """fp64 layer output for a Workload-like object (fields x, W, bias, ids,
    ranks, A, B, scale; or slices, A_s, B_s for a merged output).  ``rows``
    selects output rows; returns [len(rows), N]."""
    if getattr(wl, "slices", None):
        return _lora_linear_slices(wl, rows, scale)
    if getattr(wl, "A8", None) is not None:
        return _lora_linear_e4m3(wl, rows, scale)
    lib = _load()
    x, W, bias = _bits(wl.x), _bits(wl.W), _bits(wl.bias)
    ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
    rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
    a_cat, b_cat = _concat(wl.A, wl.K), _concat(wl.B, wl.N)
    r, nrows = _rows_arg(rows, wl.M)
    y = np.zeros((nrows, wl.N), dtype=np.float64)
    s = wl.scale if scale is None else scale
    asc = _adapter_scale(wl)
    lib.oracle_lora_linear_rows(_ptr(x), wl.M, wl.K, _ptr(W), wl.N, _ptr(bias), _ptr(ids),
                                len(wl.ranks), _ptr(rk), _ptr(a_cat), _ptr(b_cat), float(s),
                                _ptr(asc), _ptr(r), nrows, _ptr(y))
    return y


def _lora_linear_e4m3(wl, rows, scale):
    """e4m3 adapters: A_i = deq_a,i e4m3(A8_i), B_i = deq_b,i e4m3(B8_i)."""
    lib = _load()
    x, W, bias = _bits(wl.x), _bits(wl.W), _bits(wl.bias)
    ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
    rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
    a8, b8, deq = _codes(wl.A8), _codes(wl.B8), _deq(wl)
    r, nrows = _rows_arg(rows, wl.M)
    y = np.zeros((nrows, wl.N), dtype=np.float64)
    s = wl.scale if scale is None else scale
    lib.oracle_lora_linear_rows_e4m3(_ptr(x), wl.M, wl.K, _ptr(W), wl.N, _ptr(bias), _ptr(ids), len(wl.ranks),
                                     _ptr(rk), _ptr(a8), _ptr(b8), _ptr(deq), float(s), _ptr(_adapter_scale(wl)),
                                     _ptr(r), nrows, _ptr(y))
    return y


def _lora_linear_slices(wl, rows, scale):
    """Merged output: one A / B pair per output slice and adapter."""
    lib = _load()
    x, W, bias = _bits(wl.x), _bits(wl.W), _bits(wl.bias)
    ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
    rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
    assert sum(wl.slices) == wl.N
    starts = np.ascontiguousarray(np.concatenate([[0], np.cumsum(wl.slices)]).astype(np.int64))
    a_cat = _concat([a for per in wl.A_s for a in per], wl.K)
    b_cat = _concat([b for per in wl.B_s for b in per], wl.N)
    r, nrows = _rows_arg(rows, wl.M)
    y = np.zeros((nrows, wl.N), dtype=np.float64)
    s = wl.scale if scale is None else scale
    lib.oracle_lora_linear_slices_rows(_ptr(x), wl.M, wl.K, _ptr(W), wl.N, _ptr(bias), _ptr(ids), len(wl.ranks),
                                       _ptr(rk), len(wl.slices), _ptr(starts), _ptr(a_cat), _ptr(b_cat), float(s),
                                       _ptr(_adapter_scale(wl)), _ptr(r), nrows, _ptr(y))
    return y


class Prepared:
    """Inputs of one workload marshalled once (bits + concatenated adapters),
    so repeated oracle calls on samples do not re-marshal the whole workload."""

    def __init__(self, wl):
        self.wl = wl
        self.x, self.W, self.bias = _bits(wl.x), _bits(wl.W), _bits(wl.bias)
        self.ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
        self.rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
        self.a_cat, self.b_cat = _concat(wl.A, wl.K), _concat(wl.B, wl.N)
        self.asc = _adapter_scale(wl)


def lora_linear_elems(prep: "Prepared", rows, cols, scale: Optional[float] = None) -> np.ndarray:
    """fp64 y[rows[q], cols[q]] for q = 0..n-1 (element samples)."""
    lib = _load()
    wl = prep.wl
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    assert r.shape == c.shape and r.ndim == 1
    assert r.size == 0 or (r.min() >= 0 and r.max() < wl.M and c.min() >= 0 and c.max() < wl.N)
    y = np.zeros(r.size, dtype=np.float64)
    s = wl.scale if scale is None else scale
    lib.oracle_lora_linear_elems(_ptr(prep.x), wl.K, _ptr(prep.W), wl.N, _ptr(prep.bias),
                                 _ptr(prep.ids), len(wl.ranks), _ptr(prep.rk), _ptr(prep.a_cat),
                                 _ptr(prep.b_cat), float(s), _ptr(prep.asc), _ptr(r), _ptr(c), r.size,
                                 _ptr(y))
    return y


def lora_linear_rows_prepared(prep: "Prepared", rows) -> np.ndarray:
    """Like lora_linear(wl, rows) but reusing marshalled inputs."""
    lib = _load()
    wl = prep.wl
    r, nrows = _rows_arg(rows, wl.M)
    y = np.zeros((nrows, wl.N), dtype=np.float64)
    lib.oracle_lora_linear_rows(_ptr(prep.x), wl.M, wl.K, _ptr(prep.W), wl.N, _ptr(prep.bias),
                                _ptr(prep.ids), len(wl.ranks), _ptr(prep.rk), _ptr(prep.a_cat),
                                _ptr(prep.b_cat), float(wl.scale), _ptr(prep.asc), _ptr(r), nrows, _ptr(y))
    return y


def shrink(wl, s_cols: int, rows=None) -> np.ndarray:
    """fp64 S = x A_id^T, [len(rows), s_cols], zero outside each row's rank."""
    lib = _load()
    x = _bits(wl.x)
    ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
    rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
    r, nrows = _rows_arg(rows, wl.M)
    S = np.zeros((nrows, s_cols), dtype=np.float64)
    if getattr(wl, "A8", None) is not None:
        lib.oracle_shrink_rows_e4m3(_ptr(x), wl.M, wl.K, _ptr(ids), len(wl.ranks), _ptr(rk), _ptr(_codes(wl.A8)),
                                    _ptr(_deq(wl)), _ptr(r), nrows, s_cols, _ptr(S))
        return S
    a_cat = _concat(wl.A, wl.K)
    lib.oracle_shrink_rows(_ptr(x), wl.M, wl.K, _ptr(ids), len(wl.ranks), _ptr(rk),
                           _ptr(a_cat), _ptr(r), nrows, s_cols, _ptr(S))
    return S


def expand(wl, S: torch.Tensor, y_in: torch.Tensor, scale: Optional[float] = None,
           rows=None) -> np.ndarray:
    """fp64 y_in + scale * S B_id^T for the given fp32 S [M, s_cols] and bf16 y_in [M, N]."""
    lib = _load()
    S_np = np.ascontiguousarray(S.detach().cpu().float().numpy())
    yin = _bits(y_in)
    ids = np.ascontiguousarray(wl.ids.numpy().astype(np.int32))
    rk = np.ascontiguousarray(np.asarray(list(wl.ranks) or [0], dtype=np.int32))
    r, nrows = _rows_arg(rows, wl.M)
    y = np.zeros((nrows, wl.N), dtype=np.float64)
    s = wl.scale if scale is None else scale
    asc = _adapter_scale(wl)
    if getattr(wl, "A8", None) is not None:
        lib.oracle_expand_rows_e4m3(_ptr(S_np), S_np.shape[1], _ptr(yin), wl.N, _ptr(ids), len(wl.ranks), _ptr(rk),
                                    _ptr(_codes(wl.B8)), _ptr(_deq(wl)), float(s), _ptr(asc), _ptr(r), nrows,
                                    _ptr(y))
        return y
    b_cat = _concat(wl.B, wl.N)
    lib.oracle_expand_rows(_ptr(S_np), S_np.shape[1], _ptr(yin), wl.N, _ptr(ids),
                           len(wl.ranks), _ptr(rk), _ptr(b_cat), float(s), _ptr(asc), _ptr(r), nrows,
                           _ptr(y))
    return y


def moe(x: torch.Tensor, W: torch.Tensor, expert: torch.Tensor, weight: torch.Tensor, rows=None) -> np.ndarray:
    """fp64 mixture-of-experts output: x bf16 [M, K], W bf16 [E, N, K],
    expert int [M, topk] (ids outside [0, E) contribute nothing), weight
    fp32 [M, topk].  Returns [len(rows), N]."""
    lib = _load()
    M, K = x.shape
    E, N, _ = W.shape
    topk = expert.shape[1]
    xb, Wb = _bits(x.contiguous()), _bits(W.contiguous())
    ex = np.ascontiguousarray(expert.numpy().astype(np.int32))
    wt = np.ascontiguousarray(weight.numpy().astype(np.float32))
    r, nrows = _rows_arg(rows, M)
    y = np.zeros((nrows, N), dtype=np.float64)
    lib.oracle_moe_rows(_ptr(xb), M, K, _ptr(Wb), N, E, topk, _ptr(ex), _ptr(wt), _ptr(r), nrows, _ptr(y))
    return y


def moe_routing(expert: torch.Tensor, num_experts: int):
    """The routing of the (token, slot) pairs: pair p = t * topk + j sorted
    stably by expert (the segment build over the pairs' expert ids), and the
    number of pairs per expert."""
    seg = build_segments(expert.reshape(-1).numpy(), num_experts, [16] * num_experts)
    counts = np.diff(seg["bucket_offsets"])[1:]
    return seg["perm"], seg["bucket_offsets"], counts
