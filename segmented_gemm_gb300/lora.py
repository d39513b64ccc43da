"""Python binding of liblora (include/lora.h), argument marshalling only.

Every entry point keeps the C name and forwards device pointers, sizes and
the current CUDA stream of PyTorch; all arithmetic runs in the library's CUDA
kernels.  PyTorch only provides device memory and streams.  There is no CPU
fallback: if the compiled library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblora.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "liblora_debug.so")   # built with LORA_DEBUG: table checks before every use

LORA_OK = 0
LORA_ERR_NULL, LORA_ERR_SHAPE, LORA_ERR_ALIGN, LORA_ERR_RANK = 1, 2, 3, 4
LORA_ERR_WORKSPACE, LORA_ERR_CUDA, LORA_ERR_UNSUPPORTED, LORA_ERR_SEGMENTS = 5, 6, 7, 8
LORA_ERR_CAPACITY, LORA_ERR_ACCESS = 9, 10
LORA_MAX_COPIES = 4
LORA_NOALLOC_SCRATCH_BYTES = 8 << 20
LORA_DEV_BAD_ID, LORA_DEV_TIMEOUT, LORA_DEV_BAD_POOL, LORA_DEV_CHECK = 1, 2, 4, 8
LORA_PATH_AUTO, LORA_PATH_TILED, LORA_PATH_SPLITK, LORA_PATH_STREAM = 0, 1, 2, 3
LORA_FLAG_STATIC_WEIGHTS = 0x100
LORA_MAX_SLICES = 4
LORA_ADAPTER_BF16, LORA_ADAPTER_E4M3 = 0, 1
LORA_MAX_LAYERS = 8
LORA_MAX_RANK, LORA_RANK_ALIGN, LORA_MAX_ADAPTERS = 128, 16, 1024

EXPORTS = ("lora_pool_layout", "lora_workspace_size", "lora_workspace_init", "lora_build_segments",
           "lora_shrink", "lora_expand", "lora_linear", "lora_linear_ex", "lora_get_status",
           "lora_status_string", "lora_linear_noalloc", "lora_moe_workspace_size", "lora_moe_route",
           "lora_moe_gemm", "lora_moe_finalize", "lora_moe", "lora_layers_workspace_size", "lora_linear_layers",
           "lora_set_wait_budget", "lora_check_segments", "lora_moe_check_route", "lora_device_pointer",
           "lora_copy_async")


class lora_pool_t(ctypes.Structure):
    _fields_ = [("a_pool", ctypes.c_void_p), ("b_pool", ctypes.c_void_p),
                ("a_offset", ctypes.c_void_p), ("b_offset", ctypes.c_void_p),
                ("rank", ctypes.c_void_p), ("a_elems", ctypes.c_int64), ("b_elems", ctypes.c_int64),
                ("num_adapters", ctypes.c_int32), ("max_rank", ctypes.c_int32),
                ("K", ctypes.c_int32), ("N", ctypes.c_int32), ("adapter_scale", ctypes.c_void_p),
                ("num_slices", ctypes.c_int32), ("slice_start", ctypes.c_int32 * (LORA_MAX_SLICES + 1)),
                ("adapter_type", ctypes.c_int32), ("dequant", ctypes.c_void_p), ("widened", ctypes.c_void_p)]


class lora_segments_t(ctypes.Structure):
    _fields_ = [("perm", ctypes.c_void_p), ("bucket_offsets", ctypes.c_void_p),
                ("seg_id", ctypes.c_void_p), ("seg_start", ctypes.c_void_p),
                ("seg_len", ctypes.c_void_p), ("seg_rank", ctypes.c_void_p),
                ("num_segments", ctypes.c_void_p), ("plan", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("num_adapters", ctypes.c_int32), ("num_slices", ctypes.c_int32)]


class lora_copy_t(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_int64)]


class lora_layer_t(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("W", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("pool", ctypes.c_void_p), ("scale", ctypes.c_float), ("y", ctypes.c_void_p)]


class LoraError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (code {code})")
        self.code = code


_libs = {}
_active = LIB_PATH


def use_debug_library(debug: bool):
    """Route every later call through liblora_debug.so (True) or liblora.so
    (False).  Both may be loaded at once; workspaces and pools serve either."""
    global _active
    _active = DEBUG_LIB_PATH if debug else LIB_PATH


def load_library():
    """Load the active library (liblora.so unless use_debug_library(True));
    raises if it has not been built."""
    path = _active
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    PP = ctypes.POINTER(lora_pool_t)
    PS = ctypes.POINTER(lora_segments_t)
    sig = {
        "lora_pool_layout": (ctypes.c_int, [I32, P, I32, I32, P, P, P, P, P]),
        "lora_workspace_size": (SZ, [I64, I32, I32]),
        "lora_workspace_init": (ctypes.c_int, [P, SZ, P]),
        "lora_build_segments": (ctypes.c_int, [P, I64, PP, PS, P, SZ, P]),
        "lora_shrink": (ctypes.c_int, [P, I64, P, PP, PS, P, I32, P, SZ, P]),
        "lora_expand": (ctypes.c_int, [P, I32, I64, P, PP, PS, F32, P, P, SZ, P]),
        "lora_linear": (ctypes.c_int, [P, I64, P, P, P, PP, F32, PS, P, P, SZ, P]),
        "lora_linear_ex": (ctypes.c_int, [P, I64, P, P, P, PP, F32, PS, P, P, SZ, P, I32]),
        "lora_get_status": (ctypes.c_int, [P, P, P]),
        "lora_linear_noalloc": (ctypes.c_int, [P, I64, P, P, P, PP, F32, P, P]),
        "lora_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "lora_moe_workspace_size": (SZ, [I64, I32, I32]),
        "lora_moe_route": (ctypes.c_int, [P, I64, I32, I32, P, SZ, P]),
        "lora_moe_gemm": (ctypes.c_int, [P, I64, I32, P, I32, I32, I32, P, P, SZ, P]),
        "lora_moe_finalize": (ctypes.c_int, [P, P, P, I64, I32, I32, I32, P, P]),
        "lora_moe": (ctypes.c_int, [P, I64, I32, P, I32, P, P, I32, I32, P, P, P, SZ, P]),
        "lora_layers_workspace_size": (SZ, [I64, I32, I32, I32]),
        "lora_linear_layers": (ctypes.c_int, [P, I32, I64, P, PS, P, SZ, P]),
        "lora_set_wait_budget": (ctypes.c_int, [I64]),
        "lora_check_segments": (ctypes.c_int, [P, I64, PP, PS, P, SZ, P]),
        "lora_moe_check_route": (ctypes.c_int, [P, I64, I32, I32, P, SZ, P]),
        "lora_device_pointer": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_void_p)]),
        "lora_copy_async": (ctypes.c_int, [ctypes.POINTER(lora_copy_t), I32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _libs[path] = lib
    return lib


def status_string(code: int) -> str:
    return load_library().lora_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != LORA_OK:
        raise LoraError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def device_pointer(t: torch.Tensor) -> int:
    """The address kernels on the current device use for t's storage: its
    own for device memory, the mapped alias for pinned host memory
    (LoraError LORA_ERR_ACCESS for pageable host memory)."""
    out = ctypes.c_void_p()
    _check(load_library().lora_device_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(out)),
           "lora_device_pointer")
    return int(out.value)


def _out_ptr(t: torch.Tensor):
    """An output the kernels write with plain stores: device memory, or a
    pinned host tensor through its device address."""
    return ctypes.c_void_p(t.data_ptr() if t.is_cuda else device_pointer(t))


def copy_async(pairs: Sequence[tuple], stream=None):
    """dst <- src for up to LORA_MAX_COPIES (dst, src) tensor pairs of equal
    byte size, in one kernel on ``stream`` (lora_copy_async): each side
    contiguous, on the device or in pinned host memory."""
    if len(pairs) > LORA_MAX_COPIES:
        raise ValueError(f"at most {LORA_MAX_COPIES} copies per call")
    arr = (lora_copy_t * max(len(pairs), 1))()
    for i, (dst, src) in enumerate(pairs):
        nb = dst.numel() * dst.element_size()
        if src.numel() * src.element_size() != nb or not dst.is_contiguous() or not src.is_contiguous():
            raise ValueError("copy_async: contiguous tensors of equal byte size")
        arr[i].dst, arr[i].src, arr[i].bytes = dst.data_ptr(), src.data_ptr(), nb
    _check(load_library().lora_copy_async(arr, len(pairs), _stream(stream)), "lora_copy_async")


# ---------------------------------------------------------------------------
# adapter pool (load-time arrangement; not part of the per-step path)
# ---------------------------------------------------------------------------

def lora_pool_layout(true_ranks: Sequence[int], K: int, N: int):
    """Rank-grouped offsets: returns (a_offset, b_offset, rank_padded, a_elems, b_elems)."""
    lib = load_library()
    n = len(true_ranks)
    rk = (ctypes.c_int32 * max(n, 1))(*true_ranks)
    ao = (ctypes.c_int64 * max(n, 1))()
    bo = (ctypes.c_int64 * max(n, 1))()
    rp = (ctypes.c_int32 * max(n, 1))()
    ae, be = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.lora_pool_layout(n, rk, K, N, ao, bo, rp, ctypes.byref(ae), ctypes.byref(be)),
           "lora_pool_layout")
    return list(ao)[:n], list(bo)[:n], list(rp)[:n], ae.value, be.value


@dataclass
class LoraPool:
    """Device-resident rank-grouped adapter pool and its C descriptor."""
    a_pool: torch.Tensor
    b_pool: torch.Tensor
    a_offset: torch.Tensor
    b_offset: torch.Tensor
    rank: torch.Tensor
    desc: lora_pool_t
    true_ranks: List[int]
    padded_ranks: List[int]
    adapter_scale: Optional[torch.Tensor] = None   # fp32 [num_adapters] factors, or None (all 1)
    dequant: Optional[torch.Tensor] = None         # e4m3 pools: fp32 [num_adapters][2]
    widened: Optional[torch.Tensor] = None         # e4m3 pools: bf16 scratch [a_elems + b_elems]

    @property
    def num_adapters(self):
        return self.desc.num_adapters


def build_pool(A: List[torch.Tensor], B: List[torch.Tensor], K: int, N: int, device="cuda",
               adapter_scale: Optional[Sequence[float]] = None) -> LoraPool:
    """Arrange adapters A_i [r_i, K], B_i [N, r_i] into the pool layout of
    include/lora.h (rank-grouped; A rows and B panels zero-padded to 16).
    ``adapter_scale``: optional per-adapter factors s_i (adapter i's delta is
    multiplied by the call's scale times s_i)."""
    ranks = [int(a.shape[0]) for a in A]
    a_off, b_off, rpad, a_elems, b_elems = lora_pool_layout(ranks, K, N)
    bf = torch.bfloat16
    a_pool = torch.zeros(max(a_elems, 8), dtype=bf, device=device)
    b_pool = torch.zeros(max(b_elems, 8), dtype=bf, device=device)
    for i, (a, b) in enumerate(zip(A, B)):
        r, rp = ranks[i], rpad[i]
        assert a.shape == (r, K) and b.shape == (N, r)
        a_pool[a_off[i]:a_off[i] + r * K] = a.to(device=device, dtype=bf).reshape(-1)
        bp = torch.zeros(N, rp, dtype=bf, device=device)
        bp[:, :r] = b.to(device=device, dtype=bf)
        panels = bp.reshape(N, rp // 16, 16).permute(1, 0, 2).contiguous()   # [rp/16, N, 16]
        b_pool[b_off[i]:b_off[i] + rp * N] = panels.reshape(-1)
    a_offset = torch.tensor(a_off or [0], dtype=torch.int64, device=device)
    b_offset = torch.tensor(b_off or [0], dtype=torch.int64, device=device)
    rank = torch.tensor(rpad or [0], dtype=torch.int32, device=device)
    asc = None
    if adapter_scale is not None:
        assert len(adapter_scale) == len(A)
        asc = torch.tensor([float(v) for v in adapter_scale] or [1.0], dtype=torch.float32, device=device)
    desc = lora_pool_t(a_pool.data_ptr(), b_pool.data_ptr(), a_offset.data_ptr(), b_offset.data_ptr(),
                       rank.data_ptr(), a_elems, b_elems, len(A), max(rpad) if rpad else 0, K, N,
                       asc.data_ptr() if asc is not None else None)
    return LoraPool(a_pool, b_pool, a_offset, b_offset, rank, desc, ranks, rpad, asc)


def build_pool_e4m3(A8: List[torch.Tensor], B8: List[torch.Tensor], deq: Sequence[tuple], K: int, N: int,
                    device="cuda", adapter_scale: Optional[Sequence[float]] = None,
                    widened: bool = True) -> LoraPool:
    """An e4m3 pool: codes A8_i uint8 [r_i, K] and B8_i uint8 [N, r_i] in the
    layout of build_pool (one byte per element), dequant factors deq[i] =
    (a, b), and (``widened``) the bf16 scratch the schedules for more than
    64 tokens widen the used adapters into."""
    ranks = [int(a.shape[0]) for a in A8]
    a_off, b_off, rpad, a_elems, b_elems = lora_pool_layout(ranks, K, N)
    u8 = torch.uint8
    a_pool = torch.zeros(max(a_elems, 16), dtype=u8, device=device)
    b_pool = torch.zeros(max(b_elems, 16), dtype=u8, device=device)
    for i, (a, b) in enumerate(zip(A8, B8)):
        r, rp = ranks[i], rpad[i]
        assert a.shape == (r, K) and b.shape == (N, r) and a.dtype == u8 and b.dtype == u8
        a_pool[a_off[i]:a_off[i] + r * K] = a.to(device).reshape(-1)
        bp = torch.zeros(N, rp, dtype=u8, device=device)
        bp[:, :r] = b.to(device)
        b_pool[b_off[i]:b_off[i] + rp * N] = bp.reshape(N, rp // 16, 16).permute(1, 0, 2).contiguous().reshape(-1)
    a_offset = torch.tensor(a_off or [0], dtype=torch.int64, device=device)
    b_offset = torch.tensor(b_off or [0], dtype=torch.int64, device=device)
    rank = torch.tensor(rpad or [0], dtype=torch.int32, device=device)
    asc = None
    if adapter_scale is not None:
        asc = torch.tensor([float(v) for v in adapter_scale] or [1.0], dtype=torch.float32, device=device)
    dq = torch.tensor([float(v) for pair in deq for v in pair] or [1.0, 1.0], dtype=torch.float32, device=device)
    wid = torch.zeros(max(a_elems + b_elems, 8), dtype=torch.bfloat16, device=device) if widened else None
    desc = lora_pool_t(a_pool.data_ptr(), b_pool.data_ptr(), a_offset.data_ptr(), b_offset.data_ptr(),
                       rank.data_ptr(), a_elems, b_elems, len(A8), max(rpad) if rpad else 0, K, N,
                       asc.data_ptr() if asc is not None else None)
    desc.adapter_type = LORA_ADAPTER_E4M3
    desc.dequant = dq.data_ptr()
    desc.widened = wid.data_ptr() if wid is not None else None
    return LoraPool(a_pool, b_pool, a_offset, b_offset, rank, desc, ranks, rpad, asc, dq, wid)


def build_pool_sliced(A_s: List[List[torch.Tensor]], B_s: List[List[torch.Tensor]], K: int, slices: Sequence[int],
                      device="cuda", adapter_scale: Optional[Sequence[float]] = None) -> LoraPool:
    """A merged-output pool (Q|K|V, gate|up): A_s[i][s] [r_i, K] and
    B_s[i][s] [N_s, r_i] for output slices of widths ``slices``.  Adapter i is
    stored as one adapter of rank S * ceil16(r_i): the slices' A stacked (each
    padded to 16 rows) and a block-diagonal B (include/lora.h, lora_pool_t)."""
    S, N = len(slices), int(sum(slices))
    assert 1 <= S <= LORA_MAX_SLICES
    starts = [0]
    for n in slices:
        starts.append(starts[-1] + int(n))
    A, B = [], []
    for a_list, b_list in zip(A_s, B_s):
        r = int(a_list[0].shape[0])
        rp = (r + 15) // 16 * 16
        a = torch.zeros(S * rp, K, dtype=torch.bfloat16)
        b = torch.zeros(N, S * rp, dtype=torch.bfloat16)
        for s in range(S):
            a[s * rp:s * rp + r] = a_list[s].to(torch.bfloat16)
            b[starts[s]:starts[s + 1], s * rp:s * rp + r] = b_list[s].to(torch.bfloat16)
        A.append(a)
        B.append(b)
    pool = build_pool(A, B, K, N, device, adapter_scale=adapter_scale)
    pool.desc.num_slices = S
    for s in range(S + 1):
        pool.desc.slice_start[s] = starts[s]
    return pool


# ---------------------------------------------------------------------------
# workspace and segments
# ---------------------------------------------------------------------------

def lora_workspace_size(M: int, N: int, num_adapters: int) -> int:
    return int(load_library().lora_workspace_size(M, N, num_adapters))


class Workspace:
    """A zero-initialised device workspace sized for (M, N, num_adapters)."""

    def __init__(self, M: int, N: int, num_adapters: int, device="cuda"):
        self.nbytes = lora_workspace_size(M, N, num_adapters)
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def lora_workspace_init(ws: Workspace, stream=None):
    _check(load_library().lora_workspace_init(ws.ptr, ws.nbytes, _stream(stream)), "lora_workspace_init")


def lora_build_segments(ids: torch.Tensor, pool: LoraPool, ws: Workspace, stream=None) -> lora_segments_t:
    out = lora_segments_t()
    _check(load_library().lora_build_segments(_ptr(ids), ids.numel(), ctypes.byref(pool.desc),
                                              ctypes.byref(out), ws.ptr, ws.nbytes, _stream(stream)),
           "lora_build_segments")
    return out


def lora_check_segments(ids: torch.Tensor, pool: LoraPool, ws: Workspace, segs: lora_segments_t, stream=None):
    """Enqueue the device check of the table in ws; its verdict is the
    LORA_DEV_CHECK bit of lora_get_status."""
    _check(load_library().lora_check_segments(_ptr(ids), ids.numel(), ctypes.byref(pool.desc), ctypes.byref(segs),
                                              ws.ptr, ws.nbytes, _stream(stream)), "lora_check_segments")


def segments_to_host(segs: lora_segments_t, ws: Workspace, M: int, num_adapters: int) -> dict:
    """Copy a device segment table (it lives inside ws) into CPU int32 tensors."""
    base = ws.buf.data_ptr()

    def grab(ptr, n):
        off = int(ptr) - base
        assert 0 <= off and off + 4 * n <= ws.buf.numel()
        return ws.buf[off:off + 4 * n].view(torch.int32).cpu()

    ns = int(grab(segs.num_segments, 1)[0])
    return dict(perm=grab(segs.perm, M), bucket_offsets=grab(segs.bucket_offsets, num_adapters + 2),
                seg_id=grab(segs.seg_id, ns), seg_start=grab(segs.seg_start, ns),
                seg_len=grab(segs.seg_len, ns), seg_rank=grab(segs.seg_rank, ns), num_segments=ns)


# ---------------------------------------------------------------------------
# compute entry points
# ---------------------------------------------------------------------------

def lora_linear(x: torch.Tensor, W: torch.Tensor, bias: Optional[torch.Tensor], ids: torch.Tensor,
                pool: LoraPool, scale: float, ws: Workspace, y: Optional[torch.Tensor] = None,
                segs: Optional[lora_segments_t] = None, path: int = LORA_PATH_AUTO,
                stream=None, static_weights: bool = False) -> torch.Tensor:
    """y = x W^T + bias + scale * (x A_id^T) B_id^T per token (id -1: base only).

    ``static_weights``: W, bias and the pool are written by no kernel that
    can still run when the call starts (LORA_FLAG_STATIC_WEIGHTS), so the call
    may start streaming them before the kernel ahead of it has finished.
    ``y`` may be a pinned host tensor: the kernels store into it directly."""
    M = x.shape[0]
    if y is None:
        y = torch.empty(M, W.shape[0], dtype=torch.bfloat16, device=x.device)
    _check(load_library().lora_linear_ex(
        _ptr(x), M, _ptr(W), _ptr(bias), _ptr(ids), ctypes.byref(pool.desc), float(scale),
        ctypes.byref(segs) if segs is not None else None, _out_ptr(y), ws.ptr, ws.nbytes,
        _stream(stream), int(path) | (LORA_FLAG_STATIC_WEIGHTS if static_weights else 0)), "lora_linear")
    return y


def lora_layers_workspace_size(M: int, max_N: int, num_adapters: int, num_layers: int) -> int:
    return int(load_library().lora_layers_workspace_size(M, max_N, num_adapters, num_layers))


class LayersWorkspace(Workspace):
    """A zero-initialised device workspace for lora_linear_layers."""

    def __init__(self, M: int, max_N: int, num_adapters: int, num_layers: int, device="cuda"):
        self.nbytes = lora_layers_workspace_size(M, max_N, num_adapters, num_layers)
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)


def lora_linear_layers(layers: Sequence[tuple], ids: torch.Tensor, ws: Workspace,
                       segs: Optional[lora_segments_t] = None, stream=None) -> List[torch.Tensor]:
    """Several LoRA layers of one step in one launch.  ``layers``: tuples
    (x, W, bias, pool, scale) or (x, W, bias, pool, scale, y); returns the
    outputs y_l = x_l W_l^T + bias_l + scale_l (x_l A_id^T) B_id^T."""
    n = len(layers)
    arr = (lora_layer_t * max(n, 1))()
    outs, keep = [], []
    for i, ly in enumerate(layers):
        x, W, bias, pool, scale = ly[:5]
        y = ly[5] if len(ly) > 5 and ly[5] is not None else torch.empty(x.shape[0], W.shape[0],
                                                                        dtype=torch.bfloat16, device=x.device)
        arr[i].x, arr[i].W = x.data_ptr(), W.data_ptr()
        arr[i].bias = None if bias is None else bias.data_ptr()
        arr[i].pool = ctypes.addressof(pool.desc)
        arr[i].scale = float(scale)
        arr[i].y = y.data_ptr()
        outs.append(y)
        keep.append(pool)
    M = layers[0][0].shape[0] if n else 0
    _check(load_library().lora_linear_layers(arr, n, M, _ptr(ids), ctypes.byref(segs) if segs is not None else None,
                                             ws.ptr, ws.nbytes, _stream(stream)), "lora_linear_layers")
    return outs


def lora_shrink(x: torch.Tensor, ids: torch.Tensor, pool: LoraPool, ws: Workspace,
                S: Optional[torch.Tensor] = None, s_cols: Optional[int] = None,
                segs: Optional[lora_segments_t] = None, stream=None) -> torch.Tensor:
    """S = x A_id^T (fp32, [M, s_cols], zero past each row's rank and on -1 rows)."""
    M = x.shape[0]
    s_cols = s_cols or max(pool.desc.max_rank, 16)
    if S is None:
        S = torch.empty(M, s_cols, dtype=torch.float32, device=x.device)
    _check(load_library().lora_shrink(
        _ptr(x), M, _ptr(ids), ctypes.byref(pool.desc),
        ctypes.byref(segs) if segs is not None else None, _ptr(S), s_cols, ws.ptr, ws.nbytes,
        _stream(stream)), "lora_shrink")
    return S


def lora_expand(S: torch.Tensor, ids: torch.Tensor, pool: LoraPool, scale: float, y: torch.Tensor,
                ws: Workspace, segs: Optional[lora_segments_t] = None, stream=None) -> torch.Tensor:
    """y += scale * S B_id^T in place (bf16 y, id -1 rows untouched)."""
    M = S.shape[0]
    _check(load_library().lora_expand(
        _ptr(S), S.shape[1], M, _ptr(ids), ctypes.byref(pool.desc),
        ctypes.byref(segs) if segs is not None else None, float(scale), _ptr(y), ws.ptr, ws.nbytes,
        _stream(stream)), "lora_expand")
    return y


def lora_linear_noalloc(x: torch.Tensor, W: torch.Tensor, bias: Optional[torch.Tensor], ids: torch.Tensor,
                        pool: LoraPool, scale: float, y: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """lora_linear for callers that cannot allocate device memory: the
    library's own static scratch array is used instead of a workspace."""
    M = x.shape[0]
    if y is None:
        y = torch.empty(M, W.shape[0], dtype=torch.bfloat16, device=x.device)
    _check(load_library().lora_linear_noalloc(
        _ptr(x), M, _ptr(W), _ptr(bias), _ptr(ids), ctypes.byref(pool.desc), float(scale), _ptr(y),
        _stream(stream)), "lora_linear_noalloc")
    return y


def lora_set_wait_budget(cycles: int):
    """Test knob: the tiled kernel's bounded waits give up after ``cycles``
    SM clock cycles (0: the default, about one second)."""
    _check(load_library().lora_set_wait_budget(int(cycles)), "lora_set_wait_budget")


def lora_get_status(ws: Workspace, stream=None) -> int:
    v = ctypes.c_int32()
    _check(load_library().lora_get_status(ws.ptr, _stream(stream), ctypes.byref(v)), "lora_get_status")
    return v.value


# ---------------------------------------------------------------------------
# mixture of experts
# ---------------------------------------------------------------------------

class MoeWorkspace:
    """Device workspace of the MoE routing and grouped GEMM, zero-filled once
    (the status word starts clear; the routing resets the rest every call)."""

    def __init__(self, M: int, topk: int, num_experts: int, device="cuda"):
        self.nbytes = int(load_library().lora_moe_workspace_size(M, topk, num_experts))
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def lora_moe(x: torch.Tensor, W: torch.Tensor, expert: torch.Tensor, weight: torch.Tensor, ws: MoeWorkspace,
             out: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = sum_j weight[:, j] * x W_{expert[:, j]}^T: routing, grouped GEMM,
    weighted finalize.  x bf16 [M, K], W bf16 [E, N, K], expert int32
    [M, topk], weight fp32 [M, topk]; out (the pairs' rows) and y are made
    when not given."""
    M, K = x.shape
    E, N, _ = W.shape
    topk = expert.shape[1]
    if out is None:
        out = torch.empty(M * topk, N, dtype=torch.bfloat16, device=x.device)
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check(load_library().lora_moe(_ptr(x), M, K, _ptr(W), N, _ptr(expert), _ptr(weight), E, topk, _ptr(out),
                                   _ptr(y), ws.ptr, ws.nbytes, _stream(stream)), "lora_moe")
    return y


def lora_moe_route(expert: torch.Tensor, num_experts: int, ws: MoeWorkspace, stream=None):
    M, topk = expert.shape
    _check(load_library().lora_moe_route(_ptr(expert), M, topk, num_experts, ws.ptr, ws.nbytes, _stream(stream)),
           "lora_moe_route")


def lora_moe_gemm(x: torch.Tensor, W: torch.Tensor, topk: int, ws: MoeWorkspace, out: torch.Tensor, stream=None):
    """The grouped GEMM alone over the routing in ws: out [M * topk, N] bf16,
    each routed pair's row x[t] W_e^T (rows of dropped slots untouched)."""
    M, K = x.shape
    E, N, _ = W.shape
    _check(load_library().lora_moe_gemm(_ptr(x), M, K, _ptr(W), N, E, topk, _ptr(out), ws.ptr, ws.nbytes,
                                         _stream(stream)), "lora_moe_gemm")


def lora_moe_check_route(expert: torch.Tensor, num_experts: int, ws: MoeWorkspace, stream=None):
    """Enqueue the device check of the routing in ws against expert int32
    [M, topk]; its verdict is the LORA_DEV_CHECK bit of lora_get_status."""
    M, topk = expert.shape
    _check(load_library().lora_moe_check_route(_ptr(expert), M, topk, num_experts, ws.ptr, ws.nbytes,
                                               _stream(stream)), "lora_moe_check_route")


def moe_routing_layout(M: int, topk: int, num_experts: int) -> dict:
    """Byte offsets of the routing's arrays in a MoE workspace, in the order
    lora_moe_workspace_size lays them out (each region 256-byte aligned)."""
    P, E = M * topk, num_experts
    max_mtiles = (P + 127) // 128 + E
    sizes = [("counters", (8 + 8) * 4), ("perm", max(P, 1) * 4), ("offsets", (E + 2) * 4),
             ("seg_id", max(E, 1) * 4), ("seg_start", max(E, 1) * 4), ("seg_len", max(E, 1) * 4),
             ("seg_rank", max(E, 1) * 4), ("num_segments", 4), ("hdr", 16 * 4), ("perm_pad", max_mtiles * 128 * 4),
             ("mt_expert", max_mtiles * 4)]
    out, o = {}, 0
    for name, n in sizes:
        out[name] = o
        o = (o + n + 255) & ~255
    out["max_mtiles"] = max_mtiles
    return out


def moe_routing_to_host(ws: MoeWorkspace, M: int, topk: int, num_experts: int):
    """The routing's perm over the pairs and its bucket offsets (CPU int32)."""
    P = M * topk
    base = ws.buf

    def grab(off, n):
        return base[off:off + 4 * n].view(torch.int32).cpu()

    lay = moe_routing_layout(M, topk, num_experts)
    return grab(lay["perm"], P), grab(lay["offsets"], num_experts + 2)
