"""CPU checks of the C ABI boundary: the library loads, exports every symbol
that include/lora.h declares, and its host-only helpers behave.  No compute
call runs here (no GPU)."""
import ctypes
import os
import re

import pytest
import torch

from segmented_gemm_gb300 import lora as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from segmented_gemm_gb300 import build
        build.build()
    return L.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(L.EXPORTS)


def test_pool_layout_rank_grouped(lib):
    a_off, b_off, rpad, ae, be = L.lora_pool_layout([8, 64, 16, 33, 20], 4096, 1024)
    assert rpad == [16, 64, 16, 48, 32]
    # grouped by padded rank: 16s (ids 0, 2), then 32 (id 4), 48 (id 3), 64 (id 1)
    order = sorted(range(5), key=lambda i: a_off[i])
    assert order == [0, 2, 4, 3, 1]
    assert all(a_off[i] % 4096 == 0 and b_off[i] % 16 == 0 for i in range(5))
    assert ae == sum(rpad) * 4096 and be == sum(rpad) * 1024
    # contiguous, non-overlapping
    for x, y in zip(order, order[1:]):
        assert a_off[y] == a_off[x] + rpad[x] * 4096
        assert b_off[y] == b_off[x] + rpad[x] * 1024


@pytest.mark.parametrize("ranks,K,N,code", [([0], 64, 64, L.LORA_ERR_RANK), ([129], 64, 64, L.LORA_ERR_RANK),
                                            ([16], 60, 64, L.LORA_ERR_SHAPE),
                                            ([16], 64, 0, L.LORA_ERR_SHAPE)])
def test_pool_layout_errors(lib, ranks, K, N, code):
    with pytest.raises(L.LoraError) as e:
        L.lora_pool_layout(ranks, K, N)
    assert e.value.code == code


def test_workspace_size_monotone(lib):
    a = L.lora_workspace_size(1024, 4096, 40)
    b = L.lora_workspace_size(8192, 4096, 40)
    assert 0 < a < b
    assert L.lora_workspace_size(-1, 64, 1) == 0


def test_status_strings(lib):
    for c in range(11):
        assert L.status_string(c)
    assert "unknown" in L.status_string(99)


def test_null_arguments_rejected_without_gpu(lib):
    # host-side validation runs before anything touches the device
    rc = lib.lora_linear_ex(None, 4, None, None, None, None, ctypes.c_float(1.0), None, None, None, 0, None, 0)
    assert rc == L.LORA_ERR_NULL
    rc = lib.lora_linear_ex(None, -1, None, None, None, None, ctypes.c_float(1.0), None, None, None, 0, None, 0)
    assert rc == L.LORA_ERR_SHAPE


def _fake_pool(adapter_scale):
    # addresses are never dereferenced: validation rejects the call first
    return L.lora_pool_t(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64 * 16, 64 * 16, 1, 16, 64, 64, adapter_scale)


def test_adapter_factors_need_ids_and_alignment_without_gpu(lib):
    f = ctypes.c_float(1.0)
    # factors are looked up by token id: a prebuilt table alone is not enough
    pool = _fake_pool(0x6000)
    rc = lib.lora_linear_ex(0x7000, 4, 0x8000, None, None, ctypes.byref(pool), f, None, 0x9000, 0xA000, 1 << 20,
                            None, 0)
    assert rc == L.LORA_ERR_NULL
    rc = lib.lora_expand(0x7000, 16, 4, None, ctypes.byref(pool), None, f, 0x9000, 0xA000, 1 << 20, None)
    assert rc == L.LORA_ERR_NULL
    # the fp32 factor table must be 4-byte aligned
    pool = _fake_pool(0x6002)
    rc = lib.lora_linear_ex(0x7000, 4, 0x8000, None, 0xB000, ctypes.byref(pool), f, None, 0x9000, 0xA000, 1 << 20,
                            None, 0)
    assert rc == L.LORA_ERR_ALIGN


def _fake_sliced_pool(starts, max_rank=48, num_slices=None):
    pool = L.lora_pool_t(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64 * 48, 768 * 48, 1, max_rank, 64, 768, None)
    pool.num_slices = len(starts) - 1 if num_slices is None else num_slices
    for s, v in enumerate(starts):
        pool.slice_start[s] = v
    return pool


@pytest.mark.parametrize("starts,max_rank,code", [
    ([0, 100, 768], 32, L.LORA_ERR_SHAPE),          # inner boundary off the 256-column grid
    ([0, 512, 256, 768], 48, L.LORA_ERR_SHAPE),     # not increasing
    ([0, 256, 512], 48, L.LORA_ERR_SHAPE),          # does not end at N
    ([0, 256, 512, 768], 32, L.LORA_ERR_RANK),      # rank not whole panels per slice
    ([0, 256, 512, 768, 768, 768], 48, L.LORA_ERR_SHAPE),   # more slices than LORA_MAX_SLICES
])
def test_sliced_pool_rejected_without_gpu(lib, starts, max_rank, code):
    pool = _fake_sliced_pool(starts, max_rank) if len(starts) <= 5 else _fake_sliced_pool(starts[:5], max_rank, 5)
    rc = lib.lora_linear_ex(0x7000, 4, 0x8000, None, 0xB000, ctypes.byref(pool), ctypes.c_float(1.0), None, 0x9000,
                            0xA000, 1 << 20, None, 0)
    assert rc == code


def test_pool_layout_accepts_rank_128(lib):
    a_off, b_off, rpad, ae, be = L.lora_pool_layout([128, 100, 16], 256, 512)
    assert rpad == [128, 112, 16]
    assert ae == (128 + 112 + 16) * 256 and be == (128 + 112 + 16) * 512


@pytest.mark.parametrize("M,topk,E", [(1, 1, 1), (37, 2, 5), (2048, 8, 64), (40000, 8, 1024)])
def test_moe_workspace_holds_every_routing_region(lib, M, topk, E):
    """The MoE workspace has room for what the routing and the grouped GEMM
    write: perm over the pairs, bucket offsets, the segment table, the padded
    expert order with each tile's expert, and the per-chunk bucket counts of
    the routing (chunks of 1024 pairs or more, at most 256 of them)."""
    def cdiv(a, b):
        return -(-a // b)
    P = M * topk
    tiles = cdiv(P, 128) + E
    chunk = max(1024, cdiv(cdiv(P, 256), 256) * 256)
    nchunks = max(1, cdiv(P, chunk))
    assert nchunks <= 256
    need = 4 * (P + (E + 2) + 4 * E + 1 + tiles * 128 + tiles + nchunks * (E + 1))
    size = lib.lora_moe_workspace_size(M, topk, E)
    assert size >= need
    assert lib.lora_moe_workspace_size(M, topk, E + 1) > size            # more experts, more room
    assert lib.lora_moe_workspace_size(-1, topk, E) == 0
    assert lib.lora_moe_workspace_size(M, 0, E) == 0


def test_moe_host_errors_without_gpu(lib):
    # shapes are checked before anything touches the device
    assert lib.lora_moe_route(None, 4, 2, 0, None, 0, None) == L.LORA_ERR_SHAPE      # no experts
    assert lib.lora_moe_route(None, 4, 3, 2, None, 0, None) == L.LORA_ERR_SHAPE      # topk > E
    assert lib.lora_moe_route(None, 4, 2, 2000, None, 0, None) == L.LORA_ERR_SHAPE   # E > LORA_MAX_ADAPTERS
    assert lib.lora_moe_route(None, 4, 2, 4, None, 0, None) == L.LORA_ERR_NULL
    assert lib.lora_moe_route(None, 0, 2, 4, None, 0, None) == L.LORA_OK             # no tokens: nothing to do
    assert lib.lora_moe_gemm(None, 4, 12, None, 64, 4, 2, None, None, 0, None) == L.LORA_ERR_SHAPE   # K % 8


def test_wait_budget_knob_validates(lib):
    assert lib.lora_set_wait_budget(-1) == L.LORA_ERR_SHAPE
    assert lib.lora_set_wait_budget(1_000_000) == L.LORA_OK
    assert lib.lora_set_wait_budget(0) == L.LORA_OK   # back to the default


def test_debug_library_exports_the_same_symbols(lib):
    """liblora_debug.so (the sources built with LORA_DEBUG) is the same ABI."""
    assert os.path.exists(L.DEBUG_LIB_PATH), "build() makes both libraries"
    dbg = ctypes.CDLL(L.DEBUG_LIB_PATH)
    for n in L.EXPORTS:
        assert hasattr(dbg, n), n


def test_device_status_bits_match_the_header():
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    bits = {m.group(1): 1 << int(m.group(2)) for m in re.finditer(r"\b(LORA_DEV_[A-Z_]+)\s*=\s*1\s*<<\s*(\d+)", src)}
    assert set(bits) == {"LORA_DEV_BAD_ID", "LORA_DEV_TIMEOUT", "LORA_DEV_BAD_POOL", "LORA_DEV_CHECK"}
    for name, v in bits.items():
        assert getattr(L, name) == v, name


def test_check_segments_host_errors_without_gpu(lib):
    seg = L.lora_segments_t()
    pool = _fake_pool(None)
    F = lib.lora_check_segments
    assert F(0x1000, 64, ctypes.byref(pool), None, 0x2000, 1 << 20, None) == L.LORA_ERR_NULL   # no table
    assert F(0x1000, -1, ctypes.byref(pool), ctypes.byref(seg), 0x2000, 1 << 20, None) == L.LORA_ERR_SHAPE
    assert F(None, 64, ctypes.byref(pool), ctypes.byref(seg), 0x2000, 1 << 20, None) == L.LORA_ERR_NULL   # no ids
    assert F(0x1000, 0, ctypes.byref(pool), ctypes.byref(seg), 0x2000, 1 << 20, None) == L.LORA_OK   # M = 0: no-op
    assert F(0x1000, 0, None, ctypes.byref(seg), 0x2000, 1 << 20, None) == L.LORA_ERR_NULL


@pytest.mark.parametrize("M,topk,E", [(1, 1, 1), (37, 2, 5), (2048, 8, 64), (40000, 8, 1024)])
def test_moe_layout_mirror_fits_the_workspace(lib, M, topk, E):
    """The binding's mirror of the routing's layout (the arrays the tests
    read and edit) ends inside the workspace the library sizes."""
    lay = L.moe_routing_layout(M, topk, E)
    order = ["counters", "perm", "offsets", "seg_id", "seg_start", "seg_len", "seg_rank", "num_segments", "hdr",
             "perm_pad", "mt_expert"]
    offs = [lay[k] for k in order]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay["mt_expert"] + 4 * lay["max_mtiles"] <= lib.lora_moe_workspace_size(M, topk, E)


def test_moe_check_route_host_errors_without_gpu(lib):
    F = lib.lora_moe_check_route
    assert F(None, 4, 2, 0, None, 0, None) == L.LORA_ERR_SHAPE      # no experts
    assert F(None, 4, 3, 2, None, 0, None) == L.LORA_ERR_SHAPE      # topk > E
    assert F(None, 4, 2, 4, None, 0, None) == L.LORA_ERR_NULL       # no expert ids
    assert F(None, 0, 2, 4, None, 0, None) == L.LORA_OK             # no tokens: nothing to check
    assert F(0x1000, 4, 2, 4, None, 0, None) == L.LORA_ERR_WORKSPACE


def test_error_codes_and_copy_limit_match_the_header():
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(LORA_ERR_[A-Z_]+)\s*=\s*(\d+)", src)}
    assert len(codes) == 10
    for name, v in codes.items():
        assert getattr(L, name) == v, name
    assert int(re.search(r"#define LORA_MAX_COPIES (\d+)", src).group(1)) == L.LORA_MAX_COPIES
    assert "access" in L.status_string(L.LORA_ERR_ACCESS)


def test_copy_async_host_errors_without_gpu(lib):
    # every check here returns before the library asks the driver anything
    C = L.lora_copy_t
    assert lib.lora_copy_async(None, 0, None) == L.LORA_OK
    assert lib.lora_copy_async(None, 1, None) == L.LORA_ERR_NULL
    assert lib.lora_copy_async((C * 5)(), 5, None) == L.LORA_ERR_SHAPE
    assert lib.lora_copy_async((C * 1)(), -1, None) == L.LORA_ERR_SHAPE
    one = (C * 1)()
    one[0].dst, one[0].src, one[0].bytes = 0x1000, 0x2000, -16
    assert lib.lora_copy_async(one, 1, None) == L.LORA_ERR_SHAPE
    one[0].bytes = 0                                   # an empty entry is skipped
    assert lib.lora_copy_async(one, 1, None) == L.LORA_OK
    one[0].dst, one[0].bytes = None, 64
    assert lib.lora_copy_async(one, 1, None) == L.LORA_ERR_NULL
    for dst, src, nb in ((0x1008, 0x2000, 64), (0x1000, 0x2004, 64), (0x1000, 0x2000, 40)):
        one[0].dst, one[0].src, one[0].bytes = dst, src, nb
        assert lib.lora_copy_async(one, 1, None) == L.LORA_ERR_ALIGN, (dst, src, nb)
    out = ctypes.c_void_p()
    assert lib.lora_device_pointer(None, ctypes.byref(out)) == L.LORA_ERR_NULL
    assert lib.lora_device_pointer(ctypes.c_void_p(0x1000), None) == L.LORA_ERR_NULL


def test_copy_async_binding_checks_its_pairs():
    a, b = torch.zeros(8), torch.zeros(4)
    with pytest.raises(ValueError):
        L.copy_async([(a, b)])                         # sizes differ
    with pytest.raises(ValueError):
        L.copy_async([(a, a)] * (L.LORA_MAX_COPIES + 1))
    with pytest.raises(ValueError):
        L.copy_async([(a[::2], b)])                    # not contiguous
