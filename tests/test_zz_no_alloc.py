"""lora_linear_noalloc: the fused layer for callers that cannot allocate
device memory (an engine hook handed no workspace, code that may not call
cudaMalloc while it runs).  It uses a scratch array built into the library
instead of a workspace.  Because the array is shared and keeps the previous
call's contents, every case below makes at least two calls in a row.  Each
call's output is compared element by element with the CPU oracle and with
lora_linear on a caller workspace, both within the parity tolerance.

This file is named so that pytest collects it last.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

TOL = 2e-2


def _dev(wl):
    d = "cuda"
    return dict(x=wl.x.to(d), W=wl.W.to(d), bias=None if wl.bias is None else wl.bias.to(d),
                ids=wl.ids.to(d), pool=L.build_pool(wl.A, wl.B, wl.K, wl.N, d))


def _with_workspace(wl, dev):
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y)
    assert L.lora_get_status(ws) == 0
    return y


def _no_alloc(wl, dev, ids=None):
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear_noalloc(dev["x"], dev["W"], dev["bias"], dev["ids"] if ids is None else ids, dev["pool"],
                          wl.scale, y=y)
    torch.cuda.synchronize()
    return y


def _assert_close(got, ref, what, rows=None):
    g = got.float().cpu().double().numpy()
    if rows is not None:
        g = g[rows]
    r = ref.float().cpu().double().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref)
    err = np.abs(g - r) / (1.0 + np.abs(r))
    bad = ~(err <= TOL)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(err):.3e}"


def _check_two_calls(wl, dev, what, oracle_rows=None):
    ref_ws = _with_workspace(wl, dev)
    ref = oracle.lora_linear(wl, rows=oracle_rows)
    for call in range(2):
        y = _no_alloc(wl, dev)
        _assert_close(y, ref_ws, f"{what} call {call} vs lora_linear")
        _assert_close(y, ref, f"{what} call {call} vs oracle", rows=oracle_rows)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_no_alloc_matches_oracle_and_lora_linear_twice(name):
    wl = workloads.make_config(name)
    _check_two_calls(wl, _dev(wl), name)


@pytest.mark.gpu
def test_no_alloc_tiled_partial_last_wave():
    # M > 128 runs the tiled schedule; here without the split-tile scratch
    # (it never fits the array), while lora_linear on a full workspace splits
    # the partial last wave along K.  Both must agree with the oracle.
    wl = workloads.make_custom(300, 512, 1024, [16, 32, 64, 16, 48], seed=811, scale=2.0)
    _check_two_calls(wl, _dev(wl), "M=300")
    wl = workloads.make_config("prefill")
    rows = sorted(set([0, wl.M - 1] + list(range(5, wl.M, 97))))
    _check_two_calls(wl, _dev(wl), "prefill", oracle_rows=rows)


@pytest.mark.gpu
def test_no_alloc_shape_changes_between_calls():
    # Each shape lays the scratch out differently, so every call must clear
    # what the previous one left behind.  The sizes cover the decode-sized,
    # mid-sized and tiled batches.
    shapes = [(32, 512, 1024, [16, 32, 64, 16]), (100, 256, 512, [16, 32]), (300, 256, 384, [16, 64, 32]),
              (32, 512, 1024, [16, 32, 64, 16])]
    for i, (M, K, N, ranks) in enumerate(shapes):
        wl = workloads.make_custom(M, K, N, ranks, seed=700 + i)
        _check_two_calls(wl, _dev(wl), f"shape {i}")


@pytest.mark.gpu
@pytest.mark.parametrize("M", [32, 100, 300])
def test_no_alloc_bad_ids_do_not_poison_the_next_call(M):
    # A call whose ids hold values outside [-1, num_adapters) treats those
    # tokens as base-only and sets a status bit in the shared array; the next
    # call clears the status and its counters and must be exact again.
    wl = workloads.make_custom(M, 256, 512, [16, 32, 64], seed=900 + M, scale=2.0)
    dev = _dev(wl)
    bad = wl.ids.clone()
    bad[::7] = wl.num_adapters + 3
    bad[3::11] = -5
    wl_bad = dataclasses.replace(wl, ids=bad)
    _assert_close(_no_alloc(wl, dev, ids=bad.to("cuda")), oracle.lora_linear(wl_bad), f"M={M} bad ids vs oracle")
    _check_two_calls(wl, dev, f"M={M} after bad ids")


def _fake_pool(N, K, A, max_rank=64):
    desc = L.lora_pool_t()
    desc.N, desc.K, desc.num_adapters, desc.max_rank = N, K, A, max_rank
    if A:
        # never dereferenced: the checks below all return on the host
        desc.a_pool = desc.b_pool = desc.a_offset = desc.b_offset = desc.rank = 4096
        desc.a_elems, desc.b_elems = max_rank * K, max_rank * N
    return desc


def test_no_alloc_capacity_rule_on_the_host():
    # Checked on the host before anything is enqueued, so no GPU is needed.
    lib = L.load_library()
    # far above the limit
    M, N, A = 16384, 4096, 1024
    assert L.lora_workspace_size(M, N, A) > L.LORA_NOALLOC_SCRATCH_BYTES
    rc = lib.lora_linear_noalloc(None, M, None, None, None, ctypes.byref(_fake_pool(N, 4096, A)), 1.0, None, None)
    assert rc == L.LORA_ERR_CAPACITY
    assert "LORA_NOALLOC_SCRATCH_BYTES" in L.status_string(rc)
    # the MLP down projection (M = 8192, N = 4096, 32 adapters): its full
    # workspace is larger than the array, but its minimal layout fits, so the
    # call passes the capacity check and stops at the null input pointers
    M, N, A = 8192, 4096, 32
    assert L.lora_workspace_size(M, N, A) > L.LORA_NOALLOC_SCRATCH_BYTES
    rc = lib.lora_linear_noalloc(None, M, None, None, None, ctypes.byref(_fake_pool(N, 12288, A)), 1.0, None, None)
    assert rc == L.LORA_ERR_NULL
    # shapes are validated before any layout arithmetic
    rc = lib.lora_linear_noalloc(None, 1 << 40, None, None, None, ctypes.byref(_fake_pool(N, 4096, A)), 1.0,
                                 None, None)
    assert rc == L.LORA_ERR_SHAPE
    rc = lib.lora_linear_noalloc(None, 64, None, None, None, ctypes.byref(_fake_pool(N, 4096, 5000)), 1.0,
                                 None, None)
    assert rc == L.LORA_ERR_SHAPE
    assert L.lora_workspace_size(1 << 40, N, A) == 0
    assert L.lora_workspace_size(64, N, 5000) == 0
