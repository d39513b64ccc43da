"""lora_linear_noalloc: the fused layer for callers that cannot allocate
device memory (an engine hook handed no workspace, code that may not call
cudaMalloc while it runs).  It uses a scratch array built into the library
instead of a workspace.  Its output must match lora_linear's for the same
inputs, call after call, because the array is shared and keeps the previous
call's contents.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _no_alloc(wl, dev):
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear_noalloc(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, y=y)
    torch.cuda.synchronize()
    return y


def _assert_close(got, ref, what):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    err = np.abs(g - r) / (1.0 + np.abs(r))
    bad = ~(err <= TOL)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(err):.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_no_alloc_matches_lora_linear_twice(name):
    wl = workloads.make_config(name)
    dev = _dev(wl)
    ref = _with_workspace(wl, dev)
    for call in range(2):
        _assert_close(_no_alloc(wl, dev), ref, f"{name} call {call}")


@pytest.mark.gpu
def test_no_alloc_shape_changes_between_calls():
    # Each shape lays the scratch out differently, so every call must clear
    # what the previous one left behind.  The sizes cover the decode-sized,
    # mid-sized and tiled batches.
    shapes = [(32, 512, 1024, [16, 32, 64, 16]), (100, 256, 512, [16, 32]), (300, 256, 384, [16, 64, 32]),
              (32, 512, 1024, [16, 32, 64, 16])]
    for i, (M, K, N, ranks) in enumerate(shapes):
        wl = workloads.make_custom(M, K, N, ranks, seed=700 + i)
        dev = _dev(wl)
        ref = _with_workspace(wl, dev)
        for call in range(2):
            _assert_close(_no_alloc(wl, dev), ref, f"shape {i} call {call}")


def test_no_alloc_rejects_oversize_problem():
    # Checked on the host before anything is enqueued, so no GPU is needed.
    lib = L.load_library()
    M, N, A = 16384, 4096, 1024
    assert L.lora_workspace_size(M, N, A) > L.LORA_NOALLOC_SCRATCH_BYTES
    desc = L.lora_pool_t()
    desc.N, desc.K, desc.num_adapters, desc.max_rank = N, 4096, A, 64
    rc = lib.lora_linear_noalloc(None, M, None, None, None, ctypes.byref(desc), 1.0, None, None)
    assert rc == L.LORA_ERR_CAPACITY
    assert "LORA_NOALLOC_SCRATCH_BYTES" in L.status_string(rc)
