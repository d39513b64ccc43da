"""Parity of e4m3 adapter pools (8-bit codes, one dequant factor per adapter
and factor) with the fp64 oracle, on every schedule and entry point.

The kernels widen the codes to bf16 exactly and fold the factors into the
per-adapter factor that scales S before its one bf16 rounding, so the bar is
the one of the bf16 pools: |gpu - oracle| <= 2e-2 (1 + |oracle|).
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-2


def assert_close(gpu, ref, tol=TOL, what="", rows=None):
    g = gpu.detach().float().cpu().double().numpy()
    if rows is not None:
        g = g[rows]
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    bad = ~(e <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(e):.3e}"


def dev8(wl8, widened=True):
    d = "cuda"
    pool = L.build_pool_e4m3(wl8.A8, wl8.B8, wl8.deq, wl8.K, wl8.N, d, adapter_scale=wl8.adapter_scale,
                             widened=widened)
    return dict(x=wl8.x.to(d), W=wl8.W.to(d), bias=None if wl8.bias is None else wl8.bias.to(d),
                ids=wl8.ids.to(d), pool=pool)


def run(wl8, dev, path, static=False, segs=False):
    ws = L.Workspace(wl8.M, wl8.N, wl8.num_adapters)
    y = torch.full((wl8.M, wl8.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    sg = L.lora_build_segments(dev["ids"], dev["pool"], ws) if segs else None
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl8.scale, ws, y=y, path=path,
                  static_weights=static, segs=sg)
    return y, L.lora_get_status(ws)


SCHEDULES = [(40, L.LORA_PATH_STREAM), (40, L.LORA_PATH_SPLITK), (100, L.LORA_PATH_SPLITK),
             (300, L.LORA_PATH_TILED), (40, L.LORA_PATH_AUTO), (300, L.LORA_PATH_AUTO)]


@pytest.mark.parametrize("M,path", SCHEDULES)
def test_e4m3_every_schedule(M, path):
    wl8 = workloads.to_e4m3(workloads.make_custom(M, 512, 384, [16, 32, 64, 48, 16], seed=400 + M, p_base=0.15,
                                                  adapter_scale="random"))
    dev = dev8(wl8)
    y, status = run(wl8, dev, path)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl8), what=f"M={M} path={path}")


@pytest.mark.parametrize("static", [False, True])
def test_e4m3_decode_config(static):
    """The decode config's adapters as e4m3: the whole output, with and
    without static weights, and twice on one workspace."""
    wl8 = workloads.to_e4m3(workloads.make_config("decode"))
    dev = dev8(wl8, widened=False)   # the decode-sized schedule reads the 8-bit pool itself
    ref = oracle.lora_linear(wl8)
    ws = L.Workspace(wl8.M, wl8.N, wl8.num_adapters)
    for call in range(2):
        y = torch.full((wl8.M, wl8.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl8.scale, ws, y=y,
                      static_weights=static)
        assert L.lora_get_status(ws) == 0
        assert_close(y, ref, what=f"decode call {call}")


def test_e4m3_prebuilt_table_and_bad_ids():
    wl8 = workloads.to_e4m3(workloads.make_custom(260, 256, 512, [32, 16, 64], seed=431, adapter_scale="random"))
    bad = wl8.ids.clone()
    bad[::11] = 9
    bad[4::13] = -4
    wl8 = dataclasses.replace(wl8, ids=bad)
    dev = dev8(wl8)
    y, status = run(wl8, dev, L.LORA_PATH_AUTO, segs=True)
    assert status == L.LORA_DEV_BAD_ID
    assert_close(y, oracle.lora_linear(wl8), what="prebuilt table, bad ids")


def test_e4m3_shrink_and_expand():
    """The standalone products: S = x A^T with A = a_deq e4m3(A8) (fp32 out),
    and y += scale s_i S B^T with B = b_deq e4m3(B8)."""
    wl8 = workloads.to_e4m3(workloads.make_custom(200, 256, 264, [16, 48, 64, 32], seed=443, id_mode="runs",
                                                  p_base=0.2, adapter_scale=[2.0, 0.5, -0.75, 1.5]))
    dev = dev8(wl8)
    ws = L.Workspace(wl8.M, wl8.N, wl8.num_adapters)
    S = torch.full((wl8.M, 64), float("nan"), dtype=torch.float32, device="cuda")
    L.lora_shrink(dev["x"], dev["ids"], dev["pool"], ws, S=S, s_cols=64)
    assert_close(S, oracle.shrink(wl8, 64), tol=1e-3, what="e4m3 shrink")
    Sin = workloads.random_fp32((wl8.M, 64), seed=17)
    y0 = workloads.random_fp32((wl8.M, wl8.N), seed=18).to(torch.bfloat16)
    y = y0.to("cuda")
    L.lora_expand(Sin.to("cuda"), dev["ids"], dev["pool"], 1.25, y, ws)
    assert_close(y, oracle.expand(wl8, Sin, y0, scale=1.25), what="e4m3 expand")


def test_e4m3_layers_one_launch():
    M = 300
    base = workloads.make_custom(M, 256, 256, [16, 32, 64], seed=451)
    wls = [workloads.to_e4m3(workloads.make_custom(M, K, N, [16, 32, 64], seed=452 + j, ids=base.ids.clone(),
                                                   scale=1.0 + 0.5 * j))
           for j, (K, N) in enumerate([(256, 512), (384, 256), (256, 256)])]
    devs = [dev8(wl) for wl in wls]
    ws = L.LayersWorkspace(M, 512, 3, len(wls))
    outs = L.lora_linear_layers([(d["x"], d["W"], d["bias"], d["pool"], wl.scale) for wl, d in zip(wls, devs)],
                                devs[0]["ids"], ws)
    assert L.lora_get_status(ws) == 0
    for j, (wl, y) in enumerate(zip(wls, outs)):
        assert_close(y, oracle.lora_linear(wl), what=f"e4m3 layer {j}")


def test_e4m3_widening_needs_its_scratch():
    """The schedules that widen the pool refuse a pool without scratch."""
    wl8 = workloads.to_e4m3(workloads.make_custom(200, 256, 256, [16, 32], seed=461))
    dev = dev8(wl8, widened=False)
    ws = L.Workspace(wl8.M, wl8.N, wl8.num_adapters)
    with pytest.raises(L.LoraError) as e:
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl8.scale, ws)
    assert e.value.code == L.LORA_ERR_NULL


@pytest.mark.parametrize("path", [L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED])
def test_e4m3_every_code_is_widened_exactly(path):
    """Every finite e4m3 code, read back exactly through a schedule: x is
    one-hot (token t selects K column t), A's first 16 columns hold the 256
    codes (A[j, k] = code 16 j + k), B is the identity (code 0x38 = 1.0),
    factors are 1 and W is zero, so y[t, n] = A[n, t] with no rounding
    anywhere.  Compared with the oracle's decode, bit for bit."""
    M, K, N, r = 16, 256, 16, 16
    codes = torch.arange(256, dtype=torch.int64).reshape(16, 16)
    codes[(codes & 0x7F) == 0x7F] = 0          # the two NaN codes
    A8 = torch.zeros(r, K, dtype=torch.uint8)
    A8[:, :16] = codes.to(torch.uint8)
    B8 = torch.zeros(N, r, dtype=torch.uint8)
    B8[torch.arange(N), torch.arange(N)] = 0x38
    pool = L.build_pool_e4m3([A8], [B8], [(1.0, 1.0)], K, N, "cuda")
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.arange(M)] = 1.0
    W = torch.zeros(N, K, dtype=torch.bfloat16)
    ids = torch.zeros(M, dtype=torch.int32)
    ws = L.Workspace(M, N, 1)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(x.cuda(), W.cuda(), None, ids.cuda(), pool, 1.0, ws, y=y, path=path)
    assert L.lora_get_status(ws) == 0
    want = torch.tensor([[oracle.e4m3_to_f64(int(codes[n, t])) for n in range(N)] for t in range(M)],
                        dtype=torch.float64)
    got = y.double().cpu()
    assert torch.equal(got, want), f"path {path}: {int((got != want).sum())} codes differ"
