"""Parity of the tiled schedule at a few hundred to a thousand tokens with the
fp64 oracle: several token tiles, a ragged last tile, shrink jobs with odd
and large numbers of rank panels, stream-K (the last partial wave split
along K) twice on one workspace, a prebuilt table reused call after call
with per-adapter factors, invalid ids, merged slices, several layers in one
launch, the standalone products and e4m3 pools.  Bar: |gpu - oracle| <=
2e-2 (1 + |oracle|), outputs NaN-prefilled.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-2


def to_dev(wl):
    d = "cuda"
    if wl.slices:
        pool = L.build_pool_sliced(wl.A_s, wl.B_s, wl.K, wl.slices, d, adapter_scale=wl.adapter_scale)
    elif wl.A8 is not None:
        pool = L.build_pool_e4m3(wl.A8, wl.B8, wl.deq, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    else:
        pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    return dict(x=wl.x.to(d), W=wl.W.to(d), bias=None if wl.bias is None else wl.bias.to(d),
                ids=wl.ids.to(d), pool=pool)


def assert_close(gpu, ref, tol=TOL, what=""):
    g = gpu.detach().float().cpu().double().numpy()
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    bad = ~(e <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(e):.3e}"


def linear(wl, dev, ws=None, path=L.LORA_PATH_AUTO, segs=None):
    ws = ws or L.Workspace(wl.M, wl.N, wl.num_adapters)
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, path=path,
                  segs=segs)
    return y, L.lora_get_status(ws)


@pytest.mark.parametrize("M", [511, 512, 600, 700, 1000])
def test_tiled_ragged_last_tile(M):
    """Token counts around 512 and ragged last tiles (600: 88 rows; 700: 60)."""
    wl = workloads.make_custom(M, 384, 768, [16, 48, 64, 32, 16], seed=900 + M, p_base=0.1, scale=0.75)
    dev = to_dev(wl)
    y, status = linear(wl, dev)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what=f"M={M}")


@pytest.mark.parametrize("ranks,mode", [([16, 48, 16, 16, 48], "runs"),   # 1 or 3 panels per segment
                                        ([64] * 6, "uniform"),             # 24 panels a tile: jobs of 16 + 8
                                        ([16] * 19, "uniform"),            # 19 panels: 16 + 3
                                        ([32], "single")])
def test_tiled_shrink_jobs_with_odd_panel_counts(ranks, mode):
    wl = workloads.make_custom(768, 256, 512, ranks, seed=len(ranks) * 7, id_mode=mode, p_base=0.05)
    dev = to_dev(wl)
    y, status = linear(wl, dev, path=L.LORA_PATH_TILED)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what=f"ranks {ranks}")


def test_tiled_stream_k_twice_on_one_workspace():
    """Fewer output tiles than CTAs: the tiles are split along K (each tail
    piece stores its partial sums in its CTA's scratch slot); the scratch
    and counters must be clean for the second call."""
    wl = workloads.make_custom(1024, 1024, 2048, [16, 32, 64, 48] * 2, seed=931, id_mode="runs", p_base=0.1)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    for call in range(2):
        y, status = linear(wl, dev, ws=ws, path=L.LORA_PATH_TILED)
        assert status == 0
        assert_close(y, ref, what=f"stream-K call {call}")


def test_tiled_prebuilt_table_repeated_calls_adapter_factors():
    wl = workloads.make_custom(900, 512, 640, [64, 16, 32, 48, 16, 64], seed=941, p_base=0.2,
                               adapter_scale="random", scale=1.5)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    for call in range(3):
        y, status = linear(wl, dev, ws=ws, segs=segs)
        assert status == 0
        assert_close(y, ref, what=f"prebuilt call {call}")


def test_tiled_all_base_and_bad_ids():
    wl = workloads.make_custom(640, 256, 512, [16, 32], seed=951, id_mode="all_base")
    dev = to_dev(wl)
    y, status = linear(wl, dev)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what="all base")
    wl = workloads.make_custom(640, 256, 512, [16, 32, 64], seed=952)
    bad = wl.ids.clone()
    bad[::9] = 7
    bad[3::13] = -5
    wl.ids.copy_(bad)
    dev = to_dev(wl)
    y, status = linear(wl, dev)
    assert status == L.LORA_DEV_BAD_ID
    assert_close(y, oracle.lora_linear(wl), what="bad ids")


def test_tiled_sliced_output():
    wl = workloads.make_sliced(1024, 512, [512, 256, 256], [16, 32, 16], seed=961, p_base=0.15)
    dev = to_dev(wl)
    y, status = linear(wl, dev)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what="sliced")


def test_tiled_layers_one_launch():
    M = 800
    base = workloads.make_custom(M, 256, 256, [16, 32, 64], seed=971)
    wls = [workloads.make_custom(M, K, N, [16, 32, 64], seed=972 + j, ids=base.ids.clone(), scale=1.0 + 0.5 * j)
           for j, (K, N) in enumerate([(256, 768), (512, 256), (256, 512)])]
    devs = [to_dev(wl) for wl in wls]
    ws = L.LayersWorkspace(M, 768, 3, len(wls))
    outs = L.lora_linear_layers([(d["x"], d["W"], d["bias"], d["pool"], wl.scale) for wl, d in zip(wls, devs)],
                                devs[0]["ids"], ws)
    assert L.lora_get_status(ws) == 0
    for j, (wl, y) in enumerate(zip(wls, outs)):
        assert_close(y, oracle.lora_linear(wl), what=f"layer {j}")


def test_tiled_shrink_and_expand_alone():
    wl = workloads.make_custom(900, 1024, 520, [16, 48, 64, 32], seed=981, id_mode="runs", p_base=0.2)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = torch.full((wl.M, 64), float("nan"), dtype=torch.float32, device="cuda")
    L.lora_shrink(dev["x"], dev["ids"], dev["pool"], ws, S=S, s_cols=64)
    assert_close(S, oracle.shrink(wl, 64), tol=1e-3, what="shrink")
    Sin = workloads.random_fp32((wl.M, 64), seed=21)
    y0 = workloads.random_fp32((wl.M, wl.N), seed=22).to(torch.bfloat16)
    y = y0.to("cuda")
    L.lora_expand(Sin.to("cuda"), dev["ids"], dev["pool"], 1.25, y, ws)
    assert_close(y, oracle.expand(wl, Sin, y0, scale=1.25), what="expand")
    base_rows = (wl.ids < 0).nonzero().flatten()
    assert torch.equal(y[base_rows.to("cuda")].cpu(), y0[base_rows])


def test_tiled_e4m3_pool():
    wl8 = workloads.to_e4m3(workloads.make_custom(700, 512, 384, [16, 32, 64, 48, 16], seed=991, p_base=0.15,
                                                  adapter_scale="random"))
    dev = to_dev(wl8)
    y, status = linear(wl8, dev)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl8), what="e4m3")
