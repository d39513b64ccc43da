"""lora_linear_layers: several LoRA layers of one step in one launch, sharing
one segment table ("vLLM-Ascend dynamic LoRA" §1.2 end, §3.2).  Every layer's
output is compared element by element with the fp64 oracle of that layer
(the oracle has no notion of a launch: a layer is a layer), with the same
bar as the other parity tests: |gpu - oracle| <= 2e-2 (1 + |oracle|)."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

TOL = 2e-2


def _assert_close(gpu, ref, what, rows=None):
    g = gpu.detach().float().cpu().double().numpy()
    if rows is not None:
        g = g[rows]
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    bad = ~(e <= TOL)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(e):.3e}"


def _layers(M, shapes, ranks, seed, ids=None, p_base=0.1, factors=False, slices=None):
    """Workloads of one step: the same ids and adapter ranks, each layer its
    own K, N and values.  slices: per layer, output slice widths (merged
    projections; every layer the same count)."""
    base = workloads.make_custom(M, shapes[0][0], shapes[0][1], ranks, seed=seed, ids=ids, p_base=p_base)
    out = []
    for j, (K, N) in enumerate(shapes):
        asc = "random" if factors else None
        if slices:
            wl = workloads.make_sliced(M, K, slices[j], ranks, seed=seed + 100 + j, ids=base.ids.clone(),
                                       scale=1.0 + 0.25 * j, adapter_scale=asc)
        else:
            wl = workloads.make_custom(M, K, N, ranks, seed=seed + 100 + j, ids=base.ids.clone(),
                                       scale=1.0 + 0.25 * j, adapter_scale=asc)
        out.append(wl)
    return out


def _dev(wl):
    d = "cuda"
    if wl.slices:
        pool = L.build_pool_sliced(wl.A_s, wl.B_s, wl.K, wl.slices, d, adapter_scale=wl.adapter_scale)
    else:
        pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    return dict(x=wl.x.to(d), W=wl.W.to(d), bias=None if wl.bias is None else wl.bias.to(d), pool=pool,
                y=torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device=d))


def _run(wls, devs, ws, ids, segs=None):
    for d in devs:
        d["y"].fill_(float("nan"))
    L.lora_linear_layers([(d["x"], d["W"], d["bias"], d["pool"], wl.scale, d["y"]) for wl, d in zip(wls, devs)],
                         ids, ws, segs=segs)
    return L.lora_get_status(ws)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 40, 300])
def test_layers_match_oracle(M):
    """Four layers of other K and N (an attention block's projections in
    small): every output against its layer's oracle, two calls in a row on
    one workspace."""
    shapes = [(256, 512), (256, 128), (256, 128), (512, 384)]
    wls = _layers(M, shapes, [16, 32, 64, 48, 16], seed=31)
    devs = [_dev(wl) for wl in wls]
    ids = wls[0].ids.to("cuda")
    ws = L.LayersWorkspace(M, max(n for _, n in shapes), wls[0].num_adapters, len(wls))
    refs = [oracle.lora_linear(wl) for wl in wls]
    for call in range(2):
        assert _run(wls, devs, ws, ids) == 0
        for j, (d, ref) in enumerate(zip(devs, refs)):
            _assert_close(d["y"], ref, f"M={M} call {call} layer {j}")


@pytest.mark.gpu
def test_layers_prebuilt_table_factors_and_bad_ids():
    """A table built once by lora_build_segments for the step; per-adapter
    factors that differ between layers; ids outside [-1, A) (treated as -1,
    flagged)."""
    M = 260
    shapes = [(384, 256), (256, 512), (128, 256)]
    wls = _layers(M, shapes, [32, 16, 64], seed=47, factors=True)
    bad = wls[0].ids.clone()
    bad[::13] = 7
    bad[5::17] = -3
    wls = [dataclasses.replace(wl, ids=bad.clone()) for wl in wls]
    devs = [_dev(wl) for wl in wls]
    ids = bad.to("cuda")
    ws = L.LayersWorkspace(M, 512, wls[0].num_adapters, len(wls))
    segs = L.lora_build_segments(ids, devs[0]["pool"], ws)
    status = _run(wls, devs, ws, ids, segs=segs)
    assert status == L.LORA_DEV_BAD_ID
    for j, d in enumerate(devs):
        _assert_close(d["y"], oracle.lora_linear(wls[j]), f"layer {j}")


@pytest.mark.gpu
def test_layers_merged_outputs():
    """Every layer a merged projection of two output slices (slice widths
    differ between layers; the slice count must not)."""
    M = 200
    slices = [[256, 256], [512, 256], [256, 512]]
    shapes = [(256, sum(s)) for s in slices]
    wls = _layers(M, shapes, [16, 32, 16], seed=53, slices=slices)
    devs = [_dev(wl) for wl in wls]
    ids = wls[0].ids.to("cuda")
    ws = L.LayersWorkspace(M, max(sum(s) for s in slices), wls[0].num_adapters, len(wls))
    assert _run(wls, devs, ws, ids) == 0
    for j, d in enumerate(devs):
        _assert_close(d["y"], oracle.lora_linear(wls[j]), f"merged layer {j}")


@pytest.mark.gpu
def test_layers_attention_block_prefill_sampled():
    """The bench's step: the prefill config's ids and adapters, four
    projections (K = 4096; N = 4096, 1024, 1024, 4096), on sampled rows."""
    base = workloads.make_config("prefill")
    shapes = [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096)]
    wls = [workloads.make_custom(base.M, K, N, base.ranks, seed=2000 + j, ids=base.ids.clone())
           for j, (K, N) in enumerate(shapes)]
    devs = [_dev(wl) for wl in wls]
    ids = base.ids.to("cuda")
    ws = L.LayersWorkspace(base.M, 4096, base.num_adapters, len(wls))
    assert _run(wls, devs, ws, ids) == 0
    rng = np.random.default_rng(3)
    rows = sorted(set([0, base.M - 1] + [int(r) for r in rng.integers(0, base.M, 14)]))
    for j, d in enumerate(devs):
        _assert_close(d["y"], oracle.lora_linear(wls[j], rows=rows), f"projection {j}", rows=rows)


@pytest.mark.gpu
def test_layers_one_layer_equals_lora_linear_schedule_choice_free():
    """One layer through lora_linear_layers and through lora_linear (tiled):
    both within the bar of the oracle."""
    wl = workloads.make_custom(333, 320, 640, [16, 64], seed=61)
    d = _dev(wl)
    ids = wl.ids.to("cuda")
    ws = L.LayersWorkspace(wl.M, wl.N, wl.num_adapters, 1)
    assert _run([wl], [d], ws, ids) == 0
    ref = oracle.lora_linear(wl)
    _assert_close(d["y"], ref, "layers call")
    ws1 = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y = L.lora_linear(d["x"], d["W"], d["bias"], ids, d["pool"], wl.scale, ws1, path=L.LORA_PATH_TILED)
    _assert_close(y, ref, "lora_linear")


def _desc_pool(N, K, A, max_rank=64, a_rows=None, b_panels=None, slices=0):
    desc = L.lora_pool_t()
    desc.N, desc.K, desc.num_adapters, desc.max_rank = N, K, A, max_rank
    if A:
        desc.a_pool = desc.b_pool = desc.a_offset = desc.b_offset = desc.rank = 4096
        desc.a_elems = (a_rows or max_rank) * K
        desc.b_elems = (b_panels or max_rank // 16) * 16 * N
    desc.num_slices = slices
    return desc


def test_layers_host_checks():
    """Refusals that the host makes before anything is enqueued (no GPU)."""
    lib = L.load_library()
    assert L.lora_layers_workspace_size(1024, 4096, 40, 4) > L.lora_layers_workspace_size(1024, 4096, 40, 1)
    assert L.lora_layers_workspace_size(1024, 4096, 40, 0) == 0
    assert L.lora_layers_workspace_size(1024, 4096, 40, L.LORA_MAX_LAYERS + 1) == 0
    assert L.lora_layers_workspace_size(-1, 4096, 40, 2) == 0

    def call(pools, n=None, M=64):
        n = len(pools) if n is None else n
        arr = (L.lora_layer_t * max(len(pools), 1))()
        for i, pd in enumerate(pools):
            arr[i].x = arr[i].W = arr[i].y = 4096
            arr[i].pool = ctypes.addressof(pd)
            arr[i].scale = 1.0
        return lib.lora_linear_layers(arr, n, M, None, None, None, 0, None)

    a, b = _desc_pool(512, 256, 4), _desc_pool(256, 512, 4)
    assert call([a, b], n=0) == L.LORA_ERR_SHAPE
    assert call([a] * 9) == L.LORA_ERR_SHAPE
    assert lib.lora_linear_layers(None, 1, 64, None, None, None, 0, None) == L.LORA_ERR_NULL
    # pools that one table cannot describe: other adapter count, max rank,
    # pool rows or slice count
    assert call([a, _desc_pool(256, 512, 5)]) == L.LORA_ERR_SHAPE
    assert call([a, _desc_pool(256, 512, 4, max_rank=32)]) == L.LORA_ERR_SHAPE
    assert call([a, _desc_pool(256, 512, 4, a_rows=128)]) == L.LORA_ERR_SHAPE
    assert call([a, _desc_pool(512, 256, 4, slices=2)]) == L.LORA_ERR_SHAPE
    # consistent pools: M == 0 is a no-op; then the missing ids / workspace
    assert call([a, b], M=0) == L.LORA_OK
    assert call([a, b]) == L.LORA_ERR_NULL
