"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Bar: segment tables and permutations bit-exact; outputs within
|gpu - oracle| <= 2e-2 * (1 + |oracle|) per element (bf16 output, fp32
accumulation, S rounded once to bf16 before the second product).
Every output buffer is pre-filled with NaN so an element the kernels never
write fails the comparison.
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


def to_dev(wl):
    d = "cuda"
    if wl.slices:
        pool = L.build_pool_sliced(wl.A_s, wl.B_s, wl.K, wl.slices, d, adapter_scale=wl.adapter_scale)
    else:
        pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    return dict(x=wl.x.to(d), W=wl.W.to(d), bias=None if wl.bias is None else wl.bias.to(d),
                ids=wl.ids.to(d), pool=pool)


def rel_err(gpu, ref):
    g = gpu.detach().float().cpu().double().numpy()
    return np.abs(g - ref) / (1.0 + np.abs(ref))


def assert_close(gpu, ref, tol=TOL, what=""):
    e = rel_err(gpu, ref)
    bad = ~(e <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(e):.3e}"


def run_linear(wl, dev, path=L.LORA_PATH_AUTO, prebuilt=False):
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws) if prebuilt else None
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                  segs=segs, path=path)
    status = L.lora_get_status(ws)
    return y, ws, status


def sample_rows(M, per_tile=3, seed=0):
    rng = np.random.default_rng(seed)
    rows = set([0, M - 1])
    for t0 in range(0, M, 128):
        hi = min(M, t0 + 128)
        rows.update(int(r) for r in rng.integers(t0, hi, size=min(per_tile, hi - t0)))
    return sorted(rows)


def check_segments(wl, dev, ws, segs):
    got = L.segments_to_host(segs, ws, wl.M, wl.num_adapters)
    want = oracle.build_segments(wl.ids.numpy(), wl.num_adapters, wl.ranks)
    assert np.array_equal(got["perm"].numpy(), want["perm"])
    assert np.array_equal(got["bucket_offsets"].numpy(), want["bucket_offsets"])
    assert got["num_segments"] == want["num_segments"]
    for k in ("seg_id", "seg_start", "seg_len", "seg_rank"):
        assert np.array_equal(got[k].numpy(), want[k]), k


# ---------------------------------------------------------------------------
# segment builder: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", workloads.CONFIG_NAMES)
def test_segments_configs(name):
    wl = workloads.make_config(name)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    check_segments(wl, dev, ws, segs)
    assert L.lora_get_status(ws) == 0


@pytest.mark.parametrize("M,A,mode", [(1, 3, "uniform"), (33, 1, "single"), (1000, 7, "runs"),
                                      (4097, 200, "uniform"), (300, 5, "all_base"),
                                      (20000, 1024, "uniform")])
def test_segments_edge(M, A, mode):
    ranks = [16 * (1 + (i % 4)) for i in range(A)]
    ids = None
    if A == 1024:
        g = torch.Generator().manual_seed(3)
        ids = torch.randint(-1, A, (M,), generator=g)
    wl = workloads.make_custom(M, 64, 64, ranks, seed=M + A, ids=ids, id_mode=mode)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    check_segments(wl, dev, ws, segs)


def test_segments_invalid_ids_flagged():
    wl = workloads.make_custom(50, 64, 64, [16, 32], seed=1, id_mode="uniform")
    wl.ids[3] = 7
    wl.ids[9] = -4
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, 2)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    check_segments(wl, dev, ws, segs)      # oracle also sorts them as -1
    assert L.lora_get_status(ws) & L.LORA_DEV_BAD_ID
    assert L.lora_get_status(ws) == 0       # reading clears the word


# ---------------------------------------------------------------------------
# the fused layer
# ---------------------------------------------------------------------------

def test_tiny_config_all_rows_both_paths():
    wl = workloads.make_config("tiny")
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in (L.LORA_PATH_AUTO, L.LORA_PATH_TILED, L.LORA_PATH_SPLITK, L.LORA_PATH_STREAM):
        y, ws, status = run_linear(wl, dev, path)
        assert status == 0
        assert_close(y, ref, what=f"tiny path={path}")


@pytest.mark.parametrize("path", [L.LORA_PATH_TILED, L.LORA_PATH_SPLITK, L.LORA_PATH_STREAM])
@pytest.mark.parametrize("M,K,N,ranks,mode", [
    (1, 64, 64, [16], "single"),
    (7, 200, 136, [8, 40, 64], "uniform"),          # K not a multiple of 64, N ragged
    (100, 320, 520, [16, 32, 48, 64, 20], "uniform"),
    (128, 256, 256, [64] * 6, "uniform"),
    (61, 512, 384, [16] * 40, "uniform"),            # many segments in one tile
    (33, 640, 1032, [48, 16, 64, 32], "uniform"),    # odd number of K blocks, 9 output tiles
    (64, 1024, 2048, [64] * 12 + [16] * 12, "uniform"),
    (16, 4096, 4096, [16, 32, 64] * 7, "uniform"),  # decode shapes, 21 adapters
    (48, 192, 392, [16, 64, 32], "uniform"),         # 3 K blocks (half K unit), N ragged
    (64, 512, 256, [16] * 64, "uniform"),            # ~40 adapters present: shrink slices span 3-4 windows
])
def test_linear_small_shapes(path, M, K, N, ranks, mode):
    if path == L.LORA_PATH_STREAM and (M > 64 or K % 64):
        pytest.skip("streaming schedule serves M <= 64 with K a multiple of 64")
    if path == L.LORA_PATH_SPLITK and M > 128:
        pytest.skip("split-K schedule serves M <= 128")
    wl = workloads.make_custom(M, K, N, ranks, seed=M * 7 + K, id_mode=mode, p_base=0.15, scale=1.5)
    dev = to_dev(wl)
    y, ws, status = run_linear(wl, dev, path)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what=f"M{M} K{K} N{N} path={path}")


@pytest.mark.parametrize("M,K,N,ranks,mode", [
    (300, 320, 520, [16, 32, 48, 64], "runs"),       # several tiles, ragged M tail
    (640, 256, 768, [64] * 5 + [16] * 5, "uniform"),
    (257, 128, 264, [64] * 20, "uniform"),           # > 16 rank panels in a tile: 2 shrink jobs
    (1000, 192, 512, [16, 32], "all_base"),          # base GEMM only
    (513, 256, 256, [32], "single"),
])
def test_linear_tiled_multi_tile(M, K, N, ranks, mode):
    wl = workloads.make_custom(M, K, N, ranks, seed=M + N, id_mode=mode, p_base=0.2, scale=0.75)
    dev = to_dev(wl)
    y, ws, status = run_linear(wl, dev)
    assert status == 0
    assert_close(y, oracle.lora_linear(wl), what=f"M{M} K{K} N{N}")


@pytest.mark.parametrize("M,K,N,ranks", [
    (1280, 256, 2560, [16, 32, 64, 48] * 3),   # ~100 output tiles on the grid: split tiles with one tail each
    (300, 320, 1032, [16, 64]),                # a few tiles over every CTA: many tails, summed by atomics
])
def test_linear_tiled_split_tiles_repeat(M, K, N, ranks):
    """The tiled schedule's last partial wave split along K (partial sums in
    the workspace), twice on one workspace: the scratch must be left clean."""
    wl = workloads.make_custom(M, K, N, ranks, seed=M + 3 * N, id_mode="runs", p_base=0.1, scale=1.25)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    for call in range(2):
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                      path=L.LORA_PATH_TILED)
        assert L.lora_get_status(ws) == 0
        assert_close(y, ref, what=f"split tiles M{M} N{N} call {call}")


def test_linear_no_bias_and_prebuilt_segments():
    wl = workloads.make_custom(200, 256, 320, [16, 64, 32], seed=77, with_bias=False)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in (L.LORA_PATH_AUTO, L.LORA_PATH_TILED):
        y, ws, status = run_linear(wl, dev, path, prebuilt=True)
        assert status == 0
        assert_close(y, ref, what=f"no-bias path={path}")


@pytest.mark.parametrize("M,paths", [(60, "tiled,splitk,stream"), (96, "tiled,splitk"), (300, "tiled")])
def test_linear_repeated_calls_reuse_workspace(M, paths):
    """Counters are left zeroed: the same workspace serves call after call, on
    every schedule that takes the batch size (M = 300 on the tiled schedule
    with a full workspace, so a partial last wave is split along K)."""
    wl = workloads.make_custom(M, 256, 512, [16, 32, 64], seed=5, scale=2.0)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    names = {"tiled": L.LORA_PATH_TILED, "splitk": L.LORA_PATH_SPLITK, "stream": L.LORA_PATH_STREAM}
    for path in (names[n] for n in paths.split(",")):
        ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
        segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
        for _ in range(4):
            y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                          segs=segs, path=path)
            assert_close(y, ref, what=f"repeat path={path}")
        assert L.lora_get_status(ws) == 0


@pytest.mark.parametrize("case", ["mix", "all_base", "four"])
def test_stream_back_to_back_calls(case):
    """Thirty decode-sized calls on one workspace with no host sync between
    them: the window sums and counters a call uses must be back at zero when
    the next one starts (a small pool shrunk whole, no LoRA token, and a
    pool whose windows every token touches)."""
    if case == "mix":
        wl = workloads.make_config("decode")
    elif case == "all_base":
        wl = workloads.make_custom(32, 4096, 4096, [16, 32, 64] * 6, seed=21, id_mode="all_base")
    else:
        wl = workloads.make_custom(32, 4096, 4096, [64, 32, 16, 64], seed=3, p_base=0.0)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    ys = [torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(30)]
    for y in ys:
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                      path=L.LORA_PATH_STREAM)
    assert L.lora_get_status(ws) == 0
    for i in (0, 1, 14, 29):
        assert_close(ys[i], ref, what=f"back to back {case} call {i}")


def test_decode_walkthrough_shapes():
    """Page's decode walk-through: ids [0, 2, -1], K 4096, N 12288, ranks 16 / 32."""
    wl = workloads.make_custom(3, 4096, 12288, [16, 16, 32], seed=34, ids=[0, 2, -1])
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in (L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED):
        y, ws, status = run_linear(wl, dev, path)
        assert status == 0
        assert_close(y, ref, what=f"walkthrough path={path}")


def test_invalid_ids_are_base_only_and_flagged():
    wl = workloads.make_custom(40, 128, 256, [16, 16], seed=8)
    wl.ids[0] = 5
    wl.ids[1] = -3
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)      # oracle treats them as -1 too
    for path in (L.LORA_PATH_TILED, L.LORA_PATH_SPLITK, L.LORA_PATH_STREAM):
        y, ws, status = run_linear(wl, dev, path)
        assert status & L.LORA_DEV_BAD_ID
        assert_close(y, ref, what=f"invalid ids path={path}")


def test_empty_batch_is_noop():
    wl = workloads.make_custom(4, 64, 64, [16], seed=2)
    dev = to_dev(wl)
    ws = L.Workspace(0, 64, 1)
    x = dev["x"][:0]
    y = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    L.lora_linear(x, dev["W"], dev["bias"], dev["ids"][:0], dev["pool"], 1.0, ws, y=y)


def test_host_errors():
    wl = workloads.make_custom(16, 64, 64, [16], seed=2)
    dev = to_dev(wl)
    ws = L.Workspace(16, 64, 1)
    small = L.Workspace(1, 8, 0)
    with pytest.raises(L.LoraError) as e:
        L.lora_linear(dev["x"], dev["W"], None, dev["ids"], dev["pool"], 1.0, small)
    assert e.value.code == L.LORA_ERR_WORKSPACE
    with pytest.raises(L.LoraError) as e:
        L.lora_linear(dev["x"], dev["W"], None, dev["ids"], dev["pool"], 1.0, ws,
                      y=torch.empty(16, 64, dtype=torch.bfloat16, device="cuda"), path=7)
    assert e.value.code == L.LORA_ERR_SHAPE



def test_linear_tiled_split_shrink_weighted_waves_repeat():
    """K >= 1024 with few waves: every shrink job runs as two K halves, each
    writing its own S panel set that the expand steps add up, and the CTAs
    that ran a half take more of the last wave's split tiles (160 output
    tiles + 32 shrink halves on the grid).  Twice on one workspace."""
    wl = workloads.make_custom(2048, 1024, 2560, [16, 32, 64, 48, 64, 16], seed=4242, id_mode="uniform",
                               p_base=0.2, scale=0.8)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    for call in range(2):
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                      path=L.LORA_PATH_TILED)
        assert L.lora_get_status(ws) == 0
        assert_close(y, ref, what=f"split shrink call {call}")

# ---------------------------------------------------------------------------
# full-size workloads: sampled rows against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["decode", "prefill", "qkv", "mlp_down"])
def test_config_full_size_sampled(name):
    wl = workloads.make_config(name)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, segs=segs)
    assert L.lora_get_status(ws) == 0
    assert not torch.isnan(y).any()
    rows = sample_rows(wl.M, per_tile=2 if wl.M > 2048 else 3)
    ref = oracle.lora_linear(wl, rows=rows)
    assert_close(y[rows], ref, what=name)


# ---------------------------------------------------------------------------
# the two products alone
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,ranks,mode", [(64, 256, [8, 8, 16, 16], "uniform"),
                                            (300, 320, [16, 48, 64, 32], "runs"),
                                            (257, 128, [64] * 20, "uniform"),
                                            (300, 1024, [16, 64, 32], "uniform")])   # two K halves add into S
def test_shrink(M, K, ranks, mode):
    wl = workloads.make_custom(M, K, 64, ranks, seed=M, id_mode=mode, p_base=0.2)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = torch.full((M, 64), float("nan"), dtype=torch.float32, device="cuda")
    L.lora_shrink(dev["x"], dev["ids"], dev["pool"], ws, S=S, s_cols=64)
    ref = oracle.shrink(wl, 64)
    assert_close(S, ref, tol=1e-3, what="shrink")


@pytest.mark.parametrize("M,N,ranks,mode", [(64, 256, [8, 8, 16, 16], "uniform"),
                                            (300, 520, [16, 48, 64, 32], "runs")])
def test_expand(M, N, ranks, mode):
    wl = workloads.make_custom(M, 64, N, ranks, seed=N, id_mode=mode, p_base=0.2)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = workloads.random_fp32((M, 64), seed=11)
    y0 = workloads.random_fp32((M, N), seed=12).to(torch.bfloat16)
    y = y0.to("cuda")
    L.lora_expand(S.to("cuda"), dev["ids"], dev["pool"], 1.25, y, ws)
    ref = oracle.expand(wl, S, y0, scale=1.25)
    assert_close(y, ref, what="expand")
    base_rows = (wl.ids < 0).nonzero().flatten()
    assert torch.equal(y[base_rows.to('cuda')].cpu(), y0[base_rows])    # -1 rows untouched


# ---------------------------------------------------------------------------
# per-adapter factors (adapter i's delta scaled by scale * s_i)
# ---------------------------------------------------------------------------

FACTOR_CASES = [
    # M, K, N, ranks, paths
    (7, 256, 384, [16, 32, 64, 16], (L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
    (64, 512, 640, [64, 16, 32, 48, 16], (L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
    (120, 320, 256, [32, 16, 64], (L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
    (700, 1024, 512, [16, 64, 32, 48, 16, 64], (L.LORA_PATH_TILED,)),   # K halves, split last wave
]


@pytest.mark.parametrize("M,K,N,ranks,paths", FACTOR_CASES)
def test_linear_adapter_factors_every_path(M, K, N, ranks, paths):
    factors = [0.25 + 0.5 * i for i in range(len(ranks))]
    factors[1] = 0.0          # an adapter switched off by its factor
    factors[-1] = -1.5        # and one with its delta reversed
    wl = workloads.make_custom(M, K, N, ranks, seed=M + K, id_mode="uniform", p_base=0.15, scale=1.25,
                               adapter_scale=factors)
    wl.ids[0] = len(ranks) + 3    # an invalid id: base only, flagged, its factor never read
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in paths:
        y, ws, status = run_linear(wl, dev, path)
        assert status == L.LORA_DEV_BAD_ID
        assert_close(y, ref, what=f"factors M{M} path={path}")


def test_linear_adapter_factors_prebuilt_segments_and_decode_config():
    """The decode-sized configuration with random factors, segments built
    first, then two back-to-back calls on one workspace."""
    base = workloads.make_config("decode")
    wl = workloads.make_custom(base.M, base.K, base.N, base.ranks, seed=77, ids=base.ids.clone(),
                               adapter_scale="random")
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    rows = sample_rows(wl.M)
    ref = oracle.lora_linear(wl, rows=rows)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    for call in range(2):
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                      segs=segs if call == 0 else None)
        assert L.lora_get_status(ws) == 0
        assert_close(y[rows], ref, what=f"decode factors call {call}")


def test_expand_adapter_factors():
    wl = workloads.make_custom(300, 64, 264, [16, 48, 64, 32], seed=5, id_mode="runs", p_base=0.2,
                               adapter_scale=[2.0, 0.5, -0.75, 1.5])
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = workloads.random_fp32((wl.M, 64), seed=13)
    y0 = workloads.random_fp32((wl.M, wl.N), seed=14).to(torch.bfloat16)
    y = y0.to("cuda")
    L.lora_expand(S.to("cuda"), dev["ids"], dev["pool"], 1.25, y, ws)
    assert_close(y, oracle.expand(wl, S, y0, scale=1.25), what="expand factors")


def test_shrink_ignores_adapter_factors():
    """S leaves the first product unscaled, factors or not."""
    wl = workloads.make_custom(200, 256, 64, [16, 32, 64], seed=8, id_mode="uniform", adapter_scale=[3.0, 0.5, 2.0])
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = torch.full((wl.M, 64), float("nan"), dtype=torch.float32, device="cuda")
    L.lora_shrink(dev["x"], dev["ids"], dev["pool"], ws, S=S, s_cols=64)
    assert_close(S, oracle.shrink(wl, 64), tol=1e-3, what="shrink with factors")


# ---------------------------------------------------------------------------
# LORA_FLAG_STATIC_WEIGHTS: weights streamed before the previous kernel ends
# ---------------------------------------------------------------------------

def test_static_weights_after_kernels_that_write_the_inputs():
    """With the flag, the decode schedule may start streaming W and the pool
    while the kernel ahead of it still runs; x and the ids must still be read
    only after that kernel.  Every call here directly follows torch kernels
    that write its x and ids (three input sets, six calls, one workspace),
    run eagerly and then replayed from a CUDA graph."""
    base = workloads.make_config("decode")
    variants = [base]
    for k in range(2):
        g = torch.Generator().manual_seed(900 + k)
        ids = torch.randint(-1, base.num_adapters, (base.M,), generator=g).to(torch.int32)
        x = workloads.random_fp32((base.M, base.K), seed=910 + k).to(torch.bfloat16)
        variants.append(dataclasses.replace(base, x=x, ids=ids))
    refs = [oracle.lora_linear(v) for v in variants]
    dev = to_dev(base)
    src_x = [v.x.to("cuda") for v in variants]
    src_ids = [v.ids.to("cuda") for v in variants]
    xd, idd = torch.empty_like(src_x[0]), torch.empty_like(src_ids[0])
    ws = L.Workspace(base.M, base.N, base.num_adapters)
    ys = [torch.empty(base.M, base.N, dtype=torch.bfloat16, device="cuda") for _ in range(6)]

    def calls():
        for c in range(6):
            v = c % 3
            torch.mul(src_x[v], 1, out=xd)        # kernels that write this call's inputs
            torch.add(src_ids[v], 0, out=idd)
            L.lora_linear(xd, dev["W"], dev["bias"], idd, dev["pool"], base.scale, ws, y=ys[c],
                          static_weights=True)

    def check(what):
        torch.cuda.synchronize()
        assert L.lora_get_status(ws) == 0
        for c in range(6):
            assert_close(ys[c], refs[c % 3], what=f"{what} call {c}")
            ys[c].fill_(float("nan"))

    for y in ys:
        y.fill_(float("nan"))
    calls()
    check("eager")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            calls()
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
        check("graph")


# ---------------------------------------------------------------------------
# the segment table a decode-sized call builds inside its own kernel
# ---------------------------------------------------------------------------

def _rebase(segs, ws_from, ws_to):
    """The same table layout, pointing into another workspace of equal size."""
    out = L.lora_segments_t()
    d = ws_to.buf.data_ptr() - ws_from.buf.data_ptr()
    for name in ("perm", "bucket_offsets", "seg_id", "seg_start", "seg_len", "seg_rank", "num_segments"):
        setattr(out, name, getattr(segs, name) + d)
    out.plan = ws_to.buf.data_ptr()
    out.M, out.num_adapters, out.num_slices = segs.M, segs.num_adapters, segs.num_slices
    return out


@pytest.mark.parametrize("static_weights", [False, True])
def test_decode_call_builds_the_segment_table(static_weights):
    """A decode-sized call given no table builds one in an extra CTA of its
    own kernel, beside the weight stream.  The table it leaves in the
    workspace equals the oracle's bit for bit, and the tiled schedule then
    runs from it (its work lists included) to the oracle's output."""
    wl = workloads.make_config("decode")
    wl.ids[5] = wl.num_adapters + 2                  # flagged, bucketed as -1
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y,
                  path=L.LORA_PATH_STREAM, static_weights=static_weights)
    assert L.lora_get_status(ws) == L.LORA_DEV_BAD_ID
    assert_close(y, ref, what="decode with in-kernel build")
    ws2 = L.Workspace(wl.M, wl.N, wl.num_adapters)   # only for the table's addresses
    segs = _rebase(L.lora_build_segments(dev["ids"], dev["pool"], ws2), ws2, ws)
    del ws2
    check_segments(wl, dev, ws, segs)
    y2 = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y2, segs=segs,
                  path=L.LORA_PATH_TILED)
    assert L.lora_get_status(ws) == 0
    assert_close(y2, ref, what="tiled from the in-kernel table")


# ---------------------------------------------------------------------------
# merged output (Q|K|V, gate|up): one adapter pair per output slice
# ---------------------------------------------------------------------------

SLICED_CASES = [
    # M, K, slices, ranks, id_mode, paths
    (300, 256, [256, 256, 512], [16, 8, 16, 4], "uniform", (L.LORA_PATH_TILED, L.LORA_PATH_AUTO)),
    (1100, 512, [512, 512], [32, 16, 24], "runs", (L.LORA_PATH_TILED,)),
    (257, 320, [256, 256, 256, 256], [16, 16], "uniform", (L.LORA_PATH_TILED,)),
    (100, 256, [256, 256, 512], [16, 8, 16, 4], "uniform", (L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
    (20, 512, [512, 256, 256], [16, 4, 12], "uniform", (L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
]


@pytest.mark.parametrize("M,K,slices,ranks,mode,paths", SLICED_CASES)
def test_linear_sliced_every_path(M, K, slices, ranks, mode, paths):
    wl = workloads.make_sliced(M, K, slices, ranks, seed=M + K, id_mode=mode, p_base=0.15, scale=1.25,
                               adapter_scale=[0.5 + 0.25 * i for i in range(len(ranks))])
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in paths:
        y, ws, status = run_linear(wl, dev, path, prebuilt=(path == L.LORA_PATH_TILED))
        assert status == 0
        assert_close(y, ref, what=f"sliced M{M} slices={slices} path={path}")


def test_sliced_qkv_shape_sampled():
    """The merged QKV shape (M=2048, K=4096, slices 4096 | 1024 | 1024), eight
    adapters of rank 16 per slice, shuffled Zipf-like ids: sampled rows."""
    base = workloads.make_config("qkv")
    wl = workloads.make_sliced(base.M, base.K, [4096, 1024, 1024], [16] * 8, seed=71, ids=base.ids.clone())
    dev = to_dev(wl)
    y, ws, status = run_linear(wl, dev)
    assert status == 0
    rows = sample_rows(wl.M, per_tile=2)
    assert_close(y[rows], oracle.lora_linear(wl, rows=rows), what="sliced qkv")


def test_sliced_table_must_match_its_pool():
    """A segment table built for a one-output pool is refused with a merged
    pool of the same adapters (its chunk lists are not slice-major)."""
    wl = workloads.make_sliced(200, 256, [256, 256], [16, 16], seed=73)
    dev = to_dev(wl)
    plain = L.build_pool([torch.cat(a) for a in wl.A_s], [torch.zeros(wl.N, 32, dtype=torch.bfloat16)] * 2,
                         wl.K, wl.N, "cuda")
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], plain, ws)
    y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.LoraError) as e:
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, segs=segs)
    assert e.value.code == L.LORA_ERR_SEGMENTS


def test_sliced_rank_not_whole_panels_is_flagged():
    """Ranks 48 and 16 with three slices: the largest rank splits into whole
    panels, the other does not; the builder flags it (no fault)."""
    wl = workloads.make_custom(64, 128, 768, [48, 16], seed=74)
    dev = to_dev(wl)
    pool = dev["pool"]
    pool.desc.num_slices = 3
    for s, v in enumerate([0, 256, 512, 768]):
        pool.desc.slice_start[s] = v
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    L.lora_build_segments(dev["ids"], pool, ws)
    assert L.lora_get_status(ws) & L.LORA_DEV_BAD_POOL


# ---------------------------------------------------------------------------
# one segment table for every layer of a step (§3.2)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", [100, 700])
def test_one_table_serves_layers_of_other_shapes(M):
    """The table is built once, with the first layer's pool; the other layers
    (other K and N, the same adapters and ranks, laid out alike) reuse it on
    the same workspace, sized for the largest N.  M=100 runs the split-K
    schedule, M=700 the tiled one."""
    ranks = [16, 32, 64, 16, 48]
    g = torch.Generator().manual_seed(M)
    ids = torch.randint(-1, len(ranks), (M,), generator=g).to(torch.int32)
    shapes = [(512, 768), (512, 256), (768, 512), (256, 1024)]   # (K, N) per layer
    layers = [workloads.make_custom(M, K, N, ranks, seed=M + 10 * j, ids=ids.clone()) for j, (K, N) in enumerate(shapes)]
    devs = [to_dev(wl) for wl in layers]
    ws = L.Workspace(M, max(N for _, N in shapes), len(ranks))
    segs = L.lora_build_segments(devs[0]["ids"], devs[0]["pool"], ws)
    for j, (wl, dev) in enumerate(zip(layers, devs)):
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, segs=segs)
        assert L.lora_get_status(ws) == 0
        assert_close(y, oracle.lora_linear(wl), what=f"layer {j} K{wl.K} N{wl.N} with the shared table")


# ---------------------------------------------------------------------------
# ranks above 64 (up to 128)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,paths", [(20, (L.LORA_PATH_STREAM, L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
                                     (100, (L.LORA_PATH_SPLITK, L.LORA_PATH_TILED)),
                                     (700, (L.LORA_PATH_TILED,))])
def test_linear_ranks_up_to_128_every_path(M, paths):
    wl = workloads.make_custom(M, 512, 640, [128, 96, 16, 80, 128, 40], seed=M + 3, id_mode="uniform", p_base=0.1)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in paths:
        y, ws, status = run_linear(wl, dev, path)
        assert status == 0
        assert_close(y, ref, what=f"ranks to 128, M{M} path={path}")


def test_sliced_rank_64_per_slice():
    """A merged gate|up with rank 64 per slice: stacked rank 128."""
    wl = workloads.make_sliced(300, 256, [512, 512], [64, 32, 64], seed=77, id_mode="runs")
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    for path in (L.LORA_PATH_TILED, L.LORA_PATH_AUTO):
        y, ws, status = run_linear(wl, dev, path)
        assert status == 0
        assert_close(y, ref, what=f"sliced rank 64 path={path}")


# ---------------------------------------------------------------------------
# mixture of experts: routing (bit-exact), grouped GEMM + finalize
# ---------------------------------------------------------------------------

def run_moe(mw):
    d = "cuda"
    x, W = mw.x.to(d), mw.W.to(d)
    ex, wt = mw.expert.to(d), mw.weight.to(d)
    ws = L.MoeWorkspace(mw.M, mw.topk, mw.E)
    out = torch.full((mw.M * mw.topk, mw.N), float("nan"), dtype=torch.bfloat16, device=d)
    y = torch.full((mw.M, mw.N), float("nan"), dtype=torch.bfloat16, device=d)
    L.lora_moe(x, W, ex, wt, ws, out=out, y=y)
    return y, ws


@pytest.mark.parametrize("M,K,N,E,topk,skew", [(1, 64, 64, 4, 1, 0.0), (37, 192, 136, 5, 2, 0.0),
                                               (300, 512, 640, 16, 4, 1.5), (1000, 256, 264, 64, 8, 3.0),
                                               (129, 128, 512, 3, 3, 0.0)])
def test_moe_matches_oracle(M, K, N, E, topk, skew):
    mw = workloads.make_moe(M, K, N, E, topk, seed=M + E, skew=skew)
    if M > 3:
        mw.expert[2, 0] = E + 5      # an invalid expert contributes nothing
        mw.expert[3, topk - 1] = -1
    y, ws = run_moe(mw)
    assert assert_close(y, oracle.moe(mw.x, mw.W, mw.expert, mw.weight), what=f"moe M{M} E{E} top{topk}") is None
    perm, off = L.moe_routing_to_host(ws, M, topk, E)
    want_perm, want_off, _ = oracle.moe_routing(mw.expert, E)
    assert np.array_equal(perm.numpy(), want_perm) and np.array_equal(off.numpy(), want_off)


@pytest.mark.parametrize("M,topk,E", [(40000, 8, 1024), (5000, 2, 7), (33, 8, 8)])
def test_moe_routing_many_chunks(M, topk, E):
    """The routing alone over many CTA chunks (320 K pairs: 250 chunks of
    1280, so a warp's range is not a whole number of id batches), bit-exact
    against the stable sort; ids outside [-1, E) set the device status."""
    g = torch.Generator().manual_seed(M + E)
    ex = torch.randint(-1, E, (M, topk), generator=g, dtype=torch.int32)
    ex[0, 0] = E          # invalid: routed with the -1 pairs
    ws = L.MoeWorkspace(M, topk, E)
    L.lora_moe_route(ex.cuda(), E, ws)
    perm, off = L.moe_routing_to_host(ws, M, topk, E)
    want_perm, want_off, _ = oracle.moe_routing(ex, E)
    assert np.array_equal(perm.numpy(), want_perm) and np.array_equal(off.numpy(), want_off)
    assert L.lora_get_status(ws) & L.LORA_DEV_BAD_ID
    ex[0, 0] = 0
    L.lora_moe_route(ex.cuda(), E, ws)
    assert L.lora_get_status(ws) == 0


def test_moe_large_sampled_rows():
    """M=2048 tokens, 64 experts, top-8, K=2048, N=1408: sampled rows."""
    mw = workloads.make_moe(2048, 2048, 1408, 64, 8, seed=91, skew=1.0)
    y, ws = run_moe(mw)
    rows = sample_rows(mw.M, per_tile=2)
    assert_close(y[rows], oracle.moe(mw.x, mw.W, mw.expert, mw.weight, rows=rows), what="moe large")
