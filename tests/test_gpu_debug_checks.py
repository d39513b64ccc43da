"""The segment-table checker and the library built with LORA_DEBUG.

lora_check_segments (both builds) reads a segment table in the workspace
against the ids it was built from ("vLLM-Ascend dynamic LoRA", §2.3: a
stable bucket sort by lora_id, one segment per adapter present; §2.4: the
work lists derived from it) and sets LORA_DEV_CHECK when they disagree.
- Every table the library builds passes, on every schedule's table: the
  stand-alone builder's and the one the decode-sized kernel builds inside
  its own launch.
- A table edited in one place on the host fails, and passes again once the
  edit is undone.  The checker reads only inside the table's arrays (every
  index it follows is range-checked first), so these edits run safely.

lora_moe_check_route does the same for the routing of a mixture-of-experts
layer (the pairs sorted stably by expert, the padded expert order, each
tile's expert), with the same two kinds of tests.

liblora_debug.so runs the checker on every table before a fused kernel
uses it, and on every routing it makes:
- on valid inputs it matches the oracle on every schedule and never raises
  LORA_DEV_CHECK;
- given a prebuilt table whose perm names a token past M, it flags the
  table before any kernel reads it: the tiled schedule leaves y untouched
  and the split-K schedule writes the base product alone.
The normal library is never given such a table.
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


def assert_close(gpu, ref, what=""):
    g = gpu.detach().float().cpu().double().numpy()
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    bad = ~(e <= TOL)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {np.nanmax(e):.3e}"


def to_dev(wl):
    d = "cuda"
    if wl.slices:
        pool = L.build_pool_sliced(wl.A_s, wl.B_s, wl.K, wl.slices, d, adapter_scale=wl.adapter_scale)
    else:
        pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    return dict(x=wl.x.to(d), W=wl.W.to(d), bias=None if wl.bias is None else wl.bias.to(d),
                ids=wl.ids.to(d), pool=pool)


@pytest.fixture
def debug_lib():
    L.use_debug_library(True)
    try:
        yield
    finally:
        L.use_debug_library(False)


# ---- the checker on tables the library built ---------------------------------

def _bad_id_workload():
    wl = workloads.make_custom(260, 256, 256, [32, 16, 64], seed=611)
    ids = wl.ids.clone()
    ids[::9] = 7      # outside [-1, A): bucketed with -1
    ids[4::13] = -3
    return workloads.make_custom(260, 256, 256, [32, 16, 64], seed=611, ids=ids)


BUILT = {
    "tiny": lambda: workloads.make_config("tiny"),
    "decode": lambda: workloads.make_config("decode"),
    "tiled_uniform": lambda: workloads.make_custom(300, 256, 512, [16, 32, 64, 48, 16], seed=601, p_base=0.15),
    "many_tiles_runs": lambda: workloads.make_custom(2000, 128, 256, [16, 64, 32, 128], seed=602, id_mode="runs"),
    "all_base": lambda: workloads.make_custom(700, 128, 256, [16, 32], seed=603, id_mode="all_base"),
    "single": lambda: workloads.make_custom(129, 128, 256, [64], seed=604, id_mode="single"),
    "sliced": lambda: workloads.make_sliced(300, 256, [256, 256, 256], [16, 32], seed=605),
    "many_adapters": lambda: workloads.make_custom(3000, 128, 256, [16, 32, 48, 64] * 50, seed=606, p_base=0.05),
    "bad_ids": _bad_id_workload,
}


@pytest.mark.parametrize("name", sorted(BUILT))
def test_checker_accepts_every_built_table(name):
    wl = BUILT[name]()
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    first = L.lora_get_status(ws)
    L.lora_check_segments(dev["ids"], dev["pool"], ws, segs)
    status = L.lora_get_status(ws)
    bad_ids = name == "bad_ids"
    assert first == (L.LORA_DEV_BAD_ID if bad_ids else 0)
    assert status == 0, f"{name}: status {status}"


@pytest.mark.parametrize("static", [False, True])
def test_checker_accepts_the_decode_kernels_own_table(static):
    """The decode-sized schedule builds its table inside its own launch (in an
    extra CTA beside the weight stream); the checker reads that table."""
    wl = workloads.make_config("decode")
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)   # the table's device pointers
    ws.buf.zero_()                                               # ... and nothing left of that build
    y = L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws,
                      static_weights=static)
    assert L.lora_get_status(ws) == 0
    L.lora_check_segments(dev["ids"], dev["pool"], ws, segs)
    assert L.lora_get_status(ws) == 0
    assert_close(y, oracle.lora_linear(wl), "decode")


# ---- the checker on tables edited in one place ----------------------------------

def _word(ws, ptr, i):
    """The int32 view of word i of the table array at device address ptr."""
    off = int(ptr) - ws.buf.data_ptr()
    assert 0 <= off and off + 4 * (i + 1) <= ws.buf.numel()
    return ws.buf[off + 4 * i: off + 4 * i + 4].view(torch.int32)


def _edits(host, M, A):
    """(name, [(array, index, new value)]) edits of a valid table, each of
    which breaks exactly one of the table's defining properties."""
    perm, off = host["perm"].tolist(), host["bucket_offsets"].tolist()
    big = max(range(A + 1), key=lambda b: off[b + 1] - off[b])        # the fullest bucket
    j = off[big]                                                        # its first position
    other = next(b for b in range(A + 1) if b != big and off[b + 1] > off[b])
    k = off[other]
    return [
        ("perm past M", [("perm", 5, M + 7)]),
        ("perm negative", [("perm", 0, -1)]),
        ("perm repeats a token", [("perm", j + 1, perm[j])]),
        ("perm not stable inside a bucket", [("perm", j, perm[j + 1]), ("perm", j + 1, perm[j])]),
        ("perm swaps tokens of two buckets", [("perm", j, perm[k]), ("perm", k, perm[j])]),
        ("a bucket offset moved", [("bucket_offsets", big + 1, off[big + 1] + 1)]),
        ("bucket_offsets[0] not 0", [("bucket_offsets", 0, 1)]),
        ("a segment length", [("seg_len", 0, host["seg_len"][0].item() + 1)]),
        ("a segment start", [("seg_start", 1, host["seg_start"][1].item() - 1)]),
        ("a segment rank", [("seg_rank", 0, host["seg_rank"][0].item() + 16)]),
        ("a segment id past the pool", [("seg_id", 0, A)]),
        ("the segment count", [("num_segments", 0, host["num_segments"] + 1)]),
    ]


def test_checker_flags_each_edit_and_passes_once_undone():
    wl = workloads.make_custom(300, 256, 256, [16, 32, 64, 48, 16], seed=621, p_base=0.15)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
    assert L.lora_get_status(ws) == 0
    host = L.segments_to_host(segs, ws, wl.M, wl.num_adapters)
    assert host["num_segments"] >= 2
    ptrs = dict(perm=segs.perm, bucket_offsets=segs.bucket_offsets, seg_id=segs.seg_id, seg_start=segs.seg_start,
                seg_len=segs.seg_len, seg_rank=segs.seg_rank, num_segments=segs.num_segments)
    for name, edit in _edits(host, wl.M, wl.num_adapters):
        saved = []
        for arr, i, v in edit:
            w = _word(ws, ptrs[arr], i)
            saved.append((w, w.clone()))
            w.fill_(v)
        L.lora_check_segments(dev["ids"], dev["pool"], ws, segs)
        status = L.lora_get_status(ws)
        for w, old in reversed(saved):
            w.copy_(old)
        assert status & L.LORA_DEV_CHECK, f"{name}: not flagged (status {status})"
        L.lora_check_segments(dev["ids"], dev["pool"], ws, segs)
        assert L.lora_get_status(ws) == 0, f"{name}: still flagged once undone"


# ---- the LORA_DEBUG library -------------------------------------------------------

DEBUG_CASES = [
    ("decode", L.LORA_PATH_AUTO),
    ("splitk", L.LORA_PATH_SPLITK),
    ("tiled", L.LORA_PATH_TILED),
    ("tiled_many", L.LORA_PATH_AUTO),
    ("sliced", L.LORA_PATH_AUTO),
]


def _debug_workload(name):
    if name == "decode":
        return workloads.make_config("decode")
    if name == "splitk":
        return workloads.make_custom(96, 512, 384, [16, 32, 64, 48], seed=631, p_base=0.1, adapter_scale="random")
    if name == "tiled":
        return workloads.make_custom(300, 512, 512, [16, 32, 64, 48, 16], seed=632, p_base=0.15)
    if name == "tiled_many":
        return workloads.make_custom(1100, 256, 768, [16, 64, 32, 128, 48], seed=633, id_mode="runs")
    return workloads.make_sliced(400, 256, [256, 512, 256], [16, 32, 16], seed=634)


@pytest.mark.parametrize("name,path", DEBUG_CASES)
def test_debug_library_matches_the_oracle_without_false_alarms(debug_lib, name, path):
    wl = _debug_workload(name)
    dev = to_dev(wl)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    for prebuilt in (False, True):   # a table built inside the call, then a prebuilt one (checked before use)
        segs = L.lora_build_segments(dev["ids"], dev["pool"], ws) if prebuilt else None
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, segs=segs,
                      path=path)
        status = L.lora_get_status(ws)
        assert status == 0, f"{name} prebuilt={prebuilt}: status {status}"
        assert_close(y, ref, f"{name} prebuilt={prebuilt}")


def test_debug_library_products_layers_e4m3_and_experts(debug_lib):
    """The standalone products, two layers in one launch, an e4m3 pool and a
    mixture-of-experts layer through the debug build: parity, no alarm."""
    wl = workloads.make_custom(260, 256, 264, [16, 48, 64, 32], seed=641, id_mode="runs", p_base=0.2)
    dev = to_dev(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    S = torch.full((wl.M, 64), float("nan"), dtype=torch.float32, device="cuda")
    L.lora_shrink(dev["x"], dev["ids"], dev["pool"], ws, S=S, s_cols=64)
    g = S.detach().cpu().double().numpy()
    ref = oracle.shrink(wl, 64)
    assert (np.abs(g - ref) <= 1e-3 * (1 + np.abs(ref))).all()
    Sin = workloads.random_fp32((wl.M, 64), seed=19)
    y0 = workloads.random_fp32((wl.M, wl.N), seed=20).to(torch.bfloat16)
    y = y0.to("cuda")
    L.lora_expand(Sin.to("cuda"), dev["ids"], dev["pool"], 1.5, y, ws)
    assert_close(y, oracle.expand(wl, Sin, y0, scale=1.5), "expand")
    assert L.lora_get_status(ws) == 0

    base = workloads.make_custom(300, 256, 256, [16, 32, 64], seed=642)
    wls = [workloads.make_custom(300, K, N, [16, 32, 64], seed=643 + j, ids=base.ids.clone())
           for j, (K, N) in enumerate([(256, 512), (384, 256)])]
    devs = [to_dev(w) for w in wls]
    lws = L.LayersWorkspace(300, 512, 3, 2)
    outs = L.lora_linear_layers([(d["x"], d["W"], d["bias"], d["pool"], w.scale) for w, d in zip(wls, devs)],
                                devs[0]["ids"], lws)
    assert L.lora_get_status(lws) == 0
    for j, (w, yj) in enumerate(zip(wls, outs)):
        assert_close(yj, oracle.lora_linear(w), f"layer {j}")

    wl8 = workloads.to_e4m3(workloads.make_custom(300, 256, 256, [16, 32, 64], seed=645, adapter_scale="random"))
    pool8 = L.build_pool_e4m3(wl8.A8, wl8.B8, wl8.deq, wl8.K, wl8.N, "cuda", adapter_scale=wl8.adapter_scale)
    ws8 = L.Workspace(wl8.M, wl8.N, wl8.num_adapters)
    y8 = L.lora_linear(wl8.x.cuda(), wl8.W.cuda(), wl8.bias.cuda(), wl8.ids.cuda(), pool8, wl8.scale, ws8)
    assert L.lora_get_status(ws8) == 0
    assert_close(y8, oracle.lora_linear(wl8), "e4m3")

    mw = workloads.make_moe(96, 256, 256, 8, 2, seed=646, skew=0.5)
    mws = L.MoeWorkspace(mw.M, 2, 8)
    ym = L.lora_moe(mw.x.cuda(), mw.W.cuda(), mw.expert.cuda(), mw.weight.cuda(), mws)
    assert L.lora_get_status(mws) == 0
    assert_close(ym, oracle.moe(mw.x, mw.W, mw.expert, mw.weight), "moe")


def test_debug_library_refuses_a_table_whose_perm_leaves_the_batch(debug_lib):
    """A prebuilt table whose perm names token M + 1000: the debug build's
    check flags it before the fused kernel reads it.  The tiled schedule then
    leaves y untouched (NaN, and the rows past y too); the split-K schedule,
    which takes only the chunk lists from the table, writes the base product
    alone.  A table built afresh works again."""
    for M, path in ((300, L.LORA_PATH_TILED), (96, L.LORA_PATH_SPLITK)):
        wl = workloads.make_custom(M, 256, 256, [16, 32, 64], seed=651 + M, p_base=0.1)
        dev = to_dev(wl)
        ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
        segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
        assert L.lora_get_status(ws) == 0
        _word(ws, segs.perm, 5).fill_(M + 1000)
        ybig = torch.full((M + 8, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = ybig[:M]
        L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, y=y, segs=segs,
                      path=path)
        status = L.lora_get_status(ws)
        assert status & L.LORA_DEV_CHECK, f"M={M}: status {status}"
        assert torch.isnan(ybig[M:].float()).all(), "a row past y was written"
        if path == L.LORA_PATH_TILED:
            assert torch.isnan(y.float()).all(), "the tiled schedule wrote y from a refused table"
        else:
            no_lora = dataclasses.replace(wl, ids=torch.full((M,), -1, dtype=torch.int32))
            assert_close(y, oracle.lora_linear(no_lora), "split-K, base product alone")
        segs = L.lora_build_segments(dev["ids"], dev["pool"], ws)
        y = L.lora_linear(dev["x"], dev["W"], dev["bias"], dev["ids"], dev["pool"], wl.scale, ws, segs=segs,
                          path=path)
        assert L.lora_get_status(ws) == 0
        assert_close(y, oracle.lora_linear(wl), f"M={M} after a fresh build")


def test_debug_library_refuses_a_bad_prebuilt_table_for_several_layers(debug_lib):
    """lora_linear_layers with a prebuilt table: the debug build checks it
    first, and a perm entry past M leaves every layer's output untouched."""
    M = 300
    base = workloads.make_custom(M, 256, 256, [16, 32, 64], seed=681)
    wls = [workloads.make_custom(M, K, N, [16, 32, 64], seed=682 + j, ids=base.ids.clone())
           for j, (K, N) in enumerate([(256, 512), (384, 256)])]
    devs = [to_dev(w) for w in wls]
    ids = devs[0]["ids"]
    ws = L.LayersWorkspace(M, 512, 3, len(wls))
    segs = L.lora_build_segments(ids, devs[0]["pool"], ws)
    assert L.lora_get_status(ws) == 0
    ys = [torch.full((M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda") for w in wls]
    layers = [(d["x"], d["W"], d["bias"], d["pool"], w.scale, y) for w, d, y in zip(wls, devs, ys)]
    L.lora_linear_layers(layers, ids, ws, segs=segs)
    assert L.lora_get_status(ws) == 0
    for j, (w, y) in enumerate(zip(wls, ys)):
        assert_close(y, oracle.lora_linear(w), f"layer {j}, prebuilt table")
    _word(ws, segs.perm, 7).fill_(M + 1000)
    for y in ys:
        y.fill_(float("nan"))
    L.lora_linear_layers(layers, ids, ws, segs=segs)
    status = L.lora_get_status(ws)
    assert status & L.LORA_DEV_CHECK, f"status {status}"
    for j, y in enumerate(ys):
        assert torch.isnan(y.float()).all(), f"layer {j} was written from a refused table"


# ---- the routing of a mixture-of-experts layer ----------------------------------

def _route(M, topk, E, seed, skew=0.0, invalid=False):
    mw = workloads.make_moe(M, 64, 64, E, topk, seed=seed, skew=skew)
    ex = mw.expert.clone()
    if invalid and M > 3:
        ex[1, 0] = E + 3       # outside [0, E): routed with the dropped slots
        ex[2, topk - 1] = -1   # a dropped slot
    return mw, ex


ROUTES = [(1, 1, 1, 0.0), (37, 2, 5, 0.0), (300, 4, 16, 2.0), (2048, 8, 64, 1.0), (5000, 2, 7, 0.0),
          (777, 8, 300, 0.5)]


@pytest.mark.parametrize("M,topk,E,skew", ROUTES)
def test_route_checker_accepts_every_routing(M, topk, E, skew):
    for invalid in (False, True):
        _, ex = _route(M, topk, E, seed=M + E, skew=skew, invalid=invalid)
        ws = L.MoeWorkspace(M, topk, E)
        L.lora_moe_route(ex.cuda(), E, ws)
        first = L.lora_get_status(ws)
        assert first == (L.LORA_DEV_BAD_ID if invalid and M > 3 else 0)
        L.lora_moe_check_route(ex.cuda(), E, ws)
        assert L.lora_get_status(ws) == 0, f"M={M} E={E} invalid={invalid}"


def test_route_checker_flags_each_edit_and_passes_once_undone():
    M, topk, E = 300, 4, 16
    _, ex = _route(M, topk, E, seed=661, skew=2.0, invalid=True)
    exd = ex.cuda()
    ws = L.MoeWorkspace(M, topk, E)
    L.lora_moe_route(exd, E, ws)
    L.lora_get_status(ws)
    lay = L.moe_routing_layout(M, topk, E)
    perm, off = (t.tolist() for t in L.moe_routing_to_host(ws, M, topk, E))
    P = M * topk

    def word(name, i):
        o = lay[name] + 4 * i
        return ws.buf[o:o + 4].view(torch.int32)

    busy = max(range(1, E + 1), key=lambda b: off[b + 1] - off[b])   # the busiest expert's bucket
    j = off[busy]
    other = next(b for b in range(1, E + 1) if b != busy and off[b + 1] > off[b])
    tiles = int(word("hdr", 4).item())   # the padded order's tile count
    pad_first = int(word("perm_pad", 0).item())
    edits = [
        ("perm past the pairs", [("perm", 3, P + 5)]),
        ("perm repeats a pair", [("perm", j + 1, perm[j])]),
        ("perm swaps pairs of two experts", [("perm", j, perm[off[other]]), ("perm", off[other], perm[j])]),
        ("a bucket offset moved", [("offsets", busy, off[busy] + 1)]),
        ("a padded row names another pair", [("perm_pad", 0, pad_first + 1 if pad_first + 1 < P else 0)]),
        ("a row past the last tile holds a pair", [("perm_pad", tiles * 128 + 5, 0)]),
        ("a tile's expert", [("mt_expert", 0, int(word("mt_expert", 0).item()) + 1)]),
        ("a tile past the last has an expert", [("mt_expert", tiles, 0)]),
        ("the tile count", [("hdr", 4, tiles + 1)]),
        ("a segment length", [("seg_len", 0, int(word("seg_len", 0).item()) + 1)]),
        ("the segment count", [("num_segments", 0, int(word("num_segments", 0).item()) - 1)]),
    ]
    assert tiles < lay["max_mtiles"]
    for name, edit in edits:
        saved = []
        for arr, i, v in edit:
            w = word(arr, i)
            saved.append((w, w.clone()))
            w.fill_(v)
        L.lora_moe_check_route(exd, E, ws)
        status = L.lora_get_status(ws)
        for w, old in reversed(saved):
            w.copy_(old)
        assert status & L.LORA_DEV_CHECK, f"{name}: not flagged (status {status})"
        L.lora_moe_check_route(exd, E, ws)
        assert L.lora_get_status(ws) == 0, f"{name}: still flagged once undone"


def test_debug_library_refuses_a_routing_that_failed_its_check(debug_lib):
    """The debug build checks the routing it makes (the layer matches the
    oracle, no alarm).  A routing edited afterwards and checked again is
    flagged, and the grouped GEMM then leaves its output untouched; routing
    afresh works again."""
    M, topk, E = 300, 4, 16
    mw = workloads.make_moe(M, 256, 192, E, topk, seed=671, skew=1.0)
    x, W, ex, wt = mw.x.cuda(), mw.W.cuda(), mw.expert.cuda(), mw.weight.cuda()
    ws = L.MoeWorkspace(M, topk, E)
    y = L.lora_moe(x, W, ex, wt, ws)
    assert L.lora_get_status(ws) == 0
    assert_close(y, oracle.moe(mw.x, mw.W, mw.expert, mw.weight), "moe through the debug build")
    lay = L.moe_routing_layout(M, topk, E)
    ws.buf[lay["perm_pad"]:lay["perm_pad"] + 4].view(torch.int32).fill_(M * topk + 100)   # a pair past the batch
    L.lora_moe_check_route(ex, E, ws)
    out = torch.full((M * topk, 192), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_moe_gemm(x, W, topk, ws, out)
    status = L.lora_get_status(ws)
    assert status & L.LORA_DEV_CHECK, f"status {status}"
    assert torch.isnan(out.float()).all(), "the grouped GEMM ran on a routing that failed its check"
    y2 = L.lora_moe(x, W, ex, wt, ws)   # routes afresh
    assert L.lora_get_status(ws) == 0
    assert_close(y2, oracle.moe(mw.x, mw.W, mw.expert, mw.weight), "moe after routing afresh")
