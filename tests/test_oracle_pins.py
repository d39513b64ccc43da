"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

None of these re-types the oracle's own loops: each compares it with an
independent route (a library matmul on a special case, a closed-form identity,
a brute-force Python loop on tiny inputs, a worked example printed on the
page, or an invariant).  Source: "vLLM-Ascend dynamic LoRA"
(pptc.cn/news/149022), sections cited per test.
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t):
    return t.to(torch.float64).numpy()


def _rel_close(a, b, rtol=1e-11):
    scale = np.maximum(1.0, np.abs(b))
    return np.max(np.abs(a - b) / scale) <= rtol


# ----------------------------------------------------------------------------
# segment table (§2.3)
# ----------------------------------------------------------------------------

def test_segments_page_example():
    """§2.3 worked example: ids [0, 2, 0, 1] -> same-id tokens contiguous."""
    g = json.load(open(os.path.join(GOLDEN, "segments_p5_example.json")))
    s = oracle.build_segments(g["ids"], g["num_adapters"], g["true_ranks"])
    assert s["perm"].tolist() == g["perm"]
    assert s["bucket_offsets"].tolist() == g["bucket_offsets"]
    got = [dict(id=int(i), start=int(a), len=int(b), rank=int(r))
           for i, a, b, r in zip(s["seg_id"], s["seg_start"], s["seg_len"], s["seg_rank"])]
    assert got == g["segments"]


@pytest.mark.parametrize("seed", range(12))
def test_segments_brute_force(seed):
    """Stable sort by (id+1, t) computed by Python's sorted() on tiny inputs."""
    rng = np.random.default_rng(seed)
    A = int(rng.integers(1, 9))
    M = int(rng.integers(0, 70))
    ranks = [int(r) for r in rng.choice([8, 16, 20, 32, 64], size=A)]
    ids = rng.integers(-1, A, size=M).astype(np.int32)
    s = oracle.build_segments(ids, A, ranks)
    want = sorted(range(M), key=lambda t: (int(ids[t]) + 1, t))
    assert s["perm"].tolist() == want
    # invariants: permutation, offsets sum to M, each segment one id and contiguous
    assert sorted(s["perm"].tolist()) == list(range(M))
    assert s["bucket_offsets"][-1] == M
    for i, st, ln, rk in zip(s["seg_id"], s["seg_start"], s["seg_len"], s["seg_rank"]):
        toks = s["perm"][st:st + ln]
        assert ln > 0 and all(ids[t] == i for t in toks)
        assert rk % 16 == 0 and rk >= ranks[i] and rk - ranks[i] < 16   # §4.3 padding
    assert list(s["seg_id"]) == sorted(set(int(v) for v in ids if v >= 0))


def test_segments_invalid_ids_are_base_only():
    s = oracle.build_segments([3, -1, 7, -5, 0], 2, [16, 16])
    assert s["invalid"] == 3
    assert s["perm"].tolist() == [0, 1, 2, 3, 4]   # 3, 7, -5 all sorted as -1
    assert s["seg_id"].tolist() == [0]


def test_segments_empty_and_all_base():
    s = oracle.build_segments([], 3, [16, 16, 16])
    assert s["num_segments"] == 0 and s["bucket_offsets"].tolist() == [0, 0, 0, 0, 0]
    s = oracle.build_segments([-1] * 9, 3, [16, 16, 16])
    assert s["num_segments"] == 0 and s["perm"].tolist() == list(range(9))


# ----------------------------------------------------------------------------
# layer output (§1.1, §2.1, §2.2, §3.4)
# ----------------------------------------------------------------------------

def test_all_base_equals_library_gemm():
    """§4.3 / §3.3: with every id -1 the layer is the plain linear x W^T + bias."""
    wl = workloads.make_custom(40, 96, 72, [16, 32], seed=3, id_mode="all_base")
    y = oracle.lora_linear(wl)
    ref = f64(wl.x) @ f64(wl.W).T + f64(wl.bias)[None, :]
    assert _rel_close(y, ref)
    wl.bias = None
    assert _rel_close(oracle.lora_linear(wl), f64(wl.x) @ f64(wl.W).T)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_single_adapter_equals_merged_weight(which):
    """§1.1: a batch where every token uses adapter i equals the merged linear
    x (W + scale * B_i A_i)^T + bias; the other adapters sit in the pool too,
    so a wrong adapter offset or a transposed operand fails here."""
    wl = workloads.make_custom(24, 80, 56, [8, 32, 16], seed=11 + which, id_mode="single",
                               scale=1.75)
    wl.ids[:] = which
    y = oracle.lora_linear(wl)
    Wm = f64(wl.W) + wl.scale * f64(wl.B[which]) @ f64(wl.A[which])
    ref = f64(wl.x) @ Wm.T + f64(wl.bias)[None, :]
    assert _rel_close(y, ref, 1e-10)


@pytest.mark.parametrize("which", [0, 2])
def test_single_adapter_with_factor_equals_merged_weight(which):
    """Per-adapter factor s_i (for instance alpha_i / r_i): a batch where every
    token uses adapter i equals x (W + scale * s_i * B_i A_i)^T + bias, with
    the other adapters' different factors sitting in the table."""
    wl = workloads.make_custom(20, 72, 40, [16, 8, 32], seed=41 + which, id_mode="single", scale=1.5,
                               adapter_scale=[0.25, 4.0, 0.75])
    wl.ids[:] = which
    y = oracle.lora_linear(wl)
    Wm = f64(wl.W) + wl.scale * wl.adapter_scale[which] * f64(wl.B[which]) @ f64(wl.A[which])
    ref = f64(wl.x) @ Wm.T + f64(wl.bias)[None, :]
    assert _rel_close(y, ref, 1e-10)


def test_equal_factors_equal_a_global_scale():
    """Every adapter with the same factor c is the same layer as scale * c."""
    wl = workloads.make_custom(26, 64, 48, [16, 32, 8], seed=44, id_mode="uniform", p_base=0.2,
                               scale=1.25, adapter_scale=[0.625] * 3)
    y = oracle.lora_linear(wl)
    wl.adapter_scale = None
    assert _rel_close(y, oracle.lora_linear(wl, scale=1.25 * 0.625), 1e-12)


def _brute(wl):
    """Per-token loop written out in Python, for tiny shapes only."""
    x, W, b = f64(wl.x), f64(wl.W), f64(wl.bias) if wl.bias is not None else None
    out = np.zeros((wl.M, wl.N))
    for t in range(wl.M):
        for n in range(wl.N):
            v = sum(x[t, k] * W[n, k] for k in range(wl.K))
            if b is not None:
                v += b[n]
            i = int(wl.ids[t])
            if 0 <= i < len(wl.ranks):
                A, B = f64(wl.A[i]), f64(wl.B[i])
                S = [sum(x[t, k] * A[j, k] for k in range(wl.K)) for j in range(wl.ranks[i])]
                si = 1.0 if wl.adapter_scale is None else wl.adapter_scale[i]
                v += wl.scale * si * sum(S[j] * B[n, j] for j in range(wl.ranks[i]))
            out[t, n] = v
    return out


@pytest.mark.parametrize("seed,adapter_scale", [(0, None), (1, None), (2, None), (3, [0.5, 3.0, 1.25])])
def test_per_token_brute_force(seed, adapter_scale):
    """§2.1 / §3.4: each token gets its own base row plus only its own adapter
    (and, when given, only its own adapter's factor on the LoRA term)."""
    wl = workloads.make_custom(8, 24, 16, [8, 16, 4], seed=seed, id_mode="uniform", p_base=0.3,
                               scale=0.5 + seed, adapter_scale=adapter_scale)
    wl.ids[0] = -1
    wl.ids[1] = 2
    wl.ids[2] = 9          # names no adapter: treated as base only
    assert _rel_close(oracle.lora_linear(wl), _brute(wl))


def test_row_independence():
    """A mixed batch's row t equals row t of a batch where every token uses id[t]."""
    wl = workloads.make_custom(30, 64, 48, [16, 8, 32, 16], seed=5, id_mode="uniform",
                               p_base=0.25)
    y = oracle.lora_linear(wl)
    for i in [-1, 0, 1, 2, 3]:
        ids = wl.ids.clone()
        wl2 = workloads.Workload(**{**wl.__dict__, "ids": torch.full_like(ids, i)})
        yi = oracle.lora_linear(wl2)
        sel = (ids == i).numpy()
        assert np.array_equal(y[sel], yi[sel])


def test_rank_padding_is_exact():
    """§4.3: zero rows in A and zero columns in B leave the result unchanged."""
    wl = workloads.make_custom(12, 48, 40, [8, 20], seed=9, id_mode="uniform", p_base=0.0)
    y = oracle.lora_linear(wl)
    A2 = [torch.cat([a, torch.zeros(16 * ((a.shape[0] + 15) // 16) - a.shape[0], a.shape[1],
                                    dtype=a.dtype)]) for a in wl.A]
    B2 = [torch.cat([b, torch.zeros(b.shape[0], a.shape[0] - b.shape[1], dtype=b.dtype)], 1)
          for a, b in zip(A2, wl.B)]
    wl2 = workloads.Workload(**{**wl.__dict__, "A": A2, "B": B2,
                                "ranks": [a.shape[0] for a in A2]})
    assert np.array_equal(y, oracle.lora_linear(wl2))


def test_rows_subset_matches_full():
    wl = workloads.make_custom(20, 32, 24, [16, 16], seed=4)
    full = oracle.lora_linear(wl)
    rows = [19, 0, 7, 7, 3]
    assert np.array_equal(oracle.lora_linear(wl, rows=rows), full[rows])


def test_decode_walkthrough_shapes():
    """§3.4 walk-through: ids [0, 2, -1], K 4096, merged QKV N 12288, ranks 16 / 32.
    The page prints no values; it pins the -1 passthrough and per-row adapters."""
    g = json.load(open(os.path.join(GOLDEN, "decode_walkthrough_p5.json")))
    ranks = [g["ranks"]["0"], 16, g["ranks"]["2"]]
    wl = workloads.make_custom(g["M"], g["K"], g["N"], ranks, seed=34, ids=g["ids"])
    y = oracle.lora_linear(wl)
    x, W, b = f64(wl.x), f64(wl.W), f64(wl.bias)
    base = x @ W.T + b
    assert _rel_close(y[2], base[2])                       # id -1 row passes through
    for row, i in [(0, 0), (1, 2)]:
        lora = wl.scale * (x[row] @ f64(wl.A[i]).T) @ f64(wl.B[i]).T
        assert _rel_close(y[row], base[row] + lora, 1e-10)
        assert not _rel_close(y[row], base[row], 1e-6)     # the LoRA term is really there


# ----------------------------------------------------------------------------
# the two steps alone (§2.2)
# ----------------------------------------------------------------------------

def test_shrink_matches_library_gemm():
    wl = workloads.make_custom(26, 72, 40, [16, 48, 8], seed=21, id_mode="uniform", p_base=0.2)
    S = oracle.shrink(wl, 64)
    x = f64(wl.x)
    for t in range(wl.M):
        i = int(wl.ids[t])
        want = np.zeros(64)
        if i >= 0:
            want[:wl.ranks[i]] = x[t] @ f64(wl.A[i]).T
        assert _rel_close(S[t], want)


@pytest.mark.parametrize("adapter_scale", [None, [2.5, 0.4]])
def test_expand_matches_library_gemm(adapter_scale):
    wl = workloads.make_custom(18, 40, 56, [16, 32], seed=22, id_mode="uniform", p_base=0.3,
                               adapter_scale=adapter_scale)
    S = workloads.random_fp32((wl.M, 32), seed=5)
    y_in = workloads.random_fp32((wl.M, wl.N), seed=6).to(torch.bfloat16)
    y = oracle.expand(wl, S, y_in, scale=1.5)
    for t in range(wl.M):
        i = int(wl.ids[t])
        want = f64(y_in[t])
        if i >= 0:
            si = 1.0 if adapter_scale is None else adapter_scale[i]
            want = want + 1.5 * si * S[t, :wl.ranks[i]].double().numpy() @ f64(wl.B[i]).T
        assert _rel_close(y[t], want)


def test_linear_is_shrink_then_expand():
    """§2.2: y = base + scale * (x A^T) B^T, via the two separate steps in fp64."""
    wl = workloads.make_custom(16, 64, 32, [16, 32, 64], seed=30, id_mode="uniform", p_base=0.2)
    y = oracle.lora_linear(wl)
    S = oracle.shrink(wl, 64)
    base = f64(wl.x) @ f64(wl.W).T + f64(wl.bias)
    for t in range(wl.M):
        i = int(wl.ids[t])
        want = base[t] if i < 0 else base[t] + wl.scale * S[t, :wl.ranks[i]] @ f64(wl.B[i]).T
        assert _rel_close(y[t], want)


def test_config_generators_shapes():
    for name in workloads.CONFIG_NAMES[:3]:
        wl = workloads.make_config(name)
        assert wl.x.shape == (wl.M, wl.K) and wl.W.shape == (wl.N, wl.K)
        assert wl.ids.shape == (wl.M,) and wl.ids.dtype == torch.int32
        assert int(wl.ids.min()) >= -1 and int(wl.ids.max()) < wl.num_adapters
        for a, b, r in zip(wl.A, wl.B, wl.ranks):
            assert a.shape == (r, wl.K) and b.shape == (wl.N, r)
    wl = workloads.make_config("prefill")
    assert sum(wl.meta["request_lengths"]) == 1024 and len(wl.meta["request_lengths"]) == 16
    # seeded: same seed -> identical draw
    assert torch.equal(workloads.make_config("tiny").x, workloads.make_config("tiny").x)


def test_element_samples_match_rows():
    """Element sampling evaluates the same definition as the row routine,
    pinned independently against a library GEMM on a mixed batch."""
    wl = workloads.make_custom(21, 48, 40, [16, 8, 32], seed=41, id_mode="uniform", p_base=0.3)
    prep = oracle.Prepared(wl)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, wl.M, 60)
    cols = rng.integers(0, wl.N, 60)
    e = oracle.lora_linear_elems(prep, rows, cols)
    x, W, b = f64(wl.x), f64(wl.W), f64(wl.bias)
    for q, (t, c) in enumerate(zip(rows, cols)):
        want = x[t] @ W[c] + b[c]
        i = int(wl.ids[t])
        if i >= 0:
            want += wl.scale * (x[t] @ f64(wl.A[i]).T) @ f64(wl.B[i])[c]
        assert abs(e[q] - want) <= 1e-11 * max(1.0, abs(want))
    full = oracle.lora_linear_rows_prepared(prep, list(range(wl.M)))
    assert np.allclose(e, full[rows, cols], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# merged output (Q|K|V, gate|up): one adapter pair per output slice
# ---------------------------------------------------------------------------

def _one_slice_as_plain(wl):
    """The same workload written as an ordinary (single-output) one."""
    return dataclasses.replace(wl, slices=None, A=[a[0] for a in wl.A_s], B=[b[0] for b in wl.B_s],
                               A_s=None, B_s=None)


def test_single_slice_is_the_plain_layer():
    wl = workloads.make_sliced(12, 48, [40], [16, 8, 32], seed=61, adapter_scale=[1.0, 0.5, 2.0])
    assert _rel_close(oracle.lora_linear(wl), oracle.lora_linear(_one_slice_as_plain(wl)), 1e-13)


@pytest.mark.parametrize("which", [0, 1])
def test_sliced_single_adapter_equals_merged_weight(which):
    """Every token uses adapter i: the merged output is x W'^T + bias with
    W' = W whose slice-s rows get scale * s_i * B_i^s A_i^s added."""
    wl = workloads.make_sliced(14, 56, [32, 16, 24], [16, 8], seed=62 + which, scale=1.5,
                               adapter_scale=[0.5, 3.0])
    wl.ids[:] = which
    Wm = f64(wl.W).copy()
    n0 = 0
    for s, n in enumerate(wl.slices):
        Wm[n0:n0 + n] += wl.scale * wl.adapter_scale[which] * f64(wl.B_s[which][s]) @ f64(wl.A_s[which][s])
        n0 += n
    ref = f64(wl.x) @ Wm.T + f64(wl.bias)[None, :]
    assert _rel_close(oracle.lora_linear(wl), ref, 1e-10)


def test_sliced_brute_force_per_element():
    wl = workloads.make_sliced(6, 12, [4, 8, 4], [4, 8, 4], seed=64, id_mode="uniform", p_base=0.3)
    x, W = f64(wl.x), f64(wl.W)
    starts = [0, 4, 12, 16]
    want = np.zeros((wl.M, wl.N))
    for t in range(wl.M):
        i = int(wl.ids[t])
        for n in range(wl.N):
            v = sum(x[t, k] * W[n, k] for k in range(wl.K)) + float(f64(wl.bias)[n])
            if i >= 0:
                s = max(q for q in range(3) if starts[q] <= n)
                A, B = f64(wl.A_s[i][s]), f64(wl.B_s[i][s])
                S = [sum(x[t, k] * A[j, k] for k in range(wl.K)) for j in range(wl.ranks[i])]
                v += wl.scale * sum(S[j] * B[n - starts[s], j] for j in range(wl.ranks[i]))
            want[t, n] = v
    assert _rel_close(oracle.lora_linear(wl), want, 1e-12)


def test_sliced_equals_stacked_block_diagonal_adapter():
    """The representation the GPU pool uses: adapter i as one adapter of rank
    S * r_i, its A the slices' A stacked and its B block-diagonal (slice s's
    rows use only columns [s r_i, (s + 1) r_i))."""
    wl = workloads.make_sliced(20, 64, [32, 16, 16], [16, 32], seed=65, adapter_scale=[2.0, 0.25])
    A, B = [], []
    for i, r in enumerate(wl.ranks):
        A.append(torch.cat(wl.A_s[i], dim=0))
        Bd = torch.zeros(wl.N, len(wl.slices) * r, dtype=torch.bfloat16)
        n0 = 0
        for s, n in enumerate(wl.slices):
            Bd[n0:n0 + n, s * r:(s + 1) * r] = wl.B_s[i][s]
            n0 += n
        B.append(Bd)
    stacked = dataclasses.replace(wl, slices=None, A_s=None, B_s=None, A=A, B=B,
                                  ranks=[len(wl.slices) * r for r in wl.ranks])
    assert _rel_close(oracle.lora_linear(wl), oracle.lora_linear(stacked), 1e-12)


def test_a_slice_pair_touches_only_its_columns():
    wl = workloads.make_sliced(16, 40, [24, 8, 16], [16], seed=66, id_mode="single")
    y0 = oracle.lora_linear(wl)
    wl.B_s[0][1] = (f64_t(wl.B_s[0][1]) * 3.0).to(torch.bfloat16)
    y1 = oracle.lora_linear(wl)
    changed = np.abs(y1 - y0).max(axis=0) > 0
    assert not changed[:24].any() and not changed[32:].any() and changed[24:32].all()


def f64_t(t):
    return t.to(torch.float64)


# ---------------------------------------------------------------------------
# mixture-of-experts layer: routing, grouped expert GEMMs, weighted finalize
# ---------------------------------------------------------------------------

def test_moe_top1_unit_weight_is_the_grouped_gemm():
    """topk 1 with weight 1: every token's row is x W_e^T of its expert,
    computed here one expert group at a time with a library matmul."""
    mw = workloads.make_moe(40, 48, 24, 5, 1, seed=81)
    mw.weight[:] = 1.0
    y = oracle.moe(mw.x, mw.W, mw.expert, mw.weight)
    ref = np.zeros_like(y)
    for e in range(mw.E):
        rows = (mw.expert[:, 0] == e).nonzero().flatten().numpy()
        if rows.size:
            ref[rows] = f64(mw.x)[rows] @ f64(mw.W[e]).T
    assert _rel_close(y, ref, 1e-12)


def test_moe_brute_force():
    mw = workloads.make_moe(5, 6, 4, 4, 2, seed=82)
    mw.expert[1, 1] = 9          # an invalid expert contributes nothing
    x, W = f64(mw.x), f64(mw.W)
    want = np.zeros((mw.M, mw.N))
    for t in range(mw.M):
        for j in range(mw.topk):
            e = int(mw.expert[t, j])
            if not 0 <= e < mw.E:
                continue
            for n in range(mw.N):
                want[t, n] += float(mw.weight[t, j]) * sum(x[t, k] * W[e, n, k] for k in range(mw.K))
    assert _rel_close(oracle.moe(mw.x, mw.W, mw.expert, mw.weight), want, 1e-12)


def test_moe_slot_order_and_weight_linearity():
    mw = workloads.make_moe(30, 32, 16, 6, 3, seed=83)
    y = oracle.moe(mw.x, mw.W, mw.expert, mw.weight)
    perm = torch.tensor([2, 0, 1])
    y_perm = oracle.moe(mw.x, mw.W, mw.expert[:, perm].contiguous(), mw.weight[:, perm].contiguous())
    assert _rel_close(y, y_perm, 1e-13)
    assert _rel_close(oracle.moe(mw.x, mw.W, mw.expert, mw.weight * 2.0), 2.0 * y, 1e-13)   # exact in fp32


def test_moe_routing_is_a_stable_sort_of_the_pairs():
    mw = workloads.make_moe(50, 8, 8, 7, 2, seed=84, skew=2.0)
    perm, off, counts = oracle.moe_routing(mw.expert, mw.E)
    flat = mw.expert.reshape(-1).tolist()
    want = sorted(range(len(flat)), key=lambda p: (flat[p] + 1 if 0 <= flat[p] < mw.E else 0, p))
    assert perm.tolist() == want
    assert counts.tolist() == [flat.count(e) for e in range(mw.E)]


# ---------------------------------------------------------------------------
# e4m3 adapters (8-bit codes with one dequant factor per adapter and factor)
# ---------------------------------------------------------------------------

def test_e4m3_decode_spec_values():
    """Values the e4m3 format fixes: bias 7, 3 mantissa bits, no infinities;
    the smallest subnormal is 2^-9, the smallest normal 2^-6, the largest
    finite magnitude 448 (0x7E); S.1111.111 is NaN."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0,
             0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, v in table.items():
        assert oracle.e4m3_to_f64(code) == v, hex(code)
    assert np.isnan(oracle.e4m3_to_f64(0x7F)) and np.isnan(oracle.e4m3_to_f64(0xFF))
    assert np.signbit(oracle.e4m3_to_f64(0x80))


def test_e4m3_codes_are_ordered_and_symmetric():
    """The 127 non-negative finite codes increase strictly with the code,
    and each negative code is the mirror of its positive one."""
    pos = [oracle.e4m3_to_f64(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(pos, pos[1:]))
    for c in range(1, 0x7F):
        assert oracle.e4m3_to_f64(c | 0x80) == -pos[c]


def _bf16_twin(wl8):
    """The bf16 workload holding e4m3 adapters decoded with unit factors
    (every e4m3 value is exact in bf16)."""
    def dec(codes):
        v = np.vectorize(oracle.e4m3_to_f64)(codes.numpy().astype(np.int64))
        return torch.tensor(v, dtype=torch.float64).to(torch.bfloat16)
    return dataclasses.replace(wl8, A=[dec(a) for a in wl8.A8], B=[dec(b) for b in wl8.B8], A8=None, B8=None,
                               deq=None)


def test_e4m3_unit_factors_equal_the_bf16_oracle():
    """An e4m3 pool with unit dequant factors is the bf16 pool of the same
    values: the two oracle paths agree bit for bit."""
    wl8 = workloads.to_e4m3(workloads.make_custom(12, 64, 48, [16, 32, 8], seed=71, p_base=0.2))
    wl8 = dataclasses.replace(wl8, deq=[(1.0, 1.0)] * 3)
    assert np.array_equal(oracle.lora_linear(wl8), oracle.lora_linear(_bf16_twin(wl8)))


def test_e4m3_factors_scale_the_delta():
    """The LoRA term is linear in each dequant factor: doubling every A
    factor and halving every B factor changes nothing; doubling every A
    factor equals doubling the call's scale."""
    wl8 = workloads.to_e4m3(workloads.make_custom(10, 96, 64, [16, 48], seed=73, p_base=0.0))
    ref = oracle.lora_linear(wl8)
    same = dataclasses.replace(wl8, deq=[(2 * a, b / 2) for a, b in wl8.deq])
    np.testing.assert_allclose(oracle.lora_linear(same), ref, rtol=1e-12, atol=1e-12)
    dbl = dataclasses.replace(wl8, deq=[(2 * a, b) for a, b in wl8.deq])
    np.testing.assert_allclose(oracle.lora_linear(dbl), oracle.lora_linear(wl8, scale=2 * wl8.scale),
                               rtol=1e-12, atol=1e-12)


def test_e4m3_per_token_brute_force():
    """Plain Python per token, with A and B factors that differ (a swapped
    factor or a wrong code offset fails)."""
    wl8 = workloads.to_e4m3(workloads.make_custom(7, 24, 20, [16, 32, 16], seed=79, p_base=0.2,
                                                  adapter_scale="random"))
    dec = np.vectorize(oracle.e4m3_to_f64)
    x = wl8.x.double().numpy()
    W = wl8.W.double().numpy()
    bias = wl8.bias.double().numpy()
    y = x @ W.T + bias
    for t in range(wl8.M):
        i = int(wl8.ids[t])
        if i < 0:
            continue
        a, b = wl8.deq[i]
        A = a * dec(wl8.A8[i].numpy().astype(np.int64))
        B = b * dec(wl8.B8[i].numpy().astype(np.int64))
        y[t] += wl8.scale * wl8.adapter_scale[i] * ((x[t] @ A.T) @ B.T)
    np.testing.assert_allclose(oracle.lora_linear(wl8), y, rtol=1e-11, atol=1e-12)


def test_e4m3_linear_is_shrink_then_expand():
    """The two steps with e4m3 adapters (A's factor in the shrink, B's in
    the expand) give the fused layer's LoRA term; S passes through fp32."""
    wl8 = workloads.to_e4m3(workloads.make_custom(9, 64, 32, [16, 32], seed=83, p_base=0.2))
    S = oracle.shrink(wl8, 32)
    base = dataclasses.replace(wl8, ids=torch.full_like(wl8.ids, -1))
    delta = oracle.lora_linear(wl8) - oracle.lora_linear(base)
    zero = torch.zeros(wl8.M, wl8.N, dtype=torch.bfloat16)
    got = oracle.expand(wl8, torch.tensor(S, dtype=torch.float32), zero)
    np.testing.assert_allclose(got, delta, rtol=1e-5, atol=1e-6)
