"""Seeded synthetic workloads for the multi-LoRA linear layer.

This module only draws inputs; it holds none of the layer's arithmetic, so the
CPU oracle and the CUDA path can both consume it without sharing any of the
computation.  Everything is drawn on the CPU with a ``torch.Generator`` seeded
per workload, in fp32, and rounded to bf16 exactly once.

Shapes and value distributions follow the five benchmark configurations of
this project (tiny / decode / prefill / merged-QKV / MLP-down).  The weight
shapes follow "vLLM-Ascend dynamic LoRA" (pptc.cn/news/149022) §1.1: A_i is
[r_i, K], B_i is [N, r_i], W is [N, K] (torch ``nn.Linear`` convention), and
``lora_id_map`` has one int32 per token with -1 meaning "no adapter" (§2.1).

Notation: ``N(0, s)`` means a normal distribution with standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

CONFIG_NAMES = ("tiny", "decode", "prefill", "qkv", "mlp_down")


@dataclass
class Workload:
    """One seeded instance of the layer's inputs (all CPU tensors)."""

    name: str
    M: int
    K: int
    N: int
    ranks: List[int]                 # true rank r_i of each adapter
    ids: torch.Tensor                # int32 [M], -1 = base only
    x: torch.Tensor                  # bf16 [M, K]
    W: torch.Tensor                  # bf16 [N, K]
    bias: Optional[torch.Tensor]     # bf16 [N] or None
    A: List[torch.Tensor]            # bf16 [r_i, K] per adapter
    B: List[torch.Tensor]            # bf16 [N, r_i] per adapter
    scale: float
    seed: int = 0
    meta: dict = field(default_factory=dict)
    # per-adapter factor on the LoRA term (e.g. alpha_i / r_i); None = 1 for all
    adapter_scale: Optional[List[float]] = None
    # merged output (e.g. Q|K|V): widths of the output slices (sum N); then each
    # adapter has one pair per slice, A_s[i][s] bf16 [r_i, K] and
    # B_s[i][s] bf16 [N_s, r_i], and A / B are None
    slices: Optional[List[int]] = None
    A_s: Optional[List[List[torch.Tensor]]] = None
    B_s: Optional[List[List[torch.Tensor]]] = None
    # e4m3 adapters: codes A8[i] uint8 [r_i, K], B8[i] uint8 [N, r_i] and
    # dequant factors deq[i] = (a, b); adapter i is then A_i = a * e4m3(A8[i]),
    # B_i = b * e4m3(B8[i]), and A / B are None
    A8: Optional[List[torch.Tensor]] = None
    B8: Optional[List[torch.Tensor]] = None
    deq: Optional[List[tuple]] = None

    @property
    def num_adapters(self) -> int:
        return len(self.ranks)

    def describe(self) -> str:
        nz = int((self.ids >= 0).sum())
        return (f"{self.name}: M={self.M} K={self.K} N={self.N} adapters={self.num_adapters} "
                f"lora_tokens={nz} scale={self.scale}")


# --------------------------------------------------------------------------
# id-structure generators (structure only, no layer arithmetic)
# --------------------------------------------------------------------------

def _zipf_probs(n: int, s: float) -> torch.Tensor:
    k = torch.arange(1, n + 1, dtype=torch.float64)
    p = k.pow(-s)
    return p / p.sum()


def _renormalise_lengths(lengths: List[int], total: int) -> List[int]:
    """Scale request lengths so they sum to ``total`` exactly.

    floor(L_j * total / sum L) (at least 1), then the remainder is handed out
    +1 at a time to the largest fractional parts, ties broken by lower j.
    """
    s = sum(lengths)
    exact = [L * total / s for L in lengths]
    out = [max(1, int(math.floor(e))) for e in exact]
    rem = total - sum(out)
    order = sorted(range(len(lengths)), key=lambda j: (-(exact[j] - math.floor(exact[j])), j))
    i = 0
    while rem > 0:
        out[order[i % len(order)]] += 1
        rem -= 1
        i += 1
    while rem < 0:  # only possible when many lengths were clamped up to 1
        j = max(range(len(out)), key=lambda q: (out[q], -q))
        out[j] -= 1
        rem += 1
    return out


def _draw_values(g: torch.Generator, M, K, N, ranks, w_std, a_std, b_std, bias_std, with_bias=True):
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, dtype=torch.float32) * w_std).to(torch.bfloat16)
    bias = None
    if with_bias:
        bias = (torch.randn(N, generator=g, dtype=torch.float32) * bias_std).to(torch.bfloat16)
    A, B = [], []
    for r in ranks:
        A.append((torch.randn(r, K, generator=g, dtype=torch.float32) * a_std).to(torch.bfloat16))
        B.append((torch.randn(N, r, generator=g, dtype=torch.float32) * b_std).to(torch.bfloat16))
    return x, W, bias, A, B


def make_config(name_or_index, seed: Optional[int] = None) -> Workload:
    """Build one of the five benchmark configurations.

    ``seed`` defaults to 1234 + the configuration index.
    """
    if isinstance(name_or_index, int):
        idx = name_or_index
        name = CONFIG_NAMES[idx]
    else:
        name = name_or_index
        idx = CONFIG_NAMES.index(name)
    if seed is None:
        seed = 1234 + idx
    g = torch.Generator().manual_seed(seed)
    meta = {}

    if name == "tiny":
        M, K, N = 64, 256, 256
        ranks = [8, 8, 16, 16]
        ids = torch.randint(-1, 4, (M,), generator=g, dtype=torch.int64)
        w_std, bias_std, b_std, scale = 0.02, 0.01, 0.02, 2.0

    elif name == "decode":
        M, K, N = 32, 4096, 4096
        nA = 20
        choices = torch.tensor([16, 32, 64])
        ranks = choices[torch.randint(0, 3, (nA,), generator=g)].tolist()
        ids = torch.randint(0, nA, (M,), generator=g, dtype=torch.int64)
        drop = torch.rand(M, generator=g) < 0.10
        ids[drop] = -1
        w_std, bias_std, b_std, scale = 0.02, 0.01, 0.02, 2.0

    elif name == "prefill":
        M, K, N = 1024, 4096, 4096
        nA, nreq = 40, 16
        choices = torch.tensor([16, 32, 64])
        ranks = choices[torch.randint(0, 3, (nA,), generator=g)].tolist()
        lengths = torch.randint(16, 129, (nreq,), generator=g).tolist()
        lengths = _renormalise_lengths(lengths, M)
        req_ids = torch.randint(0, nA, (nreq,), generator=g).tolist()
        base_only = (torch.rand(nreq, generator=g) < 0.05).tolist()
        parts = []
        for L, a, b in zip(lengths, req_ids, base_only):
            parts.append(torch.full((L,), -1 if b else a, dtype=torch.int64))
        ids = torch.cat(parts)
        meta["request_lengths"] = lengths
        w_std, bias_std, b_std, scale = 0.02, 0.01, 0.02, 2.0

    elif name == "qkv":
        M, K, N = 2048, 4096, 6144
        nA = 8
        ranks = [64] * nA
        p = _zipf_probs(nA, 1.1)
        ids = torch.multinomial(p, M, replacement=True, generator=g).to(torch.int64)
        drop = torch.rand(M, generator=g) < 0.20
        ids[drop] = -1
        w_std, bias_std, b_std, scale = 0.02, 0.01, 0.02, 2.0

    elif name == "mlp_down":
        M, K, N = 8192, 12288, 4096
        nA = 32
        choices = torch.tensor([16, 32, 64])
        ranks = choices[torch.randint(0, 3, (nA,), generator=g)].tolist()
        p = _zipf_probs(nA, 1.1)
        lengths, total = [], 0
        while total < M:
            L = int(torch.randint(64, 513, (1,), generator=g))
            L = min(L, M - total)
            lengths.append(L)
            total += L
        nreq = len(lengths)
        req_ids = torch.multinomial(p, nreq, replacement=True, generator=g).tolist()
        base_only = (torch.rand(nreq, generator=g) < 0.20).tolist()
        parts = []
        for L, a, b in zip(lengths, req_ids, base_only):
            parts.append(torch.full((L,), -1 if b else a, dtype=torch.int64))
        ids = torch.cat(parts)
        meta["request_lengths"] = lengths
        w_std, bias_std, b_std, scale = 0.01, 0.01, 0.02, 1.0
    else:
        raise ValueError(f"unknown config {name!r}")

    a_std = 1.0 / math.sqrt(K)
    x, W, bias, A, B = _draw_values(g, M, K, N, ranks, w_std, a_std, b_std, bias_std)
    return Workload(name=name, M=M, K=K, N=N, ranks=list(ranks), ids=ids.to(torch.int32),
                    x=x, W=W, bias=bias, A=A, B=B, scale=scale, seed=seed, meta=meta)


def make_custom(M: int, K: int, N: int, ranks: List[int], seed: int, ids=None,
                id_mode: str = "uniform", p_base: float = 0.1, scale: float = 2.0,
                with_bias: bool = True, w_std: float = 0.02, adapter_scale=None) -> Workload:
    """A free-form workload for edge cases.

    ``ids`` may be given explicitly; otherwise ``id_mode`` picks the structure:
    "uniform" (i.i.d. over adapters, then -1 with probability p_base),
    "runs" (contiguous runs of random length), "all_base" (every id -1),
    "single" (every token uses adapter 0).  ``adapter_scale`` is an optional
    per-adapter factor on the LoRA term; "random" draws one from U(0.25, 2).
    """
    g = torch.Generator().manual_seed(seed)
    nA = len(ranks)
    if ids is not None:
        ids = torch.as_tensor(ids, dtype=torch.int64)
    elif id_mode == "all_base" or nA == 0:
        ids = torch.full((M,), -1, dtype=torch.int64)
    elif id_mode == "single":
        ids = torch.zeros(M, dtype=torch.int64)
    elif id_mode == "uniform":
        ids = torch.randint(0, nA, (M,), generator=g, dtype=torch.int64)
        ids[torch.rand(M, generator=g) < p_base] = -1
    elif id_mode == "runs":
        parts, total = [], 0
        while total < M:
            L = min(int(torch.randint(1, 200, (1,), generator=g)), M - total)
            a = int(torch.randint(-1, nA, (1,), generator=g))
            parts.append(torch.full((L,), a, dtype=torch.int64))
            total += L
        ids = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)
    else:
        raise ValueError(id_mode)
    a_std = 1.0 / math.sqrt(K)
    x, W, bias, A, B = _draw_values(g, M, K, N, ranks, w_std, a_std, 0.02, 0.01, with_bias)
    if isinstance(adapter_scale, str) and adapter_scale == "random":
        adapter_scale = [float(v) for v in (torch.rand(nA, generator=g) * 1.75 + 0.25)]
    return Workload(name=f"custom_M{M}_K{K}_N{N}", M=M, K=K, N=N, ranks=list(ranks),
                    ids=ids.to(torch.int32), x=x, W=W, bias=bias, A=A, B=B, scale=scale, seed=seed,
                    adapter_scale=None if adapter_scale is None else [float(v) for v in adapter_scale])


def make_sliced(M: int, K: int, slices: List[int], ranks: List[int], seed: int, ids=None,
                id_mode: str = "uniform", p_base: float = 0.1, scale: float = 2.0, with_bias: bool = True,
                adapter_scale=None) -> Workload:
    """A merged-output workload: output slices of widths ``slices`` (for a
    merged QKV projection, [q, k, v]) and, per adapter, one A / B pair per
    slice with the adapter's rank.  Ids and the base tensors are drawn as in
    make_custom (same seed, same structure); A ~ N(0, 1/sqrt(K)),
    B ~ N(0, 0.02)."""
    N = int(sum(slices))
    base = make_custom(M, K, N, ranks, seed, ids=ids, id_mode=id_mode, p_base=p_base, scale=scale,
                       with_bias=with_bias, adapter_scale=adapter_scale)
    g = torch.Generator().manual_seed(seed + 7919)
    a_std = 1.0 / math.sqrt(K)
    A_s, B_s = [], []
    for r in ranks:
        A_s.append([(torch.randn(r, K, generator=g) * a_std).to(torch.bfloat16) for _ in slices])
        B_s.append([(torch.randn(n, r, generator=g) * 0.02).to(torch.bfloat16) for n in slices])
    base.name = f"sliced_M{M}_K{K}_N{'+'.join(str(n) for n in slices)}"
    base.A, base.B = None, None
    base.slices, base.A_s, base.B_s = [int(n) for n in slices], A_s, B_s
    return base


@dataclass
class MoeWorkload:
    """Inputs of a mixture-of-experts layer (CPU tensors)."""

    name: str
    M: int
    K: int
    N: int
    E: int
    topk: int
    x: torch.Tensor          # bf16 [M, K]
    W: torch.Tensor          # bf16 [E, N, K]: expert e's weight, nn.Linear layout
    expert: torch.Tensor     # int32 [M, topk]: the experts of each token (distinct)
    weight: torch.Tensor     # fp32 [M, topk]: their routing weights (softmax over the chosen)
    seed: int = 0


def make_moe(M: int, K: int, N: int, E: int, topk: int, seed: int, skew: float = 0.0) -> MoeWorkload:
    """Seeded MoE inputs: x ~ N(0, 1), W ~ N(0, 0.02), router logits ~ N(0, 1)
    plus ``skew`` * (a per-expert bias ~ N(0, 1)) so that some experts are
    busier; each token takes its topk largest logits and a softmax over them."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)
    logits = torch.randn(M, E, generator=g) + skew * torch.randn(1, E, generator=g)
    top, idx = torch.topk(logits, topk, dim=1)
    weight = torch.softmax(top, dim=1).to(torch.float32)
    return MoeWorkload(name=f"moe_M{M}_K{K}_N{N}_E{E}_top{topk}", M=M, K=K, N=N, E=E, topk=topk, x=x, W=W,
                       expert=idx.to(torch.int32).contiguous(), weight=weight.contiguous(), seed=seed)


def random_fp32(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """A seeded fp32 tensor (used as the given S input of the expand step)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def to_e4m3(wl: Workload) -> Workload:
    """The same workload with its adapters stored as e4m3 codes: per adapter
    and factor, a dequant factor d = max|value| / 448 (the largest e4m3
    magnitude) and codes e4m3(value / d), round to nearest even (torch's
    float8_e4m3fn cast).  This is input preparation: the oracle decodes the
    codes itself, and the layer is defined by codes and factors."""
    A8, B8, deq = [], [], []
    for a, b in zip(wl.A, wl.B):
        da = float(a.float().abs().max()) / 448.0 or 1.0
        db = float(b.float().abs().max()) / 448.0 or 1.0
        A8.append((a.float() / da).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        B8.append((b.float() / db).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        deq.append((da, db))
    return dataclasses.replace(wl, A=None, B=None, A8=A8, B8=B8, deq=deq, name=wl.name + "_e4m3")
