"""Moving a step's inputs and outputs across the host link with the SMs:
lora_copy_async (pinned host <-> device copies by a kernel) and a fused
layer writing y straight into pinned host memory.

Copies are compared byte for byte.  A layer's host-side y must match the
fp64 oracle within the parity bar, and equal the same call's y in device
memory: bit for bit where the schedule sums in a fixed order (the split-K
schedule's atomics do not).  Host-side argument checks that need no GPU run
in test_boundary.py.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _pinned(shape, dtype, fill=None):
    t = torch.empty(shape, dtype=dtype).pin_memory()
    if fill is not None:
        t.copy_(fill)
    return t


def test_copy_round_trip_several_buffers():
    g = torch.Generator().manual_seed(7)
    srcs = [torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, generator=g) for n in (4, 1024, 65536, 12)]
    hs = [_pinned(s.shape, s.dtype, s) for s in srcs]
    ds = [torch.full(s.shape, -7, dtype=s.dtype, device="cuda") for s in srcs]
    L.copy_async(list(zip(ds, hs)))                  # host -> device
    outs = [_pinned(s.shape, s.dtype, torch.zeros_like(s)) for s in srcs]
    L.copy_async(list(zip(outs, ds)))                # device -> host
    torch.cuda.synchronize()
    for s, d, o in zip(srcs, ds, outs):
        assert torch.equal(d.cpu(), s)
        assert torch.equal(o, s)


def test_copy_device_to_device_and_empty_entries():
    src = torch.arange(4096, dtype=torch.float32, device="cuda")
    dst = torch.zeros_like(src)
    empty = torch.empty(0, dtype=torch.float32, device="cuda")
    L.copy_async([(dst, src), (empty, empty)])
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
    L.copy_async([])                                 # nothing to do


def test_copy_refuses_pageable_and_unaligned_memory():
    pageable = torch.zeros(64, dtype=torch.int32)    # not pinned: the GPU cannot address it through this call
    dst = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LoraError) as e:
        L.copy_async([(dst, pageable)])
    assert e.value.code == L.LORA_ERR_ACCESS
    h = _pinned((80,), torch.int32, torch.arange(80, dtype=torch.int32))
    with pytest.raises(L.LoraError) as e:
        L.copy_async([(dst[:60], h[2:62])])          # 8 bytes past a 16-byte boundary
    assert e.value.code == L.LORA_ERR_ALIGN
    with pytest.raises(L.LoraError) as e:
        L.device_pointer(pageable)
    assert e.value.code == L.LORA_ERR_ACCESS
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), torch.zeros(64, dtype=torch.int32))   # nothing was written


def test_device_pointer_of_device_and_pinned_memory():
    d = torch.zeros(16, device="cuda")
    assert L.device_pointer(d) == d.data_ptr()
    h = _pinned((16,), torch.float32)
    assert L.device_pointer(h) != 0


# name: (workload, whether two identical calls give identical bits).  The
# split-K schedule adds its K pieces' partial sums with fp32 atomics, whose
# order varies from call to call; the other schedules sum in a fixed order.
CASES = {
    "decode": (lambda: workloads.make_config("decode"), True),                                 # weight streaming
    "splitk": (lambda: workloads.make_custom(96, 512, 384, [16, 32, 64], seed=771), False),    # split-K
    "tiled": (lambda: workloads.make_custom(300, 256, 512, [16, 32, 64, 48], seed=772), True),  # tiled
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_writes_y_into_pinned_host_memory(name):
    make, same_bits = CASES[name]
    wl = make()
    d = "cuda"
    pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    x, W, ids = wl.x.to(d), wl.W.to(d), wl.ids.to(d)
    bias = None if wl.bias is None else wl.bias.to(d)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y_dev = torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device=d)
    L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, y=y_dev)
    y_host = _pinned((wl.M, wl.N), torch.bfloat16, torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16))
    L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, y=y_host)
    assert L.lora_get_status(ws) == 0            # synchronises the stream
    assert not torch.isnan(y_host.float()).any()     # every element was written
    if same_bits:
        assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    else:
        assert torch.allclose(y_host.float(), y_dev.cpu().float(), rtol=1e-2, atol=1e-2)
    rows = sorted(set([0, wl.M - 1] + list(range(0, wl.M, 37))))
    ref = oracle.lora_linear(wl, rows=rows)
    got = y_host[rows].float().double().numpy()
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert (err <= TOL).all(), f"{name}: max err {err.max():.3e}"


def test_one_stream_step_graph_with_host_link_copies():
    """The end-to-end step the bench times: x and ids copied in by
    copy_async, the layer writing y into pinned host memory, captured in a
    CUDA graph and replayed over two input sets."""
    wl = workloads.make_config("decode")
    d = "cuda"
    pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d, adapter_scale=wl.adapter_scale)
    W = wl.W.to(d)
    bias = None if wl.bias is None else wl.bias.to(d)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    g = torch.Generator().manual_seed(5)
    hx = [_pinned(wl.x.shape, wl.x.dtype, wl.x), _pinned(wl.x.shape, wl.x.dtype, wl.x.flip(0))]
    hids = [_pinned(wl.ids.shape, wl.ids.dtype, wl.ids),
            _pinned(wl.ids.shape, wl.ids.dtype, wl.ids[torch.randperm(wl.M, generator=g)])]
    hy = [_pinned((wl.M, wl.N), torch.bfloat16) for _ in range(2)]
    dx = [torch.empty_like(wl.x, device=d) for _ in range(2)]
    dids = [torch.empty_like(wl.ids, device=d) for _ in range(2)]
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for b in range(2):   # warm-up outside the capture
            L.copy_async([(dx[b], hx[b]), (dids[b], hids[b])], stream=stream)
            L.lora_linear(dx[b], W, bias, dids[b], pool, wl.scale, ws, y=hy[b], stream=stream, static_weights=True)
        stream.synchronize()
        for b in range(2):
            hy[b].fill_(float("nan"))
        with torch.cuda.graph(graph, stream=stream):
            for b in range(2):
                L.copy_async([(dx[b], hx[b]), (dids[b], hids[b])], stream=stream)
                L.lora_linear(dx[b], W, bias, dids[b], pool, wl.scale, ws, y=hy[b], stream=stream,
                              static_weights=True)
    graph.replay()
    torch.cuda.synchronize()
    assert L.lora_get_status(ws) == 0
    for b in range(2):
        y_ref = L.lora_linear(hx[b].to(d), W, bias, hids[b].to(d), pool, wl.scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(hy[b].view(torch.int16), y_ref.cpu().view(torch.int16)), b
