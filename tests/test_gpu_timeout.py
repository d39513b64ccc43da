"""A bounded wait that runs out: the kernel gives up, reports it in the
device status word and returns, and the GPU context stays usable.

The failure is made on the host, without faulting anything: after the
segment table is built, one S-ready counter of the tiled schedule (the
counter block opens the workspace; the per-tile counters start at int32 8,
token tile 0 of layer 0 first) is set so low that the shrink jobs can never
bring it to its target.  The producers of that token tile's output tiles
then wait until their budget (about one second) runs out, raise their CTA's
abort flag and set LORA_DEV_TIMEOUT; every role of the kernel keeps going
with short waits, so the launch completes.  Only the tiled schedule is
exercised: its roles never leave their loops on a timeout, so they all
reach the final barrier, where each waits (bounded) for its own loads and
tensor-core work in flight before the tensor memory is freed.  The wait
budget is shortened for the failing call (lora_set_wait_budget) so the test
takes milliseconds, and restored for the calls that check the context.
"""
import time

import numpy as np
import pytest
import torch

from oracle import oracle
from segmented_gemm_gb300 import lora as L
from segmented_gemm_gb300 import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-2
CNT_S_READY_TILE0 = 8   # int32 index of token tile 0's S-ready counter in the workspace


def _close(y, ref, what):
    g = y.float().cpu().double().numpy()
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    assert (e <= TOL).all(), f"{what}: max err {np.nanmax(e):.3e}"


def test_unsatisfiable_wait_times_out_and_the_context_survives():
    wl = workloads.make_custom(300, 256, 512, [16, 32, 64], seed=991, p_base=0.1)
    d = "cuda"
    x, W, bias, ids = wl.x.to(d), wl.W.to(d), wl.bias.to(d), wl.ids.to(d)
    pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(ids, pool, ws)
    ws.buf.view(torch.int32)[CNT_S_READY_TILE0] = -(1 << 30)   # no number of shrink jobs reaches the target
    torch.cuda.synchronize()
    y = torch.zeros(wl.M, wl.N, dtype=torch.bfloat16, device=d)
    L.lora_set_wait_budget(20_000_000)   # about 10 ms at 2 GHz
    try:
        t0 = time.perf_counter()
        L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, y=y, segs=segs, path=L.LORA_PATH_TILED)
        status = L.lora_get_status(ws)   # synchronises the stream
        waited = time.perf_counter() - t0
    finally:
        L.lora_set_wait_budget(0)
    assert status & L.LORA_DEV_TIMEOUT, f"status {status}"
    assert waited < 5.0, f"the launch took {waited:.1f} s"
    assert L.lora_get_status(ws) == 0   # reading the status clears it
    # the context is usable: a fresh workspace gives the right answer ...
    ws2 = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y2 = L.lora_linear(x, W, bias, ids, pool, wl.scale, ws2, path=L.LORA_PATH_TILED)
    assert L.lora_get_status(ws2) == 0
    _close(y2, ref, "fresh workspace after the timeout")
    # ... and so does the failed call's workspace once re-initialised
    L.lora_workspace_init(ws)
    y3 = L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, path=L.LORA_PATH_TILED)
    assert L.lora_get_status(ws) == 0
    _close(y3, ref, "re-initialised workspace after the timeout")
