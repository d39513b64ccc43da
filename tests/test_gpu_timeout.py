"""A bounded wait that runs out: the kernel gives up, reports it in the
device status word and returns, and the GPU context stays usable.

The failure is made on the host, without faulting anything: after the
segment table is built, one S-ready counter in the workspace's counter block
(which opens the workspace) is set so low that the shrink results can never
bring it to its target:
- the tiled schedule (M > 128): token tile 0's counter (int32 8, the first
  per-tile counter), which the producers of that tile's output tiles wait on;
- the split-K schedule (64 < M <= 128): its single count of reduced shrink
  tiles (int32 3), which every producer with expand steps waits on.
Those waits run until their budget runs out, raise their CTA's abort flag
and set LORA_DEV_TIMEOUT; every role keeps going with short waits and,
before the CTA ends, waits (bounded) for its own loads and tensor-core work
in flight, so the launch completes and frees its tensor memory.  The wait
budget is shortened for the failing call (lora_set_wait_budget) so the test
takes milliseconds, and restored for the calls that check the context.  The
cluster schedule (M <= 64) is not exercised.
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


def _close(y, ref, what):
    g = y.float().cpu().double().numpy()
    e = np.abs(g - ref) / (1.0 + np.abs(ref))
    assert (e <= TOL).all(), f"{what}: max err {np.nanmax(e):.3e}"


@pytest.mark.parametrize("M,path,counter", [(300, L.LORA_PATH_TILED, 8), (96, L.LORA_PATH_SPLITK, 3)])
def test_unsatisfiable_wait_times_out_and_the_context_survives(M, path, counter):
    wl = workloads.make_custom(M, 256, 512, [16, 32, 64], seed=991, p_base=0.1)
    d = "cuda"
    x, W, bias, ids = wl.x.to(d), wl.W.to(d), wl.bias.to(d), wl.ids.to(d)
    pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, d)
    ref = oracle.lora_linear(wl)
    ws = L.Workspace(wl.M, wl.N, wl.num_adapters)
    segs = L.lora_build_segments(ids, pool, ws)
    ws.buf.view(torch.int32)[counter] = -(1 << 30)   # no number of shrink results reaches the target
    torch.cuda.synchronize()
    y = torch.zeros(wl.M, wl.N, dtype=torch.bfloat16, device=d)
    L.lora_set_wait_budget(20_000_000)   # about 10 ms at 2 GHz
    try:
        t0 = time.perf_counter()
        L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, y=y, segs=segs, path=path)
        status = L.lora_get_status(ws)   # synchronises the stream
        waited = time.perf_counter() - t0
    finally:
        L.lora_set_wait_budget(0)
    assert status & L.LORA_DEV_TIMEOUT, f"status {status}"
    assert waited < 5.0, f"the launch took {waited:.1f} s"
    assert L.lora_get_status(ws) == 0   # reading the status clears it
    # the context is usable: a fresh workspace gives the right answer ...
    ws2 = L.Workspace(wl.M, wl.N, wl.num_adapters)
    y2 = L.lora_linear(x, W, bias, ids, pool, wl.scale, ws2, path=path)
    assert L.lora_get_status(ws2) == 0
    _close(y2, ref, "fresh workspace after the timeout")
    # ... and so does the failed call's workspace once re-initialised
    L.lora_workspace_init(ws)
    y3 = L.lora_linear(x, W, bias, ids, pool, wl.scale, ws, path=path)
    assert L.lora_get_status(ws) == 0
    _close(y3, ref, "re-initialised workspace after the timeout")
