"""Fp4Linear.step_host: the host-buffer path through the C ABI (pinned host
inputs copied in, the step, outputs copied back) gives, call after call, the
bits `step` gives on device buffers. Three calls alternate two input sets, so
both sets of device buffers are used and one is reused while the other call's
copies may still be in flight."""
import pytest
import torch

import fp4_block_scaled_02_gb300 as fb

pytestmark = pytest.mark.gpu


def test_step_host_matches_step_over_alternating_buffers():
    T, K, N = 256, 512, 256
    g = torch.Generator().manual_seed(11)

    def inputs():
        x = torch.randn((T, K), generator=g).bfloat16()
        w = (0.05 * torch.randn((N, K), generator=g)).bfloat16()
        dy = (0.01 * torch.randn((T, N), generator=g)).bfloat16()
        return x, w, dy

    sets = [inputs(), inputs()]
    L = fb.Fp4Linear(T, K, N, rht=True, seed=5)
    order = [0, 1, 0]
    host_out = []
    for i in order:
        x, w, dy = (t.pin_memory() for t in sets[i])
        outs = (torch.empty((T, N), dtype=torch.bfloat16).pin_memory(),
                torch.empty((T, K), dtype=torch.bfloat16).pin_memory(),
                torch.empty((N, K), dtype=torch.float32).pin_memory())
        L.step_host(x, w, dy, *outs)
        host_out.append(outs)
    torch.cuda.synchronize()
    assert fb.fp4_device_status() == 0
    ref = fb.Fp4Linear(T, K, N, rht=True, seed=5)
    for i, outs in zip(order, host_out):
        x, w, dy = (t.cuda() for t in sets[i])
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
        ref.step(x, w, dy, y, dx, dw)
        torch.cuda.synchronize()
        for got, want in zip(outs, (y, dx, dw)):
            assert torch.equal(got.view(torch.int16 if got.dtype == torch.bfloat16 else torch.int32),
                               want.cpu().view(torch.int16 if want.dtype == torch.bfloat16 else torch.int32))
