"""The failure path of a bounded device wait, exercised without faulting or hanging the GPU.

Every pipeline wait in the GEMM kernels gives up after a wall-clock limit, records
MOE_LORA_DEV_TIMEOUT in the call's device status word and winds the kernel down
(copies and MMAs in flight drained, TMEM freed).  The test hook
moe_lora_debug_set_acc_wait_ns shortens ONE of those waits -- the gate_up epilogue's
wait for its accumulator -- so that it runs out on an ordinary decode layer, whose
accumulators take microseconds.  Every other wait keeps its normal limit.  The test
checks the status bit, the host-buffer entry's MOE_LORA_EDEVICE, and that the next
call with the default limit gives the bytes of a call that never timed out.
"""
import numpy as np
import pytest

from expert_gemm_gb300 import workloads as W
from gpu_harness import dev_weights, dims_of, inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def ml(torch):
    from expert_gemm_gb300 import build, moe_lora
    build.build()
    moe_lora.load()
    return moe_lora


def test_accumulator_wait_timeout_is_reported_and_the_next_call_is_clean(ml, torch):
    wl = W.get("decode")   # 16-row weight-streaming tiles: single-CTA kernels
    logits, lora, x, w = inputs(wl)
    d = dims_of(wl, 0, ml)
    assert ml.plan(d)["block_m"] <= 128
    layer = ml.Layer(d, dev_weights(w, torch))
    lg, lr, xd = to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch)
    fresh = layer.step(lg, lr, xd).clone()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0

    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()   # noqa: E731
    lg_h, lr_h, x_h = pin(logits), pin(lora), pin(x.view(np.int16))
    out_h = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    ml.debug_set_acc_wait_ns(1)
    try:
        layer.step(lg, lr, xd)
        torch.cuda.synchronize()
        st = int(layer.status.item())
        assert st & ml.DEV_TIMEOUT, st
        with pytest.raises(ml.MoeLoraError) as ei:
            layer.step_host(lg_h, lr_h, x_h, out_h)
        assert ei.value.status == ml.EDEVICE
    finally:
        ml.debug_set_acc_wait_ns(0)

    # default limits again: the same bytes as before the timeouts, the context usable
    for _ in range(2):
        again = layer.step(lg, lr, xd)
        torch.cuda.synchronize()
        assert int(layer.status.item()) == 0
        assert torch.equal(fresh.view(torch.int16), again.view(torch.int16))
    assert layer.step_host(lg_h, lr_h, x_h, out_h) == 0
    assert torch.equal(out_h.cuda(), fresh.view(torch.int16))
