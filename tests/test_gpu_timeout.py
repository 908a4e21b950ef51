"""The error path of the bounded device-side waits, exercised without faulting or hanging the GPU.

gptq_set_test_stall makes the small-M kernel's copy producer issue no copy at all, so nothing is
ever in flight and every consumer wait runs into a 1 ms limit (a barrier that nothing completes).
The kernel then records the timeout in the handle's host-visible error word and returns; the test
checks that the next gptq_gemm on that handle refuses with GPTQ_ERR_TIMEOUT without a device
synchronize inside the library, that gptq_device_status reports and clears it, and that the context
stays usable: the same handle, with the hook off, and a fresh handle both match the oracle again.
"""
import numpy as np
import pytest
import torch

from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack

pytestmark = pytest.mark.gpu

# (spec, M): a single-tile CTA (identity order); a 16-warp CTA with act-order x permuted in shared
# memory; act-order with the gather pre-pass (which still runs normally); the K split, whose first
# CTA of each cluster still waits for the other CTAs' sends after its own waits gave up; the K split
# at two m-tiles, whose clusters still pass their tile sums through both receive slots
CASES = [(synth.LayerSpec(1024, 512, 4, 128, False, False, "fp16"), 1),
         (synth.LayerSpec(512, 16384, 4, 128, True, False, "bf16"), 1),
         (synth.LayerSpec(512, 1024, 3, 64, True, False, "fp16"), 4),
         (synth.LayerSpec(4096, 512, 4, 128, False, False, "bf16"), 1),
         (synth.LayerSpec(8192, 8192, 4, 128, False, False, "bf16"), 16)]


def _id(c):
    s, M = c
    return f"K{s.K}N{s.N}b{s.bits}{'da' if s.desc_act else ''}M{M}"


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_stalled_waits_report_timeout_and_the_context_recovers(case):
    spec, M = case
    ck = synth.make_checkpoint(spec, seed=spec.N + M)
    x = synth.make_x(M, spec.K, spec.dtype, seed=M)
    ref = oracle_y(ck, x)
    h = repack(ck)
    plan = gptq.gptq_gemm_plan(h, M, gptq.PATH_SMALL_M)
    xd = x.cuda()
    y = torch.zeros((M, spec.N), dtype=xd.dtype, device="cuda")

    gptq.gptq_set_test_stall(h, True, 1_000_000)
    gptq.gptq_gemm_path(h, xd, y, gptq.PATH_SMALL_M)     # launches; its waits give up after 1 ms
    torch.cuda.synchronize()
    with pytest.raises(gptq.GptqError) as ei:           # refused on the host, nothing launched
        gptq.gptq_gemm_path(h, xd, y, gptq.PATH_SMALL_M)
    assert ei.value.status == 9
    with pytest.raises(gptq.GptqError) as ei:
        gptq.gptq_device_status(h)
    assert ei.value.status == 9
    gptq.gptq_device_status(h)                          # the record is cleared

    gptq.gptq_set_test_stall(h, False)
    y.fill_(float("nan"))
    gptq.gptq_gemm_path(h, xd, y, gptq.PATH_SMALL_M)
    torch.cuda.synchronize()
    gptq.gptq_device_status(h)
    compare(y.cpu(), ref)

    h2 = repack(ck)
    y2 = torch.full_like(y, float("nan"))
    gptq.gptq_gemm(h2, xd, y2)
    torch.cuda.synchronize()
    gptq.gptq_device_status(h2)
    compare(y2.cpu(), ref)
    assert plan.consumer_warps in (8, 16)


def test_stall_hook_rejects_bad_limits():
    ck = synth.make_checkpoint(synth.LayerSpec(256, 256), seed=1)
    h = repack(ck)
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(gptq.GptqError) as ei:
            gptq.gptq_set_test_stall(h, True, bad)
        assert ei.value.status == 1
    gptq.gptq_set_test_stall(h, False)
