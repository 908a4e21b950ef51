"""GPU parity of the small-M path's two-pass calls against the oracle.  At M = 17 .. 32, when x of M
rows would be staged in four or more K panels and the layer has at least one 32-column tile per
SM, gptq_gemm runs the first 16 rows and then the rest as two launches over row slices of x and y."""
import pytest
import torch

from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# K = 4096: x of 24 or more rows takes four panels; N = 5120 gives 160 tiles (>= 152 SMs)
SPECS = [
    synth.LayerSpec(4096, 5120, 4, 128, False, True, "bf16"),
    synth.LayerSpec(4096, 5120, 4, 128, True, False, "fp16"),     # act-order: a gather pass per slice
    synth.LayerSpec(4352, 5120, 3, 64, False, False, "bf16"),
    synth.LayerSpec(4096, 5120, 8, 32, True, False, "bf16"),
]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{s.dtype}"


@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("M", [24, 28, 32])
def test_two_passes_parity(spec, M):
    assert (spec.N + 31) // 32 >= _sms()
    ck = synth.make_checkpoint(spec, seed=spec.K + spec.N + M)
    h = repack(ck)
    plan = gptq.gptq_gemm_plan(h, M, gptq.PATH_SMALL_M)
    assert plan.row_passes == 2 and plan.m_tiles == 2                  # the first pass: 16 rows
    assert plan.launches == gptq.gptq_gemm_launches(h, M, gptq.PATH_SMALL_M)
    assert plan.launches == (2 if spec.desc_act else 1) * 2
    x = synth.make_x(M, spec.K, spec.dtype, seed=M + 40)
    y = run_gemm(h, x, spec.N, gptq.PATH_SMALL_M)
    compare(y, oracle_y(ck, x))


def test_one_pass_where_two_do_not_pay():
    """Three panels (M = 20 at K = 4096), or fewer tiles than SMs: one launch, four m-tiles."""
    h = repack(synth.make_checkpoint(synth.LayerSpec(4096, 5120, 4, 128, False, True, "bf16"), seed=1))
    assert gptq.gptq_gemm_plan(h, 20, gptq.PATH_SMALL_M).row_passes == 1
    assert gptq.gptq_gemm_plan(h, 16, gptq.PATH_SMALL_M).row_passes == 1
    h2 = repack(synth.make_checkpoint(synth.LayerSpec(4096, 4096, 4, 128, False, True, "bf16"), seed=2))
    p = gptq.gptq_gemm_plan(h2, 28, gptq.PATH_SMALL_M)
    assert p.row_passes == 1 and p.m_tiles == 4 and p.k_panels >= 4
    assert gptq.gptq_gemm_plan(h2, 64, gptq.PATH_LARGE_M).row_passes == 1


def test_two_passes_in_a_graph():
    spec = synth.LayerSpec(4096, 5120, 4, 128, True, False, "fp16")
    ck = synth.make_checkpoint(spec, seed=9)
    h = repack(ck)
    xs = {M: synth.make_x(M, spec.K, "fp16", seed=M).cuda() for M in (28, 4)}
    ys = {M: torch.empty(M, spec.N, dtype=torch.float16, device="cuda") for M in xs}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            for M in (28, 4, 28):
                gptq.gptq_gemm_path(h, xs[M], ys[M], gptq.PATH_SMALL_M)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    gptq.gptq_device_status(h)
    for M in (28, 4):
        compare(ys[M].cpu(), oracle_y(ck, xs[M].cpu()))


def test_auto_takes_two_passes_up_to_32_rows():
    """gptq_gemm sends M = 29 .. 32 to the small-M kernel where it runs as two passes, and to the
    large-M kernel where it would not."""
    spec = synth.LayerSpec(4096, 5120, 4, 128, False, True, "bf16")
    ck = synth.make_checkpoint(spec, seed=11)
    h = repack(ck)
    for M in (29, 32):
        p = gptq.gptq_gemm_plan(h, M, gptq.PATH_AUTO)
        assert p.path == gptq.PATH_SMALL_M and p.row_passes == 2
    assert gptq.gptq_gemm_plan(h, 33, gptq.PATH_AUTO).path == gptq.PATH_LARGE_M
    x = synth.make_x(30, spec.K, spec.dtype, seed=12)
    compare(run_gemm(h, x, spec.N, gptq.PATH_AUTO), oracle_y(ck, x))
    h2 = repack(synth.make_checkpoint(synth.LayerSpec(4096, 4096, 4, 128, False, True, "bf16"), seed=13))
    assert gptq.gptq_gemm_plan(h2, 30, gptq.PATH_AUTO).path == gptq.PATH_LARGE_M   # fewer tiles than SMs


def test_two_passes_with_bias_awq_and_fp8():
    """The second pass writes y at a row offset and adds the bias again: AWQ with a bias, and an FP8
    block-scaled layer, both at M = 28 in two passes."""
    import oracle
    K, N = 4096, 5120
    b = torch.randn(N, generator=torch.Generator().manual_seed(21)) * 0.1
    ck = synth.make_awq_checkpoint(K, N, 128, "fp16", seed=22)
    h = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), 128)
    gptq.gptq_set_bias(h, b.half().cuda())
    assert gptq.gptq_gemm_plan(h, 28, gptq.PATH_SMALL_M).row_passes == 2
    x = synth.make_x(28, K, "fp16", seed=23)
    y_ref = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, 128, "fp16", x) + b.half().double().numpy()[None, :]
    compare(run_gemm(h, x, N, gptq.PATH_SMALL_M), y_ref)
    f8 = synth.make_fp8_checkpoint(K, N, "bf16", seed=24)
    h8 = gptq.gptq_repack_fp8(f8.weight.cuda(), f8.scale_inv.cuda(), torch.bfloat16)
    assert gptq.gptq_gemm_plan(h8, 28, gptq.PATH_AUTO).row_passes == 2
    x8 = synth.make_x(28, K, "bf16", seed=25)
    compare(run_gemm(h8, x8, N, gptq.PATH_AUTO), oracle.fp8_linear(f8.weight, f8.scale_inv, "bf16", x8))
