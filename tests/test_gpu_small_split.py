"""GPU parity of the small-M kernel's K split against the oracle.  The K panels of a tile are the
CTAs of one thread-block cluster, and the first CTA of the cluster adds the others' sums (sent into
its shared memory) in panel order.  Two cases split:
  * layers with fewer 32-column tiles than SMs at M <= 8: one tile per cluster;
  * M = 9 .. 16 when x over all of K does not fit in shared memory: each cluster walks a run of
    tiles, and the sums travel through two receive slots that the first CTA frees tile by tile."""
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm

pytestmark = pytest.mark.gpu

SPECS = [
    synth.LayerSpec(8192, 2048, 4, -1, False, False, "fp16"),     # two panels
    synth.LayerSpec(4096, 1024, 4, 128, True, False, "fp16"),     # act-order: the in-kernel permute per panel
    synth.LayerSpec(6144, 512, 3, 64, True, False, "bf16"),
    synth.LayerSpec(8320, 288, 8, 32, False, False, "fp16"),      # 65 blocks: a short last panel; ragged N
    synth.LayerSpec(8192, 512, 2, -1, False, True, "bf16"),
    synth.LayerSpec(8192, 256, 4, 128, False, True, "bf16"),      # 8 tiles: eight panels
]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{s.dtype}"


@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_small_split_parity_and_determinism(spec, M):
    ck = synth.make_checkpoint(spec, seed=spec.K + spec.N + M)
    h = repack(ck)                                                   # no workspace needed
    x = synth.make_x(M, spec.K, spec.dtype, seed=M)
    splits = gptq.gptq_gemm_k_splits(h, M, gptq.PATH_SMALL_M)
    assert splits > 1
    plan = gptq.gptq_gemm_plan(h, M, gptq.PATH_SMALL_M)
    assert plan.k_splits == splits and plan.consumer_warps == 16
    y1 = run_gemm(h, x, spec.N, gptq.PATH_SMALL_M)
    compare(y1, oracle_y(ck, x))
    assert torch.equal(y1, run_gemm(h, x, spec.N, gptq.PATH_SMALL_M))   # same sum order every call


def test_small_split_only_at_small_m_and_few_tiles():
    spec = synth.LayerSpec(8192, 256, 4, 128, True, False, "fp16")
    h = repack(synth.make_checkpoint(spec, seed=1))
    gptq.gptq_reserve(h, 64)
    assert gptq.gptq_gemm_k_splits(h, 1, gptq.PATH_SMALL_M) == 8
    assert gptq.gptq_gemm_plan(h, 1, gptq.PATH_SMALL_M).grid == 8      # one CTA per tile and panel
    # two m-tiles: x over K = 8192 does not fit, x of half of K does
    for M in (9, 16):
        assert gptq.gptq_gemm_k_splits(h, M, gptq.PATH_SMALL_M) == 2
    for M in (17, 28, 32):
        assert gptq.gptq_gemm_k_splits(h, M, gptq.PATH_SMALL_M) == 1
    assert gptq.gptq_gemm_k_splits(h, 64, gptq.PATH_AUTO) == gptq.gptq_gemm_k_splits(h, 64, gptq.PATH_LARGE_M)
    # a layer with at least as many tiles as SMs does not split, nor one whose panels would save
    # too few blocks per CTA
    for K, N in ((1024, 14336), (4096, 2048)):
        hw = repack(synth.make_checkpoint(synth.LayerSpec(K, N, 4, 128, False, True, "bf16"), seed=2))
        assert gptq.gptq_gemm_k_splits(hw, 1, gptq.PATH_SMALL_M) == 1


def test_small_split_with_bias_awq_and_fp8():
    K, N = 4096, 512
    b = torch.randn(N, generator=torch.Generator().manual_seed(2)) * 0.1
    ck = synth.make_awq_checkpoint(K, N, 128, "fp16", seed=3)
    h = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), 128)
    gptq.gptq_set_bias(h, b.half().cuda())
    assert gptq.gptq_gemm_k_splits(h, 4, gptq.PATH_SMALL_M) > 1
    x = synth.make_x(4, K, "fp16", seed=4)
    y_ref = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, 128, "fp16", x) + b.half().double().numpy()[None, :]
    compare(run_gemm(h, x, N, gptq.PATH_SMALL_M), y_ref)
    f8 = synth.make_fp8_checkpoint(K, N, "bf16", seed=5)
    h8 = gptq.gptq_repack_fp8(f8.weight.cuda(), f8.scale_inv.cuda(), torch.bfloat16)
    assert gptq.gptq_gemm_k_splits(h8, 1, gptq.PATH_SMALL_M) > 1
    x8 = synth.make_x(1, K, "bf16", seed=6)
    compare(run_gemm(h8, x8, N, gptq.PATH_SMALL_M), oracle.fp8_linear(f8.weight, f8.scale_inv, "bf16", x8))


def test_small_split_back_to_back_calls_and_graphs():
    """Back-to-back calls of one handle (the next call's CTAs start while this one finishes) and
    of two M values, captured in a CUDA graph and replayed: every result stays right."""
    spec = synth.LayerSpec(8192, 2048, 4, 128, False, False, "bf16")
    ck = synth.make_checkpoint(spec, seed=7)
    h = repack(ck)
    assert gptq.gptq_gemm_k_splits(h, 1, gptq.PATH_SMALL_M) > 1
    xs = {M: synth.make_x(M, spec.K, "bf16", seed=M).cuda() for M in (1, 8)}
    ys = {M: torch.empty(M, spec.N, dtype=torch.bfloat16, device="cuda") for M in xs}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(4):
            for M in (1, 1, 8):
                gptq.gptq_gemm_path(h, xs[M], ys[M], gptq.PATH_SMALL_M)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    for M in (1, 8):
        compare(ys[M].cpu(), oracle_y(ck, xs[M].cpu()))


# M = 9 .. 16: K long enough that x over all of K does not fit in shared memory.  With 76 clusters
# of two CTAs (or 38 of four) on 152 SMs, the 192 to 256 tiles of these layers give runs of two
# to four tiles, so both receive slots are used and freed again.
SPECS_2MT = [
    (synth.LayerSpec(8192, 8192, 4, 128, True, False, "fp16"), (9, 16), 2),    # act-order (pre-pass)
    (synth.LayerSpec(4608, 6144, 3, 64, False, False, "bf16"), (16,), 2),      # panels of 20 and 16 blocks
    (synth.LayerSpec(9216, 4096, 8, 32, True, False, "bf16"), (12,), 2),
    (synth.LayerSpec(9216, 4096, 8, 32, True, False, "bf16"), (16,), 4),       # four panels, the last short
    (synth.LayerSpec(8192, 4096, 2, -1, False, True, "bf16"), (16,), 2),
]


def _id2(c):
    s, Ms, S = c
    return f"{_id(s)}M{'-'.join(map(str, Ms))}S{S}"


@pytest.mark.parametrize("case", SPECS_2MT, ids=_id2)
def test_two_m_tile_split_parity_and_determinism(case):
    spec, Ms, S = case
    ck = synth.make_checkpoint(spec, seed=spec.K + 3 * spec.N)
    h = repack(ck)
    for M in Ms:
        assert gptq.gptq_gemm_k_splits(h, M, gptq.PATH_SMALL_M) == S
        plan = gptq.gptq_gemm_plan(h, M, gptq.PATH_SMALL_M)
        assert plan.k_splits == S and plan.consumer_warps == 8 and plan.m_tiles == 2
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        cap = min(spec.N // 32, sms // S)                         # clusters: runs of tiles, as many
        assert cap * 3 // 4 <= plan.grid <= cap                   # as the GPU holds at once
        x = synth.make_x(M, spec.K, spec.dtype, seed=M + 20)
        y1 = run_gemm(h, x, spec.N, gptq.PATH_SMALL_M)
        compare(y1, oracle_y(ck, x))
        assert torch.equal(y1, run_gemm(h, x, spec.N, gptq.PATH_SMALL_M))   # same sum order every call


def test_two_m_tile_split_with_bias_awq_and_fp8():
    K, N = 8192, 6144
    b = torch.randn(N, generator=torch.Generator().manual_seed(12)) * 0.1
    ck = synth.make_awq_checkpoint(K, N, 128, "fp16", seed=13)
    h = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), 128)
    gptq.gptq_set_bias(h, b.half().cuda())
    assert gptq.gptq_gemm_k_splits(h, 16, gptq.PATH_SMALL_M) == 2
    x = synth.make_x(16, K, "fp16", seed=14)
    y_ref = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, 128, "fp16", x) + b.half().double().numpy()[None, :]
    compare(run_gemm(h, x, N, gptq.PATH_SMALL_M), y_ref)
    f8 = synth.make_fp8_checkpoint(K, N, "bf16", seed=15)
    h8 = gptq.gptq_repack_fp8(f8.weight.cuda(), f8.scale_inv.cuda(), torch.bfloat16)
    assert gptq.gptq_gemm_k_splits(h8, 13, gptq.PATH_SMALL_M) == 2
    x8 = synth.make_x(13, K, "bf16", seed=16)
    compare(run_gemm(h8, x8, N, gptq.PATH_SMALL_M), oracle.fp8_linear(f8.weight, f8.scale_inv, "bf16", x8))


def test_two_m_tile_split_back_to_back_calls_and_graphs():
    """Runs of three and four tiles, called back to back with M = 16 and M = 10 and replayed from a
    CUDA graph: the receive slots' phases carry over no state from one call to the next."""
    spec = synth.LayerSpec(8192, 8192, 4, 128, False, False, "bf16")
    ck = synth.make_checkpoint(spec, seed=17)
    h = repack(ck)
    assert gptq.gptq_gemm_k_splits(h, 16, gptq.PATH_SMALL_M) == 2
    xs = {M: synth.make_x(M, spec.K, "bf16", seed=M + 30).cuda() for M in (10, 16)}
    ys = {M: torch.empty(M, spec.N, dtype=torch.bfloat16, device="cuda") for M in xs}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            for M in (16, 16, 10):
                gptq.gptq_gemm_path(h, xs[M], ys[M], gptq.PATH_SMALL_M)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    gptq.gptq_device_status(h)
    for M in (10, 16):
        compare(ys[M].cpu(), oracle_y(ck, xs[M].cpu()))
