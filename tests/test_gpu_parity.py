"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle.

Repack results are compared bit for bit with the oracle's runtime-layout function;
GEMM results element by element within max|y - y_ref| <= 4e-3 max|y_ref|.
Sizes span several tiles and a ragged tail; the full-size layers are compared on
sampled rows with all columns.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm, to_device

pytestmark = pytest.mark.gpu

SPECS = [
    synth.LayerSpec(256, 256, 4, 128, False, False, "fp16", 0.005, 0.02),     # tiny layer
    synth.LayerSpec(512, 288, 4, 128, True, False, "bf16"),                   # ragged N tile, act-order
    synth.LayerSpec(320, 96, 2, 64, False, False, "fp16"),                    # K not a multiple of 128
    synth.LayerSpec(384, 320, 3, 128, True, False, "bf16"),
    synth.LayerSpec(384, 320, 3, 128, True, False, "fp16"),
    synth.LayerSpec(256, 256, 8, 32, True, False, "bf16"),
    synth.LayerSpec(256, 256, 8, 32, False, False, "fp16"),
    synth.LayerSpec(1024, 512, 4, -1, False, False, "bf16"),
    synth.LayerSpec(1024, 512, 4, 96, False, True, "fp16"),                   # groups padded to 128
    synth.LayerSpec(1024, 512, 2, 128, False, True, "bf16"),
]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{'sym' if s.sym else ''}{s.dtype}"


@pytest.mark.parametrize("spec", SPECS, ids=_id)
def test_repack_bit_exact(spec):
    ck = synth.make_checkpoint(spec, seed=spec.K + spec.bits)
    h = repack(ck)
    got = gptq.gptq_copy_runtime(h)
    ref = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size)
    for key in ("Kr", "Np", "G"):
        assert got[key] == ref[key], key
    for key in ("perm", "cgid", "s_r", "z_r", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    info = gptq.gptq_get_info(h)
    assert info.identity == int(np.array_equal(ref["perm"], np.arange(ref["Kr"])) and ref["Kr"] == spec.K)


@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 16, 17, 40])
def test_gemm_parity_small_layers(spec, M):
    ck = synth.make_checkpoint(spec, seed=spec.N + spec.bits)
    h = repack(ck)
    gptq.gptq_reserve(h, 64)
    x = synth.make_x(M, spec.K, spec.dtype, seed=M)
    compare(run_gemm(h, x, spec.N), oracle_y(ck, x))


def test_unbalanced_g_idx_parity():
    spec = synth.LayerSpec(512, 256, 4, 64, dtype="bf16")
    ck = synth.make_checkpoint(spec, seed=3)
    rng = np.random.default_rng(1)
    g = rng.integers(0, spec.G, size=spec.K).astype(np.int32)
    g[g == 3] = 2                                        # an empty group
    ck.g_idx = torch.from_numpy(g)
    h = repack(ck)
    got = gptq.gptq_copy_runtime(h)
    ref = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 64)
    for key in ("perm", "cgid", "s_r", "z_r", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    x = synth.make_x(6, spec.K, "bf16", seed=4)
    compare(run_gemm(h, x, spec.N), oracle_y(ck, x))


def test_one_hot_probes_read_single_weights():
    """x = e_k gives y[:, n] = round(W[n, k]): pins the perm direction, the group lookup and the
    tile order.  The product of an exact integer (code - zero) and the scale is rounded once."""
    spec = synth.LayerSpec(512, 256, 4, 64, True, False, "fp16")
    ck = synth.make_checkpoint(spec, seed=21)
    h = repack(ck)
    W = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 64, "fp16")
    ks = [0, 1, 63, 64, 127, 200, 511]
    x = torch.zeros(len(ks), spec.K, dtype=torch.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = run_gemm(h, x, spec.N).float().numpy()
    for i, k in enumerate(ks):
        expect = torch.from_numpy(W[:, k]).to(torch.float16).float().numpy()
        assert np.array_equal(y[i], expect), k


def test_m_zero_launches_nothing():
    spec = synth.LayerSpec(256, 256, 4, 128)
    h = repack(synth.make_checkpoint(spec))
    x = torch.zeros(0, 256, dtype=torch.float16, device="cuda")
    y = torch.zeros(0, 256, dtype=torch.float16, device="cuda")
    gptq.gptq_gemm(h, x, y, 0)
    assert gptq.gptq_gemm_launches(h, 0) == 0


def test_invalid_g_idx_value_is_reported():
    spec = synth.LayerSpec(256, 256, 4, 128, True)
    ck = synth.make_checkpoint(spec)
    ck.g_idx = ck.g_idx.clone()
    ck.g_idx[77] = spec.G                                 # selects no scale row (GPTQ-004)
    with pytest.raises(gptq.GptqError) as ei:
        repack(ck)
    assert ei.value.status == 4 and "g_idx[77]" in str(ei.value)


@pytest.mark.parametrize("spec", SPECS[:4] + SPECS[5:8], ids=_id)
@pytest.mark.parametrize("M", [17, 24, 32])
def test_small_path_four_m_tiles(spec, M):
    """The small-M kernel forced at 17 <= M <= 32 (four 8-row m-tiles)."""
    ck = synth.make_checkpoint(spec, seed=spec.K + 3 * spec.N + M)
    h = repack(ck)
    x = synth.make_x(M, spec.K, spec.dtype, seed=M + 11)
    compare(run_gemm(h, x, spec.N, gptq.PATH_SMALL_M), oracle_y(ck, x))
    gptq.gptq_device_status(h)


def test_small_path_refuses_m_above_its_tiles():
    spec = synth.LayerSpec(256, 256, 4, 128)
    h = repack(synth.make_checkpoint(spec))
    x = torch.zeros(33, 256, dtype=torch.float16, device="cuda")
    y = torch.zeros(33, 256, dtype=torch.float16, device="cuda")
    with pytest.raises(gptq.GptqError) as e:
        gptq.gptq_gemm_path(h, x, y, gptq.PATH_SMALL_M)
    assert e.value.status == 1                          # INVALID_ARG


def test_workspace_required_above_reserve():
    spec = synth.LayerSpec(256, 256, 4, 128, True)
    h = repack(synth.make_checkpoint(spec))
    info = gptq.gptq_get_info(h)
    assert info.identity == 0 and info.reserved_M == 32
    x = torch.zeros(40, 256, dtype=torch.float16, device="cuda")
    y = torch.zeros(40, 256, dtype=torch.float16, device="cuda")
    try:
        gptq.gptq_gemm_path(h, x, y, gptq.PATH_LARGE_M)
    except gptq.GptqError as e:
        assert e.status in (2, 6)                         # UNSUPPORTED until the large-M kernel exists
    else:
        pytest.fail("large-M call above the reserved M must fail")


def test_repeated_calls_and_two_handles_on_two_streams():
    specs = [synth.LayerSpec(512, 256, 4, 128, False, False, "bf16"), synth.LayerSpec(512, 512, 4, 128, True, False, "bf16")]
    cks = [synth.make_checkpoint(s, seed=i) for i, s in enumerate(specs)]
    hs = [repack(c) for c in cks]
    xs = [synth.make_x(8, 512, "bf16", seed=i) for i in range(2)]
    refs = [oracle_y(c, x) for c, x in zip(cks, xs)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty(8, s.N, dtype=torch.bfloat16, device="cuda") for s in specs]
    xd = [x.cuda() for x in xs]
    torch.cuda.synchronize()
    for _ in range(5):
        for i in range(2):
            gptq.gptq_gemm(hs[i], xd[i], outs[i], 8, streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        compare(outs[i].cpu(), refs[i])
    first = outs[0].clone()
    gptq.gptq_gemm(hs[0], xd[0], outs[0], 8)
    torch.cuda.synchronize()
    assert torch.equal(first, outs[0])                    # deterministic reduction order
    for h in hs:
        gptq.gptq_destroy(h)
