"""GPU parity of the format extensions, through the C ABI, against the oracle: gptq_v2 zero
fields (gptq_repack_ex, GPTQ_REPACK_ZEROS_V2), float32 scales rounded to the layer dtype
(GPTQ_REPACK_SCALES_FP32) and the optional bias (gptq_set_bias).  Layouts bit for bit, GEMMs
element by element within max|y - y_ref| <= 4e-3 max|y_ref|, on both kernel families."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare

pytestmark = pytest.mark.gpu

SPECS = [
    synth.LayerSpec(256, 256, 4, 128, False, False, "fp16"),
    synth.LayerSpec(512, 288, 4, 128, True, False, "bf16"),        # act-order, ragged N tile
    synth.LayerSpec(384, 320, 3, 128, True, False, "fp16"),
    synth.LayerSpec(256, 256, 8, 32, False, False, "bf16"),
    synth.LayerSpec(320, 96, 2, 64, False, False, "fp16"),
]
PATHS = [(gptq.PATH_SMALL_M, [1, 5, 24]), (gptq.PATH_LARGE_M, [1, 40, 129])]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{s.dtype}"


def _dt(name):
    return torch.float16 if name == "fp16" else torch.bfloat16


def _run(h, x_cpu, N, path):
    x = x_cpu.cuda()
    y = torch.full((x.shape[0], N), float("nan"), dtype=x.dtype, device="cuda")
    gptq.gptq_gemm_path(h, x, y, path)
    torch.cuda.synchronize()
    return y.cpu()


def _dev(ck):
    return (ck.qweight.cuda(), ck.qzeros.cuda(), None if ck.g_idx is None else ck.g_idx.cuda())


# ------------------------------------------------------------------ gptq_v2 zero fields
@pytest.mark.parametrize("spec", SPECS, ids=_id)
def test_v2_zeros_layout_and_gemm(spec):
    """Random words are valid v2 checkpoints too: every field 0 .. 2^bits - 1 is a zero."""
    ck = synth.make_checkpoint(spec, seed=spec.K + 3)
    qw, qz, gi = _dev(ck)
    h = gptq.gptq_repack(qw, qz, ck.scales.cuda(), gi, spec.bits, spec.group_size, zeros_v2=True)
    torch.cuda.synchronize()
    info = gptq.gptq_get_info(h)
    assert info.zero_offset == 0
    got = gptq.gptq_copy_runtime(h)
    ref = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size)
    for key in ("perm", "cgid", "s_r", "z_r", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    gptq.gptq_reserve(h, 160)
    for path, Ms in PATHS:
        for M in Ms:
            x = synth.make_x(M, spec.K, spec.dtype, seed=M)
            y_ref = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size,
                                  spec.dtype, x, zero_offset=0)
            compare(_run(h, x, spec.N, path), y_ref)


# ------------------------------------------------------------------ float32 scales
@pytest.mark.parametrize("spec", SPECS, ids=_id)
def test_fp32_scales_rounded_once(spec):
    ck = synth.make_checkpoint(spec, seed=spec.N + 5)
    gen = torch.Generator().manual_seed(spec.K)
    s32 = (torch.rand((spec.G, spec.N), generator=gen, dtype=torch.float64) * 0.008 + 0.002).float()
    s32[0, :8] = torch.tensor([0.0029296875 + 2 ** -21, 1.0009765625, 2 ** -14, 0.01, 65504.0 / 2 ** 20,
                               1.00390625, 3.0517578125e-05, 0.0078125])   # ties and binade edges
    qw, qz, gi = _dev(ck)
    h = gptq.gptq_repack(qw, qz, s32.cuda(), gi, spec.bits, spec.group_size, dtype=_dt(spec.dtype))
    torch.cuda.synchronize()
    s_bits = oracle.round_fp32(s32, spec.dtype)
    got = gptq.gptq_copy_runtime(h)
    ref = oracle.runtime_layout(ck.qweight, ck.qzeros, s_bits, ck.g_idx, spec.bits, spec.group_size)
    for key in ("s_r", "z_r", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    gptq.gptq_reserve(h, 160)
    for path, Ms in PATHS:
        M = Ms[-1]
        x = synth.make_x(M, spec.K, spec.dtype, seed=M + 1)
        y_ref = oracle.linear(ck.qweight, ck.qzeros, s_bits, ck.g_idx, spec.bits, spec.group_size, spec.dtype, x)
        compare(_run(h, x, spec.N, path), y_ref)


# ------------------------------------------------------------------ bias
@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("bias_fp32", [False, True])
def test_bias_in_the_epilogue(spec, bias_fp32):
    ck = synth.make_checkpoint(spec, seed=spec.N + 7)
    qw, qz, gi = _dev(ck)
    h = gptq.gptq_repack(qw, qz, ck.scales.cuda(), gi, spec.bits, spec.group_size)
    gptq.gptq_reserve(h, 160)
    b = torch.randn(spec.N, generator=torch.Generator().manual_seed(3)) * 0.5
    b = b if bias_fp32 else b.to(_dt(spec.dtype))
    gptq.gptq_set_bias(h, b.cuda())
    assert gptq.gptq_get_info(h).has_bias == 1
    for path, Ms in PATHS:
        for M in Ms:
            x = synth.make_x(M, spec.K, spec.dtype, seed=M + 2)
            y_ref = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size,
                                  spec.dtype, x, bias=b)
            compare(_run(h, x, spec.N, path), y_ref)
    # detaching gives back exactly the output of a handle that never had a bias
    x = synth.make_x(5, spec.K, spec.dtype, seed=9)
    gptq.gptq_set_bias(h, None)
    assert gptq.gptq_get_info(h).has_bias == 0
    h0 = gptq.gptq_repack(qw, qz, ck.scales.cuda(), gi, spec.bits, spec.group_size)
    for path, _ in PATHS:
        assert torch.equal(_run(h, x, spec.N, path), _run(h0, x, spec.N, path))


def test_bias_with_awq_handle_and_graph_capture():
    """A bias on an AWQ handle equals the bias on the GPTQ handle of the same weights, also when
    the calls are replayed from a CUDA graph captured after the bias was attached."""
    K, N, gs = 512, 256, 128
    ck = synth.make_awq_checkpoint(K, N, gs, "fp16", seed=4)
    gen = torch.Generator().manual_seed(5)
    zeros = torch.randint(1, 16, (ck.G, N), generator=gen, dtype=torch.uint8).numpy()
    ck.qzeros = torch.from_numpy(oracle.awq_pack(zeros))
    codes = oracle.awq_unpack(ck.qweight)
    h_awq = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), gs)
    h_gptq = gptq.gptq_repack(torch.from_numpy(oracle.pack_codes(codes, 4)).cuda(),
                              torch.from_numpy(oracle.pack_zeros(zeros.astype(np.int32), 4)).cuda(),
                              ck.scales.cuda(), None, 4, gs)
    b = (torch.randn(N, generator=gen) * 0.25).half().cuda()
    gptq.gptq_set_bias(h_awq, b)
    gptq.gptq_set_bias(h_gptq, b)
    for M in (3, 64):
        x = synth.make_x(M, K, "fp16", seed=M).cuda()
        ya = torch.empty(M, N, dtype=torch.float16, device="cuda")
        yg = torch.empty_like(ya)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            gptq.gptq_gemm(h_awq, x, ya)
            gptq.gptq_gemm(h_gptq, x, yg)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ya, yg)
        y_ref = oracle.linear(oracle.pack_codes(codes, 4), oracle.pack_zeros(zeros.astype(np.int32), 4), ck.scales,
                              None, 4, gs, "fp16", x.cpu(), bias=b.cpu())
        compare(ya.cpu(), y_ref)


def test_repack_ex_rejects_unknown_flags_and_fp32_scales_need_a_dtype():
    spec = synth.LayerSpec(256, 256, 4, 128)
    ck = synth.make_checkpoint(spec, seed=1)
    qw, qz, _ = _dev(ck)
    sc = ck.scales.cuda()
    out = C.c_void_p()
    rc = gptq.lib().gptq_repack_ex(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), None, 256, 256, 4, 128, 0, 4,
                                   None, C.byref(out))
    assert rc == 1 and not out.value
    with pytest.raises(gptq.GptqError):
        gptq.gptq_repack(qw, qz, sc.float(), None, 4, 128)
    h = gptq.gptq_repack(qw, qz, sc, None, 4, 128)
    with pytest.raises(gptq.GptqError):
        gptq.gptq_set_bias(h, torch.zeros(255, dtype=torch.float16, device="cuda"))
