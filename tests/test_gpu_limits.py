"""GPU parity at the size limits the boundary documents (K up to 131072, N up to 262144), on both
kernel families, on sampled outputs against the oracle.  Very long K makes the per-block and
per-group tables of both kernels large; the planners then fall back to narrower layouts."""
import numpy as np
import pytest
import torch

from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm

pytestmark = pytest.mark.gpu


def _sampled(ck, h, M, path, rows_n=2, cols_n=96, seed=0):
    s = ck.spec
    x = synth.make_x(M, s.K, s.dtype, seed=M + seed)
    y = run_gemm(h, x, s.N, path)
    rows = np.unique(np.linspace(0, M - 1, min(M, rows_n)).astype(np.int32))
    cols = np.sort(np.random.default_rng(M).choice(s.N, min(cols_n, s.N), replace=False)).astype(np.int32)
    compare(y[rows][:, cols], oracle_y(ck, x, rows, cols))


@pytest.mark.parametrize("K,gs,da", [(131072, 128, False), (65536, 128, True), (131072, 32, False)])
def test_longest_k(K, gs, da):
    spec = synth.LayerSpec(K, 256, 4, gs, da, False, "bf16")
    ck = synth.make_checkpoint(spec, seed=K // 1024 + gs)
    h = repack(ck)
    gptq.gptq_reserve(h, 300)
    for M in (1, 8, 16, 28):
        _sampled(ck, h, M, gptq.PATH_SMALL_M)
    for M in (40, 129, 300):
        _sampled(ck, h, M, gptq.PATH_LARGE_M)


def test_widest_n():
    spec = synth.LayerSpec(256, 262144, 4, 128, False, False, "fp16")
    ck = synth.make_checkpoint(spec, seed=5)
    h = repack(ck)
    gptq.gptq_reserve(h, 64)
    for M, path in ((1, gptq.PATH_SMALL_M), (8, gptq.PATH_SMALL_M), (64, gptq.PATH_LARGE_M)):
        _sampled(ck, h, M, path, cols_n=256)


def test_beyond_the_limits_is_refused():
    """One row or column past the documented limits: refused by the host checks (UNSUPPORTED, no
    handle) before any device memory is touched."""
    import ctypes as C
    ck = synth.make_checkpoint(synth.LayerSpec(256, 256, 4, 128), seed=1)
    q, z, sc = ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda()
    for K, N in ((131072 + 32, 256), (256, 262144 + 32)):
        out = C.c_void_p()
        rc = gptq.lib().gptq_repack(q.data_ptr(), z.data_ptr(), sc.data_ptr(), None, K, N, 4, 128, 0, None, C.byref(out))
        assert rc == 2 and out.value is None
