"""C ABI checks that need no GPU: the library builds, loads and exports every function
include/gptq.h declares, and its host-side argument checks reject bad input before any
device work (tensref.org "GPTQ packed checkpoint", "Reject the file when")."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
from weight_only_quantized_gb300 import gptq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gptq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gptq_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 10
    L = gptq.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(gptq.SIGNATURES)


def test_status_strings():
    for code, name in gptq.STATUS.items():
        assert gptq.gptq_status_string(code) == name


def _cs(bits, qw, qz, sc, glen, gs):
    K, N = C.c_int(-1), C.c_int(-1)
    s = gptq.lib().gptq_check_shapes(bits, qw[0], qw[1], qz[0], qz[1], sc[0], sc[1], glen, gs, C.byref(K), C.byref(N))
    return s, K.value, N.value


def test_example_header_shapes_accepted():
    # small-gptq.safetensors: qweight [32,32], qzeros [8,4], scales [8,32], g_idx [256], bits 4
    s, K, N = _cs(4, (32, 32), (8, 4), (8, 32), 256, 32)
    assert s == 0 and (K, N) == (256, 32)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("gs", [-1, 32, 128, 96])
def test_shape_rules_agree_with_oracle(bits, gs):
    """The library's rules and the oracle's independent transcription accept and reject the
    same declared shapes (GPTQ-001..004)."""
    K, N = 512, 64
    G = 1 if gs == -1 else -(-K // gs)
    good = dict(qw=(K // 32 * bits, N), qz=(G, N // 32 * bits), sc=(G, N), glen=K)
    variants = [good,
                dict(good, qw=(K // 32 * bits + 1, N)),
                dict(good, qz=(G, N // 32 * bits + 1)),
                dict(good, sc=(G, N - 1)),
                dict(good, glen=K - 32)]
    for v in variants:
        s, _, _ = _cs(bits, v["qw"], v["qz"], v["sc"], v["glen"], gs)
        g = np.zeros(v["glen"], np.int32)
        in_f = v["qw"][0] * 32 // bits if (v["qw"][0] * 32) % bits == 0 else -1
        rule = oracle.check_rules(bits, v["qw"], v["qz"], v["sc"], in_f, g)
        assert (s == 0) == (rule == 0), (v, s, rule)


@pytest.mark.parametrize("bits,status", [(5, 2), (1, 2), (16, 2)])
def test_bad_bits_rejected(bits, status):
    s, _, _ = _cs(bits, (128, 32), (1, 4), (1, 32), 0, -1)
    assert s == status
    assert "GPTQ-001" in gptq.gptq_last_error_message()


def test_repack_host_checks_fail_before_device_work():
    L = gptq.lib()
    out = C.c_void_p(123)
    dummy = C.c_void_p(4096)        # never dereferenced: every case fails a host check first
    assert L.gptq_repack(None, dummy, dummy, None, 256, 256, 4, 128, 0, None, C.byref(out)) == 1
    assert out.value is None
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 256, 5, 128, 0, None, C.byref(out)) == 2
    assert L.gptq_repack(dummy, dummy, dummy, None, 250, 256, 4, 128, 0, None, C.byref(out)) == 3
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 250, 4, 128, 0, None, C.byref(out)) == 3
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 256, 4, 0, 0, None, C.byref(out)) == 1
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 256, 4, 128, 7, None, C.byref(out)) == 2
    assert L.gptq_repack(C.c_void_p(4098), dummy, dummy, None, 256, 256, 4, 128, 0, None, C.byref(out)) == 5
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 256, 4, 128, 0, None, None) == 1


def test_null_handle_calls():
    L = gptq.lib()
    assert L.gptq_gemm(None, None, None, 1, None) == 1
    assert L.gptq_reserve(None, 4) == 1
    assert L.gptq_destroy(None) == 0
    assert L.gptq_gemm_launches(None, 1, 0) == -1
    assert L.gptq_get_info(None, None) == 1
