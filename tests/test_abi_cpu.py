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


def test_null_handle_plan_and_stall_hook():
    L = gptq.lib()
    plan = gptq.GptqPlan()
    assert L.gptq_gemm_plan(None, 1, 0, C.byref(plan)) == 1
    assert L.gptq_set_test_stall(None, 1, 1000000) == 1


def _noalloc_args(K=512, N=256, bits=4, gs=128):
    import torch
    from weight_only_quantized_gb300 import synth
    ck = synth.make_checkpoint(synth.LayerSpec(K, N, bits, gs), seed=3)
    G, Np = ck.spec.G, -(-N // 256) * 256
    kr_cap = -(-(K + 31 * G) // 128) * 128
    bufs = dict(wr=torch.empty(kr_cap // 128 * bits * Np * 16, dtype=torch.uint8),
                perm=torch.empty(kr_cap, dtype=torch.int32), cgid=torch.empty(kr_cap // 32, dtype=torch.int32),
                s_r=torch.empty((G, Np), dtype=torch.int16), z_r=torch.empty((G, Np), dtype=torch.uint8))
    return ck, bufs


@pytest.mark.parametrize("short", ["cgid", "s_r", "z_r"])
def test_noalloc_wrapper_rejects_short_outputs_before_any_launch(short):
    """The C entry point takes no capacity for cgid, s_r and z_r, so the binding checks them: a short
    one is refused on the host, before the library is called (these CPU tensors would be refused as
    not on the GPU only after the sizes)."""
    import torch
    ck, b = _noalloc_args()
    b[short] = b[short].flatten()[:-1] if short != "cgid" else b[short][:-1]
    with pytest.raises(gptq.GptqError) as ei:
        gptq.gptq_repack_noalloc(ck.qweight, ck.qzeros, ck.scales, None, 4, 128, b["wr"], b["perm"], b["cgid"],
                                 b["s_r"], b["z_r"])
    assert ei.value.status == 1 and short in str(ei.value)


def test_noalloc_wrapper_rejects_wrong_dtype_and_host_tensors():
    import torch
    ck, b = _noalloc_args()
    bad = dict(b, perm=b["perm"].view(torch.float32))
    with pytest.raises(gptq.GptqError) as ei:
        gptq.gptq_repack_noalloc(ck.qweight, ck.qzeros, ck.scales, None, 4, 128, **bad)
    assert ei.value.status == 1 and "int32" in str(ei.value)
    with pytest.raises(gptq.GptqError) as ei:     # right sizes, but host memory
        gptq.gptq_repack_noalloc(ck.qweight, ck.qzeros, ck.scales, None, 4, 128, **b)
    assert ei.value.status == 1 and "CUDA device" in str(ei.value)


def test_limits_shared_by_header_and_library():
    text = open(HEADER).read()
    assert "#define GPTQ_MAX_K      131072" in text and "#define GPTQ_MAX_N      262144" in text
    L = gptq.lib()
    out = C.c_void_p()
    dummy = C.c_void_p(4096)
    # one step past each limit is refused before any device work, by both repack entry points
    assert L.gptq_repack(dummy, dummy, dummy, None, 131072 + 32, 256, 4, 128, 0, None, C.byref(out)) == 2
    assert L.gptq_repack(dummy, dummy, dummy, None, 256, 262144 + 32, 4, 128, 0, None, C.byref(out)) == 2
    kr = C.c_int()
    args = [dummy, dummy, dummy, None, 131072 + 32, 256, 4, 128, 0, dummy, C.c_size_t(1 << 40), dummy, dummy,
            1 << 20, dummy, dummy, C.byref(kr), None]
    assert L.gptq_repack_noalloc(*args) == 2


def _c_layout(struct, fields):
    """sizeof and offsetof of a header struct, from a C program compiled against include/gptq.h."""
    import subprocess
    import tempfile
    body = "\n".join(f'  printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields)
    src = (f'#include <stdio.h>\n#include <stddef.h>\n#include "gptq.h"\n'
           f'int main(void) {{\n  printf("sizeof %zu\\n", sizeof({struct}));\n{body}\n  return 0;\n}}\n')
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True,
                       capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


@pytest.mark.parametrize("struct,cls", [("gptq_plan_t", gptq.GptqPlan), ("gptq_info_t", gptq.GptqInfo)])
def test_binding_structs_match_the_header(struct, cls):
    """The ctypes mirrors in the binding have the header's size and field offsets, so a field added
    on one side only is caught without a GPU."""
    fields = [f for f, _ in cls._fields_]
    lay = _c_layout(struct, fields)
    assert lay["sizeof"] == C.sizeof(cls)
    for f in fields:
        assert lay[f] == getattr(cls, f).offset, f
