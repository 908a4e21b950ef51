"""ctypes + numpy wrapper around gptq_oracle.c (test infrastructure only).

Arrays cross as numpy buffers: int32 words, uint16 bit patterns of fp16/bf16
values, float32 / float64 results.  Torch tensors are accepted and converted on
the CPU; nothing here touches a GPU.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gptq_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_SO = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DT = {"fp16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile gptq_oracle.c into oracle/lib/liboracle.so (OpenMP when available)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _SO + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC], check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            I = C.c_int
            sigs = {
                "oracle_unpack_codes": [P, I, I, I, P],
                "oracle_pack_codes": [P, I, I, I, P],
                "oracle_unpack_zeros": [P, I, I, I, P],
                "oracle_pack_zeros": [P, I, I, I, P],
                "oracle_num_groups": [I, I],
                "oracle_dequant": [P, P, P, I, P, I, I, I, I, P],
                "oracle_linear": [P, P, P, I, P, I, I, I, I, P, I, P, I, P, I, P],
                "oracle_dequant_ex": [P, P, P, I, P, I, I, I, I, I, P],
                "oracle_linear_ex": [P, P, P, I, P, I, I, I, I, I, P, I, P, I, P, I, P, I, P],
                "oracle_round_fp32": [P, C.c_long, I, P],
                "oracle_e4m3_to_float": [P, C.c_long, P],
                "oracle_fp8_dequant": [P, P, I, I, P],
                "oracle_fp8_linear": [P, P, I, I, I, P, I, P, I, P, I, P],
                "oracle_runtime_layout_fp8": [P, I, I, P, P, P],
                "oracle_check_rules": [I, I, I, I, I, I, I, I, P, I],
                "oracle_runtime_dims": [P, I, I, I, P, P],
                "oracle_runtime_layout": [P, P, P, P, I, I, I, I, P, P, P, P, P],
                "oracle_num_threads": [],
                "oracle_set_num_threads": [I],
                "oracle_awq_unpack": [P, I, I, P],
                "oracle_awq_pack": [P, I, I, P],
                "oracle_awq_dequant": [P, P, P, I, I, I, I, P],
                "oracle_awq_linear": [P, P, P, I, I, I, I, P, I, P, I, P, I, P],
                "oracle_awq_to_gptq_fields": [P, P, I, I, I, P, P],
            }
            for name, args in sigs.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = I
            L.oracle_set_num_threads.restype = None
            L.oracle_half_to_float.argtypes = [C.c_uint16, I]
            L.oracle_half_to_float.restype = C.c_float
            _lib = L
    return _lib


def _np(a, dtype):
    """torch tensor or array -> contiguous numpy array viewed as dtype (bit patterns kept)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype in (torch.float16, torch.bfloat16):
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:
        pass
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype != np.dtype(dtype):
        a = a.view(dtype)
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle: {what} rejected its arguments")


def num_groups(K: int, group_size: int) -> int:
    return lib().oracle_num_groups(K, group_size)


def unpack_codes(qweight, bits: int) -> np.ndarray:
    qw = _np(qweight, np.int32)
    K, N = qw.shape[0] * 32 // bits, qw.shape[1]
    out = np.empty((K, N), np.uint8)
    _check(lib().oracle_unpack_codes(_p(qw), K, N, bits, _p(out)), "unpack_codes")
    return out


def pack_codes(codes, bits: int) -> np.ndarray:
    c = _np(codes, np.uint8)
    K, N = c.shape
    out = np.empty((K * bits // 32, N), np.int32)
    _check(lib().oracle_pack_codes(_p(c), K, N, bits, _p(out)), "pack_codes")
    return out


def unpack_zeros(qzeros, N: int, bits: int) -> np.ndarray:
    qz = _np(qzeros, np.int32)
    G = qz.shape[0]
    out = np.empty((G, N), np.int32)
    _check(lib().oracle_unpack_zeros(_p(qz), G, N, bits, _p(out)), "unpack_zeros")
    return out


def pack_zeros(z, bits: int) -> np.ndarray:
    zz = _np(z, np.int32)
    G, N = zz.shape
    out = np.empty((G, N * bits // 32), np.int32)
    _check(lib().oracle_pack_zeros(_p(zz), G, N, bits, _p(out)), "pack_zeros")
    return out


def dequant(qweight, qzeros, scales, g_idx, bits: int, group_size: int, dtype: str,
            zero_offset: int = 1) -> np.ndarray:
    """Dense W float32 [N, K].  zero_offset: 1 for v1 zero fields (stored minus one), 0 for gptq_v2."""
    qw, qz = _np(qweight, np.int32), _np(qzeros, np.int32)
    sc, gi = _np(scales, np.uint16), _np(g_idx, np.int32)
    K, N = qw.shape[0] * 32 // bits, qw.shape[1]
    W = np.empty((N, K), np.float32)
    if zero_offset == 1:
        _check(lib().oracle_dequant(_p(qw), _p(qz), _p(sc), DT[dtype], _p(gi), K, N, bits, group_size, _p(W)),
               "dequant")
    else:
        _check(lib().oracle_dequant_ex(_p(qw), _p(qz), _p(sc), DT[dtype], _p(gi), K, N, bits, group_size,
                                       zero_offset, _p(W)), "dequant_ex")
    return W


def linear(qweight, qzeros, scales, g_idx, bits: int, group_size: int, dtype: str, x,
           rows=None, cols=None, zero_offset: int = 1, bias=None) -> np.ndarray:
    """y[rows][cols] = x[rows] . W[cols]^T (+ bias[cols]) in float64 (all rows / columns by default).

    zero_offset: 1 for v1 zero fields (stored minus one), 0 for gptq_v2.  bias: None, or [N]
    float16 / bfloat16 / float32 (a torch tensor or a numpy float16/float32 array)."""
    qw, qz = _np(qweight, np.int32), _np(qzeros, np.int32)
    sc, gi = _np(scales, np.uint16), _np(g_idx, np.int32)
    xx = _np(x, np.uint16)
    K, N = qw.shape[0] * 32 // bits, qw.shape[1]
    M = xx.shape[0]
    assert xx.shape[1] == K
    r = np.arange(M, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    y = np.empty((len(r), len(c)), np.float64)
    if zero_offset == 1 and bias is None:
        _check(lib().oracle_linear(_p(qw), _p(qz), _p(sc), DT[dtype], _p(gi), K, N, bits, group_size,
                                   _p(xx), M, _p(r), len(r), _p(c), len(c), _p(y)), "linear")
        return y
    b, kind = _bias(bias, N)
    _check(lib().oracle_linear_ex(_p(qw), _p(qz), _p(sc), DT[dtype], _p(gi), K, N, bits, group_size, zero_offset,
                                  _p(b), kind, _p(xx), M, _p(r), len(r), _p(c), len(c), _p(y)), "linear_ex")
    return y


def _bias(bias, N):
    """(array, kind) for oracle_linear_ex: kind 0 fp16 bits, 1 bf16 bits, 2 float32."""
    if bias is None:
        return None, 0
    import torch
    if isinstance(bias, torch.Tensor):
        t = bias.detach().cpu().contiguous()
        assert t.numel() == N
        if t.dtype == torch.float32:
            return t.numpy(), 2
        kind = {torch.float16: 0, torch.bfloat16: 1}[t.dtype]
        return t.view(torch.int16).numpy().view(np.uint16), kind
    a = np.ascontiguousarray(bias)
    assert a.size == N
    if a.dtype == np.float32:
        return a, 2
    assert a.dtype == np.float16
    return a.view(np.uint16), 0


def round_fp32(values, dtype: str) -> np.ndarray:
    """float32 values -> fp16 / bf16 bits (uint16), round to nearest even."""
    import torch
    if isinstance(values, torch.Tensor):
        values = values.detach().cpu().contiguous().numpy()
    v = np.ascontiguousarray(values, np.float32)
    out = np.empty(v.shape, np.uint16)
    _check(lib().oracle_round_fp32(_p(v.view(np.uint32)), v.size, DT[dtype], _p(out)), "round_fp32")
    return out


def check_rules(bits, qweight_shape, qzeros_shape, scales_shape, in_features, g_idx=None) -> int:
    gi = _np(g_idx, np.int32)
    n = 0 if gi is None else gi.shape[0]
    return lib().oracle_check_rules(bits, qweight_shape[0], qweight_shape[1], qzeros_shape[0],
                                    qzeros_shape[1], scales_shape[0], scales_shape[1], in_features,
                                    _p(gi), n)


def runtime_dims(g_idx, K: int, N: int, group_size: int) -> tuple[int, int]:
    gi = _np(g_idx, np.int32)
    kr, npad = C.c_int(), C.c_int()
    _check(lib().oracle_runtime_dims(_p(gi), K, N, group_size, C.byref(kr), C.byref(npad)), "runtime_dims")
    return kr.value, npad.value


def runtime_layout(qweight, qzeros, scales, g_idx, bits: int, group_size: int) -> dict:
    """Expected contents of a runtime handle: wr bytes, perm, cgid, s_r (uint16 bits), z_r."""
    qw, qz = _np(qweight, np.int32), _np(qzeros, np.int32)
    sc, gi = _np(scales, np.uint16), _np(g_idx, np.int32)
    K, N = qw.shape[0] * 32 // bits, qw.shape[1]
    G = num_groups(K, group_size)
    Kr, Np = runtime_dims(gi, K, N, group_size)
    out = dict(
        Kr=Kr, Np=Np, G=G,
        wr=np.empty(Kr // 128 * bits * Np * 16, np.uint8),
        perm=np.empty(Kr, np.int32),
        cgid=np.empty(Kr // 32, np.int32),
        s_r=np.empty((G, Np), np.uint16),
        z_r=np.empty((G, Np), np.uint8),
    )
    _check(lib().oracle_runtime_layout(_p(qw), _p(qz), _p(sc), _p(gi), K, N, bits, group_size,
                                       _p(out["wr"]), _p(out["perm"]), _p(out["cgid"]),
                                       _p(out["s_r"]), _p(out["z_r"])), "runtime_layout")
    return out


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Thread count of the following oracle calls (timing only; results do not depend on it)."""
    lib().oracle_set_num_threads(int(n))


def half_to_float(bits_u16: int, dtype: str) -> float:
    return lib().oracle_half_to_float(bits_u16, DT[dtype])


# ---- AutoAWQ GEMM checkpoints (4-bit, packed along the output dimension) ----

def awq_unpack(packed) -> np.ndarray:
    """int32 [rows, N/8] in AWQ's interleaved order -> uint8 codes [rows, N]."""
    pk = _np(packed, np.int32)
    rows, N = pk.shape[0], pk.shape[1] * 8
    out = np.empty((rows, N), np.uint8)
    _check(lib().oracle_awq_unpack(_p(pk), rows, N, _p(out)), "awq_unpack")
    return out


def awq_pack(codes) -> np.ndarray:
    c = _np(codes, np.uint8)
    rows, N = c.shape
    out = np.empty((rows, N // 8), np.int32)
    _check(lib().oracle_awq_pack(_p(c), rows, N, _p(out)), "awq_pack")
    return out


def awq_dequant(qweight, qzeros, scales, group_size: int, dtype: str) -> np.ndarray:
    """Dense W float32 [N, K] of an AWQ checkpoint."""
    qw, qz, sc = _np(qweight, np.int32), _np(qzeros, np.int32), _np(scales, np.uint16)
    K, N = qw.shape[0], qw.shape[1] * 8
    W = np.empty((N, K), np.float32)
    _check(lib().oracle_awq_dequant(_p(qw), _p(qz), _p(sc), DT[dtype], K, N, group_size, _p(W)), "awq_dequant")
    return W


def awq_linear(qweight, qzeros, scales, group_size: int, dtype: str, x, rows=None, cols=None) -> np.ndarray:
    """y[rows][cols] = x[rows] . W[cols]^T in float64 for an AWQ checkpoint."""
    qw, qz, sc = _np(qweight, np.int32), _np(qzeros, np.int32), _np(scales, np.uint16)
    xx = _np(x, np.uint16)
    K, N = qw.shape[0], qw.shape[1] * 8
    M = xx.shape[0]
    assert xx.shape[1] == K
    r = np.arange(M, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    y = np.empty((len(r), len(c)), np.float64)
    _check(lib().oracle_awq_linear(_p(qw), _p(qz), _p(sc), DT[dtype], K, N, group_size, _p(xx), M,
                                   _p(r), len(r), _p(c), len(c), _p(y)), "awq_linear")
    return y


def awq_to_gptq_fields(qweight, qzeros, group_size: int) -> tuple[np.ndarray, np.ndarray]:
    """The AWQ codes and zero fields in GPTQ packing (zero field = the AWQ zero itself)."""
    qw, qz = _np(qweight, np.int32), _np(qzeros, np.int32)
    K, N = qw.shape[0], qw.shape[1] * 8
    G = num_groups(K, group_size)
    qwg = np.empty((K // 8, N), np.int32)
    qzg = np.empty((G, N // 8), np.int32)
    _check(lib().oracle_awq_to_gptq_fields(_p(qw), _p(qz), K, N, group_size, _p(qwg), _p(qzg)), "awq_to_gptq_fields")
    return qwg, qzg


# ---- FP8 block-scaled layers (float8_e4m3fn weight [N, K], float32 scale_inv per 128 x 128) ----

def _fp8_bytes(weight) -> np.ndarray:
    import torch
    if isinstance(weight, torch.Tensor):
        t = weight.detach().cpu().contiguous()
        return t.view(torch.uint8).numpy() if t.dtype != torch.uint8 else t.numpy()
    return np.ascontiguousarray(weight, np.uint8)


def e4m3_to_float(codes) -> np.ndarray:
    b = _fp8_bytes(codes)
    out = np.empty(b.shape, np.float32)
    _check(lib().oracle_e4m3_to_float(_p(b), b.size, _p(out)), "e4m3_to_float")
    return out


def fp8_dequant(weight, scale_inv) -> np.ndarray:
    """Dense W float32 [N, K]."""
    w, s = _fp8_bytes(weight), _np(scale_inv, np.float32)
    N, K = w.shape
    W = np.empty((N, K), np.float32)
    _check(lib().oracle_fp8_dequant(_p(w), _p(s), K, N, _p(W)), "fp8_dequant")
    return W


def fp8_linear(weight, scale_inv, dtype: str, x, rows=None, cols=None) -> np.ndarray:
    """y[rows][cols] = x[rows] . W[cols]^T in float64."""
    w, s, xx = _fp8_bytes(weight), _np(scale_inv, np.float32), _np(x, np.uint16)
    N, K = w.shape
    M = xx.shape[0]
    assert xx.shape[1] == K
    r = np.arange(M, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    y = np.empty((len(r), len(c)), np.float64)
    _check(lib().oracle_fp8_linear(_p(w), _p(s), DT[dtype], K, N, _p(xx), M, _p(r), len(r), _p(c), len(c),
                                   _p(y)), "fp8_linear")
    return y


def runtime_layout_fp8(weight) -> dict:
    w = _fp8_bytes(weight)
    N, K = w.shape
    Kr, Np = runtime_dims(None, K, N, 128)
    out = dict(Kr=Kr, Np=Np, G=num_groups(K, 128), wr=np.empty(Kr // 128 * 8 * Np * 16, np.uint8),
               perm=np.empty(Kr, np.int32), cgid=np.empty(Kr // 32, np.int32))
    _check(lib().oracle_runtime_layout_fp8(_p(w), K, N, _p(out["wr"]), _p(out["perm"]), _p(out["cgid"])),
           "runtime_layout_fp8")
    return out
