"""Python binding of the C ABI in include/gptq.h (argument marshalling only).

Every function here has the C entry point's name and does nothing but turn torch
tensors into pointers and sizes, call the library, and raise on a non-OK status.
All work runs in the CUDA library; there is no Python or CPU fallback: if the
library cannot be built or loaded, the call raises.
"""
from __future__ import annotations

import ctypes as C
import threading
from typing import Optional

import torch

from . import build as _build

GPTQ_OK = 0
STATUS = {0: "GPTQ_OK", 1: "GPTQ_ERR_INVALID_ARG", 2: "GPTQ_ERR_UNSUPPORTED", 3: "GPTQ_ERR_SHAPE",
          4: "GPTQ_ERR_INVALID_GIDX", 5: "GPTQ_ERR_ALIGNMENT", 6: "GPTQ_ERR_WORKSPACE", 7: "GPTQ_ERR_CUDA",
          8: "GPTQ_ERR_DEVICE", 9: "GPTQ_ERR_TIMEOUT"}
PATH_AUTO, PATH_SMALL_M, PATH_LARGE_M = 0, 1, 2
DTYPE = {torch.float16: 0, torch.bfloat16: 1}
REPACK_ZEROS_V2, REPACK_SCALES_FP32 = 1, 2

_lock = threading.Lock()
_lib = None

# Every symbol include/gptq.h declares, with its ctypes signature.
_P, _I, _L = C.c_void_p, C.c_int, C.c_int64


class GptqInfo(C.Structure):
    _fields_ = [("K", C.c_int), ("N", C.c_int), ("bits", C.c_int), ("group_size", C.c_int), ("G", C.c_int),
                ("K_sorted", C.c_int), ("N_padded", C.c_int), ("identity", C.c_int), ("dtype", C.c_int),
                ("reserved_M", C.c_int), ("zero_offset", C.c_int), ("has_bias", C.c_int), ("fp8", C.c_int),
                ("weight_bytes", C.c_size_t),
                ("device_bytes", C.c_size_t)]


class GptqPlan(C.Structure):
    _fields_ = [("path", C.c_int), ("launches", C.c_int), ("grid", C.c_int), ("threads", C.c_int),
                ("smem_bytes", C.c_int), ("consumer_warps", C.c_int), ("m_tiles", C.c_int),
                ("act_order_in_kernel", C.c_int), ("k_splits", C.c_int), ("k_panels", C.c_int),
                ("stages", C.c_int), ("row_passes", C.c_int)]


SIGNATURES = {
    "gptq_check_shapes": (_I, [_I, _L, _L, _L, _L, _L, _L, _L, _I, _P, _P]),
    "gptq_repack": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "gptq_repack_awq": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "gptq_repack_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, C.c_uint, _P, _P]),
    "gptq_set_bias": (_I, [_P, _P, _I, _P]),
    "gptq_repack_fp8": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "gptq_reserve": (_I, [_P, _I]),
    "gptq_gemm": (_I, [_P, _P, _P, _I, _P]),
    "gptq_gemm_path": (_I, [_P, _P, _P, _I, _I, _P]),
    "gptq_gemm_launches": (_I, [_P, _I, _I]),
    "gptq_gemm_k_splits": (_I, [_P, _I, _I]),
    "gptq_destroy": (_I, [_P]),
    "gptq_get_info": (_I, [_P, C.POINTER(GptqInfo)]),
    "gptq_copy_runtime": (_I, [_P, _P, _P, _P, _P, _P]),
    "gptq_device_status": (_I, [_P]),
    "gptq_repack_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, C.c_size_t, _P, _P, _I, _P, _P, _P, _P]),
    "gptq_gemm_plan": (_I, [_P, _I, _I, C.POINTER(GptqPlan)]),
    "gptq_set_test_stall": (_I, [_P, _I, C.c_uint64]),
    "gptq_status_string": (C.c_char_p, [_I]),
    "gptq_last_error_message": (C.c_char_p, []),
}


def lib():
    """The loaded CUDA library (built in-tree on first use if missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


class GptqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def _check(status: int):
    if status != GPTQ_OK:
        msg = lib().gptq_last_error_message().decode()
        raise GptqError(status, msg or STATUS.get(status, str(status)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def gptq_status_string(status: int) -> str:
    return lib().gptq_status_string(status).decode()


def gptq_last_error_message() -> str:
    return lib().gptq_last_error_message().decode()


def gptq_check_shapes(bits: int, qweight_shape, qzeros_shape, scales_shape, g_idx_len: int,
                      group_size: int) -> tuple[int, int]:
    K, N = C.c_int(), C.c_int()
    _check(lib().gptq_check_shapes(bits, qweight_shape[0], qweight_shape[1], qzeros_shape[0], qzeros_shape[1],
                                   scales_shape[0], scales_shape[1], g_idx_len, group_size, C.byref(K), C.byref(N)))
    return K.value, N.value


class Handle:
    """Owns one runtime handle; gptq_destroy runs when it is closed or collected."""

    def __init__(self, raw: int):
        self.raw = raw

    def close(self):
        if self.raw:
            _check(lib().gptq_destroy(C.c_void_p(self.raw)))
            self.raw = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def ptr(self):
        if not self.raw:
            raise GptqError(1, "handle is closed")
        return C.c_void_p(self.raw)


def gptq_repack(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor, g_idx: Optional[torch.Tensor],
                bits: int, group_size: int, stream=None, *, zeros_v2: bool = False,
                dtype: Optional[torch.dtype] = None) -> Handle:
    """Checkpoint tensors (on the current CUDA device) -> runtime handle.

    zeros_v2: the qzeros fields hold the zero itself (gptq_v2) instead of zero - 1.  Float32
    scales are accepted with `dtype` (float16 / bfloat16) naming the layer's compute type; they are
    rounded to it once.  Either option goes through gptq_repack_ex."""
    K, N = gptq_check_shapes(bits, tuple(qweight.shape), tuple(qzeros.shape), tuple(scales.shape),
                             0 if g_idx is None else g_idx.numel(), group_size)
    for name, t, dt in (("qweight", qweight, torch.int32), ("qzeros", qzeros, torch.int32)):
        if t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise GptqError(1, f"{name} must be a contiguous int32 CUDA tensor")
    if scales.dtype not in (torch.float16, torch.bfloat16, torch.float32) or not scales.is_contiguous() \
            or not scales.is_cuda:
        raise GptqError(2, "scales must be a contiguous fp16, bf16 or float32 CUDA tensor")
    flags = REPACK_ZEROS_V2 if zeros_v2 else 0
    if scales.dtype == torch.float32:
        if dtype not in DTYPE:
            raise GptqError(2, "float32 scales need dtype=torch.float16 or torch.bfloat16 (the layer's compute type)")
        flags |= REPACK_SCALES_FP32
    else:
        dtype = scales.dtype if dtype is None else dtype
        if dtype != scales.dtype:
            raise GptqError(2, "16-bit scales must have the layer's dtype")
    if g_idx is not None and (g_idx.dtype != torch.int32 or not g_idx.is_contiguous() or not g_idx.is_cuda):
        raise GptqError(1, "g_idx must be a contiguous int32 CUDA tensor")
    out = C.c_void_p()
    if flags:
        _check(lib().gptq_repack_ex(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), K, N, bits, group_size,
                                    DTYPE[dtype], flags, _stream(stream), C.byref(out)))
    else:
        _check(lib().gptq_repack(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), K, N, bits, group_size,
                                 DTYPE[dtype], _stream(stream), C.byref(out)))
    return Handle(out.value)


def gptq_set_bias(h: Handle, bias: Optional[torch.Tensor], stream=None):
    """Attach bias [N] (the handle's dtype or float32, on the device) to the handle; None detaches."""
    if bias is None:
        _check(lib().gptq_set_bias(h.ptr, None, 0, _stream(stream)))
        return
    info = gptq_get_info(h)
    if bias.dim() != 1 or bias.numel() != info.N or not bias.is_contiguous() or not bias.is_cuda:
        raise GptqError(3, f"bias must be a contiguous CUDA tensor of {info.N} elements")
    handle_dt = torch.bfloat16 if info.dtype == 1 else torch.float16
    if bias.dtype not in (handle_dt, torch.float32):
        raise GptqError(2, f"bias must be {handle_dt} or float32")
    _check(lib().gptq_set_bias(h.ptr, _ptr(bias), 1 if bias.dtype == torch.float32 else 0, _stream(stream)))


def gptq_repack_awq(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor, group_size: int,
                    stream=None) -> Handle:
    """AutoAWQ GEMM tensors (qweight int32 [K, N/8], qzeros int32 [G, N/8], scales [G, N], 4-bit,
    on the current CUDA device) -> runtime handle."""
    for name, t in (("qweight", qweight), ("qzeros", qzeros)):
        if t.dtype != torch.int32 or t.dim() != 2 or not t.is_contiguous() or not t.is_cuda:
            raise GptqError(1, f"{name} must be a contiguous 2-d int32 CUDA tensor")
    if scales.dtype not in DTYPE or scales.dim() != 2 or not scales.is_contiguous() or not scales.is_cuda:
        raise GptqError(2, "scales must be a contiguous 2-d fp16 or bf16 CUDA tensor")
    K, N = qweight.shape[0], qweight.shape[1] * 8
    if group_size != -1 and group_size < 1:
        raise GptqError(1, "group_size must be -1 or >= 1")
    G = 1 if group_size == -1 else -(-K // group_size)
    if tuple(qzeros.shape) != (G, N // 8) or tuple(scales.shape) != (G, N):
        raise GptqError(3, f"AWQ qweight [{K}, {N // 8}] needs qzeros [{G}, {N // 8}] and scales [{G}, {N}]")
    out = C.c_void_p()
    _check(lib().gptq_repack_awq(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size,
                                 DTYPE[scales.dtype], _stream(stream), C.byref(out)))
    return Handle(out.value)


def gptq_repack_fp8(weight: torch.Tensor, scale_inv: torch.Tensor, dtype: torch.dtype, stream=None) -> Handle:
    """FP8 block-scaled layer (weight float8_e4m3fn or its uint8 bytes [N, K], scale_inv float32
    [ceil(N/128), ceil(K/128)], on the current CUDA device) -> runtime handle computing in dtype."""
    if weight.dim() != 2 or weight.element_size() != 1 or not weight.is_contiguous() or not weight.is_cuda:
        raise GptqError(1, "weight must be a contiguous 2-d float8_e4m3fn (or uint8) CUDA tensor")
    if scale_inv.dtype != torch.float32 or not scale_inv.is_contiguous() or not scale_inv.is_cuda:
        raise GptqError(1, "scale_inv must be a contiguous float32 CUDA tensor")
    if dtype not in DTYPE:
        raise GptqError(2, "dtype must be torch.float16 or torch.bfloat16")
    N, K = weight.shape
    if tuple(scale_inv.shape) != (-(-N // 128), -(-K // 128)):
        raise GptqError(3, f"scale_inv must be [{-(-N // 128)}, {-(-K // 128)}] for a [{N}, {K}] weight")
    out = C.c_void_p()
    _check(lib().gptq_repack_fp8(_ptr(weight), _ptr(scale_inv), K, N, DTYPE[dtype], _stream(stream), C.byref(out)))
    return Handle(out.value)


def gptq_reserve(h: Handle, max_M: int):
    _check(lib().gptq_reserve(h.ptr, max_M))


def gptq_gemm(h: Handle, x: torch.Tensor, y: torch.Tensor, M: Optional[int] = None, stream=None):
    """y[:M] = x[:M] . W^T on the stream (default: torch's current stream)."""
    M = x.shape[0] if M is None else M
    _check(lib().gptq_gemm(h.ptr, _ptr(x), _ptr(y), M, _stream(stream)))


def gptq_gemm_path(h: Handle, x: torch.Tensor, y: torch.Tensor, path: int, M: Optional[int] = None, stream=None):
    M = x.shape[0] if M is None else M
    _check(lib().gptq_gemm_path(h.ptr, _ptr(x), _ptr(y), M, path, _stream(stream)))


def gptq_gemm_launches(h: Handle, M: int, path: int = PATH_AUTO) -> int:
    return lib().gptq_gemm_launches(h.ptr, M, path)


def gptq_gemm_k_splits(h: Handle, M: int, path: int = PATH_LARGE_M) -> int:
    return lib().gptq_gemm_k_splits(h.ptr, M, path)


def gptq_destroy(h: Handle):
    h.close()


def gptq_device_status(h: Handle):
    """Raise GptqError(GPTQ_ERR_TIMEOUT) if a kernel of this handle gave up a bounded wait."""
    _check(lib().gptq_device_status(h.ptr))


def gptq_repack_noalloc(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
                        g_idx: Optional[torch.Tensor], bits: int, group_size: int, wr: torch.Tensor,
                        perm: torch.Tensor, cgid: torch.Tensor, s_r: torch.Tensor, z_r: torch.Tensor,
                        stream=None) -> int:
    """Repack into caller-owned device tensors; the library allocates nothing.  Returns K_sorted.

    wr: uint8 (capacity = numel), perm: int32 [kr_capacity], cgid: int32 [kr_capacity // 32],
    s_r: fp16/bf16-sized 2-byte [G, N_padded], z_r: uint8 [G, N_padded].  Every output is checked
    (dtype, contiguity, size, device) before the library is called, since the C entry point takes no
    capacity for cgid, s_r and z_r."""
    K, N = gptq_check_shapes(bits, tuple(qweight.shape), tuple(qzeros.shape), tuple(scales.shape),
                             0 if g_idx is None else g_idx.numel(), group_size)
    if scales.dtype not in DTYPE:
        raise GptqError(2, "scales must be fp16 or bf16")
    G = 1 if group_size == -1 else -(-K // group_size)
    Np = -(-N // 256) * 256
    outs = (("wr", wr, 1), ("perm", perm, 4), ("cgid", cgid, 4), ("s_r", s_r, 2), ("z_r", z_r, 1))
    for name, t, es in outs:
        if not isinstance(t, torch.Tensor) or not t.is_contiguous() or t.element_size() != es:
            raise GptqError(1, f"{name} must be a contiguous tensor of {es}-byte elements")
    if perm.dtype != torch.int32 or cgid.dtype != torch.int32:
        raise GptqError(1, "perm and cgid must be int32")
    if z_r.dtype != torch.uint8:
        raise GptqError(1, "z_r must be uint8")
    if cgid.numel() * 32 < perm.numel():
        raise GptqError(1, f"cgid holds {cgid.numel()} chunks; perm's capacity of {perm.numel()} rows needs "
                           f"{-(-perm.numel() // 32)}")
    if s_r.numel() < G * Np or z_r.numel() < G * Np:
        raise GptqError(1, f"s_r and z_r need at least G * N_padded = {G} * {Np} elements")
    dev = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t, _ in outs:
        if not t.is_cuda or t.device.index != dev:
            raise GptqError(1, f"{name} must be on the current CUDA device")
    kr = C.c_int()
    _check(lib().gptq_repack_noalloc(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), K, N, bits, group_size,
                                     DTYPE[scales.dtype], _ptr(wr), wr.numel() * wr.element_size(), _ptr(perm),
                                     _ptr(cgid), perm.numel(), _ptr(s_r), _ptr(z_r), C.byref(kr), _stream(stream)))
    return kr.value


def gptq_gemm_plan(h: Handle, M: int, path: int = PATH_AUTO) -> GptqPlan:
    """The launch plan gptq_gemm_path would use at M (host only)."""
    plan = GptqPlan()
    _check(lib().gptq_gemm_plan(h.ptr, M, path, C.byref(plan)))
    return plan


def gptq_set_test_stall(h: Handle, on: bool, wait_limit_ns: int = 1_000_000):
    """Test hook: the small-M kernel's producer issues no copy and every wait gives up after
    wait_limit_ns (see include/gptq.h).  Not for production use."""
    _check(lib().gptq_set_test_stall(h.ptr, 1 if on else 0, int(wait_limit_ns)))


def gptq_get_info(h: Handle) -> GptqInfo:
    info = GptqInfo()
    _check(lib().gptq_get_info(h.ptr, C.byref(info)))
    return info


def gptq_copy_runtime(h: Handle) -> dict:
    """The handle's runtime layout, copied to host numpy arrays."""
    import numpy as np
    info = gptq_get_info(h)
    out = dict(Kr=info.K_sorted, Np=info.N_padded, G=info.G,
               wr=np.empty(info.weight_bytes, np.uint8), perm=np.empty(info.K_sorted, np.int32),
               cgid=np.empty(info.K_sorted // 32, np.int32), s_r=np.empty((info.G, info.N_padded), np.uint16),
               z_r=np.empty((info.G, info.N_padded), np.uint8))
    p = lambda a: a.ctypes.data_as(C.c_void_p)
    _check(lib().gptq_copy_runtime(h.ptr, p(out["wr"]), p(out["perm"]), p(out["cgid"]), p(out["s_r"]), p(out["z_r"])))
    return out


class GptqLinear:
    """A GPTQ linear layer on the current CUDA device: repack once, then y = layer(x)."""

    def __init__(self, qweight, qzeros, scales, g_idx, bits: int, group_size: int, stream=None, *, bias=None,
                 zeros_v2: bool = False, dtype: Optional[torch.dtype] = None, _handle=None):
        self.handle = _handle if _handle is not None else gptq_repack(qweight, qzeros, scales, g_idx, bits,
                                                                        group_size, stream, zeros_v2=zeros_v2,
                                                                        dtype=dtype)
        info = gptq_get_info(self.handle)
        self.K, self.N = info.K, info.N
        self.dtype = torch.bfloat16 if info.dtype == 1 else torch.float16
        if bias is not None:
            gptq_set_bias(self.handle, bias, stream)

    @classmethod
    def from_fp8(cls, weight, scale_inv, dtype: torch.dtype, stream=None, *, bias=None) -> "GptqLinear":
        """The same layer object built from an FP8 block-scaled checkpoint (W8A16)."""
        return cls(None, None, None, None, 8, 128, stream, bias=bias,
                   _handle=gptq_repack_fp8(weight, scale_inv, dtype, stream))

    @classmethod
    def from_awq(cls, qweight, qzeros, scales, group_size: int, stream=None, *, bias=None) -> "GptqLinear":
        """The same layer object built from an AutoAWQ GEMM checkpoint."""
        return cls(None, None, scales, None, 4, group_size, stream, bias=bias,
                   _handle=gptq_repack_awq(qweight, qzeros, scales, group_size, stream))

    def __call__(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if x.dtype != self.dtype or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise GptqError(1, f"x must be a contiguous [M, {self.K}] {self.dtype} tensor")
        y = out if out is not None else torch.empty((x.shape[0], self.N), dtype=self.dtype, device=x.device)
        gptq_gemm(self.handle, x, y, x.shape[0], stream)
        return y
