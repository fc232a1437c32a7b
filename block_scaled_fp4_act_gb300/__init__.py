"""Python binding of libfp4moe.so: the quantized MoE expert projection on GB300.

Argument marshalling only. Each function takes torch tensors that already live on the
current CUDA device, passes their pointers and sizes to the C ABI declared in
include/fp4moe.h, and raises Fp4Error on a non-zero status. Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch fallback.
If the compiled library is missing, the first call raises.
"""
import ctypes
import os

from . import build as _build

NVFP4 = 0
MXFP4 = 1

FP4_OK = 0
FP4_ERR_ARG = -1
FP4_ERR_SHAPE = -2
FP4_ERR_ALIGN = -3
FP4_ERR_LAUNCH = -4
FP4_ERR_DEVICE = -5
FP4_ERR_WORKSPACE = -6

FP4_DEVERR_OFFSETS = 1
FP4_DEVERR_ROW_ID = 2
FP4_DEVERR_TIMEOUT = 4

PATH_AUTO = 0
PATH_STREAM = 1
PATH_TC = 2

LIB_PATH = _build.LIB
_lib = None


class Fp4Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        lib = _lib
        name = lib.fp4_status_string(status).decode() if lib else str(status)
        detail = lib.fp4_last_error().decode() if lib else ""
        super().__init__("%s failed: %s %s" % (what, name, detail))


def lib():
    """The loaded C library with argument types set (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfp4moe.so is not built; run block_scaled_fp4_act_gb300.build"
                               ".build() (nvcc, sm_103a) first")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                ctypes.c_size_t)
        L.act_quant_fp8.argtypes = [P, P, P, i64, i64, P]
        L.act_quant_fp8.restype = i32
        L.fp4_expert_gemm.argtypes = [P, P, P, f32, i32, P, i64, i64, i64, P, P, P, sz, P]
        L.fp4_expert_gemm.restype = i32
        L.fp4_grouped_workspace_size.argtypes = [i64, i64, i64, i64, i32]
        L.fp4_grouped_workspace_size.restype = sz
        L.fp4_grouped_expert_gemm.argtypes = [P, i64, P, P, i32, i64, P, P, P, i32, P, i64, i64,
                                              P, sz, P]
        L.fp4_grouped_expert_gemm.restype = i32
        L.fp4_grouped_expert_gemm_noalloc.argtypes = [P, i64, P, P, i32, i64, P, P, P, i32, P,
                                                       i64, i64, P]
        L.fp4_grouped_expert_gemm_noalloc.restype = i32
        L.fp4_gemm_mirror.argtypes = [P, P, P, P, f32, i32, P, i64, i64, i64, P]
        L.fp4_gemm_mirror.restype = i32
        L.fp4_swiglu_quant.argtypes = [P, P, i64, f32, i64, i64, P, P, P, P]
        L.fp4_swiglu_quant.restype = i32
        L.fp4_gemm_path.argtypes = [i64, i32, i64, i64, i32, i32]
        L.fp4_gemm_path.restype = i32
        L.fp4_error_ops.argtypes = [i32, i32, i64]
        L.fp4_error_ops.restype = ctypes.c_double
        L.fp4_force_path.argtypes = [i32]
        L.fp4_force_path.restype = None
        L.fp4_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
        L.fp4_get_device_error.restype = i32
        L.fp4_last_error.argtypes = []
        L.fp4_last_error.restype = ctypes.c_char_p
        L.fp4_status_string.argtypes = [i32]
        L.fp4_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != FP4_OK:
        raise Fp4Error(status, what)


def _need(t, dtype, shape, name):
    import torch
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.device != torch.device("cuda", torch.cuda.current_device()):
        raise ValueError("%s is not on the current CUDA device" % name)


def group_size(recipe):
    return 16 if recipe == NVFP4 else 32


# ---------------------------------------------------------------- entry points

def act_quant_fp8(x, codes=None, scales=None, stream=None):
    """x [rows, k] f32 -> (codes [rows, k] u8, scales [rows, k/128] f32)."""
    import torch
    rows, k = x.shape
    _need(x, torch.float32, None, "x")
    if codes is None:
        codes = torch.empty((rows, k), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, k // 128), dtype=torch.float32, device=x.device)
    _need(codes, torch.uint8, (rows, k), "codes")
    _need(scales, torch.float32, (rows, k // 128), "scales")
    _check(lib().act_quant_fp8(_ptr(x), _ptr(codes), _ptr(scales), rows, k, _stream(stream)),
           "act_quant_fp8")
    return codes, scales


def fp4_expert_gemm(x, w, wscale, scale2, recipe, out=None, codes_out=None, scales_out=None,
                    workspace=None, stream=None):
    """One expert: x [g,k] f32, w [n,k/2] u8, wscale [n,k/gs] u8 -> out [g,n] f32."""
    import torch
    g, k = x.shape
    n = w.shape[0]
    _need(x, torch.float32, None, "x")
    _need(w, torch.uint8, (n, k // 2), "w")
    _need(wscale, torch.uint8, (n, k // group_size(recipe)), "wscale")
    if out is None:
        out = torch.empty((g, n), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, (g, n), "out")
    if codes_out is not None:
        _need(codes_out, torch.uint8, (g, k), "codes_out")
        _need(scales_out, torch.float32, (g, k // 128), "scales_out")
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, torch.uint8, None, "workspace")
        ws_bytes = workspace.numel()
    _check(lib().fp4_expert_gemm(_ptr(x), _ptr(w), _ptr(wscale), float(scale2), int(recipe),
                                 _ptr(out), g, n, k, _ptr(codes_out), _ptr(scales_out),
                                 _ptr(workspace), ws_bytes, _stream(stream)),
           "fp4_expert_gemm")
    return out


def fp4_grouped_workspace_size(num_tokens, total_rows, n, k, recipe):
    return int(lib().fp4_grouped_workspace_size(num_tokens, total_rows, n, k, int(recipe)))


def fp4_grouped_expert_gemm(x, row_ids, offsets, w, wscale, scale2, recipe, out=None,
                            workspace=None, stream=None):
    """All experts of one projection.

    x [T,k] f32; row_ids [P] int32 or None; offsets [E+1] int32; w [E,n,k/2] u8;
    wscale [E,n,k/gs] u8; scale2 [E] f32 (NVFP4) -> out [P,n] f32."""
    import torch
    T, k = x.shape
    E, n = w.shape[0], w.shape[1]
    _need(x, torch.float32, None, "x")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    if row_ids is not None:
        _need(row_ids, torch.int32, None, "row_ids")
        P = row_ids.numel()
    else:
        P = T
    _need(w, torch.uint8, (E, n, k // 2), "w")
    _need(wscale, torch.uint8, (E, n, k // group_size(recipe)), "wscale")
    if scale2 is not None:
        _need(scale2, torch.float32, (E,), "scale2")
    if out is None:
        out = torch.empty((P, n), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, (P, n), "out")
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, torch.uint8, None, "workspace")
        ws_bytes = workspace.numel()
    _check(lib().fp4_grouped_expert_gemm(_ptr(x), T, _ptr(row_ids), _ptr(offsets), E, P, _ptr(w),
                                         _ptr(wscale), _ptr(scale2), int(recipe), _ptr(out), n, k,
                                         _ptr(workspace), ws_bytes, _stream(stream)),
           "fp4_grouped_expert_gemm")
    return out


def fp4_grouped_expert_gemm_noalloc(x, row_ids, offsets, w, wscale, scale2, recipe, out=None,
                                    stream=None):
    """As fp4_grouped_expert_gemm, for callers that cannot allocate device memory: runs the
    tensor-core path with the library's fixed 32 MiB scratch (total_rows*k*2+1024 bytes at
    most) instead of a workspace. Calls that overlap on the GPU race on that scratch."""
    import torch
    T, k = x.shape
    E, n = w.shape[0], w.shape[1]
    _need(x, torch.float32, None, "x")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    if row_ids is not None:
        _need(row_ids, torch.int32, None, "row_ids")
        P = row_ids.numel()
    else:
        P = T
    _need(w, torch.uint8, (E, n, k // 2), "w")
    _need(wscale, torch.uint8, (E, n, k // group_size(recipe)), "wscale")
    if scale2 is not None:
        _need(scale2, torch.float32, (E,), "scale2")
    if out is None:
        out = torch.empty((P, n), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, (P, n), "out")
    _check(lib().fp4_grouped_expert_gemm_noalloc(_ptr(x), T, _ptr(row_ids), _ptr(offsets), E, P,
                                                 _ptr(w), _ptr(wscale), _ptr(scale2), int(recipe),
                                                 _ptr(out), n, k, _stream(stream)),
           "fp4_grouped_expert_gemm_noalloc")
    return out


def fp4_gemm_mirror(codes, scales, w, wscale, scale2, recipe, out=None, stream=None):
    """One expert from quantised activations in the page's own kernel order, bit for bit:
    codes [g,k] u8, scales [g,k/128] f32, w [n,k/2] u8, wscale [n,k/gs] u8 -> out [g,n]."""
    import torch
    g, k = codes.shape
    n = w.shape[0]
    _need(codes, torch.uint8, (g, k), "codes")
    _need(scales, torch.float32, (g, k // 128), "scales")
    _need(w, torch.uint8, (n, k // 2), "w")
    _need(wscale, torch.uint8, (n, k // group_size(recipe)), "wscale")
    if out is None:
        out = torch.empty((g, n), dtype=torch.float32, device=codes.device)
    _need(out, torch.float32, (g, n), "out")
    _check(lib().fp4_gemm_mirror(_ptr(codes), _ptr(scales), _ptr(w), _ptr(wscale), float(scale2),
                                 int(recipe), _ptr(out), g, n, k, _stream(stream)),
           "fp4_gemm_mirror")
    return out


def fp4_swiglu_quant(gate, up, limit, want_h=False, codes=None, scales=None, h_out=None,
                     stream=None):
    """SwiGLU with the swiglu_limit clamps, fused with the e4m3 requantisation of h.

    gate, up: f32 CUDA tensors [rows, inter] with unit column stride and the same row
    stride (e.g. the two halves of a fused gate/up output). Returns (codes [rows, inter]
    u8, scales [rows, inter/128] f32, h [rows, inter] f32 or None)."""
    import torch
    if gate.dtype != torch.float32 or up.dtype != torch.float32 or not gate.is_cuda:
        raise ValueError("gate and up must be f32 CUDA tensors")
    if gate.shape != up.shape or gate.dim() != 2:
        raise ValueError("gate and up must have the same 2-D shape")
    if gate.stride(1) != 1 or up.stride(1) != 1 or gate.stride(0) != up.stride(0):
        raise ValueError("gate and up need unit column stride and one row stride")
    rows, inter = gate.shape
    ld = gate.stride(0) if rows > 1 else inter
    if codes is None:
        codes = torch.empty((rows, inter), dtype=torch.uint8, device=gate.device)
    if scales is None:
        scales = torch.empty((rows, inter // 128), dtype=torch.float32, device=gate.device)
    _need(codes, torch.uint8, (rows, inter), "codes")
    _need(scales, torch.float32, (rows, inter // 128), "scales")
    if want_h and h_out is None:
        h_out = torch.empty((rows, inter), dtype=torch.float32, device=gate.device)
    if h_out is not None:
        _need(h_out, torch.float32, (rows, inter), "h_out")
    _check(lib().fp4_swiglu_quant(_ptr(gate), _ptr(up), ld, float(limit), rows, inter,
                                  _ptr(h_out), _ptr(codes), _ptr(scales), _stream(stream)),
           "fp4_swiglu_quant")
    return codes, scales, h_out


def fp4_gemm_path(total_rows, num_experts, n, k, recipe, have_workspace=True):
    return int(lib().fp4_gemm_path(total_rows, num_experts, n, k, int(recipe),
                                   1 if have_workspace else 0))


def fp4_error_ops(path, recipe, k):
    return float(lib().fp4_error_ops(int(path), int(recipe), int(k)))


def fp4_force_path(path):
    lib().fp4_force_path(int(path))


def fp4_get_device_error(stream=None):
    """Synchronise the stream; return the device error bits (0 = none) and clear them."""
    bits = ctypes.c_uint(0)
    st = lib().fp4_get_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (FP4_OK, FP4_ERR_DEVICE):
        raise Fp4Error(st, "fp4_get_device_error")
    return int(bits.value)


def workspace_for(num_tokens, total_rows, n, k, recipe, device=None):
    """Allocate (with torch) the workspace a grouped call of this shape may use."""
    import torch
    nbytes = fp4_grouped_workspace_size(num_tokens, total_rows, n, k, recipe)
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
