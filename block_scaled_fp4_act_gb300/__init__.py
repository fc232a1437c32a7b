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
FP4_DEVERR_EXPERT_ID = 8

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
        L.fp4_grouped_gate_up_swiglu.argtypes = [P, i64, P, P, i32, i64, P, P, P, i32, f32, P,
                                                 i64, i64, P, sz, P]
        L.fp4_grouped_gate_up_swiglu.restype = i32
        L.fp4_grouped_quantize.argtypes = [P, i64, P, i64, i64, i32, P, sz, P]
        L.fp4_grouped_quantize.restype = i32
        L.fp4_grouped_gemm_quantized.argtypes = [P, sz, i64, P, P, i32, i64, P, P, P, i32, P,
                                                 i64, i64, P]
        L.fp4_grouped_gemm_quantized.restype = i32
        L.fp4_route_topk.argtypes = [P, i64, i32, i32, i32, P, P, P]
        L.fp4_route_topk.restype = i32
        L.fp4_route_csr_workspace_size.argtypes = [i64, i32]
        L.fp4_route_csr_workspace_size.restype = sz
        L.fp4_route_csr.argtypes = [P, i64, i32, i32, P, P, P, P, sz, P]
        L.fp4_route_csr.restype = i32
        L.fp4_moe_combine.argtypes = [P, i64, P, P, i64, i32, i64, P, P]
        L.fp4_moe_combine.restype = i32
        L.fp4_gemm_mirror.argtypes = [P, P, P, P, f32, i32, P, i64, i64, i64, P]
        L.fp4_gemm_mirror.restype = i32
        L.fp4_swiglu_quant.argtypes = [P, P, i64, f32, i64, i64, P, P, P, P]
        L.fp4_swiglu_quant.restype = i32
        L.act_quant_w4a4.argtypes = [P, P, P, P, i64, i64, P]
        L.act_quant_w4a4.restype = i32
        L.fp4_w4a4_workspace_size.argtypes = [i64, i64, i64]
        L.fp4_w4a4_workspace_size.restype = sz
        L.fp4_grouped_expert_gemm_w4a4.argtypes = [P, i64, P, P, i32, i64, P, P, P, P, i64,
                                                   i64, P, sz, P]
        L.fp4_grouped_expert_gemm_w4a4.restype = i32
        L.fp4_w4a4_quantize.argtypes = [P, i64, P, i64, i64, P, sz, P]
        L.fp4_w4a4_quantize.restype = i32
        L.fp4_w4a4_gemm_quantized.argtypes = [P, sz, i64, P, P, i32, i64, P, P, P, P, i64, i64,
                                              P]
        L.fp4_w4a4_gemm_quantized.restype = i32
        L.fp4_w4a4_error_ops.argtypes = [i64]
        L.fp4_w4a4_error_ops.restype = ctypes.c_double
        L.fp4_gemm_path.argtypes = [i64, i32, i64, i64, i32, i32]
        L.fp4_gemm_path.restype = i32
        L.fp4_error_ops.argtypes = [i32, i32, i64]
        L.fp4_error_ops.restype = ctypes.c_double
        L.fp4_force_path.argtypes = [i32]
        L.fp4_force_path.restype = None
        L.fp4_test_stall_next_gemm.argtypes = [i64]
        L.fp4_test_stall_next_gemm.restype = None
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


def fp4_grouped_gate_up_swiglu(x, row_ids, offsets, w, wscale, scale2, recipe, limit,
                               workspace, h=None, stream=None):
    """The gate/up projection with SwiGLU in its epilogue (tensor-core path).

    w [E, 2*inter, k/2] u8 (gate rows, then up rows, per expert) -> h [P, inter] f32."""
    import torch
    T, k = x.shape
    E, n = w.shape[0], w.shape[1]
    inter = n // 2
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
    if h is None:
        h = torch.empty((P, inter), dtype=torch.float32, device=x.device)
    _need(h, torch.float32, (P, inter), "h")
    _need(workspace, torch.uint8, None, "workspace")
    _check(lib().fp4_grouped_gate_up_swiglu(_ptr(x), T, _ptr(row_ids), _ptr(offsets), E, P,
                                            _ptr(w), _ptr(wscale), _ptr(scale2), int(recipe),
                                            float(limit), _ptr(h), inter, k, _ptr(workspace),
                                            workspace.numel(), _stream(stream)),
           "fp4_grouped_gate_up_swiglu")
    return h


def fp4_grouped_quantize(x, row_ids, total_rows, recipe, workspace, stream=None):
    """Stage 1 of the tensor-core path: every routed row of x (x[row_ids[p]], or x[p]
    without row ids) quantised into `workspace` (a uint8 CUDA tensor of at least
    fp4_grouped_workspace_size(...) bytes) for fp4_grouped_gemm_quantized."""
    import torch
    T, k = x.shape
    _need(x, torch.float32, None, "x")
    if row_ids is not None:
        _need(row_ids, torch.int32, (total_rows,), "row_ids")
    _need(workspace, torch.uint8, None, "workspace")
    _check(lib().fp4_grouped_quantize(_ptr(x), T, _ptr(row_ids), int(total_rows), k, int(recipe),
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_grouped_quantize")
    return workspace


def fp4_grouped_gemm_quantized(workspace, num_tokens, row_ids, offsets, w, wscale, scale2,
                               recipe, out, stream=None):
    """Stage 2 on the tensor cores from a workspace fp4_grouped_quantize filled for the same
    tokens, row ids, routed rows, k and recipe: offsets [E+1] int32, w [E,n,k/2],
    wscale [E,n,k/gs], scale2 [E] (NVFP4) -> out [P,n] f32 (caller-owned)."""
    import torch
    E, n = w.shape[0], w.shape[1]
    k = w.shape[2] * 2
    P = out.shape[0]
    if row_ids is not None:
        _need(row_ids, torch.int32, (P,), "row_ids")
    _need(workspace, torch.uint8, None, "workspace")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w, torch.uint8, (E, n, k // 2), "w")
    _need(wscale, torch.uint8, (E, n, k // group_size(recipe)), "wscale")
    if scale2 is not None:
        _need(scale2, torch.float32, (E,), "scale2")
    _need(out, torch.float32, (P, n), "out")
    _check(lib().fp4_grouped_gemm_quantized(_ptr(workspace), workspace.numel(), int(num_tokens),
                                            _ptr(row_ids), _ptr(offsets), E, P, _ptr(w),
                                            _ptr(wscale), _ptr(scale2), int(recipe), _ptr(out), n,
                                            k, _stream(stream)),
           "fp4_grouped_gemm_quantized")
    return out


def fp4_grouped_expert_gemm_noalloc(x, row_ids, offsets, w, wscale, scale2, recipe, out,
                                    stream=None):
    """As fp4_grouped_expert_gemm, for callers that cannot allocate device memory: runs the
    tensor-core path with the library's fixed 32 MiB scratch instead of a workspace (the call
    needs fp4_grouped_workspace_size(...) bytes of it). `out` is required: this binding
    allocates nothing either. Calls that overlap on the GPU race on that scratch."""
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
        raise ValueError("fp4_grouped_expert_gemm_noalloc needs a caller-owned `out`")
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


def fp4_route_topk(logits, topk, renormalize=False, ids=None, weights=None, stream=None):
    """Router: logits [T, E] f32 -> (ids [T, topk] int32, weights [T, topk] f32): the topk
    largest logits per token (ties: lower expert id), best first; softmax weights over all
    experts, or over the selected ones with renormalize."""
    import torch
    T, E = logits.shape
    _need(logits, torch.float32, None, "logits")
    if ids is None:
        ids = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    _need(ids, torch.int32, (T, topk), "ids")
    _need(weights, torch.float32, (T, topk), "weights")
    _check(lib().fp4_route_topk(_ptr(logits), T, E, int(topk), 1 if renormalize else 0, _ptr(ids),
                                _ptr(weights), _stream(stream)), "fp4_route_topk")
    return ids, weights


def fp4_route_csr(ids, num_experts, workspace=None, offsets=None, row_ids=None, pair_rows=None,
                  stream=None):
    """CSR routing from expert ids [T, topk] int32: (offsets [E+1], row_ids [T*topk],
    pair_rows [T, topk]), routed rows grouped by expert in token order."""
    import torch
    T, topk = ids.shape
    _need(ids, torch.int32, None, "ids")
    dev = ids.device
    if workspace is None:
        nbytes = int(lib().fp4_route_csr_workspace_size(T, int(num_experts)))
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    if offsets is None:
        offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    if row_ids is None:
        row_ids = torch.empty(T * topk, dtype=torch.int32, device=dev)
    if pair_rows is None:
        pair_rows = torch.empty((T, topk), dtype=torch.int32, device=dev)
    _need(offsets, torch.int32, (num_experts + 1,), "offsets")
    _need(row_ids, torch.int32, (T * topk,), "row_ids")
    _need(pair_rows, torch.int32, (T, topk), "pair_rows")
    _need(workspace, torch.uint8, None, "workspace")
    _check(lib().fp4_route_csr(_ptr(ids), T, topk, int(num_experts), _ptr(offsets), _ptr(row_ids),
                               _ptr(pair_rows), _ptr(workspace), workspace.numel(),
                               _stream(stream)), "fp4_route_csr")
    return offsets, row_ids, pair_rows


def fp4_moe_combine(out, pair_rows, weights, y=None, stream=None):
    """y [T, n] = per token, sum over its slots j of weights[t, j] * out[pair_rows[t, j]]."""
    import torch
    P, n = out.shape
    T, topk = pair_rows.shape
    _need(out, torch.float32, None, "out")
    _need(pair_rows, torch.int32, None, "pair_rows")
    _need(weights, torch.float32, (T, topk), "weights")
    if y is None:
        y = torch.empty((T, n), dtype=torch.float32, device=out.device)
    _need(y, torch.float32, (T, n), "y")
    _check(lib().fp4_moe_combine(_ptr(out), P, _ptr(pair_rows), _ptr(weights), T, int(topk), n,
                                 _ptr(y), _stream(stream)), "fp4_moe_combine")
    return y


# --------------------------------------------------------------------------- W4A4 variant

def act_quant_w4a4(x, codes=None, scales=None, rowscale=None, stream=None):
    """Two-level W4A4 quantisation: x [rows, k] f32 -> (codes [rows, k/2] u8 nibble pairs,
    scales [rows, k/16] u8 e4m3, rowscale [rows] f32)."""
    import torch
    rows, k = x.shape
    _need(x, torch.float32, None, "x")
    if codes is None:
        codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, k // 16), dtype=torch.uint8, device=x.device)
    if rowscale is None:
        rowscale = torch.empty((rows,), dtype=torch.float32, device=x.device)
    _need(codes, torch.uint8, (rows, k // 2), "codes")
    _need(scales, torch.uint8, (rows, k // 16), "scales")
    _need(rowscale, torch.float32, (rows,), "rowscale")
    _check(lib().act_quant_w4a4(_ptr(x), _ptr(codes), _ptr(scales), _ptr(rowscale), rows, k,
                                _stream(stream)), "act_quant_w4a4")
    return codes, scales, rowscale


def fp4_w4a4_workspace_size(num_tokens, total_rows, k):
    return int(lib().fp4_w4a4_workspace_size(int(num_tokens), int(total_rows), int(k)))


def w4a4_workspace_for(num_tokens, total_rows, k, device=None):
    """A uint8 CUDA tensor sized for the W4A4 grouped calls of this shape."""
    import torch
    b = fp4_w4a4_workspace_size(num_tokens, total_rows, k)
    return torch.empty((max(b, 1),), dtype=torch.uint8, device=device or "cuda")


def fp4_grouped_expert_gemm_w4a4(x, row_ids, offsets, w, wscale, scale2, out=None,
                                 workspace=None, stream=None):
    """All experts of one NVFP4 projection with W4A4 activations: x [T,k] f32, row_ids [P]
    int32 or None, offsets [E+1] int32, w [E,n,k/2] u8, wscale [E,n,k/16] u8, scale2 [E] f32
    -> out [P,n] f32."""
    import torch
    T, k = x.shape
    E, n = w.shape[0], w.shape[1]
    P = row_ids.shape[0] if row_ids is not None else T
    _need(x, torch.float32, None, "x")
    if row_ids is not None:
        _need(row_ids, torch.int32, (P,), "row_ids")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w, torch.uint8, (E, n, k // 2), "w")
    _need(wscale, torch.uint8, (E, n, k // 16), "wscale")
    _need(scale2, torch.float32, (E,), "scale2")
    if out is None:
        out = torch.empty((P, n), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, (P, n), "out")
    if workspace is None:
        workspace = w4a4_workspace_for(T, P, k, x.device)
    _need(workspace, torch.uint8, None, "workspace")
    _check(lib().fp4_grouped_expert_gemm_w4a4(_ptr(x), T, _ptr(row_ids), _ptr(offsets), E, P,
                                              _ptr(w), _ptr(wscale), _ptr(scale2), _ptr(out), n,
                                              k, _ptr(workspace), workspace.numel(),
                                              _stream(stream)),
           "fp4_grouped_expert_gemm_w4a4")
    return out


def fp4_w4a4_quantize(x, row_ids, total_rows, workspace, stream=None):
    """The W4A4 quantise pass into `workspace` (see fp4_grouped_expert_gemm_w4a4)."""
    import torch
    T, k = x.shape
    _need(x, torch.float32, None, "x")
    if row_ids is not None:
        _need(row_ids, torch.int32, (total_rows,), "row_ids")
    _need(workspace, torch.uint8, None, "workspace")
    _check(lib().fp4_w4a4_quantize(_ptr(x), T, _ptr(row_ids), int(total_rows), k,
                                   _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_w4a4_quantize")
    return workspace


def fp4_w4a4_gemm_quantized(workspace, num_tokens, row_ids, offsets, w, wscale, scale2, out,
                            stream=None):
    """The W4A4 GEMM from a workspace fp4_w4a4_quantize filled for the same tokens, row
    ids, routed rows and k -> out [P,n] f32 (caller-owned)."""
    import torch
    E, n = w.shape[0], w.shape[1]
    k = w.shape[2] * 2
    P = out.shape[0]
    if row_ids is not None:
        _need(row_ids, torch.int32, (P,), "row_ids")
    _need(workspace, torch.uint8, None, "workspace")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w, torch.uint8, (E, n, k // 2), "w")
    _need(wscale, torch.uint8, (E, n, k // 16), "wscale")
    _need(scale2, torch.float32, (E,), "scale2")
    _need(out, torch.float32, (P, n), "out")
    _check(lib().fp4_w4a4_gemm_quantized(_ptr(workspace), workspace.numel(), int(num_tokens),
                                         _ptr(row_ids), _ptr(offsets), E, P, _ptr(w),
                                         _ptr(wscale), _ptr(scale2), _ptr(out), n, k,
                                         _stream(stream)),
           "fp4_w4a4_gemm_quantized")
    return out


def fp4_w4a4_error_ops(k):
    return float(lib().fp4_w4a4_error_ops(int(k)))


def fp4_gemm_path(total_rows, num_experts, n, k, recipe, have_workspace=True):
    return int(lib().fp4_gemm_path(total_rows, num_experts, n, k, int(recipe),
                                   1 if have_workspace else 0))


def fp4_error_ops(path, recipe, k):
    return float(lib().fp4_error_ops(int(path), int(recipe), int(k)))


def fp4_force_path(path):
    lib().fp4_force_path(int(path))


def fp4_test_stall_next_gemm(wait_limit_cycles):
    """Test hook: the next tensor-core GEMM launched from this thread stalls one pipeline
    wait, gives up after wait_limit_cycles and reports FP4_DEVERR_TIMEOUT."""
    lib().fp4_test_stall_next_gemm(int(wait_limit_cycles))


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
