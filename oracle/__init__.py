"""CPU oracle of the quantized MoE expert projection -- TEST INFRASTRUCTURE.

A plain, slow, obviously-correct reference (oracle.c, compiled by build.py) wrapped for
numpy. Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package; the library under `block_scaled_fp4_act_gb300/` never does.

Functions and the page passages they follow (memra-engine docs.rs source pages):
  act_quant           0.98.0 src/bin/dsv4_native_gemm_gate.rs, fn quant_rows
  gemm_ref            same page, fn f64_ref (f64 reference + sum of |scaled products|)
  grouped_ref_sampled quant_rows + f64_ref per routed row (CSR expert offsets as in
                      0.71.0 src/bin/kernel_check.rs, grouped MoE GEMM section)
  e4m3_decode         0.71.0 src/bin/kernel_check.rs, F8-E4M3 MMVQ section's decoder
  mirror_gemm         same page, fn mirror_gemm: the page's own kernel order in f32
                      (128 strided partials per output + a fixed halving tree)
  route_topk          0.125.0 src/bin/qwen4exp_gpu_gate.rs, the device-router arm (softmax
                      top-k; body not printed: the reading is stated in oracle.c)
  route_csr           0.71.0 kernel_check.rs, grouped MoE GEMM section (CSR offsets)
  moe_combine         same section (per-routed-row factor on the output), summed per token
  swiglu              0.98.0 dsv4_native_gemm_gate.rs, swiglu_limit saturation cell and
                      the f64 check of main: h = min(g,L) * sigmoid(min(g,L)) * clamp(u,-L,L)
  within_bound        the error model stated in the header comment of
                      dsv4_native_gemm_gate.rs and applied in its f64 comparison:
                      |gpu - f64| <= n_ops * 2^-24 * sum|p_scaled|
  max_rel             the `rel` convention of kernel_check.rs:
                      max|gpu - ref| / max(max|ref|, 1e-3)
  act_quant_w4a4      0.71.0 kernel_check.rs, NVFP4 W4A4 MMQ GEMM section: two-level
                      scaling (row scale + e4m3 micro-scale per 16; readings in oracle.c)
  act_quant_w4a4_v1   same section, the sub-block-only quantiser it is compared with
  gemm_ref_w4a4       f64 GEMM of the dequantised W4A4 operands (+ sum of |products|)
  per_token_rel       same section, the dynamic-range arm's per-token relative error

Pins (tests/test_oracle_pins.py) tie every function to something other than itself.
"""
import ctypes

import numpy as np

from . import build as _build

NVFP4 = 0
MXFP4 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u8, f32, f64, i64, i32 = (ctypes.c_uint8, ctypes.c_float, ctypes.c_double,
                                  ctypes.c_int64, ctypes.c_int)
        P = ctypes.c_void_p
        lib.orc_e4m3_decode.argtypes = [u8]
        lib.orc_e4m3_decode.restype = f64
        lib.orc_e2m1_decode.argtypes = [u8]
        lib.orc_e2m1_decode.restype = f64
        lib.orc_e8m0_decode.argtypes = [u8]
        lib.orc_e8m0_decode.restype = f64
        lib.orc_e4m3_encode.argtypes = [f32]
        lib.orc_e4m3_encode.restype = u8
        lib.orc_pow2_ceil.argtypes = [f32]
        lib.orc_pow2_ceil.restype = f32
        lib.orc_act_quant.argtypes = [P, i64, i64, P, P]
        lib.orc_act_quant.restype = None
        lib.orc_gemm_ref.argtypes = [P, P, P, P, f32, i32, i64, i64, i64, P, P]
        lib.orc_gemm_ref.restype = None
        lib.orc_mirror_gemm.argtypes = [P, P, P, P, f32, i32, i64, i64, i64, P]
        lib.orc_mirror_gemm.restype = None
        lib.orc_swiglu.argtypes = [P, P, i64, i64, i64, f32, P]
        lib.orc_swiglu.restype = None
        lib.orc_grouped_ref_sampled.argtypes = [P, i64, i64, P, P, i32, i64, P, P, P, i32, i64,
                                                P, P, i64, P, P, P, P]
        lib.orc_grouped_ref_sampled.restype = i32
        lib.orc_route_topk.argtypes = [P, i64, i32, i32, i32, P, P]
        lib.orc_route_topk.restype = None
        lib.orc_route_csr.argtypes = [P, i64, i32, i32, P, P, P]
        lib.orc_route_csr.restype = i32
        lib.orc_moe_combine.argtypes = [P, P, P, i64, i32, i64, P, P]
        lib.orc_moe_combine.restype = None
        lib.orc_e2m1_encode.argtypes = [f32]
        lib.orc_e2m1_encode.restype = u8
        lib.orc_act_quant_w4a4.argtypes = [P, i64, i64, P, P, P]
        lib.orc_act_quant_w4a4.restype = None
        lib.orc_act_quant_w4a4_v1.argtypes = [P, i64, i64, P, P]
        lib.orc_act_quant_w4a4_v1.restype = None
        lib.orc_gemm_ref_w4a4.argtypes = [P, P, P, P, P, f32, i64, i64, i64, P, P]
        lib.orc_gemm_ref_w4a4.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- codecs

def e4m3_decode(codes):
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e2m1_decode(nibbles):
    lib = _load()
    table = np.array([lib.orc_e2m1_decode(i) for i in range(16)], dtype=np.float64)
    return table[np.asarray(nibbles, dtype=np.uint8) & 0x0F]


def e8m0_decode(exps):
    lib = _load()
    table = np.array([lib.orc_e8m0_decode(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(exps, dtype=np.uint8)]


def e4m3_encode(values):
    """Element-wise nearest-even e4m3 code of f32 values (one C call per element)."""
    lib = _load()
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    enc = lib.orc_e4m3_encode
    for i in range(flat_v.size):
        flat_o[i] = enc(float(flat_v[i]))
    return out


def pow2_ceil(values):
    lib = _load()
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.float32)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    for i in range(flat_v.size):
        flat_o[i] = lib.orc_pow2_ceil(float(flat_v[i]))
    return out


def e4m3_threshold(code):
    """Smallest non-negative f32 whose oracle encoding is `code` (0 <= code <= 0x7E).

    Bisection over f32 bit patterns, which are ordered like their values for x >= 0;
    the encoder is monotone there."""
    lib = _load()
    if code == 0:
        return np.float32(0.0)
    lo, hi = 0, 0x43E00000  # bits of 0.0 and 448.0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        v = float(np.array([mid], dtype=np.uint32).view(np.float32)[0])
        if lib.orc_e4m3_encode(v) >= code:
            hi = mid
        else:
            lo = mid
    return np.array([hi], dtype=np.uint32).view(np.float32)[0]


# --------------------------------------------------------------------------- the method

def act_quant(x):
    """x f32 [rows, k] -> (codes u8 [rows, k], scales f32 [rows, k/128])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % 128 == 0
    codes = np.empty((rows, k), dtype=np.uint8)
    scales = np.empty((rows, k // 128), dtype=np.float32)
    _load().orc_act_quant(_ptr(x), rows, k, _ptr(codes), _ptr(scales))
    return codes, scales


def mirror_gemm(codes, scales, w, sc, scale2, recipe):
    """The page's mirror order in f32: codes [g,k] u8, scales [g,k/128] f32, w [n,k/2],
    sc [n,k/gs] -> out f32 [g,n]."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    w = _c(w, np.uint8)
    sc = _c(sc, np.uint8)
    g, k = codes.shape
    n = w.shape[0]
    out = np.empty((g, n), dtype=np.float32)
    _load().orc_mirror_gemm(_ptr(codes), _ptr(scales), _ptr(w), _ptr(sc), float(scale2),
                            int(recipe), g, n, k, _ptr(out))
    return out


def swiglu(gate, up, limit):
    """gate, up f32 [rows, inter] -> h f64 [rows, inter] (the SwiGLU of the page, with
    the swiglu_limit clamps: up on both sides, gate from above, before the sigmoid)."""
    gate = _c(gate, np.float32)
    up = _c(up, np.float32)
    assert gate.shape == up.shape and gate.ndim == 2
    rows, inter = gate.shape
    h = np.empty((rows, inter), dtype=np.float64)
    _load().orc_swiglu(_ptr(gate), _ptr(up), inter, rows, inter, float(limit), _ptr(h))
    return h


def gemm_ref(codes, scales, w, sc, scale2, recipe):
    """f64 reference of one expert: codes [g,k], scales [g,k/128], w [n,k/2], sc [n,k/gs].

    Returns (out f64 [g,n], absp f64 [g,n]) with absp the sum of |scaled products|."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.float32)
    w, sc = _c(w, np.uint8), _c(sc, np.uint8)
    g, k = codes.shape
    n = w.shape[0]
    gs = 16 if recipe == NVFP4 else 32
    assert w.shape == (n, k // 2) and sc.shape == (n, k // gs) and scales.shape == (g, k // 128)
    out = np.empty((g, n), dtype=np.float64)
    absp = np.empty((g, n), dtype=np.float64)
    _load().orc_gemm_ref(_ptr(codes), _ptr(scales), _ptr(w), _ptr(sc), float(scale2), int(recipe),
                         g, n, k, _ptr(out), _ptr(absp))
    return out, absp


def grouped_ref_sampled(x, row_ids, offsets, w, sc, scale2, recipe, sample_p, sample_col):
    """Reference outputs of a grouped call at (routed row, column) samples.

    x [T,k] f32; row_ids [P] int32 or None (routed row p reads x[p]); offsets [E+1];
    w [E,n,k/2]; sc [E,n,k/gs]; scale2 [E] f32 (NVFP4). Returns (out, absp) per sample."""
    x = _c(x, np.float32)
    T, k = x.shape
    offsets = _c(offsets, np.int32)
    E = offsets.size - 1
    P = int(offsets[-1])
    w, sc = _c(w, np.uint8), _c(sc, np.uint8)
    n = w.shape[1]
    s2 = _c(scale2 if scale2 is not None else np.zeros(E), np.float32)
    rid = None if row_ids is None else _c(row_ids, np.int32)
    sp, scol = _c(sample_p, np.int64), _c(sample_col, np.int64)
    order = np.argsort(sp, kind="stable")
    sp_s, sc_s = np.ascontiguousarray(sp[order]), np.ascontiguousarray(scol[order])
    out_s = np.empty(sp.size, dtype=np.float64)
    absp_s = np.empty(sp.size, dtype=np.float64)
    tmpc = np.empty(k, dtype=np.uint8)
    tmps = np.empty(k // 128, dtype=np.float32)
    rc = _load().orc_grouped_ref_sampled(_ptr(x), T, k, _ptr(rid), _ptr(offsets), E, P, _ptr(w),
                                         _ptr(sc), _ptr(s2), int(recipe), n, _ptr(sp_s),
                                         _ptr(sc_s), sp.size, _ptr(out_s), _ptr(absp_s),
                                         _ptr(tmpc), _ptr(tmps))
    if rc != 0:
        raise ValueError("oracle: routed row, row id or column out of range")
    out = np.empty_like(out_s)
    absp = np.empty_like(absp_s)
    out[order] = out_s
    absp[order] = absp_s
    return out, absp


# --------------------------------------------------------------------------- W4A4 variant

def e2m1_encode(values):
    """Element-wise nearest E2M1 code (ties to the even code, saturating at 6, sign kept)."""
    lib = _load()
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    enc = lib.orc_e2m1_encode
    for i in range(flat_v.size):
        flat_o[i] = enc(float(flat_v[i]))
    return out


def act_quant_w4a4(x):
    """Two-level W4A4 activation quantisation: x f32 [rows, k] (k % 16 == 0) ->
    (codes u8 [rows, k/2] nibble pairs, scales u8 [rows, k/16] e4m3, rowscale f32 [rows])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % 16 == 0
    codes = np.empty((rows, k // 2), dtype=np.uint8)
    scales = np.empty((rows, k // 16), dtype=np.uint8)
    rs = np.empty(rows, dtype=np.float32)
    _load().orc_act_quant_w4a4(_ptr(x), rows, k, _ptr(codes), _ptr(scales), _ptr(rs))
    return codes, scales, rs


def act_quant_w4a4_v1(x):
    """The page's sub-block-only quantiser (V1): (codes [rows, k/2], scales [rows, k/16])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % 16 == 0
    codes = np.empty((rows, k // 2), dtype=np.uint8)
    scales = np.empty((rows, k // 16), dtype=np.uint8)
    _load().orc_act_quant_w4a4_v1(_ptr(x), rows, k, _ptr(codes), _ptr(scales))
    return codes, scales


def unpack_nibbles(packed):
    """[rows, k/2] nibble pairs -> [rows, k] nibbles (low nibble = even k)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def dequant_w4a4(codes, scales, rowscale=None):
    """x^ f64 [rows, k] = E2M1(code) * e4m3(scale of its 16-block) * rowscale."""
    q = e2m1_decode(unpack_nibbles(codes))
    s = np.repeat(e4m3_decode(scales), 16, axis=-1)
    x = q * s
    if rowscale is not None:
        x = x * np.asarray(rowscale, dtype=np.float64)[:, None]
    return x


def gemm_ref_w4a4(codes, scales, rowscale, w, sc, scale2):
    """f64 W4A4 reference: codes [g,k/2], scales [g,k/16], rowscale [g] or None,
    w [n,k/2], sc [n,k/16] e4m3, scale2 -> (out f64 [g,n], absp f64 [g,n])."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    w, sc = _c(w, np.uint8), _c(sc, np.uint8)
    g, k2 = codes.shape
    k = 2 * k2
    n = w.shape[0]
    assert scales.shape == (g, k // 16) and w.shape == (n, k2) and sc.shape == (n, k // 16)
    rs = None if rowscale is None else _c(rowscale, np.float32)
    out = np.empty((g, n), dtype=np.float64)
    absp = np.empty((g, n), dtype=np.float64)
    _load().orc_gemm_ref_w4a4(_ptr(codes), _ptr(scales), _ptr(rs), _ptr(w), _ptr(sc),
                              float(scale2), g, n, k, _ptr(out), _ptr(absp))
    return out, absp


def per_token_rel(y, ref):
    """The dynamic-range arm's measure: max over rows of max|y - ref| / max|ref| (rows
    whose reference is all zero count 0)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    worst = 0.0
    for i in range(ref.shape[0]):
        s = float(np.max(np.abs(ref[i]))) if ref.shape[1] else 0.0
        if s > 0.0:
            worst = max(worst, float(np.max(np.abs(y[i] - ref[i]))) / s)
    return worst


# --------------------------------------------------------------------------- routing front-end

def route_topk(logits, topk, renormalize=False):
    """logits f32 [T, E] -> (ids int32 [T, topk], weights f64 [T, topk]): the topk largest
    logits per token (ties: lower expert id first), best first; softmax weights over all
    experts, or over the selected ones with renormalize."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float64)
    _load().orc_route_topk(_ptr(logits), T, E, topk, 1 if renormalize else 0, _ptr(ids), _ptr(w))
    return ids, w


def route_csr(ids, num_experts):
    """ids int32 [T, topk] -> (offsets int32 [E+1], row_ids int32 [T*topk], pair_rows int32
    [T, topk]): routed rows grouped by expert, token order within an expert."""
    ids = _c(ids, np.int32)
    T, topk = ids.shape
    offsets = np.empty(num_experts + 1, dtype=np.int32)
    row_ids = np.empty(T * topk, dtype=np.int32)
    pair_rows = np.empty((T, topk), dtype=np.int32)
    rc = _load().orc_route_csr(_ptr(ids), T, topk, num_experts, _ptr(offsets), _ptr(row_ids),
                               _ptr(pair_rows))
    if rc != 0:
        raise ValueError("oracle: expert id outside [0, num_experts)")
    return offsets, row_ids, pair_rows


def moe_combine(out, pair_rows, weights):
    """out f32 [P, n], pair_rows int32 [T, topk], weights f32 [T, topk] -> (y f64 [T, n],
    absy f64 [T, n]): y[t] = sum_j weights[t, j] * out[pair_rows[t, j]]."""
    out = _c(out, np.float32)
    pair_rows = _c(pair_rows, np.int32)
    weights = _c(weights, np.float32)
    T, topk = pair_rows.shape
    n = out.shape[1]
    y = np.empty((T, n), dtype=np.float64)
    absy = np.empty((T, n), dtype=np.float64)
    _load().orc_moe_combine(_ptr(out), _ptr(pair_rows), _ptr(weights), T, topk, n, _ptr(y),
                            _ptr(absy))
    return y, absy


# --------------------------------------------------------------------------- acceptance

U32 = 2.0 ** -24


def within_bound(gpu, ref, absp, n_ops, abs_floor=0.0):
    """Per-output check of the stated f32 model |gpu - ref| <= n_ops * 2^-24 * absp
    (+ abs_floor: the absolute error of roundings that land in the f32 subnormal range,
    2^-150 each under gradual underflow; 0 where no result can be subnormal).

    Returns (ok, worst err/bound ratio, index of the worst output)."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    absp = np.asarray(absp, dtype=np.float64).reshape(-1)
    err = np.abs(gpu - ref)
    bound = n_ops * U32 * absp + abs_floor
    ok = bool(np.all(err <= bound))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
    i = int(np.argmax(ratio)) if ratio.size else 0
    return ok, float(ratio[i]) if ratio.size else 0.0, i


def max_rel(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(gpu - ref)) / max(float(np.max(np.abs(ref))), 1e-3))


def lib_path():
    return _build.build()


__all__ = ["NVFP4", "MXFP4", "e4m3_decode", "e2m1_decode", "e8m0_decode", "e4m3_encode",
           "pow2_ceil", "e4m3_threshold", "act_quant", "gemm_ref", "grouped_ref_sampled",
           "route_topk", "route_csr", "moe_combine", "within_bound", "max_rel", "lib_path",
           "U32", "e2m1_encode", "act_quant_w4a4", "act_quant_w4a4_v1", "unpack_nibbles",
           "dequant_w4a4", "gemm_ref_w4a4", "per_token_rel"]
