"""The C ABI without a GPU: the library loads, exports every function the header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

import block_scaled_fp4_act_gb300 as fp4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4moe.h")


@pytest.fixture(scope="module")
def lib():
    fp4.build.build()
    return fp4.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["act_quant_fp8", "fp4_expert_gemm", "fp4_grouped_expert_gemm",
                 "fp4_grouped_workspace_size", "fp4_get_device_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fp4.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_host_side_argument_checks(lib):
    V = ctypes.c_void_p
    a16 = V(0x10000)           # never dereferenced: every call below fails its checks first
    odd = V(0x10004)
    # act_quant_fp8
    assert lib.act_quant_fp8(a16, a16, a16, 4, 100, None) == fp4.FP4_ERR_SHAPE
    assert lib.act_quant_fp8(a16, a16, a16, -1, 128, None) == fp4.FP4_ERR_ARG
    assert lib.act_quant_fp8(None, a16, a16, 4, 128, None) == fp4.FP4_ERR_ARG
    assert lib.act_quant_fp8(odd, a16, a16, 4, 128, None) == fp4.FP4_ERR_ALIGN
    assert lib.act_quant_fp8(None, None, None, 0, 128, None) == fp4.FP4_OK  # empty: no-op
    # fp4_expert_gemm
    g = lib.fp4_expert_gemm
    assert g(a16, a16, a16, 1.0, 7, a16, 1, 1, 128, None, None, None, 0, None) == fp4.FP4_ERR_ARG
    assert g(a16, a16, a16, 1.0, 0, a16, 1, 1, 96, None, None, None, 0, None) == fp4.FP4_ERR_SHAPE
    assert g(a16, a16, a16, 1.0, 0, a16, 1, 0, 128, None, None, None, 0, None) == fp4.FP4_ERR_SHAPE
    assert g(a16, None, a16, 1.0, 0, a16, 1, 4, 128, None, None, None, 0, None) == fp4.FP4_ERR_ARG
    assert g(a16, a16, a16, 1.0, 0, odd, 1, 4, 128, None, None, None, 0, None) == fp4.FP4_ERR_ALIGN
    assert g(a16, a16, a16, 1.0, 0, a16, 1, 4, 128, a16, None, None, 0, None) == fp4.FP4_ERR_ARG
    assert g(None, None, None, 1.0, 0, None, 0, 4, 128, None, None, None, 0, None) == fp4.FP4_OK
    # fp4_grouped_expert_gemm
    G = lib.fp4_grouped_expert_gemm
    assert G(a16, 8, None, a16, 0, 8, a16, a16, a16, 0, a16, 4, 128, None, 0, None) == \
        fp4.FP4_ERR_ARG                                  # zero experts
    assert G(a16, 8, None, a16, 2, 8, a16, a16, None, 0, a16, 4, 128, None, 0, None) == \
        fp4.FP4_ERR_ARG                                  # NVFP4 without scale2
    assert G(a16, 4, None, a16, 2, 8, a16, a16, a16, 0, a16, 4, 128, None, 0, None) == \
        fp4.FP4_ERR_SHAPE                                # no row ids but fewer tokens than rows
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, 1, a16, 4, 130, None, 0, None) == \
        fp4.FP4_ERR_SHAPE
    assert G(a16, 8, None, a16, 2, 8, odd, a16, a16, 1, a16, 4, 128, None, 0, None) == \
        fp4.FP4_ERR_ALIGN
    assert G(a16, 8, None, a16, 2, 0, a16, a16, a16, 1, a16, 4, 128, None, 0, None) == fp4.FP4_OK
    # fp4_grouped_quantize(x, T, row_ids, P, k, recipe, workspace, ws_bytes, stream)
    Q = lib.fp4_grouped_quantize
    big = 1 << 40
    assert Q(a16, 8, None, 8, 512, 5, a16, big, None) == fp4.FP4_ERR_ARG          # recipe
    assert Q(a16, 8, None, 8, 384, 0, a16, big, None) == fp4.FP4_ERR_SHAPE        # k % 256
    assert Q(a16, 8, None, 8, 768, 1, a16, big, None) == fp4.FP4_ERR_SHAPE        # k % 512
    assert Q(a16, 8, None, 8, 512, 0, None, 0, None) == fp4.FP4_ERR_WORKSPACE
    assert Q(a16, 8, None, 8, 512, 0, a16, 100, None) == fp4.FP4_ERR_WORKSPACE    # too small
    assert Q(None, 8, None, 8, 512, 0, a16, big, None) == fp4.FP4_ERR_ARG
    assert Q(a16, 4, None, 8, 512, 0, a16, big, None) == fp4.FP4_ERR_SHAPE        # T < P
    assert Q(odd, 8, None, 8, 512, 0, a16, big, None) == fp4.FP4_ERR_ALIGN
    assert Q(None, 0, None, 0, 512, 0, None, 0, None) == fp4.FP4_OK               # empty
    # fp4_grouped_gemm_quantized(ws, ws_bytes, T, row_ids, offsets, E, P, w, wscale, scale2,
    #                            recipe, out, n, k, stream)
    R = lib.fp4_grouped_gemm_quantized
    assert R(a16, big, 8, None, a16, 0, 8, a16, a16, a16, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_ARG
    assert R(None, 0, 8, None, a16, 2, 8, a16, a16, a16, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_WORKSPACE
    assert R(a16, big, 8, None, a16, 2, 8, a16, a16, None, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_ARG
    assert R(a16, big, 8, None, None, 2, 8, a16, a16, a16, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_ARG
    assert R(a16, big, 8, None, a16, 2, 8, odd, a16, a16, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_ALIGN
    assert R(a16, big, 8, None, a16, 2, 8, a16, a16, None, 1, a16, 256, 768, None) == \
        fp4.FP4_ERR_SHAPE
    assert R(a16, big, 8, None, a16, 2, 8, a16, a16, a16, 0, a16, 0, 512, None) == \
        fp4.FP4_ERR_SHAPE
    assert R(a16, big, 4, None, a16, 2, 8, a16, a16, a16, 0, a16, 256, 512, None) == \
        fp4.FP4_ERR_SHAPE                                # no row ids, fewer tokens than rows
    assert R(a16, big, 8, None, a16, 2, 0, a16, a16, a16, 0, a16, 256, 512, None) == fp4.FP4_OK
    # fp4_grouped_gate_up_swiglu(x, T, row_ids, offsets, E, P, w, wscale, scale2, recipe,
    #                            limit, h, inter, k, ws, ws_bytes, stream)
    G = lib.fp4_grouped_gate_up_swiglu
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, 0, 0.0, a16, 128, 512, a16, big, None) == \
        fp4.FP4_ERR_ARG                                  # limit <= 0
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, 0, 7.0, a16, 100, 512, a16, big, None) == \
        fp4.FP4_ERR_SHAPE                                # inter % 64
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, 0, 7.0, a16, 128, 512, None, 0, None) == \
        fp4.FP4_ERR_WORKSPACE
    assert G(None, 8, None, a16, 2, 8, a16, a16, a16, 0, 7.0, a16, 128, 512, a16, big, None) == \
        fp4.FP4_ERR_ARG
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, 0, 7.0, odd, 128, 512, a16, big, None) == \
        fp4.FP4_ERR_ALIGN
    assert G(a16, 8, None, a16, 2, 0, a16, a16, a16, 0, 7.0, a16, 128, 512, a16, big, None) == \
        fp4.FP4_OK                                       # no routed rows
    # fp4_route_topk(logits, T, E, topk, renorm, ids, weights, stream)
    K = lib.fp4_route_topk
    assert K(a16, 4, 0, 1, 0, a16, a16, None) == fp4.FP4_ERR_ARG
    assert K(a16, 4, 2048, 8, 0, a16, a16, None) == fp4.FP4_ERR_SHAPE          # E > 1024
    assert K(a16, 4, 8, 9, 0, a16, a16, None) == fp4.FP4_ERR_SHAPE             # topk > E
    assert K(a16, 4, 64, 33, 0, a16, a16, None) == fp4.FP4_ERR_SHAPE           # topk > 32
    assert K(None, 4, 64, 8, 0, a16, a16, None) == fp4.FP4_ERR_ARG
    assert K(odd, 4, 64, 8, 0, a16, a16, None) == fp4.FP4_ERR_ALIGN
    assert K(None, 0, 64, 8, 0, None, None, None) == fp4.FP4_OK
    # fp4_route_csr(ids, T, topk, E, offsets, row_ids, pair_rows, ws, ws_bytes, stream)
    C = lib.fp4_route_csr
    need = lib.fp4_route_csr_workspace_size(100, 16)
    assert need == 4 * (2 * 16 * 4 + 16)
    assert C(a16, 100, 2, 0, a16, a16, a16, a16, need, None) == fp4.FP4_ERR_ARG
    assert C(a16, 100, 2, 16, None, a16, a16, a16, need, None) == fp4.FP4_ERR_ARG
    assert C(a16, 100, 2, 16, a16, a16, a16, a16, need - 1, None) == fp4.FP4_ERR_WORKSPACE
    assert C(a16, 100, 2, 16, a16, a16, a16, odd, need, None) == fp4.FP4_ERR_ALIGN
    # fp4_moe_combine(out, P, pair_rows, weights, T, topk, n, y, stream)
    B = lib.fp4_moe_combine
    assert B(a16, 8, a16, a16, 4, 2, 6, a16, None) == fp4.FP4_ERR_SHAPE           # n % 4
    assert B(a16, 8, a16, a16, 4, 0, 8, a16, None) == fp4.FP4_ERR_ARG
    assert B(None, 8, a16, a16, 4, 2, 8, a16, None) == fp4.FP4_ERR_ARG
    assert B(a16, 8, a16, a16, 4, 2, 8, odd, None) == fp4.FP4_ERR_ALIGN
    assert B(None, 0, None, None, 0, 2, 8, None, None) == fp4.FP4_OK
    # fp4_gemm_mirror(codes, scales, w, wscale, scale2, recipe, out, g, n, k, stream)
    M = lib.fp4_gemm_mirror
    assert M(a16, a16, a16, a16, 1.0, 5, a16, 2, 4, 128, None) == fp4.FP4_ERR_ARG      # recipe
    assert M(a16, a16, a16, a16, 1.0, 0, a16, 2, 4, 100, None) == fp4.FP4_ERR_SHAPE    # k % 128
    assert M(a16, None, a16, a16, 1.0, 0, a16, 2, 4, 128, None) == fp4.FP4_ERR_ARG
    assert M(None, None, None, None, 1.0, 0, None, 0, 4, 128, None) == fp4.FP4_OK     # empty
    # fp4_swiglu_quant(gate, up, ld, limit, rows, inter, h_out, codes, scales, stream)
    S = lib.fp4_swiglu_quant
    assert S(a16, a16, 256, 0.0, 2, 256, None, a16, a16, None) == fp4.FP4_ERR_ARG     # limit <= 0
    assert S(a16, a16, 256, float("inf"), 2, 256, None, a16, a16, None) == fp4.FP4_ERR_ARG
    assert S(a16, a16, 256, float("nan"), 2, 256, None, a16, a16, None) == fp4.FP4_ERR_ARG
    assert S(a16, a16, 200, 7.0, 2, 200, None, a16, a16, None) == fp4.FP4_ERR_SHAPE   # inter % 128
    assert S(a16, a16, 128, 7.0, 2, 256, None, a16, a16, None) == fp4.FP4_ERR_SHAPE   # ld < inter
    assert S(a16, a16, 258, 7.0, 2, 256, None, a16, a16, None) == fp4.FP4_ERR_SHAPE   # ld % 4
    assert S(None, a16, 256, 7.0, 2, 256, None, a16, a16, None) == fp4.FP4_ERR_ARG
    assert S(a16, a16, 256, 7.0, 2, 256, None, None, a16, None) == fp4.FP4_ERR_ARG
    assert S(odd, a16, 256, 7.0, 2, 256, None, a16, a16, None) == fp4.FP4_ERR_ALIGN
    assert S(a16, a16, 256, 7.0, 2, 256, odd, a16, a16, None) == fp4.FP4_ERR_ALIGN
    assert S(None, None, 256, 7.0, 0, 256, None, None, None, None) == fp4.FP4_OK      # empty


def test_status_strings_and_error_model(lib):
    assert lib.fp4_status_string(fp4.FP4_ERR_WORKSPACE) == b"FP4_ERR_WORKSPACE"
    assert lib.fp4_status_string(123) == b"FP4_ERR_UNKNOWN"
    for recipe, gs in ((fp4.NVFP4, 16), (fp4.MXFP4, 32)):
        extra = 2 if recipe == fp4.NVFP4 else 0
        for k in (128, 1536, 4096, 7168, 28544):
            # up to k = 28544 the streaming path is the warp-MMA kernel: one f32 rounding
            # per 16-product MMA step, as on the tcgen05 path
            n_ops = fp4.fp4_error_ops(fp4.PATH_STREAM, recipe, k)
            assert n_ops == k // 16 + extra + 1
            assert n_ops == fp4.fp4_error_ops(fp4.PATH_TC, recipe, k)
        for k in (28672, 65536):
            # beyond it, the FMA streaming kernel: the order of the pages' own kernel,
            # (gs-1) + ceil(groups/128) + 7
            n_ops = fp4.fp4_error_ops(fp4.PATH_STREAM, recipe, k)
            assert gs - 1 < n_ops <= (gs - 1) + k / 256 + 8


def test_path_choice_by_shape(lib):
    # decode-sized (about one row per expert) always streams
    assert fp4.fp4_gemm_path(64, 64, 3072, 4096, fp4.NVFP4, True) == fp4.PATH_STREAM
    # the tensor-core path from 9 routed rows per expert on average, given a workspace
    assert fp4.fp4_gemm_path(8 * 64, 64, 3072, 4096, fp4.NVFP4, True) == fp4.PATH_STREAM
    assert fp4.fp4_gemm_path(9 * 64, 64, 3072, 4096, fp4.NVFP4, True) == fp4.PATH_TC
    # without a workspace there is only the streaming path
    assert fp4.fp4_gemm_path(32768, 256, 2048, 7168, fp4.NVFP4, False) == fp4.PATH_STREAM
    fp4.fp4_force_path(fp4.PATH_TC)
    try:
        assert fp4.fp4_gemm_path(64, 64, 3072, 4096, fp4.NVFP4, True) == fp4.PATH_TC
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    assert fp4.fp4_gemm_path(64, 64, 3072, 4096, fp4.NVFP4, True) == fp4.PATH_STREAM


def test_w4a4_host_side_checks(lib):
    V = ctypes.c_void_p
    a16 = V(0x10000)           # never dereferenced: every call below fails its checks first
    odd = V(0x10004)
    Q = lib.act_quant_w4a4     # (x, codes, scales, rowscale, rows, k, stream)
    assert Q(a16, a16, a16, a16, 4, 24, None) == fp4.FP4_ERR_SHAPE       # k % 16
    assert Q(a16, a16, a16, a16, -1, 32, None) == fp4.FP4_ERR_ARG
    assert Q(None, a16, a16, a16, 4, 32, None) == fp4.FP4_ERR_ARG
    assert Q(a16, a16, a16, None, 4, 32, None) == fp4.FP4_ERR_ARG
    assert Q(a16, a16, odd, a16, 4, 32, None) == fp4.FP4_ERR_ALIGN
    assert Q(None, None, None, None, 0, 32, None) == fp4.FP4_OK           # empty: no-op
    # workspace size: 1024 + R(P k/2) + R(P k/16) + R(4P) (+ the token rows when T < P)
    R = lambda b: (b + 1023) // 1024 * 1024
    k, P, T = 7168, 32768, 4096
    assert fp4.fp4_w4a4_workspace_size(T, P, k) == \
        1024 + R(P * k // 2) + R(P * k // 16) + R(4 * P) + R(T * k // 2) + R(T * k // 16) + R(4 * T)
    assert fp4.fp4_w4a4_workspace_size(P, P, k) == 1024 + R(P * k // 2) + R(P * k // 16) + R(4 * P)
    assert fp4.fp4_w4a4_workspace_size(8, 8, 128) == 0                    # k % 256
    # fp4_grouped_expert_gemm_w4a4(x, T, row_ids, offsets, E, P, w, wscale, scale2, out, n, k,
    #                              ws, ws_bytes, stream)
    G = lib.fp4_grouped_expert_gemm_w4a4
    big = 1 << 40
    assert G(a16, 8, None, a16, 0, 8, a16, a16, a16, a16, 4, 256, a16, big, None) == \
        fp4.FP4_ERR_ARG                                                  # zero experts
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, a16, 4, 384, a16, big, None) == \
        fp4.FP4_ERR_SHAPE                                                # k % 256
    assert G(a16, 8, None, a16, 1025, 8, a16, a16, a16, a16, 4, 256, a16, big, None) == \
        fp4.FP4_ERR_SHAPE                                                # > 1024 experts
    assert G(a16, 4, None, a16, 2, 8, a16, a16, a16, a16, 4, 256, a16, big, None) == \
        fp4.FP4_ERR_SHAPE                                                # T < P, no row ids
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, a16, 4, 256, None, 0, None) == \
        fp4.FP4_ERR_WORKSPACE
    assert G(a16, 8, None, a16, 2, 8, a16, a16, a16, a16, 4, 256, a16, 1024, None) == \
        fp4.FP4_ERR_WORKSPACE
    assert G(odd, 8, None, a16, 2, 8, a16, a16, a16, a16, 4, 256, a16, big, None) == \
        fp4.FP4_ERR_ALIGN
    assert G(None, 0, None, None, 2, 0, None, None, None, None, 4, 256, None, 0, None) == \
        fp4.FP4_OK                                                       # empty
    M = lib.fp4_w4a4_gemm_quantized
    assert M(a16, big, 8, None, a16, 2, 8, a16, a16, None, a16, 4, 256, None) == fp4.FP4_ERR_ARG
    assert M(a16, big, 8, None, a16, 2, 8, odd, a16, a16, a16, 4, 256, None) == \
        fp4.FP4_ERR_ALIGN
    assert fp4.fp4_w4a4_error_ops(7168) == 7168 // 16 + 3
