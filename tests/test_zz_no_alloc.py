"""The allocation-free grouped entry point, through the C ABI.

fp4_grouped_expert_gemm_noalloc serves callers that may not allocate device memory: it
runs the tensor-core path with the library's fixed scratch array instead of a caller
workspace. Its output must match the existing entry point (given a workspace, on the same
path) within the error model the other tests use, on two different calls in a row (the
second smaller, so stale scratch contents from the first are present during it).
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import gemm_bound, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problem(recipe, E, T, topk, n, k, seed):
    gen = torch.Generator().manual_seed(seed)
    scores = torch.rand(T, E, generator=gen)
    choices = torch.argsort(scores, dim=1)[:, :topk]
    r = synth.routing_from_choices(choices, E)
    bank = synth.make_bank(recipe, E, n, k, seed + 1, "cpu", scale2_value=5.9945243e-5)
    x = torch.randn(T, k, generator=gen) * 2
    return x, r, bank


def _raw_noalloc(x, r, bank, out):
    """Call the entry point with plain pointers (the C ABI, no binding helper)."""
    L = fp4.lib()
    V = ctypes.c_void_p
    T, k = x.shape
    return L.fp4_grouped_expert_gemm_noalloc(
        V(x.data_ptr()), T, V(r.row_ids.data_ptr()), V(r.offsets.data_ptr()), bank.w.shape[0],
        r.row_ids.numel(), V(bank.w.data_ptr()), V(bank.sc.data_ptr()),
        V(bank.scale2.data_ptr()) if bank.recipe == fp4.NVFP4 else None, bank.recipe,
        V(out.data_ptr()), bank.w.shape[1], k, V(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    fp4.build.build()
    cases = [(fp4.NVFP4, 8, 300, 2, 384, 1024, 11), (fp4.MXFP4, 4, 64, 2, 256, 512, 12)]
    for recipe, E, T, topk, n, k, seed in cases:
        x, r, bank = _problem(recipe, E, T, topk, n, k, seed)
        xd, rid, off = x.to(DEV), r.row_ids.to(DEV), r.offsets.to(DEV)
        w, sc, s2 = bank.w.to(DEV), bank.sc.to(DEV), bank.scale2.to(DEV)
        P = r.P
        # the existing entry point with a caller workspace, on the same (tensor-core) path
        fp4.fp4_force_path(fp4.PATH_TC)
        try:
            ws = fp4.workspace_for(T, P, n, k, recipe)
            ref = fp4.fp4_grouped_expert_gemm(xd, rid, off, w, sc, s2, recipe, workspace=ws)
        finally:
            fp4.fp4_force_path(fp4.PATH_AUTO)
        out = torch.full((P, n), float("nan"), device=DEV)
        dev_bank = synth.Bank(recipe, w, sc, s2)
        st = _raw_noalloc(xd, synth.Routing(off, rid), dev_bank, out)
        assert st == fp4.FP4_OK, fp4.lib().fp4_last_error()
        assert fp4.fp4_get_device_error() == 0
        a, b = to_np(out), to_np(ref)
        # tolerance of the parity tests: the stated error model around the f64 reference
        sp = np.repeat(np.arange(P), n)
        scol = np.tile(np.arange(n), P)
        _, absp = oracle.grouped_ref_sampled(x.numpy(), r.row_ids.numpy(), r.offsets.numpy(),
                                             bank.w.numpy(), bank.sc.numpy(),
                                             bank.scale2.numpy(), recipe, sp, scol)
        n_ops = gemm_bound(fp4.PATH_TC, recipe, k)
        ok, worst, i = oracle.within_bound(a.reshape(-1), b.reshape(-1), absp, 2 * n_ops)
        assert ok, (worst, i)
        assert oracle.max_rel(a, b) <= 1e-3
        assert np.array_equal(a, b)  # same kernels, same order: identical bits


def test_noalloc_rejects_calls_beyond_its_scratch():
    fp4.build.build()
    L = fp4.lib()
    V = ctypes.c_void_p
    a16 = V(0x10000)  # never dereferenced: the size check fails first
    st = L.fp4_grouped_expert_gemm_noalloc(a16, 8192, a16, a16, 8, 8192, a16, a16, a16,
                                           fp4.NVFP4, a16, 2048, 7168, None)
    assert st == fp4.FP4_ERR_WORKSPACE
    assert b"scratch" in L.fp4_last_error()
