"""fp4_gemm_mirror against the oracle's mirror order (fn mirror_gemm of
dsv4_native_gemm_gate.rs), through the C ABI: equal bit for bit, as the page requires of
its own kernel."""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(rng, g, n, k, recipe, scale=2.0):
    x = (rng.standard_normal((g, k)) * scale).astype(np.float32)
    x[0, : min(k, 64)] *= 50.0                       # a row with an outlier block
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    gs = fp4.group_size(recipe)
    sc = (rng.integers(0x20, 0x41, (n, k // gs)) if recipe == fp4.NVFP4
          else rng.integers(118, 135, (n, k // gs))).astype(np.uint8)
    codes, scales = oracle.act_quant(x)
    return x, codes, scales, w, sc


def _gpu(codes, scales, w, sc, s2, recipe):
    t = lambda a: torch.as_tensor(a).to(DEV)
    out = fp4.fp4_gemm_mirror(t(codes), t(scales), t(w), t(sc), s2, recipe)
    return out.cpu().numpy()


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
@pytest.mark.parametrize("g,n,k", [(4, 256, 512), (3, 136, 128), (2, 64, 8192), (16, 512, 2048)])
def test_mirror_bit_exact(recipe, g, n, k):
    fp4.build.build()
    rng = np.random.default_rng(7 + recipe + k)
    for s2 in ([1.0 / 64, 5.9945243e-5] if recipe == fp4.NVFP4 else [0.0]):
        _, codes, scales, w, sc = _inputs(rng, g, n, k, recipe)
        got = _gpu(codes, scales, w, sc, s2, recipe)
        want = oracle.mirror_gemm(codes, scales, w, sc, s2, recipe)
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, "recipe %d %s: %d outputs differ, first %d: %r vs %r" % (
            recipe, (g, n, k), bad.size, bad[0], got.reshape(-1)[bad[0]], want.reshape(-1)[bad[0]])


def test_mirror_after_gpu_act_quant():
    """The page's chain: act_quant on the GPU (bit-exact), then the mirror GEMM."""
    rng = np.random.default_rng(99)
    g, n, k = 5, 192, 1024
    x, codes, scales, w, sc = _inputs(rng, g, n, k, fp4.NVFP4)
    gcodes, gscales = fp4.act_quant_fp8(torch.as_tensor(x).to(DEV))
    assert np.array_equal(gcodes.cpu().numpy(), codes)
    out = fp4.fp4_gemm_mirror(gcodes, gscales, torch.as_tensor(w).to(DEV),
                              torch.as_tensor(sc).to(DEV), 1.0 / 64, fp4.NVFP4)
    want = oracle.mirror_gemm(codes, scales, w, sc, 1.0 / 64, fp4.NVFP4)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_mirror_tree_order_example_on_gpu():
    """The oracle pin's worked example: only the halving-tree order gives 32 + 2^-18."""
    k, gs = 2048, 16
    codes = np.zeros((1, k), np.uint8)
    scales = np.ones((1, k // 128), np.float32)
    w = np.zeros((1, k // 2), np.uint8)
    sc = np.full((1, k // gs), 0x38, np.uint8)
    codes[0, 0], w[0, 0], sc[0, 0] = 0x40, 0x06, 0x48
    for grp in (1, 65):
        codes[0, grp * gs], w[0, grp * gs // 2], sc[0, grp] = 0x01, 0x01, 0x01
    got = _gpu(codes, scales, w, sc, 1.0, fp4.NVFP4)[0, 0]
    assert got == np.float32(32.0 + 2.0 ** -18)
