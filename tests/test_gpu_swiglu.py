"""Parity of fp4_swiglu_quant (SwiGLU with the swiglu_limit clamps + e4m3 requantisation,
the step after the gate/up projection) with the CPU oracle, through the C ABI.

The page (dsv4_native_gemm_gate.rs, swiglu_limit saturation cell) accepts the GPU's h
within 2e-6 * max|h| of the CPU's (the exp ulp class); the requantised codes and scales
must be act_quant of the GPU's own h, bit for bit. Rows scaled x50 drive both clamps, as
the page's saturation cell does.
"""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4

pytestmark = pytest.mark.gpu
DEV = "cuda"
H_TOL = 2e-6


def _gate_up(rows, inter, seed, sat_every=4, scale=3.0):
    """Fused gate/up output [rows, 2*inter] (gate first): N(0, scale) with every
    sat_every-th row scaled x50 (the page's saturation rows)."""
    gen = torch.Generator().manual_seed(seed)
    gu = torch.randn(rows, 2 * inter, generator=gen) * scale
    if sat_every:
        gu[::sat_every] *= 50.0
    return gu


def _check(gate, up, limit, codes, scales, h, what):
    g_np = gate.cpu().numpy()
    u_np = up.cpu().numpy()
    ref = oracle.swiglu(g_np, u_np, limit)
    h_np = h.cpu().numpy().astype(np.float64)
    err = np.max(np.abs(h_np - ref))
    assert err <= H_TOL * np.max(np.abs(ref)), "%s: h max err %.3g vs %.3g" % (
        what, err, H_TOL * np.max(np.abs(ref)))
    want_c, want_s = oracle.act_quant(h.cpu().numpy())
    got_c = codes.cpu().numpy()
    got_s = scales.cpu().numpy()
    bad = np.flatnonzero(got_c.reshape(-1) != want_c.reshape(-1))
    assert bad.size == 0, "%s: %d codes differ, first %d: %d vs %d" % (
        what, bad.size, bad[0], got_c.reshape(-1)[bad[0]], want_c.reshape(-1)[bad[0]])
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), what
    return err / np.max(np.abs(ref))


@pytest.mark.parametrize("limit", [7.0, 10.0])
def test_swiglu_fused_bank_layout(limit):
    fp4.build.build()
    rows, inter = 37, 512
    gu = _gate_up(rows, inter, 1).to(DEV)
    gate, up = gu[:, :inter], gu[:, inter:]
    codes, scales, h = fp4.fp4_swiglu_quant(gate, up, limit, want_h=True)
    rel = _check(gate, up, limit, codes, scales, h, "fused L=%g" % limit)
    # the test input drives both clamps
    g_np, u_np = gate.cpu().numpy(), up.cpu().numpy()
    assert (g_np > limit).sum() > 0 and (np.abs(u_np) > limit).sum() > 0
    assert (g_np < -limit).sum() > 0  # gate values below -L pass unclamped
    print("swiglu fused L=%g: h rel err %.3g" % (limit, rel))


def test_swiglu_separate_tensors_and_without_h():
    rows, inter = 64, 1024
    gu = _gate_up(rows, inter, 2, sat_every=3).to(DEV)
    gate = gu[:, :inter].contiguous()
    up = gu[:, inter:].contiguous()
    codes, scales, h = fp4.fp4_swiglu_quant(gate, up, 7.0, want_h=True)
    _check(gate, up, 7.0, codes, scales, h, "separate")
    codes2, scales2, h2 = fp4.fp4_swiglu_quant(gate, up, 7.0)
    assert h2 is None
    assert torch.equal(codes2, codes) and torch.equal(scales2, scales)
    # the fused layout gives the same result
    codes3, scales3, _ = fp4.fp4_swiglu_quant(gu[:, :inter], gu[:, inter:], 7.0)
    assert torch.equal(codes3, codes) and torch.equal(scales3, scales)


def test_swiglu_edge_rows():
    # one row, one group; a zero row (scale floor); a row of huge negative gates (h ~ 0)
    inter = 128
    gate = torch.zeros(3, inter)
    up = torch.randn(3, inter)
    gate[0] = torch.linspace(-5, 5, inter)
    gate[2] = -1.0e4
    gate, up = gate.to(DEV), up.to(DEV)
    codes, scales, h = fp4.fp4_swiglu_quant(gate, up, 7.0, want_h=True)
    _check(gate, up, 7.0, codes, scales, h, "edge")
    assert torch.all(h[1] == 0) and torch.all(h[2].abs() < 1e-30)
    assert fp4.fp4_swiglu_quant(gate[:0], up[:0], 7.0)[0].numel() == 0


def test_swiglu_prefill_shape_sampled():
    """The prefill gate/up output shape (32,768 routed rows, inter 1024), rows sampled."""
    rows, inter = 32768, 1024
    gu = _gate_up(rows, inter, 3, sat_every=97).to(DEV)
    codes, scales, h = fp4.fp4_swiglu_quant(gu[:, :inter], gu[:, inter:], 7.0, want_h=True)
    rng = np.random.default_rng(3)
    sel = np.unique(np.concatenate([[0, rows - 1, 97, 194], rng.integers(0, rows, 60)]))
    idx = torch.as_tensor(sel, device=DEV)
    g = gu[idx, :inter]
    u = gu[idx, inter:]
    _check(g, u, 7.0, codes[idx], scales[idx], h[idx], "prefill sampled")


@pytest.mark.parametrize("recipe", [0, 1])
@pytest.mark.parametrize("inter", [64, 192])
def test_fused_gate_up_swiglu_ragged(recipe, inter):
    """fp4_grouped_gate_up_swiglu with inter a multiple of 64 but not of 128 (one and three
    64-column tiles), ragged and empty experts: h against the oracle's SwiGLU of the same
    call's unfused gate/up output (computed on the tensor cores too), within 2e-6 max|h|."""
    from block_scaled_fp4_act_gb300 import synth
    fp4.build.build()
    gen = torch.Generator().manual_seed(90 + inter + recipe)
    sizes = [0, 37, 200, 1, 0, 65]
    E, T, k, limit = len(sizes), 96, 512, 6.0
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(torch.tensor(sizes), 0).to(torch.int32)
    P = int(offsets[-1])
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    bank = synth.make_bank(recipe, E, 2 * inter, k, 91 + recipe, "cpu")
    x = torch.randn(T, k, generator=gen) * 3
    x[::5] *= 50.0
    xd, rid, off = x.to(DEV), row_ids.to(DEV), offsets.to(DEV)
    w, sc, s2 = bank.w.to(DEV), bank.sc.to(DEV), bank.scale2.to(DEV)
    ws = fp4.workspace_for(T, P, 2 * inter, k, recipe)
    fp4.fp4_force_path(fp4.PATH_TC)
    try:
        gu = fp4.fp4_grouped_expert_gemm(xd, rid, off, w, sc, s2, recipe, workspace=ws)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    h = fp4.fp4_grouped_gate_up_swiglu(xd, rid, off, w, sc, s2, recipe, limit, ws)
    g_np, u_np = gu[:, :inter].cpu().numpy(), gu[:, inter:].cpu().numpy()
    assert (g_np > limit).any() and (np.abs(u_np) > limit).any()
    ref = oracle.swiglu(g_np, u_np, limit)
    err = np.max(np.abs(h.cpu().numpy().astype(np.float64) - ref))
    assert err <= H_TOL * np.max(np.abs(ref)), err
    assert fp4.fp4_get_device_error() == 0
