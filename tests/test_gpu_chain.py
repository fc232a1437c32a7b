"""The page's swiglu_limit saturation cell as a chain, through the C ABI: a row scaled x50
goes through act_quant -> gate GEMM (w1) and up GEMM (w3) -> SwiGLU with the swiglu_limit
clamps -> e4m3 requantisation -> down GEMM (w2), on both recipes and both GEMM paths
(dsv4_native_gemm_gate.rs, swiglu_limit saturation cell).

Each leg is checked against the oracle on the inputs the GPU leg actually received, as the
page does (its GEMM legs are compared with the CPU on the same codes): the gate/up GEMMs
against the f64 reference of act_quant(x), within the stated bound; h against the oracle's
SwiGLU of the GPU's own gate/up outputs, within 2e-6 max|h|; the requantised codes and
scales against act_quant of the GPU's h, bit for bit; the down GEMM against the f64
reference of those codes, within the bound. Both clamps must engage (gate above +L, |up|
above L), and gate values below -L must pass unclamped.
"""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import check_gemm, gemm_bound, grouped_sampled_check, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
H_TOL = 2e-6


def _expert(recipe, n, k, seed):
    b = synth.make_bank(recipe, 1, n, k, seed, "cpu", scale2_value=5.9945243e-5 * 64)
    return b.w[0].numpy(), b.sc[0].numpy(), float(b.scale2[0])


def _gemm(x_dev, w, sc, s2, recipe, path):
    """One expert through fp4_expert_gemm on `path`; returns (out, codes, scales) with
    the codes the call quantised."""
    g, k = x_dev.shape
    n = w.shape[0]
    codes = torch.empty(g, k, dtype=torch.uint8, device=DEV)
    scales = torch.empty(g, k // 128, dtype=torch.float32, device=DEV)
    ws = fp4.workspace_for(g, g, n, k, recipe) if path == fp4.PATH_TC else None
    fp4.fp4_force_path(path)
    try:
        out = fp4.fp4_expert_gemm(x_dev, torch.as_tensor(w).to(DEV), torch.as_tensor(sc).to(DEV),
                                  s2, recipe, codes_out=codes, scales_out=scales, workspace=ws)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    return out, codes, scales


@pytest.mark.parametrize("path", [fp4.PATH_STREAM, fp4.PATH_TC])
@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_saturation_cell_chain(recipe, path):
    fp4.build.build()
    hidden, inter, limit = 2048, 1024, 7.0
    gen = torch.Generator().manual_seed(31 + recipe)
    x = torch.randn(4, hidden, generator=gen)
    x[0] *= 50.0                                   # the page's x50 row
    w1, s1, q1 = _expert(recipe, inter, hidden, 41)
    w3, s3, q3 = _expert(recipe, inter, hidden, 43)
    w2, s2, q2 = _expert(recipe, hidden, inter, 42)
    xd = x.to(DEV)

    # gate and up legs: codes bit-exact with the oracle's act_quant, outputs within bound
    g1, c1, sc1 = _gemm(xd, w1, s1, q1, recipe, path)
    g3, c3, sc3 = _gemm(xd, w3, s3, q3, recipe, path)
    xc, xs = oracle.act_quant(x.numpy())
    for c, sc in ((c1, sc1), (c3, sc3)):
        assert np.array_equal(to_np(c), xc)
        assert np.array_equal(to_np(sc).view(np.uint32), xs.view(np.uint32))
    n_up = gemm_bound(path, recipe, hidden)
    for out, w, sc, q, tag in ((g1, w1, s1, q1, "w1"), (g3, w3, s3, q3, "w3")):
        ref, absp = oracle.gemm_ref(xc, xs, w, sc, q, recipe)
        check_gemm(to_np(out), ref, absp, n_up, "chain %s recipe %d path %d" % (tag, recipe, path))

    # the clamps engage on the x50 row (gate from above, up on both sides)
    g_np, u_np = to_np(g1), to_np(g3)
    assert (g_np[0] > limit).sum() > 0 and (np.abs(u_np[0]) > limit).sum() > 0
    assert (g_np[0] < -limit).sum() > 0

    # SwiGLU + requantisation of the GPU's gate/up outputs
    hc, hs, h = fp4.fp4_swiglu_quant(g1, g3, limit, want_h=True)
    h_ref = oracle.swiglu(g_np, u_np, limit)
    h_np = to_np(h).astype(np.float64)
    assert np.max(np.abs(h_np - h_ref)) <= H_TOL * np.max(np.abs(h_ref))
    want_c, want_s = oracle.act_quant(to_np(h))
    assert np.array_equal(to_np(hc), want_c)
    assert np.array_equal(to_np(hs).view(np.uint32), want_s.view(np.uint32))

    # down leg on h: the codes it quantises equal the requantised codes, output within bound
    d, dc, ds = _gemm(h, w2, s2, q2, recipe, path)
    assert torch.equal(dc, hc) and torch.equal(ds, hs)
    ref, absp = oracle.gemm_ref(want_c, want_s, w2, s2, q2, recipe)
    worst, rel = check_gemm(to_np(d), ref, absp, gemm_bound(path, recipe, inter),
                            "chain w2 recipe %d path %d" % (recipe, path))
    assert fp4.fp4_get_device_error() == 0
    print("chain recipe %d path %d: gate sat %d, up sat %d, w2 worst err/bound %.3g" % (
        recipe, path, int((g_np[0] > limit).sum()), int((np.abs(u_np[0]) > limit).sum()), worst))


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_saturation_cell_chain_fused_epilogue(recipe):
    """The same cell over routed rows of several experts, with SwiGLU in the gate/up
    epilogue (fp4_grouped_gate_up_swiglu): its h must equal, bit for bit, fp4_swiglu_quant's
    h of the unfused gate/up output; the gate/up output, h and the down projection of h
    (whose quantise pass is the requantisation) are checked against the oracle."""
    fp4.build.build()
    E, T, topk, hidden, inter, limit = 3, 96, 2, 2048, 1024, 7.0
    gen = torch.Generator().manual_seed(57 + recipe)
    x = torch.randn(T, hidden, generator=gen)
    x[::7] *= 50.0                                              # saturation rows
    choices = torch.stack([torch.randperm(E, generator=gen)[:topk] for _ in range(T)])
    r = synth.routing_from_choices(choices, E)
    gu_bank = synth.make_bank(recipe, E, 2 * inter, hidden, 61 + recipe, "cpu",
                              scale2_value=5.9945243e-5 * 64)
    dn_bank = synth.make_bank(recipe, E, hidden, inter, 67 + recipe, "cpu",
                              scale2_value=5.9945243e-5 * 64)
    routing = synth.Routing(r.offsets.to(DEV), r.row_ids.to(DEV))
    gu = synth.Bank(recipe, gu_bank.w.to(DEV), gu_bank.sc.to(DEV), gu_bank.scale2.to(DEV))
    dn = synth.Bank(recipe, dn_bank.w.to(DEV), dn_bank.sc.to(DEV), dn_bank.scale2.to(DEV))
    xd = x.to(DEV)
    P = r.P

    # unfused: the gate/up projection on the tensor cores, then fp4_swiglu_quant
    ws = fp4.workspace_for(T, P, 2 * inter, hidden, recipe)
    fp4.fp4_force_path(fp4.PATH_TC)
    try:
        gu_out = fp4.fp4_grouped_expert_gemm(xd, routing.row_ids, routing.offsets, gu.w, gu.sc,
                                             gu.scale2, recipe, workspace=ws)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    _, _, h_unf = fp4.fp4_swiglu_quant(gu_out[:, :inter], gu_out[:, inter:], limit, want_h=True)

    # fused
    h = fp4.fp4_grouped_gate_up_swiglu(xd, routing.row_ids, routing.offsets, gu.w, gu.sc,
                                       gu.scale2, recipe, limit, ws)
    assert torch.equal(h, h_unf), float((h - h_unf).abs().max())

    # the gate/up leg against the oracle, the clamps engaged, h against the oracle's SwiGLU
    proj_gu = synth.Projection("gu", xd, routing, gu)
    grouped_sampled_check(proj_gu, gu_out, fp4.PATH_TC, np.arange(P), "fused chain gate/up")
    g_np, u_np = to_np(gu_out[:, :inter]), to_np(gu_out[:, inter:])
    assert (g_np > limit).sum() > 0 and (np.abs(u_np) > limit).sum() > 0
    assert (g_np < -limit).sum() > 0
    h_ref = oracle.swiglu(g_np, u_np, limit)
    assert np.max(np.abs(to_np(h).astype(np.float64) - h_ref)) <= H_TOL * np.max(np.abs(h_ref))

    # the down projection takes h as its routed rows (no row ids): its quantise pass is the
    # requantisation; checked against the oracle's act_quant + f64 reference of h
    ws_dn = fp4.workspace_for(P, P, hidden, inter, recipe)
    fp4.fp4_force_path(fp4.PATH_TC)
    try:
        d = fp4.fp4_grouped_expert_gemm(h, None, routing.offsets, dn.w, dn.sc, dn.scale2, recipe,
                                        workspace=ws_dn)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    proj_dn = synth.Projection("dn", h, synth.Routing(routing.offsets, routing.row_ids), dn,
                               row_ids_used=False)
    worst, rel = grouped_sampled_check(proj_dn, d, fp4.PATH_TC, np.arange(P), "fused chain down")
    assert fp4.fp4_get_device_error() == 0
    print("fused chain recipe %d: h bit-equal to the unfused chain; down worst err/bound %.3g" % (
        recipe, worst))
