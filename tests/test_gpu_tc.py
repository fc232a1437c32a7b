"""Parity of the tensor-core (tcgen05) path with the CPU oracle, through the C ABI.

Small forced-path cases cover ragged weight-row blocks (n not a multiple of 128), ragged
routed-row blocks (expert sizes around the 256-row block and the 16-row MMA step), empty
experts and both recipes; the lossless special case must be bit-equal to a float64
matmul.
"""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import (check_gemm, expert_reference, gemm_bound, grouped_sampled_check,
                         run_projection, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def force_tc():
    fp4.build.build()
    fp4.fp4_force_path(fp4.PATH_TC)
    yield
    fp4.fp4_force_path(fp4.PATH_AUTO)


def _projection(recipe, sizes, n, k, T=None, seed=0, scale2=5.9945243e-5):
    """Grouped projection whose expert e has exactly sizes[e] routed rows (row ids drawn
    at random from T tokens)."""
    gen = torch.Generator().manual_seed(seed)
    E = len(sizes)
    P = int(sum(sizes))
    T = T or max(P, 1)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(torch.tensor(sizes, dtype=torch.int64), 0).to(torch.int32)
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    bank = synth.make_bank(recipe, E, n, k, 900 + seed, "cpu", scale2_value=scale2)
    x = torch.randn(T, k, generator=gen) * 3
    return synth.Projection("tc", x.to(DEV), synth.Routing(offsets.to(DEV), row_ids.to(DEV)),
                            synth.Bank(recipe, bank.w.to(DEV), bank.sc.to(DEV),
                                       bank.scale2.to(DEV)))


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_small_grouped_all_outputs(recipe):
    proj = _projection(recipe, [5, 0, 16, 1, 33, 0, 17], n=136, k=512, T=40, seed=1)
    out, path = run_projection(proj)
    assert path == fp4.PATH_TC
    worst, rel = grouped_sampled_check(proj, out, path, np.arange(proj.routing.P), "tc small")
    assert fp4.fp4_get_device_error() == 0
    print("tc small recipe %d: worst err/bound %.3g max_rel %.3g" % (recipe, worst, rel))


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_multi_block_experts(recipe):
    """Experts spanning several 256-row blocks with ragged tails, several weight blocks."""
    proj = _projection(recipe, [257, 0, 512, 300, 15, 256], n=384, k=1024, T=600, seed=2)
    out, path = run_projection(proj)
    assert path == fp4.PATH_TC
    worst, rel = grouped_sampled_check(proj, out, path, np.arange(proj.routing.P), "tc multi")
    assert fp4.fp4_get_device_error() == 0
    print("tc multi recipe %d: worst err/bound %.3g max_rel %.3g" % (recipe, worst, rel))


@pytest.mark.parametrize("n", [130, 132, 36])
def test_tc_output_row_stride_forms(n):
    """Whole 32-row chunks leave the epilogue through tensor stores when an output row is a
    multiple of 16 bytes (n = 132: the last weight block's box is cut at column 132; n = 36:
    one partly valid warp) and through per-value stores otherwise (n = 130); ragged chunks
    always take per-value stores."""
    proj = _projection(fp4.NVFP4, [64, 33, 0, 200, 7], n=n, k=512, T=300, seed=3)
    out, path = run_projection(proj)
    assert path == fp4.PATH_TC
    worst, rel = grouped_sampled_check(proj, out, path, np.arange(proj.routing.P), "tc n=%d" % n)
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_exact_special_case(recipe, golden_dir):
    """Lossless inputs: every partial sum is exact in f32, so the tensor-core result must
    equal the float64 matmul bit for bit."""
    from test_oracle_pins import _dense_weights, _exact_inputs, golden_e2m1
    rng = np.random.default_rng(5 + recipe)
    table = golden_e2m1(golden_dir)
    for g, n, k in [(40, 128, 512), (300, 200, 2048)]:
        x, w, sc = _exact_inputs(rng, g, n, k, recipe)
        ws = fp4.workspace_for(g, g, n, k, recipe)
        out = fp4.fp4_expert_gemm(torch.as_tensor(x).to(DEV), torch.as_tensor(w).to(DEV),
                                  torch.as_tensor(sc).to(DEV), 1.0, recipe, workspace=ws)
        want = x.astype(np.float64) @ _dense_weights(w, table).T
        got = to_np(out).astype(np.float64)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, "first mismatch %d: got %r want %r" % (bad[0], got.reshape(-1)[bad[0]],
                                                                    want.reshape(-1)[bad[0]])


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_single_expert_with_workspace(recipe):
    rng = np.random.default_rng(9 + recipe)
    g, n, k = 100, 320, 2048
    x = (rng.standard_normal((g, k)) * 2).astype(np.float32)
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    gs = fp4.group_size(recipe)
    sc = (rng.integers(0x20, 0x41, (n, k // gs)) if recipe == fp4.NVFP4
          else rng.integers(118, 135, (n, k // gs))).astype(np.uint8)
    s2 = 1.0 / 64 if recipe == fp4.NVFP4 else 0.0
    ws = fp4.workspace_for(g, g, n, k, recipe)
    out = fp4.fp4_expert_gemm(torch.as_tensor(x).to(DEV), torch.as_tensor(w).to(DEV),
                              torch.as_tensor(sc).to(DEV), s2, recipe, workspace=ws)
    _, _, ref, absp = expert_reference(x, w, sc, s2, recipe)
    worst, rel = check_gemm(to_np(out), ref, absp, gemm_bound(fp4.PATH_TC, recipe, k), "tc one")
    print("tc single recipe %d: worst err/bound %.3g max_rel %.3g" % (recipe, worst, rel))


def test_tc_matches_stream_path_closely():
    """Both paths on the same inputs agree within the sum of their bounds."""
    proj = _projection(fp4.NVFP4, [70, 3, 190], n=256, k=1024, T=100, seed=4)
    out_tc, _ = run_projection(proj)
    fp4.fp4_force_path(fp4.PATH_STREAM)
    out_st, _ = run_projection(proj)
    fp4.fp4_force_path(fp4.PATH_TC)
    d = (out_tc - out_st).abs().max().item()
    assert d <= 1e-3 * out_st.abs().max().item()


def _scaled_rows_projection(recipe, gaps, n=256, k=1024, seed=7):
    """One expert; routed row r has its 128-blocks scaled by 2^-u, u uniform in [0, gaps[r]]
    (block scale spread of about 2^gaps[r] within the row)."""
    rng = np.random.default_rng(seed)
    rows = len(gaps)
    x = rng.standard_normal((rows, k))
    for r, gmax in enumerate(gaps):
        u = rng.uniform(0, gmax, k // 128)
        u[0], u[-1] = 0.0, gmax
        x[r] *= np.repeat(np.exp2(-u), 128)
    x = x.astype(np.float32)
    return _projection_from(recipe, x, n, k, seed)


def _projection_from(recipe, x, n, k, seed):
    rows = x.shape[0]
    offsets = torch.tensor([0, rows], dtype=torch.int32)
    row_ids = torch.arange(rows, dtype=torch.int32)
    bank = synth.make_bank(recipe, 1, n, k, 910 + seed, "cpu", scale2_value=5.9945243e-5)
    return synth.Projection("scaled", torch.as_tensor(x).to(DEV),
                            synth.Routing(offsets.to(DEV), row_ids.to(DEV)),
                            synth.Bank(recipe, bank.w.to(DEV), bank.sc.to(DEV),
                                       bank.scale2.to(DEV)))


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_rows_with_wide_block_scale_spread(recipe):
    """Block scales spread up to about 2^12 within a row keep the NVFP4 f16 activation route
    (small codes become f16 subnormals); a row spread over 2^30 sends the whole call to the
    bf16 route. Both must stay within the bound."""
    for gaps, tag in [([0, 6, 10, 12] * 10, "f16"), ([0, 6, 30, 3] * 10, "bf16")]:
        proj = _scaled_rows_projection(recipe, gaps)
        out, path = run_projection(proj)
        assert path == fp4.PATH_TC
        worst, rel = grouped_sampled_check(proj, out, path, np.arange(proj.routing.P),
                                           "spread %s" % tag)
        assert fp4.fp4_get_device_error() == 0
        print("spread %s recipe %d: worst err/bound %.3g max_rel %.3g" % (tag, recipe, worst, rel))


def test_tc_full_size_prefill_repeatable_and_matches_stream():
    """Every output of both prefill projections (256 NVFP4 experts, 4096 tokens top-8,
    Zipf routing), several runs. The tensor-core path computes each output in one fixed
    MMA sequence, so runs must agree bit for bit: a pipeline race (a ring slot reused
    before its reader finished) shows up as run-to-run changes in a few weight rows of a
    tile. Each run must also agree with the streaming path to 1e-3 of the output's
    magnitude (floored at 1e-2 of the projection's largest output); the race gave errors
    of 10-30%."""
    wl = synth.workload("c4", device=DEV)
    for proj in wl.projections:
        fp4.fp4_force_path(fp4.PATH_STREAM)
        ref, _ = run_projection(proj)
        fp4.fp4_force_path(fp4.PATH_TC)
        floor = 1e-2 * ref.abs().max()
        first = None
        for rep in range(4):
            out, path = run_projection(proj)
            assert path == fp4.PATH_TC
            assert fp4.fp4_get_device_error() == 0
            bad = (out - ref).abs() > 1e-3 * (ref.abs() + floor)
            nbad = int(bad.sum().item())
            assert nbad == 0, "%s run %d: %d outputs off the streaming path, first at %s" % (
                proj.name, rep, nbad, tuple(bad.nonzero()[0].tolist()))
            if first is None:
                first = out
            else:
                diff = int((out != first).sum().item())
                assert diff == 0, "%s run %d: %d outputs differ from run 0" % (proj.name, rep, diff)
            del out
        del ref, first


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_two_phase_calls_match_one_call_and_share_the_quantised_input(recipe):
    """fp4_grouped_quantize + fp4_grouped_gemm_quantized are the launches of one grouped
    call on this path: same bits. One quantised input then serves a second bank (the gate
    and up projections of one x), checked against the oracle on every output."""
    proj = _projection(recipe, [40, 0, 100, 9, 1], n=256, k=1024, T=120, seed=3)
    one, _ = run_projection(proj)
    bank, r = proj.bank, proj.routing
    T, k = proj.x.shape
    ws = fp4.workspace_for(T, r.P, bank.n, k, recipe)
    fp4.fp4_grouped_quantize(proj.x, r.row_ids, r.P, recipe, ws)
    two = torch.empty_like(one)
    fp4.fp4_grouped_gemm_quantized(ws, T, r.row_ids, r.offsets, bank.w, bank.sc, bank.scale2,
                                   recipe, two)
    assert torch.equal(one, two)
    other = synth.make_bank(recipe, bank.E, bank.n, k, 977, DEV, scale2_value=1.0 / 64.0)
    three = torch.empty_like(one)
    fp4.fp4_grouped_gemm_quantized(ws, T, r.row_ids, r.offsets, other.w, other.sc, other.scale2,
                                   recipe, three)
    proj2 = synth.Projection("second bank", proj.x, r, other)
    grouped_sampled_check(proj2, three, fp4.PATH_TC, np.arange(r.P), "second bank")
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_tc_quantise_pass_long_rows(recipe):
    """k past what the quantise pass holds in registers (8 warps x 8 groups of 128): the
    row is read twice. NVFP4 rows within the f16 route, then one row that forces the bf16
    pass."""
    for gaps, tag in [([0, 5, 9, 3, 12], "f16"), ([0, 5, 25, 3, 12], "bf16")]:
        rng = np.random.default_rng(17)
        k = 9216
        x = rng.standard_normal((len(gaps), k))
        for r, gmax in enumerate(gaps):
            u = rng.uniform(0, gmax, k // 128)
            u[0], u[-1] = 0.0, gmax
            x[r] *= np.repeat(np.exp2(-u), 128)
        proj = _projection_from(recipe, x.astype(np.float32), 200, k, 21)
        out, path = run_projection(proj)
        assert path == fp4.PATH_TC
        grouped_sampled_check(proj, out, path, np.arange(proj.routing.P), "long rows " + tag)
        assert fp4.fp4_get_device_error() == 0
