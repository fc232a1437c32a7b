"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on one GPU.

act_quant codes and scales must be bit-exact; GEMM outputs must satisfy
|gpu - f64 reference| <= n_ops 2^-24 sum|p| per output with the n_ops the library states
for the path that ran, and max_rel <= 1e-3 (the error model and `rel` convention of the
pages: dsv4_native_gemm_gate.rs, kernel_check.rs).
"""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import (check_gemm, expert_reference, gemm_bound, grouped_sampled_check,
                         run_projection, sample_rows, to_np)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    fp4.build.build()
    fp4.lib()
    torch.cuda.init()
    fp4.fp4_force_path(fp4.PATH_AUTO)
    yield
    fp4.fp4_force_path(fp4.PATH_AUTO)


def _gpu(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(device=DEV, dtype=dtype)


# ------------------------------------------------------------------ act_quant

@pytest.mark.parametrize("case", ["normal", "student_t", "outliers", "bf16", "tiny", "zeros"])
def test_act_quant_bit_exact(case):
    g = torch.Generator().manual_seed(hash(case) % 1000)
    rows, k = 37, 1536
    x = torch.randn(rows, k, generator=g)
    if case == "student_t":
        x = synth.student_t((rows, k), 3, g, "cpu")
    elif case == "outliers":
        x = synth.with_outliers(x, g, p=0.01)
    elif case == "bf16":
        x = synth.bf16_rounded(x)
    elif case == "tiny":
        x = x * 1e-6
        x[0, :5] = torch.tensor([1e-40, -1e-42, 0.0, -0.0, 3e-39])
    elif case == "zeros":
        x[:5] = 0.0
        x[5, :128] = -0.0
    codes, scales = fp4.act_quant_fp8(x.to(DEV))
    c_ref, s_ref = oracle.act_quant(x.numpy())
    assert np.array_equal(to_np(scales).view(np.uint32), s_ref.view(np.uint32))
    diff = np.flatnonzero(to_np(codes) != c_ref)
    assert diff.size == 0, "first code mismatch at %d: x=%r gpu=%#x cpu=%#x" % (
        diff[0], x.numpy().reshape(-1)[diff[0]], to_np(codes).reshape(-1)[diff[0]],
        c_ref.reshape(-1)[diff[0]])


def test_act_quant_golden_examples(golden_dir):
    from test_oracle_pins import _parse_examples
    ex = _parse_examples(golden_dir)
    x = np.stack([e[1] for e in ex])
    codes, scales = fp4.act_quant_fp8(_gpu(x))
    for r, (ident, _, scale, want) in enumerate(ex):
        assert to_np(scales)[r, 0] == scale, ident
        for i, c in want.items():
            assert to_np(codes)[r, i] == c, (ident, i)


def test_act_quant_edge_shapes():
    for rows, k in [(1, 128), (3, 256), (1, 7168), (4096 + 3, 128)]:
        x = torch.randn(rows, k) * 3
        codes, scales = fp4.act_quant_fp8(x.to(DEV))
        c_ref, s_ref = oracle.act_quant(x.numpy())
        assert np.array_equal(to_np(codes), c_ref)
        assert np.array_equal(to_np(scales), s_ref)
    # rows == 0 is a no-op
    empty = torch.empty(0, 256, device=DEV)
    c, s = fp4.act_quant_fp8(empty)
    assert c.shape == (0, 256)


def _sweep_chunk(start_bits, count):
    """Codes of `count` consecutive f32 bit patterns starting at start_bits, computed by
    act_quant with one 448 per group so that the group scale is exactly 1."""
    groups = (count + 126) // 127
    bits = torch.arange(start_bits, start_bits + groups * 127, dtype=torch.int64, device=DEV)
    vals = bits.to(torch.int32).view(torch.float32)
    last = start_bits + count - 1
    vals = torch.where(bits <= last, vals, vals[count - 1])
    x = torch.empty(groups, 128, device=DEV)
    x[:, 0] = 448.0
    x[:, 1:] = vals.view(groups, 127)
    codes, scales = fp4.act_quant_fp8(x)
    assert bool(torch.all(scales == 1.0))
    return to_np(codes[:, 1:].reshape(-1)[:count])


def test_act_quant_encoder_exhaustive_sweep():
    """Every f32 in [-448, 448] (P-SWEEP): the GPU codes form the step function whose steps
    are the oracle's thresholds, so every code equals the oracle's."""
    thresholds = np.array([oracle.e4m3_threshold(c) for c in range(1, 0x7F)],
                          dtype=np.float32).view(np.uint32).astype(np.int64)
    top = int(np.array([448.0], dtype=np.float32).view(np.uint32)[0])
    chunk = 127 << 19
    for sign in (0, 0x80000000):
        start = 0
        while start <= top:
            count = min(chunk, top + 1 - start)
            codes = _sweep_chunk(start + sign if sign == 0 else
                                 (start | sign) - (1 << 32), count)
            mag = codes & 0x7F
            assert np.all((codes & 0x80) == (0x80 if sign else 0))
            first = oracle.e4m3_encode(np.array([start], dtype=np.uint32).view(np.float32))[0]
            assert mag[0] == first
            steps = np.flatnonzero(np.diff(mag.astype(np.int16)) != 0) + 1
            assert np.all(np.diff(mag.astype(np.int16)) >= 0)
            assert np.all(np.diff(mag.astype(np.int16)) <= 1)
            want = thresholds[(thresholds > start) & (thresholds < start + count)] - start
            assert np.array_equal(steps, want)
            start += count


# ------------------------------------------------------------------ single expert

@pytest.mark.parametrize("cfg", [1, 2])
def test_expert_gemm_configs(cfg):
    x, bank = synth.single_expert(cfg, device="cpu")
    w, sc, s2 = bank.w[0], bank.sc[0], float(bank.scale2[0])
    codes = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    scales = torch.empty(x.shape[0], x.shape[1] // 128, device=DEV)
    out = fp4.fp4_expert_gemm(x.to(DEV), w.to(DEV), sc.to(DEV), s2, bank.recipe,
                              codes_out=codes, scales_out=scales)
    c_ref, s_ref, ref, absp = expert_reference(x.numpy(), w.numpy(), sc.numpy(), s2, bank.recipe)
    assert np.array_equal(to_np(codes), c_ref) and np.array_equal(to_np(scales), s_ref)
    n_ops = gemm_bound(fp4.PATH_STREAM, bank.recipe, x.shape[1])
    check_gemm(to_np(out), ref, absp, n_ops, "c%d" % cfg)
    out2 = fp4.fp4_expert_gemm(x.to(DEV), w.to(DEV), sc.to(DEV), s2, bank.recipe)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
@pytest.mark.parametrize("g,n,k", [(1, 1, 128), (3, 200, 256), (5, 64, 1536), (9, 129, 512),
                                   (2, 70, 7168), (17, 100, 384), (3, 40, 28672)])
def test_expert_gemm_shapes(recipe, g, n, k):
    """Ragged n (not a multiple of the tile), short k (idle lanes), k that is not a
    multiple of 256 or 1024, rows not a multiple of the rows per pass, and a k too long
    for the warp-MMA kernel's shared memory (the FMA streaming kernel takes it)."""
    rng = np.random.default_rng(g * 1000 + n + k + recipe)
    x = (rng.standard_normal((g, k)) * rng.choice([1e-3, 1, 100], (g, 1))).astype(np.float32)
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    gs = fp4.group_size(recipe)
    if recipe == fp4.NVFP4:
        sc = rng.integers(0x08, 0x7E, (n, k // gs), dtype=np.uint8)
        s2 = 5.9945243e-5
    else:
        sc = rng.integers(100, 150, (n, k // gs), dtype=np.uint8)
        s2 = 0.0
    out = fp4.fp4_expert_gemm(_gpu(x), _gpu(w), _gpu(sc), s2, recipe)
    _, _, ref, absp = expert_reference(x, w, sc, s2, recipe)
    check_gemm(to_np(out), ref, absp, gemm_bound(fp4.PATH_STREAM, recipe, k), "shape")


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
@pytest.mark.parametrize("spreads", [(0, 15, 3, 0), (16, 0, 0, 0), (15, 15, 40, 7), (60, 0, 0, 0)])
def test_expert_gemm_block_scale_spread(recipe, spreads):
    """Rows whose 128-blocks have act scales 2^j far apart: within 2^15 of the row's
    largest, the decode kernel takes f16 activations scaled by the row's largest block;
    a wider spread in any row of the pass takes bf16 for the whole pass. Block amax is
    448 * 2^j exactly, so the scale is 2^j, and every block keeps codes down to 2^-9."""
    rng = np.random.default_rng(91 + recipe + sum(spreads))
    g, n, k = len(spreads), 96, 2048
    x = rng.uniform(-1.0, 1.0, (g, k)).astype(np.float32)
    x[:, ::128] = 1.0                                            # amax exactly 448 * 2^j
    x[:, 1::128] = 2.0 ** -9 / 448.0                             # the smallest e4m3 code
    for r, spread in enumerate(spreads):
        j = np.full(k // 128, -10.0 + rng.integers(-3, 4))     # above the 1e-4 amax floor
        j[::2] += spread
        x[r] *= np.repeat(448.0 * 2.0 ** j, 128).astype(np.float32)
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    if recipe == fp4.NVFP4:
        sc = rng.integers(0x08, 0x7E, (n, k // 16), dtype=np.uint8)
        s2 = 5.9945243e-5
    else:
        sc = rng.integers(100, 150, (n, k // 32), dtype=np.uint8)
        s2 = 0.0
    codes = torch.empty((g, k), dtype=torch.uint8, device=DEV)
    scales = torch.empty((g, k // 128), device=DEV)
    out = fp4.fp4_expert_gemm(_gpu(x), _gpu(w), _gpu(sc), s2, recipe, codes_out=codes,
                              scales_out=scales)
    c_ref, s_ref, ref, absp = expert_reference(x, w, sc, s2, recipe)
    assert np.array_equal(to_np(codes), c_ref) and np.array_equal(to_np(scales), s_ref)
    exps = np.log2(s_ref)
    assert np.all(exps == np.round(exps))
    assert [int(exps[r].max() - exps[r].min()) for r in range(g)] == list(spreads)
    check_gemm(to_np(out), ref, absp, gemm_bound(fp4.PATH_STREAM, recipe, k), "spread")
    # each row alone (its own pass, its own route) agrees with the oracle too
    for r in range(g):
        one = fp4.fp4_expert_gemm(_gpu(x[r:r + 1]), _gpu(w), _gpu(sc), s2, recipe)
        check_gemm(to_np(one), ref[r:r + 1], absp[r:r + 1],
                   gemm_bound(fp4.PATH_STREAM, recipe, k), "spread row %d" % r)


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_expert_gemm_exact_special_case(recipe, golden_dir):
    """P-EXACT: lossless quantisation, unit weight scales -> bit-equal to a float64 matmul."""
    from test_oracle_pins import _dense_weights, _exact_inputs, golden_e2m1
    rng = np.random.default_rng(77 + recipe)
    table = golden_e2m1(golden_dir)
    for g, n, k in [(3, 5, 256), (8, 64, 1024), (4, 96, 2048)]:
        x, w, sc = _exact_inputs(rng, g, n, k, recipe)
        out = fp4.fp4_expert_gemm(_gpu(x), _gpu(w), _gpu(sc), 1.0, recipe)
        want = x.astype(np.float64) @ _dense_weights(w, table).T
        assert np.array_equal(to_np(out).astype(np.float64), want)


# ------------------------------------------------------------------ grouped

def _small_grouped(recipe, device=DEV, E=6, T=40, topk=3, n=136, k=512, empty=(1, 4)):
    gen = torch.Generator(device="cpu").manual_seed(100 + recipe)
    scores = torch.rand(T, E, generator=gen)
    for e in empty:
        scores[:, e] = -1.0
    choices = torch.argsort(scores, dim=1, descending=True)[:, :topk]
    r = synth.routing_from_choices(choices, E)
    bank = synth.make_bank(recipe, E, n, k, 555, "cpu", scale2_value=5.9945243e-5)
    x = torch.randn(T, k, generator=gen) * 4
    proj = synth.Projection("small", x.to(device), synth.Routing(r.offsets.to(device),
                                                                  r.row_ids.to(device)),
                            synth.Bank(recipe, bank.w.to(device), bank.sc.to(device),
                                       bank.scale2.to(device)))
    return proj


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
@pytest.mark.parametrize("path", [fp4.PATH_STREAM])
def test_grouped_small_all_outputs(recipe, path):
    proj = _small_grouped(recipe)
    fp4.fp4_force_path(path)
    try:
        out, used = run_projection(proj)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    assert used == path
    P = proj.routing.P
    grouped_sampled_check(proj, out, path, np.arange(P), "small grouped")
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_grouped_decode_many_experts_ragged_passes(recipe):
    """The weight-streaming decode path over hundreds of experts holding 0-19 routed rows
    each (passes of up to 8 rows, item runs that split a pass across CTAs), ragged n and a
    k of several 512-k ring stages: every output against the oracle."""
    gen = torch.Generator().manual_seed(31 + recipe)
    E, T, n, k = 300, 64, 200, 1024
    sizes = torch.randint(0, 20, (E,), generator=gen)
    sizes[::7] = 0
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(sizes, 0).to(torch.int32)
    P = int(offsets[-1])
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    bank = synth.make_bank(recipe, E, n, k, 777 + recipe, "cpu", scale2_value=5.9945243e-5)
    x = torch.randn(T, k, generator=gen) * 2
    proj = synth.Projection("many", x.to(DEV), synth.Routing(offsets.to(DEV), row_ids.to(DEV)),
                            synth.Bank(recipe, bank.w.to(DEV), bank.sc.to(DEV),
                                       bank.scale2.to(DEV)))
    fp4.fp4_force_path(fp4.PATH_STREAM)
    try:
        out, used = run_projection(proj)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    assert used == fp4.PATH_STREAM
    grouped_sampled_check(proj, out, used, np.arange(P), "decode many experts")
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("E", [1024, 1025])
def test_grouped_decode_expert_limit(E):
    """The most experts the TMA-fed decode kernel takes (1024), and one more (the
    per-lane-load kernel then runs): routed rows on a few hundred experts, every output."""
    gen = torch.Generator().manual_seed(E)
    n, k, T = 64, 512, 32
    sizes = torch.zeros(E, dtype=torch.int64)
    hot = torch.randperm(E, generator=gen)[:300]
    sizes[hot] = torch.randint(1, 4, (300,), generator=gen)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(sizes, 0).to(torch.int32)
    P = int(offsets[-1])
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    bank = synth.make_bank(fp4.NVFP4, E, n, k, 555, "cpu", scale2_value=5.9945243e-5)
    x = torch.randn(T, k, generator=gen)
    proj = synth.Projection("limit", x.to(DEV), synth.Routing(offsets.to(DEV), row_ids.to(DEV)),
                            synth.Bank(fp4.NVFP4, bank.w.to(DEV), bank.sc.to(DEV),
                                       bank.scale2.to(DEV)))
    out, used = run_projection(proj, workspace=None)
    assert used == fp4.PATH_STREAM
    grouped_sampled_check(proj, out, used, np.arange(P), "decode %d experts" % E)
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_grouped_decode_back_to_back_dependency(recipe):
    """Two decode-path calls queued back to back on one stream, the second reading the
    first's output as its activations (as a down projection reads h). The second kernel may
    be scheduled while the first drains, and must read nothing before the first has
    finished: the first output starts as NaN, and every output of the second call is checked
    against the oracle run on the first call's final output."""
    gen = torch.Generator().manual_seed(909 + recipe)
    E, T, n1, k1, n2 = 24, 16, 1536, 1024, 512
    sizes = torch.randint(0, 4, (E,), generator=gen)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(sizes, 0).to(torch.int32)
    P = int(offsets[-1])
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    b1 = synth.make_bank(recipe, E, n1, k1, 901, "cpu", scale2_value=5.9945243e-5)
    b2 = synth.make_bank(recipe, E, n2, n1, 902, "cpu", scale2_value=1.0 / 64.0)
    bank1 = synth.Bank(recipe, b1.w.to(DEV), b1.sc.to(DEV), b1.scale2.to(DEV))
    bank2 = synth.Bank(recipe, b2.w.to(DEV), b2.sc.to(DEV), b2.scale2.to(DEV))
    x = (torch.randn(T, k1, generator=gen) * 2).to(DEV)
    off_d, rid_d = offsets.to(DEV), row_ids.to(DEV)
    ident = torch.arange(P, dtype=torch.int32, device=DEV)
    assert fp4.fp4_gemm_path(P, E, n1, k1, recipe, False) == fp4.PATH_STREAM
    for _ in range(3):
        h = torch.full((P, n1), float("nan"), device=DEV)
        torch.cuda.synchronize()
        fp4.fp4_grouped_expert_gemm(x, rid_d, off_d, bank1.w, bank1.sc, bank1.scale2, recipe,
                                    out=h)
        y = fp4.fp4_grouped_expert_gemm(h, ident, off_d, bank2.w, bank2.sc, bank2.scale2,
                                        recipe)
        torch.cuda.synchronize()
        assert not torch.isnan(h).any()
        proj = synth.Projection("chained", h, synth.Routing(off_d, ident), bank2)
        grouped_sampled_check(proj, y, fp4.PATH_STREAM, np.arange(P), "decode chained")
    assert fp4.fp4_get_device_error() == 0


def test_grouped_row_equals_single_row_launch():
    """P-ROW: a routed row's output equals the single-expert call on that row alone."""
    proj = _small_grouped(fp4.NVFP4)
    fp4.fp4_force_path(fp4.PATH_STREAM)
    try:
        out, _ = run_projection(proj)
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    off = to_np(proj.routing.offsets)
    rid = to_np(proj.routing.row_ids)
    for p in [0, 5, int(off[-1]) - 1]:
        e = int(np.searchsorted(off, p, side="right") - 1)
        t = int(rid[p])
        one = fp4.fp4_expert_gemm(proj.x[t:t + 1].contiguous(), proj.bank.w[e], proj.bank.sc[e],
                                  float(proj.bank.scale2[e]), proj.bank.recipe)
        assert torch.equal(one[0], out[p])


def test_grouped_device_checks_flag_bad_routing():
    proj = _small_grouped(fp4.NVFP4)
    assert fp4.fp4_get_device_error() == 0
    bad = proj.routing.row_ids.clone()
    bad[3] = proj.x.shape[0] + 5
    fp4.fp4_force_path(fp4.PATH_STREAM)
    try:
        fp4.fp4_grouped_expert_gemm(proj.x, bad, proj.routing.offsets, proj.bank.w, proj.bank.sc,
                                    proj.bank.scale2, proj.bank.recipe)
        assert fp4.fp4_get_device_error() & fp4.FP4_DEVERR_ROW_ID
        off = proj.routing.offsets.clone()
        off[2], off[3] = off[3].clone(), off[2].clone()
        if int(off[2]) == int(off[3]):
            off[2] += 1
        fp4.fp4_grouped_expert_gemm(proj.x, proj.routing.row_ids, off, proj.bank.w,
                                    proj.bank.sc, proj.bank.scale2, proj.bank.recipe)
        assert fp4.fp4_get_device_error() & fp4.FP4_DEVERR_OFFSETS
    finally:
        fp4.fp4_force_path(fp4.PATH_AUTO)
    # the context stays usable and the word is cleared
    assert fp4.fp4_get_device_error() == 0
    out, path = run_projection(proj)
    grouped_sampled_check(proj, out, path, np.arange(proj.routing.P), "after errors")


@pytest.mark.parametrize("scale2", [1.0 / 64.0, 5.9945243e-5])
def test_grouped_decode_c3_full_size(scale2):
    wl = synth.decode_c3(device=DEV, scale2_value=scale2)
    rng = np.random.default_rng(3)
    for proj in wl.projections:
        out, path = run_projection(proj)
        rows = np.arange(proj.routing.P)          # 64 routed rows: check them all
        grouped_sampled_check(proj, out, path, rows, "c3 " + proj.name)
    assert fp4.fp4_get_device_error() == 0
    del rng


@pytest.mark.parametrize("variant", ["mxfp4", "nvfp4_wide_spread"])
def test_grouped_decode_shapes_full_size_variants(variant):
    """The decode workload's shapes (64 experts, 8 tokens top-8, gate/up [3072, 4096] and
    down [4096, 1536]) with an MXFP4 bank, and with NVFP4 activations whose 128-blocks
    alternate between x 2^8 and x 2^-10 (block scales about 2^18 apart, past the f16
    route's 2^15): both take the bf16 operands of the no-workspace kernel. Every routed
    row, every column."""
    wl = synth.decode_c3(device=DEV)
    for proj in wl.projections:
        bank, x = proj.bank, proj.x
        if variant == "mxfp4":
            bank = synth.make_bank(fp4.MXFP4, bank.E, bank.n, bank.k, 1203, DEV)
        else:
            blocks = torch.arange(x.shape[1] // 128, device=DEV)
            f = torch.where(blocks % 2 == 0, 2.0 ** 8, 2.0 ** -10).repeat_interleave(128)
            x = (x * f).contiguous()
        proj = synth.Projection(proj.name, x, proj.routing, bank, row_ids_used=proj.row_ids_used)
        if variant != "mxfp4":
            _, scales = oracle.act_quant(to_np(x[:4]))
            e = np.log2(scales)
            assert np.all(e.max(axis=1) - e.min(axis=1) > 15)
        out, path = run_projection(proj)
        assert path == fp4.PATH_STREAM
        grouped_sampled_check(proj, out, path, np.arange(proj.routing.P),
                              "c3 %s %s" % (variant, proj.name))
    assert fp4.fp4_get_device_error() == 0


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_grouped_prefill_full_size_sampled(name):
    wl = synth.workload(name, device=DEV)
    rng = np.random.default_rng(4)
    for proj in wl.projections:
        out, path = run_projection(proj)
        rows = sample_rows(to_np(proj.routing.offsets).astype(np.int64), proj.routing.P, rng, 48)
        grouped_sampled_check(proj, out, path, rows, "%s %s" % (name, proj.name))
        del out
    assert fp4.fp4_get_device_error() == 0
