"""Pins of the CPU oracle to things other than itself (no GPU).

Each test ties an oracle function to a library routine, a hand-derived worked example
from the pages' definitions, a closed form, an invariant, or brute force on tiny inputs,
so that a dropped term, a wrong sign or index, or a transposed operand fails one of them.
Pages: memra-engine 0.98.0 src/bin/dsv4_native_gemm_gate.rs (fn quant_rows, fn f64_ref,
struct ExpertRaw) and 0.71.0 src/bin/kernel_check.rs (e4m3 decoder, FP4 grid facts).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

# ----------------------------------------------------------------- independent decoders

def torch_e4m3(codes):
    """Library decode (torch float8_e4m3fn) -> float64."""
    c = torch.as_tensor(np.asarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(values):
    v = torch.as_tensor(np.asarray(values, dtype=np.float32))
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def golden_e2m1(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "e2m1_grid.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    table = np.zeros(16)
    for c in range(8):
        table[c] = vals[c]
        table[c + 8] = -vals[c]
    return table


# ----------------------------------------------------------------- e4m3

def test_e4m3_decode_matches_library_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = torch_e4m3(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}  # exponent 15 with mantissa 7
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_e4m3_decode_page_facts():
    d = oracle.e4m3_decode(np.array([0x7E, 0x01, 0x07, 0x08, 0x38, 0x80, 0xFE], dtype=np.uint8))
    assert d[0] == 448.0                 # largest finite
    assert d[1] == 2.0 ** -9             # exponent 0: mantissa * 2^-9
    assert d[2] == 7 * 2.0 ** -9
    assert d[3] == 2.0 ** -6             # smallest normal, bias 7
    assert d[4] == 1.0
    assert d[5] == 0.0 and np.signbit(d[5])
    assert d[6] == -448.0


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def _sweep_values():
    grid = np.sort(np.unique(np.abs(torch_e4m3(np.arange(0, 0x7F, dtype=np.uint8)))))
    mids = (grid[:-1] + grid[1:]) / 2.0          # exact in f32 (<= 5 significant bits)
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(0))
    rng = np.random.default_rng(7)
    rnd = (2.0 ** rng.uniform(-24, math.log2(448), 20000)).astype(np.float32)
    rnd = np.minimum(rnd, np.float32(448))
    tiny = np.array([0.0, 1e-30, 1e-9, 2.0 ** -10, 2.0 ** -11, 2.0 ** -10 * 1.0000001],
                    dtype=np.float32)
    pos = np.concatenate([grid.astype(np.float32), mids32, up, dn, rnd, tiny])
    return np.concatenate([pos, -pos, np.array([-0.0], dtype=np.float32)])


def test_e4m3_encode_matches_library_rne():
    v = _sweep_values()
    assert np.all(np.abs(v) <= 448)
    assert np.array_equal(oracle.e4m3_encode(v), torch_encode(v))


def test_e4m3_encode_is_nearest_by_brute_force():
    """Nearest of all 254 finite codes, ties to the even code, sign kept."""
    codes = np.array([c for c in range(0x7F)], dtype=np.uint8)
    grid = torch_e4m3(codes)
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1e-2, 3000)]).astype(np.float32)
    got = oracle.e4m3_encode(v)
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1)
    for i in range(v.size):
        cands = np.flatnonzero(d[i] == best[i])
        c = cands[0] if cands.size == 1 else [c for c in cands if c % 2 == 0][0]
        want = c | (0x80 if np.signbit(v[i]) else 0)
        assert got[i] == want, (v[i], got[i], want)


def test_e4m3_thresholds_match_library():
    for code in range(0, 0x7F):
        t = oracle.e4m3_threshold(code)
        assert torch_encode([t])[0] == code
        if code > 0:
            below = np.nextafter(np.float32(t), np.float32(0))
            assert torch_encode([below])[0] == code - 1


# ----------------------------------------------------------------- e2m1 / e8m0

def test_e2m1_grid_matches_golden(golden_dir):
    got = oracle.e2m1_decode(np.arange(16))
    want = golden_e2m1(golden_dir)
    assert np.array_equal(np.abs(got), np.abs(want))
    assert np.array_equal(got[1:8], want[1:8]) and np.array_equal(got[9:], want[9:])
    assert np.all(np.signbit(got[8:])) and not np.any(np.signbit(got[:8]))
    # page facts: 8 grid points per sign, top point 6
    assert len(set(np.abs(got).tolist())) == 8 and np.max(np.abs(got)) == 6.0
    assert np.all(np.diff(got[:8]) > 0)


def test_e8m0_closed_form():
    e = np.arange(255, dtype=np.uint8)
    got = oracle.e8m0_decode(e)
    assert np.array_equal(got, np.ldexp(1.0, e.astype(np.int64) - 127))
    assert np.isnan(oracle.e8m0_decode(np.array([255], dtype=np.uint8))[0])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127


# ----------------------------------------------------------------- pow2_ceil

def test_pow2_ceil_invariants():
    rng = np.random.default_rng(3)
    x = (2.0 ** rng.uniform(-40, 100, 5000)).astype(np.float32)
    x = np.concatenate([x, np.ldexp(np.float32(1), np.arange(-30, 30)).astype(np.float32),
                        np.array([2.2321428e-07, 1.0, 0.75, 1.5, 3.0], dtype=np.float32)])
    s = oracle.pow2_ceil(x)
    m, _ = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)                         # a power of two
    xs = x.astype(np.float64)
    ss = s.astype(np.float64)
    assert np.all(ss >= xs) and np.all(ss / 2 < xs)  # the smallest one >= x


# ----------------------------------------------------------------- act_quant

def _parse_examples(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "act_quant_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ident, fill, over, slog, codes = [p.strip() for p in line.split("|")]
            x = np.full(128, float(fill), dtype=np.float32)
            if over != "-":
                for item in over.split(","):
                    i, v = item.split(":")
                    x[int(i)] = np.float32(float(v))
            exp = {int(i): int(c, 16) for i, c in (it.split(":") for it in codes.split(","))}
            out.append((ident, x, float(2.0 ** int(slog)), exp))
    return out


def test_act_quant_worked_examples(golden_dir):
    ex = _parse_examples(golden_dir)
    assert len(ex) >= 7
    for ident, x, scale, codes in ex:
        c, s = oracle.act_quant(x[None, :])
        assert s[0, 0] == scale, ident
        for i, want in codes.items():
            assert c[0, i] == want, (ident, i, hex(c[0, i]), hex(want))


def _random_rows(rng, rows, k):
    x = rng.standard_normal((rows, k)).astype(np.float32)
    x[1] *= 1e-6                                   # floor territory
    x[2, :128] = 0.0                               # all-zero group
    x[3] = (rng.standard_t(3, k) * 100).astype(np.float32)
    mask = rng.random((rows, k)) < 0.01
    x[mask] *= 50.0
    x[4, :64] = np.float32(1e-40) * rng.standard_normal(64).astype(np.float32)  # subnormals
    x[5] = torch.tensor(x[5]).to(torch.bfloat16).float().numpy()  # bf16-range ties
    return x


def test_act_quant_invariants_and_brute_force_codes():
    rng = np.random.default_rng(5)
    rows, k = 8, 512
    x = _random_rows(rng, rows, k)
    codes, scales = oracle.act_quant(x)
    grid_codes = np.array([c for c in range(0x7F)], dtype=np.uint8)
    grid = torch_e4m3(grid_codes)
    for r in range(rows):
        for g in range(k // 128):
            grp = x[r, g * 128:(g + 1) * 128].astype(np.float64)
            s = float(scales[r, g])
            m, _ = np.frexp(s)
            assert m == 0.5                                   # power of two
            amax = max(np.max(np.abs(grp)), float(np.float32(1e-4)))
            assert s * 448 >= amax * (1 - 2.0 ** -23)         # x/s never needs the clamp
            dec = torch_e4m3(codes[r, g * 128:(g + 1) * 128])
            if np.max(np.abs(grp)) >= 1e-4:
                top = np.max(np.abs(dec))
                assert 224 <= top <= 448, (r, g, top)
            if np.all(grp == 0):
                assert s == 2.0 ** -22 and np.all(codes[r, g * 128:(g + 1) * 128] == 0)
            q = grp / s                                       # exact (power of two)
            d = np.abs(np.abs(q)[:, None] - grid[None, :])
            best = d.min(axis=1)
            for i in range(128):
                cands = np.flatnonzero(d[i] == best[i])
                c = cands[0] if cands.size == 1 else [c for c in cands if c % 2 == 0][0]
                want = c | (0x80 if np.signbit(q[i]) else 0)
                assert codes[r, g * 128 + i] == want


def test_act_quant_matches_library_pipeline():
    """Same steps with numpy f32 arithmetic and torch's e4m3 conversion."""
    rng = np.random.default_rng(9)
    x = _random_rows(rng, 8, 1024)
    codes, scales = oracle.act_quant(x)
    g = x.reshape(8, 8, 128)
    amax = np.maximum(np.max(np.abs(g), axis=2), np.float32(1e-4)).astype(np.float32)
    t = (amax * np.float32(1.0 / 448.0)).astype(np.float32)
    s = np.exp2(np.ceil(np.log2(t.astype(np.float64)))).astype(np.float32)
    assert np.array_equal(s, scales)
    q = np.clip((g / s[:, :, None]).astype(np.float32), -448, 448)
    assert np.array_equal(torch_encode(q.reshape(8, 1024)), codes)


# ----------------------------------------------------------------- GEMM reference

def _exact_inputs(rng, g, n, k, recipe):
    """Lossless special case: per-group amax exactly 448*2^m with integer codes, unit weight
    scales. Returns x, w, sc, and the decoded dense matrices."""
    kq = k // 128
    m = rng.integers(-1, 2, (g, kq))
    c = rng.integers(-16, 17, (g, k)).astype(np.float64)
    c.reshape(g, kq, 128)[:, :, 0] = 448.0 * rng.choice([-1, 1], (g, kq))
    x = (c.reshape(g, kq, 128) * np.exp2(m)[:, :, None]).reshape(g, k).astype(np.float32)
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    gs = 16 if recipe == oracle.NVFP4 else 32
    sc = np.full((n, k // gs), 0x38 if recipe == oracle.NVFP4 else 127, dtype=np.uint8)
    return x, w, sc


def _dense_weights(w, table):
    n, kh = w.shape
    lo = table[w & 0x0F]
    hi = table[w >> 4]
    dense = np.empty((n, kh * 2))
    dense[:, 0::2] = lo       # low nibble = even k (struct ExpertRaw / mirror_gemm)
    dense[:, 1::2] = hi
    return dense


@pytest.mark.parametrize("recipe", [oracle.NVFP4, oracle.MXFP4])
def test_gemm_exact_special_case_is_plain_matmul(recipe, golden_dir):
    rng = np.random.default_rng(21 + recipe)
    table = golden_e2m1(golden_dir)
    for g, n, k in [(3, 5, 256), (8, 64, 1024)]:
        x, w, sc = _exact_inputs(rng, g, n, k, recipe)
        codes, scales = oracle.act_quant(x)
        # quantisation is lossless here
        deq = torch_e4m3(codes) * np.repeat(scales.astype(np.float64), 128, axis=1)
        assert np.array_equal(deq, x.astype(np.float64))
        out, absp = oracle.gemm_ref(codes, scales, w, sc, 1.0, recipe)
        want = x.astype(np.float64) @ _dense_weights(w, table).T
        assert np.array_equal(out, want)
        assert np.array_equal(absp, np.abs(x.astype(np.float64)) @ np.abs(_dense_weights(w, table)).T)


def _rational_ref(codes, scales, w, sc, scale2, recipe, table):
    g, k = codes.shape
    n = w.shape[0]
    gs = 16 if recipe == oracle.NVFP4 else 32
    adec = torch_e4m3(codes)
    wd = _dense_weights(w, table)
    out = np.empty((g, n), dtype=object)
    absp = np.empty((g, n), dtype=object)
    for r in range(g):
        for col in range(n):
            acc = Fraction(0)
            ab = Fraction(0)
            for j in range(k // gs):
                if recipe == oracle.NVFP4:
                    ws = np.float32(torch_e4m3([sc[col, j]])[0]) * np.float32(scale2)
                else:
                    ws = np.float32(math.ldexp(1.0, int(sc[col, j]) - 127))
                f = Fraction(float(ws)) * Fraction(float(scales[r, (j * gs) // 128]))
                for i in range(gs):
                    kk = j * gs + i
                    p = Fraction(float(adec[r, kk])) * Fraction(float(wd[col, kk])) * f
                    acc += p
                    ab += abs(p)
            out[r, col] = acc
            absp[r, col] = ab
    return out, absp


@pytest.mark.parametrize("recipe,scale2", [(oracle.NVFP4, 1 / 64), (oracle.NVFP4, 5.9945243e-5),
                                           (oracle.MXFP4, 0.0)])
def test_gemm_matches_exact_rational_sum(recipe, scale2, golden_dir):
    rng = np.random.default_rng(31 + recipe)
    table = golden_e2m1(golden_dir)
    for g, n, k in [(2, 3, 128), (1, 4, 256)]:
        codes = rng.integers(0, 256, (g, k), dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C
        scales = np.exp2(rng.integers(-12, 4, (g, k // 128))).astype(np.float32)
        w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
        gs = 16 if recipe == oracle.NVFP4 else 32
        if recipe == oracle.NVFP4:
            sc = rng.integers(0x20, 0x41, (n, k // gs), dtype=np.uint8)
        else:
            sc = rng.integers(118, 135, (n, k // gs), dtype=np.uint8)
        out, absp = oracle.gemm_ref(codes, scales, w, sc, scale2, recipe)
        ex, exabs = _rational_ref(codes, scales, w, sc, scale2, recipe, table)
        for r in range(g):
            for c in range(n):
                e = float(ex[r, c])
                assert abs(out[r, c] - e) <= k * 2.0 ** -53 * float(exabs[r, c])
                assert abs(absp[r, c] - float(exabs[r, c])) <= k * 2.0 ** -53 * float(exabs[r, c])


def test_gemm_nibble_order_and_scale_indexing_worked_example():
    """Hand-computed outputs for one-hot activations (values from the definitions):
    row 0 is one-hot at k=1, row 1 one-hot at k=16, row 2 one-hot at k=128."""
    k, n = 256, 2
    x = np.zeros((3, k), dtype=np.float32)
    x[0, 1] = 1.0      # group 0: amax 1 -> s = 2^-8, code 256
    x[1, 16] = -2.0    # group 0: s = 2^-7, code -256
    x[2, 128] = 3.0    # group 1: s = 2^-7, code 384
    codes, scales = oracle.act_quant(x)
    w = np.zeros((n, k // 2), dtype=np.uint8)
    w[0, 0] = 0x21     # col 0: k=0 -> code 1 (0.5), k=1 -> code 2 (1.0)
    w[0, 8] = 0x0D     # col 0: k=16 -> code 13 (-3.0), k=17 -> 0
    w[1, 64] = 0x07    # col 1: k=128 -> code 7 (6.0)
    w[1, 0] = 0xF0     # col 1: k=1 -> code 15 (-6.0)
    sc = np.full((n, k // 16), 0x38, dtype=np.uint8)   # 1.0
    sc[0, 1] = 0x40    # col 0, k in [16, 32): 2.0
    sc[1, 8] = 0x30    # col 1, k in [128, 144): 0.5
    out, _ = oracle.gemm_ref(codes, scales, w, sc, 0.25, oracle.NVFP4)
    # out[r, c] = code * E2M1 * (e4m3 scale * scale2) * activation scale
    assert out[0, 0] == 256 * 1.0 * (1.0 * 0.25) * 2.0 ** -8      # = 0.25
    assert out[0, 1] == 256 * -6.0 * (1.0 * 0.25) * 2.0 ** -8     # = -1.5
    assert out[1, 0] == -256 * -3.0 * (2.0 * 0.25) * 2.0 ** -7    # = 3.0
    assert out[1, 1] == 0.0
    assert out[2, 0] == 0.0
    assert out[2, 1] == 384 * 6.0 * (0.5 * 0.25) * 2.0 ** -7      # = 2.25
    # MXFP4: per-32 scale, e8m0 128 = 2.0 on k in [0, 32) of col 0
    sc2 = np.full((n, k // 32), 127, dtype=np.uint8)
    sc2[0, 0] = 128
    out2, _ = oracle.gemm_ref(codes, scales, w, sc2, 0.0, oracle.MXFP4)
    assert out2[0, 0] == 256 * 1.0 * 2.0 * 2.0 ** -8               # = 2.0
    assert out2[1, 0] == -256 * -3.0 * 2.0 * 2.0 ** -7             # = 12.0
    assert out2[2, 1] == 384 * 6.0 * 1.0 * 2.0 ** -7               # = 18.0


def test_grouped_reference_routing_worked_example():
    """Expert 1 empty; routed rows gather tokens out of order; each sampled output must
    equal the single-expert reference on the hand-picked token and expert."""
    rng = np.random.default_rng(41)
    T, k, n, E = 5, 256, 6, 3
    x = rng.standard_normal((T, k)).astype(np.float32)
    offsets = np.array([0, 2, 2, 5], dtype=np.int32)
    row_ids = np.array([4, 0, 1, 1, 3], dtype=np.int32)
    expert_of_row = [0, 0, 2, 2, 2]
    w = rng.integers(0, 256, (E, n, k // 2), dtype=np.uint8)
    sc = rng.integers(0x20, 0x41, (E, n, k // 16), dtype=np.uint8)
    s2 = np.array([1 / 64, 1 / 32, 1 / 16], dtype=np.float32)
    sp = np.repeat(np.arange(5), n)
    scol = np.tile(np.arange(n), 5)
    out, absp = oracle.grouped_ref_sampled(x, row_ids, offsets, w, sc, s2, oracle.NVFP4, sp, scol)
    for p in range(5):
        e = expert_of_row[p]
        codes, scales = oracle.act_quant(x[row_ids[p]][None, :])
        ref, rabs = oracle.gemm_ref(codes, scales, w[e], sc[e], s2[e], oracle.NVFP4)
        assert np.array_equal(out[p * n:(p + 1) * n], ref[0])
        assert np.array_equal(absp[p * n:(p + 1) * n], rabs[0])
    with pytest.raises(ValueError):
        oracle.grouped_ref_sampled(x, np.array([4, 0, 1, 1, 9], dtype=np.int32), offsets, w, sc,
                                   s2, oracle.NVFP4, np.array([4]), np.array([0]))


def test_bound_checker_catches_planted_error():
    ref = np.array([1.0, -2.0, 3.0])
    absp = np.array([4.0, 4.0, 4.0])
    ok, ratio, _ = oracle.within_bound(ref + 4.0 * 2.0 ** -24 * 4.0 * np.array([1, -1, 0.5]),
                                       ref, absp, 4.0)
    assert ok and ratio <= 1.0
    ok, ratio, i = oracle.within_bound(ref + np.array([0, 0, 1e-3]), ref, absp, 4.0)
    assert not ok and i == 2
    assert oracle.max_rel(ref + 3e-3, ref) == pytest.approx(1e-3)


# ---------------------------------------------------------------- SwiGLU (next row)
# The page (dsv4_native_gemm_gate.rs, swiglu_limit saturation cell and the f64 check of
# main) defines h = g * sigmoid(g) * u with u = clamp(up, -L, L) and g = min(gate, L).

def _silu_tanh(x):
    # logistic through tanh, an identity independent of the oracle's exp form:
    # sigmoid(x) = (1 + tanh(x / 2)) / 2
    x = np.asarray(x, dtype=np.float64)
    return x * 0.5 * (1.0 + np.tanh(0.5 * x))


def test_swiglu_matches_tanh_form_inside_the_clamps():
    rng = np.random.default_rng(11)
    L = 7.0
    gate = rng.uniform(-L, L, (4, 256)).astype(np.float32)
    up = rng.uniform(-L, L, (4, 256)).astype(np.float32)
    h = oracle.swiglu(gate, up, L)
    want = _silu_tanh(gate) * up.astype(np.float64)
    assert np.max(np.abs(h - want)) <= 1e-13 * np.max(np.abs(want))


def test_swiglu_odd_part_identity():
    # silu(x) - silu(-x) = x, so h(g, u) - h(-g, u) = g * u for |g| <= L
    rng = np.random.default_rng(12)
    L = 10.0
    g = rng.uniform(-L, L, (2, 512)).astype(np.float32)
    u = rng.uniform(-L, L, (2, 512)).astype(np.float32)
    d = oracle.swiglu(g, u, L) - oracle.swiglu(-g, u, L)
    want = g.astype(np.float64) * u.astype(np.float64)
    assert np.max(np.abs(d - want)) <= 1e-12 * np.max(np.abs(want))


def test_swiglu_clamp_semantics():
    L = 7.0
    one = np.ones((1, 1), np.float32)

    def h(g, u):
        return oracle.swiglu(np.full((1, 1), g, np.float32), np.full((1, 1), u, np.float32), L)[0, 0]

    # gate clamped from above, before the sigmoid: min(silu(2L), L) would give L instead
    assert h(2 * L, 1.0) == h(L, 1.0)
    assert abs(h(L, 1.0) - _silu_tanh(L)) < 1e-12 and h(L, 1.0) < L
    # gate not clamped from below: silu(-3L) is far smaller than silu(-L)
    assert abs(h(-3 * L, 1.0) - _silu_tanh(-3 * L)) < 1e-15
    assert abs(h(-3 * L, 1.0)) < abs(h(-L, 1.0)) / 100
    # up clamped on both sides
    assert h(1.0, 5 * L) == h(1.0, L)
    assert h(1.0, -5 * L) == h(1.0, -L)
    assert h(1.0, -5 * L) == -h(1.0, 5 * L)
    # silu(0) = 0 whatever the up value
    assert h(0.0, 3.0) == 0.0
    del one


def test_swiglu_row_stride_and_shape():
    rng = np.random.default_rng(13)
    gate = rng.standard_normal((3, 128)).astype(np.float32) * 4
    up = rng.standard_normal((3, 128)).astype(np.float32) * 4
    h = oracle.swiglu(gate, up, 6.0)
    assert h.shape == (3, 128) and h.dtype == np.float64
    # rows are independent
    h1 = oracle.swiglu(gate[1:2], up[1:2], 6.0)
    assert np.array_equal(h1[0], h[1])


# ---------------------------------------------------------------- mirror order (next row)
# fn mirror_gemm of dsv4_native_gemm_gate.rs: the page's kernel order in f32.

@pytest.mark.parametrize("recipe", [oracle.NVFP4, oracle.MXFP4])
def test_mirror_lossless_case_is_plain_matmul(recipe, golden_dir):
    # every partial sum is exact in f32 here (half-integers, |sum| <= k * 448 * 2 * 6
    # < 2^23 for k <= 1024), so any order gives the exact matmul
    rng = np.random.default_rng(41 + recipe)
    table = golden_e2m1(golden_dir)
    for g, n, k in [(3, 5, 256), (4, 9, 1024)]:
        x, w, sc = _exact_inputs(rng, g, n, k, recipe)
        codes, scales = oracle.act_quant(x)
        got = oracle.mirror_gemm(codes, scales, w, sc, 1.0, recipe).astype(np.float64)
        want = x.astype(np.float64) @ _dense_weights(w, table).T
        assert np.array_equal(got, want)


@pytest.mark.parametrize("recipe", [oracle.NVFP4, oracle.MXFP4])
def test_mirror_within_the_pages_bound(recipe):
    # the page states |mirror-order kernel - f64| <= n_ops 2^-24 sum|p| with
    # n_ops = (gs - 1) + ceil((k/gs)/128) + 7, for exactly this summation structure
    rng = np.random.default_rng(43 + recipe)
    gs = 16 if recipe == oracle.NVFP4 else 32
    for g, n, k in [(4, 32, 512), (3, 16, 8192)]:
        x = (rng.standard_normal((g, k)) * 3).astype(np.float32)
        w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
        sc = (rng.integers(0x20, 0x41, (n, k // gs)) if recipe == oracle.NVFP4
              else rng.integers(118, 135, (n, k // gs))).astype(np.uint8)
        s2 = 1.0 / 64 if recipe == oracle.NVFP4 else 0.0
        codes, scales = oracle.act_quant(x)
        ref, absp = oracle.gemm_ref(codes, scales, w, sc, s2, recipe)
        got = oracle.mirror_gemm(codes, scales, w, sc, s2, recipe)
        n_ops = (gs - 1) + int(np.ceil((k / gs) / 128)) + 7
        ok, worst, _ = oracle.within_bound(got, ref, absp, n_ops)
        assert ok, worst
        assert np.any(got.astype(np.float64) != ref)  # it does round


def test_mirror_halving_tree_order():
    """Worked example, k = 2048 (128 NVFP4 groups: partial t holds group t alone).
    Group 0 gives 32, groups 1 and 65 give 32 * 2^-24 each. The halving tree adds
    groups 1 and 65 first (offset 64), then that 2^-18 to 32 (offset 1): 32 + 2^-18,
    exact in f32. Adding left to right would give 32 (each 2^-19 is a tie to even)."""
    k, gs = 2048, 16
    codes = np.zeros((1, k), np.uint8)
    scales = np.ones((1, k // 128), np.float32)
    w = np.zeros((1, k // 2), np.uint8)
    sc = np.full((1, k // gs), 0x38, np.uint8)          # weight scale e4m3 1.0
    # group 0: a = 2 (0x40), w = 4 (E2M1 code 6, even k -> low nibble), ws = 4 (0x48): 32
    codes[0, 0] = 0x40
    w[0, 0] = 0x06
    sc[0, 0] = 0x48
    # groups 1 and 65: a = 2^-9 (0x01), w = 0.5 (code 1), ws = 2^-9 (0x01): 2^-19 each
    for grp in (1, 65):
        codes[0, grp * gs] = 0x01
        w[0, grp * gs // 2] = 0x01
        sc[0, grp] = 0x01
    got = oracle.mirror_gemm(codes, scales, w, sc, 1.0, oracle.NVFP4)[0, 0]
    assert got == np.float32(32.0 + 2.0 ** -18)
    seq = np.float32(32.0)
    for _ in range(2):
        seq = np.float32(seq + np.float32(2.0 ** -19))
    assert seq == np.float32(32.0)          # the order matters for this input
    ref, _ = oracle.gemm_ref(codes, scales, w, sc, 1.0, oracle.NVFP4)
    assert ref[0, 0] == 32.0 + 2.0 ** -18   # and the tree result is the exact sum


# ------------------------------------------------------------------ routing front-end

def _parse_routing(golden_dir):
    topk, csr = [], []
    with open(os.path.join(golden_dir, "routing_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("topk:"):
                parts = [p.strip() for p in line[5:].split(";")]
                topk.append((np.array(parts[0].split(), dtype=np.float32), int(parts[1]),
                             [int(v) for v in parts[2].split()], float(parts[3])))
            elif line.startswith("csr:"):
                parts = [p.strip() for p in line[4:].split(";")]
                ids = np.array([[int(v) for v in g.split()] for g in parts[1].split("|")],
                               dtype=np.int32)
                csr.append((int(parts[0]), ids, [int(v) for v in parts[2].split()],
                            [int(v) for v in parts[3].split()],
                            np.array([int(v) for v in parts[4].split()]).reshape(ids.shape)))
    return topk, csr


def test_route_topk_worked_examples(golden_dir):
    topk, _ = _parse_routing(golden_dir)
    assert len(topk) >= 4
    for logits, k, want_ids, want_w0 in topk:
        ids, w = oracle.route_topk(logits[None, :], k)
        assert ids[0].tolist() == want_ids
        assert abs(w[0, 0] - want_w0) <= 5e-9   # the fixture prints 9 decimals


def test_route_topk_matches_sort_and_softmax():
    """Selection = a stable sort of the experts by descending logit (numpy lexsort),
    weights = the softmax (closed form in numpy, f64), renormalised or not; logits drawn
    from a few values so that ties straddle the top-k boundary often."""
    rng = np.random.default_rng(71)
    for E, k in [(8, 2), (64, 8), (512, 10)]:
        logits = rng.choice(np.linspace(-3, 3, 13), size=(40, E)).astype(np.float32)
        logits[0] = 1.5                                   # all equal
        logits[1, :] = -200.0
        logits[1, 3] = 200.0                              # others underflow
        for renorm in (False, True):
            ids, w = oracle.route_topk(logits, k, renormalize=renorm)
            for t in range(logits.shape[0]):
                order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
                assert ids[t].tolist() == order[:k].tolist()
                z = np.exp(logits[t].astype(np.float64) - logits[t].max())
                p = z / z.sum()
                want = p[order[:k]] / (p[order[:k]].sum() if renorm else 1.0)
                np.testing.assert_allclose(w[t], want, rtol=1e-12, atol=0)
    ids, _ = oracle.route_topk(np.full((1, 16), 0.5, np.float32), 4)
    assert ids[0].tolist() == [0, 1, 2, 3]


def test_route_csr_worked_examples(golden_dir):
    _, csr = _parse_routing(golden_dir)
    assert len(csr) >= 3
    for E, ids, off, rid, prows in csr:
        o, r, p = oracle.route_csr(ids, E)
        assert o.tolist() == off and r.tolist() == rid
        assert np.array_equal(p, prows)


def test_route_csr_matches_stable_sort():
    """Routed rows = the (token, slot) pairs stably sorted by expert (numpy argsort, kind
    stable, over the token-major pair list); offsets = the cumulative counts."""
    rng = np.random.default_rng(72)
    for T, E, k in [(1, 4, 1), (37, 16, 3), (300, 64, 8)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        off, rid, prow = oracle.route_csr(ids, E)
        flat = ids.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert rid.tolist() == (order // k).tolist()
        pos = np.empty_like(order)
        pos[order] = np.arange(order.size)
        assert prow.reshape(-1).tolist() == pos.tolist()
        assert off.tolist() == [0] + np.cumsum(np.bincount(flat, minlength=E)).tolist()
    with pytest.raises(ValueError):
        oracle.route_csr(np.array([[0, 4]], np.int32), 4)


def test_moe_combine_closed_forms():
    rng = np.random.default_rng(73)
    T, k, n = 5, 3, 64
    out = rng.standard_normal((T * k, n)).astype(np.float32)
    prow = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    onehot = np.zeros((T, k), np.float32)
    onehot[:, 1] = 1.0
    y, absy = oracle.moe_combine(out, prow, onehot)
    assert np.array_equal(y, out[prow[:, 1]].astype(np.float64))     # selection, exact
    w = rng.random((T, k)).astype(np.float32)
    y, absy = oracle.moe_combine(out, prow, w)
    want = np.einsum("tj,tjc->tc", w.astype(np.float64), out[prow].astype(np.float64))
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(absy, np.einsum("tj,tjc->tc", np.abs(w.astype(np.float64)),
                                               np.abs(out[prow].astype(np.float64))), rtol=1e-13)


# ----------------------------------------------------------------- W4A4 variant
# NVFP4 W4A4 MMQ GEMM section of memra-engine 0.71.0 src/bin/kernel_check.rs: two-level
# activation scaling (row scale + e4m3 micro-scale per 16), its sub-block-only form (V1),
# the informational rel band and the dynamic-range arm.

def _w4a4_examples(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "w4a4_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ident, vals, rs, sc, by, v1sc, v1by = [p.strip() for p in line.split("|")]
            x = np.zeros(32, dtype=np.float32)
            if vals != "-":
                for item in vals.split(","):
                    i, v = item.split(":")
                    x[int(i)] = np.float32(float(v))
            if "/" in rs:
                a, b = rs.split("/")
                rsv = np.float32(float(a)) / np.float32(float(b))
            else:
                rsv = np.float32(float(rs))

            def table(spec, size):
                t = np.zeros(size, dtype=np.uint8)
                if spec != "-":
                    for item in spec.split(","):
                        i, v = item.split(":")
                        t[int(i)] = int(v, 16)
                return t
            scales, codes = table(sc, 2), table(by, 16)
            v1s = scales if v1sc == "=" else table(v1sc, 2)
            v1c = codes if v1by == "=" else table(v1by, 16)
            out.append((ident, x, rsv, scales, codes, v1s, v1c))
    return out


def test_w4a4_quant_worked_examples(golden_dir):
    ex = _w4a4_examples(golden_dir)
    assert len(ex) >= 5
    for ident, x, rs, scales, codes, v1s, v1c in ex:
        c, s, r = oracle.act_quant_w4a4(x[None, :])
        assert r[0] == rs, (ident, r[0], rs)
        assert np.array_equal(s[0], scales), (ident, s[0], scales)
        assert np.array_equal(c[0], codes), (ident, [hex(v) for v in c[0]])
        c1, s1 = oracle.act_quant_w4a4_v1(x[None, :])
        assert np.array_equal(s1[0], v1s), (ident, s1[0], v1s)
        assert np.array_equal(c1[0], v1c), (ident, [hex(v) for v in c1[0]])


def test_e2m1_encode_thresholds_and_ties(golden_dir):
    """Midpoints of the E2M1 grid (values from the golden grid file): the tie goes to the
    even code, one f32 ulp either side goes to the nearer neighbour; above 6 saturates."""
    grid = golden_e2m1(golden_dir)[:8]
    for c in range(7):
        mid = np.float32((grid[c] + grid[c + 1]) / 2)
        even = c if c % 2 == 0 else c + 1
        assert oracle.e2m1_encode([mid])[0] == even, (c, mid)
        assert oracle.e2m1_encode([np.nextafter(mid, np.float32(0))])[0] == c
        assert oracle.e2m1_encode([np.nextafter(mid, np.float32(10))])[0] == c + 1
        assert oracle.e2m1_encode([-mid])[0] == even | 8
    assert oracle.e2m1_encode([6.0, 6.5, 100.0, 3e38])[:].tolist() == [7, 7, 7, 7]
    assert oracle.e2m1_encode([-0.0, -1e-30, 0.0])[:].tolist() == [8, 8, 0]
    # brute force on random values: nearest grid value, ties cannot occur off the midpoints
    v = np.random.default_rng(3).uniform(-8, 8, 4000).astype(np.float32)
    got = oracle.e2m1_encode(v)
    mag = np.abs(v.astype(np.float64))
    want = np.argmin(np.abs(mag[:, None] - grid[None, :]), axis=1)
    assert np.array_equal(got & 7, want)
    assert np.array_equal(got >> 3, (v < 0).astype(np.uint8))


def _w4a4_rows(rng, rows, k):
    x = rng.uniform(-1, 1, (rows, k)).astype(np.float32) * np.float32(0.1)
    x[1] *= np.float32(1e-5)                          # a quiet token
    x[2, 16:48] = 0.0                                 # two all-zero blocks
    x[3] = (rng.standard_t(3, k) * 10).astype(np.float32)
    x[4, ::37] *= 300.0                               # outlier channels
    x[5] = 0.0                                        # a zero row
    return x


def test_w4a4_quant_block_brute_force_and_invariants(golden_dir):
    """Each code is the nearest E2M1 point (brute force over the golden grid) to the
    row-normalised value over its block's micro-scale, both quotients formed in numpy f32;
    the micro-scale is the e4m3 code nearest max|y|/6 (torch's e4m3 rounding); the block
    holding the row's amax gets 0x7E and that element a magnitude-6 code."""
    grid = golden_e2m1(golden_dir)[:8]
    rng = np.random.default_rng(11)
    rows, k = 6, 256
    x = _w4a4_rows(rng, rows, k)
    codes, scales, rs = oracle.act_quant_w4a4(x)
    nib = oracle.unpack_nibbles(codes)
    for r in range(rows):
        amax = np.max(np.abs(x[r]))
        assert rs[r] == np.float32(amax) / np.float32(2688.0)
        if rs[r] == 0:
            assert not scales[r].any() and not codes[r].any()
            continue
        y = x[r] / rs[r]                               # numpy f32 division
        for j in range(k // 16):
            yb = y[16 * j:16 * j + 16]
            m = np.max(np.abs(yb))
            assert scales[r, j] == torch_encode([m / np.float32(6.0)])[0], (r, j)
            S = np.float32(torch_e4m3([scales[r, j]])[0])
            qb = nib[r, 16 * j:16 * j + 16]
            if S == 0:
                assert not qb.any()
                continue
            t = (yb / S).astype(np.float64)
            d = np.abs(np.abs(t)[:, None] - grid[None, :])
            want = np.argmin(d, axis=1)
            tie = np.sort(d, axis=1)[:, 1] - np.sort(d, axis=1)[:, 0] == 0
            assert np.array_equal((qb & 7)[~tie], want[~tie]), (r, j)
        jmax = int(np.argmax(np.abs(x[r]))) // 16
        assert scales[r, jmax] == 0x7E
        assert nib[r, int(np.argmax(np.abs(x[r])))] & 7 == 7


def _w4a4_weights(rng, n, k):
    w = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    sc = torch_encode(np.exp2(rng.uniform(-3, 1, (n, k // 16))).astype(np.float32))
    return w, sc


def test_w4a4_gemm_ref_is_dequantised_matmul(golden_dir):
    """The reference equals a float64 matmul of the dequantised operands, each decoded
    here from the golden E2M1 grid and torch's e4m3 (not the oracle's decoders)."""
    table = golden_e2m1(golden_dir)
    rng = np.random.default_rng(12)
    g, n, k = 6, 24, 256
    x = _w4a4_rows(rng, g, k)
    codes, scales, rs = oracle.act_quant_w4a4(x)
    w, sc = _w4a4_weights(rng, n, k)
    s2 = np.float32(5.9945243e-5 * 64)
    out, absp = oracle.gemm_ref_w4a4(codes, scales, rs, w, sc, s2)
    xa = _dense_weights(codes, table) * np.repeat(torch_e4m3(scales), 16, axis=1) \
        * rs.astype(np.float64)[:, None]
    wd = _dense_weights(w, table) * np.repeat(torch_e4m3(sc), 16, axis=1) * float(s2)
    want = xa @ wd.T
    wabs = np.abs(xa) @ np.abs(wd).T
    assert np.all(np.abs(out - want) <= 1e-12 * wabs)
    assert np.allclose(absp, wabs, rtol=1e-12, atol=0)


def test_w4a4_gemm_ref_exact_rational(golden_dir):
    table = golden_e2m1(golden_dir)
    rng = np.random.default_rng(13)
    g, n, k = 2, 3, 64
    x = _w4a4_rows(rng, 6, k)[[0, 3]]
    codes, scales, rs = oracle.act_quant_w4a4(x)
    w, sc = _w4a4_weights(rng, n, k)
    s2 = np.float32(1 / 64)
    out, absp = oracle.gemm_ref_w4a4(codes, scales, rs, w, sc, s2)
    an = _dense_weights(codes, table)
    wn = _dense_weights(w, table)
    for r in range(g):
        for c in range(n):
            acc = Fraction(0)
            ab = Fraction(0)
            for kk in range(k):
                p = (Fraction(float(an[r, kk])) * Fraction(float(torch_e4m3([scales[r, kk // 16]])[0]))
                     * Fraction(float(wn[c, kk])) * Fraction(float(torch_e4m3([sc[c, kk // 16]])[0]))
                     * Fraction(float(rs[r])) * Fraction(float(s2)))
                acc += p
                ab += abs(p)
            assert abs(out[r, c] - float(acc)) <= k * 2.0 ** -52 * float(ab)
            assert abs(absp[r, c] - float(ab)) <= k * 2.0 ** -52 * float(ab)


def _dense_nvfp4(w, sc, s2, table):
    return _dense_weights(w, table) * np.repeat(torch_e4m3(sc), 16, axis=1) * float(s2)


def test_w4a4_informational_band_and_two_level_gain():
    """The section's arms on synthetic NVFP4 weights: uniform 0.1-scale activations stay in
    the informational band (rel < 0.2 against the unquantised activations), and on
    activations whose tokens span 1e-3..1e3 the two-level quantiser beats the sub-block
    one per token (the section's hard gate)."""
    table = np.array([oracle.e2m1_decode(i) for i in range(16)]).reshape(-1)
    rng = np.random.default_rng(14)
    n, k = 64, 512
    w, sc = _w4a4_weights(rng, n, k)
    s2 = np.float32(1 / 64)
    wd = _dense_nvfp4(w, sc, s2, table)
    x = (rng.uniform(-1, 1, (16, k)) * 0.1).astype(np.float32)
    cpu = x.astype(np.float64) @ wd.T
    c, s, r = oracle.act_quant_w4a4(x)
    out, _ = oracle.gemm_ref_w4a4(c, s, r, w, sc, s2)
    rel = oracle.max_rel(out, cpu)
    assert 0.0 < rel < 0.2, rel
    tokens = np.arange(16)
    dec = np.power(10.0, (tokens % 7) - 3).astype(np.float32)
    xd = (rng.uniform(-1, 1, (16, k)) * 0.1).astype(np.float32) * dec[:, None]
    cpu = xd.astype(np.float64) @ wd.T
    c, s, r = oracle.act_quant_w4a4(xd)
    two, _ = oracle.gemm_ref_w4a4(c, s, r, w, sc, s2)
    c1, s1 = oracle.act_quant_w4a4_v1(xd)
    one, _ = oracle.gemm_ref_w4a4(c1, s1, None, w, sc, s2)
    rel2, rel1 = oracle.per_token_rel(two, cpu), oracle.per_token_rel(one, cpu)
    assert rel2 < 0.2 and rel2 < rel1, (rel2, rel1)
    # the quiet tokens are where V1 fails: their micro-scales clamp and whole rows vanish
    assert rel1 > 0.5


def test_per_token_rel_closed_form():
    ref = np.array([[1.0, -2.0], [0.0, 0.0], [10.0, 5.0]])
    y = np.array([[1.5, -2.0], [3.0, 0.0], [10.0, 4.0]])
    assert oracle.per_token_rel(y, ref) == 0.25


def test_bound_checker_absolute_floor():
    """The gradual-underflow term: a one-ulp error in the subnormal range passes with the
    2^-149 floor and fails without it; an error above the floor still fails."""
    ref = np.array([2.0 ** -140, 1.0])
    absp = np.array([2.0 ** -140, 1.0])
    got = ref + np.array([2.0 ** -149, 0.0])
    assert not oracle.within_bound(got, ref, absp, 4.0)[0]
    assert oracle.within_bound(got, ref, absp, 4.0, 2.0 ** -149)[0]
    assert not oracle.within_bound(ref + np.array([2.0 ** -147, 0.0]), ref, absp, 4.0,
                                   2.0 ** -149)[0]


def test_pow2_scale_multiply_equals_divide_every_f32():
    """fn quant_rows forms the scale as pow2_ceil(amax * f32(1/448)); the plain statement of
    the method divides by 448. Over every f32 amax from the 1e-4 floor to 3e38 (about 1.18e9
    values, in chunks) the two give the same power of two, so either reading yields the
    same scales (and, the codes being x / s, the same codes)."""
    lo = int(np.array([1e-4], dtype=np.float32).view(np.uint32)[0])
    hi = int(np.array([3e38], dtype=np.float32).view(np.uint32)[0])
    inv = np.float32(1.0 / 448.0)
    d = np.float32(448.0)

    def p2c(t):
        b = t.view(np.uint32)
        m = b & np.uint32(0x007FFFFF)
        e = b & np.uint32(0x7F800000)
        return np.where(m == 0, b, e + np.uint32(0x00800000))

    step = 1 << 26
    for start in range(lo, hi + 1, step):
        bits = np.arange(start, min(start + step, hi + 1), dtype=np.uint32)
        a = bits.view(np.float32)
        same = p2c(a * inv) == p2c(a / d)
        assert same.all(), a[~same][:4]
