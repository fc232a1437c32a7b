"""The W4A4 NVFP4 variant through the C ABI against the oracle (memra-engine 0.71.0,
src/bin/kernel_check.rs, the NVFP4 W4A4 MMQ GEMM section).

* act_quant_w4a4: codes, micro-scales and row scales bit for bit with the oracle's
  two-level quantiser (both sides take every rounding in f32 in the same order).
* fp4_grouped_expert_gemm_w4a4: every output (or a sample at full size) against the f64
  reference over the oracle's quantised activations and the NVFP4 weights, within
  fp4_w4a4_error_ops(k) * 2^-24 * sum|p| and max_rel <= 1e-3.
* The section's own arms, on synthetic NVFP4 weights: the informational band (rel < 0.2
  against the unquantised activations) and the dynamic-range gate (tokens spanning
  1e-3..1e3: the two-level GPU path beats the sub-block-only quantiser per token).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import record_error, sample_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def built():
    fp4.build.build()
    yield
    fp4.fp4_test_stall_next_gemm(0)


def _rows(rng, rows, k):
    x = rng.uniform(-1, 1, (rows, k)).astype(np.float32) * np.float32(0.1)
    if rows > 6:
        x[1] *= np.float32(1e-5)                          # a quiet token
        x[2, 16:48] = 0.0                                 # zero blocks
        x[3] = (rng.standard_t(3, k) * 10).astype(np.float32)
        x[4, ::37] *= 300.0                               # outlier channels
        x[5] = 0.0                                        # a zero row
        x[6] = np.float32(1e-40) * rng.standard_normal(k).astype(np.float32)  # subnormals
    return x


def _check_quant(x):
    codes, scales, rs = fp4.act_quant_w4a4(torch.as_tensor(x).to(DEV))
    oc, osc, ors = oracle.act_quant_w4a4(x)
    assert np.array_equal(to_np(rs).view(np.uint32), ors.view(np.uint32))
    assert np.array_equal(to_np(scales), osc)
    gc = to_np(codes)
    if not np.array_equal(gc, oc):
        bad = np.argwhere(gc != oc)[0]
        raise AssertionError("code byte %s: gpu %#x oracle %#x" % (bad, gc[tuple(bad)],
                                                                   oc[tuple(bad)]))


@pytest.mark.parametrize("rows,k", [(9, 32), (16, 48), (33, 2048), (12, 7168), (3, 16),
                                    (5, 512), (7, 1040), (4, 4096), (3, 8192), (2, 8720)])
def test_act_quant_w4a4_bit_exact(rows, k):
    """Bit-exact against the oracle on row lengths from one 16-group to past 8192, ragged
    against the CTA's 128 threads x 4 values and exact multiples of it."""
    rng = np.random.default_rng(rows * 131 + k)
    _check_quant(_rows(rng, rows, k))


def test_act_quant_w4a4_worked_examples_and_ties():
    """The golden examples' rows, and rows built on the E2M1 midpoints (every tie of the
    grid at several micro-scales), through the GPU quantiser."""
    rng = np.random.default_rng(7)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 0.0, -0.0, -0.25, -2.5,
                     -5.0, 1.0, 0.5], dtype=np.float32)
    rows = []
    for top in (2688.0, 448.0, 12.0, 1.0, 3e-3):
        r = np.tile(mids, 4) * np.float32(top / 6.0)
        r[0] = np.float32(top)                        # the row amax sets r
        rows.append(r.astype(np.float32))
    x = np.stack(rows)
    _check_quant(x)
    _check_quant(rng.uniform(-1, 1, (64, 256)).astype(np.float32) * np.float32(1e3))


def _bank_np(E, n, k, seed, s2=5.9945243e-5 * 64):
    b = synth.make_bank(fp4.NVFP4, E, n, k, seed, "cpu", scale2_value=s2)
    return b.w.numpy(), b.sc.numpy(), b.scale2.numpy()


def _run(x, row_ids, offsets, w, sc, s2):
    xd = torch.as_tensor(x).to(DEV)
    rid = None if row_ids is None else torch.as_tensor(row_ids, dtype=torch.int32).to(DEV)
    off = torch.as_tensor(offsets, dtype=torch.int32).to(DEV)
    out = fp4.fp4_grouped_expert_gemm_w4a4(xd, rid, off, torch.as_tensor(w).to(DEV),
                                           torch.as_tensor(sc).to(DEV),
                                           torch.as_tensor(s2).to(DEV))
    torch.cuda.synchronize()
    return to_np(out)


# The epilogue's two f32 multiplies (x r, x scale2) round into the subnormal range when r
# is tiny (rows of subnormal inputs): under gradual underflow each such rounding adds up to
# 2^-150 absolute on top of the relative model.
ABS_FLOOR = 2.0 ** -149


def _check_all(out, x, row_ids, offsets, w, sc, s2, what):
    k = x.shape[1]
    n_ops = fp4.fp4_w4a4_error_ops(k)
    codes, scales, rs = oracle.act_quant_w4a4(x)
    worst, rel_all, count = 0.0, 0.0, 0
    for e in range(offsets.size - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        src = np.arange(r0, r1) if row_ids is None else row_ids[r0:r1]
        ref, absp = oracle.gemm_ref_w4a4(codes[src], scales[src], rs[src], w[e], sc[e], s2[e])
        ok, wst, i = oracle.within_bound(out[r0:r1], ref, absp, n_ops, ABS_FLOOR)
        assert ok, "%s expert %d: output %d gpu %r ref %r err/bound %.3g" % (
            what, e, i, out[r0:r1].reshape(-1)[i], ref.reshape(-1)[i], wst)
        rel = oracle.max_rel(out[r0:r1], ref)
        assert rel <= 1e-3, (what, e, rel)
        worst, rel_all, count = max(worst, wst), max(rel_all, rel), count + ref.size
    record_error(what, None, fp4.NVFP4, k, n_ops, worst, rel_all, count)
    return worst, rel_all


@pytest.mark.parametrize("k,n", [(256, 128), (512, 200), (2048, 384), (7168, 256)])
def test_grouped_w4a4_every_output(k, n):
    """Ragged experts: empty ones, one- and 17-row ones, and ones spanning several 160-row
    tiles; n not a multiple of 128 in one case; repeated tokens through row ids."""
    rng = np.random.default_rng(k + n)
    sizes = np.array([0, 1, 17, 160, 161, 333, 0, 40])
    E = sizes.size
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    T = 300
    x = _rows(rng, T, k)
    row_ids = rng.integers(0, T, P).astype(np.int32)
    w, sc, s2 = _bank_np(E, n, k, 400 + k)
    out = _run(x, row_ids, offsets, w, sc, s2)
    worst, rel = _check_all(out, x, row_ids, offsets, w, sc, s2, "w4a4 k=%d n=%d" % (k, n))
    print("w4a4 k=%d n=%d: worst err/bound %.3g max_rel %.3g" % (k, n, worst, rel))


def test_grouped_w4a4_without_row_ids_and_zero_rows():
    rng = np.random.default_rng(5)
    k, n = 1024, 256
    sizes = np.array([70, 0, 90])
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    x = _rows(rng, P, k)
    x[100] = 0.0                                     # a zero row: r = 0, output exactly 0
    w, sc, s2 = _bank_np(3, n, k, 77)
    out = _run(x, None, offsets, w, sc, s2)
    assert not out[100].any()
    _check_all(out, x, None, offsets, w, sc, s2, "w4a4 no row ids")
    assert fp4.fp4_get_device_error() == 0


def test_grouped_w4a4_bad_row_id_gives_zero_row_and_error_bit():
    rng = np.random.default_rng(6)
    k, n, T = 512, 128, 40
    offsets = np.array([0, 30, 64], dtype=np.int32)
    row_ids = rng.integers(0, T, 64).astype(np.int32)
    row_ids[5] = T + 3                               # outside [0, T)
    x = _rows(rng, T, k)
    w, sc, s2 = _bank_np(2, n, k, 78)
    out = _run(x, row_ids, offsets, w, sc, s2)
    bits = fp4.fp4_get_device_error()
    assert bits == fp4.FP4_DEVERR_ROW_ID, bits
    assert not out[5].any()
    keep = np.ones(64, dtype=bool)
    keep[5] = False
    ok_ids = np.where(keep, row_ids, 0).astype(np.int32)
    codes, scales, rs = oracle.act_quant_w4a4(x)
    for e in range(2):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        ref, absp = oracle.gemm_ref_w4a4(codes[ok_ids[r0:r1]], scales[ok_ids[r0:r1]],
                                         rs[ok_ids[r0:r1]], w[e], sc[e], s2[e])
        m = keep[r0:r1]
        ok, wst, _ = oracle.within_bound(out[r0:r1][m], ref[m], absp[m],
                                         fp4.fp4_w4a4_error_ops(k), ABS_FLOOR)
        assert ok, wst


def test_grouped_w4a4_full_prefill_shape_sampled():
    """The prefill routing (256 experts, 4096 tokens top-8 Zipf(1.1)) on a gate and up bank
    of the layer body ([2 x 2048, 7168], k as the benchmark's gate/up projection, twice its
    n), in the launch configuration the benchmark uses; two runs bit-identical; sampled
    routed rows, the first and last weight block, against the oracle."""
    E, T, topk, n, k = 256, 4096, 8, 4096, 7168
    routing = synth.zipf_topk(T, E, topk, 1234, "cpu")
    gen = torch.Generator().manual_seed(99)
    x = (torch.rand(T, k, generator=gen) * 2 - 1) * 0.1
    bank = synth.make_bank(fp4.NVFP4, E, n, k, 4321, DEV, scale2_value=5.9945243e-5 * 64)
    call = lambda: fp4.fp4_grouped_expert_gemm_w4a4(x.to(DEV), routing.row_ids.to(DEV),
                                                    routing.offsets.to(DEV), bank.w, bank.sc,
                                                    bank.scale2)
    out = call()
    again = call()                                   # the same inputs: bit-identical outputs
    torch.cuda.synchronize()
    assert torch.equal(out, again)
    del again
    assert fp4.fp4_get_device_error() == 0
    offs = routing.offsets.numpy()
    rng = np.random.default_rng(3)
    rows = sample_rows(offs, routing.P, rng, 24)
    xn = x.numpy()
    rid = routing.row_ids.numpy()
    n_ops = fp4.fp4_w4a4_error_ops(k)
    cols = np.concatenate([np.arange(0, 128), np.arange(n - 128, n)])
    worst, rel_all = 0.0, 0.0
    for p in rows:
        e = int(np.searchsorted(offs, p, side="right") - 1)
        c, s, r = oracle.act_quant_w4a4(xn[rid[p]][None, :])
        w = to_np(bank.w[e])[cols]
        sc = to_np(bank.sc[e])[cols]
        ref, absp = oracle.gemm_ref_w4a4(c, s, r, w, sc, float(bank.scale2[e]))
        got = to_np(out[p])[cols][None, :]
        ok, wst, i = oracle.within_bound(got, ref, absp, n_ops)
        assert ok, (p, e, i, wst)
        worst, rel_all = max(worst, wst), max(rel_all, oracle.max_rel(got, ref))
    assert rel_all <= 1e-3
    record_error("w4a4 prefill shape sampled", None, fp4.NVFP4, k, n_ops, worst, rel_all,
                 rows.size * cols.size)
    print("w4a4 full shape: %d rows sampled, worst err/bound %.3g max_rel %.3g"
          % (rows.size, worst, rel_all))


def _dense_w(w, sc, s2):
    return oracle.dequant_w4a4(w, sc) * float(s2)


@pytest.mark.parametrize("T", [16, 128])
def test_w4a4_informational_band_and_dynamic_range_gate(T):
    """The section's arms on one synthetic NVFP4 expert (its gate weight stands in for the
    page's blk.0.ffn_gate): uniform 0.1-scale activations give rel < 0.2 against the
    unquantised activations; with token j scaled by 10^((j % 7) - 3) the GPU's two-level
    path has a lower per-token rel than the sub-block-only quantiser (the hard gate)."""
    k, n = 2048, 512
    rng = np.random.default_rng(T)
    w, sc, s2 = _bank_np(1, n, k, 555, s2=1 / 64)
    wd = _dense_w(w[0], sc[0], s2[0])
    offsets = np.array([0, T], dtype=np.int32)
    x = (rng.uniform(-1, 1, (T, k)) * 0.1).astype(np.float32)
    out = _run(x, None, offsets, w, sc, s2)
    rel = oracle.max_rel(out, x.astype(np.float64) @ wd.T)
    assert rel < 0.2, rel
    dec = np.power(10.0, (np.arange(T) % 7) - 3).astype(np.float32)
    xd = (rng.uniform(-1, 1, (T, k)) * 0.1).astype(np.float32) * dec[:, None]
    cpu = xd.astype(np.float64) @ wd.T
    out = _run(xd, None, offsets, w, sc, s2)
    c1, s1 = oracle.act_quant_w4a4_v1(xd)
    v1, _ = oracle.gemm_ref_w4a4(c1, s1, None, w[0], sc[0], s2[0])
    rel2, rel1 = oracle.per_token_rel(out, cpu), oracle.per_token_rel(v1, cpu)
    assert rel2 < rel1, (rel2, rel1)
    print("W4A4 T=%d: rel %.3e (band 0.2); dynamic range per-token rel %.3e vs sub-block only "
          "%.3e" % (T, rel, rel2, rel1))


def test_w4a4_stalled_launch_times_out_and_the_next_call_is_correct():
    """The bounded-wait abort path of the W4A4 kernel (the test hook withholds one
    scale-factor arrival of CTA 0); the next call is normal and correct."""
    rng = np.random.default_rng(8)
    E, rows, n, k, T = 80, 160, 256, 512, 1024
    offsets = np.arange(0, E * rows + 1, rows).astype(np.int32)
    row_ids = rng.integers(0, T, E * rows).astype(np.int32)
    x = _rows(rng, T, k)
    w, sc, s2 = _bank_np(E, n, k, 88)
    assert fp4.fp4_get_device_error() == 0
    fp4.fp4_test_stall_next_gemm(20_000_000)
    t0 = time.perf_counter()
    _run(x, row_ids, offsets, w, sc, s2)
    bits = fp4.fp4_get_device_error()
    elapsed = time.perf_counter() - t0
    assert bits == fp4.FP4_DEVERR_TIMEOUT, bits
    assert elapsed < 5.0, elapsed
    out = _run(x, row_ids, offsets, w, sc, s2)
    assert fp4.fp4_get_device_error() == 0
    sub = offsets[:5]
    _check_all(out[:int(sub[-1])], x, row_ids[:int(sub[-1])], sub, w, sc, s2,
               "w4a4 after a stalled launch")


def test_grouped_w4a4_expert_limit():
    """1024 experts (the kernel's limit: its tile prefix lives in shared memory), most empty,
    a few with rows; 1025 experts are refused on the host."""
    rng = np.random.default_rng(9)
    E, n, k, T = 1024, 128, 256, 64
    sizes = np.zeros(E, dtype=np.int64)
    hot = rng.choice(E, 40, replace=False)
    sizes[hot] = rng.integers(1, 9, 40)
    sizes[E - 1] = 3                                   # the last expert has rows
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    row_ids = rng.integers(0, T, P).astype(np.int32)
    x = _rows(rng, T, k)
    w = rng.integers(0, 256, (E, n, k // 2), dtype=np.uint8)
    sc = torch.exp2(torch.empty(E, n, k // 16).uniform_(-3, 1)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()
    s2 = np.full(E, 1 / 64, dtype=np.float32)
    out = _run(x, row_ids, offsets, w, sc, s2)
    assert fp4.fp4_get_device_error() == 0
    _check_all(out, x, row_ids, offsets, w, sc, s2, "w4a4 1024 experts")
    off = torch.as_tensor(np.concatenate([offsets, [P]]).astype(np.int32)).to(DEV)
    wd = torch.as_tensor(np.concatenate([w, w[:1]])).to(DEV)
    scd = torch.as_tensor(np.concatenate([sc, sc[:1]])).to(DEV)
    with pytest.raises(fp4.Fp4Error, match="FP4_ERR_SHAPE"):
        fp4.fp4_grouped_expert_gemm_w4a4(torch.as_tensor(x).to(DEV),
                                         torch.as_tensor(row_ids).to(DEV), off, wd, scd,
                                         torch.ones(E + 1, device=DEV))
