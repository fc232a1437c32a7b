"""Parity of the routing front-end (router, CSR construction, weighted combine) with the
oracle, through the C ABI.

The router's selected ids and their order must be exact (qwen4exp_gpu_gate.rs, device-
router arm); its weights are compared with the oracle's f64 softmax within a bound
derived from the f32 arithmetic: exp within 2 ulp, the rounding of (logit - max) which
moves exp by up to |logit - max| ulps, the f32 sums (E/32 sequential adds per lane and 5
shuffle levels, or topk terms when renormalising) and the division. The CSR layout must
equal the oracle's exactly; the combine must meet |y - f64| <= topk 2^-24 sum|terms| (one
f32 fma per slot).
"""
import numpy as np
import pytest
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import grouped_sampled_check, run_projection, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def built():
    fp4.build.build()
    fp4.lib()


def _logits(T, E, seed, ties=False):
    rng = np.random.default_rng(seed)
    if ties:
        x = rng.choice(np.linspace(-2, 2, 9), size=(T, E))
        x[0] = 0.75                      # all equal
        x[1] = -150.0
        x[1, E // 2] = 150.0             # everything else underflows in f32
        x[2, : E // 2] = 1.0             # a tie that straddles the top-k boundary
    else:
        x = rng.standard_normal((T, E)) * 2
    return x.astype(np.float32)


def _check_router(logits, topk, renorm):
    ids, w = fp4.fp4_route_topk(torch.as_tensor(logits).to(DEV), topk, renormalize=renorm)
    ids_ref, w_ref = oracle.route_topk(logits, topk, renormalize=renorm)
    bad = np.flatnonzero((to_np(ids) != ids_ref).any(axis=1))
    assert bad.size == 0, "token %d: gpu %s oracle %s" % (bad[0], to_np(ids)[bad[0]], ids_ref[bad[0]])
    E = logits.shape[1]
    span = (logits.max(axis=1) - logits.min(axis=1)).astype(np.float64)[:, None]
    rtol = (2.0 * span + E / 32.0 + topk + 16.0) * U
    err = np.abs(to_np(w).astype(np.float64) - w_ref)
    assert np.all(err <= rtol * w_ref + 1e-38), float(np.max(err / (rtol * w_ref + 1e-38)))
    return to_np(ids), to_np(w)


@pytest.mark.parametrize("T,E,topk,ties", [(4096, 256, 8, False), (777, 512, 10, True),
                                           (300, 64, 1, True), (64, 1024, 32, False),
                                           (50, 8, 8, True), (33, 40, 5, True)])
@pytest.mark.parametrize("renorm", [False, True])
def test_router_matches_oracle(T, E, topk, ties, renorm):
    _check_router(_logits(T, E, T + E + topk, ties), topk, renorm)


@pytest.mark.parametrize("T,E,topk", [(4096, 256, 8), (1, 4, 1), (37, 16, 3), (16384, 128, 8),
                                      (8, 64, 8), (1000, 1000, 2)])
def test_csr_matches_oracle(T, E, topk):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    if T > 10:
        ids[:, 0] = np.minimum(ids[:, 0], 3)  # a few hot experts, many empty ones
        for t in range(T):  # keep ids distinct within a token
            row = list(dict.fromkeys(ids[t].tolist()))
            spare = [e for e in range(E) if e not in row]
            ids[t] = row + spare[: topk - len(row)]
    off, rid, prow = fp4.fp4_route_csr(torch.as_tensor(ids).to(DEV), E)
    off_ref, rid_ref, prow_ref = oracle.route_csr(ids, E)
    assert np.array_equal(to_np(off), off_ref)
    assert np.array_equal(to_np(rid), rid_ref)
    assert np.array_equal(to_np(prow), prow_ref)
    assert fp4.fp4_get_device_error() == 0


def test_csr_flags_bad_ids():
    ids = torch.tensor([[0, 1], [2, 2], [1, 9]], dtype=torch.int32, device=DEV)
    fp4.fp4_route_csr(ids, 4)
    assert fp4.fp4_get_device_error() & fp4.FP4_DEVERR_EXPERT_ID
    assert fp4.fp4_get_device_error() == 0  # read and cleared
    off, rid, prow = fp4.fp4_route_csr(ids[:1], 4)
    assert to_np(off).tolist() == [0, 1, 2, 2, 2]


@pytest.mark.parametrize("T,topk,n", [(4096, 8, 2048), (5, 3, 4), (333, 2, 7168)])
def test_combine_matches_oracle(T, topk, n):
    rng = np.random.default_rng(T)
    P = T * topk
    out = rng.standard_normal((P, n)).astype(np.float32)
    prow = rng.permutation(P).reshape(T, topk).astype(np.int32)
    w = rng.random((T, topk)).astype(np.float32)
    y = fp4.fp4_moe_combine(torch.as_tensor(out).to(DEV), torch.as_tensor(prow).to(DEV),
                            torch.as_tensor(w).to(DEV))
    ref, absy = oracle.moe_combine(out, prow, w)
    ok, worst, i = oracle.within_bound(to_np(y), ref, absy, topk)
    assert ok, (worst, i)
    assert fp4.fp4_get_device_error() == 0


def test_routing_chain_around_a_grouped_projection():
    """logits -> router -> CSR -> grouped projection -> combine, each step checked against
    the oracle on the inputs it received."""
    T, E, topk, n, k = 512, 64, 8, 1024, 2048
    logits = _logits(T, E, 5)
    ids, w = _check_router(logits, topk, True)
    off, rid, prow = fp4.fp4_route_csr(torch.as_tensor(ids).to(DEV), E)
    off_ref, rid_ref, prow_ref = oracle.route_csr(ids, E)
    assert np.array_equal(to_np(off), off_ref) and np.array_equal(to_np(rid), rid_ref)
    bank = synth.make_bank(fp4.NVFP4, E, n, k, 55, DEV)
    x = torch.randn(T, k, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV)
    proj = synth.Projection("routed", x, synth.Routing(off, rid), bank)
    out, path = run_projection(proj)
    rows = np.unique(np.concatenate([prow_ref[:3].reshape(-1), prow_ref[-2:].reshape(-1)]))
    grouped_sampled_check(proj, out, path, rows, "routed projection")
    y = fp4.fp4_moe_combine(out, prow, torch.as_tensor(w).to(DEV))
    ref, absy = oracle.moe_combine(to_np(out), to_np(prow), w)
    ok, worst, i = oracle.within_bound(to_np(y), ref, absy, topk)
    assert ok, (worst, i)
    assert fp4.fp4_get_device_error() == 0
