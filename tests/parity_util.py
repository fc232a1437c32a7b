"""Helpers for the parity tests: run the CUDA path through the C ABI, run the oracle on
the same inputs, and compare under the stated error model."""
import json
import os

import numpy as np
import torch

import oracle
import block_scaled_fp4_act_gb300 as fp4


def to_np(t):
    return t.detach().cpu().numpy()


def gemm_bound(path, recipe, k):
    n_ops = fp4.fp4_error_ops(path, recipe, k)
    # The stated n_ops must come from a real summation structure, not a loose constant:
    # no more than one rounding per 16 products plus a fixed epilogue depth.
    assert 0 < n_ops <= 64 + k / 16, n_ops
    return n_ops


def page_n_ops(recipe, k):
    """n_ops of the pages' own kernel for this recipe and k: (gs-1) + ceil(groups/128) + 7
    (dsv4_native_gemm_gate.rs, the f64 check in main)."""
    gs = 16 if recipe == fp4.NVFP4 else 32
    return (gs - 1) + -(-(k // gs) // 128) + 7


def record_error(what, path, recipe, k, n_ops, worst, rel, count):
    """With FP4_ERR_REPORT set to a file name, append the worst |err| / (2^-24 sum|p|) seen
    by a parity check (its error in units of the error model's step), beside the stated
    n_ops of the path and the pages' own n_ops for the shape."""
    dest = os.environ.get("FP4_ERR_REPORT")
    if not dest:
        return
    rec = {"what": what, "path": int(path) if path is not None else None, "recipe": int(recipe),
           "k": int(k), "outputs": int(count), "n_ops": float(n_ops),
           "page_n_ops": page_n_ops(recipe, k), "worst_units": float(worst) * float(n_ops),
           "max_rel": float(rel)}
    with open(dest, "a") as f:
        f.write(json.dumps(rec) + "\n")


def check_gemm(gpu_out, ref, absp, n_ops, what=""):
    ok, worst, i = oracle.within_bound(gpu_out, ref, absp, n_ops)
    rel = oracle.max_rel(gpu_out, ref)
    g = np.asarray(gpu_out, dtype=np.float64).reshape(-1)
    r = np.asarray(ref).reshape(-1)
    assert ok, "%s: output %d gpu %r ref %r err/bound %.3g (n_ops %g)" % (
        what, i, g[i], r[i], worst, n_ops)
    assert rel <= 1e-3, "%s: max_rel %.3g" % (what, rel)
    return worst, rel


def expert_reference(x_np, w_np, sc_np, scale2, recipe):
    codes, scales = oracle.act_quant(x_np)
    out, absp = oracle.gemm_ref(codes, scales, w_np, sc_np, scale2, recipe)
    return codes, scales, out, absp


def sample_rows(offsets_np, P, rng, count):
    """Routed rows to check: each expert's first and last row, plus random ones."""
    picks = set()
    E = offsets_np.size - 1
    sizes = np.diff(offsets_np)
    for e in np.argsort(-sizes)[:8]:                       # hottest experts
        if sizes[e] > 0:
            picks.update([int(offsets_np[e]), int(offsets_np[e + 1] - 1)])
    nonempty = np.flatnonzero(sizes > 0)
    for e in rng.choice(nonempty, size=min(8, nonempty.size), replace=False):
        picks.update([int(offsets_np[e]), int(offsets_np[e + 1] - 1)])
    while len(picks) < min(count, P):
        picks.add(int(rng.integers(0, P)))
    return np.array(sorted(picks), dtype=np.int64)


def grouped_sampled_check(proj, out_gpu, path, rows, what):
    """Compare routed rows `rows` (all n columns) of a grouped call with the oracle."""
    x = to_np(proj.x)
    off = to_np(proj.routing.offsets).astype(np.int64)
    rid = to_np(proj.routing.row_ids).astype(np.int64) if proj.row_ids_used else None
    bank = proj.bank
    n, k = bank.n, bank.k
    out_np = to_np(out_gpu[torch.as_tensor(rows, device=out_gpu.device)])
    n_ops = gemm_bound(path, bank.recipe, k)
    worst_all, rel_refs, rel_gpu = 0.0, [], []
    experts = np.searchsorted(off, rows, side="right") - 1
    for e in np.unique(experts):
        sel = np.flatnonzero(experts == e)
        toks = rid[rows[sel]] if rid is not None else rows[sel]
        w = to_np(bank.w[int(e)])
        sc = to_np(bank.sc[int(e)])
        s2 = float(to_np(bank.scale2[int(e)]))
        _, _, ref, absp = expert_reference(x[toks], w, sc, s2, bank.recipe)
        worst, _ = check_gemm(out_np[sel], ref, absp, n_ops, "%s expert %d" % (what, e))
        worst_all = max(worst_all, worst)
        rel_refs.append(ref)
        rel_gpu.append(out_np[sel])
    rel = oracle.max_rel(np.concatenate([g.reshape(-1) for g in rel_gpu]),
                         np.concatenate([r.reshape(-1) for r in rel_refs]))
    assert rel <= 1e-3, (what, rel)
    record_error(what, path, bank.recipe, k, n_ops, worst_all, rel, len(rows) * n)
    return worst_all, rel


def run_projection(proj, workspace="auto"):
    """Run one grouped projection through the C ABI; returns (out, path)."""
    bank = proj.bank
    T, k = proj.x.shape
    P = proj.routing.P
    if workspace == "auto":
        workspace = fp4.workspace_for(T, P, bank.n, k, bank.recipe, device=proj.x.device)
    out = fp4.fp4_grouped_expert_gemm(proj.x, proj.routing.row_ids if proj.row_ids_used else None,
                                      proj.routing.offsets, bank.w, bank.sc, bank.scale2,
                                      bank.recipe, workspace=workspace)
    path = fp4.fp4_gemm_path(P, bank.E, bank.n, k, bank.recipe, workspace is not None)
    return out, path
