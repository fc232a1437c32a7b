"""The bounded-wait abort path of both tensor-core GEMM kernels, made to run out on purpose.

The library's test hook (fp4_test_stall_next_gemm) makes the next tensor-core GEMM launch
withhold one pipeline arrival in its first CTA (a converter warp's "A stage full" on the
NVFP4 kernel, a scale-factor warp's "scale factors full" on the MXFP4 kernel; neither
guards an asynchronous copy) and bounds its waits by a short limit. That launch must
return, report FP4_DEVERR_TIMEOUT, and leave the context usable: the next, normal call
must match the oracle and report no error. The shape gives the first CTA two tiles, so the
abort also stops the MMA warp at a tile start.
"""
import time

import numpy as np
import pytest
import torch

import block_scaled_fp4_act_gb300 as fp4
from block_scaled_fp4_act_gb300 import synth
from parity_util import grouped_sampled_check, run_projection, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def force_tc():
    fp4.build.build()
    fp4.fp4_force_path(fp4.PATH_TC)
    yield
    fp4.fp4_test_stall_next_gemm(0)
    fp4.fp4_force_path(fp4.PATH_AUTO)


def _projection(recipe, E, rows, n, k, T, seed):
    gen = torch.Generator().manual_seed(seed)
    P = E * rows
    offsets = torch.arange(0, P + 1, rows, dtype=torch.int32)
    row_ids = torch.randint(0, T, (P,), generator=gen, dtype=torch.int32)
    bank = synth.make_bank(recipe, E, n, k, 950 + seed, "cpu")
    x = torch.randn(T, k, generator=gen)
    return synth.Projection("stall", x.to(DEV), synth.Routing(offsets.to(DEV), row_ids.to(DEV)),
                            synth.Bank(recipe, bank.w.to(DEV), bank.sc.to(DEV),
                                       bank.scale2.to(DEV)))


@pytest.mark.parametrize("recipe", [fp4.NVFP4, fp4.MXFP4])
def test_stalled_launch_times_out_and_the_next_call_is_correct(recipe):
    # 80 experts x 192 rows x 2 weight blocks = 160 tiles: more than one per SM
    proj = _projection(recipe, E=80, rows=192, n=256, k=512, T=2048, seed=recipe)
    assert fp4.fp4_get_device_error() == 0
    fp4.fp4_test_stall_next_gemm(20_000_000)  # about 10 ms of clock64 cycles
    t0 = time.perf_counter()
    _, path = run_projection(proj)
    bits = fp4.fp4_get_device_error()
    elapsed = time.perf_counter() - t0
    assert path == fp4.PATH_TC
    assert bits & fp4.FP4_DEVERR_TIMEOUT, bits
    assert bits == fp4.FP4_DEVERR_TIMEOUT, bits  # nothing else went wrong
    assert elapsed < 5.0, elapsed

    # the request was used once: the same call again runs normally and is correct
    out, path = run_projection(proj)
    assert fp4.fp4_get_device_error() == 0
    rng = np.random.default_rng(5)
    rows = sample_rows(proj.routing.offsets.cpu().numpy(), proj.routing.P, rng, 160)
    worst, rel = grouped_sampled_check(proj, out, path, rows, "after a stalled launch")
    print("recipe %d: stalled launch %.1f ms, then worst err/bound %.3g max_rel %.3g"
          % (recipe, elapsed * 1e3, worst, rel))
