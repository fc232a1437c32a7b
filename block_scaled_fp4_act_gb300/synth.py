"""Seeded synthetic workloads for the quantized MoE expert projection.

Input generation only: this module holds none of the method's arithmetic (no
quantisation, no scale arithmetic, no GEMM). Both the CUDA path's tests/benchmark and
the CPU oracle's tests draw their inputs here. Random draws go through a
torch.Generator seeded per tensor family, on the device the tensors are made on (the
same seed gives different numbers on CPU and CUDA; each run is still reproducible).

Workloads (shapes and distributions):
  c1  single expert NVFP4: g=4, k=512, n=256; x ~ N(0,1); nibble bytes uniform 0..255;
      per-16 scale bytes = e4m3(2^u), u ~ U[-3,1] (torch's float8_e4m3fn conversion);
      scale2 = 1/64.
  c2  single expert MXFP4: g=16, k=2048, n=1024; x = 0.5 * Student-t(4); e8m0 scale
      bytes uniform in [122, 130].
  c3  decode: 64 NVFP4 experts, gate/up bank [n=2*1536, k=4096], down bank [n=4096,
      k=1536]; 8 tokens, top-8 distinct experts uniform; x ~ N(0,1), each element x50
      with probability 0.001; the down input is 64 routed rows of the same law.
  c4  prefill: 256 NVFP4 experts, gate/up [n=2048, k=7168], down [n=7168, k=2048];
      4096 tokens, top-8 without replacement, P(expert of rank r) ~ r^-1.1 over a seeded
      permutation; x = bf16-rounded N(0,1) (as f32); the down input is one row per
      routed pair, same law.
  c5  mixed: 128 NVFP4 + 128 MXFP4 experts, each [n=2048, k=4096]; per recipe 16384
      tokens, top-8 uniform; x ~ Student-t(3).
Seeds: weights 1000 + c, activations c, routing 2000 + c.
"""
from dataclasses import dataclass
from typing import Optional

import torch

NVFP4 = 0
MXFP4 = 1


def group_size(recipe: int) -> int:
    return 16 if recipe == NVFP4 else 32


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


@dataclass
class Bank:
    """One projection's expert bank: w [E,n,k/2] u8, sc [E,n,k/gs] u8, scale2 [E] f32."""
    recipe: int
    w: torch.Tensor
    sc: torch.Tensor
    scale2: torch.Tensor

    @property
    def E(self):
        return self.w.shape[0]

    @property
    def n(self):
        return self.w.shape[1]

    @property
    def k(self):
        return self.w.shape[2] * 2


@dataclass
class Routing:
    """CSR routing: routed row p reads token row_ids[p] and belongs to expert e with
    offsets[e] <= p < offsets[e+1]."""
    offsets: torch.Tensor  # [E+1] int32
    row_ids: torch.Tensor  # [P] int32

    @property
    def P(self):
        return int(self.row_ids.numel())


# ------------------------------------------------------------------ element draws

def nibble_bytes(shape, gen, device):
    return torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.uint8)


def nvfp4_scale_bytes(shape, gen, device, lo_exp=-3.0, hi_exp=1.0):
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.exp2(lo_exp + (hi_exp - lo_exp) * u)
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


def mxfp4_scale_bytes(shape, gen, device, lo=122, hi=130):
    return torch.randint(lo, hi + 1, shape, generator=gen, device=device, dtype=torch.uint8)


def normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def student_t(shape, nu: int, gen, device):
    """Z / sqrt(chi2_nu / nu), chi2 from nu squared standard normals."""
    z = normal(shape, gen, device)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2 += normal(shape, gen, device) ** 2
    return z / torch.sqrt(chi2 / nu)


def with_outliers(x, gen, p=0.001, factor=50.0):
    mask = torch.rand(x.shape, generator=gen, device=x.device) < p
    return torch.where(mask, x * factor, x)


def bf16_rounded(x):
    return x.to(torch.bfloat16).to(torch.float32)


# ------------------------------------------------------------------ banks and routing

def make_bank(recipe, E, n, k, seed, device, scale2_value=1.0 / 64.0):
    gen = _gen(seed, device)
    gs = group_size(recipe)
    w = nibble_bytes((E, n, k // 2), gen, device)
    if recipe == NVFP4:
        sc = nvfp4_scale_bytes((E, n, k // gs), gen, device)
        s2 = torch.full((E,), float(scale2_value), dtype=torch.float32, device=device)
    else:
        sc = mxfp4_scale_bytes((E, n, k // gs), gen, device)
        s2 = torch.zeros((E,), dtype=torch.float32, device=device)
    return Bank(recipe, w, sc, s2)


def routing_from_choices(choices: torch.Tensor, E: int) -> Routing:
    """choices [T, topk] expert ids -> CSR routing sorted by (expert, token)."""
    T, topk = choices.shape
    device = choices.device
    tokens = torch.arange(T, device=device, dtype=torch.int64).repeat_interleave(topk)
    experts = choices.reshape(-1).to(torch.int64)
    key = experts * T + tokens
    order = torch.argsort(key)
    row_ids = tokens[order].to(torch.int32)
    counts = torch.bincount(experts, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(counts, 0)
    return Routing(offsets.to(torch.int32), row_ids.contiguous())


def uniform_topk(T, E, topk, seed, device) -> Routing:
    gen = _gen(seed, device)
    keys = torch.rand((T, E), generator=gen, device=device)
    choices = torch.argsort(keys, dim=1)[:, :topk]
    return routing_from_choices(choices, E)


def zipf_topk(T, E, topk, seed, device, alpha=1.1) -> Routing:
    gen = _gen(seed, device)
    ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
    p_rank = ranks ** (-alpha)
    perm = torch.randperm(E, generator=gen, device=device)
    probs = torch.empty(E, device=device, dtype=torch.float64)
    probs[perm] = p_rank / p_rank.sum()
    choices = torch.multinomial(probs.float().expand(T, E).contiguous(), topk, replacement=False,
                                generator=gen)
    return routing_from_choices(choices, E)


# ------------------------------------------------------------------ workloads

@dataclass
class Projection:
    """One grouped call: x [T,k] f32, routing, bank, and the tokens' row mapping."""
    name: str
    x: torch.Tensor
    routing: Routing
    bank: Bank
    row_ids_used: bool = True


@dataclass
class Workload:
    name: str
    projections: list
    description: str = ""


def single_expert(cfg: int, device="cpu", g: Optional[int] = None, n: Optional[int] = None,
                  k: Optional[int] = None):
    """c1 (NVFP4) or c2 (MXFP4); returns (x [g,k], Bank with E=1)."""
    if cfg == 1:
        g, n, k = g or 4, n or 256, k or 512
        bank = make_bank(NVFP4, 1, n, k, 1000 + cfg, device)
        x = normal((g, k), _gen(cfg, device), device)
    elif cfg == 2:
        g, n, k = g or 16, n or 1024, k or 2048
        bank = make_bank(MXFP4, 1, n, k, 1000 + cfg, device)
        x = 0.5 * student_t((g, k), 4, _gen(cfg, device), device)
    else:
        raise ValueError(cfg)
    return x, bank


def decode_c3(device="cpu", E=64, T=8, topk=8, inter=1536, hidden=4096, scale2_value=1.0 / 64.0):
    gen_x = _gen(3, device)
    r = uniform_topk(T, E, topk, 2003, device)
    gu = make_bank(NVFP4, E, 2 * inter, hidden, 1003, device, scale2_value)
    dn = make_bank(NVFP4, E, hidden, inter, 1103, device, scale2_value)
    x = with_outliers(normal((T, hidden), gen_x, device), gen_x)
    h = with_outliers(normal((r.P, inter), gen_x, device), gen_x)
    ident = Routing(r.offsets, torch.arange(r.P, dtype=torch.int32, device=device))
    return Workload("c3_decode", [Projection("gate_up", x, r, gu),
                                  Projection("down", h, ident, dn, row_ids_used=False)],
                    "64 NVFP4 experts, 8 tokens top-8 uniform")


def prefill_c4(device="cpu", E=256, T=4096, topk=8, inter=2048, hidden=7168):
    gen_x = _gen(4, device)
    r = zipf_topk(T, E, topk, 2004, device)
    gu = make_bank(NVFP4, E, inter, hidden, 1004, device)
    dn = make_bank(NVFP4, E, hidden, inter, 1104, device)
    x = bf16_rounded(normal((T, hidden), gen_x, device))
    h = bf16_rounded(normal((r.P, inter), gen_x, device))
    ident = Routing(r.offsets, torch.arange(r.P, dtype=torch.int32, device=device))
    return Workload("c4_prefill", [Projection("gate_up", x, r, gu),
                                   Projection("down", h, ident, dn, row_ids_used=False)],
                    "256 NVFP4 experts, 4096 tokens top-8 Zipf(1.1)")


def mixed_c5(device="cpu", E=128, T=16384, topk=8, n=2048, k=4096):
    gen_x = _gen(5, device)
    projs = []
    for recipe, tag, off in ((NVFP4, "nvfp4", 0), (MXFP4, "mxfp4", 100)):
        r = uniform_topk(T, E, topk, 2005 + off, device)
        bank = make_bank(recipe, E, n, k, 1005 + off, device)
        x = student_t((T, k), 3, gen_x, device)
        projs.append(Projection(tag, x, r, bank))
    return Workload("c5_mixed", projs, "128 NVFP4 + 128 MXFP4 experts, 16384 tokens top-8")


def workload(name: str, device="cpu", **kw) -> Workload:
    if name in ("c3", "decode"):
        return decode_c3(device, **kw)
    if name in ("c4", "prefill"):
        return prefill_c4(device, **kw)
    if name in ("c5", "mixed"):
        return mixed_c5(device, **kw)
    raise ValueError(name)
