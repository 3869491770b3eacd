"""Seeded synthetic inputs for one sparse MoE layer.

This module only draws random numbers and prepares them in the library's
canonical layouts; it holds none of the layer's arithmetic (no routing, no
dispatch, no FFN). Both the CUDA path and the CPU oracle receive exactly the
tensors produced here.

Recipe (fixed so every run of every consumer sees the same bits):

* ``torch.Generator().manual_seed(seed)`` on the CPU, fp32 draws in the order
  x, W_r, b_r. Expert e = 0..E-1 has a generator of its own,
  ``manual_seed(expert_seed(seed, e))``, drawing W_gate[e], W_up[e], W_down[e]
  in that order; so the experts can be drawn in parallel threads and the bits
  do not depend on how many threads there are.
* x ~ N(0, 1); every weight ~ N(0, 0.02). Weights are drawn directly in the
  ``[out][in]`` layout (reduction index contiguous): W_r [E][d], gate/up
  [E][f][d], down [E][d][f].
* bf16 tensors are the fp32 draws rounded to nearest even.
* int4 g128 experts: per output row and per 128 consecutive reduction indices,
  s = bf16(max|w| / 7) and q = clamp(round_half_even(w / s), -7, 7) (q = 0 when
  s = 0), packed two's-complement, low nibble = even index; scales bf16
  [..][cols/128].
* MX experts (OCP Microscaling): per output row and per 32 consecutive
  reduction indices, the shared exponent is floor(log2(max|w|)) - emax with
  emax = 8 (E4M3) or 2 (E2M1); the scale byte is that exponent + 127 (E8M0;
  127 for an all-zero block); each element is w / 2^exponent rounded to
  nearest even in the element format and saturated at its largest normal
  (448, 6). E4M3 codes are bytes [..][cols]; E2M1 codes are nibbles packed
  two per byte, low nibble = even index; scales [..][cols/32].
* Router bias: none, or the skewed-routing rule
  b_e = alpha * ln p(rank(e)) with Zipf(s) popularity p(r) = r^-s / H over the
  ranks r = 1..E, the ranks assigned by a seeded permutation; alpha is the
  smallest value on a 0.05 grid for which the hottest expert takes >= 24% of
  the assignments and >= 3 experts receive none (found by a script that runs
  the oracle's router, stored in ``SKEWED_ALPHA``); or "hot0": +30 on expert 0.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import torch

F32, BF16, I4G128, MXFP8, MXFP4 = 0, 1, 2, 3, 4
DTYPE_CODE = {"f32": F32, "bf16": BF16, "i4g128": I4G128, "mxfp8": MXFP8, "mxfp4": MXFP4}
GROUP = 128
MX_BLOCK = 32
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)  # magnitudes of codes 0..7

# Zipf exponent and the bias scale chosen for the skewed-routing layer
# (T=16384, d=2048, E=64, k=4, seed 0).
ZIPF_S = 1.2
SKEWED_ALPHA = 1.1


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    act: str = "bf16"      # "f32" | "bf16"
    wdt: str = "bf16"      # "f32" | "bf16" | "i4g128" | "mxfp8" | "mxfp4"
    bias: str = "none"     # "none" | "zipf" | "hot0"
    alpha: float = SKEWED_ALPHA
    slots: int = 0         # handle option: experts kept in HBM (0 = all); the rest in host memory
    promotions: int = 0    # handle option: hot-set promotions per forward

    @property
    def act_code(self) -> int:
        return DTYPE_CODE[self.act]

    @property
    def w_code(self) -> int:
        return DTYPE_CODE[self.wdt]

    @property
    def n_assign(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEShape":
        return replace(self, **kw)


# The five workloads: a tiny fp32 layer; a Mixtral-8x7B-shaped layer at a
# decode batch and at prefill (8 sequences x 512 tokens); a fine-grained
# 256-expert layer with int4 experts; a skewed-routing stress layer. The
# others measure quantised experts (int4, MX) at decode and prefill batches
# and the residency tier.
CONFIGS = {
    "tiny_fp32": MoEShape("tiny_fp32", T=64, d=256, E=8, k=2, f=512, act="f32", wdt="f32"),
    "mixtral_decode": MoEShape("mixtral_decode", T=32, d=4096, E=8, k=2, f=14336),
    "mixtral_prefill": MoEShape("mixtral_prefill", T=4096, d=4096, E=8, k=2, f=14336),
    "fine_int4": MoEShape("fine_int4", T=256, d=6144, E=256, k=8, f=2048, wdt="i4g128"),
    "skewed": MoEShape("skewed", T=16384, d=2048, E=64, k=4, f=1408, bias="zipf"),
    # beside the five: the Mixtral-shaped prefill layer with int4 g128
    # experts (~1024 rows per expert), for the quantised tensor-core GEMM; and
    # the two decode layers with block-scaled (OCP MX) experts
    "mixtral_prefill_int4": MoEShape("mixtral_prefill_int4", T=4096, d=4096, E=8, k=2,
                                     f=14336, wdt="i4g128"),
    "mixtral_decode_mxfp8": MoEShape("mixtral_decode_mxfp8", T=32, d=4096, E=8, k=2, f=14336,
                                     wdt="mxfp8"),
    "fine_mxfp4": MoEShape("fine_mxfp4", T=256, d=6144, E=256, k=8, f=2048, wdt="mxfp4"),
    # the Mixtral-shaped prefill layer with MXFP8 experts (tensor-core GEMM
    # with the weights dequantised into tensor memory)
    "mixtral_prefill_mxfp8": MoEShape("mixtral_prefill_mxfp8", T=4096, d=4096, E=8, k=2,
                                      f=14336, wdt="mxfp8"),
    # the decode layer with its experts in host memory and 2 of 8 in HBM:
    # 6 active experts stream over NVLink-C2C every forward
    "mixtral_decode_tier": MoEShape("mixtral_decode_tier", T=32, d=4096, E=8, k=2, f=14336,
                                    slots=2, promotions=0),
}


def _cast(w: torch.Tensor, code: int) -> torch.Tensor:
    return w if code == F32 else w.to(torch.bfloat16)


def quantize_i4g128(w: torch.Tensor):
    """fp32 [rows][cols] -> (packed uint8 [rows][cols/2], bf16 scales [rows][cols/128])."""
    rows, cols = w.shape
    assert cols % GROUP == 0, "int4 groups need cols % 128 == 0"
    g = w.reshape(rows, cols // GROUP, GROUP)
    s = (g.abs().amax(dim=-1) / 7.0).to(torch.bfloat16)
    sf = s.float().unsqueeze(-1)
    q = torch.where(sf > 0, torch.round(g / torch.where(sf > 0, sf, torch.ones_like(sf))),
                    torch.zeros_like(g))
    q = q.clamp_(-7, 7).to(torch.int16).reshape(rows, cols)
    nib = (q & 0xF).to(torch.uint8)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return packed.contiguous(), s.contiguous()


def quantize_mx(w: torch.Tensor, fmt: str):
    """fp32 [rows][cols] -> (codes, E8M0 scales uint8 [rows][cols/32]) for
    fmt "mxfp8" (E4M3 bytes [rows][cols]) or "mxfp4" (E2M1 nibbles packed
    [rows][cols/2])."""
    rows, cols = w.shape
    assert cols % MX_BLOCK == 0, "MX blocks need cols % 32 == 0"
    g = w.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    amax = g.abs().amax(dim=-1)
    emax = 8 if fmt == "mxfp8" else 2
    _, ex = torch.frexp(amax)                      # amax = m * 2^ex, m in [0.5, 1)
    shared = torch.where(amax > 0, ex.to(torch.int32) - 1 - emax, torch.zeros_like(ex))
    shared = shared.clamp(-127, 127)
    scales = (shared + 127).to(torch.uint8)
    v = g / torch.pow(2.0, shared.to(torch.float32)).unsqueeze(-1)
    if fmt == "mxfp8":
        codes = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        return codes.reshape(rows, cols).contiguous(), scales.contiguous()
    a = v.abs().clamp(max=6.0).double()
    grid = torch.tensor(E2M1_GRID, dtype=torch.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    code = torch.bucketize(a, mids, right=False)   # a == mids[j] -> j (lower neighbour)
    tie = (code < 7) & (a == mids[code.clamp(max=6)]) & (code % 2 == 1)
    code = code + tie.to(code.dtype)               # ties go to the even code
    code = code.to(torch.uint8) | (torch.signbit(v).to(torch.uint8) << 3)
    code = code.reshape(rows, cols)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), scales.contiguous()


def zipf_bias(E: int, alpha: float, perm: torch.Tensor, s: float = ZIPF_S) -> torch.Tensor:
    """b_e = alpha * ln p(rank(e)), p Zipf(s) over ranks 1..E, rank(e) = perm[e] + 1."""
    h = sum(r ** -s for r in range(1, E + 1))
    logp = torch.tensor([math.log((r ** -s) / h) for r in range(1, E + 1)], dtype=torch.float64)
    return (alpha * logp[perm.long()]).to(torch.float32)


def expert_seed(seed: int, e: int) -> int:
    """Seed of expert e's own generator (distinct for e < 2^20)."""
    return (seed << 20) + 1 + e


def _draw_experts(E: int, seed: int, one):
    """one(e, generator) for every expert, in parallel threads (torch ops
    release the interpreter lock); each expert has its own seeded generator."""
    def job(e):
        one(e, torch.Generator().manual_seed(expert_seed(seed, e)))
    workers = max(1, min(E, os.cpu_count() or 1, 32))
    if workers == 1:
        for e in range(E):
            job(e)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(job, range(E)))


def make_layer(shape: MoEShape, seed: int = 0, experts: bool = True) -> dict:
    """All inputs of one layer as CPU tensors in the canonical layouts.

    Keys: x [T][d], w_router [E][d] (act dtype), b_router [E] f32 or None,
    w_gate/w_up [E][f][d], w_down [E][d][f] (f32/bf16, or int4 bytes
    [E][f][d/2] / [E][d][f/2]) and, for int4, s_gate/s_up [E][f][d/128] and
    s_down [E][d][f/128] (bf16). ``experts=False`` skips the expert weights.
    """
    T, d, E, f = shape.T, shape.d, shape.E, shape.f
    g = torch.Generator().manual_seed(seed)
    x = _cast(torch.randn(T, d, generator=g), shape.act_code)
    w_r = _cast(torch.randn(E, d, generator=g) * 0.02, shape.act_code)
    if shape.bias == "zipf":
        b_r = zipf_bias(E, shape.alpha, torch.randperm(E, generator=g))
    elif shape.bias == "hot0":
        b_r = torch.zeros(E, dtype=torch.float32)
        b_r[0] = 30.0
    else:
        b_r = None
    out = {"x": x, "w_router": w_r, "b_router": b_r}
    if not experts:
        return out
    if shape.wdt == "i4g128":
        assert d % GROUP == 0 and f % GROUP == 0
        wg = torch.empty(E, f, d // 2, dtype=torch.uint8)
        wu = torch.empty(E, f, d // 2, dtype=torch.uint8)
        wd = torch.empty(E, d, f // 2, dtype=torch.uint8)
        sg = torch.empty(E, f, d // GROUP, dtype=torch.bfloat16)
        su = torch.empty(E, f, d // GROUP, dtype=torch.bfloat16)
        sd = torch.empty(E, d, f // GROUP, dtype=torch.bfloat16)
        def one(e, ge):
            wg[e], sg[e] = quantize_i4g128(torch.randn(f, d, generator=ge) * 0.02)
            wu[e], su[e] = quantize_i4g128(torch.randn(f, d, generator=ge) * 0.02)
            wd[e], sd[e] = quantize_i4g128(torch.randn(d, f, generator=ge) * 0.02)
        _draw_experts(E, seed, one)
        out.update(w_gate=wg, w_up=wu, w_down=wd, s_gate=sg, s_up=su, s_down=sd)
    elif shape.wdt in ("mxfp8", "mxfp4"):
        assert d % MX_BLOCK == 0 and f % MX_BLOCK == 0
        bpe = 1 if shape.wdt == "mxfp8" else 2     # elements per byte
        wg = torch.empty(E, f, d // bpe, dtype=torch.uint8)
        wu = torch.empty(E, f, d // bpe, dtype=torch.uint8)
        wd = torch.empty(E, d, f // bpe, dtype=torch.uint8)
        sg = torch.empty(E, f, d // MX_BLOCK, dtype=torch.uint8)
        su = torch.empty(E, f, d // MX_BLOCK, dtype=torch.uint8)
        sd = torch.empty(E, d, f // MX_BLOCK, dtype=torch.uint8)

        def one(e, ge):
            wg[e], sg[e] = quantize_mx(torch.randn(f, d, generator=ge) * 0.02, shape.wdt)
            wu[e], su[e] = quantize_mx(torch.randn(f, d, generator=ge) * 0.02, shape.wdt)
            wd[e], sd[e] = quantize_mx(torch.randn(d, f, generator=ge) * 0.02, shape.wdt)
        _draw_experts(E, seed, one)
        out.update(w_gate=wg, w_up=wu, w_down=wd, s_gate=sg, s_up=su, s_down=sd)
    else:
        dt = torch.float32 if shape.w_code == F32 else torch.bfloat16
        wg = torch.empty(E, f, d, dtype=dt)
        wu = torch.empty(E, f, d, dtype=dt)
        wd = torch.empty(E, d, f, dtype=dt)
        def one(e, ge):
            wg[e] = torch.randn(f, d, generator=ge) * 0.02
            wu[e] = torch.randn(f, d, generator=ge) * 0.02
            wd[e] = torch.randn(d, f, generator=ge) * 0.02
        _draw_experts(E, seed, one)
        out.update(w_gate=wg, w_up=wu, w_down=wd, s_gate=None, s_up=None, s_down=None)
    return out


def random_assignments(T: int, E: int, k: int, seed: int = 0) -> torch.Tensor:
    """topk_idx [T][k] int32: k distinct experts per token, uniformly drawn."""
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def random_rows(n: int, d: int, act: int, seed: int = 0, scale: float = 1.0) -> torch.Tensor:
    """[n][d] ~ N(0, scale^2) in the act dtype (f32 or bf16)."""
    g = torch.Generator().manual_seed(seed)
    return _cast(torch.randn(n, d, generator=g) * scale, act)


def random_gates(T: int, k: int, seed: int = 0) -> torch.Tensor:
    """[T][k] positive f32 weights summing to one per token."""
    g = torch.Generator().manual_seed(seed)
    w = torch.rand(T, k, generator=g) + 0.05
    return (w / w.sum(dim=1, keepdim=True)).to(torch.float32)
