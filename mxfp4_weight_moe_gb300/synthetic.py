"""Seeded synthetic inputs for the MoE layer (harness code).

This module draws random numbers and packs them into the byte formats the
layer consumes.  It holds none of the layer's own arithmetic (no routing,
permutation, activation quantisation, GEMM, SwiGLU or combine); both the CUDA
path and the CPU oracle consume exactly the bytes it returns.

Recipes (sizes from the workloads the pages describe):
  * expert weights: W ~ N(0, 0.02) (0.02 read as the standard deviation),
    packed to MXFP4 the way a checkpoint converter would: per 32-element block
    along K the shared exponent floor(log2 amax) - 2 (OCP MX v1.0 rule; e2m1
    emax = 2), elements rounded to nearest-even on the e2m1 grid, saturating
    at +-6.  Expert e is drawn from its own generator (seed, e), so any
    subset of experts can be regenerated alone.
  * hidden: N(0, 1) rounded to bf16.
  * router logits: "normal" N(0,1); "hot_cold" N(0,1) with column 0 + 8 (every
    token picks it) and column E-1 - 8 (no token picks it); "zipf"
    ln p_pi(e) + Gumbel(0,1) with p_r ~ r^-1.1 and pi a seeded permutation
    (Gumbel top-k = sampling k experts without replacement ~ Zipf(1.1));
    "uniform" U[0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# e2m1 rounding thresholds between consecutive magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6
# and whether a value exactly on the threshold goes up (the upper code is even).
_E2M1_THRESHOLDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_E2M1_TIE_UP = (False, True, False, True, False, True, False)


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    logits: str
    seed: int = 0
    layers: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def S(self) -> int:
        return self.T * self.k


CONFIGS: dict[str, MoEConfig] = {
    # FlashInfer's official MXFP8 x MXFP4 test shape (T, H, E, k, I) = (1, 128, 2, 2, 128)
    "tiny": MoEConfig("tiny", T=1, H=128, E=2, k=2, I=128, logits="normal",
                      notes="w13 [2,256,128], w2 [2,128,128]; k = E so both experts are picked"),
    # token counts 1/2/8/32 with one always-picked and one never-picked expert
    "small_T1": MoEConfig("small_T1", T=1, H=1024, E=16, k=4, I=512, logits="hot_cold"),
    "small_T2": MoEConfig("small_T2", T=2, H=1024, E=16, k=4, I=512, logits="hot_cold"),
    "small_T8": MoEConfig("small_T8", T=8, H=1024, E=16, k=4, I=512, logits="hot_cold"),
    "small_T32": MoEConfig("small_T32", T=32, H=1024, E=16, k=4, I=512, logits="hot_cold"),
    # DeepSeek-V4-Flash-shaped layer (synthetic sizes), Zipf(1.1) expert skew
    "dsv4": MoEConfig("dsv4", T=4096, H=4096, E=256, k=6, I=2048, logits="zipf"),
    # Kimi-K3-shaped layer (SwiGLU in place of SiTU), uniform router logits
    "kimi_T16": MoEConfig("kimi_T16", T=16, H=7168, E=896, k=16, I=3584, logits="uniform"),
    "kimi_T8192": MoEConfig("kimi_T8192", T=8192, H=7168, E=896, k=16, I=3584, logits="uniform"),
    # profiling-sized Kimi-K3-shaped layers: 64 of the 896 experts, so that a
    # multi-pass ncu capture holds a few GB on the device; tiles as in
    # kimi_T16 (16 token rows) and kimi_T8192 (about 176 rows per chunk)
    "kimi_T16_e64": MoEConfig("kimi_T16_e64", T=16, H=7168, E=64, k=16, I=3584, logits="uniform"),
    "kimi_T2048_e64": MoEConfig("kimi_T2048_e64", T=2048, H=7168, E=64, k=16, I=3584, logits="uniform"),
    # layerwise prefill: 43 DSV4-shaped layers, layer l's logits use seed l
    "layerwise": MoEConfig("layerwise", T=16384, H=4096, E=256, k=6, I=2048, logits="zipf", layers=43),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def pack_mxfp4(W: torch.Tensor):
    """Pack float weights [..., K] (K % 32 == 0) into (fp4x2 [..., K/2], e8m0 [..., K/32]).

    Checkpoint-converter rule: per block exponent X = floor(log2 amax) - 2,
    clamped to [-127, 127] (all-zero block: -127); element = RNE(w * 2^-X) on
    the e2m1 grid, saturating at 6; element 2i in the low nibble of byte i."""
    *lead, K = W.shape
    assert K % 32 == 0
    Wb = W.float().reshape(*lead, K // 32, 32)
    amax = Wb.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)                      # amax = m * 2^ex, m in [0.5, 1)
    X = (ex.to(torch.int32) - 1 - 2)
    X = torch.where(amax > 0, X, torch.full_like(X, -127)).clamp(-127, 127)
    v = torch.ldexp(Wb, (-X).unsqueeze(-1).float())
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.uint8)
    for thr, up in zip(_E2M1_THRESHOLDS, _E2M1_TIE_UP):
        code += ((a > thr) | ((a == thr) & up)).to(torch.uint8)
    nib = code | (torch.signbit(v).to(torch.uint8) << 3)
    nib = nib.reshape(*lead, K)
    packed = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return packed.contiguous(), (X + 127).to(torch.uint8).contiguous()


def make_expert(e: int, H: int, I: int, seed: int, device="cpu", std: float = 0.02):
    """Expert e's (w13, w13_sf, w2, w2_sf): w13 [2I, H/2], w2 [H, I/2] + scales."""
    g = _gen(device, seed * 1_000_003 + 7919 * e + 1)
    w13f = torch.randn(2 * I, H, generator=g, device=device) * std
    w13, w13_sf = pack_mxfp4(w13f)
    del w13f
    w2f = torch.randn(H, I, generator=g, device=device) * std
    w2, w2_sf = pack_mxfp4(w2f)
    return w13, w13_sf, w2, w2_sf


def make_weights(E: int, H: int, I: int, seed: int = 0, device="cpu", std: float = 0.02):
    """All experts' packed weights: w13 [E,2I,H/2], w13_sf [E,2I,H/32], w2 [E,H,I/2], w2_sf [E,H,I/32]."""
    w13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
    w13_sf = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
    w2_sf = torch.empty(E, H, I // 32, dtype=torch.uint8, device=device)
    for e in range(E):
        a, b, c, d = make_expert(e, H, I, seed, device, std)
        w13[e].copy_(a)
        w13_sf[e].copy_(b)
        w2[e].copy_(c)
        w2_sf[e].copy_(d)
    return w13, w13_sf, w2, w2_sf


def make_hidden(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """bf16 [T, H] drawn from N(0, 1)."""
    g = _gen(device, seed * 7 + 3)
    return torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)


def make_logits(T: int, E: int, recipe: str, seed: int = 0, device="cpu") -> torch.Tensor:
    """f32 [T, E] router logits by recipe ("normal", "hot_cold", "zipf", "uniform")."""
    g = _gen(device, seed * 13 + 5)
    if recipe == "normal":
        return torch.randn(T, E, generator=g, device=device)
    if recipe == "hot_cold":
        lg = torch.randn(T, E, generator=g, device=device)
        lg[:, 0] += 8.0
        lg[:, E - 1] -= 8.0
        return lg
    if recipe == "uniform":
        return torch.rand(T, E, generator=g, device=device)
    if recipe == "zipf":
        r = torch.arange(1, E + 1, device=device, dtype=torch.float64)
        p = r.pow(-1.1)
        p = p / p.sum()
        pi = torch.randperm(E, generator=g, device=device)
        logp = torch.log(p)[pi].float()
        u = torch.rand(T, E, generator=g, device=device).clamp_(1e-12, 1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        return logp.unsqueeze(0) + gumbel
    raise ValueError(f"unknown logits recipe {recipe!r}")


def bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """uint16-compatible int16 view of a bf16 tensor (same bytes)."""
    assert x.dtype == torch.bfloat16
    return x.view(torch.int16)


def make_inputs(cfg: MoEConfig | str, device="cpu", seed: int | None = None, layer: int = 0,
                with_weights: bool = True):
    """hidden, logits and (optionally) packed weights for one layer of a config."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    s = cfg.seed if seed is None else seed
    out = {
        "cfg": cfg,
        "hidden": make_hidden(cfg.T, cfg.H, s, device),
        "logits": make_logits(cfg.T, cfg.E, cfg.logits, s + layer, device),
    }
    if with_weights:
        out["w13"], out["w13_sf"], out["w2"], out["w2_sf"] = make_weights(cfg.E, cfg.H, cfg.I, s + 1000 * layer,
                                                                          device)
    return out
