"""Seeded synthetic KV caches for speculative KV coding.

This module serves both the CUDA path and the oracle.  It draws inputs only:
true caches, predictor means mu, the per-channel sigma table and the
calibration histogram behind p-hat.  It holds none of the coder's arithmetic
(no rank, bin, CDF or rANS step).

The Qwen3 models and the C4 text behind the pages' measurements ("推测式 KV
编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding), section "早期结果"
(early results)) are not available, so seeded draws with the Qwen3 cache
shapes stand in for them:

* per-channel scale[l, kv, h, d] = exp(N(0, 1)), drawn once per workload with
  model seed 0; workloads marked ``outliers`` multiply 4 channels per
  (l, kv, h), picked by a seeded permutation, by 10;
* a draw with seed s: x = bf16(scale * N(0, 1)); residual r from
  0.95 N(0, sc^2) + 0.03 N(0, (3 sc)^2) + 0.02 Laplace(0, b = 20 sc) with
  sc = ``sigma_c`` * scale; mu = bf16(fp32(x) + r);
* sigma table: sc itself, or (``calibrated_sigma``) the RMS of x - mu over the
  calibration draws at (l, kv, h, d) granularity -- the page's optimum
  sigma^2 = E[(KV - mu)^2] from section "q 应是什么样的";
* p-hat counts: a histogram of the calibration draws' x by bf16 bit pattern
  (seed 1 for the tiny workload, seeds 1..128 of 512 tokens otherwise);
* e4m3 workloads: s = absmax|x| / 448 per (layer, head), x8 = e4m3(x / s)
  saturated to +-448, mu = bf16(fp32(mu) / s), sigma = sc / s;
* position-varying error scale (``drift`` > 0; the pages, section "下一步计划",
  note that sigma varies with prompt and position): sc is multiplied by
  exp(drift * W(t)) per (layer, kv, head), W a Brownian path over the tokens
  with Var W(T) = 1 (cumulative sums of N(0, 1/T)), drawn per seed, so the
  static sigma table sees only its average.

Torch is used as the random-number and array library on whatever device the
caller names; the bytes it produces are what both sides consume.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch

BF16, E4M3 = 0, 1


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    dtype: int
    L: int
    H: int
    T: int
    D: int
    sigma_c: float
    outliers: bool
    calib_draws: int
    calib_tokens: int          # 0: same T as the evaluation draw
    calibrated_sigma: bool
    Tb: int
    G: int
    drift: float = 0.0         # std of the log error scale's walk over the sequence

    @property
    def n(self) -> int:
        return self.L * 2 * self.H * self.T * self.D

    def scaled(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 2 x {K,V} x 2 heads x 256 tokens x 64: 131,072 scalars
    "tiny-bf16": Spec("tiny-bf16", BF16, 2, 2, 256, 64, 0.02, False, 1, 0, False, 256, 4),
    # Qwen3-0.6B-shaped: 28 x {K,V} x 8 x 4096 x 128 = 234.9M scalars
    "qwen3-0.6b-bf16": Spec("qwen3-0.6b-bf16", BF16, 28, 8, 4096, 128, 0.03, True, 128, 512,
                            False, 256, 16),
    # Qwen3-32B-shaped: 64 x {K,V} x 8 x 8192 x 128 = 1.07G scalars, calibrated sigma
    "qwen3-32b-bf16": Spec("qwen3-32b-bf16", BF16, 64, 8, 8192, 128, 0.015, True, 128, 512,
                           True, 256, 16),
    # Qwen3-8B-shaped FP8: 36 x {K,V} x 8 x 16384 x 128 = 1.21G e4m3 scalars
    "qwen3-8b-e4m3": Spec("qwen3-8b-e4m3", E4M3, 36, 8, 16384, 128, 0.03, True, 0, 512, False,
                          256, 8),
    # the Qwen3-0.6B shape as an FP8 cache: 234.9M e4m3 scalars, small enough for
    # a detailed profile of the e4m3 kernels (about 1.5 GB on the device); 16
    # lanes per chunk fill the GPU as the larger caches do
    "qwen3-0.6b-e4m3": Spec("qwen3-0.6b-e4m3", E4M3, 28, 8, 4096, 128, 0.03, True, 0, 512, False,
                            256, 16),
    # long-context FP8 stress: 64 x {K,V} x 8 x 32768 x 128 = 2^32 e4m3 scalars
    "long-32k-e4m3": Spec("long-32k-e4m3", E4M3, 64, 8, 32768, 128, 0.03, True, 0, 512, False,
                          128, 4),
    # the Qwen3-0.6B shape with an error scale that drifts along the sequence
    "qwen3-0.6b-bf16-drift": Spec("qwen3-0.6b-bf16-drift", BF16, 28, 8, 4096, 128, 0.03, True,
                                  128, 512, False, 256, 16, 1.0),
}


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def channel_scale(spec: Spec, device) -> torch.Tensor:
    """[L, 2, H, D] fp32 per-channel scale (model seed 0)."""
    g = _gen(device, spec.name, "scale", 0)
    scale = torch.exp(torch.randn(spec.L, 2, spec.H, spec.D, generator=g, device=device))
    if spec.outliers:
        go = _gen("cpu", spec.name, "outliers", 0)
        boost = torch.ones(spec.L * 2 * spec.H, spec.D)
        for row in range(spec.L * 2 * spec.H):
            idx = torch.randperm(spec.D, generator=go)[:4]
            boost[row, idx] = 10.0
        scale = scale * boost.view(spec.L, 2, spec.H, spec.D).to(device)
    return scale


def _draw_layer(spec: Spec, scale_l: torch.Tensor, seed: int, layer: int, T: int, device):
    """One layer of a draw: (x bf16, mu bf16), both [2, H, T, D]."""
    g = _gen(device, spec.name, "draw", seed, layer)
    shp = (2, spec.H, T, spec.D)
    s = scale_l[:, :, None, :]
    x = (s * torch.randn(shp, generator=g, device=device)).to(torch.bfloat16)
    sc = spec.sigma_c * s
    if spec.drift > 0:
        gd = _gen(device, spec.name, "drift", seed, layer)
        walk = torch.cumsum(torch.randn(2, spec.H, T, generator=gd, device=device), dim=2)
        sc = sc * torch.exp(spec.drift * walk / T ** 0.5)[..., None]
    u = torch.rand(shp, generator=g, device=device)
    n = torch.randn(shp, generator=g, device=device)
    e = torch.empty(shp, device=device).exponential_(1.0, generator=g)
    sgn = torch.where(torch.rand(shp, generator=g, device=device) < 0.5, -1.0, 1.0)
    r = torch.where(u < 0.95, sc * n, torch.where(u < 0.98, 3.0 * sc * n, 20.0 * sc * sgn * e))
    mu = (x.float() + r).to(torch.bfloat16)
    return x, mu


@dataclasses.dataclass
class Workload:
    spec: Spec
    kv: torch.Tensor         # [L,2,H,T,D] bfloat16 or uint8 (e4m3 codes)
    mu: torch.Tensor         # [L,2,H,T,D] bfloat16
    sigma: torch.Tensor      # [L,2,H,D] float32
    counts: torch.Tensor | None  # [65536] int64 histogram by bf16 pattern (bf16 only)
    fp8_scale: torch.Tensor | None = None  # [L, H] (e4m3 only)

    @property
    def n(self):
        return self.spec.n


def _calibrate(spec: Spec, scale: torch.Tensor, device):
    """Histogram of x by bf16 pattern and, optionally, RMS(x - mu) per channel."""
    counts = torch.zeros(65536, dtype=torch.int64, device=device)
    sq = torch.zeros(spec.L, 2, spec.H, spec.D, dtype=torch.float64, device=device)
    T = spec.calib_tokens or spec.T
    for d in range(1, spec.calib_draws + 1):
        for l in range(spec.L):
            x, mu = _draw_layer(spec, scale[l], d, l, T, device)
            pat = x.view(torch.int16).to(torch.int64) & 0xFFFF
            counts += torch.bincount(pat.reshape(-1), minlength=65536)
            if spec.calibrated_sigma:
                diff = x.double() - mu.double()
                sq[l] += (diff * diff).sum(dim=2)
    rms = None
    if spec.calibrated_sigma:
        rms = torch.sqrt(sq / (spec.calib_draws * T)).float()
    return counts, rms


def make(spec: Spec | str, device="cpu", seed: int = 0, layers=None) -> Workload:
    """Draw the evaluation cache (seed 0 by default) and its calibration tables.

    layers = (l0, l1): only layers l0 .. l1 - 1 of that cache, as a workload of
    l1 - l0 layers (what one rank holds when a cache is split by layers): the
    same bytes as those layers of the whole draw, with their rows of the sigma
    table; the calibration histogram is the whole cache's."""
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    device = torch.device(device)
    scale = channel_scale(spec, device)
    l0, l1 = layers if layers is not None else (0, spec.L)
    if not 0 <= l0 < l1 <= spec.L:
        raise ValueError("layer range %r outside 0..%d" % (layers, spec.L))
    part = spec if (l0, l1) == (0, spec.L) else spec.scaled(L=l1 - l0)
    shape = (l1 - l0, 2, spec.H, spec.T, spec.D)
    x = torch.empty(shape, dtype=torch.bfloat16, device=device)
    mu = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for l in range(l0, l1):
        x[l - l0], mu[l - l0] = _draw_layer(spec, scale[l], seed, l, spec.T, device)
    sigma_c = (spec.sigma_c * scale).float()
    if spec.dtype == BF16:
        counts, rms = _calibrate(spec, scale, device)
        sigma = rms if spec.calibrated_sigma else sigma_c
        return Workload(part, x, mu, sigma[l0:l1].contiguous(), counts)
    # e4m3: per-(layer, head) absmax / 448 scale shared by K and V
    s = x.float().abs().amax(dim=(1, 3, 4)) / 448.0          # [L, H]
    s = torch.where(s > 0, s, torch.ones_like(s))
    sb = s[:, None, :, None, None]
    x8 = (x.float() / sb).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    mu8 = (mu.float() / sb).to(torch.bfloat16)
    sigma = (sigma_c[l0:l1] / s[:, None, :, None]).float().contiguous()
    del x, mu
    return Workload(part, x8.contiguous(), mu8.contiguous(), sigma, None, s)


def to_numpy(w: Workload):
    """Host copies as raw bit patterns: (kv u16/u8, mu u16, sigma f32, counts u64|None)."""
    import numpy as np
    if w.spec.dtype == BF16:
        kv = w.kv.view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        kv = w.kv.cpu().numpy().view(np.uint8)
    mu = w.mu.view(torch.int16).cpu().numpy().view(np.uint16)
    sigma = w.sigma.cpu().numpy().astype(np.float32)
    counts = None if w.counts is None else w.counts.cpu().numpy().astype(np.uint64)
    return kv, mu, sigma, counts
