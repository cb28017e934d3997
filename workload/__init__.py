"""Seeded synthetic inputs for the slot-cache MoE layer.

This module holds input generation only: random expert banks in the NVFP4
storage layout, bf16 activations and router logits with the routing statistics
the pages describe.  It contains none of the method's arithmetic (no routing,
no dequantisation, no cache logic) and imports neither the CUDA library nor the
oracle, so both can be fed from it.

Routing model (the pages' frozen routing trace is not available, so this
stands in for it): expert popularity is Zipf(s) over a seeded permutation of
the experts, and step t's logits are
    l_t[e] = -s * ln(rank_e) + n_t[e],   n_t = rho * n_{t-1} + sqrt(1 - rho^2) * G_t,
with G_t iid standard Gumbel.  The first term is log-popularity and the
Gumbel noise makes top-k a draw without replacement from the Zipf law; rho
controls how many experts consecutive steps share ("GB300 GLM 5.3 Testing",
trace analysis: step-to-step overlap 0.27, cross-layer overlap at chance).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# purposes for independent random streams
_P_WEIGHTS, _P_X, _P_ROUTE, _P_PERM, _P_DRAFT, _P_GSCALE, _P_XWIDE = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    layers: int
    hidden: int
    inter: int
    experts: int
    top_k: int
    slots: int
    rows: int
    steps: int
    zipf_s: float
    rho: float
    seed: int
    literal_normal_bias: bool = False  # logits = N(0,1) + ln-Zipf bias, iid per step
    streams: int = 1                   # multi-row rounds: streams x (1 + drafts)
    drafts: int = 0
    draft_shared: int = 0              # ids a draft row keeps from its stream's row 0
    # scales: "literal" = block scales from the 16 E4M3 codes 0x30..0x3F and every
    # global scale 1/64 (the tiny configuration as stated); "wide" = block scales
    # over every finite positive E4M3 code 0x01..0x7E (subnormals included) and a
    # distinct seeded global scale per (expert, matrix)
    scales: str = "wide"


CONFIGS = {
    # 1 layer, H256/I128, 16 experts, top-2, S=4, 64 steps, N(0,1) + Zipf(1.1) bias
    "tiny": Config("tiny", 1, 256, 128, 16, 2, 4, 1, 64, 1.1, 0.0, 0, literal_normal_bias=True,
                   scales="literal"),
    # the same layer with wide block scales and per-(expert, matrix) global scales
    "tiny_wide": Config("tiny_wide", 1, 256, 128, 16, 2, 4, 1, 64, 1.1, 0.0, 5,
                        literal_normal_bias=True),
    # a small layer whose dimensions are multiples of 256 (the grouped MMA's TMA
    # tiles): H512/I256, 16 experts, top-4, S=8, wide scales
    "small": Config("small", 1, 512, 256, 16, 4, 8, 1, 64, 1.1, 0.0, 9,
                    literal_normal_bias=True),
    # the same with one 256-element chunk of K for gate/up and a 4-chunk down pass
    # (H256/I1024, top-2, S=4), and with the hidden size 1024 (H1024/I256, top-4, S=8)
    "small_wide_i": Config("small_wide_i", 1, 256, 1024, 16, 2, 4, 1, 64, 1.1, 0.0, 10,
                           literal_normal_bias=True),
    "small_wide_h": Config("small_wide_h", 1, 1024, 256, 16, 4, 8, 1, 64, 1.1, 0.0, 11,
                           literal_normal_bias=True),
    # GLM-5.3-shaped layer: H6144/I2048, 256 experts, top-8, S=128, M=1, 300 churn steps
    "glm": Config("glm", 1, 6144, 2048, 256, 8, 128, 1, 300, 1.1, 0.1, 1),
    # Flash-shaped stack: 16 layers, H4096/I2048, 288 experts top-8, S=54, 512 steps
    "flash": Config("flash", 16, 4096, 2048, 288, 8, 54, 1, 512, 1.05, 0.1, 2),
    # multi-row rounds: GLM shape, 16 layers, S=128, M=16 = 4 streams x (1 + 3 drafts)
    "multirow": Config("multirow", 16, 6144, 2048, 256, 8, 128, 16, 256, 1.1, 0.1, 3,
                       streams=4, drafts=3, draft_shared=4),
    # prefill bypass (M=512) then an S sweep at M=1: GLM shape, 8 layers
    "prefill": Config("prefill", 8, 6144, 2048, 256, 8, 128, 512, 300, 1.1, 0.1, 4),
}
SWEEP_SLOTS = (32, 64, 128, 192)


def storage_bytes(hidden: int, inter: int) -> tuple[int, int]:
    """Bytes of one expert's codes and scales in the storage layout (3 matrices of
    hidden*inter 4-bit codes, one 8-bit scale per 16 codes)."""
    n = 3 * hidden * inter
    return n // 2, n // 16


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, *stream])


def fill_bank(w: np.ndarray, s: np.ndarray, experts: int, hidden: int, inter: int,
              seed: int, layer: int = 0, scales: str = "literal") -> None:
    """Fill one layer's expert bank in place.

    Codes: uniform over all 16 nibbles (uniform random bytes).  Scales
    ("literal"): uniform over the 16 E4M3 codes 0x30..0x3F (values 0.5 ..
    1.875); ("wide"): uniform over the 126 finite positive E4M3 codes
    0x01..0x7E (2^-9 .. 448, subnormals included)."""
    bw, bs = storage_bytes(hidden, inter)
    assert w.size >= experts * bw and s.size >= experts * bs
    assert scales in ("literal", "wide")
    for e in range(experts):
        r = rng_for(seed, _P_WEIGHTS, layer, e)
        w[e * bw:(e + 1) * bw] = np.frombuffer(r.bytes(bw), np.uint8)
        sb = np.frombuffer(r.bytes(bs), np.uint8)
        if scales == "literal":
            s[e * bs:(e + 1) * bs] = 0x30 | (sb & 0x0F)
        else:
            # 0x01 + (16-bit draw mod 126): the bias of the modulus is below 2e-3
            u = np.frombuffer(r.bytes(2 * bs), np.uint16)
            s[e * bs:(e + 1) * bs] = (1 + u % 126).astype(np.uint8)


def global_scales(experts: int, scales: str = "literal", seed: int = 0,
                  layer: int = 0) -> np.ndarray:
    """fp32 (gate, up, down) global scales per expert.  "literal": all 1/64.
    "wide": 2^(j - 13) * (1 + u) per (expert, matrix), j uniform in {-1, 0, 1}
    and u uniform in [0, 1), so the three matrices of an expert, and the
    experts, all differ; 2^-13 * 1.5 offsets the wide block scales' larger
    magnitude (RMS ~100 against ~1.16 for the literal codes), keeping the
    layer's outputs near the literal configuration's scale."""
    if scales == "literal":
        return np.full((experts, 3), 1.0 / 64.0, np.float32)
    assert scales == "wide"
    r = rng_for(seed, _P_GSCALE, layer)
    j = r.integers(-1, 2, size=(experts, 3))
    u = r.random((experts, 3))
    return (np.ldexp(1.0 + u, j - 13)).astype(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def activations(seed: int, layer: int, steps: int, rows: int, hidden: int) -> np.ndarray:
    """bf16 bits [steps, rows, hidden] of N(0,1), fresh every step."""
    r = rng_for(seed, _P_X, layer)
    return to_bf16_bits(r.standard_normal((steps, rows, hidden), dtype=np.float32))


def activations_wide(seed: int, layer: int, steps: int, rows: int, hidden: int) -> np.ndarray:
    """bf16 bits [steps, rows, hidden]: N(0,1) with, in every row, 4 elements of
    magnitude U(1e3, 4e3), 2 of magnitude U(3.3e4, 6e4) (above the f16 range's
    half, so a kernel that holds x in f16 must rescale the row) and 4 of
    magnitude U(1e-6, 1e-5) (below f16's normal range), random signs and
    positions."""
    r = rng_for(seed, _P_XWIDE, layer)
    a = r.standard_normal((steps, rows, hidden), dtype=np.float32)
    for t in range(steps):
        for m in range(rows):
            pos = r.choice(hidden, size=10, replace=False)
            mag = np.concatenate([r.uniform(1e3, 4e3, 4), r.uniform(3.3e4, 6e4, 2),
                                  r.uniform(1e-6, 1e-5, 4)])
            a[t, m, pos] = (mag * r.choice([-1.0, 1.0], size=10)).astype(np.float32)
    return to_bf16_bits(a)


class Routing:
    """Router logits for one layer: Zipf popularity + AR(1) Gumbel noise."""

    def __init__(self, cfg: Config, layer: int = 0):
        self.cfg = cfg
        E = cfg.experts
        perm = rng_for(cfg.seed, _P_PERM, layer).permutation(E)
        rank = np.empty(E, np.float64)
        rank[perm] = np.arange(1, E + 1)
        self.bias = -cfg.zipf_s * np.log(rank)
        self.rng = rng_for(cfg.seed, _P_ROUTE, layer)
        self.draft_rng = rng_for(cfg.seed, _P_DRAFT, layer)
        self.noise = None

    def _gumbel(self, shape, rng=None) -> np.ndarray:
        rng = self.rng if rng is None else rng
        return rng.gumbel(size=shape)

    def step(self, rows: int | None = None) -> np.ndarray:
        """Logits fp32 [rows, E] for the next step."""
        c = self.cfg
        M = c.rows if rows is None else rows
        E = c.experts
        if c.literal_normal_bias:
            return (self.bias + self.rng.standard_normal((M, E))).astype(np.float32)
        if c.streams > 1 and M == c.streams * (1 + c.drafts):
            return self._round()
        if self.noise is None or self.noise.shape != (M, E):
            self.noise = self._gumbel((M, E))
        else:
            self.noise = c.rho * self.noise + math.sqrt(1 - c.rho ** 2) * self._gumbel((M, E))
        return (self.bias + self.noise).astype(np.float32)

    def _round(self) -> np.ndarray:
        """One multi-row round: each stream's row 0 follows the AR process; each of
        its draft rows keeps `draft_shared` of row 0's top-k ids (forced to the top
        of the draft's logits) and fills the rest from a fresh draw."""
        c = self.cfg
        E, k = c.experts, c.top_k
        if self.noise is None or self.noise.shape != (c.streams, E):
            self.noise = self._gumbel((c.streams, E))
        else:
            self.noise = c.rho * self.noise + math.sqrt(1 - c.rho ** 2) * self._gumbel((c.streams, E))
        base = self.bias + self.noise
        out = np.empty((c.streams * (1 + c.drafts), E), np.float64)
        for st in range(c.streams):
            r0 = st * (1 + c.drafts)
            out[r0] = base[st]
            top = np.argsort(-base[st], kind="stable")[:k]
            for d in range(1, 1 + c.drafts):
                fresh = self.bias + self._gumbel(E, self.draft_rng)
                keep = self.draft_rng.choice(top, size=c.draft_shared, replace=False)
                fresh[keep] = fresh.max() + 50.0 + np.arange(c.draft_shared)
                out[r0 + d] = fresh
        return out.astype(np.float32)


def prefill_logits(cfg: Config, layer: int, rows: int) -> np.ndarray:
    """Prefill chunk: every token's logits drawn independently (bias + Gumbel)."""
    rt = Routing(cfg, layer)
    return (rt.bias + rt._gumbel((rows, cfg.experts))).astype(np.float32)
