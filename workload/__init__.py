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
_P_WEIGHTS, _P_X, _P_ROUTE, _P_PERM, _P_DRAFT = 1, 2, 3, 4, 5


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


CONFIGS = {
    # 1 layer, H256/I128, 16 experts, top-2, S=4, 64 steps, N(0,1) + Zipf(1.1) bias
    "tiny": Config("tiny", 1, 256, 128, 16, 2, 4, 1, 64, 1.1, 0.0, 0, literal_normal_bias=True),
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
              seed: int, layer: int = 0) -> None:
    """Fill one layer's expert bank in place.

    Codes: uniform over all 16 nibbles (uniform random bytes).  Scales: uniform
    over the 16 E4M3 codes 0x30..0x3F (values 0.5 .. 1.875)."""
    bw, bs = storage_bytes(hidden, inter)
    assert w.size >= experts * bw and s.size >= experts * bs
    for e in range(experts):
        r = rng_for(seed, _P_WEIGHTS, layer, e)
        w[e * bw:(e + 1) * bw] = np.frombuffer(r.bytes(bw), np.uint8)
        sb = np.frombuffer(r.bytes(bs), np.uint8)
        s[e * bs:(e + 1) * bs] = 0x30 | (sb & 0x0F)


def global_scales(experts: int) -> np.ndarray:
    """fp32 (gate, up, down) global scales per expert: all 1/64."""
    return np.full((experts, 3), 1.0 / 64.0, np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def activations(seed: int, layer: int, steps: int, rows: int, hidden: int) -> np.ndarray:
    """bf16 bits [steps, rows, hidden] of N(0,1), fresh every step."""
    r = rng_for(seed, _P_X, layer)
    return to_bf16_bits(r.standard_normal((steps, rows, hidden), dtype=np.float32))


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
