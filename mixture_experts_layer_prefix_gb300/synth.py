"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

Nothing here computes any part of the MoE layer: it only draws numbers and
rounds them to the storage type. Every tensor is a deterministic function of
(seed, tensor name, expert index), so any expert's weights can be drawn alone
(the oracle checks large layers on sampled experts) and the same values reach
the GPU and the oracle.

Workloads follow the benchmark definitions of the 8- vs 128-expert top-4
study in "Introducing Olmo-core 3" (page 1 intro: pool grown from 8 to 128
experts with four chosen per token), with synthetic values:
  x ~ N(0, 1); dy ~ N(0, 1); w_gate, w_up ~ N(0, 1/d); w_down ~ N(0, 1/f);
  router w_r ~ N(0, 1/d) for the tiny fp32 layer, N(0, 0.02^2) otherwise.
Skewed routing adds a per-expert logit bias alpha * ln p_e with
p_e proportional to rank_e^-s over a seeded random ranking of the experts.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    dtype: str = "bf16"          # "f32" | "bf16" | "mxfp8"
    router_std: float | None = None   # None -> 1/sqrt(d)
    zipf_s: float | None = None       # per-expert logit bias exponent (None: no bias)
    zipf_alpha: float = 1.0
    n_dead: int = 0                   # experts pinned to a -1e4 bias (guaranteed empty)

    @property
    def R(self) -> int:
        return self.T * self.k


# alpha for the skewed 128-expert layer: chosen (bisection over alpha, routing
# computed by the fp64 oracle on these exact inputs) so that the 8 most loaded
# experts take about 40% of the T*k assignments. Recomputed by
# tests/golden/calibrate_skew.py, which calls only the oracle.
SKEW_ALPHA_E128 = 0.3537

CONFIGS = {
    "tiny_fp32": MoEShape("tiny_fp32", 512, 256, 8, 2, 512, "f32", None),
    "e8_top4": MoEShape("e8_top4", 16384, 2048, 8, 4, 1024, "bf16", 0.02),
    "e128_top4": MoEShape("e128_top4", 16384, 2048, 128, 4, 1024, "bf16", 0.02),
    "e128_top4_skew": MoEShape("e128_top4_skew", 16384, 2048, 128, 4, 1024, "bf16", 0.02,
                               zipf_s=1.2, zipf_alpha=SKEW_ALPHA_E128, n_dead=4),
    "e128_top4_mxfp8": MoEShape("e128_top4_mxfp8", 32768, 2048, 128, 4, 1024, "mxfp8", 0.02),
    "e128_top4_bf16_twin": MoEShape("e128_top4_bf16_twin", 32768, 2048, 128, 4, 1024, "bf16", 0.02),
    "stress_e256_top8": MoEShape("stress_e256_top8", 65536, 4096, 256, 8, 2048, "bf16", 0.02,
                                 zipf_s=1.0, zipf_alpha=1.0),
}


def shape(name: str, **over) -> MoEShape:
    return dataclasses.replace(CONFIGS[name], **over) if over else CONFIGS[name]


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) & np.uint32(0xFFFF0000)).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _rng(seed: int, name: str, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), zlib.crc32(name.encode()), int(sub)])


class Inputs:
    """Lazy, seeded inputs for one MoEShape. Values are float32 arrays that are
    exactly representable in the storage type (bf16-rounded unless f32)."""

    def __init__(self, s: MoEShape, seed: int = 0):
        self.s = s
        self.seed = seed
        self._cache = {}

    def _round(self, a):
        return a if self.s.dtype == "f32" else round_bf16(a)

    def _normal(self, name, shape_, std, sub=0):
        a = _rng(self.seed, name, sub).standard_normal(shape_, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return self._round(a)

    def _get(self, key, fn):
        if key not in self._cache:
            self._cache[key] = fn()
        return self._cache[key]

    def x(self):
        return self._get("x", lambda: self._normal("x", (self.s.T, self.s.d), 1.0))

    def dy(self):
        return self._get("dy", lambda: self._normal("dy", (self.s.T, self.s.d), 1.0))

    def w_r(self):
        std = self.s.router_std if self.s.router_std is not None else 1.0 / np.sqrt(self.s.d)
        return self._get("w_r", lambda: self._normal("w_r", (self.s.d, self.s.E), std))

    def w_gate_e(self, e):
        return self._normal("w_gate", (self.s.d, self.s.f), 1.0 / np.sqrt(self.s.d), e)

    def w_up_e(self, e):
        return self._normal("w_up", (self.s.d, self.s.f), 1.0 / np.sqrt(self.s.d), e)

    def w_down_e(self, e):
        return self._normal("w_down", (self.s.f, self.s.d), 1.0 / np.sqrt(self.s.f), e)

    def _stack(self, fn, experts=None):
        ex = range(self.s.E) if experts is None else experts
        return np.stack([fn(e) for e in ex])

    def w_gate(self, experts=None):
        return self._stack(self.w_gate_e, experts)

    def w_up(self, experts=None):
        return self._stack(self.w_up_e, experts)

    def w_down(self, experts=None):
        return self._stack(self.w_down_e, experts)

    def bias(self):
        """Per-expert fp32 logit bias, or None for unbiased routing."""
        s = self.s
        if s.zipf_s is None and s.n_dead == 0:
            return None

        def make():
            rng = _rng(self.seed, "bias_rank")
            rank = rng.permutation(s.E) + 1
            b = np.zeros(s.E, np.float32)
            if s.zipf_s is not None:
                p = rank.astype(np.float64) ** (-s.zipf_s)
                p /= p.sum()
                b = (s.zipf_alpha * np.log(p)).astype(np.float32)
                b -= b.max()
            if s.n_dead:
                dead = rng.choice(s.E, size=s.n_dead, replace=False)
                b[dead] = -1.0e4
            return b

        return self._get("bias", make)

    def for_experts(self, experts):
        """Stacked weights of a subset of experts (for sampled oracle checks)."""
        ex = list(experts)
        return dict(w_gate=self.w_gate(ex), w_up=self.w_up(ex), w_down=self.w_down(ex))
