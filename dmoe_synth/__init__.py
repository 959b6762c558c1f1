"""Seeded synthetic inputs for the dropless MoE block.

This module is shared by the CPU oracle, the CUDA path's tests and the
benchmark.  It holds none of the method's arithmetic: it only draws random
numbers, shapes them into the five workloads and encodes them as bf16 / fp32,
exactly as both sides consume them.

Workloads (all dimensions in elements):

=========  =====  =====  ===  =====  ===  ======  =======  =========================
name       T      d      E    F      k    act     renorm   routing logits
=========  =====  =====  ===  =====  ===  ======  =======  =========================
tiny       512    256    4    512    1    gelu    no       N(0,1)
moe_xs     8192   512    64   2048   1    gelu    no       N(0,1)
skewed     16384  1024   64   4096   1    gelu    no       N(0,1) + 8 on a Zipf draw
mixtral    8192   4096   8    14336  2    swiglu  yes      N(0,1)
fine       4096   3584   64   2560   8    swiglu  no       N(0,1)
=========  =====  =====  ===  =====  ===  ======  =======  =========================

T tokens, d model width, E experts, F hidden width of one expert, k experts
per token.  Weights follow the per-expert layer of the MegaBlocks section of
George Lin's blog post on MoE training (section 1.2: expert i has
W_i^1 in R^{d x F}); all experts are stored side by side:

* ``w1``, ``w3``: bf16 ``[d, E*F]`` (expert e owns columns e*F .. e*F+F-1)
* ``w2``: bf16 ``[E*F, d]`` (expert e owns rows e*F .. e*F+F-1)

Value distributions: ``tiny`` draws x and all weights from N(0, 0.02) as its
description fixes.  The other workloads state none, so they use unit-scale
activations and fan-in scaled weights (x ~ N(0,1), W1/W3 ~ N(0, 1/d),
W2 ~ N(0, 1/F)) which keep every intermediate O(1).  The upstream gradient
``dy`` is N(0,1) everywhere.

The skewed workload draws each token's expert from a Zipf law (exponent
1.254 over 62 live ranks, mapped to experts by a seeded permutation; the
two remaining experts receive no token), then adds +8 to that expert's
logit.  The top-10 experts then receive about 75% of the tokens, the load
skew FlexMoE reports for a 64-expert GPT-MoE (same post, section 2.1).

bf16 tensors are returned as ``numpy.uint16`` bit patterns (round to nearest
even from fp32).  Each tensor comes from its own PCG64 stream keyed by
``(seed, stream id)``, so any subset can be generated independently.
"""

from __future__ import annotations

import dataclasses
import numpy as np

BLOCK = 128

STREAM_LOGITS = 1
STREAM_X = 2
STREAM_W1 = 3
STREAM_W3 = 4
STREAM_W2 = 5
STREAM_DY = 6
STREAM_ROUTE = 7


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    d: int
    E: int
    F: int
    k: int
    act: str  # "gelu" or "swiglu"
    renorm: bool
    routing: str  # "normal" or "zipf"
    init: str  # "n002" or "fanin"
    seed: int

    @property
    def A(self) -> int:
        """Number of (token, slot) assignments."""
        return self.T * self.k

    @property
    def P_max(self) -> int:
        """Upper bound on the padded row count for any routing."""
        return padded_rows_max(self.T, self.k, self.E)

    @property
    def nnz_max(self) -> int:
        return (self.P_max // BLOCK) * (self.F // BLOCK)

    def scaled(self, T: int) -> "Config":
        return dataclasses.replace(self, T=T, name=f"{self.name}_T{T}")


def padded_rows_max(T: int, k: int, E: int, block: int = BLOCK) -> int:
    """Largest possible sum over experts of ceil(T_e/B)*B with sum T_e = T*k.

    At most min(E, A) experts are non-empty and each adds at most B-1 pad
    rows, so P <= A + (B-1)*min(E, A), rounded down to a multiple of B.
    """
    A = T * k
    live = min(E, A)
    return ((A + live * (block - 1)) // block) * block


CONFIGS = {
    c.name: c
    for c in [
        Config("tiny", 512, 256, 4, 512, 1, "gelu", False, "normal", "n002", 1001),
        Config("moe_xs", 8192, 512, 64, 2048, 1, "gelu", False, "normal", "fanin", 1002),
        Config("skewed", 16384, 1024, 64, 4096, 1, "gelu", False, "zipf", "fanin", 1003),
        Config("mixtral", 8192, 4096, 8, 14336, 2, "swiglu", True, "normal", "fanin", 1004),
        Config("fine", 4096, 3584, 64, 2560, 8, "swiglu", False, "normal", "fanin", 1005),
    ]
}


def custom(name, T, d, E, F, k, act="gelu", renorm=False, routing="normal", init="fanin", seed=7) -> Config:
    """A config for tests with shapes outside the five named workloads."""
    return Config(name, T, d, E, F, k, act, renorm, routing, init, seed)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk_rows: int = 256) -> np.ndarray:
    """N(0, std^2) drawn in fp32, scaled, rounded to bf16 bits; row-chunked."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        z = rng.standard_normal((r1 - r0,) + tuple(shape[1:]), dtype=np.float32)
        z *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(z)
    return out


def zipf_experts(cfg: Config) -> np.ndarray:
    """Per-token expert draw for the skewed workload (int64 [T])."""
    rng = _rng(cfg.seed, STREAM_ROUTE)
    live = cfg.E - 2
    ranks = np.arange(1, live + 1, dtype=np.float64)
    p = ranks ** -1.254
    p /= p.sum()
    perm = rng.permutation(cfg.E)
    drawn = rng.choice(live, size=cfg.T, p=p)
    return perm[drawn]


def make_logits(cfg: Config) -> np.ndarray:
    rng = _rng(cfg.seed, STREAM_LOGITS)
    logits = rng.standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if cfg.routing == "zipf":
        drawn = zipf_experts(cfg)
        logits[np.arange(cfg.T), drawn] += np.float32(8.0)
    elif cfg.routing != "normal":
        raise ValueError(cfg.routing)
    return logits


def _stds(cfg: Config):
    if cfg.init == "n002":
        return 0.02, 0.02, 0.02
    if cfg.init == "fanin":
        return 1.0, 1.0 / np.sqrt(cfg.d), 1.0 / np.sqrt(cfg.F)
    raise ValueError(cfg.init)


def make_x(cfg: Config) -> np.ndarray:
    sx, _, _ = _stds(cfg)
    return _normal_bf16(_rng(cfg.seed, STREAM_X), (cfg.T, cfg.d), sx)


# Weights of expert block b (deeper experts stack several SDD -> DSD blocks)
# come from their own streams; block 0 keeps the streams of the one-block
# layer.
STREAM_BLOCK_STRIDE = 16


def make_w1(cfg: Config, block: int = 0) -> np.ndarray:
    _, s1, _ = _stds(cfg)
    return _normal_bf16(_rng(cfg.seed, STREAM_W1 + STREAM_BLOCK_STRIDE * block), (cfg.d, cfg.E * cfg.F), s1)


def make_w3(cfg: Config, block: int = 0) -> np.ndarray:
    _, s1, _ = _stds(cfg)
    return _normal_bf16(_rng(cfg.seed, STREAM_W3 + STREAM_BLOCK_STRIDE * block), (cfg.d, cfg.E * cfg.F), s1)


def make_w2(cfg: Config, block: int = 0) -> np.ndarray:
    _, _, s2 = _stds(cfg)
    return _normal_bf16(_rng(cfg.seed, STREAM_W2 + STREAM_BLOCK_STRIDE * block), (cfg.E * cfg.F, cfg.d), s2)


def make_deep_weights(cfg: Config, depth: int) -> dict:
    """w1s, w2s (and w3s for SwiGLU): lists of ``depth`` expert blocks."""
    out = {"w1s": [make_w1(cfg, b) for b in range(depth)], "w2s": [make_w2(cfg, b) for b in range(depth)]}
    if cfg.act == "swiglu":
        out["w3s"] = [make_w3(cfg, b) for b in range(depth)]
    return out


def make_dy(cfg: Config) -> np.ndarray:
    return _normal_bf16(_rng(cfg.seed, STREAM_DY), (cfg.T, cfg.d), 1.0)


def make_inputs(cfg: Config, parts=("logits", "x", "w1", "w3", "w2", "dy")) -> dict:
    """Generate the requested inputs; ``w3`` is skipped for GELU layers."""
    makers = {
        "logits": make_logits,
        "x": make_x,
        "w1": make_w1,
        "w3": make_w3,
        "w2": make_w2,
        "dy": make_dy,
    }
    out = {}
    for p in parts:
        if p == "w3" and cfg.act != "swiglu":
            continue
        out[p] = makers[p](cfg)
    return out


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """Free-standing seeded bf16 tensor, for unit tests of single calls."""
    return _normal_bf16(_rng(seed, stream), tuple(shape), std)


def normal_f32(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    z = _rng(seed, stream).standard_normal(tuple(shape), dtype=np.float32)
    return z * np.float32(std)


def integers(seed: int, stream: int, low: int, high: int, shape) -> np.ndarray:
    return _rng(seed, stream).integers(low, high, size=tuple(shape), dtype=np.int64)
