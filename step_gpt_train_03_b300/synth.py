"""Seeded synthetic inputs shared by the CUDA path, the tests and the bench.

This module holds random draws only: model initialisation, token streams and the
standalone layernorm inputs.  It contains none of the training step's arithmetic,
so both the CUDA library and the CPU checker can consume its output without
sharing any computation.

Input recipe (all numpy PCG64 via ``numpy.random.default_rng``):

* Weights: every matrix and both embedding tables ~ N(0, 0.02); the two residual
  projections (attention output projection, MLP output projection) are further
  scaled by 1/sqrt(2L); layernorm gains 1, biases 0; the padded vocabulary rows of
  the token table (ids >= V) are 0.  Drawn from ``default_rng(1000 + seed)`` in the
  fixed tensor order of ``PARAM_ORDER``.
* Tokens: either uniform in [0, V) (tokens then targets, two draws) or a bounded
  Zipf stream with p(k) proportional to (k+1)^-s over k in [0, V), sampled by
  inverse CDF.  A stream of n*B*T+1 ids gives n batches; batch i is the window
  [i*BT, (i+1)*BT) and its targets are the same window shifted by one.  The
  heavy-tailed id frequencies stand in for tokenised text (the pages train on
  tinyshakespeare / TinyStories / FineWeb, none of which is available here).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

PARAM_ORDER = (
    "wte", "wpe",
    "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
    "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb",
    "lnfw", "lnfb",
)


@dataclass(frozen=True)
class ModelShape:
    max_seq_len: int
    vocab_size: int
    padded_vocab_size: int
    num_layers: int
    num_heads: int
    channels: int


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape | None
    B: int
    T: int
    seed: int
    precision: str            # "fp32" or "bf16"
    steps: int
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    tokens: str = "zipf"      # "uniform" or "zipf"
    fixed_batch: bool = False


GPT2_124M = ModelShape(1024, 50257, 50304, 12, 12, 768)
GPT2_350M = ModelShape(1024, 50257, 50304, 24, 16, 1024)
TINY = ModelShape(32, 512, 512, 2, 4, 64)
# the tiny model with one head of size 64, the head size of the bf16 (tensor-core) path
TINY_HS64 = ModelShape(32, 512, 512, 2, 1, 64)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", TINY, 2, 32, 0, "fp32", 1, tokens="uniform"),
    "gpt2_124m_fp32_b4_t64": Workload("gpt2_124m_fp32_b4_t64", GPT2_124M, 4, 64, 1, "fp32", 10,
                                      fixed_batch=True),
    "layernorm_8192x768_fp32": Workload("layernorm_8192x768_fp32", None, 8192, 1, 2, "fp32", 1),
    "gpt2_124m_bf16_b16_t1024": Workload("gpt2_124m_bf16_b16_t1024", GPT2_124M, 16, 1024, 2, "bf16",
                                         50, lr=6e-4, weight_decay=0.1),
    "gpt2_350m_bf16_b8_t1024": Workload("gpt2_350m_bf16_b8_t1024", GPT2_350M, 8, 1024, 3, "bf16",
                                        20, lr=3e-4, weight_decay=0.1),
    # the 124M bf16 workload in the fp8 mode (e4m3 qkv and fc products)
    "gpt2_124m_fp8_b16_t1024": Workload("gpt2_124m_fp8_b16_t1024", GPT2_124M, 16, 1024, 2, "fp8",
                                        50, lr=6e-4, weight_decay=0.1),
}


def param_shapes(s: ModelShape) -> dict[str, tuple[int, ...]]:
    """Shapes of the sixteen parameter tensors (per-layer tensors stacked over L)."""
    C, L, Vp = s.channels, s.num_layers, s.padded_vocab_size
    return {
        "wte": (Vp, C), "wpe": (s.max_seq_len, C),
        "ln1w": (L, C), "ln1b": (L, C),
        "qkvw": (L, 3 * C, C), "qkvb": (L, 3 * C),
        "attprojw": (L, C, C), "attprojb": (L, C),
        "ln2w": (L, C), "ln2b": (L, C),
        "fcw": (L, 4 * C, C), "fcb": (L, 4 * C),
        "fcprojw": (L, C, 4 * C), "fcprojb": (L, C),
        "lnfw": (C,), "lnfb": (C,),
    }


def init_params(s: ModelShape, seed: int) -> dict[str, np.ndarray]:
    """Seeded float32 initial weights, one array per tensor in ``PARAM_ORDER``."""
    rng = np.random.default_rng(1000 + seed)
    shapes = param_shapes(s)
    resid_scale = np.float32(0.02 / np.sqrt(2.0 * s.num_layers))
    out = {}
    for name in PARAM_ORDER:
        shp = shapes[name]
        if name in ("ln1w", "ln2w", "lnfw"):
            a = np.ones(shp, np.float32)
        elif name.endswith("b"):
            a = np.zeros(shp, np.float32)
        else:
            a = rng.standard_normal(shp, dtype=np.float32)
            a *= resid_scale if name in ("attprojw", "fcprojw") else np.float32(0.02)
            if name == "wte":
                a[s.vocab_size:] = 0.0
        out[name] = a
    return out


def uniform_tokens(V: int, B: int, T: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    rng = np.random.default_rng(seed)
    tokens = rng.integers(0, V, (B, T), dtype=np.int32)
    targets = rng.integers(0, V, (B, T), dtype=np.int32)
    return tokens, targets


def zipf_stream(n: int, V: int, seed: int, s: float = 1.1) -> np.ndarray:
    """n ids from the bounded Zipf law p(k) ~ (k+1)^-s on [0, V), by inverse CDF."""
    rng = np.random.default_rng(seed)
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int32)


def zipf_batches(V: int, B: int, T: int, n_batches: int, seed: int):
    """List of (tokens, targets) int32 (B, T) windows over one seeded Zipf stream."""
    BT = B * T
    x = zipf_stream(n_batches * BT + 1, V, seed)
    return [(x[i * BT:(i + 1) * BT].reshape(B, T).copy(),
             x[i * BT + 1:(i + 1) * BT + 1].reshape(B, T).copy()) for i in range(n_batches)]


def workload_batches(w: Workload, n_batches: int | None = None):
    """The batches a workload trains on, in step order."""
    s = w.shape
    n = w.steps if n_batches is None else n_batches
    if w.tokens == "uniform":
        b = uniform_tokens(s.vocab_size, w.B, w.T, w.seed)
        return [b] * n
    if w.fixed_batch:
        b = zipf_batches(s.vocab_size, w.B, w.T, 1, w.seed)[0]
        return [b] * n
    return zipf_batches(s.vocab_size, w.B, w.T, n, w.seed)


def layernorm_inputs(N: int, C: int, seed: int):
    """x ~ 3 N(0,1) + 0.5, gamma ~ N(1, 0.1), beta ~ N(0, 0.1), dy ~ N(0, 1); float32."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((N, C)) * 3.0 + 0.5).astype(np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    b = (0.1 * rng.standard_normal(C)).astype(np.float32)
    dy = rng.standard_normal((N, C)).astype(np.float32)
    return x, w, b, dy
