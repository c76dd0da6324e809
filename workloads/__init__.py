"""Seeded synthetic inputs for the MoE dispatch / combine path.

This module only draws inputs: hidden states, router logits turned into top-k expert ids and
probabilities, expert outputs and upstream gradients.  It holds none of the dispatch, layout,
quantisation or combine arithmetic, so both the CPU oracle and the CUDA path can take their
inputs from here without sharing any of the method.

Every array is a plain numpy array.  BF16 tensors are carried as ``uint16`` bit patterns.

Recipe (all draws from ``numpy.random.Generator(PCG64(seed))``):

* hidden states ``x``: standard normal drawn in float32, rounded to bf16 (RNE);
  config-specific structure (outlier rows x50, all-zero rows) is applied in float32 before
  the bf16 rounding;
* router: logits drawn in float64, top-k by logit (descending, ties to the lower expert id),
  probabilities computed in float64 and rounded to float32;
* expert outputs ``y`` and gradients: standard normal in float32 rounded to bf16.

The "balanced" router draws nothing: slot k of token t names expert (t*K + k) mod E with
probability 1/K (static benchmark routing: the row count is identical on every dispatch).

Seeds per config index c: x 1000+c, logits 2000+c, expert bias 3000+c, Zipf draws 4000+c,
outlier / zero-row choice 5000+c, grad_out 6000+c, expert outputs 7000+c, grad rows 8000+c.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "Config", "CONFIGS", "bf16_bits_from_f32", "f32_from_bf16_bits", "make_x", "make_routing",
    "make_expert_out", "make_grad_out", "make_grad_rows", "make_inputs", "r_max", "scaled",
]


@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic MoE-layer workload.

    T tokens, H hidden size, E routed experts, K top-k slots, S fused shared expert (0/1),
    P logical expert partitions (E % P == 0) and C the per-partition token capacity.
    """
    index: int
    name: str
    T: int
    H: int
    E: int
    K: int
    S: int = 0
    P: int = 1
    C: int | None = None          # None: capacity = T (never overflows)
    router: str = "softmax"       # softmax | dsv3 | zipf | hot | balanced
    outlier_frac: float = 0.0     # fraction of rows scaled x50
    zero_frac: float = 0.0        # fraction of all-zero rows
    rerun_C: int | None = None    # capacity of the full rerun after an overflow run
    pad_multiple: int = 1         # rows of every group padded to a multiple of this
    num_permuted_tokens: int | None = None   # static row capacity (None: the most any routing needs)

    @property
    def capacity(self) -> int:
        return self.T if self.C is None else self.C


CONFIGS: dict[str, Config] = {
    "tiny": Config(1, "tiny", T=128, H=256, E=8, K=2),
    "qwen3": Config(2, "qwen3", T=8192, H=2048, E=128, K=8, outlier_frac=0.01),
    "dsv3": Config(3, "dsv3", T=4096, H=7168, E=256, K=8, S=1, P=8, C=4096, router="dsv3"),
    "mixtral": Config(4, "mixtral", T=16384, H=4096, E=8, K=2, router="zipf"),
    "dsv3_large": Config(5, "dsv3_large", T=32768, H=7168, E=256, K=8, P=8, C=20000,
                         router="hot", zero_frac=0.001, rerun_C=40000),
    # benchmark static routing: balanced and noise-free, so the row count (T*K/E = 128 rows per
    # expert, plus the shared rows) is the same on every dispatch and is passed as a static row
    # capacity; groups padded to 128
    "dsv3_static": Config(6, "dsv3_static", T=4096, H=7168, E=256, K=8, S=1, P=8, C=4096,
                          router="balanced", pad_multiple=128, num_permuted_tokens=4096 * 8 + 4096),
}


def scaled(cfg: Config, T: int | None = None, H: int | None = None, **kw) -> Config:
    """Same recipe as ``cfg`` at a different size (for parity cases the oracle finishes fast)."""
    upd = {}
    if T is not None:
        upd["T"] = T
    if H is not None:
        upd["H"] = H
    upd.update(kw)
    return dataclasses.replace(cfg, **upd)


def r_max(cfg: Config) -> int:
    """Rows of the dispatched buffers: every (token, slot) pair plus one shared row per token."""
    return cfg.T * cfg.K + cfg.S * cfg.T


# ----------------------------------------------------------------------------------------
# bf16 bit patterns (the generator's own rounding; used only to produce inputs)
# ----------------------------------------------------------------------------------------
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal_bf16(seed: int, shape) -> np.ndarray:
    rng = _rng(seed)
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    chunk = 1 << 24
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        flat[s:s + n] = bf16_bits_from_f32(rng.standard_normal(n, dtype=np.float32))
    return out


# ----------------------------------------------------------------------------------------
# hidden states
# ----------------------------------------------------------------------------------------
def make_x(cfg: Config) -> np.ndarray:
    """Hidden states [T, H] as bf16 bits: N(0,1) with the config's outlier / zero rows."""
    c = cfg.index
    rng = _rng(1000 + c)
    sel = _rng(5000 + c)
    n_out = int(round(cfg.outlier_frac * cfg.T))
    n_zero = int(round(cfg.zero_frac * cfg.T))
    out_rows = np.sort(sel.choice(cfg.T, size=n_out, replace=False)) if n_out else np.zeros(0, np.int64)
    zero_rows = np.sort(sel.choice(cfg.T, size=n_zero, replace=False)) if n_zero else np.zeros(0, np.int64)
    x = np.empty((cfg.T, cfg.H), dtype=np.uint16)
    rows_per_chunk = max(1, (1 << 24) // cfg.H)
    scale = np.ones(cfg.T, dtype=np.float32)
    scale[out_rows] = 50.0
    scale[zero_rows] = 0.0
    for r0 in range(0, cfg.T, rows_per_chunk):
        r1 = min(cfg.T, r0 + rows_per_chunk)
        v = rng.standard_normal((r1 - r0, cfg.H), dtype=np.float32)
        v *= scale[r0:r1, None]
        x[r0:r1] = bf16_bits_from_f32(v)
    return x


# ----------------------------------------------------------------------------------------
# routing: top-k expert ids [T, K] int32 and probabilities [T, K] float32
# ----------------------------------------------------------------------------------------
def _topk_desc(score: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, by descending score, ties to the lower index."""
    order = np.argsort(-score, axis=1, kind="stable")
    return order[:, :k]


def _softmax_rows(v: np.ndarray) -> np.ndarray:
    m = v.max(axis=1, keepdims=True)
    e = np.exp(v - m)
    return e / e.sum(axis=1, keepdims=True)


def make_routing(cfg: Config) -> tuple[np.ndarray, np.ndarray]:
    """(topk_ids int32 [T,K], probs float32 [T,K]) per the config's router recipe."""
    c = cfg.index
    T, E, K = cfg.T, cfg.E, cfg.K
    if cfg.router == "zipf":
        # K distinct experts drawn without replacement from p(e) ~ (e+1)^-1.2; slot 0 = first draw
        w = (np.arange(E, dtype=np.float64) + 1.0) ** -1.2
        rng = _rng(4000 + c)
        ids = np.empty((T, K), dtype=np.int64)
        avail = np.broadcast_to(w, (T, E)).copy()
        for k in range(K):
            cdf = np.cumsum(avail, axis=1)
            u = rng.random(T) * cdf[:, -1]
            pick = np.minimum((cdf <= u[:, None]).sum(axis=1), E - 1)
            # never pick an exhausted (zero-weight) expert
            while True:
                bad = avail[np.arange(T), pick] == 0
                if not bad.any():
                    break
                pick[bad] = (pick[bad] + 1) % E
            ids[:, k] = pick
            avail[np.arange(T), pick] = 0.0
        logits = _rng(2000 + c).standard_normal((T, K))
        probs = _softmax_rows(logits)
        return ids.astype(np.int32), probs.astype(np.float32)

    if cfg.router == "balanced":
        # slot k of token t names expert (t*K + k) mod E: K distinct experts per token (K <= E)
        # and, when E divides T*K, exactly T*K/E rows per expert; equal probabilities 1/K
        t = np.arange(T, dtype=np.int64)[:, None]
        k = np.arange(K, dtype=np.int64)[None, :]
        ids = (t * K + k) % E
        probs = np.full((T, K), 1.0 / K)
        return ids.astype(np.int32), probs.astype(np.float32)
    logits = _rng(2000 + c).standard_normal((T, E))
    if cfg.router == "dsv3":
        bias = 0.5 * _rng(3000 + c).standard_normal(E)
        ids = _topk_desc(logits + bias[None, :], K)
        raw = np.take_along_axis(logits, ids, axis=1)
        sig = 1.0 / (1.0 + np.exp(-raw))
        probs = sig / sig.sum(axis=1, keepdims=True)
    elif cfg.router == "hot":
        biased = logits.copy()
        biased[:, :4] += 3.0
        ids = _topk_desc(biased, K)
        probs = _softmax_rows(np.take_along_axis(biased, ids, axis=1))
    else:
        ids = _topk_desc(logits, K)
        probs = _softmax_rows(np.take_along_axis(logits, ids, axis=1))
    return ids.astype(np.int32), probs.astype(np.float32)


# ----------------------------------------------------------------------------------------
# expert outputs and gradients
# ----------------------------------------------------------------------------------------
def make_expert_out(cfg: Config) -> np.ndarray:
    """Expert outputs [R_max, H] bf16 bits, N(0,1)."""
    return _normal_bf16(7000 + cfg.index, (r_max(cfg), cfg.H))


def make_grad_out(cfg: Config) -> np.ndarray:
    """Gradient of the combined output [T, H] bf16 bits, N(0,1)."""
    return _normal_bf16(6000 + cfg.index, (cfg.T, cfg.H))


def make_grad_rows(cfg: Config) -> np.ndarray:
    """Gradient of the dispatched rows [R_max, H] bf16 bits, N(0,1)."""
    return _normal_bf16(8000 + cfg.index, (r_max(cfg), cfg.H))


def make_inputs(cfg: Config) -> dict:
    ids, probs = make_routing(cfg)
    return {"x": make_x(cfg), "topk_ids": ids, "probs": probs}
