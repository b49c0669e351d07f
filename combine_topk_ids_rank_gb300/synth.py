"""Seeded synthetic inputs for the top-k dispatch / combine path.

This module is the single source of inputs for both the CUDA library's tests
and benchmark and the CPU oracle.  It only draws random numbers; it contains
none of the routing, dispatch or combine arithmetic.

Every tensor is drawn from its own numpy PCG64 stream keyed by
(seed, stream id, indices), so that
  * rows of one source rank do not depend on how many tokens another rank has,
  * the first T tokens of a source are the same for every T (ladder rungs are
    prefixes of each other),
  * expert-output rows of plane (d, s) can be drawn plane by plane.

bf16 tensors are returned as numpy uint16 bit patterns, rounded from float32
by torch's round-to-nearest-even conversion.

Workloads (the shapes of the pages' decode/prefill ladders: hidden 7168,
256 experts, top-8; the ep_size ranks are logical partitions of one GPU):
  tiny     R=2,  T=16,  H=128,  E=8,   K=2, uniform, identity experts,
           unweighted, unfused
  decode   R=8,  T=64,  H=7168, E=256, K=8, uniform, weighted + residual +
           RMSNorm (eps 1e-6)
  prefill  R=8,  T=4096,H=7168, E=256, K=8, Zipf(1.2) expert popularity,
           weighted + residual + RMSNorm
  wide     R=16, T=1024 (max 2048), H=4096, E=512, K=8, uniform,
           unweighted, unfused
  ladder   R=8,  T in {1, 2, 4, ..., 8192} (max 8192), H=7168, E=256, K=8,
           uniform, weighted + residual + RMSNorm
"""
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
import os

import numpy as np

# stream ids: one per kind of tensor
IDS, LOGITS, X, RESIDUAL, GAMMA, EXPERT_OUT = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    ep_size: int            # R, logical ranks
    tokens_per_rank: int    # T for this call
    max_tokens: int         # M, the workspace is sized once for it
    runtime_max: int        # m, plane stride of this call (T <= m <= M)
    hidden: int             # H
    num_experts: int        # E
    top_k: int              # K
    routing: str            # "uniform" or "zipf"
    zipf_s: float = 1.2
    weighted: bool = True
    fused: bool = True
    identity_experts: bool = False
    eps: float = 1e-6

    @property
    def tokens(self) -> int:
        return self.ep_size * self.tokens_per_rank

    def rung(self, T: int) -> "Workload":
        """Same workload with T tokens per rank (and runtime max T)."""
        return replace(self, tokens_per_rank=T, runtime_max=T,
                       name="%s_T%d" % (self.name.split("_T")[0], T))


WORKLOADS = {
    "tiny": Workload("tiny", 2, 16, 16, 16, 128, 8, 2, "uniform",
                     weighted=False, fused=False, identity_experts=True),
    "decode": Workload("decode", 8, 64, 64, 64, 7168, 256, 8, "uniform"),
    "prefill": Workload("prefill", 8, 4096, 4096, 4096, 7168, 256, 8, "zipf"),
    "wide": Workload("wide", 16, 1024, 2048, 1024, 4096, 512, 8, "uniform",
                     weighted=False, fused=False),
    "ladder": Workload("ladder", 8, 8192, 8192, 8192, 7168, 256, 8, "uniform"),
    # one expert per rank with many rows each: the shape at which the expert-side
    # product (expert layout) is bound by the tensor cores rather than by weights
    "moe_layer": Workload("moe_layer", 8, 4096, 4096, 4096, 7168, 8, 2, "uniform"),
}
LADDER_RUNGS = tuple(2 ** i for i in range(14))   # 1 .. 8192


def rng(seed: int, stream: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([int(seed), int(stream), *map(int, key)])))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _pmap(fn, items):
    items = list(items)
    if len(items) <= 1:
        return [fn(i) for i in items]
    with ThreadPoolExecutor(_threads()) as pool:
        return list(pool.map(fn, items))


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# -- routing ---------------------------------------------------------------

def _top_k_by_keys(keys: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest keys per row, largest first."""
    part = np.argpartition(-keys, K - 1, axis=1)[:, :K]
    order = np.argsort(-np.take_along_axis(keys, part, axis=1), axis=1)
    return np.take_along_axis(part, order, axis=1)


def topk_ids(seed: int, R: int, T: int, E: int, K: int, routing: str = "uniform",
             zipf_s: float = 1.2) -> np.ndarray:
    """int32 [R, T, K]: K distinct expert ids per token.

    uniform: a uniformly random ordered K-subset of the E experts.
    zipf:    K draws without replacement with P(e) proportional to
             (e + 1) ** -zipf_s, renormalised after every draw (expert 0 is
             the most popular; no permutation, so contiguous placement makes
             rank 0 the hottest).
    Both use the Gumbel-top-k construction: adding independent Gumbel noise
    to log-probabilities and keeping the K largest yields exactly sequential
    sampling without replacement, in draw order."""
    if K > E:
        raise ValueError("top_k > num_experts")
    if routing == "uniform":
        logp = np.zeros(E)
    elif routing == "zipf":
        logp = -zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
    else:
        raise ValueError(routing)
    out = np.empty((R, T, K), np.int32)
    for s in range(R):
        g = rng(seed, IDS, s).gumbel(size=(T, E))
        out[s] = _top_k_by_keys(logp[None, :] + g, K)
    return out


def topk_weights(seed: int, R: int, T: int, K: int) -> np.ndarray:
    """float32 [R, T, K]: softmax over each token's K logits, logits N(0,1)."""
    out = np.empty((R, T, K), np.float32)
    for s in range(R):
        z = rng(seed, LOGITS, s).standard_normal((T, K))
        z = np.exp(z - z.max(axis=1, keepdims=True))
        out[s] = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return out


# -- payloads ----------------------------------------------------------------

def normal_rows(seed: int, stream: int, key, rows: int, H: int) -> np.ndarray:
    """bf16 bits [rows, H] of N(0,1) from the stream keyed by `key`."""
    key = key if isinstance(key, tuple) else (key,)
    return to_bf16_bits(rng(seed, stream, *key).standard_normal((rows, H), dtype=np.float32))


def per_rank_rows(seed: int, stream: int, R: int, T: int, H: int) -> np.ndarray:
    """bf16 bits [R, T, H]; source rank s uses its own stream."""
    out = np.empty((R, T, H), np.uint16)

    def fill(s):
        out[s] = normal_rows(seed, stream, s, T, H)
    _pmap(fill, range(R))
    return out


def gamma(seed: int, H: int) -> np.ndarray:
    """bf16 bits [H]: 1 + 0.1 * N(0,1)."""
    g = 1.0 + 0.1 * rng(seed, GAMMA).standard_normal(H)
    return to_bf16_bits(g.astype(np.float32))


def expert_out_planes(seed: int, R: int, m: int, H: int, rows_per_plane,
                      out: np.ndarray = None) -> np.ndarray:
    """bf16 bits [R, R, m, H] of N(0,1) expert outputs.

    rows_per_plane[d][s] rows are drawn for plane (d, s) (its first rows; a
    plane is drawn from its own stream, so the first j rows do not depend on
    how many more are drawn).  Other rows are left as in `out` (np.empty by
    default; untouched pages cost no memory)."""
    if out is None:
        out = np.empty((R, R, m, H), np.uint16)

    def fill(ds):
        d, s = ds
        n = int(rows_per_plane[d][s])
        if n:
            out[d, s, :n] = normal_rows(seed, EXPERT_OUT, (d, s), n, H)
    _pmap(fill, [(d, s) for d in range(R) for s in range(R)])
    return out


def inputs(w: Workload, seed: int = 0, payloads: bool = True) -> dict:
    """Host inputs of one call: ids, weights, and (if payloads) x, residual,
    gamma as bf16 bits.  Expert outputs are drawn separately with
    expert_out_planes once the per-plane counts are known."""
    R, T, H = w.ep_size, w.tokens_per_rank, w.hidden
    d = dict(topk_ids=topk_ids(seed, R, T, w.num_experts, w.top_k, w.routing, w.zipf_s),
             topk_w=topk_weights(seed, R, T, w.top_k))
    if payloads:
        d["x"] = per_rank_rows(seed, X, R, T, H)
        if w.fused:
            d["residual"] = per_rank_rows(seed, RESIDUAL, R, T, H)
            d["gamma"] = gamma(seed, H)
    return d
