"""Seeded synthetic inputs shaped like the workloads of the MXFP8 expert-MLP pages.

This module only draws random numbers and arranges them (routing, sorting by expert); it holds
none of the method's arithmetic, so both the CUDA path's tests and the oracle's tests use it.
bf16 tensors are returned as their uint16 bit patterns (round-to-nearest-even from float32).

Workloads (the pages train Mixtral-8x7B and Llama-3.1 models on datasets that are not
available here; these synthetic tensors of the same shapes stand in for them):
  tiny      T=256 tokens, top-2, E=4, H=256, F=512; router logits N(0,1)
  llama     dense Llama-3.1-8B MLP as one group: E=1, T=8192, H=4096, F=14336, gate = 1
  mixtral   Mixtral-8x7B experts: E=8, top-2, T=16384, H=4096, F=14336;
            logits N(0,1) + per-expert bias N(0, 0.5)
  fine      fine-grained skewed MoE: E=64, top-8, T=32768, H=2048, F=1408; Zipf(1.2)
            popularity over a random permutation of experts, the 3 least popular get none;
            top-8 without replacement (Gumbel-top-k on log popularity); gates Dirichlet(1)
x ~ N(0,1) and weights ~ N(0, 0.02) everywhere.  W1 is [E, 2F, H] (rows [0,F) gate, [F,2F) up),
W2 is [E, H, F]; both are returned flattened to [E*2F, H] and [E*H, F].
"""
from __future__ import annotations

import concurrent.futures as _cf
from dataclasses import dataclass

import numpy as np

MOE_SHAPES = {
    "tiny": dict(T=256, topk=2, E=4, H=256, F=512),
    "llama": dict(T=8192, topk=1, E=1, H=4096, F=14336),
    "mixtral": dict(T=16384, topk=2, E=8, H=4096, F=14336),
    "fine": dict(T=32768, topk=8, E=64, H=2048, F=1408),
}

QUANT_SWEEP = [(4096, 4096), (8192, 4096), (16384, 14336)]


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_bits(a)


def _parallel_normal_bf16(seed_seq: np.random.SeedSequence, nchunks: int, chunk_shape, std: float,
                          threads: int = 16) -> np.ndarray:
    """nchunks independent chunks, each from its own spawned generator (thread-count independent)."""
    kids = seed_seq.spawn(nchunks)
    out = np.empty((nchunks,) + tuple(chunk_shape), dtype=np.uint16)

    def one(i):
        out[i] = _normal_bf16(np.random.default_rng(kids[i]), chunk_shape, std)

    with _cf.ThreadPoolExecutor(max_workers=max(1, min(threads, nchunks))) as ex:
        list(ex.map(one, range(nchunks)))
    return out


def quant_matrix(M: int, K: int, seed: int = 0) -> np.ndarray:
    """[M, K] bf16 bits: N(0,1), 0.1% of entries (uniform positions) x200, and in every row one
    32-wide block (uniform block index) set to zero."""
    rng = np.random.default_rng([seed, M, K])
    a = rng.standard_normal(size=(M, K), dtype=np.float32)
    n_out = max(1, (M * K) // 1000)
    idx = rng.integers(0, M * K, size=n_out)
    a.reshape(-1)[idx] *= np.float32(200.0)
    if K >= 32:
        blk = rng.integers(0, K // 32, size=M)
        cols = blk[:, None] * 32 + np.arange(32)[None, :]
        a[np.arange(M)[:, None], cols] = 0.0
    return bf16_bits(a)


@dataclass
class MoEInputs:
    name: str
    T: int
    topk: int
    E: int
    H: int
    F: int
    x_sorted: np.ndarray          # [R, H] bf16 bits, rows grouped by expert
    split_sizes: np.ndarray       # [E] int32
    gates: np.ndarray | None      # [R] float32 routing weights in sorted order (None = all ones)
    w1: np.ndarray                # [E*2F, H] bf16 bits
    w2: np.ndarray                # [E*H, F] bf16 bits
    token_of_row: np.ndarray      # [R] int64 source token of each sorted row
    x_tokens: np.ndarray | None = None      # [T, H] bf16 bits before the sort (routed workloads)
    topk_experts: np.ndarray | None = None  # [T, k] int32 router choices
    topk_gates: np.ndarray | None = None    # [T, k] float32 routing weights

    @property
    def R(self) -> int:
        return int(self.x_sorted.shape[0])

    def flops(self) -> float:
        """6*R*H*F: two GEMMs of 2*R*H*F (gate and up) plus one of 2*R*F*H."""
        return 6.0 * self.R * self.H * self.F


def _route_topk_softmax(logits: np.ndarray, k: int):
    """softmax over experts, top-k (ties -> lower expert index), renormalized over the k."""
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(p, order, axis=1)
    sel = sel / sel.sum(axis=1, keepdims=True)
    return order, sel.astype(np.float32)


def _sort_by_expert(experts: np.ndarray, weights: np.ndarray, E: int):
    """Stable sort of (token, slot) pairs by expert id -> (token_of_row, gates, split_sizes)."""
    T, k = experts.shape
    flat_e = experts.reshape(-1)
    flat_t = np.repeat(np.arange(T, dtype=np.int64), k)
    flat_w = weights.reshape(-1)
    order = np.argsort(flat_e, kind="stable")
    split = np.bincount(flat_e, minlength=E).astype(np.int32)
    return flat_t[order], flat_w[order].astype(np.float32), split


def _weights(ss: np.random.SeedSequence, E: int, H: int, F: int):
    s1, s2 = ss.spawn(2)
    w1 = _parallel_normal_bf16(s1, E * 2, (F, H), 0.02).reshape(E * 2 * F, H)
    w2 = _parallel_normal_bf16(s2, E, (H, F), 0.02).reshape(E * H, F)
    return w1, w2


def moe_workload(name: str, seed: int = 0) -> MoEInputs:
    shp = MOE_SHAPES[name]
    T, k, E, H, F = shp["T"], shp["topk"], shp["E"], shp["H"], shp["F"]
    ss = np.random.SeedSequence([seed, 0x6D78])
    s_x, s_w, s_r = ss.spawn(3)
    x = _parallel_normal_bf16(s_x, 8, (T // 8, H), 1.0).reshape(T, H) if T % 8 == 0 else \
        _normal_bf16(np.random.default_rng(s_x), (T, H), 1.0)
    w1, w2 = _weights(s_w, E, H, F)
    rng = np.random.default_rng(s_r)
    if name == "llama":
        token_of_row = np.arange(T, dtype=np.int64)
        gates = None
        split = np.array([T], dtype=np.int32)
    elif name in ("tiny", "mixtral"):
        logits = rng.standard_normal(size=(T, E))
        if name == "mixtral":
            logits = logits + rng.normal(0.0, 0.5, size=E)[None, :]
        experts, w = _route_topk_softmax(logits, k)
        token_of_row, gates, split = _sort_by_expert(experts, w, E)
    elif name == "fine":
        rank_weight = 1.0 / np.arange(1, E + 1, dtype=np.float64) ** 1.2
        rank_weight[-3:] = 0.0                       # the three least popular experts get no tokens
        perm = rng.permutation(E)                    # expert perm[r] has popularity rank r
        pop = np.zeros(E)
        pop[perm] = rank_weight
        pop /= pop.sum()
        with np.errstate(divide="ignore"):
            logp = np.log(pop)
        keys = logp[None, :] + rng.gumbel(size=(T, E))
        experts = np.argsort(-keys, axis=1, kind="stable")[:, :k]
        w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
        token_of_row, gates, split = _sort_by_expert(experts, w, E)
    else:
        raise KeyError(name)
    x_sorted = np.ascontiguousarray(x[token_of_row])
    if name == "llama":
        return MoEInputs(name, T, k, E, H, F, x_sorted, split, gates, w1, w2, token_of_row)
    return MoEInputs(name, T, k, E, H, F, x_sorted, split, gates, w1, w2, token_of_row, x,
                     experts.astype(np.int32), w.astype(np.float32))


def custom_moe(split_sizes, H: int, F: int, seed: int = 0, with_gates: bool = True,
               x_std: float = 1.0, w_std: float = 0.02) -> MoEInputs:
    """Explicit per-expert row counts (for ragged / empty-expert parity cases)."""
    split = np.asarray(split_sizes, dtype=np.int32)
    E = split.size
    R = int(split.sum())
    ss = np.random.SeedSequence([seed, 0x6375, E, H, F, R])
    s_x, s_w, s_g = ss.spawn(3)
    s_w1, s_w2 = s_w.spawn(2)
    x = _normal_bf16(np.random.default_rng(s_x), (R, H), x_std)
    w1 = _normal_bf16(np.random.default_rng(s_w1), (E * 2 * F, H), w_std)
    w2 = _normal_bf16(np.random.default_rng(s_w2), (E * H, F), w_std)
    gates = np.random.default_rng(s_g).uniform(0.05, 1.0, size=R).astype(np.float32) if with_gates else None
    return MoEInputs("custom", R, 1, E, H, F, x, split, gates, w1, w2, np.arange(R, dtype=np.int64))


def sample_rows(split_sizes, seed: int = 0, first: int = 8, last: int = 8, rand: int = 64,
                tile: int = 128) -> np.ndarray:
    """Deterministic row sample per expert: the first and last rows, random rows, and the rows on
    both sides of every `tile`-row boundary inside the expert (sorted, unique)."""
    split = np.asarray(split_sizes, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(split)])
    rng = np.random.default_rng([seed, 0x5A4D])
    rows = []
    for e in range(split.size):
        n = int(split[e])
        if n == 0:
            continue
        base = int(off[e])
        loc = set(range(min(first, n))) | set(range(max(0, n - last), n))
        if rand:
            loc |= set(rng.integers(0, n, size=min(rand, n)).tolist())
        for b in range(tile, n, tile):
            loc |= {b - 1, b}
        rows.extend(base + r for r in sorted(loc))
    return np.array(sorted(set(rows)), dtype=np.int64)
