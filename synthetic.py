"""Seeded synthetic inputs for the quantized MoE layer (weights, activations, token ids).

This module only draws random numbers and writes them into the canonical byte
layouts; it holds none of the layer's arithmetic (no dequantisation, no routing,
no matmul). Both the CPU oracle and the CUDA path read the bytes it produces.

Workloads (the five benchmark shapes of the quantized MoE layer):

  0  tiny-q8      d=256, 8 routed experts, top-2, f=128, shared f=128, all Q8_0, 4 tokens
  1  decode-1     d=4096, 256 experts, top-8, f=2048, routed Q2_K, shared Q8_0, 1 token
  2  decode-16    as 1, 16 tokens, router logit bias ~ N(0, 1)
  3  prefill-512  as 1, 512 tokens, Zipf(1.1) popularity bias over a random expert order
  4  prefill-4096 as 1, 4096 tokens; the first 1024 are hash-routed by token id through a
                  [129280 x 8] table of distinct expert ids, the rest use the learned router

Canonical byte layouts (little endian, one quantised row = its blocks back to back along K,
rows row-major, experts back to back):

  Q8_0 block, 32 weights, 34 bytes:  fp16 scale | 32 x int8 q            w = scale * q
  Q2_K super-block, 256 weights, 84 bytes:
      16 bytes of sub-block scales (byte j: low nibble s_j, high nibble m_j)
      64 bytes of 2-bit quants (weight i in byte i >> 2, bits 2*(i & 3))
      fp16 d | fp16 dmin                                  w_i = d*s_j*q_i - dmin*m_j, j = i // 16

Random streams: every named tensor draws from its own generator
``default_rng(SeedSequence(seed, spawn_key=(tag, expert)))`` so that any single expert's
tensor can be produced without drawing the others.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

Q8_0_BLOCK = 32
Q8_0_BYTES = 34
Q2_K_BLOCK = 256
Q2_K_BYTES = 84

FMT_BLOCK = {"q8_0": (Q8_0_BLOCK, Q8_0_BYTES), "q2_k": (Q2_K_BLOCK, Q2_K_BYTES)}

# stream tags
TAG_ROUTER_W, TAG_ROUTER_B, TAG_GATE, TAG_UP, TAG_DOWN = 1, 2, 3, 4, 5
TAG_S_GATE, TAG_S_UP, TAG_S_DOWN, TAG_X, TAG_TOKEN_IDS, TAG_HASH = 6, 7, 8, 9, 10, 11

HASH_VOCAB = 129280


@dataclass(frozen=True)
class Spec:
    name: str
    d: int
    n_experts: int
    top_k: int
    f: int
    f_shared: int
    n_shared: int
    fmt_gate_up: str
    fmt_down: str
    fmt_shared: str
    n_tokens: int
    seed: int
    bias: Optional[str] = None  # None | "normal" | "zipf"
    n_hash: int = 0
    hash_vocab: int = 0
    zipf_s: float = 1.1
    bias_std: float = 1.0

    def with_(self, **kw) -> "Spec":
        return replace(self, **kw)


_DS = dict(d=4096, n_experts=256, top_k=8, f=2048, f_shared=2048, n_shared=1,
           fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0")

CONFIGS = {
    0: Spec("tiny-q8", d=256, n_experts=8, top_k=2, f=128, f_shared=128, n_shared=1,
            fmt_gate_up="q8_0", fmt_down="q8_0", fmt_shared="q8_0", n_tokens=4, seed=0),
    1: Spec("decode-1", n_tokens=1, seed=1, **_DS),
    2: Spec("decode-16", n_tokens=16, seed=2, bias="normal", **_DS),
    3: Spec("prefill-512", n_tokens=512, seed=3, bias="zipf", **_DS),
    4: Spec("prefill-4096", n_tokens=4096, seed=4, n_hash=1024, hash_vocab=HASH_VOCAB, **_DS),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=tuple(key)))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def row_bytes(fmt: str, k: int) -> int:
    blk, nb = FMT_BLOCK[fmt]
    if k % blk:
        raise ValueError(f"K={k} is not a multiple of the {fmt} block ({blk})")
    return k // blk * nb


def quant_tensor(fmt: str, rows: int, k: int, seed: int, *key: int) -> np.ndarray:
    """Random quantised [rows x k] matrix in canonical bytes, shape (rows, row_bytes)."""
    rng = _rng(seed, *key)
    if fmt == "q8_0":
        nb = k // Q8_0_BLOCK
        scale = rng.uniform(0.5e-3, 2e-3, size=(rows, nb)).astype(np.float16)
        q = rng.integers(-127, 128, size=(rows, nb, 32), dtype=np.int8)
        out = np.empty((rows, nb, Q8_0_BYTES), dtype=np.uint8)
        out[:, :, 0:2] = scale.view(np.uint8).reshape(rows, nb, 2)
        out[:, :, 2:] = q.view(np.uint8)
        return out.reshape(rows, nb * Q8_0_BYTES)
    if fmt == "q2_k":
        nb = k // Q2_K_BLOCK
        scales = rng.integers(0, 256, size=(rows, nb, 16), dtype=np.uint8)  # s, m uniform 0..15
        qs = rng.integers(0, 256, size=(rows, nb, 64), dtype=np.uint8)      # q uniform 0..3
        dd = rng.uniform(1e-3, 4e-3, size=(rows, nb, 2)).astype(np.float16)  # d, dmin
        out = np.empty((rows, nb, Q2_K_BYTES), dtype=np.uint8)
        out[:, :, 0:16] = scales
        out[:, :, 16:80] = qs
        out[:, :, 80:84] = dd.view(np.uint8).reshape(rows, nb, 4)
        return out.reshape(rows, nb * Q2_K_BYTES)
    raise ValueError(f"unknown format {fmt}")


class ExpertStack:
    """Lazy [E, rows, row_bytes] stack of one routed projection; experts drawn on demand."""

    def __init__(self, fmt: str, n_experts: int, rows: int, k: int, seed: int, tag: int):
        self.fmt, self.n, self.rows, self.k, self.seed, self.tag = fmt, n_experts, rows, k, seed, tag
        self.row_bytes = row_bytes(fmt, k)
        self._cache: dict[int, np.ndarray] = {}
        self._full: Optional[np.ndarray] = None

    def __len__(self) -> int:
        return self.n

    def __getitem__(self, e: int) -> np.ndarray:
        e = int(e)
        if not 0 <= e < self.n:
            raise IndexError(e)
        if self._full is not None:
            return self._full[e]
        t = self._cache.get(e)
        if t is None:
            t = quant_tensor(self.fmt, self.rows, self.k, self.seed, self.tag, e)
            self._cache[e] = t
        return t

    def full(self) -> np.ndarray:
        if self._full is None:
            full = np.empty((self.n, self.rows, self.row_bytes), dtype=np.uint8)
            for e in range(self.n):
                full[e] = self[e]
            self._full = full
            self._cache.clear()
        return self._full


@dataclass
class Problem:
    spec: Spec
    router_w: np.ndarray                 # fp32 [E, d]
    router_b: Optional[np.ndarray]       # fp32 [E] or None
    gate: ExpertStack                    # [E, f, row_bytes(d)]
    up: ExpertStack
    down: ExpertStack                    # [E, d, row_bytes(f)]
    shared_gate: Optional[np.ndarray]    # [f_s, row_bytes(d)]
    shared_up: Optional[np.ndarray]
    shared_down: Optional[np.ndarray]    # [d, row_bytes(f_s)]
    hash_table: Optional[np.ndarray]     # int32 [V, k]
    x_bits: np.ndarray                   # uint16 bf16 bit patterns [N, d]
    token_ids: Optional[np.ndarray]      # int32 [n_hash]
    extra: dict = field(default_factory=dict)


def hash_table(n_rows: int, n_experts: int, k: int, seed: int) -> np.ndarray:
    """Rows of k distinct expert ids: the first k entries of an independent uniform random
    permutation of 0..E-1 per row (partial Fisher-Yates, vectorised over rows)."""
    rng = _rng(seed, TAG_HASH)
    perm = np.tile(np.arange(n_experts, dtype=np.int32), (n_rows, 1))
    rows = np.arange(n_rows)
    for i in range(k):
        j = rng.integers(i, n_experts, size=n_rows)
        a = perm[rows, i].copy()
        perm[rows, i] = perm[rows, j]
        perm[rows, j] = a
    return np.ascontiguousarray(perm[:, :k])


def router_bias(spec: Spec) -> Optional[np.ndarray]:
    if spec.bias is None:
        return None
    rng = _rng(spec.seed, TAG_ROUTER_B)
    if spec.bias == "normal":
        return (rng.standard_normal(spec.n_experts) * spec.bias_std).astype(np.float32)
    if spec.bias == "zipf":
        # popularity ~ rank^-s over a random order of the experts; the logit bias is the log
        # of that weight (temperature 1): b_e = -s * ln(rank_e)
        rank = rng.permutation(spec.n_experts) + 1
        return (-spec.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)
    raise ValueError(spec.bias)


def activations(spec: Spec, n_tokens: Optional[int] = None) -> np.ndarray:
    n = spec.n_tokens if n_tokens is None else n_tokens
    rng = _rng(spec.seed, TAG_X)
    return f32_to_bf16_bits(rng.standard_normal((n, spec.d), dtype=np.float32))


def make_problem(spec: Spec | int) -> Problem:
    if isinstance(spec, int):
        spec = CONFIGS[spec]
    s = spec
    rng = _rng(s.seed, TAG_ROUTER_W)
    router_w = (rng.standard_normal((s.n_experts, s.d)) * 0.02).astype(np.float32)
    gate = ExpertStack(s.fmt_gate_up, s.n_experts, s.f, s.d, s.seed, TAG_GATE)
    up = ExpertStack(s.fmt_gate_up, s.n_experts, s.f, s.d, s.seed, TAG_UP)
    down = ExpertStack(s.fmt_down, s.n_experts, s.d, s.f, s.seed, TAG_DOWN)
    if s.n_shared:
        sg = quant_tensor(s.fmt_shared, s.f_shared, s.d, s.seed, TAG_S_GATE, 0)
        su = quant_tensor(s.fmt_shared, s.f_shared, s.d, s.seed, TAG_S_UP, 0)
        sd = quant_tensor(s.fmt_shared, s.d, s.f_shared, s.seed, TAG_S_DOWN, 0)
    else:
        sg = su = sd = None
    table = tids = None
    if s.hash_vocab:
        table = hash_table(s.hash_vocab, s.n_experts, s.top_k, s.seed)
        tids = _rng(s.seed, TAG_TOKEN_IDS).integers(0, s.hash_vocab, size=s.n_hash).astype(np.int32)
    return Problem(s, router_w, router_bias(s), gate, up, down, sg, su, sd, table,
                   activations(s), tids)
