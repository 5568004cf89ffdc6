"""Seeded synthetic inputs for the verification step.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It draws random numbers and stores them; it holds none of the
verification arithmetic (no softmax, no acceptance rule, no residual). Draft
tokens are drawn with the Gumbel-max construction (the argmax of l/T plus
independent Gumbel noise is an exact sample of softmax(l/T)), so no
normaliser is computed here either.

Every request ``b`` of a workload draws from its own Philox stream, keyed by
``SeedSequence([seed, b])``, so requests can be generated on several threads
and any one request can be regenerated alone. Batch-level draws (the Zipf
permutation) use the key ``SeedSequence([seed, 2**31])``. ``seed`` is
``1000 * config + k``.

Workloads (B requests, gamma draft tokens, vocabulary V):
  1 tiny      B=1,   gamma=4, V=32,     fp32, T=1    target ~ N(0, 2^2)
  2 greedy    B=8,   gamma=5, V=32000,  bf16, T=0    target ~ N(0, 3^2)
  3 sampling  B=64,  gamma=4, V=128256, fp32, T=0.7  N(0, 3^2) + 20 hot tokens
                                                     per row, boosted by +8
  4 mixed     B=256, gamma=8, V=128256, bf16, T in {0, 0.3, 0.7, 1} per request
  5 large     B=512, gamma=7, V=152064, bf16, T=1    N(0, 3^2) + Zipf bias
Draft logits are the target logits of the first gamma positions plus
Gaussian noise (sigma 1, 1, 0.7, U(0.3, 2.0) per request, 1). Draft tokens
are the argmax of the stored draft logits at T = 0 and a draw from
softmax(draft / T) otherwise. Uniforms are binary32 values (x >> 8) * 2^-24.
Logits are generated in binary32 and stored as binary32 or as bfloat16 by
round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    config: int
    name: str
    B: int
    gamma: int
    V: int
    dtype: str  # "f32" or "bf16"
    temperatures: tuple  # values T is drawn from, uniformly per request
    target_sigma: float
    draft_sigma: tuple  # (lo, hi): per-request sigma ~ U(lo, hi); lo == hi fixes it
    hot_tokens: int = 0
    hot_boost: float = 0.0
    zipf_s: float = 0.0
    description: str = field(default="", compare=False)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def scaled(self, B: int) -> "Workload":
        """The same recipe with another batch size (for bounded samples)."""
        return dataclasses.replace(self, B=B)

    def variant(self, **changes) -> "Workload":
        """The same recipe with other fields (e.g. a smaller V for quick checks)."""
        return dataclasses.replace(self, **changes)


WORKLOADS = {
    1: Workload(1, "tiny", 1, 4, 32, "f32", (1.0,), 2.0, (1.0, 1.0),
                description="tiny sampling verify B=1 gamma=4 V=32 fp32 T=1"),
    2: Workload(2, "greedy", 8, 5, 32000, "bf16", (0.0,), 3.0, (1.0, 1.0),
                description="greedy verify B=8 gamma=5 V=32000 bf16 T=0"),
    3: Workload(3, "sampling", 64, 4, 128256, "f32", (0.7,), 3.0, (0.7, 0.7),
                hot_tokens=20, hot_boost=8.0,
                description="sampling verify B=64 gamma=4 V=128256 fp32 T=0.7"),
    4: Workload(4, "mixed", 256, 8, 128256, "bf16", (0.0, 0.3, 0.7, 1.0), 3.0, (0.3, 2.0),
                description="mixed-batch verify B=256 gamma=8 V=128256 bf16 T in {0,.3,.7,1}"),
    5: Workload(5, "large", 512, 7, 152064, "bf16", (1.0,), 3.0, (1.0, 1.0), zipf_s=1.1,
                description="large-vocab verify B=512 gamma=7 V=152064 bf16 T=1"),
}
BY_NAME = {w.name: w for w in WORKLOADS.values()}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> binary32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Batch:
    workload: Workload
    seed: int
    target: np.ndarray       # [B, gamma+1, V] float32 or uint16 (bf16 bits)
    draft: np.ndarray        # [B, gamma, V]
    tokens: np.ndarray       # [B, gamma] int32
    u_accept: np.ndarray     # [B, gamma] float32
    u_sample: np.ndarray     # [B] float32
    temperature: np.ndarray  # [B] float32

    @property
    def B(self):
        return self.target.shape[0]

    def slice(self, lo: int, hi: int) -> "Batch":
        return Batch(self.workload.scaled(hi - lo), self.seed, self.target[lo:hi],
                     self.draft[lo:hi], self.tokens[lo:hi], self.u_accept[lo:hi],
                     self.u_sample[lo:hi], self.temperature[lo:hi])

    def arrays(self):
        return (self.target, self.draft, self.tokens, self.u_accept, self.u_sample,
                self.temperature)


def request_rng(seed: int, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, b])))


def batch_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 2 ** 31])))


def zipf_bias(w: Workload, seed: int) -> np.ndarray | None:
    """Additive bias -s * ln(rank), ranks given by a random permutation."""
    if w.zipf_s == 0.0:
        return None
    perm = batch_rng(seed).permutation(w.V)
    rank = np.empty(w.V, dtype=np.float64)
    rank[perm] = np.arange(1, w.V + 1, dtype=np.float64)
    return (-w.zipf_s * np.log(rank)).astype(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return x.astype(np.float32) if dtype == "f32" else f32_to_bf16_bits(x)


def _stored_values(x: np.ndarray, dtype: str) -> np.ndarray:
    return x if dtype == "f32" else bf16_bits_to_f32(x)


def _gen_request(w: Workload, seed: int, b: int, bias, out: Batch) -> None:
    rng = request_rng(seed, b)
    G, V = w.gamma, w.V
    T = float(w.temperatures[rng.integers(len(w.temperatures))]) if len(w.temperatures) > 1 \
        else float(w.temperatures[0])
    lo, hi = w.draft_sigma
    sigma_d = float(rng.uniform(lo, hi)) if hi > lo else float(lo)
    tgt = rng.standard_normal((G + 1, V), dtype=np.float32)
    tgt *= np.float32(w.target_sigma)
    if w.hot_tokens:
        for i in range(G + 1):
            hot = rng.choice(V, size=w.hot_tokens, replace=False)
            tgt[i, hot] += np.float32(w.hot_boost)
    if bias is not None:
        tgt += bias[None, :]
    noise = rng.standard_normal((G, V), dtype=np.float32)
    noise *= np.float32(sigma_d)
    dft = tgt[:G] + noise
    out.target[b] = _store(tgt, w.dtype)
    out.draft[b] = _store(dft, w.dtype)
    dvals = _stored_values(out.draft[b], w.dtype).astype(np.float64)
    if T == 0.0:
        out.tokens[b] = np.argmax(dvals, axis=1)
    else:
        gumbel = -np.log(-np.log(rng.random((G, V))))
        out.tokens[b] = np.argmax(dvals / T + gumbel, axis=1)
    out.u_accept[b] = rng.random(G, dtype=np.float32)
    out.u_sample[b] = rng.random(dtype=np.float32)
    out.temperature[b] = np.float32(T)


def generate(w: Workload | int | str, k: int = 0, B: int | None = None,
             threads: int | None = None, seed: int | None = None) -> Batch:
    """Generate workload ``w`` (a Workload, its config number or its name) with
    seed ``1000 * config + k`` (or ``seed``); ``B`` overrides the batch size
    (requests 0..B-1 of the same streams)."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    elif isinstance(w, str):
        w = BY_NAME[w]
    if B is not None:
        w = w.scaled(B)
    seed = 1000 * w.config + k if seed is None else seed
    store_dt = np.float32 if w.dtype == "f32" else np.uint16
    out = Batch(w, seed,
                np.empty((w.B, w.gamma + 1, w.V), dtype=store_dt),
                np.empty((w.B, w.gamma, w.V), dtype=store_dt),
                np.empty((w.B, w.gamma), dtype=np.int32),
                np.empty((w.B, w.gamma), dtype=np.float32),
                np.empty((w.B,), dtype=np.float32),
                np.empty((w.B,), dtype=np.float32))
    bias = zipf_bias(w, seed)
    threads = max(1, min(threads or os.cpu_count() or 1, w.B))
    if threads == 1:
        for b in range(w.B):
            _gen_request(w, seed, b, bias, out)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda b: _gen_request(w, seed, b, bias, out), range(w.B)))
    return out


# ---------------------------------------------------------------- token histories

@dataclass
class Histories:
    """Token histories for the n-gram proposer and the commit step."""
    token_buf: np.ndarray  # [B, max_len] int32, padding 0
    seq_lens: np.ndarray   # [B] int32


def histories(B: int, max_len: int, lengths=(256, 4096), vocab: int = 32000, copy_prob: float = 0.5,
              span=(4, 32), seed: int = 0) -> Histories:
    """Synthetic histories shaped like the workloads n-gram lookup targets
    (summaries, extraction, code rewriting, RAG): each request draws a length
    L ~ U[lengths], a random prefix of L // 4 tokens (the prompt), then extends
    it in spans: with probability ``copy_prob`` a span copies tokens from a
    random earlier position, otherwise it is fresh random tokens. Span lengths
    ~ U[span]. Request b uses the Philox stream SeedSequence([seed, b])."""
    buf = np.zeros((B, max_len), dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    for b in range(B):
        rng = request_rng(seed, b)
        L = int(min(max_len, rng.integers(lengths[0], lengths[1] + 1)))
        h = list(rng.integers(0, vocab, max(1, L // 4)))
        while len(h) < L:
            s = int(rng.integers(span[0], span[1] + 1))
            if rng.random() < copy_prob and len(h) > 1:
                j = int(rng.integers(0, len(h) - 1))
                h.extend(h[j:j + s])
            else:
                h.extend(rng.integers(0, vocab, s))
        buf[b, :L] = np.asarray(h[:L], dtype=np.int32)
        lens[b] = L
    return Histories(buf, lens)


def tree_parents(B: int, gamma: int, seed: int = 5) -> np.ndarray:
    """Candidate-tree shapes [B, gamma] for a batch (parent of node j at
    j - 1): node j's parent is node j - 1 half the time (a chain, whose
    tokens, the workload's draft tokens, stay plausible), else uniform over
    0..j-1 (a branch). One numpy Generator seeded with ``seed``, drawn in
    request then node order."""
    rng = np.random.default_rng(seed)
    return np.array([[j - 1 if rng.random() < 0.5 else rng.integers(0, j) for j in range(1, gamma + 1)]
                     for _ in range(B)], np.int32)
