"""Seeded synthetic inputs for the speculative-decoding verification step.

This module is shared by the tests, the smoke check and the benchmark, and
by both sides of every parity test (the CPU oracle and the GPU library).  It
holds none of the verification arithmetic: no softmax, no normaliser, no
acceptance test, no residual and no inverse CDF.  It draws logits, draft
tokens, candidate trees and uniforms, nothing else.

Workloads (the five verification batches the library is measured on):

  c1  B=1 (replicated into independent steps), k=3, V=32, fp32.  Target
      logits ~ N(0, 2^2), drawn once; draft = target + N(0, 0.7^2); T=1, no
      top-p.  Each step has fresh draft tokens x~_i ~ q_i and k+1 uniforms.
  c2  B=8, k=4, V=32000, fp32.  Logits = -1.1*log(rank) over a random
      permutation of the vocabulary, plus N(0, 1.5^2); draft = target +
      N(0, 1^2); T=0.8; stochastic and greedy.
  c3  B=64, k=5, V=151936, bf16.  Same generator; draft noise sigma_b in
      {0.3, 1.0, 3.0} by b mod 3; T=1.
  c4  B=128, k=3, V=128256, bf16.  Same generator, draft noise 0.8, T=0.7,
      top-p 0.95 on target and draft.
  c5  greedy tree: B=16, 85 nodes (branching 4 at depths 1-3), V=32000,
      fp32.  Each node's 4 children carry 4 distinct tokens drawn without
      replacement from the top-8 of (the node's target row + N(0, 1^2)).

Draft tokens are drawn by the Gumbel-max rule, argmax_x (l(x)/T + G(x))
with G = -log(-log U), which samples softmax(l/T) without forming it.  With
top-p on (c4) the drafter restricts the draw to the 16 largest draft logits,
a top-16 drafter; on c4 one draft in 384 lands outside its row's 0.95-nucleus
(a row whose nucleus is smaller than 16 tokens), where q = 0 and the accept
rule's q = 0 case applies.  bf16 logits are made by round-to-nearest-even from fp32 and stored as
uint16 bit patterns; both sides of a parity test read the same bits.
Uniforms are fp32 multiples of 2^-24 in [0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32, BF16 = "f32", "bf16"
STOCHASTIC, GREEDY = "stochastic", "greedy"


# ------------------------------------------------------------------ storage

def to_bf16_bits(x):
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    bits = rounded.astype(np.uint16)
    nan = np.isnan(np.asarray(x, np.float32))
    if nan.any():
        bits[nan] = 0x7FC0
    return bits


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_f32(logits):
    """Storage array (float32, or uint16 bf16 bits) -> float32 values."""
    return bf16_bits_to_f32(logits) if logits.dtype == np.uint16 else logits


# ------------------------------------------------------------------ drawing

def uniforms(rng, shape):
    """fp32 uniforms on the grid j * 2^-24, j in [0, 2^24): exactly in [0, 1)."""
    return (rng.integers(0, 1 << 24, size=shape, dtype=np.int64) * (1.0 / (1 << 24))).astype(np.float32)


def zipf_gauss(rng, rows, V, sigma):
    """[rows, V] fp32 logits: -1.1*log(rank(v)) + N(0, sigma^2), with a fresh
    random rank permutation (ranks 1..V) per row."""
    log_rank = np.log(np.arange(1, V + 1, dtype=np.float64))
    out = np.empty((rows, V), np.float32)
    for r in range(rows):
        perm = rng.permutation(V)
        out[r] = -1.1 * log_rank[perm] + rng.normal(0.0, sigma, V)
    return out


def _gumbel(rng, shape):
    u = rng.random(shape)
    u = np.where(u > 0.0, u, np.finfo(np.float64).tiny)
    return -np.log(-np.log(u))


def gumbel_draw(rng, logits_f32, T, top=None):
    """Draft tokens by Gumbel-max over the last axis of [..., V] logits.

    top=None samples softmax(l/T) exactly; top=m restricts the draw to the m
    largest logits of each row (a top-m drafter)."""
    l = np.asarray(logits_f32)
    V = l.shape[-1]
    flat = l.reshape(-1, V)
    R = flat.shape[0]
    out = np.empty(R, np.int32)
    if top is not None:
        cand = np.argpartition(-flat, top - 1, axis=1)[:, :top]
        vals = np.take_along_axis(flat, cand, 1).astype(np.float64)
        pick = np.argmax(vals / T + _gumbel(rng, vals.shape), axis=1)
        out[:] = cand[np.arange(R), pick]
    else:
        step = max(1, (1 << 22) // V)
        for s in range(0, R, step):
            blk = flat[s:s + step].astype(np.float64)
            out[s:s + step] = np.argmax(blk / T + _gumbel(rng, blk.shape), axis=1)
    return out.reshape(l.shape[:-1])


def draft_prob_rows(rng, target_f32, k, favoured=64, boost=2e5, alpha=0.3):
    """Draft probability rows [B, k, V] fp32 and tokens drawn from them, for
    the form of the step that takes the draft as probabilities.

    Input synthesis only: each row is Gamma(alpha) noise, multiplied on the
    `favoured` largest target logits of the same position by boost / r^1.5
    (r = 1, 2, ... their rank), so that drafts agree with the target often
    enough to be accepted; then scaled to sum 1 in fp64 and stored as fp32.
    Each draft token is drawn from its stored row with numpy's categorical
    sampler."""
    t = np.asarray(target_f32)
    B, _, V = t.shape
    q = np.empty((B, k, V), np.float32)
    toks = np.empty((B, k), np.int32)
    m = min(favoured, V)
    ramp = boost / np.arange(1, m + 1, dtype=np.float64) ** 1.5
    for b in range(B):
        for i in range(k):
            w = rng.gamma(alpha, 1.0, V)
            top = np.argpartition(-t[b, i], m - 1)[:m]
            top = top[np.argsort(-t[b, i][top], kind="stable")]
            w[top] *= ramp
            q[b, i] = w / w.sum()
            row = q[b, i].astype(np.float64)
            toks[b, i] = rng.choice(V, p=row / row.sum())
    return q, toks


# ---------------------------------------------------------------- workloads

@dataclass
class Chain:
    """One chain-verification batch (inputs for spec_verify_sample)."""
    name: str
    B: int
    k: int
    V: int
    dtype: str
    T: float
    top_p: float
    target: np.ndarray        # [B, k+1, V] float32 or uint16 (bf16 bits)
    draft: np.ndarray         # [B, k, V]
    draft_tokens: np.ndarray  # [B, k] int32
    uniforms: np.ndarray      # [B, k+1] float32
    modes: tuple = (STOCHASTIC,)

    def logit_bytes(self, mode=STOCHASTIC):
        esz = 4 if self.dtype == F32 else 2
        rows = self.B * (2 * self.k + 1 if mode == STOCHASTIC else self.k + 1)
        return rows * self.V * esz


@dataclass
class Tree:
    """One greedy tree-verification batch (inputs for spec_verify_tree)."""
    name: str
    B: int
    N: int
    V: int
    D: int
    dtype: str
    target: np.ndarray        # [B, N, V]
    parents: np.ndarray       # [N] int32, parents[0] = -1
    node_tokens: np.ndarray   # [B, N] int32
    modes: tuple = field(default=("tree",))

    def logit_bytes(self, mode="tree"):
        return self.B * self.N * self.V * (4 if self.dtype == F32 else 2)


def _streams(seed):
    s = np.random.SeedSequence(seed).spawn(3)
    return tuple(np.random.default_rng(x) for x in s)


def _store(x, dtype):
    return to_bf16_bits(x) if dtype == BF16 else np.ascontiguousarray(x, np.float32)


def zipf_chain(name, B, k, V, dtype, T, top_p, sigma_target, sigma_draft, seed,
               drafter_top=None, modes=(STOCHASTIC,)):
    """Zipf+Gaussian chain batch; sigma_draft is a number or a per-b callable."""
    r_logit, r_draft, r_unif = _streams(seed)
    tgt = zipf_gauss(r_logit, B * (k + 1), V, sigma_target).reshape(B, k + 1, V)
    drf = np.empty((B, k, V), np.float32)
    for b in range(B):
        s = sigma_draft(b) if callable(sigma_draft) else sigma_draft
        drf[b] = tgt[b, :k] + r_logit.normal(0.0, s, (k, V)).astype(np.float32)
    target = _store(tgt, dtype)
    draft = _store(drf, dtype)
    toks = gumbel_draw(r_draft, as_f32(draft), T, top=drafter_top).astype(np.int32)
    return Chain(name, B, k, V, dtype, T, top_p, target, draft, toks,
                 uniforms(r_unif, (B, k + 1)), modes)


def c1(steps=100_000, seed=0):
    """Tiny exactness case, replicated into `steps` independent verify steps."""
    r_logit, r_draft, r_unif = _streams(seed)
    k, V = 3, 32
    tgt = r_logit.normal(0.0, 2.0, (1, k + 1, V)).astype(np.float32)
    drf = (tgt[:, :k] + r_logit.normal(0.0, 0.7, (1, k, V))).astype(np.float32)
    target = np.ascontiguousarray(np.broadcast_to(tgt, (steps, k + 1, V)))
    draft = np.ascontiguousarray(np.broadcast_to(drf, (steps, k, V)))
    toks = gumbel_draw(r_draft, draft, 1.0).astype(np.int32)
    return Chain("c1", steps, k, V, F32, 1.0, 1.0, target, draft, toks,
                 uniforms(r_unif, (steps, k + 1)), (STOCHASTIC,))


def c2(seed=2):
    return zipf_chain("c2", 8, 4, 32000, F32, 0.8, 1.0, 1.5, 1.0, seed,
                      modes=(STOCHASTIC, GREEDY))


def c3(seed=3, B=64, V=151936):
    return zipf_chain("c3", B, 5, V, BF16, 1.0, 1.0, 1.5,
                      lambda b: (0.3, 1.0, 3.0)[b % 3], seed)


def c4(seed=4, B=128, V=128256):
    """The top-p batch.  Its draft tokens come from a top-16 drafter over the
    draft logits at temperature T (Gumbel-max restricted to the 16 largest),
    not from the processed q (temperature and top-p 0.95): this module holds
    none of the method's arithmetic, and top-p is part of it.  So the draws
    are not x~ ~ q: about 1 in 384 lands on a token outside the draft's
    nucleus, where q = 0 (every such draft is then accepted only if p > 0
    there, by the ratio rule's q = 0 case).  Parity is unaffected (the step
    is a fixed function of its inputs), but c4's acceptance statistics do
    not describe the method's own x~ ~ q setting."""
    return zipf_chain("c4", B, 3, V, BF16, 0.7, 0.95, 1.5, 0.8, seed, drafter_top=16)


def bfs_parents(branching=4, depth=3):
    """Parent array of a full tree flattened breadth-first; parents[0] = -1."""
    parents, level = [-1], [0]
    for _ in range(depth):
        nxt = []
        for p in level:
            for _ in range(branching):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    return np.asarray(parents, np.int32)


def c5(seed=5, B=16, V=32000, branching=4, depth=3, dtype=F32):
    r_logit, r_draft, _ = _streams(seed)
    parents = bfs_parents(branching, depth)
    N = parents.shape[0]
    tgt = zipf_gauss(r_logit, B * N, V, 1.5).reshape(B, N, V)
    target = _store(tgt, dtype)
    tvals = as_f32(target)
    node_tokens = np.zeros((B, N), np.int32)
    children = {}
    for n in range(1, N):
        children.setdefault(int(parents[n]), []).append(n)
    for b in range(B):
        for p, kids in children.items():
            noisy = tvals[b, p].astype(np.float64) + r_draft.normal(0.0, 1.0, V)
            top8 = np.argpartition(-noisy, 7)[:8]
            pick = r_draft.choice(top8, size=len(kids), replace=False)
            node_tokens[b, kids] = pick
    return Tree("c5", B, N, V, depth, dtype, target, parents, node_tokens)


@dataclass
class SampledTree:
    """One stochastic tree-verification batch (spec_verify_tree_sample)."""
    name: str
    B: int
    N: int
    V: int
    D: int
    dtype: str
    T: float
    target: np.ndarray        # [B, N, V]
    draft: np.ndarray         # [B, N, V]: row n drew node n's children
    parents: np.ndarray       # [N] int32
    node_tokens: np.ndarray   # [B, N] int32
    uniforms: np.ndarray      # [B, N] float32: 0 the final draw, c node c's test

    def logit_bytes(self):
        return 2 * self.B * self.N * self.V * (4 if self.dtype == F32 else 2)


def c5s(seed=55, B=16, V=32000, branching=4, depth=3, dtype=F32, T=1.0, noise=1.0):
    """c5's tree shape and target generator, sampled: draft = target + N(0,
    noise^2); every node's children drawn independently (Gumbel-max over
    draft row / T) from its draft row; uniforms for every node."""
    r_logit, r_draft, r_u = _streams(seed)
    parents = bfs_parents(branching, depth)
    N = parents.shape[0]
    tgt = zipf_gauss(r_logit, B * N, V, 1.5).reshape(B, N, V)
    drf = (tgt + r_draft.normal(0.0, noise, tgt.shape)).astype(np.float32)
    node_tokens = np.zeros((B, N), np.int32)
    par = parents.astype(np.int64)
    for n in range(1, N):
        node_tokens[:, n] = gumbel_draw(r_draft, drf[:, par[n]], T)
    return SampledTree("c5s", B, N, V, depth, dtype, T, _store(tgt, dtype), _store(drf, dtype),
                       parents, node_tokens, uniforms(r_u, (B, N)))


CONFIGS = {"c1": c1, "c2": c2, "c3": c3, "c4": c4, "c5": c5}
