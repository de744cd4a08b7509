"""Seeded synthetic inputs for the verification step.

This module produces logits, draft tokens, uniforms and draft trees with the
shapes and value distributions of the five benchmark workloads.  It holds none
of the verification arithmetic: no softmax, no accept ratio, no residual.  The
drafter is simulated by Gumbel-max sampling (argmax of logits/T plus Gumbel
noise), which draws from softmax(logits/T) without ever forming it, and the
tree generator only needs the row argmax of the target logits to plant
matching tokens.

Both the CUDA path and the fp64 oracle are fed from here; nothing here
depends on either of them.

Workloads (B sequences, gamma drafts, V vocabulary, T temperature):

  chain-small   B=1   gamma=4 V=1000   fp32  target N(0,2^2), draft = target + N(0,0.5^2), T=1, seed 0
  chain-b8      B=8   gamma=7 V=151936 bf16  target N(0,3^2) + 20 boosted (+8) per row,
                                               draft = target + N(0,1^2), T=1, seed 1
  chain-b64     B=64  gamma=7 V=151936 bf16  as chain-b8, T=0.6, draft noise sigma_b in
                                               (0.25, 1, 4)[b mod 3], seed 2
  chain-b256    B=256 gamma=4 V=128256 fp32  target N(0,2.5^2), draft = 0.8 target + 0.2 N(0,2.5^2),
                                               T=1, seed 3
  tree-b32      B=32  N=36    V=151936 bf16  node logits as chain-b8's target, tree = root +
                                               7-node main chain + 4 single-node branches at each
                                               of depths 1..7, node token = argmax of the parent's
                                               row with probability 0.7, seed 4

  ngram-b64     B=64  token streams of 32768..65536 tokens (n_max 65536), V=151936: Zipf-like
                tokens with repeated spans (a block copies an earlier span with
                probability 0.35), the last 32 tokens copied from earlier in the
                stream for 70% of the sequences (a lexical hit), query w=3,
                draft L=7, up to 64 matches kept, seed 5

  cosine-b64    B=64  windows of W=240 hidden states (30 forward steps of 8 positions),
                d=4096 (Qwen3-8B's hidden size), bf16: N(0,1) rows and query; half
                the sequences hold 3 near copies of the query (noise sigma 0.2,
                0.5, 1.0); delta=4, seed 6

The vocabulary 151936 is Qwen3's and gamma=7 matches the K=7 of the DLite
reading notes (section "Experimental setup").  Every workload can be shrunk
(B, gamma, V overrides) with the same recipe for parity tests.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "WORKLOADS", "ChainInputs", "TreeInputs", "NgramInputs", "CosineInputs", "make_chain",
    "make_tree", "make_ngram", "make_cosine",
    "tree_topology", "to_bf16_exact", "gumbel_argmax",
]


@dataclasses.dataclass(frozen=True)
class ChainWorkload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str          # "f32" or "bf16"
    T: float
    seed: int
    family: str         # "gauss" (chain-small), "boosted" (chain-b8/b64), "mixed" (chain-b256)
    target_sigma: float
    draft_sigma: tuple  # per-sequence draft noise (cycled over b)


@dataclasses.dataclass(frozen=True)
class TreeWorkload:
    name: str
    B: int
    N: int
    V: int
    dtype: str
    seed: int
    depth: int          # main-chain length
    branches: int       # single-node branches per depth
    match_prob: float


@dataclasses.dataclass(frozen=True)
class NgramWorkload:
    name: str
    B: int
    n_max: int
    n_min: int
    V: int
    w: int
    L: int
    max_matches: int
    seed: int
    copy_prob: float     # a block repeats an earlier span
    hit_prob: float      # the stream ends with a copied span


@dataclasses.dataclass(frozen=True)
class CosineWorkload:
    name: str
    B: int
    W: int
    d: int
    dtype: str
    delta: int
    seed: int


WORKLOADS = {
    "chain-small": ChainWorkload("chain-small", 1, 4, 1000, "f32", 1.0, 0, "gauss", 2.0, (0.5,)),
    "chain-b8": ChainWorkload("chain-b8", 8, 7, 151936, "bf16", 1.0, 1, "boosted", 3.0, (1.0,)),
    "chain-b64": ChainWorkload("chain-b64", 64, 7, 151936, "bf16", 0.6, 2, "boosted", 3.0,
                               (0.25, 1.0, 4.0)),
    "chain-b256": ChainWorkload("chain-b256", 256, 4, 128256, "f32", 1.0, 3, "mixed", 2.5, (2.5,)),
    "tree-b32": TreeWorkload("tree-b32", 32, 36, 151936, "bf16", 4, 7, 4, 0.7),
    "ngram-b64": NgramWorkload("ngram-b64", 64, 65536, 32768, 151936, 3, 7, 64, 5, 0.35, 0.7),
    "cosine-b64": CosineWorkload("cosine-b64", 64, 240, 4096, "bf16", 4, 6),
}


@dataclasses.dataclass
class CosineInputs:
    hidden: np.ndarray     # [B, W, d] float32 (bf16-exact for dtype "bf16")
    query: np.ndarray      # [B, d]
    positions: np.ndarray  # [B, W] int32 context positions of the window rows
    delta: int
    dtype: str
    name: str


def make_cosine(name: str = "cosine-b64", *, B: Optional[int] = None, W: Optional[int] = None,
                d: Optional[int] = None, seed: Optional[int] = None) -> CosineInputs:
    """Windows of hidden states for the semantic fallback: N(0,1) rows and
    query; every even sequence plants 3 near copies of its query (noise sigma
    0.2, 0.5, 1.0) at random window rows.  Row j of a window is context
    position len_b - W + j for a context length len_b in [W, 65536]."""
    wl = WORKLOADS[name]
    assert isinstance(wl, CosineWorkload), name
    B = wl.B if B is None else B
    W = wl.W if W is None else W
    d = wl.d if d is None else d
    seed = wl.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((B, W, d), dtype=np.float32)
    q = rng.standard_normal((B, d), dtype=np.float32)
    for b in range(0, B, 2):
        rows = rng.choice(W, size=min(3, W), replace=False)
        for r, sig in zip(rows, (0.2, 0.5, 1.0)):
            H[b, r] = q[b] + np.float32(sig) * rng.standard_normal(d, dtype=np.float32)
    H = _round(H, wl.dtype)
    q = _round(q, wl.dtype)
    lens = rng.integers(W, 65537, size=B)
    pos = (lens[:, None] - W + np.arange(W)[None, :]).astype(np.int32)
    return CosineInputs(H, q, pos, wl.delta, wl.dtype, name)


@dataclasses.dataclass
class NgramInputs:
    tokens: np.ndarray     # [B, n_max] int32 (zero past each length)
    lengths: np.ndarray    # [B] int32
    w: int
    L: int
    max_matches: int
    name: str


def make_ngram(name: str = "ngram-b64", *, B: Optional[int] = None, n_max: Optional[int] = None,
               n_min: Optional[int] = None, seed: Optional[int] = None) -> NgramInputs:
    """Token streams for lexical retrieval: Zipf-like tokens (80% from 2000
    frequent ids, 20% uniform over V) in blocks of 64..512 tokens, each block
    copying an earlier span of the same stream with probability copy_prob;
    with probability hit_prob the stream ends with a 32-token copy of an
    earlier span, so its last w tokens occur earlier."""
    wl = WORKLOADS[name]
    assert isinstance(wl, NgramWorkload), name
    B = wl.B if B is None else B
    n_max = wl.n_max if n_max is None else n_max
    n_min = min(wl.n_min, n_max) if n_min is None else n_min
    seed = wl.seed if seed is None else seed
    ss = np.random.SeedSequence(seed).spawn(3)
    r_len, r_tok, r_blk = (np.random.default_rng(x) for x in ss)
    lengths = r_len.integers(n_min, n_max + 1, size=B).astype(np.int32)
    freq = (r_tok.permutation(wl.V)[:2000]).astype(np.int32)
    ranks = 1.0 / np.arange(1, 2001) ** 1.1
    ranks /= ranks.sum()
    tokens = np.zeros((B, n_max), np.int32)
    for b in range(B):
        n = int(lengths[b])
        out = np.empty(n, np.int32)
        pos = 0
        while pos < n:
            blk = min(int(r_blk.integers(64, 513)), n - pos)
            if pos > blk and r_blk.random() < wl.copy_prob:
                src = int(r_blk.integers(0, pos - blk + 1))
                out[pos:pos + blk] = out[src:src + blk]
            else:
                fr = r_tok.random(blk) < 0.8
                out[pos:pos + blk] = np.where(fr, freq[r_tok.choice(2000, blk, p=ranks)],
                                              r_tok.integers(0, wl.V, blk)).astype(np.int32)
            pos += blk
        if n > 128 and r_blk.random() < wl.hit_prob:
            src = int(r_blk.integers(0, n - 64))
            out[n - 32:] = out[src:src + 32]
        tokens[b, :n] = out
    return NgramInputs(tokens, lengths, wl.w, wl.L, wl.max_matches, name)

BOOSTED_PER_ROW = 20
BOOST = 8.0


@dataclasses.dataclass
class ChainInputs:
    """One verification batch.  Logit arrays are float32; for dtype "bf16"
    every value is exactly representable in bfloat16."""
    target: np.ndarray        # [B, gamma+1, V] float32
    draft: np.ndarray         # [B, gamma, V]   float32
    draft_tokens: np.ndarray  # [B, gamma] int32, sampled from softmax(draft/T)
    greedy_tokens: np.ndarray # [B, gamma] int32, argmax of each draft row
    uniforms: np.ndarray      # [B, gamma+1] float32 in [0, 1)
    T: float
    dtype: str
    B: int
    gamma: int
    V: int
    name: str

    def logit_bytes(self, greedy: bool = False) -> int:
        elt = 2 if self.dtype == "bf16" else 4
        rows = self.B * (self.gamma + 1) + (0 if greedy else self.B * self.gamma)
        return rows * self.V * elt


@dataclasses.dataclass
class TreeInputs:
    target: np.ndarray        # [B, N, V] float32 (bf16-exact for dtype "bf16")
    node_tokens: np.ndarray   # [B, N] int32 (node 0 holds -1: the root carries no draft)
    parents: np.ndarray       # [B, N] int32, parents[:, 0] = -1, parents[:, n] < n
    dtype: str
    B: int
    N: int
    V: int
    name: str

    def logit_bytes(self) -> int:
        elt = 2 if self.dtype == "bf16" else 4
        return self.B * self.N * self.V * elt


def to_bf16_exact(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even) and return
    them as float32.  Finite inputs only (|x| < 2^128, so the 32-bit
    arithmetic below cannot wrap)."""
    y = np.array(x, dtype=np.float32, copy=True, order="C")
    b = y.reshape(-1).view(np.uint32)
    step = 1 << 22
    for i in range(0, b.size, step):
        c = b[i:i + step]
        c += np.uint32(0x7FFF) + ((c >> np.uint32(16)) & np.uint32(1))
        c &= np.uint32(0xFFFF0000)
    return y


def gumbel_argmax(rng: np.random.Generator, logits: np.ndarray, T: float) -> np.ndarray:
    """Draw one index per row of `logits` ([R, V]) from softmax(logits/T) by
    the Gumbel-max construction.  Rows are processed one at a time to bound
    memory."""
    out = np.empty(logits.shape[0], dtype=np.int32)
    for r in range(logits.shape[0]):
        u = rng.random(logits.shape[1])                 # float64 in [0, 1)
        g = -np.log(-np.log(np.maximum(u, 1e-300)))
        out[r] = int(np.argmax(logits[r].astype(np.float64) / T + g))
    return out


def distinct_indices(rng: np.random.Generator, V: int, k: int) -> np.ndarray:
    """k distinct indices uniform over [0, V) (without replacement), in draw order."""
    if 2 * k > V:
        return rng.permutation(V)[:k]
    out, seen = [], set()
    while len(out) < k:
        for j in rng.integers(0, V, 2 * k):
            j = int(j)
            if j not in seen:
                seen.add(j)
                out.append(j)
                if len(out) == k:
                    break
    return np.array(out, dtype=np.int64)


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_exact(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def make_chain(name: str, *, B: Optional[int] = None, gamma: Optional[int] = None,
               V: Optional[int] = None, seed: Optional[int] = None,
               T: Optional[float] = None) -> ChainInputs:
    """Generate the chain workload `name` (optionally shrunk)."""
    w = WORKLOADS[name]
    assert isinstance(w, ChainWorkload), name
    B = w.B if B is None else B
    gamma = w.gamma if gamma is None else gamma
    V = w.V if V is None else V
    seed = w.seed if seed is None else seed
    T = w.T if T is None else T
    s_logits, s_noise, s_draft, s_unif = np.random.SeedSequence(seed).spawn(4)
    r_logits = np.random.default_rng(s_logits)
    r_noise = np.random.default_rng(s_noise)
    r_draft = np.random.default_rng(s_draft)
    r_unif = np.random.default_rng(s_unif)

    zt = r_logits.standard_normal((B, gamma + 1, V), dtype=np.float32)
    zt *= np.float32(w.target_sigma)
    if w.family == "boosted":
        k = min(BOOSTED_PER_ROW, V)
        for b in range(B):
            for i in range(gamma + 1):
                idx = distinct_indices(r_logits, V, k)
                zt[b, i, idx] += np.float32(BOOST)
    zt = _round(zt, w.dtype)

    noise = r_noise.standard_normal((B, gamma, V), dtype=np.float32)
    if w.family == "mixed":
        # draft = 0.8 * target + 0.2 * independent N(0, sigma^2)
        zd = np.float32(0.8) * zt[:, :gamma, :] + np.float32(0.2 * w.draft_sigma[0]) * noise
    else:
        sig = np.array([w.draft_sigma[b % len(w.draft_sigma)] for b in range(B)],
                       dtype=np.float32)[:, None, None]
        zd = zt[:, :gamma, :] + sig * noise
    del noise
    zd = _round(zd, w.dtype)

    if gamma > 0:
        tok = gumbel_argmax(r_draft, zd.reshape(B * gamma, V), T).reshape(B, gamma)
        gtok = np.argmax(zd, axis=2).astype(np.int32)
    else:
        tok = np.zeros((B, 0), np.int32)
        gtok = np.zeros((B, 0), np.int32)
    u = r_unif.random((B, gamma + 1), dtype=np.float32)
    return ChainInputs(np.ascontiguousarray(zt), np.ascontiguousarray(zd), tok, gtok, u,
                       float(T), w.dtype, B, gamma, V, name)


def tree_topology(depth: int, branches: int) -> np.ndarray:
    """Parent array of the draft tree: node 0 is the root (the last verified
    token), nodes 1..depth form the main chain (parent of node d is d-1), and
    node depth+1+branches*(d-1)+k (k < branches) is a single-node branch that
    is a sibling of main-chain node d (parent d-1).  depth=7, branches=4 gives
    the 36-node tree of the tree-b32 workload."""
    n = 1 + depth + depth * branches
    par = np.empty(n, dtype=np.int32)
    par[0] = -1
    for d in range(1, depth + 1):
        par[d] = d - 1
        for k in range(branches):
            par[depth + 1 + branches * (d - 1) + k] = d - 1
    return par


def make_tree(name: str = "tree-b32", *, B: Optional[int] = None, V: Optional[int] = None,
              seed: Optional[int] = None, depth: Optional[int] = None,
              branches: Optional[int] = None, match_prob: Optional[float] = None) -> TreeInputs:
    w = WORKLOADS[name]
    assert isinstance(w, TreeWorkload), name
    B = w.B if B is None else B
    V = w.V if V is None else V
    seed = w.seed if seed is None else seed
    depth = w.depth if depth is None else depth
    branches = w.branches if branches is None else branches
    mp = w.match_prob if match_prob is None else match_prob
    par = tree_topology(depth, branches)
    N = par.shape[0]
    s_logits, s_tok = np.random.SeedSequence(seed).spawn(2)
    r_logits = np.random.default_rng(s_logits)
    r_tok = np.random.default_rng(s_tok)
    z = r_logits.standard_normal((B, N, V), dtype=np.float32) * np.float32(3.0)
    k = min(BOOSTED_PER_ROW, V)
    for b in range(B):
        for n in range(N):
            idx = distinct_indices(r_logits, V, k)
            z[b, n, idx] += np.float32(BOOST)
    z = _round(z, w.dtype)
    g = np.argmax(z, axis=2)                      # planted-match reference per node row
    tok = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for n in range(1, N):
            gp = int(g[b, par[n]])
            if r_tok.random() < mp or V == 1:
                tok[b, n] = gp
            else:
                r = int(r_tok.integers(0, V - 1))
                tok[b, n] = r + 1 if r >= gp else r
    parents = np.ascontiguousarray(np.broadcast_to(par, (B, N)), dtype=np.int32)
    return TreeInputs(np.ascontiguousarray(z), tok, parents, w.dtype, B, N, V, name)
