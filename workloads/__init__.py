"""Seeded synthetic inputs for tree-attention speculative verification.

This module only *draws* inputs: trees (parent arrays), draft tokens, query /
key / value tensors, paged KV pools with block tables, and target logits with a
planted greedy path.  It holds none of the method's arithmetic: it builds no
ancestry masks, computes no attention, and runs no acceptance walk.  Both the
oracle (``oracle/``) and the CUDA path consume what it returns, so it is the one
piece of code the two sides share.

Every random draw goes through numpy's PCG64 with a ``SeedSequence`` keyed on
(seed, tag, chunk), so the same call returns bit-identical arrays on x86 and
Arm hosts, whatever the thread count.

bf16 tensors are returned as their raw 16-bit patterns (``uint16``), rounded
from fp32 with round-to-nearest-even; the GPU side views them as bfloat16 and
the oracle widens them to fp64 exactly.

The five named workloads (``c1`` … ``c5``) follow the shapes, sizes and tree
structures listed for the verification pass being modelled; the tree shapes and
planting rules that the workload list leaves open are chosen here and stated
on each builder.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_CHUNK = 1 << 22          # elements per independently seeded chunk
_POOL: Optional[ThreadPoolExecutor] = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _seedseq(seed: int, tag: str) -> np.random.SeedSequence:
    return np.random.SeedSequence([int(seed) & 0xFFFFFFFF, *tag.encode()])


def rng(seed: int, tag: str) -> np.random.Generator:
    """A PCG64 generator for one named stream of draws."""
    return np.random.Generator(np.random.PCG64(_seedseq(seed, tag)))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_f32(seed: int, tag: str, shape) -> np.ndarray:
    """N(0,1) fp32 of the given shape, drawn in independently seeded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    nchunks = max(1, -(-n // _CHUNK))
    kids = _seedseq(seed, tag).spawn(nchunks)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(kids[c]))
        g.standard_normal(out=out[lo:hi], dtype=np.float32)

    list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


def normal_bf16(seed: int, tag: str, shape, row_scale: Optional[np.ndarray] = None) -> np.ndarray:
    """N(0,1) drawn in fp32, optionally scaled per row (last axis = row), cast to bf16 bits."""
    x = normal_f32(seed, tag, shape)
    if row_scale is not None:
        x *= row_scale.reshape(row_scale.shape + (1,)).astype(np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.size, np.uint16)
    nchunks = max(1, -(-flat.size // _CHUNK))

    def conv(c):
        lo, hi = c * _CHUNK, min(flat.size, (c + 1) * _CHUNK)
        out[lo:hi] = bf16_bits(flat[lo:hi])

    list(_pool().map(conv, range(nchunks)))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# tree shapes
# ----------------------------------------------------------------------------

def tree_worked_example() -> np.ndarray:
    """The five-node demo tree of the news article's code listing: root 0 with
    children 1 and 2; node 3 under 1; node 4 under 2 (breadth-first order)."""
    return np.array([-1, 0, 0, 1, 2], np.int32)


def tree_random_levels(g: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """A random n-node tree whose deepest level index is ``max_depth``.

    Every non-root node gets a depth: one node is forced onto each level
    1..max_depth so the depth is reached, the rest draw their level uniformly
    from [1, max_depth].  Nodes are then numbered level by level (breadth-first
    order) and each node's parent is drawn uniformly from the nodes one level
    up.  Parents therefore always precede children.
    """
    if n < 1:
        raise ValueError("n >= 1")
    if n == 1:
        return np.array([-1], np.int32)
    max_depth = min(max_depth, n - 1)
    levels = list(range(1, max_depth + 1))
    levels += list(g.integers(1, max_depth + 1, size=n - 1 - max_depth))
    levels = np.sort(np.array([0] + levels, np.int64), kind="stable")
    parent = np.full(n, -1, np.int32)
    first = {}
    for i, d in enumerate(levels):
        first.setdefault(int(d), []).append(i)
    for i in range(1, n):
        cands = first[int(levels[i]) - 1]
        parent[i] = cands[int(g.integers(0, len(cands)))]
    return parent


def tree_from_widths(widths) -> np.ndarray:
    """A fixed tree from per-depth branching widths [w1, w2, ...].

    The root has w1 children.  For each deeper level d >= 2, the first
    w_{d-1} nodes of level d-1 (in flattened order) each get w_d children.
    Widths [4, 3, 2, 1, 1] give levels of 1, 4, 12, 6, 2, 1 nodes: 26 nodes.
    """
    parent = [-1]
    level = [0]
    for d, w in enumerate(widths):
        takers = level if d == 0 else level[: widths[d - 1]]
        nxt = []
        for p in takers:
            for _ in range(w):
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.array(parent, np.int32)


def tree_chain(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def tree_star(n: int) -> np.ndarray:
    p = np.zeros(n, np.int32)
    p[0] = -1
    return p


def forest_random(g: np.random.Generator, n: int, roots: int, max_depth: int) -> np.ndarray:
    """A forest of ``roots`` random trees (``tree_random_levels``) with ``n`` nodes in
    all, flattened level by level with the trees interleaved (node 0 is a root)."""
    sizes = np.full(roots, n // roots)
    sizes[: n % roots] += 1
    comps = [tree_random_levels(g, int(k), min(max_depth, int(k) - 1)) if k > 1 else np.array([-1], np.int32)
             for k in sizes]
    nodes = []  # (level, tiebreak, component, local index)
    for ci, par in enumerate(comps):
        lv = _levels_of(par)
        for j in range(len(par)):
            nodes.append((int(lv[j]), float(g.random()), ci, j))
    nodes.sort()
    where = {(ci, j): k for k, (_, _, ci, j) in enumerate(nodes)}
    out = np.full(n, -1, np.int32)
    for k, (_, _, ci, j) in enumerate(nodes):
        p = int(comps[ci][j])
        out[k] = -1 if p < 0 else where[(ci, p)]
    return out


def tree_random_recursive(g: np.random.Generator, n: int) -> np.ndarray:
    """parent[i] uniform over [0, i): a random recursive tree (deep-ish, irregular)."""
    p = np.full(n, -1, np.int32)
    for i in range(1, n):
        p[i] = int(g.integers(0, i))
    return p


def _levels_of(parent: np.ndarray) -> np.ndarray:
    """Level of each node by following parents (inputs are topologically ordered;
    every root, parent -1, is level 0)."""
    lv = np.zeros(len(parent), np.int64)
    for i in range(1, len(parent)):
        lv[i] = 0 if parent[i] < 0 else lv[parent[i]] + 1
    return lv


def _children_of(parent: np.ndarray):
    ch = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        if parent[i] >= 0:
            ch[int(parent[i])].append(i)
    return ch


# ----------------------------------------------------------------------------
# draft tokens and planted target logits
# ----------------------------------------------------------------------------

def draft_tokens(g: np.random.Generator, parent: np.ndarray, vocab: int) -> np.ndarray:
    """Draft ids uniform in [0, vocab), redrawn until siblings are distinct."""
    n = len(parent)
    tok = g.integers(0, vocab, size=n).astype(np.int32)
    for kids in _children_of(parent):
        seen = set()
        for c in kids:
            while int(tok[c]) in seen:
                tok[c] = int(g.integers(0, vocab))
            seen.add(int(tok[c]))
    return tok


def planted_logits(g: np.random.Generator, parent: np.ndarray, draft: np.ndarray,
                   vocab: int, length: int, seed: int, tag: str, target: Optional[int] = None):
    """fp32 N(0,1) logits [N, vocab] whose greedy path accepts ``length`` drafts.

    A target node t at level ``length`` is chosen (uniformly unless given); the
    path root -> t is x0..xL.  Row x_k (k < L) gets its largest entry planted
    at the draft token of x_{k+1}; every other row (t itself and every node off
    the path) gets it planted at a token that is no child's draft.  The planted
    entry is the row's drawn maximum plus 1.0, so it is the unique maximum.
    With distinct sibling drafts, exactly the nodes x0..xL are accepted.
    Returns (logits, t, planted_argmax).
    """
    n = len(parent)
    lv = _levels_of(parent)
    if target is None:
        cands = np.nonzero(lv == length)[0]
        if len(cands) == 0:
            raise ValueError(f"no node at level {length}")
        target = int(cands[int(g.integers(0, len(cands)))])
    path = []
    x = int(target)
    while x != -1:
        path.append(x)
        x = int(parent[x])
    path = path[::-1]
    kids = _children_of(parent)
    want = np.empty(n, np.int64)
    on_path_next = {path[k]: path[k + 1] for k in range(len(path) - 1)}
    for y in range(n):
        if y in on_path_next:
            want[y] = int(draft[on_path_next[y]])
        else:
            forbid = {int(draft[c]) for c in kids[y]}
            a = int(g.integers(0, vocab))
            while a in forbid:
                a = int(g.integers(0, vocab))
            want[y] = a
    logits = normal_f32(seed, tag, (n, vocab))
    rows = np.arange(n)
    logits[rows, want] = logits.max(axis=1) + np.float32(1.0)
    return logits, int(target), want.astype(np.int32)


# ----------------------------------------------------------------------------
# paged KV pool
# ----------------------------------------------------------------------------

def paged_layout(g: np.random.Generator, prefix_len: np.ndarray, bs: int, permute: bool, spare: int = 0):
    """Block table for per-sequence prefixes over a shared pool of ``bs``-token blocks.

    The pool holds exactly sum_b ceil((P_b + spare) / bs) blocks (at least one in
    total): ``spare`` tokens of room per sequence past its prefix (for appending
    accepted tokens).  With ``permute`` the block ids are a random permutation,
    otherwise sequence b owns a contiguous run.  Unused table entries are -1.
    """
    nblk = [-(-(int(p) + spare) // bs) for p in prefix_len]
    total = max(1, sum(nblk))
    ids = g.permutation(total).astype(np.int32) if permute else np.arange(total, dtype=np.int32)
    maxb = max(1, max(nblk))
    table = np.full((len(prefix_len), maxb), -1, np.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = ids[off:off + k]
        off += k
    return table, total


# ----------------------------------------------------------------------------
# a full case
# ----------------------------------------------------------------------------

@dataclass
class Case:
    name: str
    B: int
    N: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    parent: np.ndarray          # [B, N] int32
    prefix_len: np.ndarray      # [B] int32
    q: np.ndarray               # [B, N, Hq, D] bf16 bits
    k_cache: np.ndarray         # [num_blocks, Hkv, bs, D] bf16 bits
    v_cache: np.ndarray         # [num_blocks, Hkv, bs, D] bf16 bits
    block_table: np.ndarray     # [B, max_blocks] int32
    k_tree: np.ndarray          # [B, N, Hkv, D] bf16 bits
    v_tree: np.ndarray          # [B, N, Hkv, D] bf16 bits
    scale: float
    vocab: int = 0
    draft: Optional[np.ndarray] = None          # [B, N] int32
    logits: Optional[np.ndarray] = None         # [B, N, V] fp32
    planted_len: Optional[np.ndarray] = None    # [B] int32
    planted_target: Optional[np.ndarray] = None # [B] int32
    planted_argmax: Optional[np.ndarray] = None # [B, N] int32
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def W(self) -> int:
        return (self.N + 63) // 64


def build_case(name: str, seed: int, parent: np.ndarray, prefix_len, Hq: int, Hkv: int, D: int,
               bs: int, permute: bool, vocab: int = 0, plant_len=None, hot_key_frac: float = 0.0,
               hot_key_scale: float = 8.0, scale: Optional[float] = None,
               plant_target=None, spare_tokens: int = 0) -> Case:
    """Draw every tensor of one verification step.

    ``parent`` is [N] (shared by the batch) or [B, N].  ``prefix_len`` is [B].
    With ``vocab`` > 0, draft tokens and logits are drawn; ``plant_len`` (an int or
    a per-sequence array) is the accepted length to plant and ``plant_target``
    optionally fixes the planted end node per sequence.  ``hot_key_frac`` scales that fraction of key rows
    (each (token, kv-head) pair independently, prefix and tree keys alike) by
    ``hot_key_scale`` before the bf16 cast.
    """
    prefix_len = np.asarray(prefix_len, np.int32)
    B = len(prefix_len)
    parent = np.asarray(parent, np.int32)
    if parent.ndim == 1:
        parent = np.tile(parent, (B, 1))
    N = parent.shape[1]
    g = rng(seed, "structure")
    table, nblocks = paged_layout(g, prefix_len, bs, permute, spare_tokens)

    row_k_cache = row_k_tree = None
    if hot_key_frac > 0.0:
        gh = rng(seed, "hot-keys")
        row_k_cache = np.where(gh.random((nblocks, Hkv, bs)) < hot_key_frac, hot_key_scale, 1.0)
        row_k_tree = np.where(gh.random((B, N, Hkv)) < hot_key_frac, hot_key_scale, 1.0)

    q = normal_bf16(seed, "q", (B, N, Hq, D))
    k_cache = normal_bf16(seed, "k_cache", (nblocks, Hkv, bs, D), row_k_cache)
    v_cache = normal_bf16(seed, "v_cache", (nblocks, Hkv, bs, D))
    k_tree = normal_bf16(seed, "k_tree", (B, N, Hkv, D), row_k_tree)
    v_tree = normal_bf16(seed, "v_tree", (B, N, Hkv, D))
    case = Case(name=name, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, bs=bs, parent=parent,
                prefix_len=prefix_len, q=q, k_cache=k_cache, v_cache=v_cache,
                block_table=table, k_tree=k_tree, v_tree=v_tree,
                scale=float(scale if scale is not None else 1.0 / np.sqrt(D)))
    if vocab > 0:
        gd = rng(seed, "draft")
        draft = np.stack([draft_tokens(gd, parent[b], vocab) for b in range(B)])
        lens = np.zeros(B, np.int32)
        tgts = np.zeros(B, np.int32)
        ams = np.zeros((B, N), np.int32)
        logits = np.empty((B, N, vocab), np.float32)
        plant = np.broadcast_to(np.asarray(0 if plant_len is None else plant_len), (B,))
        for b in range(B):
            tgt = None if plant_target is None else int(plant_target[b])
            lg, t, am = planted_logits(gd, parent[b], draft[b], vocab, int(plant[b]),
                                       seed, f"logits{b}", target=tgt)
            logits[b] = lg
            lens[b] = int(plant[b])
            tgts[b] = t
            ams[b] = am
        case.vocab = vocab
        case.draft = draft
        case.logits = logits
        case.planted_len = lens
        case.planted_target = tgts
        case.planted_argmax = ams
    return case


# ----------------------------------------------------------------------------
# inputs of stochastic (temperature) verification
# ----------------------------------------------------------------------------

@dataclass
class StochasticInputs:
    """What a sampled verification step consumes besides the tree."""
    draft: np.ndarray        # [B, N] int32; children of u drawn without replacement from q[u]
    logits: np.ndarray       # [B, N, V] fp32 target logits
    q: np.ndarray            # [B, N, V] fp32 draft probabilities (each row sums to 1 in fp64)
    coins: np.ndarray        # [B, N] fp32 uniforms in [0, 1)
    temperature: float


def stochastic_inputs(seed: int, parent: np.ndarray, vocab: int, temperature: float = 1.0,
                      logit_scale: float = 2.0, draft_noise: float = 0.5,
                      tag: str = "stoch") -> StochasticInputs:
    """Target logits, a draft model's distributions, sampled draft tokens and coins.

    Target logits are ``logit_scale`` * N(0, 1).  The draft model is modelled as
    the target with its logits perturbed by ``draft_noise`` * N(0, 1): its
    distribution at node u is that perturbed row at temperature T, normalised
    in fp64 and stored in fp32.  The children of every node take tokens drawn
    from the parent's draft distribution without replacement, in index order
    (the ordered top-k of log q + Gumbel noise).  The coins are the uniforms
    the verifier consumes.
    """
    parent = np.asarray(parent, np.int32)
    B, N = parent.shape
    logits = normal_f32(seed, f"{tag}-target", (B, N, vocab)) * np.float32(logit_scale)
    noise = normal_f32(seed, f"{tag}-draft", (B, N, vocab))
    q = np.empty((B, N, vocab), np.float32)
    draft = np.zeros((B, N), np.int32)

    def one(b):
        z = (logits[b].astype(np.float64) + draft_noise * noise[b].astype(np.float64)) / temperature
        w = np.exp(z - z.max(axis=1, keepdims=True))
        q[b] = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
        g = rng(seed, f"{tag}-tokens{b}")
        for u, kids in enumerate(_children_of(parent[b])):
            if not kids:
                continue
            qu = q[b, u].astype(np.float64)
            with np.errstate(divide="ignore"):
                key = np.log(qu) - np.log(-np.log(g.random(vocab)))
            top = np.argpartition(-key, len(kids) - 1)[: len(kids)]
            top = top[np.argsort(-key[top], kind="stable")]
            draft[b, kids] = top.astype(np.int32)

    list(_pool().map(one, range(B)))
    coins = rng(seed, f"{tag}-coins").random((B, N), dtype=np.float32)
    return StochasticInputs(draft=draft, logits=logits, q=q, coins=coins, temperature=float(temperature))


def workload_trees(name: str, seed: int, batch: int = 64, forest_roots: int = 0) -> np.ndarray:
    """The [B, N] parent arrays of a named workload (the same draws its builder
    makes).  With ``forest_roots`` > 0 each sequence is instead a forest of that
    many trees (``forest_random``) with the same node count and depth."""
    if name == "c1":
        if forest_roots:
            raise ValueError("c1 has a fixed tree")
        return tree_worked_example()[None, :]
    g = rng(seed, "tree" if not forest_roots else f"forest{forest_roots}")
    shape = {"c2": (1, 64, 6), "c4": (batch, 64, 8), "c5": (4, 192, 10)}
    if name not in shape:
        raise ValueError(f"{name} has no draft tokens to verify")
    B, N, depth = shape[name]
    if forest_roots:
        return np.stack([forest_random(g, N, forest_roots, depth) for _ in range(B)])
    return np.stack([tree_random_levels(g, N, depth) for _ in range(B)])


SEEDS = {"c1": 20260001, "c2": 20260002, "c3": 20260003, "c4": 20260004, "c5": 20260005}
# Deepest level each workload's tree generator draws (every level up to it is
# populated, so it is also the depth of the deepest node).
LEVELS = {"c1": 2, "c2": 6, "c3": 5, "c4": 8, "c5": 10}
VOCAB = {"c1": 1000, "c2": 128256, "c4": 128256, "c5": 128256}


def stochastic_workload(name: str, temperature: float = 1.0, batch: int = 64, tag: str = "stoch"):
    """Trees of a named workload with inputs for stochastic verification.
    Returns (parent [B, N], StochasticInputs)."""
    parent = workload_trees(name, SEEDS[name], batch=batch)
    return parent, stochastic_inputs(SEEDS[name], parent, VOCAB[name], temperature=temperature, tag=tag)


# ----------------------------------------------------------------------------
# candidate pools for dynamic tree construction
# ----------------------------------------------------------------------------

@dataclass
class CandidatePool:
    """What a draft hands over before reranking: an expanded candidate tree."""
    parent: np.ndarray   # [B, M] int32, topological, parent[:, 0] = -1
    logp: np.ndarray     # [B, M] fp32, the draft's log-probability of each candidate given its parent (root 0)
    token: np.ndarray    # [B, M] int32, distinct among siblings


def candidate_pool(seed: int, batch: int, depth: int, topk: int, vocab: int, tag: str = "pool") -> CandidatePool:
    """A draft expansion of ``depth`` levels.  The root gets ``topk`` children;
    on every later level the ``topk`` candidates of the previous level that the
    draft gave the highest probability (given their own parent) get ``topk``
    children each.  A parent's children
    carry probabilities c * d, with d ~ Dirichlet(0.5, ..., 0.5) sorted in
    descending order and c ~ U(0.5, 1) the mass the draft puts on its top-k,
    and distinct uniform tokens.  Pool order is level by level."""
    g = rng(seed, tag)
    M = 1 + topk + (depth - 1) * topk * topk
    parent = np.full((batch, M), -1, np.int32)
    logp = np.zeros((batch, M), np.float32)
    token = np.zeros((batch, M), np.int32)
    for b in range(batch):
        nxt = 1
        level = [0]
        for d in range(depth):
            grow = level if d == 0 else sorted(sorted(level, key=lambda c: (-float(logp[b, c]), c))[:topk])
            new_level = []
            for u in grow:
                probs = np.sort(g.dirichlet(np.full(topk, 0.5)))[::-1] * g.uniform(0.5, 1.0)
                toks = g.choice(vocab, size=topk, replace=False)
                for k in range(topk):
                    parent[b, nxt] = u
                    with np.errstate(divide="ignore"):
                        logp[b, nxt] = np.float32(np.log(probs[k]))
                    token[b, nxt] = toks[k]
                    new_level.append(nxt)
                    nxt += 1
            level = new_level
        assert nxt == M
    return CandidatePool(parent=parent, logp=logp, token=token)


# The five workloads.  Seeds: 20260000 + k unless overridden.

def c1(seed: int = 20260001, **extra) -> Case:
    """Tiny reference: batch 1, the five-node demo tree, prefix 16, 2 heads (no GQA),
    head_dim 64; vocab 1000 with the greedy path 0 -> 1 -> 3 planted."""
    return build_case("c1", seed, tree_worked_example(), [16], Hq=2, Hkv=2, D=64, bs=16,
                      permute=False, vocab=1000, plant_len=2, plant_target=[3], **extra)


def c2(seed: int = 20260002, vocab: int = 128256, forest_roots: int = 0, **extra) -> Case:
    """Llama-3-8B-shaped layer: batch 1, 32 q / 8 kv heads, head_dim 128, contiguous
    4096-token prefix, a random 64-node tree of depth 6.  The workload lists no
    logits for this shape; the verification step here draws them over the
    Llama-3 vocabulary (128256) with a planted accepted length uniform in [0, 6]."""
    parent = workload_trees("c2", seed, forest_roots=forest_roots)[0]
    plant = int(rng(seed, "plant").integers(0, 7))
    case = build_case("c2", seed, parent, [4096], Hq=32, Hkv=8, D=128, bs=4096, permute=False,
                      vocab=vocab, plant_len=plant, **extra)
    return case


def c3(seed: int = 20260003, **extra) -> Case:
    """Batched serving: batch 16, prefixes uniform in [1024, 16384], 32 q / 8 kv heads,
    head_dim 128, paged KV (block 16, permuted table), the fixed 26-node tree with
    widths [4, 3, 2, 1, 1] shared by the batch.  Attention only."""
    g = rng(seed, "prefix")
    plen = g.integers(1024, 16385, size=16).astype(np.int32)
    parent = tree_from_widths([4, 3, 2, 1, 1])
    return build_case("c3", seed, parent, plen, Hq=32, Hkv=8, D=128, bs=16, permute=True, **extra)


def c4(seed: int = 20260004, batch: int = 64, forest_roots: int = 0, **extra) -> Case:
    """70B-shaped layer: batch 64, 64 q / 8 kv heads, head_dim 128, paged KV (block 16),
    prefix 8192; per-sequence random 64-node trees of depth 8; logits over 128256
    with planted accepted lengths uniform in [0, 8]."""
    parents = workload_trees("c4", seed, batch=batch, forest_roots=forest_roots)
    plant = rng(seed, "plant").integers(0, 9, size=batch)
    return build_case("c4", seed, parents, [8192] * batch, Hq=64, Hkv=8, D=128, bs=16,
                      permute=True, vocab=128256, plant_len=plant, **extra)


def c5(seed: int = 20260005, prefix: int = 131072, forest_roots: int = 0, **extra) -> Case:
    """Long-context wide tree: batch 4, prefix 131072, 32 q / 8 kv heads, head_dim 128,
    paged KV (block 64); a random 192-node tree of depth 10; 1% of key rows scaled by
    8; logits over 128256.  No accepted length is given for this shape; one uniform
    in [0, 10] is planted per sequence so that the walk is exercised."""
    parents = workload_trees("c5", seed, forest_roots=forest_roots)
    plant = rng(seed, "plant").integers(0, 11, size=4)
    return build_case("c5", seed, parents, [prefix] * 4, Hq=32, Hkv=8, D=128, bs=64,
                      permute=True, vocab=128256, plant_len=plant, hot_key_frac=0.01, **extra)


CONFIGS = {"c1": c1, "c2": c2, "c3": c3, "c4": c4, "c5": c5}


def make(name: str, **kw) -> Case:
    """A named workload; extra keywords (e.g. ``spare_tokens``) go to ``build_case``."""
    return CONFIGS[name](**kw)
