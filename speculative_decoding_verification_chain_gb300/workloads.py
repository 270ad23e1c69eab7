"""Seeded synthetic inputs for the verify-and-accept step.

This module only *makes inputs*: target logits, draft tokens, draft
probabilities, temperatures, uniforms, token trees and KV slot maps.  It holds
none of the verification arithmetic, so both the CUDA path and the CPU oracle
can be fed from it without sharing any of the method's code.

Workloads (shapes and value laws follow the speculative-decoding pages:
"Speculative Decoding" / "Accept or Reject" on the EAGLE-3 review page, and the
acceptance-rule section of the serving-book chapter):

* ``chain_tiny``      fp32 logits N(0, 2^2), rows fixed and replicated across
                      trials; draft logits = target + N(0, 0.5^2), q = softmax.
* ``chain_greedy``    bf16 logits N(0, 3^2); draft token = row argmax with
                      probability ``p_match`` else uniform over V.  T = 0.
* ``chain_sampled``   bf16 logits of Zipf shape, -1.1 ln(rank) + N(0, 0.3^2)
                      with a random rank permutation per row; the draft is
                      q = softmax(((1 - lam) z + lam n) / T) with n an
                      independent Zipf-shaped draw; draft tokens ~ q.
* ``tree_greedy``     bf16 logits N(0, 3^2) over an EAGLE-style level tree;
                      node token = argmax of its parent's row with probability
                      ``p_match`` else uniform.

Every random draw the method itself consumes (accept / resample uniforms) is
generated here as ``u = m * 2**-24`` with integer ``m`` in [0, 2**24), so every
consumer sees bit-identical float32 values.

Logits are produced in float32 and rounded to bfloat16 with round-to-nearest-
even; bf16 tensors are carried as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence, Tuple

import numpy as np

BF16 = 0
FP32 = 1

# Padding value written into slot_mapping for rejected positions.
PADDING_SLOT_ID = -1

# Slot layout: each request owns a contiguous region of this many tokens
# (4096 of context plus a 16-token block of headroom), so bases are 16-aligned.
SLOT_REGION = 4096 + 16


# ----------------------------------------------------------------------------
# bf16 helpers (bit-level representation changes only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to the float32 values they denote (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def logits_as_f32(logits: np.ndarray, dtype: int) -> np.ndarray:
    return bf16_bits_to_f32(logits) if dtype == BF16 else np.asarray(logits, dtype=np.float32)


# ----------------------------------------------------------------------------
# containers
# ----------------------------------------------------------------------------
@dataclass
class ChainInputs:
    """One batch of chain verification inputs (row i of logits checks token i)."""
    logits: np.ndarray               # [B, k+1, V]  uint16 (bf16 bits) or float32
    dtype: int                       # BF16 / FP32
    draft_tokens: np.ndarray         # [B, k] int32
    temperature: np.ndarray          # [B] float32, 0 = greedy
    u_sample: np.ndarray             # [B, k+1] float32
    draft_probs: Optional[np.ndarray] = None   # [B, k, V] float32 (sampled only)
    u_accept: Optional[np.ndarray] = None      # [B, k] float32 (sampled only)
    slot_mapping: Optional[np.ndarray] = None  # [B, k+1] int64
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def k(self) -> int:
        return self.logits.shape[1] - 1

    @property
    def V(self) -> int:
        return self.logits.shape[2]


@dataclass
class TreeInputs:
    """One batch of greedy token-tree inputs (logits row n belongs to node n)."""
    logits: np.ndarray               # [B, N+1, V]
    dtype: int
    node_tokens: np.ndarray          # [B, N] int32, node n (1..N) at column n-1
    parent: np.ndarray               # [N+1] int32, parent[0] = -1
    tree_choices: list               # list of tuples, level order
    slot_mapping: Optional[np.ndarray] = None  # [B, N+1] int64
    name: str = ""
    meta: dict = field(default_factory=dict)
    # sampled trees only
    draft_probs: Optional[np.ndarray] = None   # [B, N+1, V] f32, row c: law of c's children
    temperature: Optional[np.ndarray] = None   # [B] f32 > 0
    u_accept: Optional[np.ndarray] = None      # [B, N] f32, node n at column n-1
    u_sample: Optional[np.ndarray] = None      # [B, N+1] f32, by the node the walk ends at

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def N(self) -> int:
        return self.logits.shape[1] - 1

    @property
    def V(self) -> int:
        return self.logits.shape[2]


# ----------------------------------------------------------------------------
# random streams
# ----------------------------------------------------------------------------
def _streams(seed: int, n: int = 6):
    """Independent generators: 0 logits, 1 draft, 2 method uniforms, 3 slots, 4 noise, 5 spare."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def method_uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    """u = m * 2^-24, m uniform on [0, 2^24): exactly representable float32 in [0, 1)."""
    m = rng.integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (m.astype(np.float64) * (2.0 ** -24)).astype(np.float32)


def slot_map(rng: np.random.Generator, B: int, P: int) -> np.ndarray:
    """slot(b, j) = b*(4096+16) + c_b + j with context length c_b ~ U[0, 4096)."""
    c = rng.integers(0, 4096, size=B, dtype=np.int64)
    base = np.arange(B, dtype=np.int64) * SLOT_REGION
    return (base + c)[:, None] + np.arange(P, dtype=np.int64)[None, :]


def _softmax_rows_f32(x: np.ndarray) -> np.ndarray:
    """Draft distribution synthesis (input side): softmax along the last axis."""
    x = x.astype(np.float32, copy=False)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True, dtype=np.float64).astype(np.float32)).astype(np.float32)


def _draw_from_rows(rng: np.random.Generator, probs: np.ndarray) -> np.ndarray:
    """Draw one index per row of ``probs`` [R, V] (drafter side, independent stream)."""
    R = probs.shape[0]
    out = np.empty(R, dtype=np.int32)
    uu = rng.random(R)
    for r in range(R):
        c = np.cumsum(probs[r], dtype=np.float64)
        j = int(np.searchsorted(c, uu[r] * c[-1], side="right"))
        out[r] = min(j, probs.shape[1] - 1)
    return out


def _zipf_rows(rng: np.random.Generator, nrows: int, V: int, jitter: float = 0.3,
               slope: float = 1.1) -> np.ndarray:
    """Rows of -slope*ln(rank) + N(0, jitter^2), rank a random permutation of 1..V per row."""
    base = (-slope * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    z = rng.permuted(np.broadcast_to(base, (nrows, V)), axis=1)
    z = z + rng.standard_normal((nrows, V), dtype=np.float32) * np.float32(jitter)
    return z.astype(np.float32, copy=False)


def _row_argmax(x: np.ndarray) -> np.ndarray:
    return np.argmax(x, axis=-1).astype(np.int32)


# ----------------------------------------------------------------------------
# chain workloads
# ----------------------------------------------------------------------------
def chain_tiny(seed: int = 1, trials: int = 1000, k: int = 4, V: int = 1000,
               temperature: float = 1.0) -> ChainInputs:
    """Fixed target/draft rows replicated over ``trials`` independent requests (fp32 logits)."""
    g = _streams(seed)
    target = (g[0].standard_normal((k + 1, V)) * 2.0).astype(np.float32)
    draft_logits = target[:k].astype(np.float64) + g[4].standard_normal((k, V)) * 0.5
    q_rows = _softmax_rows_f32(draft_logits.astype(np.float32))
    logits = np.broadcast_to(target, (trials, k + 1, V)).copy()
    q = np.broadcast_to(q_rows, (trials, k, V)).copy()
    tokens = np.empty((trials, k), dtype=np.int32)
    for i in range(k):
        c = np.cumsum(q_rows[i], dtype=np.float64)
        uu = g[1].random(trials) * c[-1]
        tokens[:, i] = np.minimum(np.searchsorted(c, uu, side="right"), V - 1)
    return ChainInputs(
        logits=logits, dtype=FP32, draft_tokens=tokens,
        temperature=np.full(trials, temperature, dtype=np.float32),
        u_sample=method_uniforms(g[2], (trials, k + 1)),
        draft_probs=q, u_accept=method_uniforms(g[2], (trials, k)),
        slot_mapping=slot_map(g[3], trials, k + 1), name="chain_tiny",
        meta=dict(target_rows=target, q_rows=q_rows))


def chain_fixed_rows(seed: int, trials: int, p_logits: np.ndarray, q_rows: np.ndarray,
                     temperature: float = 1.0) -> ChainInputs:
    """Caller-chosen fixed rows (fp32 logits [k+1, V], q [k, V]) replicated over trials;
    draft tokens drawn from q.  Used for the small-V statistical constructions."""
    g = _streams(seed)
    p_logits = np.asarray(p_logits, dtype=np.float32)
    q_rows = np.asarray(q_rows, dtype=np.float32)
    k1, V = p_logits.shape
    k = k1 - 1
    tokens = np.empty((trials, k), dtype=np.int32)
    for i in range(k):
        c = np.cumsum(q_rows[i], dtype=np.float64)
        uu = g[1].random(trials) * c[-1]
        tokens[:, i] = np.minimum(np.searchsorted(c, uu, side="right"), V - 1)
    return ChainInputs(
        logits=np.broadcast_to(p_logits, (trials, k + 1, V)).copy(), dtype=FP32,
        draft_tokens=tokens, temperature=np.full(trials, temperature, dtype=np.float32),
        u_sample=method_uniforms(g[2], (trials, k + 1)),
        draft_probs=np.broadcast_to(q_rows, (trials, k, V)).copy(),
        u_accept=method_uniforms(g[2], (trials, k)),
        slot_mapping=slot_map(g[3], trials, k + 1), name="chain_fixed_rows")


def chain_greedy(seed: int = 2, B: int = 64, k: int = 5, V: int = 128256,
                 p_match: float = 0.8, dtype: int = BF16, sigma: float = 3.0) -> ChainInputs:
    """Greedy chain: logits N(0, sigma^2); token i+1 = argmax(row i) w.p. p_match else uniform."""
    g = _streams(seed)
    logits = np.empty((B, k + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    tokens = np.empty((B, k), dtype=np.int32)
    blk = max(1, (1 << 24) // max(1, (k + 1) * V))
    for b0 in range(0, B, blk):
        b1 = min(B, b0 + blk)
        x = g[0].standard_normal((b1 - b0, k + 1, V), dtype=np.float32) * np.float32(sigma)
        if dtype == BF16:
            bits = f32_to_bf16_bits(x)
            logits[b0:b1] = bits
            xv = bf16_bits_to_f32(bits)
        else:
            logits[b0:b1] = x
            xv = x
        am = _row_argmax(xv[:, :k, :])
        match = g[1].random((b1 - b0, k)) < p_match
        rnd = g[1].integers(0, V, size=(b1 - b0, k), dtype=np.int64).astype(np.int32)
        tokens[b0:b1] = np.where(match, am, rnd)
    return ChainInputs(
        logits=logits, dtype=dtype, draft_tokens=tokens,
        temperature=np.zeros(B, dtype=np.float32),
        u_sample=method_uniforms(g[2], (B, k + 1)),
        slot_mapping=slot_map(g[3], B, k + 1), name="chain_greedy",
        meta=dict(p_match=p_match))


def chain_sampled(seed: int = 3, B: int = 32, k: int = 4, V: int = 128256,
                  temperature: float = 0.7, lam: float = 0.3, dtype: int = BF16) -> ChainInputs:
    """Sampled chain on Zipf-shaped logits; q = softmax(((1-lam) z + lam n) / T)."""
    g = _streams(seed)
    logits = np.empty((B, k + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    q = np.empty((B, k, V), dtype=np.float32)
    tokens = np.empty((B, k), dtype=np.int32)
    T = np.float32(temperature)
    for b in range(B):
        z = _zipf_rows(g[0], k + 1, V)
        if dtype == BF16:
            bits = f32_to_bf16_bits(z)
            logits[b] = bits
            zv = bf16_bits_to_f32(bits)
        else:
            logits[b] = z
            zv = z
        n = _zipf_rows(g[4], k, V)
        mix = (np.float32(1.0 - lam) * zv[:k] + np.float32(lam) * n) / T
        q[b] = _softmax_rows_f32(mix)
        tokens[b] = _draw_from_rows(g[1], q[b])
    return ChainInputs(
        logits=logits, dtype=dtype, draft_tokens=tokens,
        temperature=np.full(B, temperature, dtype=np.float32),
        u_sample=method_uniforms(g[2], (B, k + 1)),
        draft_probs=q, u_accept=method_uniforms(g[2], (B, k)),
        slot_mapping=slot_map(g[3], B, k + 1), name="chain_sampled",
        meta=dict(lam=lam))


def chain_mixed(seed: int, B: int, k: int, V: int, dtype: int = BF16,
                greedy_fraction: float = 0.5, temperature: float = 0.8, lam: float = 0.3,
                p_match: float = 0.8) -> ChainInputs:
    """Mixed batch: some requests greedy (T = 0), the rest sampled (Zipf recipe)."""
    s = chain_sampled(seed=seed, B=B, k=k, V=V, temperature=temperature, lam=lam, dtype=dtype)
    g = _streams(seed + 7919)
    greedy = g[0].random(B) < greedy_fraction
    zf = logits_as_f32(s.logits, dtype)
    am = _row_argmax(zf[:, :k, :])
    match = g[1].random((B, k)) < p_match
    rnd = g[1].integers(0, V, size=(B, k), dtype=np.int64).astype(np.int32)
    tok_g = np.where(match, am, rnd)
    s.draft_tokens = np.where(greedy[:, None], tok_g, s.draft_tokens).astype(np.int32)
    s.temperature = np.where(greedy, np.float32(0.0), s.temperature).astype(np.float32)
    s.name = "chain_mixed"
    return s


# ----------------------------------------------------------------------------
# tree workloads
# ----------------------------------------------------------------------------
@dataclass
class RaggedChainInputs:
    """Chains with a different number of drafts per request, packed as the
    vLLM walkthrough's per-step metadata lays them out: request b's k_b drafts
    at cu[b] .. cu[b+1]-1 and its k_b + 1 target rows at cu[b] + b .. cu[b+1] + b."""
    logits: np.ndarray               # [cu[B] + B, V] uint16 (bf16 bits) or float32
    dtype: int
    cu: np.ndarray                   # [B+1] int32 cu_num_draft_tokens
    draft_tokens: np.ndarray         # [cu[B]] int32
    temperature: np.ndarray          # [B] float32, 0 = greedy
    u_sample: np.ndarray             # [cu[B] + B] float32
    draft_probs: Optional[np.ndarray]   # [cu[B], V] float32 (None: every request greedy)
    u_accept: Optional[np.ndarray]      # [cu[B]] float32
    slot_mapping: np.ndarray         # [cu[B] + B] int64
    parts: list                      # the per-request ChainInputs (B = 1 each)
    name: str = "chain_ragged"

    @property
    def B(self) -> int:
        return self.cu.shape[0] - 1

    @property
    def V(self) -> int:
        return self.logits.shape[1]

    @property
    def max_k(self) -> int:
        return int(np.max(np.diff(self.cu))) if self.B else 0


def chain_ragged(seed: int, B: int, max_k: int, V: int, mode: str = "greedy", dtype: int = BF16,
                 temperature: float = 0.8, lam: float = 0.3, p_match: float = 0.8,
                 min_k: int = 0) -> RaggedChainInputs:
    """Per-request k_b uniform in [min_k, max_k]; each request drawn by the
    greedy or sampled chain recipe (mode "greedy", "sampled" or "mixed": half
    of the requests greedy, at random), then packed."""
    rng = np.random.default_rng(seed)
    ks = rng.integers(min_k, max_k + 1, size=B)
    greedy = np.ones(B, bool) if mode == "greedy" else (np.zeros(B, bool) if mode == "sampled"
                                                        else rng.random(B) < 0.5)
    parts = []
    for b in range(B):
        s = seed * 7919 + 13 * b + 1
        if greedy[b]:
            parts.append(chain_greedy(seed=s, B=1, k=int(ks[b]), V=V, p_match=p_match, dtype=dtype))
        else:
            parts.append(chain_sampled(seed=s, B=1, k=int(ks[b]), V=V, temperature=temperature, lam=lam,
                                       dtype=dtype))
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(ks)
    total = int(cu[-1])
    logits = np.concatenate([x.logits[0] for x in parts], axis=0)
    tokens = np.concatenate([x.draft_tokens[0] for x in parts]).astype(np.int32) if total else np.zeros(0, np.int32)
    sampled = not greedy.all()
    q = ua = None
    if sampled:
        q = np.concatenate([x.draft_probs[0] if x.draft_probs is not None else np.zeros((x.k, V), np.float32)
                            for x in parts], axis=0) if total else np.zeros((0, V), np.float32)
        ua = np.concatenate([x.u_accept[0] if x.u_accept is not None else np.zeros(x.k, np.float32)
                             for x in parts]).astype(np.float32) if total else np.zeros(0, np.float32)
    us = np.concatenate([x.u_sample[0] for x in parts]).astype(np.float32)
    T = np.array([x.temperature[0] for x in parts], np.float32)
    slots = np.concatenate([x.slot_mapping[0] + 100000 * b for b, x in enumerate(parts)]).astype(np.int64)
    return RaggedChainInputs(logits=logits, dtype=dtype, cu=cu, draft_tokens=tokens, temperature=T,
                             u_sample=us, draft_probs=q, u_accept=ua, slot_mapping=slots, parts=parts)


def ngram_texts(seed: int, B: int, Lmax: int, V: int = 128256, copy_frac: float = 0.5,
                span: Tuple[int, int] = (4, 48), min_len: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """Token texts for n-gram lookup: a random prompt of half the length, then
    text in which spans copied from earlier (lengths uniform in `span`) make up
    about `copy_frac` of the tokens, the rest drawn at random (the copy-heavy
    tasks the lookup suits: summarising, editing code).  Lengths uniform in
    [min_len, Lmax]; tokens past a row's length are 0.  Returns (tokens
    [B, Lmax] int32, lengths [B] int32)."""
    rng = np.random.default_rng(seed)
    tokens = np.zeros((B, Lmax), np.int32)
    lengths = rng.integers(min_len, Lmax + 1, size=B).astype(np.int32)
    for b in range(B):
        L = int(lengths[b])
        t = rng.integers(0, V, size=L, dtype=np.int64).astype(np.int32)
        pos = max(1, L // 2)
        while pos < L:
            if rng.random() < copy_frac and pos > 1:
                n = int(rng.integers(span[0], span[1] + 1))
                src = int(rng.integers(0, pos))
                n = min(n, L - pos, pos - src)
                t[pos:pos + n] = t[src:src + n]
                pos += max(1, n)
            else:
                pos += int(rng.integers(1, span[1] + 1))
        tokens[b, :L] = t
    return tokens, lengths


def level_tree_choices(children_per_level: Sequence[int]) -> list:
    """tree_choices (list of index tuples, level order) for a tree in which every
    node of level L-1 has children_per_level[L] children (level 0 = root)."""
    levels = [[()]]
    for c in children_per_level:
        nxt = []
        for node in levels[-1]:
            for i in range(c):
                nxt.append(node + (i,))
        levels.append(nxt)
    out = []
    for lvl in levels[1:]:
        out.extend(lvl)
    return out


def parents_in_order(children_per_level: Sequence[int]) -> np.ndarray:
    """Parent-index array for the level tree: node j of level L (0-based inside
    its level) hangs under node floor(j / c_L) of level L-1; nodes are numbered
    1..N in level order, root = 0."""
    parent = [-1]
    first_prev, count_prev = 0, 1
    nxt = 1
    for c in children_per_level:
        count = count_prev * c
        for j in range(count):
            parent.append(first_prev + j // c)
        first_prev, count_prev = nxt, count
        nxt += count
    return np.asarray(parent, dtype=np.int32)


def tree_greedy(seed: int = 4, B: int = 16, V: int = 128256,
                children_per_level: Sequence[int] = (4, 2, 2, 1, 1), p_match: float = 0.7,
                dtype: int = BF16, sigma: float = 3.0,
                parent: Optional[np.ndarray] = None) -> TreeInputs:
    """Greedy token tree: logits N(0, sigma^2) [B, N+1, V]; token of node n equals
    argmax of row parent[n] w.p. p_match, else uniform over V."""
    g = _streams(seed)
    if parent is None:
        parent = parents_in_order(children_per_level)
        choices = level_tree_choices(children_per_level)
    else:
        parent = np.asarray(parent, dtype=np.int32)
        choices = []
    N = parent.shape[0] - 1
    logits = np.empty((B, N + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    toks = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        x = g[0].standard_normal((N + 1, V), dtype=np.float32) * np.float32(sigma)
        if dtype == BF16:
            bits = f32_to_bf16_bits(x)
            logits[b] = bits
            xv = bf16_bits_to_f32(bits)
        else:
            logits[b] = x
            xv = x
        am = _row_argmax(xv)
        match = g[1].random(N) < p_match
        rnd = g[1].integers(0, V, size=N, dtype=np.int64).astype(np.int32)
        toks[b] = np.where(match, am[parent[1:]], rnd)
    return TreeInputs(
        logits=logits, dtype=dtype, node_tokens=toks, parent=parent,
        tree_choices=choices, slot_mapping=slot_map(g[3], B, N + 1), name="tree_greedy",
        meta=dict(p_match=p_match, children_per_level=tuple(children_per_level)))


def tree_sampled(seed: int = 6, B: int = 16, V: int = 128256,
                 children_per_level: Sequence[int] = (4, 2, 2, 1, 1), temperature: float = 0.7,
                 lam: float = 0.3, dtype: int = BF16, parent: Optional[np.ndarray] = None) -> TreeInputs:
    """Sampled token tree: Zipf-shaped logits per node (as the sampled chain);
    row c of draft_probs is q_c = softmax(((1-lam) z_c + lam n_c) / T) with n_c
    an independent Zipf-shaped draw; the children of c are drawn i.i.d. from q_c
    (with replacement, so siblings may repeat a token)."""
    g = _streams(seed)
    if parent is None:
        parent = parents_in_order(children_per_level)
        choices = level_tree_choices(children_per_level)
    else:
        parent = np.asarray(parent, dtype=np.int32)
        choices = []
    N = parent.shape[0] - 1
    logits = np.empty((B, N + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    q = np.empty((B, N + 1, V), dtype=np.float32)
    toks = np.empty((B, N), dtype=np.int32)
    T = np.float32(temperature)
    for b in range(B):
        z = _zipf_rows(g[0], N + 1, V)
        if dtype == BF16:
            bits = f32_to_bf16_bits(z)
            logits[b] = bits
            zv = bf16_bits_to_f32(bits)
        else:
            logits[b] = z
            zv = z
        n = _zipf_rows(g[4], N + 1, V)
        q[b] = _softmax_rows_f32((np.float32(1.0 - lam) * zv + np.float32(lam) * n) / T)
        if N > 0:
            toks[b] = _draw_from_rows(g[1], q[b][parent[1:]])
    return TreeInputs(
        logits=logits, dtype=dtype, node_tokens=toks, parent=parent, tree_choices=choices,
        slot_mapping=slot_map(g[3], B, N + 1), name="tree_sampled",
        meta=dict(lam=lam, children_per_level=tuple(children_per_level)),
        draft_probs=q, temperature=np.full(B, temperature, dtype=np.float32),
        u_accept=method_uniforms(g[2], (B, N)), u_sample=method_uniforms(g[2], (B, N + 1)))


def redraw(x, seed: int):
    """The same logits and draft distributions with fresh draws: draft tokens
    drawn again from q (children of c i.i.d. from q_c for trees) and new method
    uniforms.  Each result is an independent trial of the accept / resample
    process on fixed distributions (the rates of rare events, such as positions
    near a flag window, are measured over many such trials without making the
    expensive rows again)."""
    from dataclasses import replace
    g = _streams(seed)
    if isinstance(x, TreeInputs):
        par = np.asarray(x.parent)
        toks = np.empty_like(x.node_tokens)
        for b in range(x.B):
            if x.N > 0:
                toks[b] = _draw_from_rows(g[1], x.draft_probs[b][par[1:]])
        return replace(x, node_tokens=toks, u_accept=method_uniforms(g[2], (x.B, x.N)),
                       u_sample=method_uniforms(g[2], (x.B, x.N + 1)))
    toks = np.empty_like(x.draft_tokens)
    for b in range(x.B):
        toks[b] = _draw_from_rows(g[1], x.draft_probs[b])
    return replace(x, draft_tokens=toks, u_accept=method_uniforms(g[2], (x.B, x.k)),
                   u_sample=method_uniforms(g[2], (x.B, x.k + 1)))


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------
def named(name: str, **kw):
    """Workloads by name: 'tiny', 'greedy', 'sampled', 'tree', 'sweep'."""
    if name == "tiny":
        return chain_tiny(**kw)
    if name == "greedy":
        return chain_greedy(**kw)
    if name == "sampled":
        return chain_sampled(**kw)
    if name == "tree":
        return tree_greedy(**kw)
    if name == "sweep":
        kw.setdefault("B", 64)
        return chain_sampled(seed=kw.pop("seed", 5), k=kw.pop("k", 8), V=kw.pop("V", 152064),
                             temperature=kw.pop("temperature", 1.0), lam=kw.pop("lam", 0.3), **kw)
    raise KeyError(name)
