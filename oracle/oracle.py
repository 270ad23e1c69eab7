"""CPU oracle for speculative-decoding verify-and-accept (ctypes binding).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the product path.  The
arithmetic lives in ``spec_oracle.c`` (plain C, IEEE double, index order); this
module only builds that file with gcc, marshals numpy arrays into it, and adds
the host-side tree metadata of the vLLM EAGLE walkthrough ("tree drafting in
detail" section) in plain Python.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspecoracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP32 = 1


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into libspecoracle.so next to it (gcc, no fast-math,
    no FMA contraction, so both host architectures evaluate the same expressions)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_verify_chain.argtypes = [P, I, P, P, P, P, P, I, I, I, P, P, P, P, P, P, I]
    lib.oracle_verify_chain.restype = I
    lib.oracle_verify_tree.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P]
    lib.oracle_verify_tree.restype = I
    lib.oracle_fixup_slots.argtypes = [P, I, I, P, P, I, ctypes.c_int64]
    lib.oracle_fixup_slots.restype = I
    lib.oracle_ngram_propose.argtypes = [P, P, I, I, I, I, I, P, P, P, P]
    lib.oracle_verify_tree_sampled.argtypes = [P, I, P, P, P, P, P, P, I, I, I, I, P, P, P, P, P, P]
    lib.oracle_verify_tree_sampled.restype = I
    L = ctypes.c_int64
    lib.oracle_prepare_next_step.argtypes = [P, I, P, P, P, I, I, I, I, I, P, P, L, L, P, P, P, P, P, P]
    lib.oracle_prepare_next_step.restype = I
    lib.oracle_compact_tree_kv.argtypes = [P, L, L, P, I, P, I, P, I, P]
    lib.oracle_compact_tree_kv.restype = I
    lib.oracle_ngram_propose.restype = I
    return lib


def load_library(path: str):
    """Bind a separately compiled copy of spec_oracle.c (the tests use this to
    check that planted mistakes are caught by the pins)."""
    return _bind(ctypes.CDLL(path))


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def verify_chain(logits: np.ndarray, dtype: int, draft_tokens: np.ndarray,
                 temperature: np.ndarray, u_sample: np.ndarray,
                 draft_probs: Optional[np.ndarray] = None, u_accept: Optional[np.ndarray] = None,
                 nthreads: int = 1, lib=None) -> dict:
    """Chain verify for every request.  Returns out_tokens [B, k+1] (-1 padded),
    num_accepted [B], flag_accept [B, k], flag_sample [B], b_alg [B] and
    accept_ratio [B, k] (p/q of each accept test that ran, NaN otherwise)."""
    lib = _load(lib)
    B, k1, V = logits.shape
    k = k1 - 1
    z = np.ascontiguousarray(logits, dtype=np.uint16 if dtype == BF16 else np.float32)
    tok = _c(draft_tokens, np.int32)
    T = _c(temperature, np.float32)
    us = _c(u_sample, np.float32)
    q = _c(draft_probs, np.float32)
    ua = _c(u_accept, np.float32)
    out = dict(
        out_tokens=np.empty((B, k + 1), np.int32), num_accepted=np.empty(B, np.int32),
        flag_accept=np.empty((B, k), np.int32), flag_sample=np.empty(B, np.int32),
        b_alg=np.empty(B, np.float64), accept_ratio=np.empty((B, k), np.float64))
    rc = lib.oracle_verify_chain(
        _ptr(z), dtype, _ptr(q), _ptr(tok), _ptr(T), _ptr(ua), _ptr(us), B, k, V,
        _ptr(out["out_tokens"]), _ptr(out["num_accepted"]), _ptr(out["flag_accept"]),
        _ptr(out["flag_sample"]), _ptr(out["b_alg"]), _ptr(out["accept_ratio"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify_chain rejected its arguments")
    return out


def verify_tree(logits: np.ndarray, dtype: int, node_tokens: np.ndarray, parent: np.ndarray,
                max_depth: Optional[int] = None, lib=None) -> dict:
    """Greedy tree verify.  Returns path [B, D+1], tokens [B, D+1], length [B], b_alg [B]."""
    lib = _load(lib)
    B, n1, V = logits.shape
    N = n1 - 1
    par = _c(parent, np.int32)
    if max_depth is None:
        max_depth = int(tree_depths(par).max()) if N > 0 else 0
    z = np.ascontiguousarray(logits, dtype=np.uint16 if dtype == BF16 else np.float32)
    toks = _c(node_tokens if N > 0 else np.zeros((B, 0), np.int32), np.int32)
    out = dict(path=np.empty((B, max_depth + 1), np.int32),
               tokens=np.empty((B, max_depth + 1), np.int32),
               length=np.empty(B, np.int32), b_alg=np.empty(B, np.float64))
    rc = lib.oracle_verify_tree(_ptr(z), dtype, _ptr(toks), _ptr(par), B, N, V, int(max_depth),
                                _ptr(out["path"]), _ptr(out["tokens"]), _ptr(out["length"]),
                                _ptr(out["b_alg"]))
    if rc != 0:
        raise ValueError("oracle_verify_tree rejected its arguments")
    return out


def verify_tree_sampled(logits: np.ndarray, dtype: int, node_tokens: np.ndarray, parent: np.ndarray,
                        temperature: np.ndarray, u_accept: np.ndarray, u_sample: np.ndarray,
                        draft_probs: np.ndarray, max_depth: Optional[int] = None, lib=None) -> dict:
    """Sampled tree verify (sequential over siblings with residual updates).
    logits [B, N+1, V]; draft_probs [B, N+1, V] (row c: the distribution the
    children of node c were drawn from); node_tokens, u_accept [B, N];
    u_sample [B, N+1] (indexed by the node the walk ends at); temperature [B] > 0.
    Returns path [B, D+1], tokens [B, D+1], length [B], flag_accept [B, N],
    flag_sample [B], b_alg [B]."""
    lib = _load(lib)
    B, n1, V = logits.shape
    N = n1 - 1
    par = _c(parent, np.int32)
    if max_depth is None:
        max_depth = int(tree_depths(par).max()) if N > 0 else 0
    z = np.ascontiguousarray(logits, dtype=np.uint16 if dtype == BF16 else np.float32)
    toks = _c(node_tokens if N > 0 else np.zeros((B, 0), np.int32), np.int32)
    ua = _c(u_accept if N > 0 else np.zeros((B, 0), np.float32), np.float32)
    q = _c(draft_probs, np.float32)
    out = dict(path=np.empty((B, max_depth + 1), np.int32), tokens=np.empty((B, max_depth + 1), np.int32),
               length=np.empty(B, np.int32), flag_accept=np.empty((B, N), np.int32),
               flag_sample=np.empty(B, np.int32), b_alg=np.empty(B, np.float64))
    rc = lib.oracle_verify_tree_sampled(
        _ptr(z), dtype, _ptr(q), _ptr(toks), _ptr(par), _ptr(_c(temperature, np.float32)), _ptr(ua),
        _ptr(_c(u_sample, np.float32)), B, N, V, int(max_depth), _ptr(out["path"]), _ptr(out["tokens"]),
        _ptr(out["length"]), _ptr(out["flag_accept"]), _ptr(out["flag_sample"]), _ptr(out["b_alg"]))
    if rc != 0:
        raise ValueError("oracle_verify_tree_sampled rejected its arguments")
    return out


def prepare_next_step(out_tokens: np.ndarray, num_accepted: np.ndarray, positions: np.ndarray,
                      block_table: np.ndarray, block_size: int, P_next: int, rows_per_req: int = 0,
                      cu: Optional[np.ndarray] = None, hidden: Optional[np.ndarray] = None, pad: int = -1,
                      lib=None) -> dict:
    """Next-step inputs after verification.  Returns next_token [B],
    next_position [B], next_slots [B, P_next] int64, last_row [B],
    hidden_out [B, row] (when hidden is given) and status."""
    lib = _load(lib)
    ot = _c(out_tokens, np.int32)
    B, stride = ot.shape
    bt = _c(block_table, np.int32)
    max_blocks = 0 if bt is None else bt.shape[1]
    hid = None if hidden is None else np.ascontiguousarray(hidden)
    row_bytes = 0 if hid is None else hid.reshape(hid.shape[0], -1).view(np.uint8).shape[1]
    out = dict(next_token=np.empty(B, np.int32), next_position=np.empty(B, np.int32),
               next_slots=np.empty((B, P_next), np.int64), last_row=np.empty(B, np.int32),
               hidden_out=None if hid is None else np.empty((B,) + hid.shape[1:], hid.dtype),
               status=np.zeros(1, np.int32))
    rc = lib.oracle_prepare_next_step(
        _ptr(ot), stride, _ptr(_c(num_accepted, np.int32)), _ptr(_c(positions, np.int32)), _ptr(bt), max_blocks,
        int(block_size), B, int(P_next), int(rows_per_req), _ptr(_c(cu, np.int32)), _ptr(hid), int(row_bytes),
        int(pad), _ptr(out["next_token"]), _ptr(out["next_position"]), _ptr(out["next_slots"]),
        _ptr(out["last_row"]), _ptr(out["hidden_out"]), _ptr(out["status"]))
    if rc != 0:
        raise ValueError("oracle_prepare_next_step rejected its arguments")
    return out


def compact_tree_kv(kv: np.ndarray, slot_mapping: np.ndarray, path: np.ndarray, out_len: np.ndarray,
                    lib=None) -> dict:
    """Tree KV compaction on a copy of kv [num_slots, ...].  Returns kv, status."""
    lib = _load(lib)
    k = np.array(kv, copy=True, order="C")
    num_slots = k.shape[0]
    row_bytes = k.reshape(num_slots, -1).view(np.uint8).shape[1] if num_slots else 1
    sm = _c(slot_mapping, np.int64)
    pa = _c(path, np.int32)
    st = np.zeros(1, np.int32)
    rc = lib.oracle_compact_tree_kv(_ptr(k), num_slots, int(row_bytes), _ptr(sm), sm.shape[1], _ptr(pa),
                                    pa.shape[1], _ptr(_c(out_len, np.int32)), sm.shape[0], _ptr(st))
    if rc != 0:
        raise ValueError("oracle_compact_tree_kv rejected its arguments")
    return dict(kv=k, status=st)


def ngram_propose(tokens: np.ndarray, lengths: np.ndarray, n_min: int, n_max: int, k: int, lib=None) -> dict:
    """n-gram lookup drafts.  tokens [B, Lmax] int32, lengths [B].  Returns
    draft [B, k] (-1 padded), count [B], match_len [B], match_end [B]."""
    lib = _load(lib)
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    B, Lmax = t.shape
    ln = _c(lengths, np.int32)
    out = dict(draft=np.empty((B, k), np.int32), count=np.empty(B, np.int32),
               match_len=np.empty(B, np.int32), match_end=np.empty(B, np.int32))
    rc = lib.oracle_ngram_propose(_ptr(t), _ptr(ln), B, Lmax, int(n_min), int(n_max), int(k),
                                  _ptr(out["draft"]), _ptr(out["count"]), _ptr(out["match_len"]),
                                  _ptr(out["match_end"]))
    if rc != 0:
        raise ValueError("oracle_ngram_propose rejected its arguments")
    return out


def fixup_slots(slot_mapping: np.ndarray, num_accepted: Optional[np.ndarray] = None,
                path: Optional[np.ndarray] = None, pad: int = -1, lib=None) -> np.ndarray:
    """Returns a fixed-up copy of slot_mapping [B, P]."""
    lib = _load(lib)
    s = np.array(slot_mapping, dtype=np.int64, copy=True, order="C")
    B, P = s.shape
    na = _c(num_accepted, np.int32)
    pa = _c(path, np.int32)
    stride = 0 if pa is None else pa.shape[1]
    rc = lib.oracle_fixup_slots(_ptr(s), B, P, _ptr(na), _ptr(pa), stride, int(pad))
    if rc != 0:
        raise ValueError("oracle_fixup_slots rejected its arguments")
    return s


# ---------------------------------------------------------------------------
# tree metadata (vLLM EAGLE walkthrough, "tree drafting in detail")
# ---------------------------------------------------------------------------
def tree_level_metadata(tree_choices: Sequence[Sequence[int]]):
    """Depth is the length of the last tuple; level l holds the tuples of length
    l+1; cu_drafts_per_level is the running total of the per-level counts and
    child_drafts_per_level[l] = count[l] // count[l-1] (count[0] at level 0)."""
    depth = len(tree_choices[-1])
    counts = [0] * depth
    for node in tree_choices:
        counts[len(node) - 1] += 1
    cu = [counts[0]]
    child = [counts[0]]
    for lvl in range(1, depth):
        cu.append(cu[-1] + counts[lvl])
        child.append(counts[lvl] // counts[lvl - 1])
    return dict(depth=depth, num_drafts_per_level=counts, cu_drafts_per_level=cu,
                child_drafts_per_level=child)


def parent_from_choices(tree_choices: Sequence[Sequence[int]]) -> np.ndarray:
    """Node n (1-based, in tree_choices order) is the tuple tree_choices[n-1]; its
    parent is the node whose tuple is that tuple minus its last entry (the empty
    tuple is the root, node 0)."""
    index = {(): 0}
    parent = [-1]
    for n, t in enumerate(tree_choices, start=1):
        t = tuple(int(v) for v in t)
        parent.append(index[t[:-1]])
        index[t] = n
    return np.asarray(parent, dtype=np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parent), dtype=np.int32)
    for n in range(1, len(parent)):
        d[n] = d[parent[n]] + 1
    return d
