"""GB300-native speculative-decoding verify-and-accept.

Every step of the path runs in the CUDA library ``libspecverify.so`` (C ABI in
``include/spec_verify.h``).  This module only marshals torch tensors into that
ABI: it checks dtypes, devices and contiguity, passes ``data_ptr()`` values and
the current CUDA stream, and keeps a zero-initialised workspace per
(device, stream).  There is no CPU fallback: if the library is missing or the
device is not sm_103, every call raises.

Entry points (names as in the C ABI):

* :func:`verify_chain`  -- chain verification, greedy (T = 0) or sampled.
* :func:`verify_tree`   -- greedy EAGLE-style token-tree verification.
* :func:`fixup_slots`   -- rewrite rejected KV slots to PADDING_SLOT_ID.
* :func:`tree_from_choices` -- tree_choices -> parent[] and level metadata.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

__all__ = ["verify_chain", "verify_tree", "fixup_slots", "tree_from_choices", "workspace_bytes",
           "SpecError", "PADDING_SLOT_ID", "STATUS_TOKEN_RANGE", "STATUS_NONFINITE",
           "STATUS_WAIT_TIMEOUT", "STATUS_BAD_OFFSETS", "STATUS_BAD_TEMPERATURE", "STATUS_SLOT_RANGE", "verify_tree_sampled", "prepare_next_step",
           "compact_tree_kv", "library_path", "load_library", "verify_chain_noalloc",
           "verify_chain_ragged", "fixup_slots_ragged", "ngram_propose"]

PADDING_SLOT_ID = -1
SPEC_BF16, SPEC_FP32 = 0, 1
STATUS_TOKEN_RANGE, STATUS_NONFINITE, STATUS_WAIT_TIMEOUT, STATUS_BAD_OFFSETS = 1, 2, 4, 8
STATUS_BAD_TEMPERATURE, STATUS_SLOT_RANGE = 16, 32
MAX_ROWS = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libspecverify.so")
_lock = threading.Lock()
_lib = None
_workspaces = {}

_STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED", 3: "SPEC_ERR_CUDA"}


class SpecError(RuntimeError):
    """A non-zero spec_status_t from the library."""

    def __init__(self, fn: str, code: int, detail: str):
        super().__init__("%s -> %s: %s" % (fn, _STATUS_NAMES.get(code, code), detail))
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libspecverify.so (built by ``__graft_entry__.build()`` or
    ``python -m speculative_decoding_verification_chain_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        import torch  # noqa: F401  (load torch's CUDA runtime first so both share it)
        if not os.path.exists(_LIB_PATH):
            raise ImportError("libspecverify.so is not built (%s); run the build step first" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.spec_workspace_bytes.argtypes = [I, I, I, I]
        lib.spec_workspace_bytes.restype = Z
        lib.spec_workspace_init.argtypes = [P, Z, P]
        lib.spec_workspace_init.restype = I
        lib.spec_verify_chain.argtypes = [P, I, P, P, P, P, P, I, I, I, P, P, P, P, Z, P]
        lib.spec_verify_chain.restype = I
        lib.spec_verify_chain_fused.argtypes = [P, I, P, P, P, P, P, I, I, I, P, P, P, ctypes.c_int64, P, P, Z, P]
        lib.spec_verify_chain_fused.restype = I
        lib.spec_verify_chain_ragged_fused.argtypes = [P, I, P, P, P, I, P, P, P, I, I, I, P, P, P, ctypes.c_int64,
                                                       P, P, Z, P]
        lib.spec_verify_chain_ragged_fused.restype = I
        lib.spec_verify_chain_ragged.argtypes = [P, I, P, P, P, I, P, P, P, I, I, I, P, P, P, P, Z, P]
        lib.spec_verify_chain_ragged.restype = I
        lib.spec_fixup_slots_ragged.argtypes = [P, I, P, I, P, ctypes.c_int64, P]
        lib.spec_fixup_slots_ragged.restype = I
        lib.spec_ngram_propose.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
        lib.spec_ngram_propose.restype = I
        lib.spec_verify_tree.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, P, Z, P]
        lib.spec_verify_tree_sampled.argtypes = [P, I, P, P, P, P, P, P, I, I, I, I, P, P, P, P, P]
        L = ctypes.c_int64
        lib.spec_prepare_next_step.argtypes = [P, I, P, P, P, I, I, I, I, I, P, P, L, L, P, P, P, P, P, P, P]
        lib.spec_compact_tree_kv.argtypes = [P, L, L, P, I, P, I, P, I, P, P]
        lib.spec_verify_tree.restype = I
        lib.spec_fixup_slots.argtypes = [P, I, I, P, P, I, ctypes.c_int64, P]
        lib.spec_fixup_slots.restype = I
        lib.spec_tree_from_choices.argtypes = [P, P, I, P, P, P, P]
        lib.spec_tree_from_choices.restype = I
        lib.spec_verify_chain_noalloc.argtypes = [P, I, P, P, P, P, P, I, I, I, P, P, P, P]
        lib.spec_verify_chain_noalloc.restype = I
        lib.spec_noalloc_scratch_bytes.argtypes = []
        lib.spec_noalloc_scratch_bytes.restype = Z
        lib.spec_last_error.argtypes = []
        lib.spec_last_error.restype = ctypes.c_char_p
        lib.spec_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.spec_set_wait_limit_ns.restype = ctypes.c_ulonglong
        lib.spec_set_tuning.argtypes = [I, I, I]
        lib.spec_set_tuning.restype = I
        _lib = lib
        return lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise SpecError(fn, rc, load_library().spec_last_error().decode(errors="replace"))


# ------------------------------------------------------------------ torch --
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_FP32
    raise TypeError("target_logits must be bfloat16 or float32, got %s" % t.dtype)


def _need(t, name, dtype, shape, device):
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if t.device != device:
        raise ValueError("%s must be on %s, got %s" % (name, device, t.device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _stream_handle(device, stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def workspace_bytes(B: int, rows: int, V: int, dtype_code: int = SPEC_BF16) -> int:
    n = load_library().spec_workspace_bytes(int(B), int(rows), int(V), int(dtype_code))
    if n == 0:
        raise SpecError("spec_workspace_bytes", 1, "invalid sizes B=%d rows=%d V=%d" % (B, rows, V))
    return int(n)


def _workspace(device, stream_handle: int, nbytes: int, layout: tuple):
    """Device workspace kept per (device, stream).  The library leaves its
    counters zero after every call for the same layout; a workspace that is
    new, grown, or last used with a different (B, rows, V, dtype) is
    zero-filled first, on the call's stream."""
    torch = _torch()
    key = (device.index, stream_handle)
    ent = _workspaces.get(key)
    if ent is None or ent[0].numel() < nbytes:
        ent = [torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device), layout]
        _workspaces[key] = ent
    elif ent[1] != layout:
        _check("spec_workspace_init", load_library().spec_workspace_init(ent[0].data_ptr(), ent[0].numel(),
                                                                       stream_handle))
        ent[1] = layout
    return ent[0]


def workspace_for(device=None, stream=None):
    """The cached workspace tensor used for calls on (device, stream), or None."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ent = _workspaces.get((device.index, _stream_handle(device, stream)))
    return None if ent is None else ent[0]


def workspace_counters(ws) -> dict:
    """Diagnostic counters the kernel accumulates at workspace offset 0:
    A units loaded / skipped, B units loaded / skipped, bytes streamed."""
    v = ws[:64].view(_torch().int64).cpu().tolist()
    return dict(a_loaded=v[0], a_skipped=v[1], b_loaded=v[2], b_skipped=v[3], bytes_loaded=v[4])


def reset_counters(ws):
    ws[:64].zero_()


def set_wait_limit_ns(ns: int) -> int:
    """spec_set_wait_limit_ns: limit of the kernels' inter-block waits (test
    setting; default 0.5 s).  Returns the previous limit."""
    return int(load_library().spec_set_wait_limit_ns(int(ns)))


def set_tuning(splits: int = 0, ahead: int = 0, path: int = 0):
    """spec_set_tuning: row splits and copy-ring depth of the persistent verify
    kernel (0 = automatic), and path (0 = automatic: sampled padded chains that
    fit go to the cluster-per-request kernel, greedy trees and greedy padded
    chains with fewer than two rows per SM to the grid of clusters; 1 = the
    persistent kernel for every batch; 2 = as 0, with every greedy padded chain
    on the grid of clusters)."""
    _check("spec_set_tuning", load_library().spec_set_tuning(int(splits), int(ahead), int(path)))


# ---------------------------------------------------------------- entries --
def verify_chain(target_logits, draft_tokens, temperature=None, u_accept=None, u_sample=None,
                 draft_probs=None, *, out_tokens=None, out_num_accepted=None, status=None,
                 workspace=None, stream=None, slot_mapping=None,
                 padding_slot_id: int = PADDING_SLOT_ID) -> Tuple[object, object]:
    """Chain verify-and-accept on the GPU.

    With ``slot_mapping`` ([B, k+1] int64 CUDA) the slot fix-up runs in the
    same launch: entries j > num_accepted[b] become ``padding_slot_id``.

    A caller-supplied ``workspace`` (uint8 CUDA tensor of at least
    workspace_bytes(B, k+1, V) bytes) must be zero-filled before its first use
    and again whenever it is reused for a different (B, k, V, dtype).

    target_logits [B, k+1, V] bf16/fp32 CUDA; draft_tokens [B, k] int32.
    Sampled requests (temperature > 0) also need draft_probs [B, k, V] fp32,
    u_accept [B, k] and u_sample [B, k+1] fp32.  With temperature None every
    request is greedy.  Returns (out_tokens [B, k+1] int32, num_accepted [B] int32).
    """
    torch = _torch()
    lib = load_library()
    z = target_logits
    if z.dim() != 3:
        raise ValueError("target_logits must be [B, k+1, V]")
    B, k1, V = z.shape
    k = k1 - 1
    dev = z.device
    if dev.type != "cuda":
        raise ValueError("target_logits must be a CUDA tensor")
    if not z.is_contiguous():
        raise ValueError("target_logits must be contiguous")
    code = _dtype_code(z)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(u_accept, "u_accept", torch.float32, (B, k), dev)
    _need(u_sample, "u_sample", torch.float32, (B, k + 1), dev)
    _need(draft_probs, "draft_probs", torch.float32, (B, k, V), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    _need(slot_mapping, "slot_mapping", torch.int64, (B, k + 1), dev)
    sh = _stream_handle(dev, stream)
    nbytes = workspace_bytes(B, k + 1, V, code)
    ws = workspace if workspace is not None else _workspace(dev, sh, nbytes, ("chain", B, k + 1, V, code))
    if slot_mapping is not None:
        rc = lib.spec_verify_chain_fused(_ptr(z), code, _ptr(draft_probs), _ptr(draft_tokens), _ptr(temperature),
                                         _ptr(u_accept), _ptr(u_sample), B, k, V, _ptr(out_tokens),
                                         _ptr(out_num_accepted), _ptr(slot_mapping), int(padding_slot_id),
                                         _ptr(status), _ptr(ws), ws.numel(), sh)
        _check("spec_verify_chain_fused", rc)
    else:
        rc = lib.spec_verify_chain(_ptr(z), code, _ptr(draft_probs), _ptr(draft_tokens), _ptr(temperature),
                                   _ptr(u_accept), _ptr(u_sample), B, k, V, _ptr(out_tokens),
                                   _ptr(out_num_accepted), _ptr(status), _ptr(ws), ws.numel(), sh)
        _check("spec_verify_chain", rc)
    return out_tokens, out_num_accepted


def verify_chain_ragged(target_logits, draft_tokens, cu_num_draft_tokens, max_k: int, temperature=None,
                        u_accept=None, u_sample=None, draft_probs=None, *, out_tokens=None,
                        out_num_accepted=None, status=None, workspace=None, stream=None, slot_mapping=None,
                        padding_slot_id: int = PADDING_SLOT_ID) -> Tuple[object, object]:
    """Chain verify-and-accept with a different number of drafts per request.

    With ``slot_mapping`` ([cu[B] + B] int64 CUDA, packed like the logits rows)
    the ragged slot fix-up runs in the same launch.

    cu_num_draft_tokens [B+1] int32 CUDA (cu[0] = 0, non-decreasing): request b
    has k_b = cu[b+1] - cu[b] <= max_k drafts.  target_logits [cu[B] + B, V]
    packed rows (request b's k_b + 1 rows from row cu[b] + b); draft_tokens and
    u_accept [cu[B]], draft_probs [cu[B], V] packed from row cu[b]; u_sample
    [cu[B] + B] packed like the logits rows; temperature [B].  Returns
    (out_tokens [B, max_k+1] int32 padded with -1, num_accepted [B] int32).
    """
    torch = _torch()
    lib = load_library()
    z = target_logits
    if z.dim() != 2 or z.device.type != "cuda" or not z.is_contiguous():
        raise ValueError("target_logits must be a contiguous [rows, V] CUDA tensor")
    rows, V = z.shape
    dev = z.device
    cu = cu_num_draft_tokens
    if cu.dtype != torch.int32 or cu.dim() != 1 or cu.device != dev or not cu.is_contiguous():
        raise ValueError("cu_num_draft_tokens must be a contiguous [B+1] int32 tensor on the logits' device")
    B = cu.shape[0] - 1
    total = rows - B
    if B < 1 or total < 0:
        raise ValueError("target_logits must hold cu[B] + B rows")
    code = _dtype_code(z)
    _need(draft_tokens, "draft_tokens", torch.int32, (total,), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(u_accept, "u_accept", torch.float32, (total,), dev)
    _need(u_sample, "u_sample", torch.float32, (total + B,), dev)
    _need(draft_probs, "draft_probs", torch.float32, (total, V), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, max_k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, max_k + 1), dev)
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    _need(slot_mapping, "slot_mapping", torch.int64, (total + B,), dev)
    sh = _stream_handle(dev, stream)
    nbytes = workspace_bytes(B, max_k + 1, V, code)
    ws = workspace if workspace is not None else _workspace(dev, sh, nbytes, ("chain", B, max_k + 1, V, code))
    if slot_mapping is not None:
        rc = lib.spec_verify_chain_ragged_fused(_ptr(z), code, _ptr(draft_probs), _ptr(draft_tokens), _ptr(cu),
                                                total, _ptr(temperature), _ptr(u_accept), _ptr(u_sample), B, max_k,
                                                V, _ptr(out_tokens), _ptr(out_num_accepted), _ptr(slot_mapping),
                                                int(padding_slot_id), _ptr(status), _ptr(ws), ws.numel(), sh)
        _check("spec_verify_chain_ragged_fused", rc)
    else:
        rc = lib.spec_verify_chain_ragged(_ptr(z), code, _ptr(draft_probs), _ptr(draft_tokens), _ptr(cu), total,
                                          _ptr(temperature), _ptr(u_accept), _ptr(u_sample), B, max_k, V,
                                          _ptr(out_tokens), _ptr(out_num_accepted), _ptr(status), _ptr(ws),
                                          ws.numel(), sh)
        _check("spec_verify_chain_ragged", rc)
    return out_tokens, out_num_accepted


def fixup_slots_ragged(slot_mapping, cu_num_draft_tokens, num_accepted, padding_slot_id: int = PADDING_SLOT_ID,
                       stream=None):
    """In-place fix-up of packed slots ([cu[B] + B] int64 CUDA): request b's
    slots start at cu[b] + b; slot j is kept iff j <= num_accepted[b]."""
    torch = _torch()
    lib = load_library()
    cu = cu_num_draft_tokens
    if slot_mapping.dtype != torch.int64 or slot_mapping.dim() != 1 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous 1-D int64 tensor")
    dev = slot_mapping.device
    if cu.dtype != torch.int32 or cu.dim() != 1 or cu.device != dev:
        raise ValueError("cu_num_draft_tokens must be a [B+1] int32 tensor on the slots' device")
    B = cu.shape[0] - 1
    total = slot_mapping.shape[0] - B
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    rc = lib.spec_fixup_slots_ragged(_ptr(slot_mapping), B, _ptr(cu), total, _ptr(num_accepted),
                                     int(padding_slot_id), _stream_handle(dev, stream))
    _check("spec_fixup_slots_ragged", rc)
    return slot_mapping


def ngram_propose(tokens, lengths, n_min: int, n_max: int, k: int, *, out_draft=None, out_count=None,
                  out_match_len=None, out_match_end=None, stream=None):
    """n-gram lookup drafts.  tokens [B, Lmax] int32 CUDA (row b's first
    lengths[b] entries are its text), lengths [B] int32 CUDA.  Returns
    (draft [B, k] int32 -1 padded, count [B], match_len [B], match_end [B])."""
    torch = _torch()
    lib = load_library()
    if tokens.dtype != torch.int32 or tokens.dim() != 2 or tokens.device.type != "cuda" or not tokens.is_contiguous():
        raise ValueError("tokens must be a contiguous [B, Lmax] int32 CUDA tensor")
    B, Lmax = tokens.shape
    dev = tokens.device
    _need(lengths, "lengths", torch.int32, (B,), dev)
    mk = lambda t, shape: t if t is not None else torch.empty(shape, dtype=torch.int32, device=dev)
    out_draft, out_count = mk(out_draft, (B, k)), mk(out_count, (B,))
    out_match_len, out_match_end = mk(out_match_len, (B,)), mk(out_match_end, (B,))
    for t, name, shape in ((out_draft, "out_draft", (B, k)), (out_count, "out_count", (B,)),
                           (out_match_len, "out_match_len", (B,)), (out_match_end, "out_match_end", (B,))):
        _need(t, name, torch.int32, shape, dev)
    rc = lib.spec_ngram_propose(_ptr(tokens), _ptr(lengths), B, Lmax, int(n_min), int(n_max), int(k), _ptr(out_draft),
                                _ptr(out_count), _ptr(out_match_len), _ptr(out_match_end), _stream_handle(dev, stream))
    _check("spec_ngram_propose", rc)
    return out_draft, out_count, out_match_len, out_match_end


def verify_tree(target_logits, node_tokens, parent: Sequence[int], max_depth: Optional[int] = None, *,
                out_path=None, out_tokens=None, out_len=None, status=None, workspace=None,
                stream=None):
    """Greedy token-tree verify on the GPU.

    target_logits [B, N+1, V] bf16/fp32 CUDA; node_tokens [B, N] int32 CUDA;
    parent: N+1 host integers (parent[0] = -1, level order).  Returns
    (out_path [B, D+1], out_tokens [B, D+1], out_len [B]) int32 CUDA tensors.
    """
    torch = _torch()
    import numpy as np
    lib = load_library()
    z = target_logits
    if z.dim() != 3:
        raise ValueError("target_logits must be [B, N+1, V]")
    B, n1, V = z.shape
    N = n1 - 1
    dev = z.device
    if dev.type != "cuda" or not z.is_contiguous():
        raise ValueError("target_logits must be a contiguous CUDA tensor")
    code = _dtype_code(z)
    par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    if par.shape != (N + 1,):
        raise ValueError("parent must hold N+1 = %d entries" % (N + 1))
    if max_depth is None:
        d = np.zeros(N + 1, np.int64)
        for n in range(1, N + 1):
            d[n] = d[par[n]] + 1 if 0 <= par[n] < n else 0
        max_depth = int(d.max())
    _need(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    D1 = max_depth + 1
    if out_path is None:
        out_path = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    sh = _stream_handle(dev, stream)
    nbytes = workspace_bytes(B, N + 1, V, code)
    ws = workspace if workspace is not None else _workspace(dev, sh, nbytes, ("tree", B, N + 1, V, code))
    rc = lib.spec_verify_tree(_ptr(z), code, _ptr(node_tokens), par.ctypes.data, B, N, V, int(max_depth),
                              _ptr(out_path), _ptr(out_tokens), _ptr(out_len), _ptr(status), _ptr(ws),
                              ws.numel(), sh)
    _check("spec_verify_tree", rc)
    return out_path, out_tokens, out_len


def verify_tree_sampled(target_logits, draft_probs, node_tokens, parent: Sequence[int], temperature, u_accept,
                        u_sample, max_depth: Optional[int] = None, *, out_path=None, out_tokens=None, out_len=None,
                        status=None, stream=None):
    """Sampled token-tree verify on the GPU (children tested in index order,
    residual after each rejected sibling, one draw where the walk stops).

    target_logits [B, N+1, V] bf16/fp32 CUDA; draft_probs [B, N+1, V] fp32
    CUDA (row c: the law of c's children); node_tokens [B, N] int32;
    temperature [B] fp32 (> 0); u_accept [B, N] and u_sample [B, N+1] fp32;
    parent: N+1 host integers.  Returns (out_path, out_tokens, out_len)."""
    torch = _torch()
    import numpy as np
    lib = load_library()
    z = target_logits
    if z.dim() != 3:
        raise ValueError("target_logits must be [B, N+1, V]")
    B, n1, V = z.shape
    N = n1 - 1
    dev = z.device
    if dev.type != "cuda" or not z.is_contiguous():
        raise ValueError("target_logits must be a contiguous CUDA tensor")
    code = _dtype_code(z)
    par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    if par.shape != (N + 1,):
        raise ValueError("parent must hold N+1 = %d entries" % (N + 1))
    if max_depth is None:
        d = np.zeros(N + 1, np.int64)
        for n in range(1, N + 1):
            d[n] = d[par[n]] + 1 if 0 <= par[n] < n else 0
        max_depth = int(d.max())
    _need(draft_probs, "draft_probs", torch.float32, (B, N + 1, V), dev)
    _need(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(u_accept, "u_accept", torch.float32, (B, N), dev)
    _need(u_sample, "u_sample", torch.float32, (B, N + 1), dev)
    D1 = max_depth + 1
    if out_path is None:
        out_path = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    rc = lib.spec_verify_tree_sampled(_ptr(z), code, _ptr(draft_probs), _ptr(node_tokens), par.ctypes.data,
                                      _ptr(temperature), _ptr(u_accept), _ptr(u_sample), B, N, V, int(max_depth),
                                      _ptr(out_path), _ptr(out_tokens), _ptr(out_len), _ptr(status),
                                      _stream_handle(dev, stream))
    _check("spec_verify_tree_sampled", rc)
    return out_path, out_tokens, out_len


def prepare_next_step(out_tokens, num_accepted, positions, block_table, block_size: int, P_next: int, *,
                      rows_per_req: Optional[int] = None, cu_num_draft_tokens=None, hidden=None,
                      padding_slot_id: int = PADDING_SLOT_ID, status=None, stream=None):
    """Next-step inputs after verification (all CUDA tensors).

    out_tokens [B, S] int32; num_accepted [B] int32 (out_len - 1 for trees);
    positions [B] int32 (sequence position of row 0); block_table [B, M]
    int32; hidden [rows, H] (any dtype) or None.  Returns (next_token [B],
    next_position [B], next_slots [B, P_next] int64, last_row [B],
    hidden_out [B, H] or None)."""
    torch = _torch()
    lib = load_library()
    if out_tokens.dtype != torch.int32 or out_tokens.dim() != 2 or out_tokens.device.type != "cuda" \
            or not out_tokens.is_contiguous():
        raise ValueError("out_tokens must be a contiguous [B, S] int32 CUDA tensor")
    B, stride = out_tokens.shape
    dev = out_tokens.device
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    _need(positions, "positions", torch.int32, (B,), dev)
    if block_table is None or block_table.dim() != 2:
        raise ValueError("block_table must be a [B, max_blocks] int32 CUDA tensor")
    _need(block_table, "block_table", torch.int32, (B, block_table.shape[1]), dev)
    if cu_num_draft_tokens is not None:
        _need(cu_num_draft_tokens, "cu_num_draft_tokens", torch.int32, (B + 1,), dev)
        rpr = 0
    else:
        rpr = int(rows_per_req if rows_per_req is not None else stride)
    row_bytes = 0
    hidden_out = None
    if hidden is not None:
        if hidden.device != dev or not hidden.is_contiguous() or hidden.dim() < 2:
            raise ValueError("hidden must be a contiguous [rows, ...] CUDA tensor on the same device")
        row_bytes = hidden[0].numel() * hidden.element_size()
        hidden_out = torch.empty((B,) + tuple(hidden.shape[1:]), dtype=hidden.dtype, device=dev)
    mk = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
    next_token, next_position, last_row = mk((B,), torch.int32), mk((B,), torch.int32), mk((B,), torch.int32)
    next_slots = mk((B, P_next), torch.int64)
    rc = lib.spec_prepare_next_step(_ptr(out_tokens), stride, _ptr(num_accepted), _ptr(positions), _ptr(block_table),
                                    block_table.shape[1], int(block_size), B, int(P_next), rpr,
                                    _ptr(cu_num_draft_tokens), _ptr(hidden), int(row_bytes), int(padding_slot_id),
                                    _ptr(next_token), _ptr(next_position), _ptr(next_slots), _ptr(last_row),
                                    _ptr(hidden_out), _ptr(status), _stream_handle(dev, stream))
    _check("spec_prepare_next_step", rc)
    return next_token, next_position, next_slots, last_row, hidden_out


def compact_tree_kv(kv, slot_mapping, path, out_len, *, status=None, stream=None):
    """Tree KV compaction in place: kv [num_slots, ...] CUDA (rows a multiple of
    16 bytes), slot_mapping [B, N+1] int64, path [B, D+1] int32, out_len [B]
    int32 (as verify_tree / verify_tree_sampled return them)."""
    torch = _torch()
    lib = load_library()
    if kv.device.type != "cuda" or not kv.is_contiguous() or kv.dim() < 1:
        raise ValueError("kv must be a contiguous CUDA tensor [num_slots, ...]")
    dev = kv.device
    num_slots = kv.shape[0]
    row_bytes = (kv[0].numel() * kv.element_size()) if num_slots else 16
    if slot_mapping.dim() != 2 or path.dim() != 2:
        raise ValueError("slot_mapping and path must be 2-D")
    B = slot_mapping.shape[0]
    _need(slot_mapping, "slot_mapping", torch.int64, tuple(slot_mapping.shape), dev)
    _need(path, "path", torch.int32, (B, path.shape[1]), dev)
    _need(out_len, "out_len", torch.int32, (B,), dev)
    rc = lib.spec_compact_tree_kv(_ptr(kv), num_slots, int(row_bytes), _ptr(slot_mapping), slot_mapping.shape[1],
                                  _ptr(path), path.shape[1], _ptr(out_len), B, _ptr(status),
                                  _stream_handle(dev, stream))
    _check("spec_compact_tree_kv", rc)
    return kv


def fixup_slots(slot_mapping, num_accepted=None, path=None, padding_slot_id: int = PADDING_SLOT_ID,
                stream=None):
    """In-place slot_mapping fix-up ([B, P] int64 CUDA).  Chain mode with
    num_accepted [B] int32, or tree mode with path [B, D+1] int32."""
    torch = _torch()
    lib = load_library()
    if slot_mapping.dtype != torch.int64 or slot_mapping.dim() != 2 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous [B, P] int64 tensor")
    B, P = slot_mapping.shape
    dev = slot_mapping.device
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    if path is not None:
        if path.dtype != torch.int32 or path.dim() != 2 or path.shape[0] != B or not path.is_contiguous():
            raise ValueError("path must be a contiguous [B, D+1] int32 tensor")
    stride = 0 if path is None else path.shape[1]
    rc = lib.spec_fixup_slots(_ptr(slot_mapping), B, P, _ptr(num_accepted), _ptr(path), stride,
                              int(padding_slot_id), _stream_handle(dev, stream))
    _check("spec_fixup_slots", rc)
    return slot_mapping


def tree_from_choices(tree_choices: Sequence[Sequence[int]]) -> dict:
    """tree_choices (level-ordered tuples) -> parent[], cu/child drafts per level, depth."""
    import numpy as np
    lib = load_library()
    n = len(tree_choices)
    lens = np.asarray([len(t) for t in tree_choices], dtype=np.int32)
    flat = np.asarray([v for t in tree_choices for v in t] or [0], dtype=np.int32)
    parent = np.zeros(n + 1, dtype=np.int32)
    cu = np.zeros(MAX_ROWS, dtype=np.int32)
    child = np.zeros(MAX_ROWS, dtype=np.int32)
    depth = ctypes.c_int(0)
    rc = lib.spec_tree_from_choices(flat.ctypes.data, lens.ctypes.data, n, parent.ctypes.data,
                                    cu.ctypes.data, child.ctypes.data, ctypes.byref(depth))
    _check("spec_tree_from_choices", rc)
    d = depth.value
    return dict(parent=parent, cu_drafts_per_level=cu[:d].tolist(),
                child_drafts_per_level=child[:d].tolist(), depth=d)


def verify_chain_noalloc(target_logits, draft_tokens, temperature=None, u_accept=None, u_sample=None,
                         draft_probs=None, *, out_tokens=None, out_num_accepted=None, status=None, stream=None):
    """verify_chain without a workspace, for callers that cannot allocate device
    memory: the library uses its own fixed 16 MiB device scratch, shared by all
    calls (serialise calls that could overlap on the GPU).  Same arguments and
    results as verify_chain; larger sizes raise SpecError."""
    torch = _torch()
    lib = load_library()
    z = target_logits
    if z.dim() != 3 or z.device.type != "cuda" or not z.is_contiguous():
        raise ValueError("target_logits must be a contiguous [B, k+1, V] CUDA tensor")
    B, k1, V = z.shape
    k = k1 - 1
    dev = z.device
    code = _dtype_code(z)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(u_accept, "u_accept", torch.float32, (B, k), dev)
    _need(u_sample, "u_sample", torch.float32, (B, k + 1), dev)
    _need(draft_probs, "draft_probs", torch.float32, (B, k, V), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, k + 1), dev)
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    rc = lib.spec_verify_chain_noalloc(_ptr(z), code, _ptr(draft_probs), _ptr(draft_tokens), _ptr(temperature),
                                       _ptr(u_accept), _ptr(u_sample), B, k, V, _ptr(out_tokens),
                                       _ptr(out_num_accepted), _ptr(status), _stream_handle(dev, stream))
    _check("spec_verify_chain_noalloc", rc)
    return out_tokens, out_num_accepted
