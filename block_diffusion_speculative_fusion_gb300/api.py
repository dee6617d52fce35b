"""Thin Python binding of libdflash (ctypes): argument marshalling only.

Every function takes torch CUDA tensors, checks their dtype, shape and
contiguity, and passes raw device pointers plus the current CUDA stream to the
C ABI declared in ``include/dflash.h``. All arithmetic runs in the library's
kernels; there is no fallback path. Workspaces are zero-initialised device
buffers cached per device and stream-ordered like every other tensor.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4
F32, BF16 = 0, 1
FLAG_ACCEPT_BOUNDARY, FLAG_CDF_BOUNDARY, FLAG_DEGENERATE, FLAG_INVALID = 1, 2, 4, 8
FLAG_GATE_BOUNDARY = 1
WS_COUNTER_BYTES = 16384
WS_ERROR_WORD_OFFSET = WS_COUNTER_BYTES - 4
DEVERR_BAD_PAGE = 100
DEVERR_BAD_N_DRAFT = 101
# recorded only by the debug library (select_library(debug=True))
DEVERR_BAD_CTX_LEN, DEVERR_BAD_COMMIT_LEN, DEVERR_BAD_POSITION = 102, 103, 104


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dflash error {code}: {msg}")
        self.code = code


c_i32 = ctypes.c_int32
c_p = ctypes.c_void_p


class CtxKvDims(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("B", "rows_max", "m", "d", "L", "Hkv", "D", "page_size",
                                     "max_pages", "num_pages", "dtype")]


class AttnDims(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("B", "n_q", "n_kv_blk", "Hq", "Hkv", "D", "page_size",
                                     "max_pages", "num_pages", "max_ctx", "dtype", "causal")]


class VerifyDims(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("B", "n_max", "V", "dtype")]


class GateDims(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("B", "k", "V", "dtype")]


class TreeDims(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("B", "n", "V", "dtype", "K", "budget")]


_SIGS = {
    "dflash_last_error": (ctypes.c_char_p, []),
    "dflash_last_launch_count": (ctypes.c_int, []),
    "dflash_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "dflash_wait_limit_ns": (ctypes.c_uint64, []),
    "dflash_verify_greedy_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(VerifyDims)]),
    "dflash_verify_greedy": (ctypes.c_int, [ctypes.POINTER(VerifyDims), c_p, c_p, c_p, c_p, c_p, c_p,
                                            c_p, c_p, c_p, ctypes.c_size_t, c_p]),
    "dflash_verify_greedy_noalloc": (ctypes.c_int, [ctypes.POINTER(VerifyDims), c_p, c_p, c_p, c_p, c_p,
                                                    c_p, c_p, c_p, c_p]),
    "dflash_verify_sample_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(VerifyDims)]),
    "dflash_verify_sample": (ctypes.c_int, [ctypes.POINTER(VerifyDims), ctypes.c_float, c_p, c_p, c_p,
                                            c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p,
                                            ctypes.c_size_t, c_p]),
    "dflash_gate_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(GateDims)]),
    "dflash_gate": (ctypes.c_int, [ctypes.POINTER(GateDims), ctypes.c_float, ctypes.c_float, c_p, c_p,
                                   c_p, c_p, c_p, c_p, c_p, c_p, ctypes.c_size_t, c_p]),
    # dims, stage, n_max, T, g, draft_logits, cand, active, c_s, cont, row_lse, flags, n_verify, ws, bytes, stream
    "dflash_gate_stage": (ctypes.c_int, [ctypes.POINTER(GateDims), ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                         ctypes.c_float] + [c_p] * 9 + [ctypes.c_size_t, c_p]),
    # dims, T, target, draft, draft_row_lse, cand, n_draft, u_accept, u_final, accept_len, bonus,
    # commit_len, out_tokens, flags, probs, workspace, ws_bytes, stream
    "dflash_verify_sample_lse": (ctypes.c_int, [ctypes.POINTER(VerifyDims), ctypes.c_float] + [c_p] * 14 +
                                 [ctypes.c_size_t, c_p]),
    "dflash_ddtree_topk": (ctypes.c_int, [ctypes.POINTER(TreeDims), ctypes.c_float, c_p, c_p, c_p, c_p]),
    "dflash_ddtree_build": (ctypes.c_int, [ctypes.POINTER(TreeDims)] + [c_p] * 9),
    "dflash_ddtree_verify_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(TreeDims)]),
    "dflash_ddtree_verify_greedy": (ctypes.c_int, [ctypes.POINTER(TreeDims)] + [c_p] * 10 + [ctypes.c_size_t, c_p]),
    "dflash_draft_select_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(VerifyDims)]),
    "dflash_draft_select": (ctypes.c_int, [ctypes.POINTER(VerifyDims), ctypes.c_float, c_p, c_p, c_p, c_p, c_p,
                                           c_p, c_p, c_p, c_p, ctypes.c_size_t, c_p]),
    "dflash_block_attn_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnDims)]),
    "dflash_block_attn": (ctypes.c_int, [ctypes.POINTER(AttnDims), c_p, c_p, c_p, c_p, c_p, c_p, c_p,
                                         ctypes.c_float, c_p, c_p, ctypes.c_size_t, c_p]),
    "dflash_block_attn_active": (ctypes.c_int, [ctypes.POINTER(AttnDims), c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p,
                                                ctypes.c_float, c_p, c_p, ctypes.c_size_t, c_p]),
    "dflash_materialize_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(CtxKvDims)]),
    "dflash_materialize_ctx_kv": (ctypes.c_int, [ctypes.POINTER(CtxKvDims), c_p, c_p, c_p, c_p, c_p,
                                                 c_p, c_p, ctypes.c_float, ctypes.c_float, c_p, c_p,
                                                 c_p, c_p, c_p, ctypes.c_size_t, c_p]),
}

_lib = None
LIB_DEBUG_PATH = os.path.join(_HERE, "libdflash_debug.so")


def select_library(debug: bool = False) -> str:
    """Use libdflash.so, or libdflash_debug.so (built by ``build.build(debug=True)``,
    whose kernels also record clamped inputs in the error word), for every later
    call; returns its path."""
    global _lib, LIB_PATH
    LIB_PATH = LIB_DEBUG_PATH if debug else os.path.join(_HERE, "libdflash.so")
    _lib = None
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libdflash.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "block_diffusion_speculative_fusion_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name, None)
            if fn is None:
                continue
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().dflash_last_error().decode()


def last_launch_count() -> int:
    return int(lib().dflash_last_launch_count())


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the tensor-core kernels' bounded waits (``dflash_set_wait_limit_ns``);
    0 restores the 2 s default."""
    _check(lib().dflash_set_wait_limit_ns(int(ns)))


def wait_limit_ns() -> int:
    return int(lib().dflash_wait_limit_ns())


def _check(rc: int):
    if rc != OK:
        raise DflashError(rc, last_error())


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
_DT = {torch.float32: F32, torch.bfloat16: BF16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DT[t.dtype]


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _opt(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    return None if t is None else _dev(t, name, dtype, shape)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


_WS: Dict[Tuple[int, int], torch.Tensor] = {}


def workspace(device: torch.device, nbytes: int, slot: int = 0) -> torch.Tensor:
    """A zero-initialised device workspace of at least ``nbytes`` (cached per
    device and slot; calls on one stream may share a slot)."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    key = (idx, slot)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, WS_COUNTER_BYTES), dtype=torch.uint8, device=f"cuda:{idx}")
        _WS[key] = ws
    return ws


def reset_workspaces():
    _WS.clear()


# ---------------------------------------------------------------------------
# (c) verify
# ---------------------------------------------------------------------------
def verify_greedy(target_logits: torch.Tensor, cand: torch.Tensor, n_draft: Optional[torch.Tensor] = None,
                  want_target_pred: bool = False, out: Optional[dict] = None, ws: Optional[torch.Tensor] = None):
    """Greedy accept rule (``dflash_verify_greedy``). Returns a dict of device
    tensors: accept_len, bonus, commit_len, out_tokens[, target_pred]."""
    _dev(target_logits, "target_logits")
    B, R, V = target_logits.shape
    n_max = R - 1
    dev = target_logits.device
    dims = VerifyDims(B, n_max, V, _dtype_code(target_logits))
    o = out if out is not None else {}
    o.setdefault("accept_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("bonus", torch.empty(B, dtype=torch.int64, device=dev))
    o.setdefault("commit_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("out_tokens", torch.empty((B, R), dtype=torch.int64, device=dev))
    if want_target_pred:
        o.setdefault("target_pred", torch.empty((B, R), dtype=torch.int64, device=dev))
    need = lib().dflash_verify_greedy_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    rc = lib().dflash_verify_greedy(
        ctypes.byref(dims), _dev(target_logits, "target_logits"), _dev(cand, "cand", torch.int64, (B, R)),
        _opt(n_draft, "n_draft", torch.int32, (B,)),
        _dev(o["accept_len"], "accept_len", torch.int32), _dev(o["bonus"], "bonus", torch.int64),
        _dev(o["commit_len"], "commit_len", torch.int32), _opt(o.get("out_tokens"), "out_tokens", torch.int64),
        _opt(o.get("target_pred"), "target_pred", torch.int64), w.data_ptr(), w.numel(), _stream(dev))
    _check(rc)
    return o


def verify_greedy_noalloc(target_logits: torch.Tensor, cand: torch.Tensor, n_draft: Optional[torch.Tensor] = None,
                          want_target_pred: bool = False, out: Optional[dict] = None):
    """Greedy accept rule on the library's fixed scratch
    (``dflash_verify_greedy_noalloc``). Outputs are caller tensors (``out``),
    created here only when not given; the C call itself allocates nothing."""
    _dev(target_logits, "target_logits")
    B, R, V = target_logits.shape
    dev = target_logits.device
    dims = VerifyDims(B, R - 1, V, _dtype_code(target_logits))
    o = out if out is not None else {}
    o.setdefault("accept_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("bonus", torch.empty(B, dtype=torch.int64, device=dev))
    o.setdefault("commit_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("out_tokens", torch.empty((B, R), dtype=torch.int64, device=dev))
    if want_target_pred:
        o.setdefault("target_pred", torch.empty((B, R), dtype=torch.int64, device=dev))
    rc = lib().dflash_verify_greedy_noalloc(
        ctypes.byref(dims), _dev(target_logits, "target_logits"), _dev(cand, "cand", torch.int64, (B, R)),
        _opt(n_draft, "n_draft", torch.int32, (B,)),
        _dev(o["accept_len"], "accept_len", torch.int32), _dev(o["bonus"], "bonus", torch.int64),
        _dev(o["commit_len"], "commit_len", torch.int32), _opt(o.get("out_tokens"), "out_tokens", torch.int64),
        _opt(o.get("target_pred"), "target_pred", torch.int64), _stream(dev))
    _check(rc)
    return o


def verify_sample(target_logits: torch.Tensor, draft_logits: torch.Tensor, cand: torch.Tensor,
                  u_accept: torch.Tensor, u_final: torch.Tensor, temperature: float = 1.0,
                  n_draft: Optional[torch.Tensor] = None, want_probs: bool = False,
                  out: Optional[dict] = None, ws: Optional[torch.Tensor] = None,
                  draft_row_lse: Optional[torch.Tensor] = None):
    """Sampled accept rule with residual resample (``dflash_verify_sample``).
    With ``draft_row_lse`` [B, n_max] (LSE(draft row / T), e.g. the DLoop
    gates' row_lse) the draft rows are not streamed
    (``dflash_verify_sample_lse``). Returns accept_len, bonus, commit_len,
    out_tokens, flags[, probs]."""
    _dev(target_logits, "target_logits")
    B, R, V = target_logits.shape
    n_max = R - 1
    dev = target_logits.device
    dt = _dtype_code(target_logits)
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("draft_logits and target_logits must share a dtype")
    dims = VerifyDims(B, n_max, V, dt)
    o = out if out is not None else {}
    o.setdefault("accept_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("bonus", torch.empty(B, dtype=torch.int64, device=dev))
    o.setdefault("commit_len", torch.empty(B, dtype=torch.int32, device=dev))
    o.setdefault("out_tokens", torch.empty((B, R), dtype=torch.int64, device=dev))
    o.setdefault("flags", torch.empty(B, dtype=torch.uint8, device=dev))
    if want_probs:
        o.setdefault("probs", torch.empty((B, 2 * n_max + 1), dtype=torch.float32, device=dev))
    need = lib().dflash_verify_sample_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    head = [ctypes.byref(dims), ctypes.c_float(temperature), _dev(target_logits, "target_logits"),
            _dev(draft_logits, "draft_logits", None, (B, n_max, V))]
    if draft_row_lse is not None:
        fn = lib().dflash_verify_sample_lse
        head.append(_dev(draft_row_lse, "draft_row_lse", torch.float32, (B, n_max)))
    else:
        fn = lib().dflash_verify_sample
    rc = fn(
        *head, _dev(cand, "cand", torch.int64, (B, R)),
        _opt(n_draft, "n_draft", torch.int32, (B,)), _dev(u_accept, "u_accept", torch.float32, (B, n_max)),
        _dev(u_final, "u_final", torch.float32, (B,)),
        _dev(o["accept_len"], "accept_len", torch.int32), _dev(o["bonus"], "bonus", torch.int64),
        _dev(o["commit_len"], "commit_len", torch.int32), _opt(o.get("out_tokens"), "out_tokens", torch.int64),
        _opt(o.get("flags"), "flags", torch.uint8), _opt(o.get("probs"), "probs", torch.float32),
        w.data_ptr(), w.numel(), _stream(dev))
    _check(rc)
    return o


# ---------------------------------------------------------------------------
# DLoop gate
# ---------------------------------------------------------------------------
def gate(draft_logits: torch.Tensor, tokens: torch.Tensor, temperature: float = 1.0, g: float = -0.5,
         active: Optional[torch.Tensor] = None, want_row_lse: bool = False,
         out: Optional[dict] = None, ws: Optional[torch.Tensor] = None):
    """DLoop block gate (``dflash_gate``). Returns c, cont, flags[, row_lse]."""
    _dev(draft_logits, "draft_logits")
    B, k, V = draft_logits.shape
    dev = draft_logits.device
    dims = GateDims(B, k, V, _dtype_code(draft_logits))
    o = out if out is not None else {}
    o.setdefault("c", torch.empty(B, dtype=torch.float32, device=dev))
    o.setdefault("cont", torch.empty(B, dtype=torch.uint8, device=dev))
    o.setdefault("flags", torch.empty(B, dtype=torch.uint8, device=dev))
    if want_row_lse:
        o.setdefault("row_lse", torch.empty((B, k), dtype=torch.float32, device=dev))
    need = lib().dflash_gate_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    rc = lib().dflash_gate(
        ctypes.byref(dims), ctypes.c_float(temperature), ctypes.c_float(g), _dev(draft_logits, "draft_logits"),
        _dev(tokens, "tokens", torch.int64, (B, k)), _opt(active, "active", torch.uint8, (B,)),
        _dev(o["c"], "c", torch.float32), _dev(o["cont"], "cont", torch.uint8),
        _opt(o.get("row_lse"), "row_lse", torch.float32), _opt(o.get("flags"), "flags", torch.uint8),
        w.data_ptr(), w.numel(), _stream(dev))
    _check(rc)
    return o


def gate_stage(draft_logits: torch.Tensor, cand: torch.Tensor, stage: int, k: int, temperature: float = 1.0,
               g: float = -0.5, active: Optional[torch.Tensor] = None, row_lse: Optional[torch.Tensor] = None,
               n_verify: Optional[torch.Tensor] = None, out: Optional[dict] = None,
               ws: Optional[torch.Tensor] = None):
    """One DLoop stage's gate on the looped layout (``dflash_gate_stage``):
    draft_logits [B, n_max, V], cand [B, n_max + 1]; stage s's rows are
    s*k .. s*k + k - 1. ``row_lse`` [B, n_max] and ``n_verify`` [B] are
    accumulated across stages. Returns c, cont, flags."""
    _dev(draft_logits, "draft_logits")
    B, n_max, V = draft_logits.shape
    dev = draft_logits.device
    dims = GateDims(B, k, V, _dtype_code(draft_logits))
    o = out if out is not None else {}
    o.setdefault("c", torch.empty(B, dtype=torch.float32, device=dev))
    o.setdefault("cont", torch.empty(B, dtype=torch.uint8, device=dev))
    o.setdefault("flags", torch.empty(B, dtype=torch.uint8, device=dev))
    need = lib().dflash_gate_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    rc = lib().dflash_gate_stage(
        ctypes.byref(dims), int(stage), int(n_max), ctypes.c_float(temperature), ctypes.c_float(g),
        _dev(draft_logits, "draft_logits"), _dev(cand, "cand", torch.int64, (B, n_max + 1)),
        _opt(active, "active", torch.uint8, (B,)), _dev(o["c"], "c", torch.float32),
        _dev(o["cont"], "cont", torch.uint8), _opt(row_lse, "row_lse", torch.float32, (B, n_max)),
        _opt(o.get("flags"), "flags", torch.uint8), _opt(n_verify, "n_verify", torch.int32, (B,)),
        w.data_ptr(), w.numel(), _stream(dev))
    _check(rc)
    return o


def draft_select(draft_logits: torch.Tensor, anchor: torch.Tensor, temperature: float = 0.0,
                 u_draft: Optional[torch.Tensor] = None, n_draft: Optional[torch.Tensor] = None,
                 out: Optional[dict] = None, ws: Optional[torch.Tensor] = None):
    """Candidates from the draft's MASK-position logits (``dflash_draft_select``):
    argmax (temperature 0) or one inverse-CDF sample per row with ``u_draft``.
    Returns cand [B, n_max+1] int64, q_x and row_lse [B, n_max] float32, flags
    [B, n_max] uint8."""
    _dev(draft_logits, "draft_logits")
    B, n_max, V = draft_logits.shape
    dev = draft_logits.device
    dims = VerifyDims(B, n_max, V, _dtype_code(draft_logits))
    o = out if out is not None else {}
    if "cand" not in o:
        o["cand"] = torch.empty((B, n_max + 1), dtype=torch.int64, device=dev)
        o["q_x"] = torch.empty((B, n_max), dtype=torch.float32, device=dev)
        o["row_lse"] = torch.empty((B, n_max), dtype=torch.float32, device=dev)
        o["flags"] = torch.empty((B, n_max), dtype=torch.uint8, device=dev)
    need = lib().dflash_draft_select_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    rc = lib().dflash_draft_select(
        ctypes.byref(dims), ctypes.c_float(temperature), _dev(draft_logits, "draft_logits"),
        _dev(anchor, "anchor", torch.int64, (B,)), _opt(n_draft, "n_draft", torch.int32, (B,)),
        _opt(u_draft if temperature > 0 else None, "u_draft", torch.float32, (B, n_max)),
        _dev(o["cand"], "cand", torch.int64, (B, n_max + 1)), _opt(o.get("q_x"), "q_x", torch.float32),
        _opt(o.get("row_lse"), "row_lse", torch.float32), _opt(o.get("flags"), "flags", torch.uint8),
        w.data_ptr(), w.numel(), _stream(dev))
    _check(rc)
    return o


# ---------------------------------------------------------------------------
# DDTree
# ---------------------------------------------------------------------------
def ddtree_topk(draft_logits: torch.Tensor, K: int, temperature: float = 1.0, out: Optional[dict] = None):
    """Top-K tokens and their log-probabilities of every drafted position
    (``dflash_ddtree_topk``): tok [B, n, K] int64, logp [B, n, K] float32."""
    _dev(draft_logits, "draft_logits")
    B, n, V = draft_logits.shape
    dev = draft_logits.device
    dims = TreeDims(B, n, V, _dtype_code(draft_logits), K, 1)
    o = out if out is not None else {}
    if "tok" not in o:
        o["tok"] = torch.empty((B, n, K), dtype=torch.int64, device=dev)
        o["logp"] = torch.empty((B, n, K), dtype=torch.float32, device=dev)
    _check(lib().dflash_ddtree_topk(ctypes.byref(dims), ctypes.c_float(temperature), _dev(draft_logits, "draft_logits"),
                                    _dev(o["tok"], "tok", torch.int64, (B, n, K)),
                                    _dev(o["logp"], "logp", torch.float32, (B, n, K)), _stream(dev)))
    return o


def ddtree_build(tok: torch.Tensor, logp: torch.Tensor, budget: int, V: int = 1, out: Optional[dict] = None):
    """Best-first draft tree within ``budget`` nodes (``dflash_ddtree_build``):
    node_token, node_parent, node_depth, node_logp [B, budget], n_nodes [B],
    flags [B]."""
    B, n, K = tok.shape
    dev = tok.device
    dims = TreeDims(B, n, max(V, K), BF16, K, budget)
    o = out if out is not None else {}
    if "node_token" not in o:
        o["node_token"] = torch.empty((B, budget), dtype=torch.int64, device=dev)
        o["node_parent"] = torch.empty((B, budget), dtype=torch.int32, device=dev)
        o["node_depth"] = torch.empty((B, budget), dtype=torch.int32, device=dev)
        o["node_logp"] = torch.empty((B, budget), dtype=torch.float32, device=dev)
        o["n_nodes"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["flags"] = torch.empty(B, dtype=torch.uint8, device=dev)
    _check(lib().dflash_ddtree_build(
        ctypes.byref(dims), _dev(tok, "tok", torch.int64, (B, n, K)), _dev(logp, "logp", torch.float32, (B, n, K)),
        _dev(o["node_token"], "node_token", torch.int64), _dev(o["node_parent"], "node_parent", torch.int32),
        _dev(o["node_depth"], "node_depth", torch.int32), _dev(o["node_logp"], "node_logp", torch.float32),
        _dev(o["n_nodes"], "n_nodes", torch.int32), _opt(o.get("flags"), "flags", torch.uint8), _stream(dev)))
    return o


def ddtree_verify_greedy(target_logits: torch.Tensor, node_token: torch.Tensor, node_parent: torch.Tensor,
                         n_nodes: torch.Tensor, n: int, K: int, out: Optional[dict] = None,
                         ws: Optional[torch.Tensor] = None):
    """Greedy walk of the verified tree (``dflash_ddtree_verify_greedy``):
    accept_len, commit_len, bonus, path [B, budget], out_tokens [B, budget+1]."""
    _dev(target_logits, "target_logits")
    B, R, V = target_logits.shape
    budget = R - 1
    dev = target_logits.device
    dims = TreeDims(B, n, V, _dtype_code(target_logits), K, budget)
    o = out if out is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["bonus"] = torch.empty(B, dtype=torch.int64, device=dev)
        o["commit_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["path"] = torch.empty((B, budget), dtype=torch.int32, device=dev)
        o["out_tokens"] = torch.empty((B, R), dtype=torch.int64, device=dev)
    need = lib().dflash_ddtree_verify_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(dev, need)
    _check(lib().dflash_ddtree_verify_greedy(
        ctypes.byref(dims), _dev(target_logits, "target_logits"),
        _dev(node_token, "node_token", torch.int64, (B, budget)), _dev(node_parent, "node_parent", torch.int32, (B, budget)),
        _dev(n_nodes, "n_nodes", torch.int32, (B,)), _dev(o["accept_len"], "accept_len", torch.int32),
        _dev(o["bonus"], "bonus", torch.int64), _dev(o["commit_len"], "commit_len", torch.int32),
        _opt(o.get("path"), "path", torch.int32), _opt(o.get("out_tokens"), "out_tokens", torch.int64),
        w.data_ptr(), w.numel(), _stream(dev)))
    return o


# ---------------------------------------------------------------------------
# (b) block attention
# ---------------------------------------------------------------------------
def block_attn(q: torch.Tensor, k_blk: torch.Tensor, v_blk: torch.Tensor, k_pool: torch.Tensor,
               v_pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
               max_ctx: Optional[int] = None, scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
               causal: bool = False, active: Optional[torch.Tensor] = None) -> torch.Tensor:
    """GQA attention of the draft block over [paged context ; block]
    (``dflash_block_attn``): unmasked, or with ``causal`` the in-block causal
    variant (query i sees the context and block rows j <= i + n_kv - n_q).
    q [B, n_q, Hq, D]; k_blk, v_blk [B, n_kv, Hkv, D]; pools [num_pages, page,
    Hkv, D]; page_table [B, max_pages] int32; ctx_len [B] int32. ``max_ctx``
    bounds every ctx_len (defaults to the page table's capacity). With
    ``active`` [B] uint8 (``dflash_block_attn_active``) only the sequences with
    active[b] != 0 are computed; the other rows of ``out`` are left as they were."""
    _dev(q, "q")
    B, n_q, Hq, D = q.shape
    n_kv, Hkv = k_blk.shape[1], k_blk.shape[2]
    num_pages, page = k_pool.shape[0], k_pool.shape[1]
    max_pages = page_table.shape[1]
    if max_ctx is None:
        max_ctx = max_pages * page
    dt = _dtype_code(q)
    for name, t in (("k_blk", k_blk), ("v_blk", v_blk), ("k_pool", k_pool), ("v_pool", v_pool)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have the dtype of q")
    dims = AttnDims(B, n_q, n_kv, Hq, Hkv, D, page, max_pages, num_pages, int(max_ctx), dt, 1 if causal else 0)
    if out is None:
        out = torch.empty_like(q)
    need = lib().dflash_block_attn_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(q.device, need, slot=1)
    args = [ctypes.byref(dims), _dev(q, "q"), _dev(k_blk, "k_blk", None, (B, n_kv, Hkv, D)),
            _dev(v_blk, "v_blk", None, (B, n_kv, Hkv, D)), _dev(k_pool, "k_pool", None, (num_pages, page, Hkv, D)),
            _dev(v_pool, "v_pool", None, (num_pages, page, Hkv, D)),
            _dev(page_table, "page_table", torch.int32, (B, max_pages)),
            _dev(ctx_len, "ctx_len", torch.int32, (B,))]
    tail = [ctypes.c_float(scale if scale is not None else D ** -0.5), _dev(out, "out", q.dtype, q.shape),
            w.data_ptr(), w.numel(), _stream(q.device)]
    if active is None:
        rc = lib().dflash_block_attn(*args, *tail)
    else:
        rc = lib().dflash_block_attn_active(*args, _dev(active, "active", torch.uint8, (B,)), *tail)
    _check(rc)
    return out


def device_error_word(ws: torch.Tensor) -> int:
    """The sticky device-side error word of a workspace (0: no error; 1-99: a
    kernel gave up a bounded wait; DEVERR_BAD_PAGE: attention met a page-table
    entry outside the pools; DEVERR_BAD_N_DRAFT: a verify or draft-select call
    met an n_draft outside [0, n_max]; with the debug library also
    DEVERR_BAD_CTX_LEN, DEVERR_BAD_COMMIT_LEN, DEVERR_BAD_POSITION).
    Synchronises with the device to read it."""
    return int(ws[WS_ERROR_WORD_OFFSET:WS_COUNTER_BYTES].view(torch.int32).item())


def clear_counters(ws: torch.Tensor) -> None:
    """Zero a workspace's counter region (after a nonzero error word), on the
    current stream."""
    ws[:WS_COUNTER_BYTES].zero_()


def error_words() -> Dict[Tuple[int, int], int]:
    """Error word of every cached workspace (see ``workspace``), keyed by
    (device, slot)."""
    return {k: device_error_word(v) for k, v in _WS.items()}


# ---------------------------------------------------------------------------
# (a) context-KV materialisation
# ---------------------------------------------------------------------------
def materialize_ctx_kv(hidden: torch.Tensor, commit_len: torch.Tensor, start_pos: torch.Tensor,
                       W_f: torch.Tensor, b_f: Optional[torch.Tensor], W_kv: torch.Tensor,
                       k_norm_w: Optional[torch.Tensor], rms_eps: float, rope_theta: float,
                       k_pools: Sequence[torch.Tensor], v_pools: Sequence[torch.Tensor],
                       page_table: torch.Tensor, new_len: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None) -> None:
    """Write the committed rows' context K/V of every draft layer into the paged
    pools (``dflash_materialize_ctx_kv``). hidden [B, rows_max, m*d];
    W_f [d, m*d]; b_f [d] or None; W_kv [L, 2, Hkv*D, d]; k_norm_w [L, D] or
    None; pools: L tensors [num_pages, page, Hkv, D]; page_table [B, max_pages]."""
    _dev(hidden, "hidden")
    B, rows_max, md = hidden.shape
    d = W_f.shape[0]
    m = md // d
    L, two, HD, d2 = W_kv.shape
    if two != 2 or d2 != d or m * d != md:
        raise ValueError("inconsistent hidden / W_f / W_kv shapes")
    if len(k_pools) != L or len(v_pools) != L:
        raise ValueError("need one K and one V pool per draft layer")
    num_pages, page, Hkv, D = k_pools[0].shape
    if Hkv * D != HD:
        raise ValueError("pool head layout does not match W_kv")
    dt = _dtype_code(hidden)
    for name, t in (("W_f", W_f), ("W_kv", W_kv)):
        if t.dtype != hidden.dtype:
            raise TypeError(f"{name} must have the dtype of hidden")
    max_pages = page_table.shape[1]
    dims = CtxKvDims(B, rows_max, m, d, L, Hkv, D, page, max_pages, num_pages, dt)
    need = lib().dflash_materialize_workspace_size(ctypes.byref(dims))
    if need == 0:
        raise DflashError(ERR_INVALID_ARG, last_error())
    w = ws if ws is not None else workspace(hidden.device, need, slot=2)
    kp = (c_p * L)(*[_dev(t, f"k_pools[{i}]", hidden.dtype, (num_pages, page, Hkv, D)) for i, t in enumerate(k_pools)])
    vp = (c_p * L)(*[_dev(t, f"v_pools[{i}]", hidden.dtype, (num_pages, page, Hkv, D)) for i, t in enumerate(v_pools)])
    rc = lib().dflash_materialize_ctx_kv(
        ctypes.byref(dims), _dev(hidden, "hidden"), _dev(commit_len, "commit_len", torch.int32, (B,)),
        _dev(start_pos, "start_pos", torch.int32, (B,)), _dev(W_f, "W_f", None, (d, md)),
        _opt(b_f, "b_f", hidden.dtype, (d,)), _dev(W_kv, "W_kv"), _opt(k_norm_w, "k_norm_w", hidden.dtype, (L, D)),
        ctypes.c_float(rms_eps), ctypes.c_float(rope_theta), ctypes.cast(kp, c_p), ctypes.cast(vp, c_p),
        _dev(page_table, "page_table", torch.int32, (B, max_pages)), _opt(new_len, "new_len", torch.int32, (B,)),
        w.data_ptr(), w.numel(), _stream(hidden.device))
    _check(rc)
