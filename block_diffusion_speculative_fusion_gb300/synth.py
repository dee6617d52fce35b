"""Seeded synthetic inputs for the DFlash hot path.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle's tests. It draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no log-sum-exp, no acceptance rule, no
attention, no projection). Sampled draft tokens are drawn with the Gumbel-max
trick, which is the upstream draft model's job, not part of the verify.

Every tensor comes from its own torch generator seeded with (seed, tag), so any
one tensor can be regenerated alone. Results are CPU tensors unless a device is
given; on a device the values come from that device's generator (the bulk KV
pools of the throughput bench), which is fine for timing but means CPU and
device draws differ.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass
from typing import Dict, List, Optional

import torch

from .workloads import Workload

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def io_dtype(wl: Workload) -> torch.dtype:
    return _TORCH_DTYPE[wl.dtype]


def _gen(seed: int, tag: str, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(tag.encode())) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _randn(shape, seed, tag, std=1.0, device="cpu"):
    g = _gen(seed, tag, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def _rand(shape, seed, tag, device="cpu"):
    return torch.rand(*shape, generator=_gen(seed, tag, device), device=device,
                      dtype=torch.float32)


def _randint(lo, hi, shape, seed, tag):
    """Integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, shape, generator=_gen(seed, tag), dtype=torch.int64)


def ctx_lengths(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Committed context length C_b per sequence, uniform on [ctx_lo, ctx_hi]."""
    return _randint(wl.ctx_lo, wl.ctx_hi, (wl.B,), seed, "ctx_len").to(torch.int32)


# ---------------------------------------------------------------------------
# Paged draft KV cache
# ---------------------------------------------------------------------------
@dataclass
class PagedCache:
    page_table: torch.Tensor     # [B, max_pages] int32, physical page per logical page
    ctx_len: torch.Tensor        # [B] int32
    num_pages: int
    max_pages: int
    k_pools: List[torch.Tensor]  # L x [num_pages, page, Hkv, D]
    v_pools: List[torch.Tensor]


def page_table(wl: Workload, ctx_len: torch.Tensor, headroom: int, seed: int = 0):
    """Assign each sequence ceil((C_b + headroom) / page) pages, drawn as a seeded
    random permutation of the pool so that logical neighbours are not physical ones."""
    P = wl.page_size
    need = [(int(c) + headroom + P - 1) // P for c in ctx_len.tolist()]
    max_pages = max(need)
    num_pages = sum(need)
    perm = torch.randperm(num_pages, generator=_gen(seed, "page_perm")).to(torch.int32)
    pt = torch.full((wl.B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, num_pages, max_pages


def paged_cache(wl: Workload, headroom: int, seed: int = 0, device: str = "cpu",
                layers: Optional[int] = None, ctx_len: Optional[torch.Tensor] = None) -> PagedCache:
    """Ctx K/V pools filled with N(0, 1) values (K after RMS norm has unit RMS;
    V is drawn at the same scale) in the I/O dtype."""
    if ctx_len is None:
        ctx_len = ctx_lengths(wl, seed)
    pt, num_pages, max_pages = page_table(wl, ctx_len, headroom, seed)
    L = wl.L if layers is None else layers
    dt = io_dtype(wl)
    shape = (num_pages, wl.page_size, wl.Hkv, wl.D)
    ks, vs = [], []
    for layer in range(L):
        ks.append(_randn(shape, seed, f"kpool{layer}", device=device).to(dt))
        vs.append(_randn(shape, seed, f"vpool{layer}", device=device).to(dt))
    return PagedCache(pt, ctx_len, num_pages, max_pages, ks, vs)


# ---------------------------------------------------------------------------
# Draft block (queries and the block's own K/V) for one draft layer
# ---------------------------------------------------------------------------
def block_qkv(wl: Workload, layer: int, seed: int = 0, n_kv_blk: Optional[int] = None,
              device: str = "cpu") -> Dict[str, torch.Tensor]:
    dt = io_dtype(wl)
    nkv = wl.k if n_kv_blk is None else n_kv_blk
    return {
        "q": _randn((wl.B, wl.k, wl.Hq, wl.D), seed, f"q{layer}", device=device).to(dt),
        "k_blk": _randn((wl.B, nkv, wl.Hkv, wl.D), seed, f"kb{layer}", device=device).to(dt),
        "v_blk": _randn((wl.B, nkv, wl.Hkv, wl.D), seed, f"vb{layer}", device=device).to(dt),
    }


# ---------------------------------------------------------------------------
# Materialisation weights and captured hidden states
# ---------------------------------------------------------------------------
def ctx_weights(wl: Workload, seed: int = 0) -> Dict[str, torch.Tensor]:
    """W_f [d, m*d], b_f [d], W_kv [L, 2, Hkv*D, d], k_norm_w [L, D] (or None)."""
    dt = io_dtype(wl)
    md = wl.m * wl.d
    std_f = wl.weight_std if wl.weight_std is not None else 1.0 / math.sqrt(md)
    std_kv = wl.weight_std if wl.weight_std is not None else 1.0 / math.sqrt(wl.d)
    std_b = wl.weight_std if wl.weight_std is not None else 1.0 / math.sqrt(md)
    out = {
        "W_f": _randn((wl.d, md), seed, "W_f", std_f).to(dt),
        "b_f": _randn((wl.d,), seed, "b_f", std_b).to(dt),
        "W_kv": _randn((wl.L, 2, wl.Hkv * wl.D, wl.d), seed, "W_kv", std_kv).to(dt),
        "k_norm_w": None,
    }
    if wl.k_norm:
        out["k_norm_w"] = (1.0 + _randn((wl.L, wl.D), seed, "k_norm_w", 0.1)).to(dt)
    return out


def captured_hidden(wl: Workload, rows: int, seed: int = 0, B: Optional[int] = None,
                    tag: str = "hidden") -> torch.Tensor:
    """Row-wise concatenation [h_l1; ...; h_lm] of the captured target layers,
    [B, rows, m*d], each entry N(0, hidden_std^2)."""
    B = wl.B if B is None else B
    return _randn((B, rows, wl.m * wl.d), seed, tag, wl.hidden_std).to(io_dtype(wl))


# ---------------------------------------------------------------------------
# Verify inputs: draft logits, target logits, candidates, uniforms
# ---------------------------------------------------------------------------
def _gumbel_pick(z: torch.Tensor, temperature: float, seed: int, tag: str) -> torch.Tensor:
    """Draw one index per row of z from softmax(z / temperature) by Gumbel-max."""
    u = _rand(z.shape, seed, tag).clamp_(min=1e-30)
    gumbel = -torch.log(-torch.log(u))
    return torch.argmax(z.float() / temperature + gumbel, dim=-1)


def draft_logits(wl: Workload, rows: int, seed: int, tag: str, B: Optional[int] = None) -> torch.Tensor:
    """Draft logits [B, rows, V]: N(0, base_std^2) plus a peak offset
    A ~ U[lo, hi] added to one uniformly chosen token of each row (or one offset
    per sequence when ``peak_per_sequence``)."""
    B = wl.B if B is None else B
    z = _randn((B, rows, wl.V), seed, tag + "_base", wl.draft_base_std)
    tok = torch.randint(0, wl.V, (B, rows), generator=_gen(seed, tag + "_tok"))
    lo, hi = wl.draft_peak
    if wl.peak_per_sequence:
        amp = (lo + (hi - lo) * _rand((B, 1), seed, tag + "_amp")).expand(B, rows)
    else:
        amp = lo + (hi - lo) * _rand((B, rows), seed, tag + "_amp")
    z.scatter_add_(2, tok.unsqueeze(-1), amp.unsqueeze(-1).contiguous())
    return z.to(io_dtype(wl))


def verify_batch(wl: Workload, seed: int = 0, sigma: Optional[float] = None,
                 n_max: Optional[int] = None, B: Optional[int] = None,
                 greedy_rows: Optional[int] = None, ragged: bool = False) -> Dict[str, torch.Tensor]:
    """One verify problem.

    target_logits [B, n_max+1, V]: row r is the target's distribution after
      consuming cand[0..r]; rows r < n_max equal the draft row r plus
      N(0, sigma^2) noise, row n_max is a fresh draft-like row plus noise.
    draft_logits [B, n_max, V]: row i-1 is the draft distribution of position i.
    cand [B, n_max+1] int64: cand[:, 0] is the anchor; cand[:, i] is the draft's
      argmax of row i-1 for greedy sequences and a draw from softmax(row/T) for
      sampled ones (the verify's q).
    n_draft [B] int32 (all n_max unless ragged), u_acc [B, n_max] and
    u_final [B] float32 uniforms on [0, 1).
    """
    B = wl.B if B is None else B
    n = wl.n_max if n_max is None else n_max
    sigma = wl.sigma if sigma is None else sigma
    n_greedy = wl.n_greedy if greedy_rows is None else greedy_rows
    n_greedy = min(n_greedy, B)
    dt = io_dtype(wl)
    zd = draft_logits(wl, n + 1, seed, "zd", B=B)          # row n: bonus-row base
    noise = _randn((B, n + 1, wl.V), seed, "zt_noise", sigma)
    zt = (zd.float() + noise).to(dt)
    zd_rows = zd[:, :n].contiguous()
    cand = torch.empty((B, n + 1), dtype=torch.int64)
    cand[:, 0] = torch.randint(0, wl.V, (B,), generator=_gen(seed, "anchor"))
    if n > 0:
        if n_greedy > 0:
            cand[:n_greedy, 1:] = torch.argmax(zd_rows[:n_greedy].float(), dim=-1)
        if n_greedy < B:
            cand[n_greedy:, 1:] = _gumbel_pick(zd_rows[n_greedy:], wl.temperature, seed, "gumbel")
    if ragged:
        n_draft = _randint(0, n, (B,), seed, "n_draft").to(torch.int32)
    else:
        n_draft = torch.full((B,), n, dtype=torch.int32)
    return {
        "target_logits": zt.contiguous(),
        "draft_logits": zd_rows,
        "cand": cand,
        "n_draft": n_draft,
        "u_acc": _rand((B, max(n, 1)), seed, "u_acc")[:, :n].contiguous(),
        "u_final": _rand((B,), seed, "u_final"),
    }


def draft_select_batch(wl: Workload, seed: int = 0, B: Optional[int] = None, n_max: Optional[int] = None,
                       ragged: bool = False) -> Dict[str, torch.Tensor]:
    """One draft-side token choice problem: the draft's MASK-position logits
    [B, n_max, V] (same law as the verify's draft rows), the anchor [B], one
    uniform per MASK position [B, n_max] and n_draft [B] (all n_max unless
    ragged)."""
    B = wl.B if B is None else B
    n = wl.n_max if n_max is None else n_max
    zd = draft_logits(wl, n, seed, "sel_zd", B=B)
    n_draft = (_randint(0, n, (B,), seed, "sel_n").to(torch.int32) if ragged
               else torch.full((B,), n, dtype=torch.int32))
    return {
        "draft_logits": zd.contiguous(),
        "anchor": torch.randint(0, wl.V, (B,), generator=_gen(seed, "sel_anchor")),
        "u_draft": _rand((B, n), seed, "sel_u"),
        "n_draft": n_draft,
    }


def ddtree_target_logits(wl: Workload, node_token: torch.Tensor, node_parent: torch.Tensor, n_nodes: torch.Tensor,
                         seed: int = 0, p_follow: float = 0.7, device: str = "cpu") -> torch.Tensor:
    """Target logits [B, budget + 1, V] for a draft tree: row 0 is the target
    after the anchor, row 1 + j after the path to node j. Each row is N(0, 1)
    noise plus a peak of 10 on one token: with probability ``p_follow`` the
    token of the row's first child in the tree (so walks run several levels),
    else a uniformly drawn token."""
    B, budget = node_token.shape
    R = budget + 1
    z = _randn((B, R, wl.V), seed, "tree_zt", device=device)
    follow = _rand((B, R), seed, "tree_follow") < p_follow
    peak = torch.randint(0, wl.V, (B, R), generator=_gen(seed, "tree_tok"))
    tok = node_token.cpu()
    par = node_parent.cpu()
    nn = n_nodes.cpu()
    for b in range(B):
        first = {}
        for j in range(int(nn[b])):
            first.setdefault(int(par[b, j]), int(tok[b, j]))
        for r in range(R):
            if bool(follow[b, r]) and (r - 1) in first:
                peak[b, r] = first[r - 1]
    z.scatter_add_(2, peak.to(z.device)[:, :, None], torch.full((B, R, 1), 10.0, device=z.device))
    return z.to(io_dtype(wl))


def gate_batch(wl: Workload, stage: int, seed: int = 0, B: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """One DLoop gate problem for draft stage ``stage``: draft logits [B, k, V] of
    the stage's k drafted tokens, the tokens drawn from softmax(logits / T), and
    an all-active mask."""
    B = wl.B if B is None else B
    z = draft_logits(wl, wl.n_draft, seed, f"gate{stage}", B=B)
    tok = _gumbel_pick(z, wl.temperature, seed, f"gate{stage}_pick")
    return {"draft_logits": z, "tokens": tok, "active": torch.ones((B,), dtype=torch.uint8)}


def plant_needles(wl: Workload, blk: Dict[str, torch.Tensor], cache: PagedCache, seed: int = 0,
                  q_shift: float = 3.0, key_norm: float = 35.0, v_offset: float = 2.0,
                  layer: int = 0) -> List[List[int]]:
    """Attention inputs in which every context page that holds a needle, and
    the block's first and last rows, carry a visible share of the output.

    Per sequence b: a random unit direction u_b is added to every query row
    (q += q_shift * u_b, all heads); "needle" keys equal key_norm * u_b (all kv
    heads) at context positions 0, C/3, C/2, 2C/3, C-1 and at block rows 0 and
    n_kv-1, each with its own value row N(0, 0.5^2) + v_offset. Needle scores
    then stand ~q_shift * key_norm / sqrt(D) above the N(0, 1) background, so
    each needle takes several percent of every row's attention and shifts the
    output by far more than the 2e-2 tolerance if its page (or block row) is
    skipped. Edits ``blk`` and ``cache`` (layer ``layer``) in place; returns
    the needle positions of each sequence."""
    B, n_kv = blk["k_blk"].shape[0], blk["k_blk"].shape[1]
    g = _gen(seed, "needles")
    dt = blk["q"].dtype
    u = torch.randn(B, wl.D, generator=g)
    u = u / u.norm(dim=1, keepdim=True)
    blk["q"].copy_((blk["q"].float() + q_shift * u[:, None, None, :]).to(dt))
    kp, vp = cache.k_pools[layer], cache.v_pools[layer]
    P = wl.page_size
    where = []
    for b in range(B):
        C = int(cache.ctx_len[b])
        pos = sorted({p for p in (0, C // 3, C // 2, (2 * C) // 3, C - 1) if 0 <= p < C})
        where.append(pos)
        for p in pos:
            page = int(cache.page_table[b, p // P])
            kp[page, p % P] = (key_norm * u[b]).to(kp.dtype).expand(wl.Hkv, wl.D)
            vp[page, p % P] = (v_offset + 0.5 * torch.randn(wl.Hkv, wl.D, generator=g)).to(vp.dtype)
        for r in sorted({0, n_kv - 1}):
            blk["k_blk"][b, r] = (key_norm * u[b]).to(dt).expand(wl.Hkv, wl.D)
            blk["v_blk"][b, r] = (v_offset + 0.5 * torch.randn(wl.Hkv, wl.D, generator=g)).to(dt)
    return where
