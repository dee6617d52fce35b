"""The attention parity inputs are strong enough that a kernel which skipped a
page, a block row or mis-weighted a split would fail the 2e-2 tolerance. The
mistakes are planted in the oracle, on the CPU: the oracle is evaluated with
one needle page left out (its page-table entry pointed at a page holding other
keys) and with the block's last row left out, and each must move the output by
far more than the tolerance."""
import dataclasses

import numpy as np
import torch

import oracle as O
from block_diffusion_speculative_fusion_gb300 import synth
from block_diffusion_speculative_fusion_gb300 import workloads as W

TOL = 2e-2


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _needle_case(ctx):
    wl = dataclasses.replace(W.LLAMA8B_B64, B=len(ctx))
    cache = synth.paged_cache(wl, headroom=16, seed=5, layers=1, ctx_len=torch.tensor(ctx, dtype=torch.int32))
    blk = synth.block_qkv(wl, 0, seed=5)
    where = synth.plant_needles(wl, blk, cache, seed=5)
    return wl, cache, blk, where


def _attn(blk, cache, wl, page_table=None, n_kv=None):
    kb, vb = f64(blk["k_blk"]), f64(blk["v_blk"])
    if n_kv is not None:
        kb, vb = kb[:, :n_kv], vb[:, :n_kv]
    pt = cache.page_table.numpy() if page_table is None else page_table
    return O.block_attn(f64(blk["q"]), kb, vb, f64(cache.k_pools[0]), f64(cache.v_pools[0]), pt,
                        cache.ctx_len.numpy(), wl.page_size)


def test_needles_make_a_skipped_page_visible():
    wl, cache, blk, where = _needle_case([8192, 3000])
    full = _attn(blk, cache, wl)
    assert np.abs(full).max() < 4.0          # outputs stay where bf16 rounding is far below 2e-2
    for b in range(2):
        for p in where[b]:
            pt = cache.page_table.numpy().copy()
            other = p // wl.page_size + 1 if p // wl.page_size + 1 < pt.shape[1] and \
                (p // wl.page_size + 1) * wl.page_size < int(cache.ctx_len[b]) else p // wl.page_size - 1
            pt[b, p // wl.page_size] = pt[b, other]      # the needle's page replaced by a neighbour
            moved = np.abs(_attn(blk, cache, wl, page_table=pt)[b] - full[b]).max()
            assert moved > 5 * TOL, (b, p, moved)


def test_needles_make_a_skipped_block_row_visible():
    wl, cache, blk, where = _needle_case([8192, 600])
    full = _attn(blk, cache, wl)
    dropped = _attn(blk, cache, wl, n_kv=wl.k - 1)
    assert np.abs(dropped - full).max(axis=(1, 2, 3)).min() > 5 * TOL
