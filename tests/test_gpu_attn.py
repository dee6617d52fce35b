"""GPU parity of the draft block attention against the CPU oracle (max-abs
2e-2 for bf16 I/O with fp32 accumulation; 1e-4 for the fp32 path)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_speculative_fusion_gb300 import api, synth
from block_diffusion_speculative_fusion_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_fusion_gb300 import build
    build.build()
    api.lib()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _case(wl, ctx, seed=0, n_q=None, n_kv=None, page=None, headroom=16, nan_tail=False):
    import dataclasses
    kw = {}
    if n_q is not None:
        kw["k"] = n_q
    if page is not None:
        kw["page_size"] = page
    w = dataclasses.replace(wl, B=len(ctx), **kw)
    ctx_len = torch.tensor(ctx, dtype=torch.int32)
    cache = synth.paged_cache(w, headroom=headroom, seed=seed, layers=1, ctx_len=ctx_len)
    blk = synth.block_qkv(w, 0, seed=seed, n_kv_blk=n_kv)
    if nan_tail:
        # rows past each context hold NaN: the kernel must mask them completely
        P = w.page_size
        for b, c in enumerate(ctx):
            for pos in range(c, cache.max_pages * P):
                pg = int(cache.page_table[b, pos // P])
                if pg >= 0:
                    cache.k_pools[0][pg, pos % P] = float("nan")
                    cache.v_pools[0][pg, pos % P] = float("nan")
    return w, cache, blk


def _run(w, cache, blk, atol, seqs=None, causal=False, repeat=1):
    args = [blk["q"].to(DEV), blk["k_blk"].to(DEV), blk["v_blk"].to(DEV), cache.k_pools[0].to(DEV),
            cache.v_pools[0].to(DEV), cache.page_table.to(DEV), cache.ctx_len.to(DEV)]
    out = api.block_attn(*args, causal=causal).clone()
    # repeated calls give the same bits: the partition of the work depends on
    # the dims and ctx_len only, and split pieces are merged in a fixed order
    for _ in range(repeat - 1):
        again = api.block_attn(*args, causal=causal)
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    torch.cuda.synchronize()
    got = f64(out)
    assert np.all(np.isfinite(got))
    seqs = range(w.B) if seqs is None else seqs
    pt = cache.page_table.numpy()
    for b in seqs:
        ref = O.block_attn(f64(blk["q"][b:b + 1]), f64(blk["k_blk"][b:b + 1]), f64(blk["v_blk"][b:b + 1]),
                           f64(cache.k_pools[0]), f64(cache.v_pools[0]), pt[b:b + 1],
                           cache.ctx_len.numpy()[b:b + 1], w.page_size, causal=causal)
        err = np.abs(got[b] - ref[0]).max()
        assert err < atol, (b, err)
    return got


def test_attn_tiny_f32_generic_path():
    wl = W.TINY_F32
    w, cache, blk = _case(wl, [32])
    _run(w, cache, blk, 1e-4)


def test_attn_tiny_f32_ragged():
    w, cache, blk = _case(W.TINY_F32, [0, 5, 31, 77], seed=3)
    _run(w, cache, blk, 1e-4)


@pytest.mark.parametrize("ctx", [[0, 1, 63, 64, 65], [37, 1024, 1100, 2100, 3000]])
def test_attn_bf16_tiles_splits_and_tails(ctx):
    w, cache, blk = _case(W.LLAMA8B_B64, ctx, seed=1)
    _run(w, cache, blk, 2e-2)


def test_attn_bf16_block_of_ten_m40():
    w, cache, blk = _case(W.LLAMA8B_B1, [2048, 700], seed=2)
    _run(w, cache, blk, 2e-2)


@pytest.mark.parametrize("stage", [1, 3])
def test_attn_bf16_dloop_stage_extra_rows(stage):
    wl = W.DLOOP_QWEN3_4B
    w, cache, blk = _case(wl, [1024, 1031, 500], seed=4, n_kv=wl.k + stage - 1)
    _run(w, cache, blk, 2e-2)


@pytest.mark.parametrize("page", [8, 32, 64])
def test_attn_bf16_page_sizes(page):
    w, cache, blk = _case(W.QWEN3_4B_B8, [1024, 333, 2049], seed=5, page=page)
    _run(w, cache, blk, 2e-2)


@pytest.mark.parametrize("ctx,hkv", [([2048], 8), ([1024, 333, 2049], 3)])
def test_attn_bf16_one_kv_head_per_item(ctx, hkv):
    # B * n_kv below one box of rows (B = 1) and an odd kv-head count both take
    # the one-head-per-item layout of the tensor-core kernel
    import dataclasses
    wl = W.LLAMA8B_B1 if hkv == 8 else dataclasses.replace(W.QWEN3_4B_B8, Hq=12, Hkv=3)
    w, cache, blk = _case(wl, ctx, seed=9)
    _run(w, cache, blk, 2e-2)


@pytest.mark.parametrize("ctx", [[17, 1030, 64], [49, 81, 113, 145, 1062, 1094, 2000, 7],
                                 [33, 65, 97, 129, 161, 193, 225, 257, 289, 321, 353, 385]])
def test_attn_bf16_masks_garbage_past_context(ctx):
    # pool rows past each context hold NaN; partial tiles land on both softmax
    # groups (tiles alternate between them), so every group must zero them
    w, cache, blk = _case(W.LLAMA8B_B64, ctx, seed=6, headroom=80, nan_tail=True)
    _run(w, cache, blk, 2e-2)


def test_attn_bf16_generic_fallback_shape():
    # D = 64 is outside the tensor-core kernel: the generic kernel serves it
    import dataclasses
    wl = dataclasses.replace(W.QWEN3_4B_B8, D=64)
    w, cache, blk = _case(wl, [100, 300], seed=7)
    _run(w, cache, blk, 2e-2)


def test_attn_full_size_batched_llama8b_b64_sampled_sequences():
    wl = W.LLAMA8B_B64
    ctx_len = synth.ctx_lengths(wl, 0)
    cache = synth.paged_cache(wl, headroom=16, seed=0, layers=1, ctx_len=ctx_len)
    blk = synth.block_qkv(wl, 0, seed=0)
    order = np.argsort(ctx_len.numpy())
    seqs = [int(order[0]), int(order[len(order) // 2]), int(order[-1]), 5]
    _run(wl, cache, blk, 2e-2, seqs=seqs, repeat=12)


def test_attn_deterministic_and_error_word_clear():
    w, cache, blk = _case(W.LLAMA8B_B64, [1500, 4000], seed=8)
    args = [blk["q"].to(DEV), blk["k_blk"].to(DEV), blk["v_blk"].to(DEV), cache.k_pools[0].to(DEV),
            cache.v_pools[0].to(DEV), cache.page_table.to(DEV), cache.ctx_len.to(DEV)]
    ws = api.workspace(torch.device(DEV), 1 << 26, slot=7)
    a = api.block_attn(*args, ws=ws).clone()
    b = api.block_attn(*args, ws=ws)
    assert torch.equal(a, b)
    assert api.device_error_word(ws) == 0


# ---- in-block causal variant: query i sees the context and block rows up to its own ----
def test_attn_causal_tiny_f32_generic_path():
    w, cache, blk = _case(W.TINY_F32, [0, 5, 31, 77], seed=5)
    _run(w, cache, blk, 1e-4, causal=True)


@pytest.mark.parametrize("ctx", [[0, 1, 63, 64, 65], [37, 1024, 1100, 2100, 3000]])
def test_attn_causal_bf16_paired_heads(ctx):
    # llama8b shape: 16 queries x 4 heads per kv head, two kv heads per item
    w, cache, blk = _case(W.LLAMA8B_B64, ctx, seed=6)
    _run(w, cache, blk, 2e-2, causal=True)


def test_attn_causal_bf16_one_kv_head_per_item_and_extra_block_rows():
    # Hkv = 3 takes one kv head per item; 3 more block rows than queries
    import dataclasses
    wl = dataclasses.replace(W.LLAMA8B_B64, Hq=12, Hkv=3)
    w, cache, blk = _case(wl, [1024, 333, 2049], seed=7, n_kv=19)
    _run(w, cache, blk, 2e-2, causal=True)


def test_attn_causal_bf16_dloop_stage_rows():
    w, cache, blk = _case(W.DLOOP_QWEN3_4B, [1024, 17, 700, 1500], seed=8, n_kv=W.DLOOP_QWEN3_4B.k + 2)
    _run(w, cache, blk, 2e-2, causal=True)


# ---- inputs that bite: needle keys in the pages (and block rows) carry a
# visible share of every output, so a skipped page, block row or a wrong split
# weight moves the output far past the tolerance ----
def _needle_full_size(seed):
    wl = W.LLAMA8B_B64
    ctx_len = synth.ctx_lengths(wl, 0)
    cache = synth.paged_cache(wl, headroom=16, seed=seed, layers=1, ctx_len=ctx_len)
    blk = synth.block_qkv(wl, 0, seed=seed)
    synth.plant_needles(wl, blk, cache, seed=seed)
    order = np.argsort(ctx_len.numpy())
    seqs = sorted({int(order[0]), int(order[1]), int(order[len(order) // 2]), int(order[-2]), int(order[-1]), 5, 40})
    return wl, cache, blk, seqs


def test_attn_full_size_needles_llama8b_b64():
    wl, cache, blk, seqs = _needle_full_size(seed=13)
    got = _run(wl, cache, blk, 2e-2, seqs=seqs, repeat=3)
    assert np.abs(got).max() > 0.5          # the needles do dominate the outputs


def test_attn_full_size_needles_causal_llama8b_b64():
    wl, cache, blk, seqs = _needle_full_size(seed=14)
    _run(wl, cache, blk, 2e-2, seqs=seqs[:4], causal=True)


@pytest.mark.parametrize("ctx", [[1024, 1025, 2048, 3000, 4097, 8192, 17, 500]])
def test_attn_needles_split_boundaries(ctx):
    # contexts near 1024-key multiples, split when the launch's mean work is small
    import dataclasses
    wl = dataclasses.replace(W.LLAMA8B_B64, B=len(ctx))
    cache = synth.paged_cache(wl, headroom=16, seed=15, layers=1, ctx_len=torch.tensor(ctx, dtype=torch.int32))
    blk = synth.block_qkv(wl, 0, seed=15)
    synth.plant_needles(wl, blk, cache, seed=15)
    _run(wl, cache, blk, 2e-2)


@pytest.mark.parametrize("B", [1, 19])
def test_attn_long_context_split_into_many_pieces(B):
    """One 8192-key context among short ones: the launch holds few tiles, so
    the partition's ranges are 8-9 tiles and each kv-head pair of the long
    context is cut into some 30 pieces. The split-merge kernel combines them
    with 8 columns per thread and eight pieces' loads at a time when fewer than
    76 (sequence, kv-head pair)s take part (B = 1), else with 16 columns and
    four pieces at a time (B = 19: 76 pairs), looping over the rest. Needles
    on the long context's pages make a lost or misplaced piece visible."""
    ctx = [8192] + [1 + 7 * i for i in range(B - 1)]
    w, cache, blk = _case(W.LLAMA8B_B64, ctx, seed=18)
    synth.plant_needles(w, blk, cache, seed=18)
    got = _run(w, cache, blk, 2e-2, seqs=sorted({0, B - 1, B // 2}), repeat=2)
    assert np.abs(got[0]).max() > 0.5


@pytest.mark.parametrize("wl,ctx", [(W.LLAMA8B_B64, [3000, 700, 5200, 1200, 64, 2500]),
                                    (W.TINY_F32, [40, 77, 20, 64])], ids=["bf16_tensor_core", "f32_generic"])
def test_active_mask_computes_only_active_sequences(wl, ctx):
    """dflash_block_attn_active (the DLoop looped draft: later stages attend
    only for the sequences whose gates continued): the active sequences' rows
    match the unmasked call (bit for bit on the fp32 path, whose blocks are
    independent; within 2e-2 on the bf16 kernel, whose static partition of the
    work then covers the active sequences only, so split merges round
    differently) and repeat bit for bit, and inactive rows are left as they
    were."""
    w, cache, blk = _case(wl, ctx, seed=17)
    args = [blk["q"].to(DEV), blk["k_blk"].to(DEV), blk["v_blk"].to(DEV), cache.k_pools[0].to(DEV),
            cache.v_pools[0].to(DEV), cache.page_table.to(DEV), cache.ctx_len.to(DEV)]
    full = api.block_attn(*args).clone()
    active = torch.tensor([1, 0, 1, 0, 1, 0][:len(ctx)], dtype=torch.uint8, device=DEV)
    out = torch.full_like(full, 7.0)
    api.block_attn(*args, out=out, active=active)
    torch.cuda.synchronize()
    on = active.bool()
    if out.dtype == torch.bfloat16:
        assert float((out[on].float() - full[on].float()).abs().max()) < 2e-2
        again = torch.full_like(full, 7.0)
        api.block_attn(*args, out=again, active=active)
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    else:
        assert torch.equal(out[on], full[on])
    assert bool((out[~on] == 7.0).all())
    # no sequence active: nothing written; all active: the unmasked call
    none = torch.full_like(full, 7.0)
    api.block_attn(*args, out=none, active=torch.zeros_like(active))
    torch.cuda.synchronize()
    assert bool((none == 7.0).all())
    every = api.block_attn(*args, active=torch.ones_like(active))
    assert torch.equal(every, full)
