"""Failure detection on the GPU without a fault.

The tensor-core kernels (bf16 attention, the context GEMMs of the
materialisation) bound every wait between their roles. With a wait limit set
far below what a working launch needs, a wait runs out: the kernel records a
code in the workspace's error word, drains its own copies and MMAs, frees its
tensor memory and returns, so the stream completes and the context stays
usable. After the limit is restored and the counter region zeroed, the next
call on the same workspace returns the same bits as a call that never failed.

A page-table entry outside the pools, inside a context, is an input error that
attention records in the same word (it reads page 0 instead, never out of
bounds).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_speculative_fusion_gb300 import api, synth
from block_diffusion_speculative_fusion_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SHORT_NS = 200          # far below the first copy of any launch


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_fusion_gb300 import build
    build.build()
    api.lib()
    yield
    api.set_wait_limit_ns(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _attn_case(ctx, seed, wl=W.LLAMA8B_B64):
    import dataclasses
    w = dataclasses.replace(wl, B=len(ctx))
    cache = synth.paged_cache(w, headroom=16, seed=seed, layers=1, ctx_len=torch.tensor(ctx, dtype=torch.int32))
    blk = synth.block_qkv(w, 0, seed=seed)
    args = [blk["q"].to(DEV), blk["k_blk"].to(DEV), blk["v_blk"].to(DEV), cache.k_pools[0].to(DEV),
            cache.v_pools[0].to(DEV), cache.page_table.to(DEV), cache.ctx_len.to(DEV)]
    return w, cache, blk, args


def test_attention_wait_limit_runs_out_then_recovers():
    w, cache, blk, args = _attn_case([4000, 3000, 8000, 1500, 700, 5000], seed=31)
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device=DEV)
    ref = api.block_attn(*args, ws=ws).clone()
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    api.set_wait_limit_ns(SHORT_NS)
    try:
        api.block_attn(*args, ws=ws)
        torch.cuda.synchronize()           # the kernel returned: no hang
    finally:
        api.set_wait_limit_ns(0)
    code = api.device_error_word(ws)
    assert 1 <= code <= 99, code
    # the context is usable and the workspace recovers once its counters are zeroed
    api.clear_counters(ws)
    again = api.block_attn(*args, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    b = 2
    want = O.block_attn(f64(blk["q"][b:b + 1]), f64(blk["k_blk"][b:b + 1]), f64(blk["v_blk"][b:b + 1]),
                        f64(cache.k_pools[0]), f64(cache.v_pools[0]), cache.page_table.numpy()[b:b + 1],
                        cache.ctx_len.numpy()[b:b + 1], w.page_size)
    assert np.abs(f64(again[b]) - want[0]).max() < 2e-2


def _mat_inputs(seed):
    wl = W.LLAMA8B_B64
    gen = torch.Generator().manual_seed(seed)
    commit = torch.randint(1, wl.k + 1, (wl.B,), generator=gen).to(torch.int32)
    start = synth.ctx_lengths(wl, 0)
    w = synth.ctx_weights(wl, seed)
    hidden = synth.captured_hidden(wl, wl.k, seed)
    cache = synth.paged_cache(wl, headroom=wl.k, seed=seed, layers=wl.L, ctx_len=start, device=DEV)
    d = {"hidden": hidden.to(DEV), "commit": commit.to(DEV), "start": start.to(DEV),
         "W_f": w["W_f"].to(DEV), "b_f": w["b_f"].to(DEV), "W_kv": w["W_kv"].to(DEV),
         "k_norm_w": w["k_norm_w"].to(DEV), "pt": cache.page_table.to(DEV)}
    return wl, d, cache


def _mat_call(wl, d, kp, vp, ws):
    api.materialize_ctx_kv(d["hidden"], d["commit"], d["start"], d["W_f"], d["b_f"], d["W_kv"], d["k_norm_w"],
                           wl.rms_eps, wl.rope_theta, kp, vp, d["pt"], ws=ws)


def test_materialize_wait_limit_runs_out_then_recovers():
    wl, d, cache = _mat_inputs(seed=32)
    dims = api.CtxKvDims(wl.B, wl.k, wl.m, wl.d, wl.L, wl.Hkv, wl.D, wl.page_size, cache.max_pages,
                         cache.num_pages, api.BF16)
    need = api.lib().dflash_materialize_workspace_size(ctypes.byref(dims))
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    k0 = [t.clone() for t in cache.k_pools]
    v0 = [t.clone() for t in cache.v_pools]
    kp, vp = [t.clone() for t in k0], [t.clone() for t in v0]
    _mat_call(wl, d, kp, vp, ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    ref_k, ref_v = [t.clone() for t in kp], [t.clone() for t in vp]
    kp, vp = [t.clone() for t in k0], [t.clone() for t in v0]
    api.set_wait_limit_ns(SHORT_NS)
    try:
        _mat_call(wl, d, kp, vp, ws)
        torch.cuda.synchronize()           # every launch of the call returned
    finally:
        api.set_wait_limit_ns(0)
    code = api.device_error_word(ws)
    assert 1 <= code <= 99, code
    api.clear_counters(ws)
    kp, vp = [t.clone() for t in k0], [t.clone() for t in v0]
    _mat_call(wl, d, kp, vp, ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    for layer in range(wl.L):
        assert torch.equal(kp[layer].view(torch.int16), ref_k[layer].view(torch.int16)), layer
        assert torch.equal(vp[layer].view(torch.int16), ref_v[layer].view(torch.int16)), layer


@pytest.mark.parametrize("wl", [W.LLAMA8B_B64, W.TINY_F32], ids=["bf16_tensor_core", "f32_generic"])
def test_attention_bad_page_entry_is_recorded(wl):
    ctx = [900, 300, 1200] if wl.dtype == "bf16" else [40, 77, 20]
    w, cache, blk, args = _attn_case(ctx, seed=33, wl=wl)
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device=DEV)
    ref = api.block_attn(*args, ws=ws).clone()
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    bad = args[5].clone()
    bad[1, 2] = cache.num_pages + 7        # logical page 2 of sequence 1 lies inside its context
    args_bad = args[:5] + [bad] + args[6:]
    api.block_attn(*args_bad, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == api.DEVERR_BAD_PAGE
    api.clear_counters(ws)
    again = api.block_attn(*args, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    assert torch.equal(again, ref)


# ---------------------------------------------------------------------------
# Inputs outside their documented range: every kernel clamps them before any
# use (never out of bounds) and records what it met in the error word; the
# debug library also records the inputs release builds clamp silently.
# ---------------------------------------------------------------------------
def _ws(size_fn, dims):
    need = getattr(api.lib(), size_fn)(ctypes.byref(dims))
    assert need > 0
    return torch.zeros(need, dtype=torch.uint8, device=DEV)


def _clamped_pair(n_draft, n_max):
    bad = n_draft.clone()
    bad[0] = n_max + 3
    bad[1] = -2
    return bad, bad.clamp(0, n_max)


def _same(a, b, keys):
    for k in keys:
        assert torch.equal(a[k], b[k]), k


def test_verify_n_draft_out_of_range_is_clamped_and_recorded():
    vb = {k: v.to(DEV) for k, v in synth.verify_batch(W.LLAMA8B_B1, seed=5, B=6, greedy_rows=3).items()}
    B, R, V = vb["target_logits"].shape
    n_max = R - 1
    bad, good = _clamped_pair(vb["n_draft"], n_max)
    dims = api.VerifyDims(B, n_max, V, api.BF16)
    keys = ("accept_len", "bonus", "commit_len", "out_tokens")
    # greedy
    ws = _ws("dflash_verify_greedy_workspace_size", dims)
    ref = {k: v.clone() for k, v in api.verify_greedy(vb["target_logits"], vb["cand"], good, ws=ws).items()}
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    got = api.verify_greedy(vb["target_logits"], vb["cand"], bad, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == api.DEVERR_BAD_N_DRAFT
    _same(got, ref, keys)
    # sampled
    ws = _ws("dflash_verify_sample_workspace_size", dims)
    args = (vb["target_logits"], vb["draft_logits"], vb["cand"], vb["u_acc"], vb["u_final"], 1.0)
    ref = {k: v.clone() for k, v in api.verify_sample(*args, n_draft=good, ws=ws).items()}
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    got = api.verify_sample(*args, n_draft=bad, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == api.DEVERR_BAD_N_DRAFT
    _same(got, ref, keys + ("flags",))
    # draft-side choice over the MASK rows
    ws = _ws("dflash_draft_select_workspace_size", dims)
    anchor = vb["cand"][:, 0].contiguous()
    ref = {k: v.clone() for k, v in api.draft_select(vb["draft_logits"], anchor, 0.0, n_draft=good, ws=ws).items()}
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == 0
    got = api.draft_select(vb["draft_logits"], anchor, 0.0, n_draft=bad, ws=ws)
    torch.cuda.synchronize()
    assert api.device_error_word(ws) == api.DEVERR_BAD_N_DRAFT
    _same(got, ref, ("cand",))


@pytest.fixture(scope="module")
def debug_library():
    from block_diffusion_speculative_fusion_gb300 import build
    path = build.build(debug=True)
    yield path
    api.select_library(debug=False)


@pytest.mark.parametrize("debug", [False, True], ids=["release", "debug"])
def test_attention_context_past_max_ctx(debug_library, debug):
    """ctx_len above max_ctx is clamped to it; only the debug library records it."""
    api.select_library(debug=debug)
    try:
        w, cache, blk, args = _attn_case([900, 2500, 300], seed=41)
        max_ctx = cache.max_pages * w.page_size
        b = int(torch.argmax(cache.ctx_len))          # every page of its table row is assigned
        ws = torch.zeros(1 << 26, dtype=torch.uint8, device=DEV)
        ok_ctx = args[6].clone()
        ok_ctx[b] = max_ctx
        ref = api.block_attn(*args[:6], ok_ctx, max_ctx=max_ctx, ws=ws).clone()
        torch.cuda.synchronize()
        assert api.device_error_word(ws) == 0
        long_ctx = ok_ctx.clone()
        long_ctx[b] = max_ctx + 40
        got = api.block_attn(*args[:6], long_ctx, max_ctx=max_ctx, ws=ws)
        torch.cuda.synchronize()
        assert api.device_error_word(ws) == (api.DEVERR_BAD_CTX_LEN if debug else 0)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    finally:
        api.select_library(debug=False)


@pytest.mark.parametrize("debug", [False, True], ids=["release", "debug"])
def test_materialize_commit_len_and_positions_out_of_range(debug_library, debug):
    """A commit_len above rows_max is clamped and a row without a pool slot is
    skipped; only the debug library records them."""
    api.select_library(debug=debug)
    try:
        wl, d, cache = _mat_inputs(seed=42)
        dims = api.CtxKvDims(wl.B, wl.k, wl.m, wl.d, wl.L, wl.Hkv, wl.D, wl.page_size, cache.max_pages,
                             cache.num_pages, api.BF16)
        ws = torch.zeros(api.lib().dflash_materialize_workspace_size(ctypes.byref(dims)), dtype=torch.uint8,
                         device=DEV)
        k0 = [t.clone() for t in cache.k_pools]
        v0 = [t.clone() for t in cache.v_pools]
        # commit_len past rows_max: the same rows as commit_len = rows_max
        kp, vp = [t.clone() for t in k0], [t.clone() for t in v0]
        d["commit"][3] = wl.k
        _mat_call(wl, d, kp, vp, ws)
        torch.cuda.synchronize()
        assert api.device_error_word(ws) == 0
        ref_k = [t.clone() for t in kp]
        kq, vq = [t.clone() for t in k0], [t.clone() for t in v0]
        d["commit"][3] = wl.k + 5
        _mat_call(wl, d, kq, vq, ws)
        torch.cuda.synchronize()
        assert api.device_error_word(ws) == (api.DEVERR_BAD_COMMIT_LEN if debug else 0)
        for layer in range(wl.L):
            assert torch.equal(kq[layer].view(torch.int16), ref_k[layer].view(torch.int16)), layer
        d["commit"][3] = wl.k
        # a negative start position: its rows have no slot and are not written
        ws.zero_()
        kr, vr = [t.clone() for t in k0], [t.clone() for t in v0]
        d["start"][5] = -3
        _mat_call(wl, d, kr, vr, ws)
        torch.cuda.synchronize()
        assert api.device_error_word(ws) == (api.DEVERR_BAD_POSITION if debug else 0)
    finally:
        api.select_library(debug=False)
