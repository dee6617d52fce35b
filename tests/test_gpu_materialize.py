"""GPU parity of the context-KV materialisation against the CPU oracle.

Written rows: max-abs 2e-2 for bf16 I/O (the GPU rounds h_ctx and the K/V
outputs to bf16; the oracle keeps float64 throughout), 1e-4 for fp32.
Rows outside the committed prefix must be left bit-for-bit untouched.
"""
import dataclasses

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


def _window_pages(B, start_pos, rows, page, seed):
    """Page table that maps only the logical pages touched by [start, start+rows)
    to a small shuffled physical pool; every other entry is -1."""
    need = [(int(s) // page, (int(s) + rows - 1) // page) for s in start_pos]
    max_pages = max(hi for _, hi in need) + 1
    total = sum(hi - lo + 1 for lo, hi in need)
    perm = torch.randperm(total, generator=torch.Generator().manual_seed(seed)).to(torch.int32)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, (lo, hi) in enumerate(need):
        pt[b, lo:hi + 1] = perm[off:off + hi - lo + 1]
        off += hi - lo + 1
    return pt, total


def _run_case(wl, commit, start, seed=0, atol=2e-2, k_norm=True, rope=True, bias=True):
    B, rows = len(commit), wl.k
    w = ctx = synth.ctx_weights(wl, seed)
    hidden = synth.captured_hidden(wl, rows, seed, B=B)
    commit_t = torch.tensor(commit, dtype=torch.int32)
    start_t = torch.tensor(start, dtype=torch.int32)
    pt, num_pages = _window_pages(B, start, rows, wl.page_size, seed)
    dt = synth.io_dtype(wl)
    shape = (num_pages, wl.page_size, wl.Hkv, wl.D)
    gen = torch.Generator().manual_seed(seed + 99)
    kp = [torch.randn(shape, generator=gen).to(dt) for _ in range(wl.L)]
    vp = [torch.randn(shape, generator=gen).to(dt) for _ in range(wl.L)]
    kn = w["k_norm_w"] if k_norm else None
    theta = wl.rope_theta if rope else 0.0
    bf = w["b_f"] if bias else None
    kd = [t.to(DEV) for t in kp]
    vd = [t.to(DEV) for t in vp]
    new_len = torch.empty(B, dtype=torch.int32, device=DEV)
    api.materialize_ctx_kv(hidden.to(DEV), commit_t.to(DEV), start_t.to(DEV), w["W_f"].to(DEV),
                           None if bf is None else bf.to(DEV), w["W_kv"].to(DEV),
                           None if kn is None else kn.to(DEV), wl.rms_eps, theta, kd, vd, pt.to(DEV), new_len)
    torch.cuda.synchronize()
    assert torch.equal(new_len.cpu(), start_t + commit_t)
    rk, rv = O.materialize_ctx_kv(f64(hidden), commit, start, f64(w["W_f"]),
                                  np.zeros(wl.d) if bf is None else f64(bf), f64(w["W_kv"]),
                                  None if kn is None else f64(kn), wl.rms_eps, theta,
                                  [f64(t) for t in kp], [f64(t) for t in vp], pt.numpy(), wl.page_size)
    written = np.zeros((num_pages, wl.page_size), bool)
    for b in range(B):
        for j in range(commit[b]):
            pos = start[b] + j
            written[int(pt[b, pos // wl.page_size]), pos % wl.page_size] = True
    for layer in range(wl.L):
        gk, gv = kd[layer].cpu(), vd[layer].cpu()
        # untouched rows: bit-exact
        assert torch.equal(gk[torch.from_numpy(~written)], kp[layer][torch.from_numpy(~written)])
        assert torch.equal(gv[torch.from_numpy(~written)], vp[layer][torch.from_numpy(~written)])
        ek = np.abs(f64(gk)[written] - rk[layer][written]).max(initial=0.0)
        ev = np.abs(f64(gv)[written] - rv[layer][written]).max(initial=0.0)
        assert ek < atol and ev < atol, (layer, ek, ev)
    return written.sum()


def test_materialize_tiny_f32():
    n = _run_case(W.TINY_F32, [3], [32], atol=1e-4)
    assert n == 3


def test_materialize_tiny_f32_batch_ragged_no_norm_no_rope():
    wl = dataclasses.replace(W.TINY_F32, B=5)
    _run_case(wl, [0, 1, 4, 2, 3], [32, 0, 17, 100, 5], seed=1, atol=1e-4, k_norm=False, rope=False, bias=False)


def test_materialize_bf16_small_shape_spans_tiles():
    wl = dataclasses.replace(W.QWEN3_4B_B8, d=256, L=2, Hkv=2, weight_std=0.05)
    _run_case(wl, [16, 0, 7, 1, 16, 9], [1024, 5, 300, 999, 16, 64], seed=2)


def test_materialize_bf16_full_llama8b_shape_b64():
    wl = W.LLAMA8B_B64
    gen = torch.Generator().manual_seed(3)
    commit = torch.randint(1, wl.k + 1, (wl.B,), generator=gen).tolist()
    start = synth.ctx_lengths(wl, 0).tolist()
    n = _run_case(wl, commit, start, seed=3)
    assert n == sum(commit)


def test_materialize_bf16_qwen3_4b_prefill_rows():
    # one sequence committing a long prompt-like block in a single call
    wl = dataclasses.replace(W.QWEN3_4B_B8, k=256)
    _run_case(wl, [256, 200], [0, 4096], seed=4)


def _prefill_case(wl, B, rows, n_check, seed):
    """Every row of every sequence committed in one call (prefill-sized
    T = B * rows), then n_check seeded rows compared with the oracle. Each row's
    K/V depends only on its own hidden row and position, so the oracle runs on
    just those rows (each as a one-row sequence at its position)."""
    w = synth.ctx_weights(wl, seed)
    hidden = synth.captured_hidden(wl, rows, seed, B=B)
    wb = dataclasses.replace(wl, B=B)
    pt, num_pages, _ = synth.page_table(wb, torch.zeros(B, dtype=torch.int32), rows, seed)
    dt = synth.io_dtype(wl)
    shape = (num_pages, wl.page_size, wl.Hkv, wl.D)
    kd = [torch.zeros(shape, dtype=dt, device=DEV) for _ in range(wl.L)]
    vd = [torch.zeros(shape, dtype=dt, device=DEV) for _ in range(wl.L)]
    commit = torch.full((B,), rows, dtype=torch.int32, device=DEV)
    start = torch.zeros(B, dtype=torch.int32, device=DEV)
    new_len = torch.empty(B, dtype=torch.int32, device=DEV)
    api.materialize_ctx_kv(hidden.to(DEV), commit, start, w["W_f"].to(DEV), w["b_f"].to(DEV), w["W_kv"].to(DEV),
                           w["k_norm_w"].to(DEV), wl.rms_eps, wl.rope_theta, kd, vd, pt.to(DEV), new_len)
    torch.cuda.synchronize()
    assert torch.all(new_len.cpu() == rows)
    rng = np.random.default_rng(seed)
    pick = rng.choice(B * rows, size=n_check, replace=False)
    bs, js = pick // rows, pick % rows
    # the picked rows as one-row sequences at their positions, one private page each
    P = wl.page_size
    tab = np.full((n_check, max(js) // P + 1), -1, dtype=np.int32)
    tab[np.arange(n_check), js // P] = np.arange(n_check)
    pool0 = [np.zeros((n_check, P, wl.Hkv, wl.D)) for _ in range(wl.L)]
    rk, rv = O.materialize_ctx_kv(f64(hidden[torch.from_numpy(bs), torch.from_numpy(js)])[:, None],
                                  [1] * n_check, js.tolist(), f64(w["W_f"]), f64(w["b_f"]), f64(w["W_kv"]),
                                  f64(w["k_norm_w"]), wl.rms_eps, wl.rope_theta, pool0,
                                  [p.copy() for p in pool0], tab, P)
    slots = torch.from_numpy(pt.numpy()[bs, js // P].astype(np.int64) * P + js % P)
    worst = 0.0
    for layer in range(wl.L):
        gk = f64(kd[layer].view(-1, wl.Hkv, wl.D)[slots.to(DEV)])
        gv = f64(vd[layer].view(-1, wl.Hkv, wl.D)[slots.to(DEV)])
        ok_ = rk[layer][np.arange(n_check), js % P]
        ov = rv[layer][np.arange(n_check), js % P]
        worst = max(worst, np.abs(gk - ok_).max(), np.abs(gv - ov).max())
    assert worst < 2e-2, worst
    return worst


def test_materialize_prefill_llama8b_t2048():
    # the Llama-3.1-8B workload's prefill: one sequence, T = 2048 rows; the
    # K/V GEMM (N = 10240) hands out whole waves of 152 tiles
    _prefill_case(W.LLAMA8B_B1, B=1, rows=2048, n_check=256, seed=11)


def test_materialize_prefill_qwen3_4b_t8192():
    # the Qwen3-4B workload's prefill: 8 sequences x 1024 rows, T = 8192; both
    # GEMMs run several waves of whole tiles before the stream-K remainder
    _prefill_case(W.QWEN3_4B_B8, B=8, rows=1024, n_check=256, seed=12)
