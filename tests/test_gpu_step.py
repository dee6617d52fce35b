"""Parity of the timed step itself against the CPU oracle.

The throughput workload (Llama-3.1-8B draft shape, B = 64, block 16, contexts
U[512, 8192] in 16-token pages, 32 greedy + 32 sampled sequences) runs as the
benchmark runs it: several consecutive steps captured in one CUDA graph, the
sampled verify on a forked stream of higher priority beside the greedy verify
on its own workspace. A decode round is attention in every draft layer, then
the accept rule, then the materialisation of commit_len = accept_len + 1 rows
(SGLang page, sections 3 and 4.1), and each round's committed rows are the
next round's context. Copies captured after every step keep that step's
outputs; the checks, per step:

  * accept_len, bonus, commit_len, out_tokens of all 64 sequences bit-exact
    against the oracle's greedy and sampled rules (oracle-flagged sequences
    reported, not compared);
  * the new context lengths = the old ones + commit_len;
  * draft layer 0's attention output of four sequences (shortest, median,
    longest -- split across CTAs -- and one more) at 2e-2, over the context
    the step saw, including the rows earlier steps materialised;
  * the rows the step materialised, in draft layers 0 and 4, for eight seeded
    sequences, at 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_speculative_fusion_gb300 import api
from block_diffusion_speculative_fusion_gb300 import workloads as W
from block_diffusion_speculative_fusion_gb300.step import DflashStep

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N_STEPS = 3
MAT_LAYERS = (0, 4)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_fusion_gb300 import build
    build.build()
    api.lib()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def npy(t):
    return t.detach().cpu().numpy()


def _context_rows(pool, page_table, b, C, page):
    """Rows 0..C-1 of sequence b from a device pool: [C, Hkv, D] float64."""
    pos = torch.arange(C, device=pool.device)
    slot = page_table[b, pos // page].long() * page + pos % page
    return f64(pool.view(-1, pool.shape[2], pool.shape[3]).index_select(0, slot))


def _rows_at(pool, page_table, b, positions, page):
    pos = torch.tensor(positions, device=pool.device, dtype=torch.long)
    slot = page_table[b, pos // page].long() * page + pos % page
    return f64(pool.view(-1, pool.shape[2], pool.shape[3]).index_select(0, slot))


@pytest.mark.parametrize("stationary", [False, True], ids=["advancing", "stationary"])
def test_timed_step_graph_matches_oracle(stationary):
    wl = W.LLAMA8B_B64
    st = DflashStep(wl, seed=0, device=DEV, headroom_steps=N_STEPS + 1, stationary=stationary)
    st.step()                      # eager: every workspace exists before capture
    torch.cuda.synchronize()
    st.reset()
    B, page = wl.B, wl.page_size
    order = np.argsort(st.ctx0.numpy())
    attn_seqs = sorted({int(order[0]), int(order[B // 2]), int(order[-1]), 37})
    sel = torch.tensor(attn_seqs, device=DEV)
    outs = [{k: torch.empty_like(v) for k, v in st.out.items()} for _ in range(N_STEPS)]
    attn = [torch.empty((len(attn_seqs),) + tuple(st.attn_out[0].shape[1:]), dtype=st.attn_out[0].dtype,
                        device=DEV) for _ in range(N_STEPS)]
    ctx = [st.ctx0.to(DEV).clone()] + [torch.empty_like(st.ctx[0]) for _ in range(N_STEPS)]

    def after(i):
        for k, v in st.out.items():
            outs[i][k].copy_(v)
        attn[i].copy_(st.attn_out[0].index_select(0, sel))
        ctx[i + 1].copy_(st.ctx[1] if stationary else st.ctx_len())

    graph = st.capture(N_STEPS, after_step=after)
    graph.replay()
    torch.cuda.synchronize()
    assert all(w == 0 for w in st.error_words()), st.error_words()

    # ---- the accept rules (the step's verify inputs are the same every round) ----
    h = st.host
    ng = wl.n_greedy
    ref_g = O.verify_greedy(f64(h["target_logits"][:ng]), npy(h["cand"][:ng]), npy(h["n_draft"][:ng]))
    ref_s = O.verify_sample(f64(h["target_logits"][ng:]), f64(h["draft_logits"]), npy(h["cand"][ng:]),
                            npy(h["n_draft"][ng:]), npy(h["u_acc"][ng:]), npy(h["u_final"][ng:]), wl.temperature)
    ok_s = ref_s["flags"] == 0
    assert ok_s.mean() >= 0.5
    ctx_h = [npy(c).astype(np.int64) for c in ctx]
    for i in range(N_STEPS):
        o = {k: npy(v) for k, v in outs[i].items()}
        for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
            np.testing.assert_array_equal(o[key][:ng], ref_g[key], err_msg=f"greedy {key} step {i}")
            np.testing.assert_array_equal(o[key][ng:][ok_s], ref_s[key][ok_s], err_msg=f"sampled {key} step {i}")
        start = ctx_h[0] if stationary else ctx_h[i]
        np.testing.assert_array_equal(ctx_h[i + 1], start + o["commit_len"], err_msg=f"context lengths step {i}")
    commit = npy(outs[0]["commit_len"]).astype(np.int64)
    assert commit.mean() > 1.5        # drafts are accepted: the rounds really advance

    # ---- attention of draft layer 0, each step over the context it saw ----
    pt = st.page_table
    for i in range(N_STEPS):
        C_i = ctx_h[0] if stationary else ctx_h[i]
        got = f64(attn[i])
        for j, b in enumerate(attn_seqs):
            C = int(C_i[b])
            kc = _context_rows(st.k_pools[0], pt, b, C, page)
            vc = _context_rows(st.v_pools[0], pt, b, C, page)
            n_pg = (C + page - 1) // page
            kp = np.zeros((n_pg * page,) + kc.shape[1:])
            vp = np.zeros_like(kp)
            kp[:C], vp[:C] = kc, vc
            ref = O.block_attn(f64(h["q0"][b:b + 1]), f64(h["k_blk0"][b:b + 1]), f64(h["v_blk0"][b:b + 1]),
                               kp.reshape(n_pg, page, *kc.shape[1:]), vp.reshape(n_pg, page, *kc.shape[1:]),
                               np.arange(n_pg, dtype=np.int32)[None], np.array([C]), page)
            err = np.abs(got[j] - ref[0]).max()
            assert err < 2e-2, (i, b, C, err)

    # ---- materialised rows of eight seeded sequences, layers 0 and 4 ----
    rng = np.random.default_rng(7)
    mat_seqs = sorted(rng.choice(B, size=8, replace=False).tolist())
    steps_checked = [N_STEPS - 1] if stationary else list(range(N_STEPS))
    hid, starts, commits, owners = [], [], [], []
    for i in steps_checked:
        s_i = ctx_h[0] if stationary else ctx_h[i]
        for b in mat_seqs:
            hid.append(f64(h["hidden"][b]))
            starts.append(int(s_i[b]))
            commits.append(int(commit[b]))
            owners.append(b)
    nb = len(owners)
    rows_max = h["hidden"].shape[1]
    # a private page table over a small pool for the oracle: only the written positions
    need = [((s // page), (s + c - 1) // page) for s, c in zip(starts, commits)]
    max_pg = max(hi for _, hi in need) + 1
    tab = np.full((nb, max_pg), -1, dtype=np.int32)
    npg = 0
    for r, (lo, hi) in enumerate(need):
        tab[r, lo:hi + 1] = np.arange(npg, npg + hi - lo + 1)
        npg += hi - lo + 1
    pool0 = [np.zeros((npg, page, wl.Hkv, wl.D)) for _ in range(wl.L)]
    rk, rv = O.materialize_ctx_kv(np.stack(hid), commits, starts, f64(st.W_f), f64(st.b_f), f64(st.W_kv),
                                  f64(st.k_norm_w), wl.rms_eps, wl.rope_theta, pool0, [p.copy() for p in pool0],
                                  tab, page)
    assert rows_max >= max(commits)
    for r in range(nb):
        b, s, c = owners[r], starts[r], commits[r]
        pos = list(range(s, s + c))
        for layer in MAT_LAYERS:
            gk = _rows_at(st.k_pools[layer], pt, b, pos, page)
            gv = _rows_at(st.v_pools[layer], pt, b, pos, page)
            ok_ = np.stack([rk[layer][tab[r, p // page], p % page] for p in pos])
            ov = np.stack([rv[layer][tab[r, p // page], p % page] for p in pos])
            assert np.abs(gk - ok_).max() < 2e-2 and np.abs(gv - ov).max() < 2e-2, (r, b, layer)
