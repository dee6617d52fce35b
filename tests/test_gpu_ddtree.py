"""GPU parity of the DDTree kernels (speculative-decoding page, section 6)
against the CPU oracle: the per-position top-K (tokens exact, log-probs within
1e-5), the best-first tree (node tokens, parents and depths exact for
sequences neither side flags as decided by a near tie; path log-probs within
1e-5) and the greedy tree walk (every output exact, given the tree)."""
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


def _tree_case(wl, B, n, K, budget, seed, temperature=1.0):
    zd = synth.draft_logits(wl, n, seed, "tree_zd", B=B)
    g = zd.to(DEV)
    tk = api.ddtree_topk(g, K, temperature)
    tr = api.ddtree_build(tk["tok"], tk["logp"], budget, V=wl.V)
    torch.cuda.synchronize()
    return zd, tk, tr


def _check_topk(zd, tk, K, temperature):
    tok, logp = O.ddtree_topk(f64(zd), K, temperature)
    np.testing.assert_array_equal(tk["tok"].cpu().numpy(), tok)
    np.testing.assert_allclose(tk["logp"].cpu().numpy(), logp, rtol=1e-5, atol=1e-5)
    return tok, logp


def _check_tree(tr, tok, logp, budget, min_live=0.0):
    """Unflagged sequences: the tree node for node. Sequences either side flags
    (a pop that a distinct path trailed by less than 1e-5, so rounding may
    order them differently): the selected path log-probabilities (unique up to
    such ties) and the validity of the GPU tree (parents first, depth =
    parent's + 1, each node's log-prob = its parent's + its token's at its
    position)."""
    ref = O.ddtree_build(tok, logp, budget)
    flags = tr["flags"].cpu().numpy()
    live = (flags == 0) & (ref["flags"] == 0)
    assert live.mean() >= min_live, (flags, ref["flags"])
    nn = tr["n_nodes"].cpu().numpy()
    np.testing.assert_array_equal(nn, ref["n_nodes"])
    got = {k: tr[k].cpu().numpy() for k in ("node_token", "node_parent", "node_depth", "node_logp")}
    for key in ("node_token", "node_parent", "node_depth"):
        np.testing.assert_array_equal(got[key][live], ref[key][live], err_msg=key)
    np.testing.assert_allclose(got["node_logp"][live], ref["node_logp"][live], rtol=1e-5, atol=1e-4)
    for b in np.nonzero(~live)[0]:
        m = int(nn[b])
        np.testing.assert_allclose(np.sort(got["node_logp"][b, :m]), np.sort(ref["node_logp"][b, :m]), atol=1e-4)
        for j in range(m):
            p, d, t = int(got["node_parent"][b, j]), int(got["node_depth"][b, j]), int(got["node_token"][b, j])
            assert p < j
            assert d == (1 if p < 0 else int(got["node_depth"][b, p]) + 1)
            r = list(tok[b, d - 1]).index(t)
            plp = 0.0 if p < 0 else float(got["node_logp"][b, p])
            assert abs(got["node_logp"][b, j] - (plp + logp[b, d - 1, r])) < 1e-4
    return live


def test_ddtree_tiny_f32():
    wl = W.TINY_F32
    zd, tk, tr = _tree_case(wl, B=3, n=3, K=4, budget=20, seed=1)
    tok, logp = _check_topk(zd, tk, 4, 1.0)
    _check_tree(tr, tok, logp, 20)


@pytest.mark.parametrize("K,budget", [(8, 512), (3, 64), (1, 16), (16, 1000)])
def test_ddtree_qwen3_4b_shape(K, budget):
    # Qwen3-4B draft shape: 15 drafted positions over a 151936-token vocabulary.
    # bf16 logits sit on a coarse grid, so distinct paths often have equal
    # log-probabilities up to rounding: those sequences are flagged on both
    # sides and only the others are compared.
    wl = W.QWEN3_4B_B8
    zd, tk, tr = _tree_case(wl, B=4, n=15, K=K, budget=budget, seed=2 + K)
    tok, logp = _check_topk(zd, tk, K, 1.0)
    _check_tree(tr, tok, logp, budget)


@pytest.mark.parametrize("K,budget", [(8, 512), (16, 2048)])
def test_ddtree_qwen3_4b_shape_f32_logits(K, budget):
    import dataclasses
    wl = dataclasses.replace(W.QWEN3_4B_B8, dtype="f32")
    zd, tk, tr = _tree_case(wl, B=4, n=15, K=K, budget=budget, seed=30 + K)
    tok, logp = _check_topk(zd, tk, K, 1.0)
    _check_tree(tr, tok, logp, budget)


def test_ddtree_topk_temperature():
    wl = W.QWEN3_4B_B8
    zd, tk, _ = _tree_case(wl, B=2, n=4, K=8, budget=8, seed=9, temperature=0.6)
    _check_topk(zd, tk, 8, 0.6)


@pytest.mark.parametrize("budget", [64, 512])
def test_ddtree_walk_matches_oracle(budget):
    # The tree both walks read is the oracle's own (oracle top-K, oracle
    # best-first build), so the walk is compared independently of the GPU build.
    wl = W.QWEN3_4B_B8
    B, n, K = 3, 15, 8
    zd = synth.draft_logits(wl, n, 20 + budget, "tree_zd", B=B)
    tok, logp = O.ddtree_topk(f64(zd), K, 1.0)
    ref_tree = O.ddtree_build(tok, logp, budget)
    node_token = torch.from_numpy(ref_tree["node_token"])
    node_parent = torch.from_numpy(ref_tree["node_parent"])
    n_nodes = torch.from_numpy(ref_tree["n_nodes"])
    zt = synth.ddtree_target_logits(wl, node_token, node_parent, n_nodes, seed=21, p_follow=0.9)
    out = api.ddtree_verify_greedy(zt.to(DEV), node_token.to(DEV), node_parent.to(DEV), n_nodes.to(DEV), n, K)
    torch.cuda.synchronize()
    ref = O.ddtree_walk_greedy(f64(zt), ref_tree["node_token"], ref_tree["node_parent"], ref_tree["n_nodes"])
    for key in ("accept_len", "commit_len", "bonus", "path", "out_tokens"):
        np.testing.assert_array_equal(out[key].cpu().numpy(), ref[key], err_msg=key)
    assert ref["accept_len"].max() >= 2     # the synthetic target follows the tree for a few levels


def test_ddtree_walk_chain_equals_greedy_verify():
    # K = 1: the tree is the DFlash draft chain, and the walk is the greedy rule
    wl = W.LLAMA8B_B64
    B, n = 8, 15
    vb = synth.verify_batch(wl, seed=5, B=B, greedy_rows=B)
    g = {k: v.to(DEV) for k, v in vb.items()}
    tk = api.ddtree_topk(g["draft_logits"], 1, 1.0)
    tr = api.ddtree_build(tk["tok"], tk["logp"], 64, V=wl.V)
    torch.cuda.synchronize()
    assert torch.equal(tr["node_token"][:, :n], g["cand"][:, 1:])
    # tree rows: 0 = after the anchor, 1 + j = after chain node j (the verify's row j + 1);
    # rows past the chain's n nodes are not read
    zt = torch.cat([g["target_logits"], g["target_logits"][:, :1].expand(B, 64 - n, -1)], 1).contiguous()
    out = api.ddtree_verify_greedy(zt, tr["node_token"], tr["node_parent"], tr["n_nodes"], n, 1)
    ver = api.verify_greedy(g["target_logits"], g["cand"], g["n_draft"])
    torch.cuda.synchronize()
    for key in ("accept_len", "bonus", "commit_len"):
        assert torch.equal(out[key], ver[key]), key
