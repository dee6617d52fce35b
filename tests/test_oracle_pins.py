"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the worked
example printed on the speculative-decoding page, closed forms, identities,
special cases that reduce to a library routine, and hand-built cases whose
answers are written out here from the pages' rules.
"""
import json
import math
import os

import numpy as np
import scipy.special
import scipy.stats
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _worked():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        return json.load(f)


def _example_inputs(u_acc, u_final):
    """The worked example as a one-draft verify: V = 5, cand = [anchor, cat]."""
    ex = _worked()
    lp = np.log(np.array(ex["p"], dtype=np.float32)).astype(np.float32)
    lq = np.log(np.array(ex["q"], dtype=np.float32)).astype(np.float32)
    B = len(u_acc)
    zt = np.zeros((B, 2, 5), dtype=np.float32)
    zt[:, 0] = lp
    zt[:, 1] = lp
    zd = np.zeros((B, 1, 5), dtype=np.float32)
    zd[:, 0] = lq
    cand = np.zeros((B, 2), dtype=np.int64)
    cand[:, 0] = 3            # anchor: any token
    cand[:, 1] = ex["tokens"].index(ex["draft_token"])
    n = np.ones(B, dtype=np.int32)
    return zt, zd, cand, n, np.array(u_acc, np.float32).reshape(B, 1), np.array(u_final, np.float32)


# ---------------------------------------------------------------------------
# sampled rule: worked example (speculative-decoding page, section 3)
# ---------------------------------------------------------------------------
def test_worked_example_ratio_beta_residual():
    ex = _worked()
    zt, zd, cand, n, ua, uf = _example_inputs([0.99], [0.3])
    r = O.verify_sample(zt, zd, cand, n, ua, uf)
    d = r["debug"][0]
    assert abs(d["p_x"][0] - 0.50) < 1e-6 and abs(d["q_x"][0] - 0.70) < 1e-6
    assert abs(d["p_x"][0] / d["q_x"][0] - ex["accept_ratio"]) < 1e-6
    assert r["accept_len"][0] == 0                     # 0.99 > 0.714: rejected
    assert abs(d["Z"] - ex["one_minus_beta"]) < 1e-6
    assert abs(d["one_minus_beta"] - ex["one_minus_beta"]) < 1e-6
    assert abs((1 - d["one_minus_beta"]) - ex["beta"]) < 1e-6
    np.testing.assert_allclose(d["final_dist"], ex["residual"], atol=1e-6)


@pytest.mark.parametrize("u,accepted,flagged", [(0.70, True, False), (0.72, False, False),
                                                (0.7142857, None, True)])
def test_worked_example_accept_decision(u, accepted, flagged):
    zt, zd, cand, n, ua, uf = _example_inputs([u], [0.3])
    r = O.verify_sample(zt, zd, cand, n, ua, uf)
    assert bool(r["flags"][0] & O.FLAG_ACCEPT_BOUNDARY) == flagged
    if accepted is not None:
        assert (r["accept_len"][0] == 1) == accepted
    if accepted:
        assert r["out_tokens"][0, 0] == 0                # cat kept


@pytest.mark.parametrize("uf,token,flagged", [(0.3, "dog", False), (0.7, "sat", False),
                                              (0.5, None, True)])
def test_worked_example_residual_draw(uf, token, flagged):
    ex = _worked()
    zt, zd, cand, n, ua, ufa = _example_inputs([0.9], [uf])
    r = O.verify_sample(zt, zd, cand, n, ua, ufa)
    assert r["accept_len"][0] == 0 and r["commit_len"][0] == 1
    assert bool(r["flags"][0] & O.FLAG_CDF_BOUNDARY) == flagged
    if token is not None:
        assert r["bonus"][0] == ex["tokens"].index(token)
        assert r["out_tokens"][0, 0] == r["bonus"][0]


def test_worked_example_not_drop_and_renormalise():
    """Dropping 'cat' and renormalising p would give 'on' 0.20; the residual
    gives it 0 (speculative-decoding page, section 3)."""
    ex = _worked()
    p = np.array(ex["p"])
    wrong = p.copy()
    wrong[0] = 0
    wrong /= wrong.sum()
    assert abs(wrong[3] - ex["wrong_renormalised_on"]) < 1e-12
    zt, zd, cand, n, ua, uf = _example_inputs([0.9], [0.3])
    d = O.verify_sample(zt, zd, cand, n, ua, uf)["debug"][0]
    assert d["final_dist"][3] < 1e-6     # 0 up to the fp32 rounding of ln p, ln q
    # and no draw ever lands on 'on' or 'cat' or 'mat' after the rejection
    for u in np.linspace(0.0, 0.999, 101):
        zt, zd, cand, n, ua, uf = _example_inputs([0.9], [u])
        y = O.verify_sample(zt, zd, cand, n, ua, uf)["bonus"][0]
        assert y in (1, 2)


# ---------------------------------------------------------------------------
# sampled rule: min(p,q) + max(0,p-q) = p, by Monte Carlo
# ---------------------------------------------------------------------------
def _chi2_pvalue(counts, probs):
    n = counts.sum()
    keep = probs > 0
    assert counts[~keep].sum() == 0
    obs = counts[keep]
    expected = probs[keep] / probs[keep].sum() * obs.sum()
    expected *= obs.sum() / expected.sum()
    stat = ((obs - expected) ** 2 / expected).sum()
    from scipy.stats import chi2
    return chi2.sf(stat, len(obs) - 1)


@pytest.mark.parametrize("V", [2, 5, 17])
def test_identity_monte_carlo(V):
    rng = np.random.default_rng(100 + V)
    trials = 60000
    lp = rng.normal(0, 1.5, V).astype(np.float32)
    lq = rng.normal(0, 1.5, V).astype(np.float32)
    p = np.exp(lp - lp.max()); p /= p.sum()
    q = np.exp(lq - lq.max()); q /= q.sum()
    x = rng.choice(V, size=trials, p=q)
    zt = np.broadcast_to(lp, (trials, 2, V)).copy()
    zd = np.broadcast_to(lq, (trials, 1, V)).copy()
    cand = np.stack([np.zeros(trials, np.int64), x], axis=1)
    ua = rng.random((trials, 1), dtype=np.float32)
    uf = rng.random(trials, dtype=np.float32)
    r = O.verify_sample(zt, zd, cand, np.ones(trials, np.int32), ua, uf)
    first = r["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=V).astype(np.float64)
    assert _chi2_pvalue(counts, p) > 1e-3
    sd = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(counts / trials - p) < 5 * sd + 1e-12)
    # acceptance rate equals beta = sum min(p, q)
    beta = np.minimum(p, q).sum()
    acc_rate = r["accept_len"].mean()
    assert abs(acc_rate - beta) < 5 * math.sqrt(beta * (1 - beta) / trials) + 1e-9


def test_identical_distributions_never_reject():
    """q == p gives beta = 1: every draft is accepted (section 4)."""
    rng = np.random.default_rng(7)
    B, n, V = 64, 6, 11
    z = rng.normal(0, 2, (B, n + 1, V)).astype(np.float32)
    cand = rng.integers(0, V, (B, n + 1))
    r = O.verify_sample(z, z[:, :n], cand, np.full(B, n), rng.random((B, n), dtype=np.float32),
                        rng.random(B, dtype=np.float32))
    assert np.all(r["accept_len"] == n)


def test_disjoint_supports_always_reject_and_draw_p():
    rng = np.random.default_rng(8)
    V, trials = 6, 20000
    lp = np.array([-1e4, -1e4, -1e4, 0.3, -0.2, 0.1], np.float32)
    lq = np.array([0.0, 0.5, -0.5, -1e4, -1e4, -1e4], np.float32)
    p = np.exp(lp - lp.max()); p /= p.sum()
    q = np.exp(lq - lq.max()); q /= q.sum()
    x = rng.choice(V, size=trials, p=q)
    zt = np.broadcast_to(lp, (trials, 2, V)).copy()
    zd = np.broadcast_to(lq, (trials, 1, V)).copy()
    cand = np.stack([np.zeros(trials, np.int64), x], axis=1)
    r = O.verify_sample(zt, zd, cand, np.ones(trials, np.int32),
                        rng.random((trials, 1), dtype=np.float32), rng.random(trials, dtype=np.float32))
    assert np.all(r["accept_len"] == 0)
    counts = np.bincount(r["bonus"], minlength=V).astype(np.float64)
    assert _chi2_pvalue(counts, p) > 1e-3


def test_one_hot_sampled_equals_greedy():
    """One-hot p and q (logit gaps of 1e4) turn the sampled rule into the greedy one."""
    rng = np.random.default_rng(9)
    B, n, V = 200, 7, 13
    tp = rng.integers(0, V, (B, n + 1))
    cand = rng.integers(0, V, (B, n + 1))
    # make about half of the drafts match
    agree = rng.random((B, n)) < 0.7
    cand[:, 1:] = np.where(agree, tp[:, :n], cand[:, 1:])
    zt = np.full((B, n + 1, V), -1e4, np.float32)
    np.put_along_axis(zt, tp[..., None], 0.0, axis=2)
    zd = np.full((B, n, V), -1e4, np.float32)
    np.put_along_axis(zd, cand[:, 1:, None], 0.0, axis=2)
    nd = rng.integers(0, n + 1, B).astype(np.int32)
    s = O.verify_sample(zt, zd, cand, nd, rng.random((B, n), dtype=np.float32),
                        rng.random(B, dtype=np.float32))
    g = O.verify_greedy(zt, cand, nd)
    for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
        np.testing.assert_array_equal(s[key], g[key])


def test_zero_q_candidate_is_flagged_invalid():
    zt = np.zeros((1, 2, 4), np.float32)
    zd = np.array([[[0.0, 0.0, 0.0, -1e4]]], np.float32)
    cand = np.array([[0, 3]])
    r = O.verify_sample(zt, zd, cand, np.array([1]), np.array([[0.5]], np.float32),
                        np.array([0.2], np.float32))
    assert r["flags"][0] & O.FLAG_INVALID
    assert r["accept_len"][0] == 1        # p/q = inf: accepted


def test_full_accept_draws_bonus_from_last_target_row():
    # p rows 0,1 put all mass on token 2; row 2 (bonus row) is uniform over 4
    zt = np.full((1, 3, 4), -1e4, np.float32)
    zt[0, 0, 2] = zt[0, 1, 2] = 0
    zt[0, 2, :] = 0
    zd = zt[:, :2].copy()
    cand = np.array([[1, 2, 2]])
    for u, y in [(0.1, 0), (0.3, 1), (0.6, 2), (0.9, 3)]:
        r = O.verify_sample(zt, zd, cand, np.array([2]), np.array([[0.5, 0.5]], np.float32),
                            np.array([u], np.float32))
        assert r["accept_len"][0] == 2 and r["bonus"][0] == y
        assert list(r["out_tokens"][0]) == [2, 2, y]


# ---------------------------------------------------------------------------
# greedy rule (SGLang page, section 3): hand-built cases
# ---------------------------------------------------------------------------
def _onehot_logits(pred, V=8):
    pred = np.asarray(pred)
    z = np.zeros(pred.shape + (V,), np.float32)
    np.put_along_axis(z, pred[..., None], 5.0, axis=-1)
    return z


def test_greedy_all_match():
    tp = [[3, 5, 1, 7]]
    cand = [[0, 3, 5, 1]]
    r = O.verify_greedy(_onehot_logits(tp), cand)
    assert r["accept_len"][0] == 3 and r["bonus"][0] == 7 and r["commit_len"][0] == 4
    assert list(r["out_tokens"][0]) == [3, 5, 1, 7]
    assert list(r["target_pred"][0]) == [3, 5, 1, 7]


def test_greedy_first_draft_wrong_commits_one():
    r = O.verify_greedy(_onehot_logits([[3, 5, 1, 7]]), [[0, 4, 5, 1]])
    assert r["accept_len"][0] == 0 and r["bonus"][0] == 3 and r["commit_len"][0] == 1
    assert list(r["out_tokens"][0]) == [3, -1, -1, -1]


def test_greedy_cumprod_stops_at_first_mismatch():
    # drafts 1 ok, 2 wrong, 3 ok: accept only the first
    r = O.verify_greedy(_onehot_logits([[3, 5, 1, 7]]), [[0, 3, 6, 1]])
    assert r["accept_len"][0] == 1 and r["bonus"][0] == 5 and r["commit_len"][0] == 2
    assert list(r["out_tokens"][0]) == [3, 5, -1, -1]


def test_greedy_ties_take_lowest_index():
    z = np.zeros((1, 2, 6), np.float32)
    z[0, 0, [2, 4]] = 1.0          # tie between 2 and 4
    z[0, 1, [5, 1]] = 2.0          # tie between 1 and 5
    r = O.verify_greedy(z, [[0, 2]])
    assert list(r["target_pred"][0]) == [2, 1]
    assert r["accept_len"][0] == 1 and r["bonus"][0] == 1
    r = O.verify_greedy(z, [[0, 4]])
    assert r["accept_len"][0] == 0 and r["bonus"][0] == 2


def test_greedy_ragged_draft_counts():
    tp = [[3, 5, 1, 7], [2, 2, 2, 2], [1, 1, 1, 1]]
    cand = [[0, 3, 5, 1], [0, 2, 2, 2], [0, 1, 9, 9]]
    r = O.verify_greedy(_onehot_logits(tp), cand, n_draft=[1, 0, 3])
    assert list(r["accept_len"]) == [1, 0, 1]
    assert list(r["bonus"]) == [5, 2, 1]
    assert list(r["commit_len"]) == [2, 1, 2]
    assert list(r["target_pred"][1]) == [2, -1, -1, -1]


# ---------------------------------------------------------------------------
# DLoop gate (DLoop page, mechanism 1)
# ---------------------------------------------------------------------------
def test_gate_uniform_logits_closed_form():
    B, k, V = 3, 7, 1000
    z = np.zeros((B, k, V), np.float32)
    tok = np.zeros((B, k), np.int64)
    r = O.gate(z, tok, None, 1.0, -0.5)
    np.testing.assert_allclose(r["c"], -k * math.log(V), rtol=1e-12)
    assert np.all(r["cont"] == 0)
    np.testing.assert_allclose(r["row_lse"], math.log(V), rtol=1e-12)


def test_gate_one_hot_is_zero_and_continues_on_tie():
    z = np.full((1, 4, 50), -1e4, np.float32)
    tok = np.array([[3, 9, 0, 49]])
    np.put_along_axis(z, tok[..., None], 0.0, axis=2)
    r = O.gate(z, tok, None, 1.0, 0.0)     # c == g exactly: >= continues
    assert r["c"][0] == 0.0 and r["cont"][0] == 1


def test_gate_explicit_probabilities_and_temperature():
    probs = np.array([0.5, 0.3, 0.2])
    z = np.log(probs)[None, None, :].repeat(2, axis=1)
    tok = np.array([[0, 1]])
    r = O.gate(z, tok, None, 1.0, -0.5)
    assert abs(r["c"][0] - (math.log(0.5) + math.log(0.3))) < 1e-12
    assert r["cont"][0] == 0
    # temperature 2: softmax(z/2) is proportional to sqrt(probs)
    r2 = O.gate(z, tok, None, 2.0, -5.0)
    s = np.sqrt(probs) / np.sqrt(probs).sum()
    assert abs(r2["c"][0] - (math.log(s[0]) + math.log(s[1]))) < 1e-12
    assert r2["cont"][0] == 1


def test_gate_inactive_sequences():
    z = np.zeros((2, 3, 10), np.float32)
    r = O.gate(z, np.zeros((2, 3), np.int64), np.array([1, 0]), 1.0, -100.0)
    assert r["cont"][0] == 1 and r["cont"][1] == 0 and r["c"][1] == 0.0


def test_dloop_stage_count():
    conts = np.array([[1, 0, 1, 1],
                      [1, 1, 0, 1],
                      [0, 1, 1, 1],
                      [1, 1, 1, 1]])
    assert list(O.dloop_stage_count(conts)) == [3, 1, 2, 4]


# ---------------------------------------------------------------------------
# block attention (DFlash page, KV injection attention equation)
# ---------------------------------------------------------------------------
def _attn_case(rng, B=2, n_q=3, Hq=4, Hkv=2, D=8, ctx=(5, 9), page=4, n_kv=None):
    n_kv = n_q if n_kv is None else n_kv
    max_pages = max((c + page - 1) // page for c in ctx) + 1
    num_pages = B * max_pages
    perm = rng.permutation(num_pages).reshape(B, max_pages)
    return dict(
        q=rng.normal(size=(B, n_q, Hq, D)), k_blk=rng.normal(size=(B, n_kv, Hkv, D)),
        v_blk=rng.normal(size=(B, n_kv, Hkv, D)),
        k_pool=rng.normal(size=(num_pages, page, Hkv, D)),
        v_pool=rng.normal(size=(num_pages, page, Hkv, D)),
        page_table=perm, ctx_len=np.array(ctx), page_size=page)


def _sdpa(q, k, v, scale):
    """torch's fp64 scaled-dot-product attention, no mask: q [H, n, D], k/v [H, m, D]."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale).numpy()


def test_attn_no_ctx_mha_matches_library():
    rng = np.random.default_rng(1)
    c = _attn_case(rng, B=1, Hq=3, Hkv=3, ctx=(0,))
    out = O.block_attn(**c)
    q = c["q"][0].transpose(1, 0, 2)
    k = c["k_blk"][0].transpose(1, 0, 2)
    v = c["v_blk"][0].transpose(1, 0, 2)
    ref = _sdpa(q, k, v, 1 / math.sqrt(8)).transpose(1, 0, 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)


def test_attn_gqa_matches_library_with_repeated_kv():
    rng = np.random.default_rng(2)
    c = _attn_case(rng, B=2, Hq=6, Hkv=2, D=8, ctx=(7, 3), page=2, n_kv=4)
    out = O.block_attn(**c)
    G = 3
    for b in range(2):
        C = c["ctx_len"][b]
        pos = np.arange(C)
        pages = c["page_table"][b][pos // 2]
        Kc = c["k_pool"][pages, pos % 2]
        Vc = c["v_pool"][pages, pos % 2]
        K = np.concatenate([Kc, c["k_blk"][b]])       # [keys, Hkv, D]
        V = np.concatenate([Vc, c["v_blk"][b]])
        Krep = np.repeat(K, G, axis=1).transpose(1, 0, 2)
        Vrep = np.repeat(V, G, axis=1).transpose(1, 0, 2)
        ref = _sdpa(c["q"][b].transpose(1, 0, 2), Krep, Vrep, 1 / math.sqrt(8)).transpose(1, 0, 2)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_attn_invariant_to_ctx_order_and_page_size():
    rng = np.random.default_rng(3)
    c = _attn_case(rng, B=1, ctx=(11,), page=4)
    base = O.block_attn(**c)
    # same rows, laid out one row per page in reversed physical order
    Kc = O.gather_ctx(c["k_pool"], c["page_table"][0], 11, 4)
    Vc = O.gather_ctx(c["v_pool"], c["page_table"][0], 11, 4)
    perm = rng.permutation(11)
    c2 = dict(c)
    c2["k_pool"] = Kc[perm][:, None]
    c2["v_pool"] = Vc[perm][:, None]
    c2["page_size"] = 1
    c2["page_table"] = np.arange(11)[None, :]
    out = O.block_attn(**c2)
    np.testing.assert_allclose(out, base, rtol=1e-12, atol=1e-12)


def test_attn_causal_no_ctx_matches_library_causal():
    # [DFlash] 块扩散的双向注意力问题 (JetSpec): position i sees positions 0 .. i.
    # With no context and n_q = n_kv this is textbook causal attention.
    rng = np.random.default_rng(11)
    c = _attn_case(rng, B=1, n_q=5, Hq=3, Hkv=3, ctx=(0,))
    out = O.block_attn(**c, causal=True)
    q = torch.from_numpy(c["q"][0].transpose(1, 0, 2))
    k = torch.from_numpy(c["k_blk"][0].transpose(1, 0, 2))
    v = torch.from_numpy(c["v_blk"][0].transpose(1, 0, 2))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=1 / math.sqrt(8)).numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)


def test_attn_causal_row_is_unmasked_attention_over_its_prefix():
    # query i sits at block row i + n_kv - n_q and keeps all context rows
    rng = np.random.default_rng(12)
    n_q, n_kv = 4, 6
    c = _attn_case(rng, B=2, n_q=n_q, Hq=4, Hkv=2, ctx=(5, 9), page=4, n_kv=n_kv)
    out = O.block_attn(**c, causal=True)
    for i in range(n_q):
        last = i + n_kv - n_q
        ci = dict(c)
        ci["q"] = c["q"][:, i:i + 1]
        ci["k_blk"] = c["k_blk"][:, :last + 1]
        ci["v_blk"] = c["v_blk"][:, :last + 1]
        ref = O.block_attn(**ci)
        np.testing.assert_allclose(out[:, i:i + 1], ref, rtol=1e-12, atol=1e-12)
    # later block rows do not reach earlier queries
    c2 = dict(c)
    c2["k_blk"] = c["k_blk"].copy()
    c2["v_blk"] = c["v_blk"].copy()
    c2["k_blk"][:, n_kv - 1] += 3.0
    c2["v_blk"][:, n_kv - 1] -= 2.0
    out2 = O.block_attn(**c2, causal=True)
    np.testing.assert_array_equal(out2[:, :n_q - 1], out[:, :n_q - 1])
    assert np.abs(out2[:, n_q - 1] - out[:, n_q - 1]).max() > 1e-3


def test_attn_causal_last_row_and_single_query_are_unmasked():
    rng = np.random.default_rng(13)
    c = _attn_case(rng, B=2, n_q=3, Hq=4, Hkv=2, ctx=(7, 2), page=2, n_kv=5)
    full = O.block_attn(**c)
    causal = O.block_attn(**c, causal=True)
    np.testing.assert_allclose(causal[:, -1], full[:, -1], rtol=1e-12, atol=1e-12)
    c1 = _attn_case(rng, B=1, n_q=1, ctx=(4,), n_kv=1)
    np.testing.assert_allclose(O.block_attn(**c1, causal=True), O.block_attn(**c1), rtol=1e-12, atol=1e-12)


def test_attn_identical_keys_average_values():
    rng = np.random.default_rng(4)
    c = _attn_case(rng, B=1, ctx=(6,), page=3)
    key = rng.normal(size=8)
    c["k_pool"][:] = key
    c["k_blk"][:] = key
    out = O.block_attn(**c)
    Vc = O.gather_ctx(c["v_pool"], c["page_table"][0], 6, 3)
    V = np.concatenate([Vc, c["v_blk"][0]])
    for h in range(4):
        np.testing.assert_allclose(out[0, :, h], np.broadcast_to(V[:, h // 2].mean(0), (3, 8)),
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# materialisation (DFlash KV injection; SGLang section 4.1)
# ---------------------------------------------------------------------------
def test_rope_against_complex_rotation():
    rng = np.random.default_rng(5)
    D, theta = 16, 10000.0
    x = rng.normal(size=(3, D))
    for pos in (0, 1, 7, 1234):
        got = O.rope_rotate_half(x, pos, theta)
        zc = (x[:, :D // 2] + 1j * x[:, D // 2:]) * np.exp(
            1j * pos * theta ** (-np.arange(0, D, 2) / D))
        ref = np.concatenate([zc.real, zc.imag], axis=1)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(O.rope_rotate_half(x, 0, theta), x)


def test_rope_relative_position_property():
    rng = np.random.default_rng(6)
    a, b = rng.normal(size=32), rng.normal(size=32)
    d1 = O.rope_rotate_half(a, 10, 500000.0) @ O.rope_rotate_half(b, 3, 500000.0)
    d2 = O.rope_rotate_half(a, 1007, 500000.0) @ O.rope_rotate_half(b, 1000, 500000.0)
    assert abs(d1 - d2) < 1e-9


def test_rms_norm_unit_weight_gives_unit_rms():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(5, 128)) * 3
    y = O.rms_norm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1.0, rtol=1e-12)


def _mat_case(rng, B=2, rows=4, m=2, d=8, L=2, Hkv=2, D=4, page=4, ctx=(3, 6)):
    max_pages = 4
    num_pages = B * max_pages
    perm = rng.permutation(num_pages).reshape(B, max_pages)
    return dict(
        hidden=rng.normal(size=(B, rows, m * d)), commit_len=np.array([2, 4]),
        start_pos=np.array(ctx), W_f=rng.normal(size=(d, m * d)) / 4, b_f=rng.normal(size=d),
        W_kv=rng.normal(size=(L, 2, Hkv * D, d)) / 3, k_norm_w=None, rms_eps=1e-6,
        rope_theta=0.0, k_pools=[rng.normal(size=(num_pages, page, Hkv, D)) for _ in range(L)],
        v_pools=[rng.normal(size=(num_pages, page, Hkv, D)) for _ in range(L)],
        page_table=perm, page_size=page)


def test_materialize_identity_weights_copy_hidden():
    rng = np.random.default_rng(8)
    c = _mat_case(rng, m=1, d=8, L=1, Hkv=2, D=4)
    c["W_f"] = np.eye(8)
    c["b_f"] = np.zeros(8)
    c["W_kv"] = np.stack([np.eye(8), 2 * np.eye(8)])[None]
    k, v = O.materialize_ctx_kv(**c)
    for b in range(2):
        for j in range(c["commit_len"][b]):
            pos = c["start_pos"][b] + j
            pg, sl = c["page_table"][b, pos // 4], pos % 4
            np.testing.assert_allclose(k[0][pg, sl].ravel(), c["hidden"][b, j], rtol=0, atol=1e-15)
            np.testing.assert_allclose(v[0][pg, sl].ravel(), 2 * c["hidden"][b, j], atol=1e-15)


def test_materialize_prefix_valid_rows_untouched_and_slots():
    rng = np.random.default_rng(9)
    c = _mat_case(rng)
    k, v = O.materialize_ctx_kv(**c)
    written = set()
    for b in range(2):
        for j in range(c["commit_len"][b]):
            pos = c["start_pos"][b] + j
            written.add((int(c["page_table"][b, pos // 4]), pos % 4))
    assert len(written) == 6
    for layer in range(2):
        for pg in range(8):
            for sl in range(4):
                if (pg, sl) not in written:
                    np.testing.assert_array_equal(k[layer][pg, sl], c["k_pools"][layer][pg, sl])
                    np.testing.assert_array_equal(v[layer][pg, sl], c["v_pools"][layer][pg, sl])


def test_materialize_matches_library_linear_chain_with_norm_and_rope():
    rng = np.random.default_rng(10)
    c = _mat_case(rng)
    c["k_norm_w"] = rng.normal(size=(2, 4)) + 1
    c["rope_theta"] = 10000.0
    k, v = O.materialize_ctx_kv(**c)
    F = torch.nn.functional
    for b in range(2):
        for j in range(c["commit_len"][b]):
            x = torch.from_numpy(c["hidden"][b, j])
            h = F.linear(x, torch.from_numpy(c["W_f"]), torch.from_numpy(c["b_f"]))
            pos = int(c["start_pos"][b] + j)
            pg, sl = c["page_table"][b, pos // 4], pos % 4
            for layer in range(2):
                kk = F.linear(h, torch.from_numpy(c["W_kv"][layer, 0])).view(2, 4)
                kk = F.rms_norm(kk, (4,), torch.from_numpy(c["k_norm_w"][layer]), eps=1e-6)
                # RoPE written as a rotation matrix acting on (x_i, x_{i+2})
                ang = pos * 10000.0 ** (-np.arange(2) * 2 / 4)
                R = np.zeros((4, 4))
                for i in range(2):
                    R[i, i], R[i, i + 2] = math.cos(ang[i]), -math.sin(ang[i])
                    R[i + 2, i], R[i + 2, i + 2] = math.sin(ang[i]), math.cos(ang[i])
                kk = kk.numpy() @ R.T
                vv = F.linear(h, torch.from_numpy(c["W_kv"][layer, 1])).view(2, 4).numpy()
                np.testing.assert_allclose(k[layer][pg, sl], kk, rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(v[layer][pg, sl], vv, rtol=1e-10, atol=1e-12)


def test_oracle_imports_nothing_from_the_cuda_path():
    import ast
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for fn in os.listdir(os.path.join(root, "oracle")):
        if not fn.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(root, "oracle", fn)).read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            for n in names:
                assert not n.startswith("block_diffusion_speculative_fusion_gb300"), (fn, n)
                # numpy and the standard library's heap queue only
                assert n.split(".")[0] in ("numpy", "heapq", "__future__", "") or n.startswith("dflash_oracle"), \
                    (fn, n)


# ---------------------------------------------------------------------------
# draft-side token choice (DFlash page, inference steps and decode listing;
# speculative-decoding page, DFlash section: one token sampled per position)
# ---------------------------------------------------------------------------
def test_draft_select_greedy_argmax_lowest_index_and_padding():
    z = np.zeros((2, 3, 6), np.float32)
    z[0, 0, [2, 4]] = 5.0          # tie: lowest index wins
    z[0, 1, 5] = 1.0
    z[0, 2, 0] = -1.0              # all others 0: the first 0 is index 1
    z[1, 0, 3] = 2.0
    r = O.draft_select(z, anchor=[7, 9], n_draft=[3, 1])
    assert r["cand"].tolist() == [[7, 2, 5, 1], [9, 3, -1, -1]]
    assert r["q_x"].tolist() == [[1.0, 1.0, 1.0], [1.0, 0.0, 0.0]]
    # row_lse is the log-sum-exp of the raw logits (scipy)
    np.testing.assert_allclose(r["row_lse"][0], scipy.special.logsumexp(z[0].astype(np.float64), axis=1),
                               rtol=1e-14)
    assert r["row_lse"][1, 1] == 0.0


def test_draft_select_greedy_matches_numpy_argmax():
    rng = np.random.default_rng(21)
    z = rng.normal(size=(3, 5, 257)).astype(np.float32)
    r = O.draft_select(z, anchor=[1, 2, 3])
    np.testing.assert_array_equal(r["cand"][:, 1:], np.argmax(z, axis=2))


def test_draft_select_sampled_closed_forms():
    V = 10
    # uniform logits: C(y) = (y + 1) / V, so y = floor(u V)
    z = np.zeros((1, 4, V), np.float32)
    u = np.array([[0.0, 0.05, 0.55, 0.999]], np.float32)
    r = O.draft_select(z, anchor=[0], u_draft=u, temperature=1.0)
    assert r["cand"][0, 1:].tolist() == [0, 0, 5, 9]
    np.testing.assert_allclose(r["q_x"][0], 0.1, rtol=1e-14)
    np.testing.assert_allclose(r["row_lse"][0], math.log(V), rtol=1e-14)
    # u exactly on a step (0.3 = C(2)) is flagged; 0.35 is not
    r2 = O.draft_select(np.zeros((1, 2, V)), anchor=[0], u_draft=np.array([[0.3, 0.35]]), temperature=1.0)
    assert r2["flags"][0].tolist() == [O.FLAG_CDF_BOUNDARY, 0]
    # one dominant logit: always that token, q = 1
    zd = np.zeros((1, 3, V), np.float32)
    zd[0, :, 6] = 1e4
    r3 = O.draft_select(zd, anchor=[0], u_draft=np.array([[0.0, 0.5, 0.999999]]), temperature=1.0)
    assert r3["cand"][0, 1:].tolist() == [6, 6, 6]
    np.testing.assert_allclose(r3["q_x"][0], 1.0)


def test_draft_select_sampled_probabilities_match_library_softmax():
    rng = np.random.default_rng(22)
    z = rng.normal(size=(2, 3, 50)) * 3
    u = rng.random((2, 3))
    for T in (0.7, 1.0, 2.0):
        r = O.draft_select(z, anchor=[0, 0], u_draft=u, temperature=T)
        p = scipy.special.softmax(z / T, axis=2)
        for b in range(2):
            for i in range(3):
                x = r["cand"][b, i + 1]
                np.testing.assert_allclose(r["q_x"][b, i], p[b, i, x], rtol=1e-12)
                # x is the inverse-CDF point of u: C(x-1) <= u < C(x)
                C = np.cumsum(p[b, i])
                assert (C[x - 1] if x > 0 else 0.0) <= u[b, i] < C[x]
        np.testing.assert_allclose(r["row_lse"], scipy.special.logsumexp(z / T, axis=2), rtol=1e-13)


def test_draft_select_sampled_histogram_is_the_softmax():
    # Monte Carlo: the draws over many uniforms follow softmax(z / T)
    rng = np.random.default_rng(23)
    V, n = 7, 20000
    z = rng.normal(size=V) * 1.5
    zz = np.broadcast_to(z, (1, n, V))
    u = rng.random((1, n))
    r = O.draft_select(zz, anchor=[0], u_draft=u, temperature=1.3)
    counts = np.bincount(r["cand"][0, 1:], minlength=V)
    p = scipy.special.softmax(z / 1.3)
    stat, pval = scipy.stats.chisquare(counts, p * n)
    assert pval > 1e-3


# ---------------------------------------------------------------------------
# DDTree (speculative-decoding page, section 6)
# ---------------------------------------------------------------------------
def test_ddtree_topk_matches_library_sort_and_log_softmax():
    rng = np.random.default_rng(31)
    z = rng.normal(size=(2, 3, 40)) * 2
    z[0, 0, [5, 9]] = 10.0                    # tie: lower index first
    tok, logp = O.ddtree_topk(z, 4, temperature=0.8)
    assert tok[0, 0, 0] == 5 and tok[0, 0, 1] == 9
    ls = scipy.special.log_softmax(z / 0.8, axis=2)
    for b in range(2):
        for i in range(3):
            ref = np.argsort(-z[b, i], kind="stable")[:4]
            np.testing.assert_array_equal(tok[b, i], ref)
            np.testing.assert_allclose(logp[b, i], ls[b, i, ref], rtol=1e-13)


def _all_paths(logp, K, n):
    """Brute force: every node of the K-ary tree of depth n as (rank path, joint log-prob)."""
    out = []
    frontier = [((), 0.0)]
    for d in range(n):
        nxt = []
        for path, lp in frontier:
            for r in range(K):
                node = (path + (r,), lp + logp[d, r])
                out.append(node)
                nxt.append(node)
        frontier = nxt
    return out


def _rank_paths(t, b):
    paths = []
    for j in range(int(t["n_nodes"][b])):
        p, rk = [], j
        while rk >= 0:
            p.append(int(t["node_rank"][b, rk]))
            rk = int(t["node_parent"][b, rk])
        paths.append(tuple(reversed(p)))
    return paths


def test_ddtree_build_is_the_top_budget_nodes_by_path_probability():
    # 6.3: the best-first tree within budget B holds the B most probable paths
    rng = np.random.default_rng(32)
    K, n = 3, 4
    z = rng.normal(size=(2, n, 12)) * 2
    tok, logp = O.ddtree_topk(z, K)
    for budget in (1, 5, 17, 40):
        t = O.ddtree_build(tok, logp, budget)
        for b in range(2):
            allp = _all_paths(logp[b], K, n)
            best = sorted(allp, key=lambda x: -x[1])[:budget]
            assert set(_rank_paths(t, b)) == {p for p, _ in best}
            # pop order: non-increasing probability, parents before children
            lp = t["node_logp"][b, :budget]
            assert np.all(np.diff(lp) <= 1e-12)
            assert np.all(t["node_parent"][b, :budget] < np.arange(budget))
            np.testing.assert_allclose(sorted(lp, reverse=True), [x for _, x in best], rtol=1e-12)


def test_ddtree_build_special_cases():
    rng = np.random.default_rng(33)
    z = rng.normal(size=(1, 3, 10))
    tok, logp = O.ddtree_topk(z, 2)
    # budget above the tree size: every node (2 + 4 + 8)
    t = O.ddtree_build(tok, logp, 50)
    assert t["n_nodes"][0] == 14
    # K = 1: the greedy draft chain
    tok1, logp1 = O.ddtree_topk(z, 1)
    t1 = O.ddtree_build(tok1, logp1, 8)
    assert t1["n_nodes"][0] == 3
    np.testing.assert_array_equal(t1["node_token"][0, :3], np.argmax(z[0], axis=1))
    np.testing.assert_array_equal(t1["node_parent"][0, :3], [-1, 0, 1])


def test_ddtree_walk_worked_example():
    # 6.5: root -> cat (accepted) -> sat (accepted) -> on (rejected); dog's subtree is dropped
    cat, dog, sat, lay, on, the = 1, 2, 3, 4, 5, 6
    node_token = np.array([[cat, dog, sat, lay, on]])
    node_parent = np.array([[-1, -1, 0, 0, 2]])
    V = 8
    tl = np.zeros((1, 6, V))
    tl[0, 0, cat] = 5      # root row: the target predicts cat
    tl[0, 1, sat] = 5      # after cat: sat
    tl[0, 2, lay] = 5      # after dog (not reached)
    tl[0, 3, the] = 5      # after sat: "the", so on is rejected
    r = O.ddtree_walk_greedy(tl, node_token, node_parent, np.array([5]))
    assert r["accept_len"][0] == 2 and r["commit_len"][0] == 3
    assert r["path"][0, :2].tolist() == [0, 2]
    assert r["out_tokens"][0, :3].tolist() == [cat, sat, the] and r["bonus"][0] == the


def test_ddtree_walk_on_a_chain_is_the_greedy_rule():
    # a K = 1 tree is the DFlash draft: the walk equals the greedy verify rule
    rng = np.random.default_rng(34)
    B, n, V = 4, 5, 6
    zt = rng.normal(size=(B, n + 1, V)) * 3
    cand = np.zeros((B, n + 1), dtype=np.int64)
    cand[:, 1:] = rng.integers(0, V, size=(B, n))
    for b in range(2):     # the first two sequences follow the target for a while
        cand[b, 1:4] = np.argmax(zt[b, :3], axis=1)
    node_token = cand[:, 1:]
    node_parent = np.tile(np.arange(-1, n - 1), (B, 1))
    r = O.ddtree_walk_greedy(zt, node_token, node_parent, np.full(B, n))
    g = O.verify_greedy(zt, cand)
    np.testing.assert_array_equal(r["accept_len"], g["accept_len"])
    np.testing.assert_array_equal(r["bonus"], g["bonus"])
    np.testing.assert_array_equal(r["out_tokens"][:, :n + 1], g["out_tokens"])
