"""GPU parity of the verify and gate kernels against the CPU oracle.

Integer outputs must match bit for bit, except for sequences the oracle flags
because a uniform sat within 1e-6 of a decision boundary; fp32 probabilities
must match within 1e-5 relative; gate scores within 1e-4 absolute (the gate's
flag band) and its decisions exactly outside that band.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_speculative_fusion_gb300 import api, synth
from block_diffusion_speculative_fusion_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_fusion_gb300 import build
    build.build()
    api.lib()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def npy(t):
    return t.detach().cpu().numpy()


def gpu(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------
def _check_greedy(vb):
    g = gpu(vb)
    out = api.verify_greedy(g["target_logits"], g["cand"], g["n_draft"], want_target_pred=True)
    torch.cuda.synchronize()
    ref = O.verify_greedy(f64(vb["target_logits"]), npy(vb["cand"]), npy(vb["n_draft"]))
    for key in ("accept_len", "bonus", "commit_len", "out_tokens", "target_pred"):
        np.testing.assert_array_equal(npy(out[key]), ref[key], err_msg=key)
    return ref


def test_greedy_tiny_f32():
    _check_greedy(synth.verify_batch(W.TINY_F32, seed=0))


def test_greedy_tiny_f32_ragged_batch():
    ref = _check_greedy(synth.verify_batch(W.TINY_F32, seed=1, B=40, ragged=True))
    assert len(set(ref["accept_len"].tolist())) > 1


def test_greedy_llama8b_b1_k10():
    _check_greedy(synth.verify_batch(W.LLAMA8B_B1, seed=0))


def test_greedy_batched_llama8b_b32_full_size():
    ref = _check_greedy(synth.verify_batch(W.LLAMA8B_B64, seed=0, B=32, greedy_rows=32))
    assert ref["accept_len"].mean() > 1.0


def test_greedy_ties_across_chunks_take_lowest_index():
    B, R, V = 3, 4, 128256
    z = torch.randn(B, R, V, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    z[0, 0, 7] = z[0, 0, V - 3] = 30.0          # far apart: different chunks
    z[1, 1, 100] = z[1, 1, 99] = 30.0
    z[2, :, :] = 1.0                             # whole rows equal: index 0
    cand = torch.zeros(B, R, dtype=torch.int64)
    cand[0, 1] = 7
    cand[1, 2] = 99
    vb = {"target_logits": z, "cand": cand, "n_draft": torch.full((B,), R - 1, dtype=torch.int32)}
    ref = _check_greedy(vb)
    assert ref["target_pred"][0, 0] == 7 and ref["target_pred"][1, 1] == 99
    assert ref["target_pred"][2].tolist() == [0, 0, 0, 0]


def test_greedy_no_drafts():
    vb = synth.verify_batch(W.TINY_F32, seed=2, B=5, n_max=0)
    ref = _check_greedy(vb)
    assert np.all(ref["accept_len"] == 0) and np.all(ref["commit_len"] == 1)


def test_greedy_odd_vocab_unaligned_rows():
    wl = W.TINY_F32
    vb = synth.verify_batch(wl, seed=3, B=7, ragged=True)
    V = 997       # rows are no longer 16-byte aligned
    vb["target_logits"] = vb["target_logits"][:, :, :V].contiguous()
    vb["cand"] = vb["cand"] % V
    _check_greedy(vb)
    vb["target_logits"] = vb["target_logits"].to(torch.bfloat16)
    _check_greedy(vb)


# ---------------------------------------------------------------------------
# sampled
# ---------------------------------------------------------------------------
def _check_sample(vb, temperature=1.0, max_flag_frac=0.5, probs_rtol=None, draft_row_lse=None):
    """A residual spread over ~1e5 tokens has CDF steps of ~1e-5, so the 1e-6
    boundary band flags a visible share of draws; flagged sequences are valid
    draws that are reported, not compared (spec rule)."""
    g = gpu(vb)
    out = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"],
                            temperature, g["n_draft"], want_probs=True, draft_row_lse=draft_row_lse)
    torch.cuda.synchronize()
    ref = O.verify_sample(f64(vb["target_logits"]), f64(vb["draft_logits"]), npy(vb["cand"]),
                          npy(vb["n_draft"]), npy(vb["u_acc"]), npy(vb["u_final"]), temperature)
    ok = ref["flags"] == 0
    assert ok.mean() >= 1.0 - max_flag_frac, ref["flags"]
    for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
        np.testing.assert_array_equal(npy(out[key])[ok], ref[key][ok], err_msg=key)
    # flagged draws mostly agree too: the fp32 error is far inside the 1e-6 band
    flagged = ~ok
    if flagged.any():
        same = np.all(npy(out["out_tokens"])[flagged] == ref["out_tokens"][flagged], axis=1)
        assert (~same).sum() <= max(1, 0.1 * flagged.sum())
    if probs_rtol is not None:
        pr = npy(out["probs"])
        n_max = vb["u_acc"].shape[1]
        for b in range(len(ok)):
            d = ref["debug"][b]
            k = len(d["p_x"])
            np.testing.assert_allclose(pr[b, :k], d["p_x"], rtol=probs_rtol)
            np.testing.assert_allclose(pr[b, n_max:n_max + k], d["q_x"], rtol=probs_rtol)
            Z = d["Z"] if d["Z"] is not None else 1.0
            np.testing.assert_allclose(pr[b, 2 * n_max], Z, rtol=probs_rtol)
    return out, ref


def test_sample_tiny_f32_probs():
    _check_sample(synth.verify_batch(W.TINY_F32, seed=0, greedy_rows=0), probs_rtol=1e-5)


def test_sample_tiny_f32_ragged_batch():
    out, ref = _check_sample(synth.verify_batch(W.TINY_F32, seed=4, B=64, greedy_rows=0, ragged=True),
                             probs_rtol=1e-5)
    assert len(set(ref["accept_len"].tolist())) > 1


@pytest.mark.parametrize("temperature", [0.7, 1.5])
def test_sample_temperature(temperature):
    _check_sample(synth.verify_batch(W.TINY_F32, seed=6, B=32, greedy_rows=0), temperature, probs_rtol=1e-5)


def _worked_inputs(u_acc, u_final):
    ex = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    lp = torch.log(torch.tensor(ex["p"], dtype=torch.float32))
    lq = torch.log(torch.tensor(ex["q"], dtype=torch.float32))
    B = len(u_acc)
    zt = lp.repeat(B, 2, 1).contiguous()
    zd = lq.repeat(B, 1, 1).contiguous()
    cand = torch.zeros(B, 2, dtype=torch.int64)
    cand[:, 0] = 3
    cand[:, 1] = ex["tokens"].index("cat")
    return ex, {"target_logits": zt, "draft_logits": zd, "cand": cand,
                "n_draft": torch.ones(B, dtype=torch.int32),
                "u_acc": torch.tensor(u_acc, dtype=torch.float32).view(B, 1),
                "u_final": torch.tensor(u_final, dtype=torch.float32)}


def test_sample_worked_example_on_gpu():
    ex, vb = _worked_inputs([0.70, 0.72, 0.9, 0.9, 0.9, 0.7142857], [0.3, 0.3, 0.3, 0.7, 0.5, 0.3])
    g = gpu(vb)
    out = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"],
                            1.0, g["n_draft"], want_probs=True)
    torch.cuda.synchronize()
    acc, bonus, flags, probs = (npy(out[k]) for k in ("accept_len", "bonus", "flags", "probs"))
    tok = ex["tokens"]
    assert acc[0] == 1 and acc[1] == 0 and acc[2] == 0
    assert bonus[1] == tok.index("dog") and bonus[2] == tok.index("dog") and bonus[3] == tok.index("sat")
    assert flags[4] & api.FLAG_CDF_BOUNDARY
    assert flags[5] & api.FLAG_ACCEPT_BOUNDARY
    assert flags[0] == 0 and flags[1] == 0
    np.testing.assert_allclose(probs[1], [0.5, 0.7, 0.2], rtol=1e-5)      # p(cat), q(cat), 1 - beta
    np.testing.assert_allclose(probs[1, 0] / probs[1, 1], ex["accept_ratio"], rtol=1e-5)


@pytest.mark.parametrize("sigma", W.QWEN3_4B_B8.sigma_sweep)
def test_sample_qwen3_4b_b8_sigma_sweep(sigma):
    out, ref = _check_sample(synth.verify_batch(W.QWEN3_4B_B8, seed=0, sigma=sigma))


def test_sample_batched_llama8b_b32_full_size():
    vb = synth.verify_batch(W.LLAMA8B_B64, seed=0, B=32, greedy_rows=0)
    out, ref = _check_sample(vb)
    assert ref["accept_len"].mean() > 0.5


def test_sample_dloop_concatenated_ragged():
    wl = W.DLOOP_QWEN3_4B
    vb = synth.verify_batch(wl, seed=0, B=8, ragged=True)
    _check_sample(vb)


def test_sample_identical_logits_never_reject():
    vb = synth.verify_batch(W.TINY_F32, seed=7, B=16, greedy_rows=0)
    vb["draft_logits"] = vb["target_logits"][:, :-1].contiguous()
    g = gpu(vb)
    out = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"], 1.0,
                            g["n_draft"])
    assert torch.all(out["accept_len"].cpu() == vb["n_draft"])


def test_sample_one_hot_equals_greedy_on_gpu():
    B, n, V = 64, 7, 300
    gen = torch.Generator().manual_seed(11)
    tp = torch.randint(0, V, (B, n + 1), generator=gen)
    cand = torch.randint(0, V, (B, n + 1), generator=gen)
    agree = torch.rand(B, n, generator=gen) < 0.7
    cand[:, 1:] = torch.where(agree, tp[:, :n], cand[:, 1:])
    zt = torch.full((B, n + 1, V), -1e4)
    zt.scatter_(2, tp.unsqueeze(-1), 0.0)
    zd = torch.full((B, n, V), -1e4)
    zd.scatter_(2, cand[:, 1:].unsqueeze(-1), 0.0)
    nd = torch.randint(0, n + 1, (B,), generator=gen).to(torch.int32)
    ua, uf = torch.rand(B, n, generator=gen), torch.rand(B, generator=gen)
    s = api.verify_sample(zt.to(DEV), zd.to(DEV), cand.to(DEV), ua.to(DEV), uf.to(DEV), 1.0, nd.to(DEV))
    gr = api.verify_greedy(zt.to(DEV), cand.to(DEV), nd.to(DEV))
    for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
        assert torch.equal(s[key].cpu(), gr[key].cpu()), key


@pytest.mark.parametrize("V", [2, 5, 17])
def test_sample_identity_monte_carlo_on_gpu(V):
    """min(p,q) + max(0,p-q) = p: the first emitted token of a one-draft verify,
    with x ~ q, is distributed as p (speculative-decoding page, section 3)."""
    rng = np.random.default_rng(200 + V)
    lp = rng.normal(0, 1.5, V).astype(np.float32)
    lq = rng.normal(0, 1.5, V).astype(np.float32)
    p = np.exp(lp.astype(np.float64) - lp.max()); p /= p.sum()
    q = np.exp(lq.astype(np.float64) - lq.max()); q /= q.sum()
    B, calls = 2000, 512
    zt = torch.from_numpy(np.broadcast_to(lp, (B, 2, V)).copy()).to(DEV)
    zd = torch.from_numpy(np.broadcast_to(lq, (B, 1, V)).copy()).to(DEV)
    counts = np.zeros(V)
    accepted = 0
    for _ in range(calls):
        x = torch.from_numpy(rng.choice(V, size=B, p=q))
        cand = torch.stack([torch.zeros(B, dtype=torch.int64), x], 1).to(DEV)
        ua = torch.from_numpy(rng.random((B, 1), dtype=np.float32)).to(DEV)
        uf = torch.from_numpy(rng.random(B, dtype=np.float32)).to(DEV)
        o = api.verify_sample(zt, zd, cand, ua, uf, 1.0)
        first = o["out_tokens"][:, 0].cpu().numpy()
        counts += np.bincount(first, minlength=V)
        accepted += int(o["accept_len"].sum())
    n = B * calls
    expected = p * n
    stat = ((counts - expected) ** 2 / expected).sum()
    from scipy.stats import chi2
    assert chi2.sf(stat, V - 1) > 1e-3
    beta = np.minimum(p, q).sum()
    assert abs(accepted / n - beta) < 5 * math.sqrt(beta * (1 - beta) / n)


def _boundary_distance(ref, vb, b):
    """How far sequence b's uniforms sit from the oracle's decision boundaries:
    every evaluated accept test with p/q < 1, and the two CDF steps around the
    drawn token (speculative-decoding page, section 3)."""
    d = ref["debug"][b]
    u = npy(vb["u_acc"])[b].astype(np.float64)
    dist = np.inf
    for i, (px, qx) in enumerate(zip(d["p_x"], d["q_x"])):
        if qx > 0 and px / qx < 1.0:
            dist = min(dist, abs(u[i] - px / qx))
    fd = d["final_dist"]
    y = int(ref["bonus"][b])
    c_hi = fd[:y + 1].sum()
    uf = float(npy(vb["u_final"])[b])
    return min(dist, abs(c_hi - fd[y] - uf), abs(c_hi - uf))


def _full_size_sample_case(name):
    if name == "llama8b_b32_sigma2":
        return synth.verify_batch(W.LLAMA8B_B64, seed=0, B=32, greedy_rows=0)
    if name.startswith("qwen3_4b_b8_sigma"):
        return synth.verify_batch(W.QWEN3_4B_B8, seed=0, sigma=float(name.split("sigma")[1]))
    return synth.verify_batch(W.DLOOP_QWEN3_4B, seed=3, B=32, ragged=True)


@pytest.mark.parametrize("name", ["llama8b_b32_sigma2", "qwen3_4b_b8_sigma0.5", "qwen3_4b_b8_sigma2",
                                  "qwen3_4b_b8_sigma4", "dloop_b32_concatenated_ragged"])
def test_sample_full_size_probs_ratio_and_flag_bands(name):
    """bf16 full-size sampled verify: p(x), q(x) of every evaluated draft and
    the drawn distribution's mass Z within 1e-5 relative; the accept ratio p/q
    within 3e-7 of the oracle's (under a third of the 1e-6 flag band); and the flags
    decided by the band: a sequence whose uniforms lie more than 1.5e-6 from
    every oracle boundary is unflagged on the GPU and bit-exact, one within
    0.5e-6 of a boundary is flagged on the GPU too."""
    vb = _full_size_sample_case(name)
    out, ref = _check_sample(vb, max_flag_frac=1.0)
    pr = npy(out["probs"]).astype(np.float64)
    n_max = vb["u_acc"].shape[1]
    gflags = npy(out["flags"])
    worst_ratio, worst_rel = 0.0, 0.0
    near = far = 0
    for b in range(len(gflags)):
        d = ref["debug"][b]
        k = len(d["p_x"])
        gp, gq = pr[b, :k], pr[b, n_max:n_max + k]
        np.testing.assert_allclose(gp, d["p_x"], rtol=1e-5, atol=1e-30)
        np.testing.assert_allclose(gq, d["q_x"], rtol=1e-5, atol=1e-30)
        worst_rel = max(worst_rel, float(np.max(np.abs(gp / np.maximum(d["p_x"], 1e-300) - 1.0), initial=0.0)))
        Z = d["Z"] if d["Z"] is not None else 1.0
        np.testing.assert_allclose(pr[b, 2 * n_max], Z, rtol=1e-5)
        for i in range(k):
            r_o = d["p_x"][i] / d["q_x"][i]
            if r_o < 1.0:
                worst_ratio = max(worst_ratio, abs(gp[i] / gq[i] - r_o))
        dist = _boundary_distance(ref, vb, b)
        if dist > 1.5e-6:
            far += 1
            assert gflags[b] == 0, (b, dist, gflags[b])
            for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
                np.testing.assert_array_equal(npy(out[key])[b], ref[key][b], err_msg=f"{key} seq {b}")
        elif dist < 0.5e-6:
            near += 1
            assert gflags[b] != 0, (b, dist)
    print(f"[{name}] sequences {len(gflags)}: far {far}, near {near}, oracle-flagged "
          f"{int((ref['flags'] != 0).sum())}, GPU-flagged {int((gflags != 0).sum())}; "
          f"max |ratio - oracle| {worst_ratio:.3e}, max rel p(x) {worst_rel:.3e}")
    # the fp32 probabilities (ratio formed in fp64) err far inside the band
    assert worst_ratio < 3e-7, worst_ratio


def test_verify_is_deterministic():
    vb = gpu(synth.verify_batch(W.QWEN3_4B_B8, seed=9))
    a = api.verify_sample(vb["target_logits"], vb["draft_logits"], vb["cand"], vb["u_acc"], vb["u_final"])
    a = {k: v.clone() for k, v in a.items()}
    b = api.verify_sample(vb["target_logits"], vb["draft_logits"], vb["cand"], vb["u_acc"], vb["u_final"])
    for k in a:
        assert torch.equal(a[k], b[k]), k


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------
def _check_gate(gb, temperature, g):
    d = gpu(gb)
    out = api.gate(d["draft_logits"], d["tokens"], temperature, g, d.get("active"), want_row_lse=True)
    torch.cuda.synchronize()
    ref = O.gate(f64(gb["draft_logits"]), npy(gb["tokens"]),
                 None if gb.get("active") is None else npy(gb["active"]), temperature, g)
    np.testing.assert_allclose(npy(out["c"]), ref["c"], atol=1e-4, rtol=0)
    np.testing.assert_allclose(npy(out["row_lse"]), ref["row_lse"], rtol=2e-6, atol=1e-5)
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(npy(out["cont"])[ok], ref["cont"][ok])
    return out, ref


def test_gate_dloop_shape_all_stages():
    wl = W.DLOOP_QWEN3_4B
    conts = []
    for s in range(wl.stages):
        out, ref = _check_gate(synth.gate_batch(wl, s, seed=0), wl.temperature, wl.gate_g)
        conts.append(ref["cont"])
    conts = np.array(conts)
    assert 0 < conts.mean() < 1            # the gate both continues and stops


def test_gate_tiny_inactive_and_temperature():
    wl = W.TINY_F32
    gb = synth.gate_batch(wl, 0, seed=1, B=9)
    gb["active"] = torch.tensor([1, 0, 1, 1, 0, 1, 1, 1, 0], dtype=torch.uint8)
    out, ref = _check_gate(gb, 0.8, -3.0)
    assert np.all(npy(out["cont"])[[1, 4, 8]] == 0) and np.all(npy(out["c"])[[1, 4, 8]] == 0)


def test_gate_uniform_logits_closed_form_on_gpu():
    B, k, V = 4, 7, 151936
    z = torch.zeros(B, k, V, dtype=torch.bfloat16, device=DEV)
    tok = torch.randint(0, V, (B, k), device=DEV)
    out = api.gate(z, tok, 1.0, -0.5, want_row_lse=True)
    np.testing.assert_allclose(npy(out["c"]), -k * math.log(V), rtol=1e-6)
    assert torch.all(out["cont"] == 0)


# ---- sampled rule fed with the draft rows' log-sum-exps (DLoop: the gates'
# row LSEs) instead of streaming the draft rows ----
def _exact_row_lse(vb, temperature):
    z = f64(vb["draft_logits"]) / temperature
    m = z.max(axis=2, keepdims=True)
    return torch.from_numpy((m[..., 0] + np.log(np.exp(z - m).sum(axis=2))).astype(np.float32)).to(DEV)


def test_sample_lse_tiny_f32_probs():
    vb = synth.verify_batch(W.TINY_F32, seed=0, greedy_rows=0)
    _check_sample(vb, probs_rtol=1e-5, draft_row_lse=_exact_row_lse(vb, 1.0))


@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_sample_lse_from_gate_dloop_concatenated(temperature):
    # the gate over the concatenated draft rows (what the stages' gate calls
    # produce) supplies the row LSEs of the looped verify
    wl = W.DLOOP_QWEN3_4B
    vb = synth.verify_batch(wl, seed=1, B=8, ragged=True)
    g = gpu(vb)
    gt = api.gate(g["draft_logits"], g["cand"][:, 1:].contiguous(), temperature, -0.5, want_row_lse=True)
    _check_sample(vb, temperature=temperature, draft_row_lse=gt["row_lse"])


def test_sample_lse_matches_streamed_rule_llama8b_b32():
    vb = synth.verify_batch(W.LLAMA8B_B64, seed=2, B=32, greedy_rows=0)
    g = gpu(vb)
    a = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"], 1.0,
                          g["n_draft"])
    a = {k: v.clone() for k, v in a.items()}
    gt = api.gate(g["draft_logits"], g["cand"][:, 1:].contiguous(), 1.0, -0.5, want_row_lse=True)
    b = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"], 1.0,
                          g["n_draft"], draft_row_lse=gt["row_lse"])
    torch.cuda.synchronize()
    ok = (npy(a["flags"]) == 0) & (npy(b["flags"]) == 0)
    for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
        np.testing.assert_array_equal(npy(a[key])[ok], npy(b[key])[ok], err_msg=key)
    assert ok.mean() > 0.5


# ---------------------------------------------------------------------------
# DLoop looped step: gates chained on the device, then one verify of the
# S_b * k concatenated candidates
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [5, 6])
def test_dloop_looped_chain_matches_oracle(seed):
    """DLoop page, mechanism 1 and the looped verify: stage s is drafted only
    while every earlier gate continued (the next stage's active mask is this
    stage's cont, on the device); the stage that stops is still verified; the
    verify checks the S_b * k concatenated candidates with the sampled rule,
    fed the gates' row LSEs. Compared with oracle.gate per stage,
    oracle.dloop_stage_count and oracle.verify_sample over n_b = S_b * k."""
    wl = W.DLOOP_QWEN3_4B
    B, k, S, T = wl.B, wl.n_draft, wl.stages, wl.temperature
    n_max = S * k
    vb = synth.verify_batch(wl, seed=seed)
    g = gpu(vb)
    row_lse = torch.zeros(B, n_max, dtype=torch.float32, device=DEV)
    n_verify = torch.zeros(B, dtype=torch.int32, device=DEV)
    conts, cvals, gflags = [], [], []
    active = None
    for s in range(S):
        o = api.gate_stage(g["draft_logits"], g["cand"], s, k, T, wl.gate_g, active=active, row_lse=row_lse,
                           n_verify=n_verify)
        conts.append(o["cont"].clone())
        cvals.append(o["c"].clone())
        gflags.append(o["flags"].clone())
        active = conts[-1]
    out = api.verify_sample(g["target_logits"], g["draft_logits"], g["cand"], g["u_acc"], g["u_final"], T,
                            n_verify, draft_row_lse=row_lse)
    torch.cuda.synchronize()
    # ---- the oracle's chain ----
    zd = f64(vb["draft_logits"])
    cand = npy(vb["cand"])
    act = np.ones(B, dtype=np.uint8)
    conts_o, flagged = [], np.zeros(B, bool)
    for s in range(S):
        ref = O.gate(zd[:, s * k:(s + 1) * k], cand[:, 1 + s * k:1 + (s + 1) * k], act, T, wl.gate_g)
        flagged |= (ref["flags"] != 0) | (npy(gflags[s]) != 0)
        ok = ~flagged
        np.testing.assert_allclose(npy(cvals[s])[ok], ref["c"][ok], atol=1e-4, rtol=0)
        np.testing.assert_array_equal(npy(conts[s])[ok], ref["cont"][ok], err_msg=f"cont stage {s}")
        conts_o.append(ref["cont"])
        act = ref["cont"].astype(np.uint8)
    S_b = O.dloop_stage_count(np.array(conts_o))
    ok = ~flagged
    np.testing.assert_array_equal(npy(n_verify)[ok], (S_b * k)[ok])
    assert 1 < len(set(S_b[ok].tolist()))            # the gates both stop and continue
    ref_v = O.verify_sample(f64(vb["target_logits"]), zd, cand, S_b * k, npy(vb["u_acc"]), npy(vb["u_final"]), T)
    ok &= ref_v["flags"] == 0
    ok &= npy(out["flags"]) == 0
    assert ok.mean() > 0.5
    for key in ("accept_len", "bonus", "commit_len", "out_tokens"):
        np.testing.assert_array_equal(npy(out[key])[ok], ref_v[key][ok], err_msg=key)
