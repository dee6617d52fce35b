"""GPU parity of the draft-side token choice (dflash_draft_select) against the
CPU oracle: candidates bit-exact (sampled rows flagged near a CDF step by either
side are reported and left out), q(x) and the row log-sum-exp within 1e-5
relative (fp32 arithmetic over up to 152k-token rows)."""
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


def _check(wl, temperature, seed, ragged=False, B=None, n_max=None):
    p = synth.draft_select_batch(wl, seed=seed, B=B, n_max=n_max, ragged=ragged)
    g = {k: v.to(DEV) for k, v in p.items()}
    got = api.draft_select(g["draft_logits"], g["anchor"], temperature, u_draft=g["u_draft"], n_draft=g["n_draft"])
    torch.cuda.synchronize()
    ref = O.draft_select(p["draft_logits"].float().numpy(), p["anchor"].numpy(), p["n_draft"].numpy(),
                         p["u_draft"].numpy(), temperature)
    cand = got["cand"].cpu().numpy()
    flags = got["flags"].cpu().numpy()
    assert np.array_equal(cand[:, 0], ref["cand"][:, 0])
    skip = (flags != 0) | (ref["flags"] != 0)
    live = ~skip
    assert np.array_equal(cand[:, 1:][live], ref["cand"][:, 1:][live]), "candidates differ"
    nd = p["n_draft"].numpy()
    pad = np.arange(cand.shape[1] - 1)[None, :] >= nd[:, None]
    assert np.all(cand[:, 1:][pad] == -1)
    q = got["q_x"].cpu().numpy().astype(np.float64)
    lse = got["row_lse"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(q[live], ref["q_x"][live], rtol=1e-5, atol=1e-30)
    np.testing.assert_allclose(lse[~pad], ref["row_lse"][~pad], rtol=1e-5, atol=1e-5)
    return int(skip.sum())


def test_draft_select_greedy_tiny_f32_ragged():
    for seed in (1, 2):
        _check(W.TINY_F32, 0.0, seed, ragged=True)


def test_draft_select_sampled_tiny_f32():
    for seed in (3, 4):
        _check(W.TINY_F32, 1.0, seed, ragged=True)


def test_draft_select_greedy_llama8b_b64():
    # 64 sequences x 16 MASK positions x 128256 tokens, bf16
    assert _check(W.LLAMA8B_B64, 0.0, seed=5) == 0


@pytest.mark.parametrize("temperature", [1.0, 0.6])
def test_draft_select_sampled_qwen3_4b_b8(temperature):
    flagged = _check(W.QWEN3_4B_B8, temperature, seed=6, ragged=True)
    assert flagged <= 2


def test_draft_select_sampled_dloop_b32():
    _check(W.DLOOP_QWEN3_4B, 1.0, seed=7)


def test_draft_select_deterministic():
    p = synth.draft_select_batch(W.QWEN3_4B_B8, seed=8)
    g = {k: v.to(DEV) for k, v in p.items()}
    a = api.draft_select(g["draft_logits"], g["anchor"], 1.0, u_draft=g["u_draft"])
    a = {k: v.clone() for k, v in a.items()}
    b = api.draft_select(g["draft_logits"], g["anchor"], 1.0, u_draft=g["u_draft"])
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k
