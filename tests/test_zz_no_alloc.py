"""dflash_verify_greedy_noalloc: the greedy verify on the library's fixed
device scratch instead of a caller workspace.

The GPU tests call it twice in a row on different inputs (the second call
starts from the counter state the first one left) and compare every output with
dflash_verify_greedy on a caller workspace; the outputs are integers, so the
comparison is exact. The host test checks the size limit, which is enforced
before any CUDA call. This file is named to be collected last, so that it also
runs after every other test has used the library in the same process.
"""
import ctypes

import pytest
import torch

from block_diffusion_speculative_fusion_gb300 import api, build, synth
from block_diffusion_speculative_fusion_gb300 import workloads as W

DEV = "cuda:0"
KEYS = ("accept_len", "bonus", "commit_len", "out_tokens", "target_pred")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def _fake_ptrs(n):
    return [ctypes.c_void_p(0x1000 + 256 * i) for i in range(n)]


def test_oversized_dims_rejected_before_launch(L):
    # B * (n_max + 1) = 32000 rows: 256000 bytes of partials + 16384 of counters
    d = api.VerifyDims(2000, 15, 1000, api.BF16)
    need = L.dflash_verify_greedy_workspace_size(ctypes.byref(d))
    assert need > 256 * 1024
    p = _fake_ptrs(8)
    rc = L.dflash_verify_greedy_noalloc(ctypes.byref(d), p[0], p[1], None, p[2], p[3], p[4], p[5], None, None)
    assert rc == api.ERR_UNSUPPORTED
    assert "scratch" in api.last_error()
    # argument errors come first, as for the workspace entry point
    rc = L.dflash_verify_greedy_noalloc(ctypes.byref(d), None, p[1], None, p[2], p[3], p[4], p[5], None, None)
    assert rc == api.ERR_INVALID_ARG


def _compare(vb):
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in vb.items()}
    ref = api.verify_greedy(g["target_logits"], g["cand"], g["n_draft"], want_target_pred=True)
    got = api.verify_greedy_noalloc(g["target_logits"], g["cand"], g["n_draft"], want_target_pred=True)
    assert api.last_launch_count() == 1
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key].cpu(), ref[key].cpu()), key
    return got


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_full_size(L):
    # llama8b shape: B = 64 sequences, 16 drafts, 128256-token vocabulary, bf16
    wl = W.LLAMA8B_B64
    first = _compare(synth.verify_batch(wl, seed=11, greedy_rows=wl.B))
    second = _compare(synth.verify_batch(wl, seed=12, greedy_rows=wl.B))
    # the two problems differ, so the second call did not replay the first
    assert not torch.equal(first["target_pred"].cpu(), second["target_pred"].cpu())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_ragged_f32(L):
    for seed in (3, 4):
        _compare(synth.verify_batch(W.TINY_F32, seed=seed, ragged=True))
