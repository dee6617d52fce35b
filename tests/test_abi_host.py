"""Host-side checks of the C ABI: the library loads without a GPU, exports every
symbol the header declares, sizes workspaces from dims alone, and rejects bad
arguments before launching anything."""
import ctypes
import os
import re

import pytest

from block_diffusion_speculative_fusion_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(dflash_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert len(names) >= 12
    for n in sorted(names):
        assert hasattr(L, n), n
    # the binding binds every declared symbol with a signature
    assert names <= set(api._SIGS), names - set(api._SIGS)


def test_workspace_sizes_need_no_gpu(L):
    d = api.VerifyDims(64, 15, 128256, api.BF16)
    g = L.dflash_verify_greedy_workspace_size(ctypes.byref(d))
    s = L.dflash_verify_sample_workspace_size(ctypes.byref(d))
    assert g > api.WS_COUNTER_BYTES and s > g
    gd = api.GateDims(32, 7, 151936, api.BF16)
    assert L.dflash_gate_workspace_size(ctypes.byref(gd)) > api.WS_COUNTER_BYTES
    bad = api.VerifyDims(0, 15, 100, api.BF16)
    assert L.dflash_verify_greedy_workspace_size(ctypes.byref(bad)) == 0
    assert "bad dims" in api.last_error()


def test_attention_causal_flag_checked_on_host(L):
    d = api.AttnDims(2, 16, 16, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 1)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(d)) > api.WS_COUNTER_BYTES
    bad = api.AttnDims(2, 16, 16, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 2)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(bad)) == 0
    assert "causal" in api.last_error()
    short = api.AttnDims(2, 16, 15, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 1)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(short)) == 0
    assert "n_kv_blk" in api.last_error()
    # the unmasked form takes a block shorter than the queries
    short0 = api.AttnDims(2, 16, 15, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 0)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(short0)) > api.WS_COUNTER_BYTES


def test_draft_select_checks_on_host(L):
    d = api.VerifyDims(64, 16, 128256, api.BF16)
    assert L.dflash_draft_select_workspace_size(ctypes.byref(d)) > api.WS_COUNTER_BYTES
    big = api.VerifyDims(512, 16, 128256, api.BF16)       # 8192 rows > one counter each
    assert L.dflash_draft_select_workspace_size(ctypes.byref(big)) == 0
    assert "rows" in api.last_error()
    p = [ctypes.c_void_p(0x1000 + 256 * i) for i in range(8)]
    ws = ctypes.c_void_p(0x100000)
    need = L.dflash_draft_select_workspace_size(ctypes.byref(d))
    # sampling without uniforms, a negative temperature, a missing output: rejected before any launch
    rc = L.dflash_draft_select(ctypes.byref(d), ctypes.c_float(1.0), p[0], p[1], None, None, p[2], None, None,
                               None, ws, need, None)
    assert rc == api.ERR_INVALID_ARG and "u_draft" in api.last_error()
    rc = L.dflash_draft_select(ctypes.byref(d), ctypes.c_float(-1.0), p[0], p[1], None, p[3], p[2], None, None,
                               None, ws, need, None)
    assert rc == api.ERR_INVALID_ARG and "temperature" in api.last_error()
    rc = L.dflash_draft_select(ctypes.byref(d), ctypes.c_float(0.0), p[0], p[1], None, None, None, None, None,
                               None, ws, need, None)
    assert rc == api.ERR_INVALID_ARG


def test_ddtree_dims_checked_on_host(L):
    d = api.TreeDims(8, 15, 151936, api.BF16, 8, 512)
    assert L.dflash_ddtree_verify_workspace_size(ctypes.byref(d)) > api.WS_COUNTER_BYTES
    assert L.dflash_ddtree_verify_workspace_size(ctypes.byref(api.TreeDims(8, 15, 151936, api.BF16, 3, 512))) > 0
    for bad, word in ((api.TreeDims(8, 15, 151936, api.BF16, 17, 512), "K=17"),
                      (api.TreeDims(8, 15, 10, api.BF16, 16, 512), "K=16"),
                      (api.TreeDims(8, 15, 151936, api.BF16, 8, 5000), "budget"),
                      (api.TreeDims(8, 300, 151936, api.BF16, 8, 512), "n=")):
        assert L.dflash_ddtree_verify_workspace_size(ctypes.byref(bad)) == 0
        assert word in api.last_error(), api.last_error()


def _p(x):
    return ctypes.c_void_p(x)


def test_verify_rejects_bad_arguments_before_launch(L):
    d = api.VerifyDims(2, 3, 100, api.BF16)
    ws_need = L.dflash_verify_greedy_workspace_size(ctypes.byref(d))
    fake = 0x10000   # never dereferenced: every call below fails validation first
    args = [_p(fake)] * 5 + [None, None]
    rc = L.dflash_verify_greedy(ctypes.byref(d), None, *args, _p(fake), ws_need, None)
    assert rc == api.ERR_INVALID_ARG and "NULL" in api.last_error()
    rc = L.dflash_verify_greedy(ctypes.byref(d), _p(fake), *args, None, ws_need, None)
    assert rc == api.ERR_WORKSPACE
    rc = L.dflash_verify_greedy(ctypes.byref(d), _p(fake), *args, _p(fake), ws_need - 1, None)
    assert rc == api.ERR_WORKSPACE and "required" in api.last_error()
    rc = L.dflash_verify_greedy(ctypes.byref(d), _p(fake), *args, _p(fake + 8), ws_need, None)
    assert rc == api.ERR_WORKSPACE and "aligned" in api.last_error()
    d2 = api.VerifyDims(2, 300, 100, api.BF16)
    rc = L.dflash_verify_greedy(ctypes.byref(d2), _p(fake), *args, _p(fake), 1 << 30, None)
    assert rc == api.ERR_UNSUPPORTED
    d3 = api.VerifyDims(2, 3, 100, 7)
    rc = L.dflash_verify_greedy(ctypes.byref(d3), _p(fake), *args, _p(fake), 1 << 30, None)
    assert rc == api.ERR_INVALID_ARG and "dtype" in api.last_error()


def test_sample_and_gate_reject_bad_temperature(L):
    d = api.VerifyDims(2, 3, 100, api.F32)
    fake = _p(0x10000)
    rc = L.dflash_verify_sample(ctypes.byref(d), ctypes.c_float(0.0), *([fake] * 13), 1 << 30, None)
    assert rc == api.ERR_INVALID_ARG and "temperature" in api.last_error()
    gd = api.GateDims(2, 3, 100, api.F32)
    rc = L.dflash_gate(ctypes.byref(gd), ctypes.c_float(-1.0), ctypes.c_float(-0.5), *([fake] * 8),
                       1 << 30, None)
    assert rc == api.ERR_INVALID_ARG


def test_binding_requires_cuda_tensors(L):
    import torch
    with pytest.raises((ValueError, TypeError)):
        api.verify_greedy(torch.zeros(1, 2, 8), torch.zeros(1, 2, dtype=torch.int64))


def test_attention_dims_checked_on_host(L):
    ok = api.AttnDims(2, 16, 16, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 0)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(ok)) > api.WS_COUNTER_BYTES
    for bad, word in ((api.AttnDims(2, 16, 16, 30, 8, 128, 16, 64, 256, 1024, api.BF16, 0), "multiple of Hkv"),
                      (api.AttnDims(2, 16, 16, 32, 8, 128, 16, 64, 256, 1025, api.BF16, 0), "max_ctx"),
                      (api.AttnDims(2, 16, 16, 32, 8, 128, 16, 64, 256, 1024, 3, 0), "dtype"),
                      (api.AttnDims(0, 16, 16, 32, 8, 128, 16, 64, 256, 1024, api.BF16, 0), "dims")):
        assert L.dflash_block_attn_workspace_size(ctypes.byref(bad)) == 0
        assert word in api.last_error(), api.last_error()
    wide = api.AttnDims(2, 16, 16, 32, 8, 512, 16, 64, 256, 1024, api.BF16, 0)
    assert L.dflash_block_attn_workspace_size(ctypes.byref(wide)) == 0 and "D=512" in api.last_error()
    # a call with a missing pointer fails before anything is launched
    need = L.dflash_block_attn_workspace_size(ctypes.byref(ok))
    fake = _p(0x10000)
    rc = L.dflash_block_attn(ctypes.byref(ok), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.088),
                             fake, fake, need, None)
    assert rc == api.ERR_INVALID_ARG and "NULL" in api.last_error()
    wide_rc = L.dflash_block_attn(ctypes.byref(wide), *([fake] * 7), ctypes.c_float(0.1), fake, fake, need, None)
    assert wide_rc == api.ERR_UNSUPPORTED


def test_materialize_dims_and_arguments_checked_on_host(L):
    ok = api.CtxKvDims(64, 16, 5, 4096, 5, 8, 128, 16, 640, 40960, api.BF16)
    need = L.dflash_materialize_workspace_size(ctypes.byref(ok))
    assert need > api.WS_COUNTER_BYTES
    for bad, word, code in ((api.CtxKvDims(64, 16, 5, 4096, 5, 8, 127, 16, 640, 40960, api.BF16), "even", None),
                            (api.CtxKvDims(64, 16, 5, 4096, 17, 8, 128, 16, 640, 40960, api.BF16), "L=17", None),
                            (api.CtxKvDims(64, 16, 5, 4100, 5, 8, 128, 16, 640, 40960, api.BF16), "16 bytes", None),
                            (api.CtxKvDims(64, 2000, 5, 4096, 5, 8, 128, 16, 640, 40960, api.BF16), "65535", None)):
        assert L.dflash_materialize_workspace_size(ctypes.byref(bad)) == 0
        assert word in api.last_error(), api.last_error()
    fake = _p(0x10000)
    pools = (ctypes.c_void_p * 5)(*([0x10000] * 5))
    pp = ctypes.cast(pools, ctypes.c_void_p)
    eps, theta = ctypes.c_float(1e-6), ctypes.c_float(5e5)
    # new_len aliasing start_pos would read and write the same array
    rc = L.dflash_materialize_ctx_kv(ctypes.byref(ok), fake, fake, _p(0x20000), fake, None, fake, None, eps, theta,
                                     pp, pp, fake, _p(0x20000), fake, need, None)
    assert rc == api.ERR_INVALID_ARG and "alias" in api.last_error()
    rc = L.dflash_materialize_ctx_kv(ctypes.byref(ok), fake, fake, fake, fake, None, fake, None, eps,
                                     ctypes.c_float(-1.0), pp, pp, fake, None, fake, need, None)
    assert rc == api.ERR_INVALID_ARG and "rope_theta" in api.last_error()
    rc = L.dflash_materialize_ctx_kv(ctypes.byref(ok), None, fake, fake, fake, None, fake, None, eps, theta,
                                     pp, pp, fake, None, fake, need, None)
    assert rc == api.ERR_INVALID_ARG and "NULL" in api.last_error()
    holes = (ctypes.c_void_p * 5)(0x10000, 0x10000, None, 0x10000, 0x10000)
    rc = L.dflash_materialize_ctx_kv(ctypes.byref(ok), fake, fake, fake, fake, None, fake, None, eps, theta,
                                     ctypes.cast(holes, ctypes.c_void_p), pp, fake, None, fake, need, None)
    assert rc == api.ERR_INVALID_ARG and "layer 2" in api.last_error()


def test_wait_limit_is_settable_and_zero_restores_default(L):
    default = L.dflash_wait_limit_ns()
    assert default == 2_000_000_000
    assert L.dflash_set_wait_limit_ns(5000) == 0
    assert L.dflash_wait_limit_ns() == 5000
    assert L.dflash_set_wait_limit_ns(0) == 0
    assert L.dflash_wait_limit_ns() == default


def test_error_word_offset_matches_header():
    hdr = open(os.path.join(ROOT, "include", "dflash.h")).read()
    assert "#define DFLASH_WS_ERROR_WORD_OFFSET (DFLASH_WS_COUNTER_BYTES - 4)" in hdr
    assert api.WS_ERROR_WORD_OFFSET == api.WS_COUNTER_BYTES - 4
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"DFLASH_DEVERR_([A-Z_]+) = (\d+)", hdr)}
    assert codes == {"BAD_PAGE": 100, "BAD_N_DRAFT": 101, "BAD_CTX_LEN": 102, "BAD_COMMIT_LEN": 103,
                     "BAD_POSITION": 104}
    for name, value in codes.items():
        assert getattr(api, "DEVERR_" + name) == value, name


def test_debug_library_builds_and_exports_every_symbol(L):
    """The DFLASH_DEBUG build of the same sources (kernels that also record
    clamped inputs in the error word) links and exports the whole ABI."""
    path = build.build(debug=True)
    assert path.endswith("libdflash_debug.so") and path != api.LIB_PATH
    D = ctypes.CDLL(path)
    missing = [n for n in sorted(_declared_functions()) if not hasattr(D, n)]
    assert not missing, missing
    assert api.select_library(debug=True) == path
    try:
        assert api.lib().dflash_wait_limit_ns() > 0
    finally:
        api.select_library(debug=False)
    assert api.LIB_PATH.endswith("libdflash.so")


def _attn_partition_slots(ctx, n_groups, TK, page_size, max_ctx, floor=8, grid=152, pt_max=512):
    """The split pieces of the attention kernel's static partition and the
    partial slot each one writes (two per range: 2v for the piece starting
    range v, 2v + 1 for a piece starting inside it), restated on the host."""
    nt = [(min(max(c, 0), max_ctx) + TK - 1) // TK + 1 for c in ctx]
    cum = [0]
    for x in nt:
        cum.append(cum[-1] + x)
    N = n_groups * cum[-1]
    window = (pt_max - 1) * page_size // TK
    share = min(window, max(floor, -(-N // grid)))
    slots = []
    for b, ntb in enumerate(nt):
        for g in range(n_groups):
            base = n_groups * cum[b] + g * ntb
            nsplit = (base + ntb - 1) // share - base // share + 1
            if nsplit < 2:
                continue
            for sp in range(nsplit):
                start = base if sp == 0 else (base // share + sp) * share
                slots.append(2 * (start // share) + (1 if start % share else 0))
    return slots


@pytest.mark.parametrize("seed", range(6))
def test_attention_workspace_holds_every_split_partial(L, seed):
    # random batches, including the adversarial one (a single long context among
    # empty ones, the smallest ranges): the pieces' slots are distinct and the
    # workspace the library sizes from the dims alone holds all of them
    import random
    rng = random.Random(seed)
    for _ in range(40):
        B = rng.choice([1, 2, 7, 19, 64, 200, 1024])
        n_q = rng.choice([4, 7, 10, 16])
        Hkv = rng.choice([1, 2, 3, 4, 8])
        Hq = Hkv * rng.choice([1, 2, 4])
        page = rng.choice([8, 16, 32, 64])
        max_ctx = rng.choice([0, 1, 100, 2048, 8192, 40000])
        n_kv = n_q
        ctx = [rng.randint(0, max_ctx) for _ in range(B)]
        if rng.random() < 0.3:
            ctx = [max_ctx] + [0] * (B - 1)
        G = Hq // Hkv
        hpi = 2 if (Hkv % 2 == 0 and 2 * n_q * G <= 128 and page >= 16 and n_kv <= 32) else 1
        Mi, n_groups, TK = hpi * n_q * G, Hkv // hpi, 64 // hpi
        slots = _attn_partition_slots(ctx, n_groups, TK, page, max_ctx)
        assert len(slots) == len(set(slots))
        max_pages = max(1, -(-max_ctx // page))
        d = api.AttnDims(B, n_q, n_kv, Hq, Hkv, 128, page, max_pages, B * max_pages, max_ctx, api.BF16, 0)
        ws = L.dflash_block_attn_workspace_size(ctypes.byref(d))
        assert ws > api.WS_COUNTER_BYTES, api.last_error()
        # fp32 O rows and (max, sum) pairs per slot, plus the plan words and at
        # most three 256-byte alignment pads
        per_slot = Mi * 128 * 4 + Mi * 8
        n_slots_min = (ws - api.WS_COUNTER_BYTES - (B + 2) * 4 - 3 * 256) // per_slot
        assert not slots or max(slots) < n_slots_min, (B, n_q, Hq, Hkv, page, max_ctx, max(slots), n_slots_min)
