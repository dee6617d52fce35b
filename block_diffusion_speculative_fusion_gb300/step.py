"""One DFlash serving step on the GPU, chained through the C ABI.

A step is the hot path of one decode round of the batched workload:
  * block attention of the draft block in each of the L draft layers
    (DFlash page, 块扩散 / KV 注入);
  * verify of the drafted candidates -- greedy for sequences [0, n_greedy),
    the min(1, p/q) rule with residual resample for the rest (SGLang page,
    section 3; speculative-decoding page, section 3);
  * context-KV materialisation of the commit_len = accept_len + 1 rows of
    every sequence into every layer's paged cache (SGLang page, section 4.1),
    which advances each sequence's committed length for the next step.

Everything stays on the device and on one stream; the step makes no host
synchronisation. Inputs that the upstream draft and target models would
produce (queries, block K/V, logits, captured hidden states) come from the
seeded generators in ``synth``.
"""
from __future__ import annotations

import ctypes
from typing import Dict, List, Optional

import torch

from . import api, synth
from .workloads import Workload


class DflashStep:
    def __init__(self, wl: Workload, seed: int = 0, device: str = "cuda:0", headroom_steps: int = 64,
                 pools_on_device: bool = True, pinned_inputs: bool = False, stationary: bool = False):
        """``stationary``: every step starts from the initial context lengths
        (the committed rows of one step are rewritten by the next), so that the
        workload does not drift as steps repeat; otherwise each step starts
        where the previous one left the cache."""
        self.wl = wl
        self.stationary = stationary
        self.dev = torch.device(device)
        dev = self.dev
        dt = synth.io_dtype(wl)
        # ---- paged draft KV cache (persistent state) ----
        ctx_len = synth.ctx_lengths(wl, seed)
        self.ctx0 = ctx_len.clone()
        headroom = wl.k * headroom_steps
        cache = synth.paged_cache(wl, headroom, seed, device=str(dev) if pools_on_device else "cpu")
        self.k_pools = [t.to(dev) for t in cache.k_pools]
        self.v_pools = [t.to(dev) for t in cache.v_pools]
        self.page_table = cache.page_table.to(dev)
        self.max_ctx = cache.max_pages * wl.page_size
        self.ctx = [ctx_len.to(dev), torch.empty_like(ctx_len, device=dev)]
        self.ctx_start = ctx_len.to(dev)
        self.cur = 0
        # ---- per-step inputs from the upstream models (host copies kept for e2e) ----
        host: Dict[str, torch.Tensor] = {}
        for layer in range(wl.L):
            for k_, v_ in synth.block_qkv(wl, layer, seed).items():
                host[f"{k_}{layer}"] = v_
        vb = synth.verify_batch(wl, seed, n_max=wl.n_draft)
        host.update(vb)
        # the draft logits are read by the sampled rule only: the step's input is
        # the sampled sub-batch's rows (the greedy sequences' candidates are given)
        host["draft_logits"] = vb["draft_logits"][wl.n_greedy:].contiguous()
        host["hidden"] = synth.captured_hidden(wl, wl.n_draft + 1, seed)
        if pinned_inputs:
            host = {k_: v_.pin_memory() for k_, v_ in host.items()}
        self.host = host
        self.inp = {k_: v_.to(dev) for k_, v_ in host.items()}
        w = synth.ctx_weights(wl, seed)
        self.W_f = w["W_f"].to(dev)
        self.b_f = w["b_f"].to(dev)
        self.W_kv = w["W_kv"].to(dev)
        self.k_norm_w = None if w["k_norm_w"] is None else w["k_norm_w"].to(dev)
        # ---- outputs ----
        B, R = wl.B, wl.n_draft + 1
        self.attn_out = [torch.empty_like(self.inp[f"q{layer}"]) for layer in range(wl.L)]
        self.out = {
            "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
            "bonus": torch.empty(B, dtype=torch.int64, device=dev),
            "commit_len": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, R), dtype=torch.int64, device=dev),
            "flags": torch.zeros(B, dtype=torch.uint8, device=dev),
        }
        ng = wl.n_greedy
        self.out_g = {k_: v_[:ng] for k_, v_ in self.out.items() if k_ != "flags"}
        self.out_s = {k_: v_[ng:] for k_, v_ in self.out.items()}
        # one workspace per call kind (calls run in order on one stream)
        self.ws = {}
        # the greedy and the sampled sub-batches are independent sequences:
        # their verify calls run concurrently, the sampled one (two dependent
        # launches, the longer path) on a forked stream of higher priority, the
        # greedy one with its own workspace (counters must not be shared)
        self.side = torch.cuda.Stream(device=dev, priority=-1)
        self.ev_fork = torch.cuda.Event()
        self.ev_join = torch.cuda.Event()
        self.ws_greedy = None
        if 0 < ng < B:
            d = api.VerifyDims(ng, wl.n_draft, wl.V, api.BF16 if wl.dtype == "bf16" else api.F32)
            need = api.lib().dflash_verify_greedy_workspace_size(ctypes.byref(d))
            self.ws_greedy = torch.zeros(need, dtype=torch.uint8, device=dev)
        self.launches_per_step = 0
        self.events: Optional[List] = None

    # ------------------------------------------------------------------
    def capture(self, n_steps: int, timer=None, after_step=None):
        """One CUDA graph holding ``n_steps`` consecutive steps, in the launch
        form the benchmark times: the verify fork onto the side stream and its
        join are captured with the launches. ``after_step(i)`` may enqueue more
        work after step i (copies of its outputs) inside the graph. Run one
        step eagerly first, so that every workspace exists before capture."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_steps):
                self.step(timer=timer)
                if after_step is not None:
                    after_step(i)
        return g

    def workspaces(self) -> List[torch.Tensor]:
        """The device workspaces this step's calls use."""
        out = [w for (dev, _), w in api._WS.items() if dev == (self.dev.index or 0)]
        if self.ws_greedy is not None:
            out.append(self.ws_greedy)
        return out

    def error_words(self) -> List[int]:
        """Device error words of the step's workspaces (all 0 unless a kernel
        gave up a bounded wait or met a bad page-table entry)."""
        return [api.device_error_word(w) for w in self.workspaces()]

    def reset(self):
        self.ctx[0].copy_(self.ctx0.to(self.dev))
        self.cur = 0

    def ctx_len(self) -> torch.Tensor:
        return self.ctx[self.cur]

    def copy_inputs_from_host(self, inp: Optional[Dict[str, torch.Tensor]] = None):
        """Host -> device copies of one step's inputs (pinned host memory) into
        ``inp`` (default: the step's own input buffers), on the current stream."""
        inp = self.inp if inp is None else inp
        for k_, v_ in inp.items():
            v_.copy_(self.host[k_], non_blocking=True)

    def second_input_set(self) -> Dict[str, torch.Tensor]:
        """A second set of device input buffers, for copying the next step's
        inputs while the current step runs."""
        return {k_: torch.empty_like(v_) for k_, v_ in self.inp.items()}

    def input_bytes(self) -> int:
        return sum(v_.numel() * v_.element_size() for v_ in self.host.values())

    def _ws(self, name: str, slot: int) -> Optional[torch.Tensor]:
        return self.ws.get(name)

    def step(self, timer=None, inp: Optional[Dict[str, torch.Tensor]] = None):
        """Enqueue one step on the current stream, reading the inputs ``inp``
        (default: the step's own input buffers). ``timer(name)`` (optional) is
        called between calls to record per-kernel events."""
        wl = self.wl
        inp = self.inp if inp is None else inp
        if self.stationary:
            cur, nxt = self.ctx_start, self.ctx[1]
        else:
            cur, nxt = self.ctx[self.cur], self.ctx[1 - self.cur]
        launches = 0
        for layer in range(wl.L):
            if timer:
                timer("attn_start")
            api.block_attn(inp[f"q{layer}"], inp[f"k_blk{layer}"], inp[f"v_blk{layer}"], self.k_pools[layer],
                           self.v_pools[layer], self.page_table, cur, max_ctx=self.max_ctx,
                           out=self.attn_out[layer])
            launches += api.last_launch_count()
            if timer:
                timer("attn_end")
        ng = wl.n_greedy
        if timer:
            timer("verify_start")
        concurrent = self.ws_greedy is not None
        main = torch.cuda.current_stream(self.dev)
        if concurrent:
            self.ev_fork.record(main)
            self.side.wait_event(self.ev_fork)
        if ng < wl.B:
            with torch.cuda.stream(self.side if concurrent else main):
                api.verify_sample(inp["target_logits"][ng:], inp["draft_logits"], inp["cand"][ng:],
                                  inp["u_acc"][ng:], inp["u_final"][ng:], wl.temperature, inp["n_draft"][ng:],
                                  out=self.out_s)
            launches += api.last_launch_count()
        if ng > 0:
            api.verify_greedy(inp["target_logits"][:ng], inp["cand"][:ng], inp["n_draft"][:ng], out=self.out_g,
                              ws=self.ws_greedy)
            launches += api.last_launch_count()
        if concurrent:
            self.ev_join.record(self.side)
            main.wait_event(self.ev_join)
        if timer:
            timer("verify_end")
            timer("mat_start")
        api.materialize_ctx_kv(inp["hidden"], self.out["commit_len"], cur, self.W_f, self.b_f, self.W_kv,
                               self.k_norm_w, wl.rms_eps, wl.rope_theta, self.k_pools, self.v_pools,
                               self.page_table, new_len=nxt)
        launches += api.last_launch_count()
        if timer:
            timer("mat_end")
        if not self.stationary:
            self.cur = 1 - self.cur
        self.launches_per_step = launches
