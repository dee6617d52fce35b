"""The five synthetic workloads of the DFlash hot path, as plain shape records.

Nothing here computes anything of the method; it only names sizes, dtypes and
the distribution parameters that ``synth`` draws inputs from.

Sources (page titles and sections of the DFlash material):
  * DFlash page, "KV injection" (fusion equation, K/V projection equation,
    attention equation) and "Draft model architecture" (5 draft layers).
  * SGLang DFlash engineering page, section 3 (block of 10, greedy rule) and
    section 4.1 (``dflash_config``: mask id 128002, target_layer_ids
    [1, 8, 15, 22, 29] for the Llama-3.1-8B draft).
  * Speculative-decoding page, section 3 (min(1, p/q) rule, residual resample).
  * DLoop page, "Mechanism 1" (gate c_s >= g with g = -0.5) and the looped
    verify of S blocks of k tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                  # "f32" or "bf16": the I/O type of every call
    B: int                      # sequences in the batch
    d: int                      # d_model of target and draft
    m: int                      # captured target layers
    L: int                      # draft layers
    Hq: int
    Hkv: int
    D: int
    k: int                      # query rows of one draft block
    n_draft: int                # drafted tokens per stage that the verify checks
    V: int                      # vocabulary
    ctx_lo: int                 # committed context length range (inclusive)
    ctx_hi: int
    page_size: int = 16
    n_greedy: int = 0           # sequences [0, n_greedy) use the greedy rule
    temperature: float = 1.0
    sigma: float = 2.0          # target logits = draft logits + N(0, sigma^2)
    hidden_std: float = 1.0     # captured hidden ~ N(0, hidden_std^2)
    weight_std: Optional[float] = None   # None: N(0, 1/fan_in)
    draft_peak: Tuple[float, float] = (8.0, 24.0)   # U[lo, hi] offset on one token per draft row
    draft_base_std: float = 1.0            # draft logits ~ N(0, std^2) + peak
    peak_per_sequence: bool = False        # DLoop: one confidence offset per sequence
    rope_theta: float = 0.0     # 0 disables RoPE on the materialised K
    k_norm: bool = False        # RMSNorm over head_dim on the materialised K
    rms_eps: float = 1e-6
    target_layer_ids: Tuple[int, ...] = ()
    mask_token_id: int = -1
    stages: int = 1             # DLoop: maximum draft stages S
    gate_g: float = -0.5        # DLoop gate threshold
    sigma_sweep: Tuple[float, ...] = field(default_factory=tuple)

    @property
    def n_sampled(self) -> int:
        return self.B - self.n_greedy

    @property
    def n_max(self) -> int:
        """Maximum drafts per sequence that one verify checks (S * n_draft)."""
        return self.stages * self.n_draft

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def kv_out(self) -> int:
        """Columns of the fused K/V projection: L * 2 * Hkv * D."""
        return self.L * 2 * self.Hkv * self.D


# Tiny fp32 instance: every call at kB scale, parity only.
TINY_F32 = Workload(
    name="tiny_f32_b1_d64_k4_v1000", dtype="f32", B=1, d=64, m=5, L=1,
    Hq=4, Hkv=2, D=16, k=4, n_draft=3, V=1000, ctx_lo=32, ctx_hi=32,
    n_greedy=1, temperature=1.0, sigma=1.5, hidden_std=1.0, weight_std=None,
    rope_theta=10000.0, k_norm=True)

# Llama-3.1-8B shape, one sequence, block 10 (anchor + 9 MASK), greedy verify.
LLAMA8B_B1 = Workload(
    name="llama8b_b1_k10_ctx2048", dtype="bf16", B=1, d=4096, m=5, L=5,
    Hq=32, Hkv=8, D=128, k=10, n_draft=9, V=128256, ctx_lo=2048, ctx_hi=2048,
    n_greedy=1, sigma=2.0, hidden_std=16.0 / 64.0, weight_std=0.02,
    rope_theta=500000.0, k_norm=True, target_layer_ids=(1, 8, 15, 22, 29),
    mask_token_id=128002)

# Qwen3-4B shape, batch 8, block 16, temperature-1 sampled verify.
QWEN3_4B_B8 = Workload(
    name="qwen3_4b_b8_k16_ctx1024", dtype="bf16", B=8, d=2560, m=5, L=5,
    Hq=32, Hkv=8, D=128, k=16, n_draft=15, V=151936, ctx_lo=1024, ctx_hi=1024,
    n_greedy=0, sigma=2.0, hidden_std=16.0 / 2560 ** 0.5, weight_std=0.02,
    rope_theta=1000000.0, k_norm=True, target_layer_ids=(1, 9, 17, 25, 33),
    sigma_sweep=(0.5, 2.0, 4.0))

# Batched serving step, Llama-3.1-8B shape: the throughput workload.
LLAMA8B_B64 = Workload(
    name="llama8b_b64_k16_ctx512-8192_paged16_mixed", dtype="bf16", B=64, d=4096,
    m=5, L=5, Hq=32, Hkv=8, D=128, k=16, n_draft=15, V=128256,
    ctx_lo=512, ctx_hi=8192, n_greedy=32, sigma=2.0, hidden_std=16.0 / 64.0,
    weight_std=0.02, rope_theta=500000.0, k_norm=True,
    target_layer_ids=(1, 8, 15, 22, 29), mask_token_id=128002)

# DLoop looped step, Qwen3-4B shape: up to 4 stages of 7 drafted tokens.
DLOOP_QWEN3_4B = Workload(
    name="dloop_qwen3_4b_b32_k7_s4", dtype="bf16", B=32, d=2560, m=5, L=5,
    Hq=32, Hkv=8, D=128, k=8, n_draft=7, V=151936, ctx_lo=1024, ctx_hi=1024,
    n_greedy=0, sigma=2.0, hidden_std=16.0 / 2560 ** 0.5, weight_std=0.02,
    draft_peak=(8.0, 32.0), draft_base_std=3.0, peak_per_sequence=True,
    rope_theta=1000000.0, k_norm=True, target_layer_ids=(1, 9, 17, 25, 33),
    stages=4, gate_g=-0.5)

ALL = (TINY_F32, LLAMA8B_B1, QWEN3_4B_B8, LLAMA8B_B64, DLOOP_QWEN3_4B)
BY_NAME = {w.name: w for w in ALL}
