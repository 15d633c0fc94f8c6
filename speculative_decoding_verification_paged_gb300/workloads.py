"""Seeded synthetic inputs for the verify step.

This module only draws inputs: shapes, random values and their layout. It holds
none of the verify step's arithmetic, so the CUDA path and the CPU oracle can
both be fed from it without sharing any computation.

The named workloads follow the pages' serving setups: an EAGLE3 chain draft of
3 tokens on a Llama-3.1-8B-shaped target with max_batch_size 128 (lmdeploy PR
#3945, "Examples"), and MTP self-speculation on a hybrid gated-delta-net +
attention model with 48 linear-attention layers and max_draft_tokens=3
(onnxruntime-genai PR #2457, Qwen3.8-27B notes). Sizes, value distributions and
mixes are fixed per workload below; nothing is read from a dataset.

Recipe (all draws from one torch.Generator seeded with `seed`, in this order):
ctx_lens, block-table permutation, q, K cache, V cache, target logits, draft
noise, per-row mode, per-row temperature, draft tokens, GDN snapshots.
  * q, K, V ~ N(0,1) rounded to bf16; cache layout [num_blocks, bs, Hkv, D];
    physical blocks are a random permutation (plus a few spare blocks), unused
    block-table entries are -1.
  * target logits ~ N(0, sigma^2) fp32; draft logits = target + N(0, noise^2);
    draft_probs = softmax(draft / T) per row (the drafter samples at the same
    temperature); sampling rows draw their draft tokens from draft_probs,
    greedy rows take argmax(draft) unless the workload says drafts are sampled.
  * GDN snapshots ~ N(0,1) fp32 [L, B, S=k+1, H*dk*dv].
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    ctx_lens: Optional[tuple] = None      # explicit lengths, else uniform in ctx_range
    ctx_range: Optional[tuple] = None     # inclusive (lo, hi)
    block_size: int = 64
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    k_draft: int = 3
    vocab: int = 128256
    logit_sigma: float = 3.0
    noise_sigma: float = 1.5
    mode: str = "sample"                  # "sample" | "greedy" | "mixed"
    temperature: tuple = (1.0, 1.0)       # uniform in [lo, hi] per row
    greedy_drafts: str = "argmax"         # "argmax" | "sampled"
    gdn_layers: int = 0                   # 0: no recurrent-state commit
    gdn_heads: int = 0
    gdn_dk: int = 0
    gdn_dv: int = 0
    seed: int = 0
    spare_blocks: int = 3

    @property
    def rows(self) -> int:
        return self.k_draft + 1

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_ctx(self) -> int:
        return max(self.ctx_lens) if self.ctx_lens else self.ctx_range[1]

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_ctx // self.block_size)

    @property
    def state_elems(self) -> int:
        return self.gdn_heads * self.gdn_dk * self.gdn_dv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 4 sequences, tiny heads and vocab: the case the oracle checks in full.
    "tiny": Workload(
        name="tiny", batch=4, ctx_lens=(17, 64, 100, 255), block_size=16, num_q_heads=4,
        num_kv_heads=1, head_dim=64, k_draft=3, vocab=1000, logit_sigma=2.0, noise_sigma=1.0,
        mode="sample", temperature=(1.0, 1.0), greedy_drafts="sampled", gdn_layers=1,
        gdn_heads=2, gdn_dk=16, gdn_dv=16, seed=0),
    # Llama-3.1-8B-shaped target, EAGLE3 chain of 3 drafts, one attention layer.
    "llama8b_eagle3": Workload(
        name="llama8b_eagle3", batch=32, ctx_lens=(2048,) * 32, block_size=64, num_q_heads=32,
        num_kv_heads=8, head_dim=128, k_draft=3, vocab=128256, logit_sigma=3.0,
        noise_sigma=1.5, mode="sample", temperature=(1.0, 1.0), seed=1),
    # The same step with the draft noise calibrated so that about 70% of drafts
    # are accepted, the rate the MTP validation runs report (the literal noise
    # of 1.5 gives about 46%).
    "llama8b_eagle3_cal": Workload(
        name="llama8b_eagle3_cal", batch=32, ctx_lens=(2048,) * 32, block_size=64, num_q_heads=32,
        num_kv_heads=8, head_dim=128, k_draft=3, vocab=128256, logit_sigma=3.0,
        noise_sigma=0.75, mode="sample", temperature=(1.0, 1.0), seed=1),
    # A full serving batch (max_batch_size 128) with ragged contexts and mixed rows.
    "serving128": Workload(
        name="serving128", batch=128, ctx_range=(512, 8192), block_size=64, num_q_heads=32,
        num_kv_heads=8, head_dim=128, k_draft=3, vocab=128256, mode="mixed",
        temperature=(0.5, 1.2), seed=2),
    # Hybrid gated-delta-net + attention MTP verify: one full-attention layer and
    # the state commit of 48 linear layers.
    "hybrid_gdn": Workload(
        name="hybrid_gdn", batch=64, ctx_range=(1024, 16384), block_size=64, num_q_heads=24,
        num_kv_heads=4, head_dim=256, k_draft=3, vocab=248320, mode="sample",
        temperature=(1.0, 1.0), gdn_layers=48, gdn_heads=32, gdn_dk=128, gdn_dv=128, seed=3),
    # Long contexts, 7 drafts, split-KV.
    "longctx": Workload(
        name="longctx", batch=8, ctx_range=(32768, 131072), block_size=128, num_q_heads=64,
        num_kv_heads=8, head_dim=128, k_draft=7, vocab=128256, mode="sample",
        temperature=(0.8, 0.8), seed=4),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_attention_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """q, paged K/V cache, block table and context lengths for workload `w`."""
    seed = w.seed if seed is None else seed
    g = _gen(device, seed)
    B, R, bs = w.batch, w.rows, w.block_size
    if w.ctx_lens is not None:
        assert len(w.ctx_lens) == B
        ctx = torch.tensor(w.ctx_lens, dtype=torch.int32)
        torch.randint(0, 2, (1,), generator=g, device=device)  # keep the draw order fixed
    else:
        lo, hi = w.ctx_range
        ctx = torch.randint(lo, hi + 1, (B,), generator=g, device=device).to("cpu", torch.int32)
    ctx = torch.clamp(ctx, min=R)
    nblk = [-(-int(c) // bs) for c in ctx.tolist()]
    total = sum(nblk)
    num_blocks = total + w.spare_blocks
    perm = torch.randperm(num_blocks, generator=g, device=device).to("cpu", torch.int32)
    max_blocks = w.max_blocks_per_seq
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    q = torch.randn((B, R, Hq, D), generator=g, device=device).to(torch.bfloat16)
    k_cache = torch.randn((num_blocks, bs, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    v_cache = torch.randn((num_blocks, bs, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    return {
        "q": q, "k_cache": k_cache, "v_cache": v_cache,
        "block_table": table.to(device), "ctx_lens": ctx.to(device),
        "num_blocks": num_blocks, "generator": g,
    }


def make_accept_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                       generator: Optional[torch.Generator] = None, mode: Optional[str] = None) -> dict:
    """Target logits, draft tokens/probabilities, per-row mode and temperature."""
    g = generator if generator is not None else _gen(device, (w.seed if seed is None else seed) + 7919)
    mode = w.mode if mode is None else mode
    B, R, k, V = w.batch, w.rows, w.k_draft, w.vocab
    target = torch.randn((B, R, V), generator=g, device=device) * w.logit_sigma
    draft_logits = target[:, :k, :] + torch.randn((B, k, V), generator=g, device=device) * w.noise_sigma
    if mode == "sample":
        modes = torch.ones(B, dtype=torch.int32, device=device)
        torch.rand((B,), generator=g, device=device)
    elif mode == "greedy":
        modes = torch.zeros(B, dtype=torch.int32, device=device)
        torch.rand((B,), generator=g, device=device)
    else:
        modes = (torch.rand((B,), generator=g, device=device) < 0.5).to(torch.int32)
    lo, hi = w.temperature
    temp = (lo + (hi - lo) * torch.rand((B,), generator=g, device=device)).to(torch.float32)
    draft_probs = torch.softmax(draft_logits / temp.view(B, 1, 1), dim=-1).contiguous()
    sampled = torch.multinomial(draft_probs.view(B * k, V), 1, generator=g).view(B, k).to(torch.int32)
    if w.greedy_drafts == "argmax":
        greedy = draft_logits.argmax(dim=-1).to(torch.int32)
        drafts = torch.where(modes.view(B, 1) == 1, sampled, greedy)
    else:
        drafts = sampled
    return {
        "target_logits": target.contiguous(), "draft_tokens": drafts.contiguous(),
        "draft_probs": draft_probs, "mode": modes.contiguous(), "temperature": temp.contiguous(),
        "philox_seed": int(w.seed if seed is None else seed),
    }


def make_gdn_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                    generator: Optional[torch.Generator] = None) -> dict:
    """Per-slot GDN state snapshots [L, B, S, H*dk*dv] and a live-state buffer."""
    g = generator if generator is not None else _gen(device, (w.seed if seed is None else seed) + 104729)
    L, B, S, E = w.gdn_layers, w.batch, w.rows, w.state_elems
    snaps = torch.empty((L, B, S, E), dtype=torch.float32, device=device)
    for l in range(L):  # per layer, to keep the peak allocation at one tensor
        snaps[l] = torch.randn((B, S, E), generator=g, device=device)
    live = torch.zeros((L, B, E), dtype=torch.float32, device=device)
    return {"snapshots": snaps, "live_state": live}


def make_gdn_verify_inputs(w: Workload, device="cpu", seed: Optional[int] = None, layers: int = 1,
                           generator: Optional[torch.Generator] = None) -> dict:
    """Inputs of the gated delta rule over the verify chain, for `layers` layers.

    q, k [layers, B, R, H, dk] are L2-normalised per head (the GatedDeltaNet layer
    normalises them before the recurrence); v ~ N(0, 1); g = log sigmoid(N(0,1) + 3)
    (decay factors near 0.95); beta = sigmoid(N(0, 1)); the live state
    [layers, B, H, dv, dk] ~ N(0, 1). scale = 1/sqrt(dk).
    """
    g = generator if generator is not None else _gen(device, (w.seed if seed is None else seed) + 15485863)
    L, B, R, H, dk, dv = layers, w.batch, w.rows, w.gdn_heads, w.gdn_dk, w.gdn_dv
    q = torch.randn((L, B, R, H, dk), generator=g, device=device)
    k = torch.randn((L, B, R, H, dk), generator=g, device=device)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn((L, B, R, H, dv), generator=g, device=device)
    gate = torch.nn.functional.logsigmoid(torch.randn((L, B, R, H), generator=g, device=device) + 3.0)
    beta = torch.sigmoid(torch.randn((L, B, R, H), generator=g, device=device))
    state = torch.empty((L, B, H, dv, dk), dtype=torch.float32, device=device)
    for l in range(L):
        state[l] = torch.randn((B, H, dv, dk), generator=g, device=device)
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(), "g": gate.contiguous(),
            "beta": beta.contiguous(), "state": state, "scale": 1.0 / float(dk) ** 0.5}


def kv_bytes(ctx_lens, num_kv_heads: int, head_dim: int) -> int:
    """Bytes of K and V (bf16) that the visible tokens occupy."""
    return int(sum(int(c) for c in ctx_lens)) * num_kv_heads * head_dim * 2 * 2


def describe(w: Workload) -> dict:
    return {k: v for k, v in dataclasses.asdict(w).items() if v not in (None, 0)}


def mean_ctx(w: Workload) -> float:
    if w.ctx_lens:
        return sum(w.ctx_lens) / len(w.ctx_lens)
    return (w.ctx_range[0] + w.ctx_range[1]) / 2.0


__all__ = ["Workload", "WORKLOADS", "make_attention_inputs", "make_accept_inputs",
           "make_gdn_inputs", "kv_bytes", "describe", "mean_ctx"]
