"""Shared helpers of the test suite: tensor conversion and parity metrics."""

import numpy as np
import torch

ATTN_MAX_ABS = 1e-2      # attention: max-abs error vs the double-precision oracle
ATTN_REL_L2 = 2e-3       # attention: relative L2 error vs the oracle
NEAR_TIE = 1e-5          # sampled decisions: |u - p/q| (or race keys this close, relative) are excused
MAX_EXCUSED_RATE = 1e-4  # ... and must stay below this share of decisions


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def attention_errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    diff = got - ref
    return float(np.abs(diff).max()), float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))


def oracle_attention_for(oracle, a: dict, seqs=None):
    return oracle.verify_attention(bf16_to_bits(a["q"]), bf16_to_bits(a["k_cache"]), bf16_to_bits(a["v_cache"]),
                                   a["block_table"].cpu().numpy(), a["ctx_lens"].cpu().numpy(), seqs=seqs)


def compare_accept(tok, alen, ref_tok, ref_alen, margin, race_gap):
    """Rows must match bit-exactly unless the oracle marks them as a near tie.

    Returns (n_mismatch_unexcused, n_excused_rows)."""
    same = (np.asarray(tok) == ref_tok).all(1) & (np.asarray(alen) == ref_alen)
    excused = (margin < NEAR_TIE) | (race_gap < NEAR_TIE)
    return int(np.sum(~same & ~excused)), int(np.sum(excused))
