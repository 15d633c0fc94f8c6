"""Gated delta rule over the verify chain on the GPU, against the oracle.

Tolerance (fp32 kernel vs double oracle, states of order one): each token's
dot products over 128 key components carry about sqrt(128) * 6e-8 ~ 1e-6 of
rounding, and at most 8 tokens are chained, so outputs and checkpoints must
agree to max-abs 1e-4 (relative to max(1, |oracle|)) and rel-L2 1e-5. The
pooled and contiguous forms run the same arithmetic and must agree bit for
bit.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAX_ABS = 1e-4
REL_L2 = 1e-5
FIELDS = ("q", "k", "v", "g", "beta")


def _close(got, ref):
    got = got.cpu().numpy() if torch.is_tensor(got) else got
    scale = max(1.0, float(np.abs(ref).max()))
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert err.max() <= MAX_ABS * scale, f"max-abs {err.max():.3e}"
    rel = np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2, f"rel-L2 {rel:.3e}"


def _gpu(sv, x, l, state=None, W=None, alignment=0):
    q, k, v, g, beta = (x[n][l] for n in FIELDS)
    B, R, H, dk = q.shape
    dv = v.shape[3]
    W = W or R
    snaps = torch.zeros((B, W, H, dv, dk), device=DEV)
    out = torch.empty((B, R, H, dv), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_gdn_verify(q, k, v, g, beta, x["state"][l] if state is None else state, snaps, out, x["scale"],
                       alignment, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return snaps, out


def _oracle(oracle_mod, x, l, rows=slice(None), state=None, W=None, alignment=0):
    arrays = [x[n][l][rows].cpu().numpy() for n in FIELDS]
    s0 = (x["state"][l] if state is None else state)[rows].cpu().numpy()
    snaps, out, rc = oracle_mod.gdn_verify(*arrays, s0, scale=x["scale"], num_slots=W or 0, alignment=alignment)
    assert rc == 0
    return snaps, out


def test_gdn_tiny_matches_oracle(sv, oracle_mod):
    """16 x 16 states (the shared-memory kernel), 4 rows, 2 heads, 4 tokens."""
    x = wl.make_gdn_verify_inputs(wl.WORKLOADS["tiny"], device=DEV)
    snaps, out = _gpu(sv, x, 0)
    ref_s, ref_o = _oracle(oracle_mod, x, 0)
    _close(snaps, ref_s)
    _close(out, ref_o)


@pytest.mark.parametrize("R", [1, 4, 8])
@pytest.mark.parametrize("alignment", [0, 1])
def test_gdn_register_kernel_matches_oracle(sv, oracle_mod, R, alignment):
    """128 x 128 states (register-resident kernel), windows two slots wider than the chain."""
    w = wl.WORKLOADS["hybrid_gdn"].replace(batch=3, k_draft=R - 1, gdn_heads=4)
    x = wl.make_gdn_verify_inputs(w, device=DEV, seed=50 + R)
    snaps, out = _gpu(sv, x, 0, W=R + 2, alignment=alignment)
    ref_s, ref_o = _oracle(oracle_mod, x, 0, W=R + 2, alignment=alignment)
    _close(snaps, ref_s)
    _close(out, ref_o)


@pytest.mark.parametrize("dk,dv", [(64, 32), (128, 64), (32, 128)])
def test_gdn_other_state_sizes(sv, oracle_mod, dk, dv):
    w = wl.WORKLOADS["hybrid_gdn"].replace(batch=2, gdn_heads=3, gdn_dk=dk, gdn_dv=dv)
    x = wl.make_gdn_verify_inputs(w, device=DEV, seed=dk + dv)
    snaps, out = _gpu(sv, x, 0)
    ref_s, ref_o = _oracle(oracle_mod, x, 0)
    _close(snaps, ref_s)
    _close(out, ref_o)


def test_gdn_full_hybrid_layer_sampled_rows(sv, oracle_mod):
    """One layer at the hybrid workload's size (64 rows x 32 heads, 128 x 128,
    4 tokens); the oracle recomputes three rows, all heads."""
    w = wl.WORKLOADS["hybrid_gdn"]
    x = wl.make_gdn_verify_inputs(w, device=DEV)
    snaps, out = _gpu(sv, x, 0)
    rows = [0, 17, w.batch - 1]
    ref_s, ref_o = _oracle(oracle_mod, x, 0, rows=rows)
    _close(snaps[rows], ref_s)
    _close(out[rows], ref_o)
    assert torch.isfinite(snaps).all() and torch.isfinite(out).all()


def test_gdn_pooled_steps_with_zero_copy_commit(sv, oracle_mod):
    """Two verify steps over a state pool with the zero-copy commit between them
    (two layers, last-aligned windows one slot wider than the chain). The pooled
    checkpoints equal the contiguous ones bit for bit, and the second step, which
    starts from the rows the commit staged, equals a contiguous step started from
    the copying commit's states; it also matches the oracle."""
    w = wl.WORKLOADS["hybrid_gdn"].replace(batch=5, gdn_heads=4)
    L, B, R, H, D = 2, w.batch, w.rows, w.gdn_heads, w.gdn_dk
    W, E = R + 1, H * D * D
    x1 = wl.make_gdn_verify_inputs(w, device=DEV, seed=81, layers=L)
    x2 = wl.make_gdn_verify_inputs(w, device=DEV, seed=82, layers=L)
    rng = np.random.default_rng(83)
    perm = rng.permutation(L * B * (W + 1)).astype(np.int32)
    live_row = torch.tensor(perm[:L * B].reshape(L, B), device=DEV)
    ckpt_rows = torch.tensor(perm[L * B:].reshape(L, B, W), device=DEV)
    pool = torch.zeros((L * B * (W + 1), E), device=DEV)
    pool[live_row.long()] = x1["state"].view(L, B, E)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    alen = torch.tensor(rng.integers(0, R, B).astype(np.int32), device=DEV)
    contiguous_live = []
    for l in range(L):  # step 1
        out = torch.empty((B, R, H, D), device=DEV)
        sv.spec_gdn_verify_pooled(*(x1[n][l] for n in FIELDS), pool, live_row[l], ckpt_rows[l], out, x1["scale"],
                                  sv.ALIGN_LAST, dev_err=err)
        snaps, out_c = _gpu(sv, x1, l, W=W, alignment=sv.ALIGN_LAST)
        torch.cuda.synchronize()
        assert torch.equal(out, out_c)
        assert torch.equal(pool[ckpt_rows[l].long()], snaps.view(B, W, E))
        live = x1["state"][l].view(B, E).clone()
        sv.spec_commit_state_aligned(snaps.view(1, B, W, E), alen, live.view(1, B, E), R, sv.ALIGN_LAST)
        contiguous_live.append(live.view(B, H, D, D))
    sv.spec_commit_select(alen, live_row, ckpt_rows, R, sv.ALIGN_LAST, dev_err=err)
    for l in range(L):  # step 2 from the staged rows
        out = torch.empty((B, R, H, D), device=DEV)
        sv.spec_gdn_verify_pooled(*(x2[n][l] for n in FIELDS), pool, live_row[l], ckpt_rows[l], out, x2["scale"],
                                  sv.ALIGN_LAST, dev_err=err)
        snaps, out_c = _gpu(sv, x2, l, state=contiguous_live[l], W=W, alignment=sv.ALIGN_LAST)
        torch.cuda.synchronize()
        assert torch.equal(out, out_c)
        assert torch.equal(pool[ckpt_rows[l].long()], snaps.view(B, W, E))
        ref_s, ref_o = _oracle(oracle_mod, x2, l, state=contiguous_live[l], W=W, alignment=sv.ALIGN_LAST)
        _close(snaps, ref_s)
        _close(out, ref_o)
    assert int(err.item()) == 0


def test_gdn_pooled_bad_row_is_flagged(sv):
    w = wl.WORKLOADS["hybrid_gdn"].replace(batch=3, gdn_heads=2)
    B, R, H, D = w.batch, w.rows, w.gdn_heads, w.gdn_dk
    x = wl.make_gdn_verify_inputs(w, device=DEV, seed=90)
    P = B * (R + 1)
    pool = torch.randn((P, H * D * D), device=DEV)
    live_row = torch.arange(B, dtype=torch.int32, device=DEV) * (R + 1)
    ckpt_rows = (live_row.view(B, 1) + 1 + torch.arange(R, dtype=torch.int32, device=DEV)).contiguous()
    ckpt_rows[1, 2] = P  # outside the pool
    before = pool.clone()
    out = torch.full((B, R, H, D), 7.0, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_gdn_verify_pooled(*(x[n][0] for n in FIELDS), pool, live_row, ckpt_rows, out, x["scale"],
                              dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & sv.DEVERR["pool_row"]
    assert torch.all(out[1] == 0)
    assert torch.equal(pool[1 * (R + 1):2 * (R + 1)], before[1 * (R + 1):2 * (R + 1)])
    assert not torch.equal(pool[:R + 1], before[:R + 1])  # the other rows ran


def test_gdn_rejects_bad_arguments(sv):
    w = wl.WORKLOADS["tiny"]
    x = wl.make_gdn_verify_inputs(w, device=DEV)
    args = [x[n][0] for n in FIELDS]
    B, R, H, dk = args[0].shape
    snaps = torch.zeros((B, R - 1, H, dk, dk), device=DEV)  # window shorter than the chain
    out = torch.empty((B, R, H, dk), device=DEV)
    with pytest.raises(RuntimeError):
        sv.spec_gdn_verify(*args, x["state"][0], snaps, out, x["scale"])
    snaps = torch.zeros((B, R, H, dk, dk), device=DEV)
    with pytest.raises(RuntimeError):
        sv.spec_gdn_verify(*args, x["state"][0], snaps, out, x["scale"], alignment=3)
    with pytest.raises(ValueError):
        sv.spec_gdn_verify(*args, x["state"][0], snaps, out[:, :1], x["scale"])
