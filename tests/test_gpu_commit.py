"""State commit on the GPU: bit-exact against the oracle and, at the hybrid
workload's full size, against the gather the definition states."""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_commit_tiny_matches_oracle(sv, oracle_mod):
    w = wl.WORKLOADS["tiny"]
    g = wl.make_gdn_inputs(w, device=DEV)
    alen = torch.tensor([0, 3, 1, 2], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_commit_state(g["snapshots"], alen, g["live_state"], dev_err=err)
    torch.cuda.synchronize()
    ref = np.zeros(tuple(g["live_state"].shape), np.float32)
    oracle_mod.commit_state(g["snapshots"].cpu().numpy(), alen.cpu().numpy(), ref)
    assert int(err.item()) == 0 and np.array_equal(g["live_state"].cpu().numpy(), ref)


def test_commit_full_hybrid_workload_bit_exact(sv, oracle_mod):
    w = wl.WORKLOADS["hybrid_gdn"]
    g = wl.make_gdn_inputs(w, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(1)
    alen = torch.randint(0, w.rows, (w.batch,), generator=gen, device=DEV, dtype=torch.int32)
    alen[0], alen[1] = 0, w.k_draft  # both ends
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_commit_state(g["snapshots"], alen, g["live_state"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = torch.arange(w.batch, device=DEV)
    for l in range(w.gdn_layers):
        assert torch.equal(g["live_state"][l], g["snapshots"][l, rows, alen.long()])
    # one (layer, row) through the oracle as well
    snap = g["snapshots"][7:8, 5:6].cpu().numpy()
    ref = np.zeros((1, 1, w.state_elems), np.float32)
    oracle_mod.commit_state(snap, alen[5:6].cpu().numpy(), ref)
    assert np.array_equal(g["live_state"][7:8, 5:6].cpu().numpy(), ref)


def test_commit_unaligned_size_and_invalid_row(sv):
    L, B, S, E = 3, 5, 4, 1001
    snaps = torch.randn((L, B, S, E), device=DEV)
    live = torch.full((L, B, E), 7.0, device=DEV)
    alen = torch.tensor([0, 4, 2, -1, 3], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_commit_state(snaps, alen, live, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & sv.DEVERR["accept_len"]
    for b in range(B):
        if 0 <= alen[b] < S:
            assert torch.equal(live[:, b], snaps[:, b, alen[b]])
        else:
            assert torch.all(live[:, b] == 7.0)


@pytest.mark.parametrize("alignment", [0, 1], ids=["token", "last"])
@pytest.mark.parametrize("E", [4096, 1001], ids=["vec", "scalar"])
def test_commit_aligned_window_matches_oracle(sv, oracle_mod, alignment, E):
    """A checkpoint window wider than the step (W = 7 slots, n = 4 tokens), both
    alignments, vectorised and element-wise copies; a bad accept_len is skipped."""
    rng = np.random.default_rng(40 + alignment)
    L, B, W, n = 3, 9, 7, 4
    snaps = torch.tensor(rng.standard_normal((L, B, W, E)).astype(np.float32), device=DEV)
    alen_np = rng.integers(0, n, B).astype(np.int32)
    alen_np[0], alen_np[1], alen_np[2] = 0, n - 1, n  # both ends and one out of range
    alen = torch.tensor(alen_np, device=DEV)
    live = torch.full((L, B, E), 5.0, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_commit_state_aligned(snaps, alen, live, n, alignment, dev_err=err)
    torch.cuda.synchronize()
    ref = np.full((L, B, E), 5.0, np.float32)
    rc = oracle_mod.commit_state_aligned(snaps.cpu().numpy(), alen_np, ref, n, alignment, check=False)
    assert rc != 0 and int(err.item()) & sv.DEVERR["accept_len"]
    assert np.array_equal(live.cpu().numpy(), ref)


def test_commit_aligned_rejects_bad_arguments(sv):
    snaps = torch.zeros((1, 2, 3, 8), device=DEV)
    live = torch.zeros((1, 2, 8), device=DEV)
    alen = torch.zeros(2, dtype=torch.int32, device=DEV)
    for n, alignment in ((4, 0), (0, 1), (2, 5)):
        with pytest.raises(RuntimeError):
            sv.spec_commit_state_aligned(snaps, alen, live, n, alignment)
