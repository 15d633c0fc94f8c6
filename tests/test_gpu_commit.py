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


def _tables(rng, L, B, W):
    perm = rng.permutation(L * B * (W + 1)).astype(np.int32)
    return perm[:L * B].reshape(L, B).copy(), perm[L * B:].reshape(L, B, W).copy()


@pytest.mark.parametrize("alignment", [0, 1])
def test_commit_select_matches_oracle(sv, oracle_mod, alignment):
    """Zero-copy commit on hybrid-sized tables (48 layers x 64 rows, a 6-slot window
    for a 4-token step), both alignments, one out-of-range row: bit-exact tables."""
    rng = np.random.default_rng(60 + alignment)
    L, B, W, n = 48, 64, 6, 4
    live_np, ckpt_np = _tables(rng, L, B, W)
    alen_np = rng.integers(0, n, B).astype(np.int32)
    alen_np[0], alen_np[1], alen_np[2] = 0, n - 1, -1
    live, ckpt = torch.tensor(live_np, device=DEV), torch.tensor(ckpt_np, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_commit_select(torch.tensor(alen_np, device=DEV), live, ckpt, n, alignment, dev_err=err)
    torch.cuda.synchronize()
    rc = oracle_mod.commit_select(alen_np, live_np, ckpt_np, n, alignment, check=False)
    assert rc != 0 and int(err.item()) & sv.DEVERR["accept_len"]
    assert np.array_equal(live.cpu().numpy(), live_np) and np.array_equal(ckpt.cpu().numpy(), ckpt_np)


def test_commit_select_stages_what_the_copy_commits(sv):
    """On a device pool, after the exchange the live rows hold exactly the states the
    copying commit writes, for every (layer, row)."""
    rng = np.random.default_rng(61)
    L, B, W, n, E = 4, 16, 5, 4, 1000
    gen = torch.Generator(device=DEV).manual_seed(61)
    pool = torch.randn((L * B * (W + 1), E), generator=gen, device=DEV)
    live_np, ckpt_np = _tables(rng, L, B, W)
    live, ckpt = torch.tensor(live_np, device=DEV), torch.tensor(ckpt_np, device=DEV)
    alen = torch.tensor(rng.integers(0, n, B).astype(np.int32), device=DEV)
    copied = pool[live.long()].clone()
    sv.spec_commit_state_aligned(pool[ckpt.long()].contiguous(), alen, copied, n, sv.ALIGN_LAST)
    sv.spec_commit_select(alen, live, ckpt, n, sv.ALIGN_LAST)
    torch.cuda.synchronize()
    assert torch.equal(pool[live.long()], copied)
    owned = torch.sort(torch.cat([live.unsqueeze(-1), ckpt], dim=-1), dim=-1).values
    before = np.sort(np.concatenate([live_np[..., None], ckpt_np], axis=-1), axis=-1)
    assert np.array_equal(owned.cpu().numpy(), before)


def test_commit_select_rejects_bad_arguments(sv):
    alen = torch.zeros(2, dtype=torch.int32, device=DEV)
    live = torch.zeros((1, 2), dtype=torch.int32, device=DEV)
    ckpt = torch.zeros((1, 2, 3), dtype=torch.int32, device=DEV)
    for n, alignment in ((4, 0), (0, 1), (2, 5)):
        with pytest.raises(RuntimeError):
            sv.spec_commit_select(alen, live, ckpt, n, alignment)
    with pytest.raises(ValueError):
        sv.spec_commit_select(alen, live, ckpt[:, :1], 2, 0)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_accept_then_select_in_one_graph(sv, oracle_mod, mode):
    """Acceptance and the zero-copy commit captured in one CUDA graph: the commit
    reads accept_len on the device with no host round trip, and each replay
    applies the exchange once more."""
    from helpers import compare_accept

    w = wl.WORKLOADS["llama8b_eagle3"]
    inp = wl.make_accept_inputs(w, device=DEV, mode=mode)
    B, R, V = inp["target_logits"].shape
    L, W, n = 48, R + 2, R
    rng = np.random.default_rng(62)
    live_np, ckpt_np = _tables(rng, L, B, W)
    live, ckpt = torch.tensor(live_np, device=DEV), torch.tensor(ckpt_np, device=DEV)
    toks = torch.empty((B, R), dtype=torch.int32, device=DEV)
    alen = torch.empty((B,), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def accept():
        sv.spec_accept(inp["target_logits"], inp["draft_tokens"], inp["draft_probs"], inp["philox_seed"],
                       inp["mode"], inp["temperature"], toks, alen, dev_err=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        accept()  # first call outside the capture (one-time function attributes)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            accept()
            sv.spec_commit_select(alen, live, ckpt, n, sv.ALIGN_LAST, dev_err=err)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert np.array_equal(live.cpu().numpy(), live_np)  # capture ran nothing
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        a = alen.cpu().numpy()
        oracle_mod.commit_select(a, live_np, ckpt_np, n, 1)
        assert np.array_equal(live.cpu().numpy(), live_np) and np.array_equal(ckpt.cpu().numpy(), ckpt_np)
    rt, ra, margin, gap, rc = oracle_mod.accept(inp["target_logits"].cpu().numpy(), inp["draft_tokens"].cpu().numpy(),
                                                inp["draft_probs"].cpu().numpy(), inp["philox_seed"],
                                                inp["mode"].cpu().numpy(), inp["temperature"].cpu().numpy())
    bad, _ = compare_accept(toks.cpu().numpy(), alen.cpu().numpy(), rt, ra, margin, gap)
    assert rc == 0 and bad == 0
