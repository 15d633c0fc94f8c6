"""Verify attention on the GPU against the double-precision oracle (parity gate).

Small cases and the named workloads at their full sizes are checked in full,
every sequence and every output element, from the same device inputs. Tolerances: max-abs <= 1e-2 and relative L2 <=
2e-3 per case. Head dims 128 and 256 have two kernels (tcgen05, the default
from 17 packed rows up, and mma.sync; SPEC_ATTN_KERNEL=tc / =mma forces one);
every case with those head dims runs both, and one case runs the default
choice.
"""

import zlib

import numpy as np
import pytest
import torch

from helpers import ATTN_MAX_ABS, ATTN_REL_L2, attention_errors, oracle_attention_for
from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (name, B, ctx_lens, bs, Hq, Hkv, D, k): every (head_dim, m-tile count) instantiation,
# ragged contexts spanning several 64-key tiles and splits, block sizes 16..128.
SMALL = [
    ("d64_mt1_bs16", 5, (4, 63, 64, 65, 700), 16, 8, 2, 64, 3),
    ("d64_mt2_bs32", 3, (9, 333, 1030), 32, 8, 2, 64, 7),
    ("d64_mt4_bs64", 2, (8, 1500), 64, 16, 2, 64, 7),
    ("d128_mt1_bs64", 4, (100, 2048, 4, 129), 64, 32, 8, 128, 3),
    ("d128_mt2_bs16", 3, (640, 77, 1999), 16, 12, 2, 128, 3),
    ("d128_mt4_bs128", 3, (129, 2000, 9), 128, 16, 2, 128, 7),
    ("d256_mt1_bs64", 3, (1000, 5, 300), 64, 4, 2, 256, 3),
    ("d256_mt2_bs64", 3, (300, 1000, 77), 64, 12, 2, 256, 3),
    ("d256_mt4_bs32", 2, (257, 900), 32, 16, 2, 256, 7),
]


# Head-dim-128 cases aimed at the tcgen05 kernel: 128-key tiles made of 8, 4, 2 or 1
# TMA pieces, contexts just below / at / above tile edges, every packed-row count
# (16, 24 -> 32, 32, 64), k = 1 and k = 7, and batches whose plan pushes the kernel
# to two stages (1600) or back to mma.sync (4096 with 64 rows).
TC_CASES = [
    ("tc_mt1_bs32_edges", 6, (4, 127, 128, 129, 255, 1100), 32, 32, 8, 128, 3),
    ("tc_mt1_k1_bs64", 4, (2, 64, 129, 3000), 64, 8, 1, 128, 1),
    ("tc_mt2_rows24_bs128", 4, (4, 128, 385, 2100), 128, 24, 4, 128, 3),
    ("tc_mt2_k7_bs64", 4, (8, 200, 513, 1500), 64, 16, 4, 128, 7),
    ("tc_mt4_bs16", 3, (5, 300, 1200), 16, 64, 4, 128, 3),
    ("tc_mt4_k7_bs32", 3, (8, 640, 1030), 32, 16, 2, 128, 7),
    # head dim 256: one 128-key stage, O^T in two 128-lane halves
    ("tc_d256_mt1_bs32", 4, (4, 127, 129, 900), 32, 8, 2, 256, 3),
    ("tc_d256_mt2_rows24_bs64", 5, (5, 64, 130, 1000, 2500), 64, 24, 4, 256, 3),
    ("tc_d256_mt2_k7_bs16", 3, (9, 385, 1400), 16, 8, 2, 256, 7),
    ("tc_d256_mt4_bs128", 3, (9, 256, 1500), 128, 16, 2, 256, 7),
]


@pytest.fixture(params=["tc", "mma"])
def attn_kernel(request, monkeypatch):
    monkeypatch.setenv("SPEC_ATTN_KERNEL", request.param)
    return request.param


def _ragged(B, lo, hi, seed):
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=B))


def run_attention(sv, a, w, **kw):
    out = torch.full((w.batch, w.rows, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft, out,
                             dev_err=err, **kw)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("case", SMALL + TC_CASES, ids=[c[0] for c in SMALL + TC_CASES])
def test_attention_small_cases_full_parity(sv, oracle_mod, case, attn_kernel):
    name, B, ctx, bs, Hq, Hkv, D, k = case
    if D == 64 and attn_kernel == "tc":
        pytest.skip("one kernel for this head dim")
    w = wl.Workload(name=name, batch=B, ctx_lens=ctx, block_size=bs, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=D, k_draft=k, seed=zlib.crc32(name.encode()) % 1000)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    ref = oracle_attention_for(oracle_mod, a)
    mx, rel = attention_errors(out.cpu().numpy(), ref)
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


def test_attention_tiny_workload(sv, oracle_mod):
    w = wl.WORKLOADS["tiny"]
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


@pytest.mark.parametrize("name", ["llama8b_eagle3", "serving128", "hybrid_gdn", "longctx"])
def test_attention_full_size_every_sequence(sv, oracle_mod, name, attn_kernel):
    """The named workloads at their full sizes, in the launch configuration the bench
    times: every sequence of the batch against the oracle, element by element, so every
    unit the stream-K plan cuts across CTAs (and merges by log-sum-exp) is compared."""
    w = wl.WORKLOADS[name]
    if w.head_dim == 64 and attn_kernel == "tc":
        pytest.skip("one kernel for this head dim")
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    assert torch.isfinite(out).all()
    ref = oracle_attention_for(oracle_mod, a)
    got = out.cpu().numpy()
    assert ref.shape == got.shape
    mx, rel = attention_errors(got, ref)
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)
    for b in range(w.batch):  # and sequence by sequence, so one bad unit cannot hide in the total
        mx_b, rel_b = attention_errors(got[b], ref[b])
        assert mx_b <= ATTN_MAX_ABS and rel_b <= ATTN_REL_L2, (b, mx_b, rel_b)


@pytest.mark.parametrize("B,Hq,k", [(1600, 32, 3), (4096, 16, 7)], ids=["b1600_mt1", "b4096_mt4"])
def test_attention_large_batch_plans(sv, oracle_mod, attn_kernel, B, Hq, k):
    """Batches whose per-sequence plan fills shared memory: every sequence is checked."""
    w = wl.Workload(name=f"big{B}", batch=B, ctx_lens=_ragged(B, k + 1, 160, B), block_size=16,
                    num_q_heads=Hq, num_kv_heads=2 if Hq == 16 else 8, head_dim=128, k_draft=k, seed=B % 997)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


@pytest.mark.parametrize("B", [8, 16, 40, 48])
@pytest.mark.parametrize("bad_row", [False, True], ids=["uniform", "one_unusable"])
def test_attention_uniform_context_split_plans(sv, oracle_mod, attn_kernel, B, bad_row):
    """Equal context lengths, so every (sequence, kv head) unit has the same tile
    count: 8 kv heads x B sequences = 64 / 128 / 320 / 384 units take, on the
    mma.sync kernel's 304-CTA grid, the even stream-K split, one whole unit per
    CTA, the stream-K split again (whole units would load 1.9x) and two whole
    units per CTA; the tcgen05 kernel's 152-CTA grid gives other cases of the
    same rule. An unusable sequence (context shorter than the chain) must not
    change the plan of the others."""
    w = wl.WORKLOADS["llama8b_eagle3"].replace(batch=B, ctx_lens=(1024,) * B, seed=B + 7 * bad_row)
    a = wl.make_attention_inputs(w, device=DEV)
    if bad_row:
        a["ctx_lens"][B // 3] = 2  # < k + 1: zero rows and an error bit, excluded from the unit lengths
    out, err = run_attention(sv, a, w)
    assert err == (sv.DEVERR["ctx_len"] if bad_row else 0)
    picks = sorted({0, B // 2, B - 1} - ({B // 3} if bad_row else set()))
    ref = oracle_attention_for(oracle_mod, a, seqs=np.array(picks, np.int32))
    mx, rel = attention_errors(out[picks].cpu().numpy(), ref)
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)
    if bad_row:
        assert torch.all(out[B // 3] == 0)


@pytest.mark.parametrize("name", ["longctx", "llama8b_eagle3"])
def test_attention_default_kernel_choice(sv, oracle_mod, monkeypatch, name):
    """No override: the library picks the kernel (tcgen05 for 64 rows, mma.sync for 16)."""
    monkeypatch.delenv("SPEC_ATTN_KERNEL", raising=False)
    w = wl.WORKLOADS[name].replace(batch=3, ctx_lens=(129, 3000, 9), ctx_range=None)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


@pytest.mark.parametrize("name,kind", [("longctx", "tc"), ("llama8b_eagle3", "mma"), ("hybrid_gdn", "tc")])
def test_attention_plan_names_the_kernel_that_runs(sv, monkeypatch, name, kind):
    """spec_verify_attention_plan names the kernel the call runs. The two kernels of
    a head dim round differently, so the default call's output equals, bit for bit,
    that of the kernel the plan names when SPEC_ATTN_KERNEL forces it, and differs
    from the other's."""
    monkeypatch.delenv("SPEC_ATTN_KERNEL", raising=False)
    w = wl.WORKLOADS[name].replace(batch=3, ctx_lens=(129, 3000, 9), ctx_range=None)
    a = wl.make_attention_inputs(w, device=DEV)
    plan_of = lambda: sv.spec_verify_attention_plan(a["q"], a["k_cache"], a["block_table"], w.k_draft)
    plan = plan_of()
    assert plan["kernel"] == kind
    assert plan["stages"] >= (1 if w.head_dim == 256 and kind == "tc" else 2)
    if kind == "tc":
        assert plan["keys_per_tile"] == 128 and plan["p_buffers"] >= 1 and plan["ctas_per_sm"] == 1
    else:
        assert plan["p_buffers"] == 0
    default, err = run_attention(sv, a, w)
    assert err == 0
    forced = {}
    for k in ("tc", "mma"):
        monkeypatch.setenv("SPEC_ATTN_KERNEL", k)
        assert plan_of()["kernel"] == k
        forced[k], err = run_attention(sv, a, w)
        assert err == 0
    other = "mma" if kind == "tc" else "tc"
    assert torch.equal(default, forced[kind])
    assert not torch.equal(default, forced[other])


def _random_shape(rng):
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32, 64, 128]))
    while True:
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
        k = int(rng.integers(1, 8))
        if (k + 1) * G <= 64 and Hkv * G <= 64:
            break
    B = int(rng.integers(1, 9))
    ctx = tuple(int(c) for c in rng.integers(k + 1, 2600, B))
    return B, ctx, bs, Hkv * G, Hkv, D, k


@pytest.mark.parametrize("seed", range(12))
def test_attention_random_shapes(sv, oracle_mod, attn_kernel, seed):
    """Seeded random shapes: every head dim, block size, GQA group and draft length
    within the supported range, ragged contexts, both kernels where D = 128 or 256."""
    rng = np.random.default_rng(1000 + seed)
    B, ctx, bs, Hq, Hkv, D, k = _random_shape(rng)
    if D == 64 and attn_kernel == "tc":
        pytest.skip("one kernel for this head dim")
    w = wl.Workload(name=f"rand{seed}", batch=B, ctx_lens=ctx, block_size=bs, num_q_heads=Hq,
                    num_kv_heads=Hkv, head_dim=D, k_draft=k, seed=seed)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (w, mx, rel)


def test_attention_is_deterministic_and_reuses_workspace(sv, attn_kernel):
    w = wl.WORKLOADS["llama8b_eagle3"].replace(batch=8, ctx_lens=(2048,) * 8)
    a = wl.make_attention_inputs(w, device=DEV)
    ws = sv.new_attention_workspace(
        sv.spec_verify_attention_workspace(a["q"], a["k_cache"], a["block_table"], w.k_draft), DEV)
    o1, _ = run_attention(sv, a, w, workspace=ws)
    o2, _ = run_attention(sv, a, w, workspace=ws)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("D,Hq", [(128, 64), (256, 24)])
def test_attention_split_units_merge_this_calls_pieces(sv, oracle_mod, attn_kernel, D, Hq):
    """Split units are merged from the pieces of the same call. Two inputs with the same shapes
    (so the same split plan and the same partial slots in one reused workspace) alternate: the
    first input's output comes back bit-identical and the second's matches the oracle. A merge
    that read a piece before its CTA had written it would pick up the other input's piece, which
    the previous call left in the workspace."""
    w = wl.Workload(name="split_reuse", batch=4, ctx_lens=(30011, 25000, 41000, 18003), block_size=128,
                    num_q_heads=Hq, num_kv_heads=8 if D == 128 else 4, head_dim=D, k_draft=7 if D == 128 else 3,
                    seed=21)
    a = wl.make_attention_inputs(w, device=DEV)
    b = wl.make_attention_inputs(w.replace(seed=22), device=DEV)
    ws = sv.new_attention_workspace(
        sv.spec_verify_attention_workspace(a["q"], a["k_cache"], a["block_table"], w.k_draft), DEV)
    o1, e1 = run_attention(sv, a, w, workspace=ws)
    o2, e2 = run_attention(sv, b, w, workspace=ws)
    o3, e3 = run_attention(sv, a, w, workspace=ws)
    assert e1 == e2 == e3 == 0
    assert torch.equal(o1, o3)
    assert not torch.equal(o1, o2)
    mx, rel = attention_errors(o2.cpu().numpy(), oracle_attention_for(oracle_mod, b))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


def test_attention_bad_block_and_bad_ctx_give_zero_rows(sv, oracle_mod, attn_kernel):
    w = wl.Workload(name="bad", batch=4, ctx_lens=(300, 300, 300, 300), block_size=16, num_q_heads=8,
                    num_kv_heads=2, head_dim=128, k_draft=3, seed=5)
    a = wl.make_attention_inputs(w, device=DEV)
    a["block_table"][1, 3] = a["num_blocks"] + 5          # out-of-range block id
    a["ctx_lens"][2] = 2                                   # ctx < k+1
    out, err = run_attention(sv, a, w)
    assert err & sv.DEVERR["block_id"] and err & sv.DEVERR["ctx_len"]
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    ref = oracle_attention_for(oracle_mod, a, seqs=np.array([0, 3], np.int32))
    mx, rel = attention_errors(out[[0, 3]].cpu().numpy(), ref)
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2


def test_attention_minimal_context_row0_is_v0(sv):
    """ctx = k+1: row 0 sees one key, so its output is that key's value."""
    w = wl.Workload(name="min", batch=3, ctx_lens=(4, 4, 4), block_size=16, num_q_heads=8, num_kv_heads=2,
                    head_dim=64, k_draft=3, seed=9)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    for b in range(3):
        phys = int(a["block_table"][b, 0])
        v0 = a["v_cache"][phys, 0].float()  # [Hkv, D]
        for h in range(8):
            assert torch.allclose(out[b, 0, h], v0[h // 4], atol=1e-6, rtol=0)


@pytest.mark.parametrize("Hq,ctx", [(16, 60000), (4, 60000), (16, 700)], ids=["rows64", "rows16", "rows64_short"])
def test_attention_one_unit_split_over_every_cta(sv, oracle_mod, attn_kernel, Hq, ctx):
    """One sequence with one kv head: its single unit is cut into a piece per CTA
    (over a hundred for a 60000-token context), and the last CTA to arrive merges
    them all; a short context gives a few pieces of one tile each."""
    w = wl.Workload(name="one_unit", batch=1, ctx_lens=(ctx,), block_size=128, num_q_heads=Hq, num_kv_heads=1,
                    head_dim=128, k_draft=3, seed=ctx % 101 + Hq)
    a = wl.make_attention_inputs(w, device=DEV)
    out, err = run_attention(sv, a, w)
    assert err == 0
    mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


@pytest.mark.parametrize("D,k,G", [(128, 7, 8), (256, 3, 8)], ids=["d128_rows64", "d256_rows32"])
def test_attention_bad_block_inside_a_split_unit(sv, oracle_mod, attn_kernel, D, k, G):
    """Two long sequences over one kv head, so each unit is cut into dozens of
    pieces and merged in several chunks; sequence 0 has an out-of-range block id
    in the middle of its context. Its rows must come out zero (the piece holding
    the bad block marks itself unusable and the merge drops the unit), the error
    bit is raised, and sequence 1 still matches the oracle. The shapes are the
    ones the tcgen05 kernel runs with four softmax warpgroups."""
    w = wl.Workload(name="bad_split", batch=2, ctx_lens=(60000, 50000), block_size=64, num_q_heads=G,
                    num_kv_heads=1, head_dim=D, k_draft=k, seed=17 + D)
    a = wl.make_attention_inputs(w, device=DEV)
    a["block_table"][0, 400] = a["num_blocks"] + 7
    out, err = run_attention(sv, a, w)
    assert err & sv.DEVERR["block_id"]
    assert torch.all(out[0] == 0)
    ref = oracle_attention_for(oracle_mod, a, seqs=np.array([1], np.int32))
    mx, rel = attention_errors(out[[1]].cpu().numpy(), ref)
    assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)
