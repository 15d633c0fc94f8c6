"""The algorithmic byte counts behind every roofline fraction bench.py reports,
checked on small cases worked out by hand (CPU only)."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_paged_gb300 import workloads as wl  # noqa: E402


def test_attention_bytes_by_hand():
    # 2 sequences of 5 and 70 tokens, 2 kv heads x 8 dims, 4 q heads, 3 drafts, blocks of 16
    w = wl.Workload(name="t", batch=2, ctx_lens=(5, 70), block_size=16, num_q_heads=4, num_kv_heads=2,
                    head_dim=8, k_draft=3)
    kv = 75 * 2 * 8 * 2 * 2        # visible tokens x kv heads x dims x bf16 x (K, V)
    qo = 2 * 4 * 4 * 8 * (2 + 4)   # rows x q heads x dims x (bf16 q in + fp32 out)
    table = (1 + 5) * 4 + 2 * 4    # block ids used (1 + 5 blocks) + ctx_lens
    assert bench.attention_bytes(w, [5, 70]) == kv + qo + table == 6368


def test_accept_bytes_by_hand():
    # V = 1000, k = 3; a greedy row that stops at 0, a sampling row that keeps all three
    # drafts and a sampling row that stops at 1; an invalid row reads nothing but the fixed part
    w = wl.Workload(name="t", batch=4, ctx_lens=(8,) * 4, vocab=1000, k_draft=3)
    greedy_0 = 1 * 4000                                # logit row 0
    sample_3 = 4 * 4000 + 0 + 3 * 32                   # rows 0..3, no residual row, q(d_j) sectors
    sample_1 = 2 * 4000 + 4000 + 1 * 32                # rows 0..1, draft row 1 of the race, q(d_0)
    fixed = 4 * (3 * 4 + 4 + 4 + 4 * 4 + 4)            # drafts, mode, temperature, out_tokens, accept_len
    got = bench.accept_bytes(w, [0, 1, 1, 1], [0, 3, 1, -1])
    assert got == greedy_0 + sample_3 + sample_1 + fixed == 32288


def test_acceptance_rate_by_hand():
    # accepted 0 + 3 + 1 drafts; decided 1 + 3 + 2 (a full row decided k drafts)
    assert bench.acceptance_rate([0, 3, 1], 3) == pytest.approx(4 / 6)
    assert bench.acceptance_rate([], 3) is None


def test_commit_and_gdn_bytes_by_hand():
    w = wl.Workload(name="t", batch=3, ctx_lens=(8,) * 3, k_draft=1, gdn_layers=2, gdn_heads=1, gdn_dk=5, gdn_dv=2)
    assert bench.commit_bytes(w) == 2 * 2 * 3 * 10 * 4           # read the kept slot, write the live state
    assert bench.commit_bytes(w, "select") == 2 * 3 * 20          # five int32 per (layer, row)
    g = wl.Workload(name="t", batch=2, ctx_lens=(8,) * 2, k_draft=1, gdn_layers=1, gdn_heads=3, gdn_dk=4, gdn_dv=4)
    states = 2 * 3 * (4 * 4 * 4) * (1 + 2)                       # read once, write one checkpoint per token
    acts = 2 * 2 * 3 * (2 * 4 + 2 * 4) * 4                       # q, k, v, out per token and head
    gates = 2 * 2 * 3 * 8                                        # g and beta
    assert bench.gdn_verify_bytes(g) == states + acts + gates == 2016


def test_recorded_traffic_follows_plan_and_kernel_sources(tmp_path, monkeypatch):
    """A recorded ncu DRAM figure is reported only for the kernel instance it was
    captured on and only while that kernel's device sources are unchanged; a record
    per unit (a smaller capture of the same kernel) scales by the call's units."""
    import json
    src = tmp_path / "k.cuh"
    src.write_text("// kernel v1\n")
    (tmp_path / "c.cu").write_text("// commit v1\n")
    plan = dict(kernel="mma", m_tiles=1, keys_per_tile=64, stages=3, p_buffers=0, ctas_per_sm=2)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"attention/mma": ["k.cuh"], "attention/tc": ["other.cuh"],
                                                  "commit": ["c.cu"]})
    record = {"attention": {"w": {"plan": plan, "kernel_sources_sha256": bench.kernel_sources_sha256(["k.cuh"]),
                                  "dram_bytes_per_call": 1234}},
              "commit": {"w": {"kernel_sources_sha256": bench.kernel_sources_sha256(["c.cu"]),
                               "dram_bytes_per_unit": 10}}}
    traffic = tmp_path / "traffic.json"
    traffic.write_text(json.dumps(record))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(traffic))
    assert bench.recorded_traffic("attention", "w", plan) == 1234
    assert bench.recorded_traffic("attention", "unrecorded", plan) is None
    assert bench.recorded_traffic("attention", "w", dict(plan, stages=4)) is None    # another instance runs
    assert bench.recorded_traffic("attention", "w", dict(plan, kernel="tc")) is None  # another kernel runs
    assert bench.recorded_traffic("commit", "w", units=7) == 70
    assert bench.recorded_traffic("accept", "w") is None                               # nothing recorded
    src.write_text("// kernel v2\n")                                                 # the kernel changed
    assert bench.recorded_traffic("attention", "w", plan) is None
    assert bench.recorded_traffic("commit", "w", units=7) == 70


def test_kernel_sources_hash_covers_names_and_bytes(tmp_path, monkeypatch):
    (tmp_path / "a").write_text("x")
    (tmp_path / "b").write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    ha, hb = bench.kernel_sources_sha256(["a"]), bench.kernel_sources_sha256(["b"])
    assert ha != hb and len(ha) == 64
    assert bench.kernel_sources_sha256(["a", "b"]) != bench.kernel_sources_sha256(["b", "a"])


def test_committed_traffic_records_name_their_kernel_sources():
    """Every committed record lists exactly the device sources bench.py hashes for its kernel."""
    import json
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    assert rec
    for kernel, per_workload in rec.items():
        for name, entry in per_workload.items():
            key = bench.traffic_key(kernel, entry.get("plan"))
            assert entry["kernel_sources"] == bench.KERNEL_SOURCES[key], (kernel, name)
            assert (entry.get("dram_bytes_per_call") or entry.get("dram_bytes_per_unit")) > 0
            for rel in entry["kernel_sources"]:
                assert os.path.exists(os.path.join(ROOT, rel)), rel
