"""The library's first calls in a process made inside a CUDA graph capture.

A serving engine may capture its verify step before it ever ran it eagerly. The
first call of each entry point does one-time launch set-up (function attributes,
occupancy queries, the tensor-map encoder); none of it may break the capture.
A fresh process captures spec_verify_attention and spec_accept as its first
calls (and, for the hybrid workload, the gated delta rule and the commit),
replays the graphs and compares the results with eager calls.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys
sys.path.insert(0, sys.argv[1])
import torch
import speculative_decoding_verification_paged_gb300 as sv
from speculative_decoding_verification_paged_gb300 import workloads as wl

dev = "cuda"
for name in ("llama8b_eagle3", "hybrid_gdn"):  # mma.sync and tcgen05 attention
    w = wl.WORKLOADS[name].replace(batch=6, ctx_range=None, ctx_lens=(700, 33, 2048, 129, 1500, 64))
    a = wl.make_attention_inputs(w, device=dev)
    acc = wl.make_accept_inputs(w, device=dev)
    B, R = w.batch, w.rows
    out = torch.empty((B, R, w.num_q_heads, w.head_dim), device=dev)
    toks = torch.empty((B, R), dtype=torch.int32, device=dev)
    alen = torch.empty((B,), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.new_attention_workspace(
        sv.spec_verify_attention_workspace(a["q"], a["k_cache"], a["block_table"], w.k_draft), dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft,
                                 out, workspace=ws, dev_err=err)
        sv.spec_accept(acc["target_logits"], acc["draft_tokens"], acc["draft_probs"], acc["philox_seed"],
                       acc["mode"], acc["temperature"], toks, alen, dev_err=err)
    # the hybrid step's other calls: the gated delta rule of one layer and the
    # commit of its checkpoint of the accepted prefix
    if name == "hybrid_gdn":
        w1 = w.replace(gdn_layers=1)
        x = wl.make_gdn_verify_inputs(w1, device=dev, layers=1)
        q, k, v, gg, beta = (x[f][0] for f in ("q", "k", "v", "g", "beta"))
        Bq, Rq, H, dk = q.shape
        dv = v.shape[3]
        snaps = torch.zeros((Bq, Rq, H, dv, dk), device=dev)
        gout = torch.empty((Bq, Rq, H, dv), device=dev)
        live = torch.zeros((1, Bq, H * dv * dk), device=dev)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=side):
            sv.spec_gdn_verify(q, k, v, gg, beta, x["state"][0], snaps, gout, x["scale"], dev_err=err)
            sv.spec_commit_state(snaps.view(1, Bq, Rq, H * dv * dk), alen, live, dev_err=err)
    g.replay()
    if name == "hybrid_gdn":
        g2.replay()
    torch.cuda.synchronize()
    if name == "hybrid_gdn":
        snaps_e = torch.zeros_like(snaps)
        gout_e = torch.empty_like(gout)
        live_e = torch.zeros_like(live)
        sv.spec_gdn_verify(q, k, v, gg, beta, x["state"][0], snaps_e, gout_e, x["scale"], dev_err=err)
        sv.spec_commit_state(snaps_e.view(1, Bq, Rq, H * dv * dk), alen, live_e, dev_err=err)
        torch.cuda.synchronize()
        assert torch.equal(snaps, snaps_e) and torch.equal(gout, gout_e) and torch.equal(live, live_e)
    out2 = torch.empty_like(out)
    toks2 = torch.empty_like(toks)
    alen2 = torch.empty_like(alen)
    sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft, out2,
                             workspace=ws, dev_err=err)
    sv.spec_accept(acc["target_logits"], acc["draft_tokens"], acc["draft_probs"], acc["philox_seed"],
                   acc["mode"], acc["temperature"], toks2, alen2, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, out2), name
    assert torch.equal(toks, toks2) and torch.equal(alen, alen2), name
print("ok")
'''


def test_first_calls_inside_a_graph_capture():
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
