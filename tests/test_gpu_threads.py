"""The library called from several host threads at once.

ctypes releases the interpreter lock during a foreign call, so these threads
really enter the library concurrently, each on its own stream, with shapes
whose launch settings differ (vocabularies with different cluster plans,
batches with different shared-memory plans). Every result must equal the
single-threaded one.
"""

import threading

import pytest
import torch

from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _accept(sv, inp, stream):
    B, R, V = inp["target_logits"].shape
    toks = torch.empty((B, R), dtype=torch.int32, device=DEV)
    alen = torch.empty((B,), dtype=torch.int32, device=DEV)
    sv.spec_accept(inp["target_logits"], inp["draft_tokens"], inp["draft_probs"], inp["philox_seed"], inp["mode"],
                   inp["temperature"], toks, alen, stream=stream)
    return toks, alen


def _attention(sv, a, w, stream):
    out = torch.empty((w.batch, w.rows, w.num_q_heads, w.head_dim), dtype=torch.float32, device=DEV)
    sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft, out,
                             stream=stream)
    return out


def test_concurrent_host_threads_match_single_threaded(sv):
    small = wl.WORKLOADS["tiny"].replace(batch=6, vocab=1000, mode="mixed")
    large = wl.WORKLOADS["llama8b_eagle3"].replace(batch=4, mode="mixed")
    acc_inputs = [wl.make_accept_inputs(w, device=DEV, seed=s) for s, w in ((5, small), (6, large))]
    att_work = [wl.WORKLOADS["serving128"].replace(batch=b, ctx_range=(64, 700), seed=b) for b in (3, 40)]
    att_inputs = [wl.make_attention_inputs(w, device=DEV) for w in att_work]
    stream0 = torch.cuda.current_stream()
    ref_acc = [tuple(t.clone() for t in _accept(sv, inp, stream0)) for inp in acc_inputs]
    ref_att = [_attention(sv, a, w, stream0).clone() for a, w in zip(att_inputs, att_work)]
    torch.cuda.synchronize()

    failures = []

    def worker(tid):
        stream = torch.cuda.Stream()
        try:
            with torch.cuda.stream(stream):
                for it in range(12):
                    i = (tid + it) % 2
                    toks, alen = _accept(sv, acc_inputs[i], stream)
                    out = _attention(sv, att_inputs[i], att_work[i], stream)
                    stream.synchronize()
                    if not (torch.equal(toks, ref_acc[i][0]) and torch.equal(alen, ref_acc[i][1])):
                        failures.append(f"thread {tid} iteration {it}: acceptance differs")
                    if not torch.equal(out, ref_att[i]):
                        failures.append(f"thread {tid} iteration {it}: attention differs")
        except Exception as e:  # surfaced below
            failures.append(f"thread {tid}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not failures, failures[:4]
