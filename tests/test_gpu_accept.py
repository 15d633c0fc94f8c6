"""Acceptance on the GPU against the oracle (parity gate) and against the
distributional facts of speculative sampling.

Greedy tokens and accept lengths must match bit-exactly. Sampled rows must
match bit-exactly except rows the oracle marks as near ties (|u - p/q| < 1e-5,
or race keys within 1e-5 relative), which are counted and must stay below
1e-4 of the decisions.
"""

import numpy as np
import pytest
import torch
from scipy import stats

from helpers import MAX_EXCUSED_RATE, compare_accept
from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_accept(sv, inp, modes, *, probs="given"):
    B, R, V = inp["target_logits"].shape
    toks = torch.full((B, R), -7, dtype=torch.int32, device=DEV)
    alen = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = inp["draft_probs"] if probs == "given" else None
    sv.spec_accept(inp["target_logits"], inp["draft_tokens"], q, inp["philox_seed"], modes, inp["temperature"],
                   toks, alen, dev_err=err)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), alen.cpu().numpy(), int(err.item())


def oracle_accept(oracle_mod, inp, modes, probs="given"):
    return oracle_mod.accept(inp["target_logits"].cpu().numpy(), inp["draft_tokens"].cpu().numpy(),
                             inp["draft_probs"].cpu().numpy() if probs == "given" else None,
                             inp["philox_seed"], modes.cpu().numpy(), inp["temperature"].cpu().numpy())


CASES = [
    ("tiny", "sample"), ("tiny", "greedy"), ("llama8b_eagle3", "sample"), ("llama8b_eagle3", "greedy"),
    ("llama8b_eagle3_cal", "sample"),
    ("serving128", "mixed"), ("hybrid_gdn", "sample"), ("hybrid_gdn", "greedy"), ("longctx", "sample"),
]


@pytest.mark.parametrize("name,mode", CASES, ids=[f"{a}-{b}" for a, b in CASES])
def test_accept_parity_named_workloads(sv, oracle_mod, name, mode):
    w = wl.WORKLOADS[name]
    inp = wl.make_accept_inputs(w, device=DEV, mode=mode)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    assert err == 0
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert rc == 0
    bad, excused = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0, f"{bad} rows differ from the oracle"
    assert np.all((alen >= 0) & (alen <= w.k_draft))
    for b in range(w.batch):
        assert np.all(tok[b, alen[b] + 1:] == -1) and tok[b, alen[b]] >= 0


def test_accept_mixed_rows_equal_single_mode_rows(sv):
    """Rows are independent on the GPU too. In a serving-shaped mixed batch (per-row modes and
    temperatures), every row gives bit-identical tokens and accept length to the same row in a
    batch run wholly in its mode, and a sampling row gives the same as when every row has its
    temperature. The kernel and its launch configuration are the same in every call, so the
    comparison needs no tolerance."""
    w = wl.WORKLOADS["serving128"].replace(batch=96)
    inp = wl.make_accept_inputs(w, device=DEV, mode="mixed")
    modes = inp["mode"]
    m = modes.cpu().numpy()
    assert 0 < m.sum() < len(m)
    t_mix, a_mix, e = run_accept(sv, inp, modes)
    assert e == 0
    t_g, a_g, e = run_accept(sv, inp, torch.zeros_like(modes))
    assert e == 0
    t_s, a_s, e = run_accept(sv, inp, torch.ones_like(modes))
    assert e == 0
    for b in range(len(m)):
        rt, ra = (t_s, a_s) if m[b] else (t_g, a_g)
        assert np.array_equal(t_mix[b], rt[b]) and a_mix[b] == ra[b], b
    temps = inp["temperature"]
    for b in np.nonzero(m)[0][:4]:
        one_t = dict(inp, temperature=torch.full_like(temps, float(temps[b])))
        t_u, a_u, e = run_accept(sv, one_t, torch.ones_like(modes))
        assert e == 0
        assert np.array_equal(t_mix[b], t_u[b]) and a_mix[b] == a_u[b], b


def test_accept_greedy_without_draft_probs(sv, oracle_mod):
    w = wl.WORKLOADS["tiny"].replace(batch=64)
    inp = wl.make_accept_inputs(w, device=DEV, mode="greedy")
    tok, alen, err = run_accept(sv, inp, inp["mode"], probs=None)
    rt, ra, _, _, _ = oracle_accept(oracle_mod, inp, inp["mode"], probs=None)
    assert err == 0 and np.array_equal(tok, rt) and np.array_equal(alen, ra)


@pytest.mark.parametrize("name", ["tiny", "llama8b_eagle3", "serving128"])
def test_accept_sampling_without_draft_probs(sv, oracle_mod, name):
    """No draft distribution: one-hot q at the drafted token, same decisions as the oracle."""
    w = wl.WORKLOADS[name]
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"], probs=None)
    assert err == 0
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"], probs=None)
    assert rc == 0
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0, f"{bad} rows differ from the oracle"
    # a rejected draft is never re-emitted as the correction token
    d = inp["draft_tokens"].cpu().numpy()
    samp = inp["mode"].cpu().numpy() == 1
    for b in np.nonzero(samp & (alen < w.k_draft))[0]:
        assert tok[b, alen[b]] != d[b, alen[b]]


def test_accept_without_draft_probs_distribution(sv):
    """Over 10^6 rows: a draft is kept with probability p(d); a rejection follows p
    with d removed."""
    B, k, V = 1_000_000, 1, 8
    rng = np.random.default_rng(6)
    l = rng.normal(0, 1.0, (k + 1, V)).astype(np.float32)
    L = torch.tensor(l, device=DEV).expand(B, k + 1, V).contiguous()
    d = torch.full((B, k), 3, dtype=torch.int32, device=DEV)
    inp = {"target_logits": L, "draft_tokens": d, "draft_probs": None, "philox_seed": 99,
           "temperature": torch.ones(B, device=DEV)}
    tok, alen, err = run_accept(sv, inp, torch.ones(B, dtype=torch.int32, device=DEV), probs=None)
    assert err == 0
    p0 = np.exp(l[0].astype(np.float64))
    p0 /= p0.sum()
    acc = alen == 1
    assert abs(acc.mean() - p0[3]) < 5 * np.sqrt(p0[3] * (1 - p0[3]) / B)
    rej = tok[~acc, 0]
    assert np.all(rej != 3)
    resid = p0.copy()
    resid[3] = 0.0
    resid /= resid.sum()
    counts = np.bincount(rej, minlength=V).astype(np.float64)
    keep = resid > 0
    assert stats.chisquare(counts[keep], resid[keep] * counts.sum()).pvalue > 1e-3


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_accept_longest_draft(sv, oracle_mod, mode):
    """k = 31, the longest supported draft, with near-copy drafts so rows run deep."""
    w = wl.WORKLOADS["tiny"].replace(batch=48, k_draft=31, vocab=3000, noise_sigma=0.2)
    inp = wl.make_accept_inputs(w, device=DEV, mode=mode)
    if mode == "greedy":
        # row b copies the target's argmax for its first b % 32 positions
        am = inp["target_logits"][:, :w.k_draft].argmax(-1).to(torch.int32)
        depth = torch.arange(w.batch, device=DEV) % (w.k_draft + 1)
        keep = torch.arange(w.k_draft, device=DEV)[None, :] < depth[:, None]
        inp["draft_tokens"] = torch.where(keep, am, inp["draft_tokens"]).contiguous()
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    assert err == 0
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert rc == 0
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0, f"{bad} rows differ from the oracle"
    assert alen.max() >= 2  # some rows accept several drafts


def test_accept_greedy_is_sequential_greedy(sv):
    """Emitted tokens = argmax of each target row, cut after the first draft miss."""
    B, k, V = 512, 5, 4000
    g = torch.Generator(device=DEV).manual_seed(3)
    L = torch.randn((B, k + 1, V), generator=g, device=DEV) * 3
    am = L.argmax(-1).to(torch.int32)
    m_true = torch.randint(0, k + 1, (B,), generator=g, device=DEV)
    d = am[:, :k].clone()
    rows = torch.arange(B, device=DEV)
    miss = m_true < k
    d[rows[miss], m_true[miss]] = (d[rows[miss], m_true[miss]] + 1) % V
    inp = {"target_logits": L, "draft_tokens": d.contiguous(), "draft_probs": None, "philox_seed": 0,
           "temperature": torch.ones(B, device=DEV)}
    tok, alen, err = run_accept(sv, inp, torch.zeros(B, dtype=torch.int32, device=DEV), probs=None)
    assert err == 0
    assert np.array_equal(alen, m_true.cpu().numpy())
    amc = am.cpu().numpy()
    for b in range(B):
        assert np.array_equal(tok[b, : alen[b] + 1], amc[b, : alen[b] + 1])


def test_accept_near_tie_rate_over_many_decisions(sv, oracle_mod):
    B, k, V = 20000, 3, 96
    w = wl.Workload(name="many", batch=B, ctx_lens=(4,) * B, vocab=V, k_draft=k, logit_sigma=2.0, noise_sigma=1.0,
                    mode="mixed", temperature=(0.5, 1.2), seed=11)
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, _ = oracle_accept(oracle_mod, inp, inp["mode"])
    bad, excused = compare_accept(tok, alen, rt, ra, margin, gap)
    decisions = int(np.sum(np.where(ra >= 0, np.minimum(ra + 1, k), 0)))
    assert err == 0 and bad == 0
    assert excused / decisions < MAX_EXCUSED_RATE, (excused, decisions)


def test_accept_vocab_not_multiple_of_four(sv, oracle_mod):
    w = wl.WORKLOADS["tiny"].replace(vocab=1001, batch=32, mode="mixed")
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, _ = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and compare_accept(tok, alen, rt, ra, margin, gap)[0] == 0


def test_accept_large_vocab_uses_full_cluster(sv, oracle_mod):
    w = wl.WORKLOADS["hybrid_gdn"].replace(vocab=700001, batch=4, mode="mixed")
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, _ = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and compare_accept(tok, alen, rt, ra, margin, gap)[0] == 0


def _chi2(samples, probs):
    counts = np.bincount(samples, minlength=len(probs)).astype(np.float64)
    return stats.chisquare(counts, probs * counts.sum()).pvalue


def test_accept_sampling_distribution_chi_square(sv):
    """Over 10^6 rows the first emitted token follows p_0, the second (given d_0 kept) p_1."""
    B, k, V, T = 1_000_000, 2, 8, 1.0
    rng = np.random.default_rng(5)
    l = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    q = np.exp(l[:k] + rng.normal(0, 1, (k, V)))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    L = torch.tensor(l, device=DEV).expand(B, k + 1, V).contiguous()
    Q = torch.tensor(q, device=DEV).expand(B, k, V).contiguous()
    g = torch.Generator(device=DEV).manual_seed(7)
    d = torch.multinomial(Q.view(B * k, V), 1, generator=g).view(B, k).to(torch.int32)
    inp = {"target_logits": L, "draft_tokens": d, "draft_probs": Q, "philox_seed": 2024,
           "temperature": torch.full((B,), T, device=DEV)}
    tok, alen, err = run_accept(sv, inp, torch.ones(B, dtype=torch.int32, device=DEV))
    assert err == 0
    p = np.exp(l.astype(np.float64) / T)
    p /= p.sum(-1, keepdims=True)
    assert _chi2(tok[:, 0], p[0]) > 1e-3
    sel = alen >= 1
    assert _chi2(tok[sel, 1], p[1]) > 1e-3
    assert _chi2(tok[:, 0], q[0].astype(np.float64) / q[0].sum()) < 1e-3  # the test has power


def test_accept_invalid_rows_flagged(sv):
    B, k, V = 4, 3, 100
    L = torch.zeros((B, k + 1, V), device=DEV)
    Q = torch.full((B, k, V), 1.0 / V, device=DEV)
    d = torch.tensor([[1, 2, 3], [1, 200, 3], [1, 2, 3], [4, 5, 6]], dtype=torch.int32, device=DEV)
    modes = torch.tensor([1, 1, 1, 2], dtype=torch.int32, device=DEV)
    temp = torch.tensor([1.0, 1.0, 0.0, 1.0], device=DEV)
    inp = {"target_logits": L, "draft_tokens": d, "draft_probs": Q, "philox_seed": 1, "temperature": temp}
    tok, alen, err = run_accept(sv, inp, modes)
    assert alen[0] == k and np.all(alen[1:] == -1) and np.all(tok[1:] == -1)
    assert err & sv.DEVERR["token"] and err & sv.DEVERR["temperature"] and err & sv.DEVERR["mode"]


@pytest.mark.parametrize("vocab", [1000, 1001], ids=["aligned", "unaligned"])
def test_accept_many_waves(sv, oracle_mod, vocab):
    """1400 rows of a 1000-word vocabulary (one CTA per row): more rows than the
    device holds at once, so each CTA walks several rows; aligned rows (16-byte
    loads) and unaligned ones (scalar loads)."""
    w = wl.WORKLOADS["tiny"].replace(vocab=vocab, batch=1400, mode="mixed")
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and rc == 0
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0


@pytest.mark.parametrize("batch", [64, 1400], ids=["one_wave", "many_waves"])
def test_accept_all_zero_residual_races_over_p(sv, oracle_mod, batch):
    """Draft probabilities at twice the target's make max(0, p - q) zero everywhere
    while drafts are still rejected (whenever u >= 1/2): the correction token is
    then drawn from p itself (a second race over the same slice)."""
    w = wl.WORKLOADS["tiny"].replace(vocab=1000, batch=batch, mode="sample")
    inp = wl.make_accept_inputs(w, device=DEV)
    T = inp["temperature"].view(-1, 1, 1)
    inp["draft_probs"] = (2.0 * torch.softmax(inp["target_logits"][:, :w.k_draft] / T, dim=-1)).contiguous()
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and rc == 0
    assert (ra < w.k_draft).sum() > batch // 4  # rejections happen (u >= 1/2 at some position)
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0


def test_binding_rejects_tensors_the_kernels_cannot_use(sv):
    """Host tensors, a malformed error word and tensors on another device are
    refused before anything is launched."""
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_accept_inputs(w, device=DEV)
    B, R, V = inp["target_logits"].shape
    toks = torch.empty((B, R), dtype=torch.int32, device=DEV)
    alen = torch.empty((B,), dtype=torch.int32, device=DEV)
    args = [inp["target_logits"], inp["draft_tokens"], inp["draft_probs"], inp["philox_seed"], inp["mode"],
            inp["temperature"], toks, alen]
    host = list(args)
    host[0] = inp["target_logits"].cpu()
    with pytest.raises(ValueError):
        sv.spec_accept(*host)
    for bad in (torch.zeros(1, dtype=torch.float32, device=DEV), torch.zeros(1, dtype=torch.int32),
                torch.zeros(0, dtype=torch.int32, device=DEV)):
        with pytest.raises(ValueError):
            sv.spec_accept(*args, dev_err=bad)
    if torch.cuda.device_count() > 1:
        other = torch.cuda.Stream(device=1)
        with pytest.raises(ValueError):
            sv.spec_accept(*args, stream=other)
    sv.spec_accept(*args, dev_err=torch.zeros(1, dtype=torch.int32, device=DEV))  # the valid call still works
    torch.cuda.synchronize()


@pytest.mark.parametrize("vocab", [40000, 40001], ids=["aligned", "unaligned"])
def test_accept_every_launch_configuration(sv, oracle_mod, monkeypatch, vocab):
    """Every (threads per CTA, CTAs per cluster) the launch can pick, forced in turn
    through SPEC_ACCEPT_CONFIG on one mixed case of 200 rows: small clusters hold
    every row at once, 16-CTA clusters walk several rows each. Each result must
    match the oracle like the launch's own choice does."""
    w = wl.WORKLOADS["serving128"].replace(vocab=vocab, batch=200, mode="mixed")
    inp = wl.make_accept_inputs(w, device=DEV)
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert rc == 0
    for threads in (128, 256):
        for csize in (1, 2, 4, 8, 16):
            monkeypatch.setenv("SPEC_ACCEPT_CONFIG", f"{threads}x{csize}")
            tok, alen, err = run_accept(sv, inp, inp["mode"])
            bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
            assert err == 0 and bad == 0, (threads, csize, err, bad)


@pytest.mark.parametrize("vocab", [1, 2, 3, 5, 7])
@pytest.mark.parametrize("k_draft", [1, 3])
def test_accept_vocabularies_smaller_than_a_few_groups(sv, oracle_mod, vocab, k_draft):
    """Vocabularies of fewer than two float4 groups (one CTA, most threads hold no
    logit, scalar loads past the row's end filled), with one or three drafts."""
    w = wl.WORKLOADS["tiny"].replace(vocab=vocab, k_draft=k_draft, batch=64, mode="mixed")
    inp = wl.make_accept_inputs(w, device=DEV)
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and rc == 0
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0
    assert np.all((tok[:, : k_draft + 1] >= -1) & (tok[:, : k_draft + 1] < vocab))


def test_accept_random_shapes(sv, oracle_mod):
    """Seeded random shapes: batch 1-160, vocabulary 1-90000 (aligned or not), 1-12
    drafts, noise and temperature ranges, mixed modes, with and without draft
    probabilities; every one against the oracle."""
    rng = np.random.default_rng(2027)
    for case in range(14):
        batch = int(rng.integers(1, 161))
        vocab = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 4096)), int(rng.integers(4096, 90000))]))
        k = int(rng.integers(1, 13))
        lo = float(rng.uniform(0.3, 1.0))
        w = wl.WORKLOADS["tiny"].replace(
            name=f"random{case}", batch=batch, vocab=vocab, k_draft=k, mode="mixed",
            logit_sigma=float(rng.uniform(0.5, 4.0)), noise_sigma=float(rng.uniform(0.1, 2.0)),
            temperature=(lo, lo + float(rng.uniform(0.0, 1.0))), seed=100 + case)
        inp = wl.make_accept_inputs(w, device=DEV)
        probs = "given" if case % 3 else "none"
        tok, alen, err = run_accept(sv, inp, inp["mode"], probs=probs)
        rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"], probs=probs)
        assert err == 0 and rc == 0, (case, batch, vocab, k)
        bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
        assert bad == 0, (case, batch, vocab, k, probs)


def test_accept_extreme_temperatures(sv, oracle_mod):
    """Per-row temperatures from 0.001 (p one-hot for practical purposes: most
    exponentials underflow) to 1000 (p nearly flat over the vocabulary)."""
    temps = [1e-3, 0.05, 0.3, 1.0, 4.0, 20.0, 1000.0]
    B = 7 * len(temps)
    w = wl.WORKLOADS["tiny"].replace(batch=B, vocab=5000, k_draft=3, mode="sample", logit_sigma=3.0, seed=77)
    inp = wl.make_accept_inputs(w, device=DEV)
    T = torch.tensor([temps[i % len(temps)] for i in range(B)], dtype=torch.float32, device=DEV)
    inp["temperature"] = T
    # draft probabilities at each row's own temperature, drafts drawn from them
    g = torch.Generator(device=DEV).manual_seed(5)
    dl = inp["target_logits"][:, :3, :] + torch.randn((B, 3, 5000), generator=g, device=DEV)
    inp["draft_probs"] = torch.softmax(dl / T.view(B, 1, 1), dim=-1).contiguous()
    inp["draft_tokens"] = torch.multinomial(inp["draft_probs"].view(B * 3, 5000), 1, generator=g).view(B, 3) \
        .to(torch.int32).contiguous()
    tok, alen, err = run_accept(sv, inp, inp["mode"])
    rt, ra, margin, gap, rc = oracle_accept(oracle_mod, inp, inp["mode"])
    assert err == 0 and rc == 0
    bad, _ = compare_accept(tok, alen, rt, ra, margin, gap)
    assert bad == 0
