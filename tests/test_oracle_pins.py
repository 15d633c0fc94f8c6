"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test ties one oracle function to something it does not compute: closed
forms, library routines (a library Philox run on the CPU, numpy argmax, scipy's
logistic function and chi-square test), invariances of the definition, or the
output layout printed on the pages. A plausible slip in the oracle (a dropped
scale, a wrong slot or block index, a transposed head mapping, a sign error in
the residual, a wrong Philox counter) fails at least one of them.
"""

import os

import numpy as np
import pytest
from scipy import special, stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Philox and the uniform map
# --------------------------------------------------------------------------

_TRITON_PHILOX = r"""
import json, sys
import torch, triton, triton.language as tl

@triton.jit
def philox_kernel(c0p, c1p, c2p, c3p, o0p, o1p, o2p, o3p, seed, N: tl.constexpr):
    offs = tl.arange(0, N)
    r0, r1, r2, r3 = tl.philox(seed, tl.load(c0p + offs), tl.load(c1p + offs), tl.load(c2p + offs),
                               tl.load(c3p + offs), 10)
    tl.store(o0p + offs, r0)
    tl.store(o1p + offs, r1)
    tl.store(o2p + offs, r2)
    tl.store(o3p + offs, r3)

cases = json.loads(sys.stdin.read())
result = []
for seed, ctrs in cases:
    n = len(ctrs)
    c = [torch.tensor([x[j] for x in ctrs], dtype=torch.int64).to(torch.uint32) for j in range(4)]
    o = [torch.zeros(n, dtype=torch.uint32) for _ in range(4)]
    philox_kernel[(1,)](*c, *o, seed, N=n)
    result.append([[int(o[j][i].to(torch.int64)) & 0xFFFFFFFF for j in range(4)] for i in range(n)])
print(json.dumps(result))
"""


def test_philox_matches_library_reference(oracle_mod):
    """Philox4x32-10 against a library implementation run on the CPU (Triton's
    tl.philox under its interpreter: the Salmon et al. round function with the
    same constants, key = seed split into its low and high words), over a sweep
    of counters and keys that includes the all-zero and all-ones corners."""
    import json
    import subprocess
    import sys

    pytest.importorskip("triton")
    rng = np.random.default_rng(2011)
    cases = []
    for seed in (0, 0xFFFFFFFFFFFFFFFF, 0x299F31D0A4093822, int(rng.integers(0, 2**63))):
        ctrs = [[0, 0, 0, 0], [0xFFFFFFFF] * 4, [1, 0, 0, 0], [0, 0, 0, 1]]
        ctrs += rng.integers(0, 2**32, size=(12, 4), dtype=np.uint64).tolist()
        cases.append([seed, [[int(v) for v in c] for c in ctrs]])
    env = dict(os.environ, TRITON_INTERPRET="1")
    proc = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps(cases), env=env,
                          capture_output=True, text=True, timeout=600, cwd=os.path.dirname(GOLDEN))
    assert proc.returncode == 0, proc.stderr[-2000:]
    ref = json.loads(proc.stdout.strip().splitlines()[-1])
    for (seed, ctrs), want in zip(cases, ref):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for c, w in zip(ctrs, want):
            assert [int(x) for x in oracle_mod.philox4x32_10(c, key)] == w, (seed, c)


def test_uniform_map_endpoints(oracle_mod):
    assert oracle_mod.uniform(0) == 2.0 ** -24
    assert oracle_mod.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle_mod.uniform(1 << 31) == 0.5 + 2.0 ** -24
    # the low 9 bits are dropped
    assert oracle_mod.uniform(0x1FF) == oracle_mod.uniform(0)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def _paged(rng, ctx, Hkv, D, bs, *, contiguous_k=None, contiguous_v=None, spare=2, perm=True):
    """Lay contiguous per-sequence K/V [B][ctx_b, Hkv, D] out in a shuffled paged cache."""
    B = len(ctx)
    nblk = [-(-c // bs) for c in ctx]
    nb = sum(nblk) + spare
    order = rng.permutation(nb) if perm else np.arange(nb)
    kc = np.zeros((nb, bs, Hkv, D), np.uint16)
    vc = np.zeros((nb, bs, Hkv, D), np.uint16)
    table = np.full((B, max(nblk)), -1, np.int32)
    pos = 0
    for b in range(B):
        for n in range(nblk[b]):
            phys = order[pos]
            pos += 1
            table[b, n] = phys
            lo, hi = n * bs, min(ctx[b], (n + 1) * bs)
            kc[phys, : hi - lo] = contiguous_k[b][lo:hi]
            vc[phys, : hi - lo] = contiguous_v[b][lo:hi]
    return kc, vc, table


def _random_case(rng, ctx, R, Hq, Hkv, D):
    q = bf16_bits(rng.standard_normal((len(ctx), R, Hq, D)).astype(np.float32))
    ks = [bf16_bits(rng.standard_normal((c, Hkv, D)).astype(np.float32)) for c in ctx]
    vs = [bf16_bits(rng.standard_normal((c, Hkv, D)).astype(np.float32)) for c in ctx]
    return q, ks, vs


def test_attention_block_layout_invariance(oracle_mod):
    """The result depends on the tokens, not on block size or physical placement."""
    rng = np.random.default_rng(1)
    ctx, R, Hq, Hkv, D = [5, 23, 40], 4, 6, 2, 16
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    ref = None
    for bs, perm in [(1, False), (4, True), (16, True), (64, False)]:
        kc, vc, table = _paged(rng, ctx, Hkv, D, bs, contiguous_k=ks, contiguous_v=vs, perm=perm)
        out = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
        if ref is None:
            ref = out
        else:
            assert np.array_equal(out, ref)


def test_attention_single_visible_key_returns_its_value(oracle_mod):
    """ctx = k+1: row 0 sees only token 0, so its output is v_0 exactly."""
    rng = np.random.default_rng(2)
    ctx, R, Hq, Hkv, D = [4, 4], 4, 4, 2, 32
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    kc, vc, table = _paged(rng, ctx, Hkv, D, 2, contiguous_k=ks, contiguous_v=vs)
    out = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    G = Hq // Hkv
    for b in range(2):
        for h in range(Hq):
            assert np.array_equal(out[b, 0, h], bits_to_f64(vs[b][0, h // G]))


def test_attention_two_keys_closed_form(oracle_mod):
    """Row 1 with ctx = k+1 sees tokens 0 and 1: o = sigmoid(s0-s1) v0 + sigmoid(s1-s0) v1."""
    rng = np.random.default_rng(3)
    ctx, R, Hq, Hkv, D = [4], 4, 2, 1, 64
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    kc, vc, table = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks, contiguous_v=vs)
    out = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    k0, k1 = bits_to_f64(ks[0][0, 0]), bits_to_f64(ks[0][1, 0])
    v0, v1 = bits_to_f64(vs[0][0, 0]), bits_to_f64(vs[0][1, 0])
    for h in range(Hq):
        qq = bits_to_f64(q[0, 1, h])
        s0, s1 = qq @ k0 / 8.0, qq @ k1 / 8.0  # 1/sqrt(64)
        want = special.expit(s0 - s1) * v0 + special.expit(s1 - s0) * v1
        np.testing.assert_allclose(out[0, 1, h], want, rtol=1e-12, atol=1e-13)


def test_attention_zero_query_gives_mean_of_visible_values(oracle_mod):
    rng = np.random.default_rng(4)
    ctx, R, Hq, Hkv, D = [9, 31], 4, 4, 2, 8
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    q[:] = 0
    kc, vc, table = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks, contiguous_v=vs)
    out = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    G = Hq // Hkv
    for b, c in enumerate(ctx):
        for i in range(R):
            n_vis = c - R + i + 1
            for h in range(Hq):
                want = bits_to_f64(vs[b][:n_vis, h // G]).mean(axis=0)
                np.testing.assert_allclose(out[b, i, h], want, rtol=1e-12, atol=1e-14)


def test_attention_causal_window(oracle_mod):
    """Row i sees tokens t <= ctx - R + i and nothing later."""
    rng = np.random.default_rng(5)
    ctx, R, Hq, Hkv, D = [12], 4, 2, 1, 16
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    kc, vc, table = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks, contiguous_v=vs)
    base = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    P = ctx[0] - R
    for t in range(P, ctx[0]):  # perturb token t (its key and value)
        ks2 = [ks[0].copy()]
        vs2 = [vs[0].copy()]
        ks2[0][t] = bf16_bits(rng.standard_normal((Hkv, D)).astype(np.float32))
        vs2[0][t] = bf16_bits(rng.standard_normal((Hkv, D)).astype(np.float32))
        kc2, vc2, table2 = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks2, contiguous_v=vs2)
        out = oracle_mod.verify_attention(q, kc2, vc2, table2, np.array(ctx, np.int32))
        for i in range(R):
            if t <= P + i:
                assert not np.array_equal(out[0, i], base[0, i])
            else:
                assert np.array_equal(out[0, i], base[0, i])


def test_attention_gqa_groups_are_contiguous(oracle_mod):
    """With V constant per kv head, query head h returns the constant of kv head h // G."""
    rng = np.random.default_rng(6)
    ctx, R, Hq, Hkv, D = [20, 7], 4, 8, 4, 8
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    consts = np.array([1.0, -2.0, 0.5, 3.0], np.float32)
    for b in range(len(ctx)):
        vs[b][:] = bf16_bits(np.broadcast_to(consts[None, :, None], (ctx[b], Hkv, D)).copy())
    kc, vc, table = _paged(rng, ctx, Hkv, D, 8, contiguous_k=ks, contiguous_v=vs)
    out = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(out[:, :, h, :], consts[h // G], rtol=1e-12)


def test_attention_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(7)
    ctx, R, Hq, Hkv, D = [6, 17, 33, 9], 4, 4, 2, 16
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    kc, vc, table = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks, contiguous_v=vs)
    full = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32))
    sub = oracle_mod.verify_attention(q, kc, vc, table, np.array(ctx, np.int32), seqs=[3, 1])
    assert np.array_equal(sub[0], full[3]) and np.array_equal(sub[1], full[1])


def test_attention_rejects_bad_block_and_ctx(oracle_mod):
    rng = np.random.default_rng(8)
    ctx, R, Hq, Hkv, D = [8, 8], 4, 2, 1, 8
    q, ks, vs = _random_case(rng, ctx, R, Hq, Hkv, D)
    kc, vc, table = _paged(rng, ctx, Hkv, D, 4, contiguous_k=ks, contiguous_v=vs)
    bad = table.copy()
    bad[1, 1] = kc.shape[0]
    out = oracle_mod.verify_attention(q, kc, vc, bad, np.array(ctx, np.int32), check=False)
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.verify_attention(q, kc, vc, bad, np.array(ctx, np.int32))
    assert e.value.code == -5
    assert np.all(out[1] == 0) and np.any(out[0] != 0)
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.verify_attention(q, kc, vc, table, np.array([3, 8], np.int32))
    assert e.value.code == -6


# --------------------------------------------------------------------------
# Greedy acceptance
# --------------------------------------------------------------------------

def test_greedy_equals_sequential_greedy_decoding(oracle_mod):
    """Speculative greedy output = the target's own greedy tokens, cut after the first miss."""
    rng = np.random.default_rng(10)
    B, k, V = 64, 5, 50
    L = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    seq_greedy = np.argmax(L, axis=-1)  # sequential greedy decoding of the same logits
    m_true = rng.integers(0, k + 1, B)
    d = seq_greedy[:, :k].copy()
    for b in range(B):
        if m_true[b] < k:
            d[b, m_true[b]] = (seq_greedy[b, m_true[b]] + 1 + rng.integers(0, V - 1)) % V
    tok, alen, _, _, rc = oracle_mod.accept(L, d, None, 0, np.zeros(B, np.int32), np.ones(B, np.float32))
    assert rc == 0
    assert np.array_equal(alen, m_true)
    for b in range(B):
        m = m_true[b]
        assert np.array_equal(tok[b, : m + 1], seq_greedy[b, : m + 1])
        assert np.all(tok[b, m + 1:] == -1)


def test_greedy_reject_sampler_fixture(oracle_mod):
    rows = [l for l in open(os.path.join(GOLDEN, "reject_sampler_fixture.txt"))
            if l.startswith("row")]
    drafts, argmaxes, expected = [], [], []
    for r in rows:
        a, b, c = r[3:].split("|")
        drafts.append([int(x) for x in a.split()])
        argmaxes.append([int(x) for x in b.split()])
        expected.append([int(x) for x in c.split()])
    B, k, V = 3, 2, 4
    L = np.zeros((B, k + 1, V), np.float32)
    for b in range(B):
        for j in range(k + 1):
            L[b, j, argmaxes[b][j]] = 5.0
    tok, alen, _, _, _ = oracle_mod.accept(L, np.array(drafts, np.int32), None, 0,
                                           np.zeros(B, np.int32), np.ones(B, np.float32))
    assert tok.tolist() == expected
    assert alen.tolist() == [2, 0, 0]


def test_greedy_ties_go_to_lowest_index(oracle_mod):
    L = np.zeros((1, 2, 6), np.float32)
    L[0, 0, [2, 4]] = 1.0
    L[0, 1, [1, 5]] = 3.0
    tok, alen, _, _, _ = oracle_mod.accept(L, np.array([[2]], np.int32), None, 0,
                                           np.zeros(1, np.int32), np.ones(1, np.float32))
    assert alen[0] == 1 and tok[0].tolist() == [2, 1]
    tok, alen, _, _, _ = oracle_mod.accept(L, np.array([[4]], np.int32), None, 0,
                                           np.zeros(1, np.int32), np.ones(1, np.float32))
    assert alen[0] == 0 and tok[0].tolist() == [2, -1]


# --------------------------------------------------------------------------
# Speculative sampling
# --------------------------------------------------------------------------

def _softmax(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def _chi2_ok(samples, probs, n_min=5):
    counts = np.bincount(samples, minlength=len(probs)).astype(np.float64)
    exp = probs * counts.sum()
    keep = exp >= n_min
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    return stats.chisquare(obs, ex).pvalue


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_sampling_first_token_follows_target(oracle_mod, T):
    """Speculative sampling emits a first token distributed as p_0 = softmax(l_0/T)."""
    rng = np.random.default_rng(11)
    B, k, V = 200_000, 2, 8
    l0 = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    dl = (l0[:k] + rng.normal(0, 1.0, (k, V))).astype(np.float32)
    q = _softmax(dl.astype(np.float64) / T).astype(np.float32)
    L = np.broadcast_to(l0, (B, k + 1, V))
    Q = np.broadcast_to(q, (B, k, V))
    d = np.stack([rng.choice(V, B, p=q[j] / q[j].sum()) for j in range(k)], 1).astype(np.int32)
    tok, alen, margin, gap, rc = oracle_mod.accept(L, d, Q, 1234, np.ones(B, np.int32),
                                                   np.full(B, T, np.float32))
    assert rc == 0
    p0 = _softmax(l0[0].astype(np.float64) / T)
    assert _chi2_ok(tok[:, 0], p0) > 1e-3
    # given d_0 accepted, the second token follows p_1
    sel = alen >= 1
    p1 = _softmax(l0[1].astype(np.float64) / T)
    assert _chi2_ok(tok[sel, 1], p1) > 1e-3
    # and the plain acceptance rate equals sum_x min(p, q)
    acc_rate = np.mean(alen >= 1)
    want = np.minimum(p0, q[0].astype(np.float64)).sum()
    assert abs(acc_rate - want) < 5 * np.sqrt(want * (1 - want) / B)
    # an unrelated statistic must fail the same test (the check has power)
    assert _chi2_ok(tok[:, 0], q[0].astype(np.float64) / q[0].sum()) < 1e-3


def test_sampling_bonus_token_follows_last_target_row(oracle_mod):
    """With q = p every draft is accepted and the bonus token follows p_k."""
    rng = np.random.default_rng(12)
    B, k, V = 100_000, 2, 16
    L = np.zeros((B, k + 1, V), np.float32)  # p_j uniform: 1/16 exactly
    lk = rng.normal(0, 1.0, V).astype(np.float32)
    L[:, k] = lk
    Q = np.full((B, k, V), 1.0 / 16, np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    tok, alen, _, _, _ = oracle_mod.accept(L, d, Q, 99, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.all(alen == k)
    assert np.array_equal(tok[:, :k], d)
    assert _chi2_ok(tok[:, k], _softmax(lk.astype(np.float64))) > 1e-3


def test_race_with_mass_spread_over_the_vocabulary_follows_target(oracle_mod):
    """The bonus token follows p_k when its mass sits on a few entries far apart in the
    vocabulary (both ends, and both sides of multiples of 4, 1024 and 8192)."""
    B, k, V = 20000, 1, 20000
    support = np.array([5, 4100, 8191, 8192, 12000, 19999])
    lk = np.full(V, -1e30, np.float32)
    lk[support] = np.array([0.0, 0.5, -0.3, 1.0, 0.2, -1.0], np.float32)
    L = np.zeros((B, k + 1, V), np.float32)
    L[:, k] = lk
    d = np.full((B, k), 7, np.int32)
    Q = np.zeros((B, k, V), np.float32)
    Q[:, 0, 7] = 1e-30  # u q < p always: the draft is kept, the bonus is raced
    tok, alen, _, _, _ = oracle_mod.accept(L, d, Q, 4242, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.all(alen == k)
    p = _softmax(lk[support].astype(np.float64))
    idx = np.searchsorted(support, tok[:, k])
    assert np.all(support[idx] == tok[:, k])
    assert _chi2_ok(idx, p) > 1e-3


def test_sampling_zero_target_probability_always_rejects(oracle_mod):
    B, k, V = 1000, 3, 10
    L = np.zeros((B, k + 1, V), np.float32)
    L[:, 0, 3] = -1e30  # p_0(3) = 0
    Q = np.full((B, k, V), 0.1, np.float32)
    d = np.full((B, k), 3, np.int32)
    tok, alen, _, _, _ = oracle_mod.accept(L, d, Q, 5, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.all(alen == 0)
    assert np.all(tok[:, 0] != 3) and np.all(tok[:, 1:] == -1)


def test_sampling_residual_support(oracle_mod):
    """p = (1/2, 1/2, 0, ...), q = (1/4, 3/4, 0, ...): a rejected draft 1 resamples token 0."""
    B, k, V = 20_000, 1, 4
    L = np.full((B, k + 1, V), -1e30, np.float32)
    L[:, 0, 0] = 0.0
    L[:, 0, 1] = 0.0
    L[:, 1, :] = 0.0
    Q = np.zeros((B, k, V), np.float32)
    Q[:, 0, 0], Q[:, 0, 1] = 0.25, 0.75
    d = np.ones((B, k), np.int32)
    tok, alen, _, _, _ = oracle_mod.accept(L, d, Q, 7, np.ones(B, np.int32), np.ones(B, np.float32))
    rej = alen == 0
    assert np.all(tok[rej, 0] == 0)
    # P(accept) = p/q = 2/3
    assert abs(np.mean(~rej) - 2 / 3) < 0.02


def test_sampling_without_draft_probs_is_one_hot(oracle_mod):
    """No draft distribution: q is one-hot at the drafted token, so a draft is kept
    with probability p(d) and a rejection draws from p with d removed."""
    rng = np.random.default_rng(31)
    B, k, V = 100_000, 1, 8
    l0 = rng.normal(0, 1.0, V).astype(np.float32)
    l1 = rng.normal(0, 1.0, V).astype(np.float32)
    L = np.broadcast_to(np.stack([l0, l1]), (B, k + 1, V))
    d = np.full((B, k), 2, np.int32)
    tok, alen, _, _, rc = oracle_mod.accept(L, d, None, 77, np.ones(B, np.int32), np.ones(B, np.float32))
    assert rc == 0
    p0 = _softmax(l0.astype(np.float64))
    acc = alen == 1
    assert abs(acc.mean() - p0[2]) < 5 * np.sqrt(p0[2] * (1 - p0[2]) / B)
    # rejected rows: never the draft, distributed as p0 without entry 2
    rej_tok = tok[~acc, 0]
    assert np.all(rej_tok != 2)
    resid = p0.copy()
    resid[2] = 0.0
    resid /= resid.sum()
    assert _chi2_ok(rej_tok, resid) > 1e-3
    assert _chi2_ok(rej_tok, p0) < 1e-3  # keeping d's mass must fail: the check has power
    # accepted rows: the bonus token follows p_1
    assert np.all(tok[acc, 0] == 2)
    assert _chi2_ok(tok[acc, 1], _softmax(l1.astype(np.float64))) > 1e-3


def test_sampling_without_draft_probs_equals_explicit_one_hot(oracle_mod):
    rng = np.random.default_rng(32)
    B, k, V = 64, 3, 50
    L = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    Q = np.zeros((B, k, V), np.float32)
    np.put_along_axis(Q, d[:, :, None], 1.0, axis=2)
    temp = rng.uniform(0.5, 1.5, B).astype(np.float32)
    a = oracle_mod.accept(L, d, None, 5, np.ones(B, np.int32), temp)
    b = oracle_mod.accept(L, d, Q, 5, np.ones(B, np.int32), temp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_sampling_uniform_uses_documented_counter(oracle_mod):
    """u_j is word 0 of Philox counter (0, j, b, 0) under key (seed lo, seed hi)."""
    B, k, V = 64, 2, 4
    seed = 0x0123456789ABCDEF
    L = np.zeros((B, k + 1, V), np.float32)
    L[:, 0, :] = np.log(np.array([0.5, 0.2, 0.2, 0.1], np.float32))
    Q = np.zeros((B, k, V), np.float32)
    Q[:, :, 0] = 1.0  # one-hot q: accept draft 0 iff u_0 < p_0(0) = 0.5
    d = np.zeros((B, k), np.int32)
    tok, alen, _, _, _ = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), np.ones(B, np.float32))
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for b in range(B):
        u0 = oracle_mod.uniform(oracle_mod.philox4x32_10([0, 0, b, 0], key)[0])
        assert (alen[b] >= 1) == (u0 < 0.5)


@pytest.mark.parametrize("V", [16, 20001])
def test_final_draw_follows_documented_race(oracle_mod, V):
    """With every draft accepted the bonus token comes from the documented race: the
    entry x with the largest p_k(x) / E_x, E_x = -ln U of word x mod 4 of Philox counter
    (x/4, k, b, 1); replayed here with the library-pinned Philox and numpy's argmax."""
    rng = np.random.default_rng(14)
    B, k = 24, 2
    seed = 777
    L = np.zeros((B, k + 1, V), np.float32)
    L[:, k] = rng.normal(0, 1.5, (B, V)).astype(np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    Q = np.zeros((B, k, V), np.float32)
    Q[np.arange(B)[:, None], np.arange(k)[None, :], d] = 1e-30  # u q < p always: every draft is kept
    tok, alen, _, gap, _ = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.all(alen == k)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for b in range(B):
        if gap[b] < 1e-9:
            continue
        words = np.array([oracle_mod.philox4x32_10([c, k, b, 1], key) for c in range((V + 3) // 4)],
                         np.uint64).reshape(-1)[:V]
        u = ((words >> np.uint64(9)).astype(np.float64) + 0.5) / 8388608.0
        p = _softmax(L[b, k].astype(np.float64))
        assert tok[b, k] == int(np.argmax(p / -np.log(u)))


def test_race_uses_the_rejected_position_counters(oracle_mod):
    """A rejection at position m races with counters (x/4, m, b, 1): a one-hot draft
    rejected at m = 1 draws from p_1 with the draft removed, keyed on m = 1, not 0."""
    rng = np.random.default_rng(17)
    B, k, V = 16, 2, 64
    seed = 4321
    L = np.zeros((B, k + 1, V), np.float32)
    L[:, 1] = rng.normal(0, 1.0, (B, V)).astype(np.float32)
    d = np.zeros((B, k), np.int32)
    d[:, 1] = 5
    L[:, 1, 5] = -1e30  # p_1(5) = 0: draft 1 is always rejected
    Q = np.zeros((B, k, V), np.float32)
    Q[:, 0, 0] = 1e-30  # draft 0 is always kept
    Q[:, 1, 5] = 1.0
    tok, alen, _, gap, _ = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.all(alen == 1)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for b in range(B):
        words = np.array([oracle_mod.philox4x32_10([c, 1, b, 1], key) for c in range(V // 4)],
                         np.uint64).reshape(-1)
        u = ((words >> np.uint64(9)).astype(np.float64) + 0.5) / 8388608.0
        w = np.maximum(_softmax(L[b, 1].astype(np.float64)) - Q[b, 1].astype(np.float64), 0.0)
        assert tok[b, 1] == int(np.argmax(np.where(w > 0, w / -np.log(u), -1.0)))


def test_sampling_is_deterministic_per_seed(oracle_mod):
    rng = np.random.default_rng(13)
    B, k, V = 256, 3, 64
    L = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    Q = _softmax(L[:, :k] + rng.normal(0, 1, (B, k, V))).astype(np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    args = (L, d, Q)
    a = oracle_mod.accept(*args, 42, np.ones(B, np.int32), np.ones(B, np.float32))
    b = oracle_mod.accept(*args, 42, np.ones(B, np.int32), np.ones(B, np.float32))
    c = oracle_mod.accept(*args, 43, np.ones(B, np.int32), np.ones(B, np.float32))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[0], c[0])


def test_mixed_rows_equal_single_mode_rows(oracle_mod):
    """Rows are independent: in a batch that mixes greedy and sampling rows with per-row
    temperatures (the serving configuration), every row's tokens and accept length equal those
    of the same row (same index, so the same Philox counters) in a batch run wholly in its mode,
    and a sampling row's equal those it gets when every row of the batch has its temperature. A
    mode or temperature read from the wrong row fails the comparison; the last check makes sure
    the temperature changes outcomes at all, so the comparison has power."""
    rng = np.random.default_rng(17)
    B, k, V = 48, 3, 97
    L = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    temp = rng.uniform(0.5, 1.2, B).astype(np.float32)
    Q = _softmax((L[:, :k] + rng.normal(0, 1, (B, k, V))) / temp[:, None, None]).astype(np.float32)
    q64 = Q.astype(np.float64)
    q64 /= q64.sum(-1, keepdims=True)
    d = np.array([[rng.choice(V, p=q64[b, j]) for j in range(k)] for b in range(B)], np.int32)
    mode = (rng.random(B) < 0.5).astype(np.int32)
    assert 0 < mode.sum() < B
    seed = 7
    tok, alen = oracle_mod.accept(L, d, Q, seed, mode, temp)[:2]
    tg, ag = oracle_mod.accept(L, d, Q, seed, np.zeros(B, np.int32), temp)[:2]
    ts, as_ = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), temp)[:2]
    for b in range(B):
        rt, ra = (ts, as_) if mode[b] else (tg, ag)
        assert np.array_equal(tok[b], rt[b]) and alen[b] == ra[b], b
    assert len(set(alen.tolist())) > 1  # a mix of accept lengths, not a degenerate batch
    changed = 0
    for b in np.nonzero(mode)[0][:8]:
        tu, au = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), np.full(B, temp[b], np.float32))[:2]
        assert np.array_equal(tok[b], tu[b]) and alen[b] == au[b], b
        tw, aw = oracle_mod.accept(L, d, Q, seed, np.ones(B, np.int32), np.full(B, 4 * temp[b], np.float32))[:2]
        changed += int(not np.array_equal(tok[b], tw[b]) or alen[b] != aw[b])
    assert changed > 0


def test_accept_invalid_rows(oracle_mod):
    B, k, V = 3, 2, 5
    L = np.zeros((B, k + 1, V), np.float32)
    Q = np.full((B, k, V), 0.2, np.float32)
    d = np.array([[0, 1], [5, 0], [1, 1]], np.int32)
    temp = np.array([1.0, 1.0, 0.0], np.float32)
    tok, alen, _, _, rc = oracle_mod.accept(L, d, Q, 1, np.array([1, 1, 1], np.int32), temp, check=False)
    assert rc != 0
    assert alen[0] >= 0 and alen[1] == -1 and alen[2] == -1
    assert np.all(tok[1] == -1) and np.all(tok[2] == -1)


# --------------------------------------------------------------------------
# State commit
# --------------------------------------------------------------------------

def test_commit_picks_accepted_slot(oracle_mod):
    rng = np.random.default_rng(20)
    L, B, S, E = 3, 5, 4, 12
    snaps = rng.standard_normal((L, B, S, E)).astype(np.float32)
    alen = np.array([0, 3, 1, 2, 3], np.int32)  # 3 = k: the last snapshot
    live = np.zeros((L, B, E), np.float32)
    assert oracle_mod.commit_state(snaps, alen, live) == 0
    for l in range(L):
        for b in range(B):
            assert np.array_equal(live[l, b], snaps[l, b, alen[b]])
    assert np.array_equal(live[:, 1], snaps[:, 1, S - 1])
    assert np.array_equal(live[:, 0], snaps[:, 0, 0])


def test_commit_aligned_windows(oracle_mod):
    """Token-indexed windows keep slot m, last-aligned windows slot W - n + m; with
    W = n both are the plain commit, and a fully accepted step keeps slot W - 1 of a
    last-aligned window (the state after its last token)."""
    rng = np.random.default_rng(21)
    L, B, W, E, n = 2, 6, 7, 5, 4
    snaps = rng.standard_normal((L, B, W, E)).astype(np.float32)
    # tag every slot with its index so the chosen slot can be read back
    snaps[..., 0] = np.arange(W, dtype=np.float32)[None, None, :]
    alen = np.array([0, 1, 2, 3, 3, 0], np.int32)
    for alignment, base in ((0, 0), (1, W - n)):
        live = np.zeros((L, B, E), np.float32)
        assert oracle_mod.commit_state_aligned(snaps, alen, live, n, alignment) == 0
        assert np.array_equal(live[..., 0], np.broadcast_to((base + alen).astype(np.float32), (L, B)))
        for l in range(L):
            for b in range(B):
                assert np.array_equal(live[l, b], snaps[l, b, base + alen[b]])
    live = np.zeros((L, B, E), np.float32)
    oracle_mod.commit_state_aligned(snaps, np.full(B, n - 1, np.int32), live, n, 1)
    assert np.all(live[..., 0] == W - 1)
    # W = n: both alignments equal the plain commit
    sq = snaps[:, :, :n].copy()
    ref = np.zeros((L, B, E), np.float32)
    oracle_mod.commit_state(sq, alen, ref)
    for alignment in (0, 1):
        live = np.zeros((L, B, E), np.float32)
        oracle_mod.commit_state_aligned(sq, alen, live, n, alignment)
        assert np.array_equal(live, ref)
    # accept_len must lie in [0, n-1]; the row is skipped and reported
    live = np.full((L, B, E), 9.0, np.float32)
    bad = alen.copy()
    bad[2] = n
    rc = oracle_mod.commit_state_aligned(snaps, bad, live, n, 1, check=False)
    assert rc != 0 and np.all(live[:, 2] == 9.0)


def _pool_tables(rng, L, B, W):
    """A pool of L*B*(W+1) rows dealt out at random: one live row and W window rows per (l, b)."""
    perm = rng.permutation(L * B * (W + 1)).astype(np.int32)
    return perm[:L * B].reshape(L, B).copy(), perm[L * B:].reshape(L, B, W).copy()


def test_commit_select_stages_the_copied_state(oracle_mod):
    """Selecting the checkpoint row leaves, as the live state of every (l, b), exactly
    the state the copying commit writes; rows never move between (l, b) units, the
    tables stay a permutation of the pool, and a row with an invalid accept_len
    keeps both tables."""
    rng = np.random.default_rng(5)
    L, B, W, E, n = 3, 7, 6, 5, 4
    pool = rng.standard_normal((L * B * (W + 1), E)).astype(np.float32)
    for alignment in (0, 1):
        live_row, ckpt_rows = _pool_tables(rng, L, B, W)
        alen = rng.integers(0, n, B).astype(np.int32)
        alen[2] = n  # out of range: skipped and reported
        expect = pool[live_row].copy()
        rc_copy = oracle_mod.commit_state_aligned(pool[ckpt_rows], alen, expect, n, alignment, check=False)
        lr, cr = live_row.copy(), ckpt_rows.copy()
        rc = oracle_mod.commit_select(alen, lr, cr, n, alignment, check=False)
        assert rc == rc_copy != 0
        assert np.array_equal(pool[lr], expect)
        assert np.array_equal(lr[:, 2], live_row[:, 2]) and np.array_equal(cr[:, 2], ckpt_rows[:, 2])
        for l in range(L):
            for b in range(B):
                before = np.sort(np.append(ckpt_rows[l, b], live_row[l, b]))
                after = np.sort(np.append(cr[l, b], lr[l, b]))
                assert np.array_equal(before, after)
                assert lr[l, b] not in cr[l, b]


def test_commit_select_follows_copying_commit_over_steps(oracle_mod):
    """A run of verify steps: each writes its checkpoints into the window rows (a
    function of the live state it starts from and fresh inputs) and commits. The
    pool's live rows track, bit for bit, a second run that copies states, so no
    step's checkpoint writes ever reach the live state it started from."""
    rng = np.random.default_rng(8)
    L, B, W, E, n = 2, 5, 5, 3, 4
    pool = np.zeros((L * B * (W + 1), E), np.float32)
    live_row, ckpt_rows = _pool_tables(rng, L, B, W)
    live_copy = rng.standard_normal((L, B, E)).astype(np.float32)
    pool[live_row] = live_copy
    for step in range(6):
        alignment = step % 2
        inputs = rng.standard_normal((L, B, W, E)).astype(np.float32)
        # checkpoints of this step: the starting state plus a running sum of inputs
        snaps_copy = live_copy[:, :, None, :] + np.cumsum(inputs, axis=2)
        pool[ckpt_rows] = pool[live_row][:, :, None, :] + np.cumsum(inputs, axis=2)
        assert np.array_equal(pool[ckpt_rows], snaps_copy)
        alen = rng.integers(0, n, B).astype(np.int32)
        oracle_mod.commit_state_aligned(snaps_copy.astype(np.float32), alen, live_copy, n, alignment)
        oracle_mod.commit_select(alen, live_row, ckpt_rows, n, alignment)
        assert np.array_equal(pool[live_row], live_copy)


def test_commit_skips_invalid_rows(oracle_mod):
    rng = np.random.default_rng(21)
    L, B, S, E = 2, 3, 4, 8
    snaps = rng.standard_normal((L, B, S, E)).astype(np.float32)
    live = np.full((L, B, E), 7.0, np.float32)
    rc = oracle_mod.commit_state(snaps, np.array([1, 4, -1], np.int32), live, check=False)
    assert rc == -7
    assert np.array_equal(live[:, 0], snaps[:, 0, 1])
    assert np.all(live[:, 1:] == 7.0)


# ---------------------------------------------------------------------------
# gated delta rule over the verify chain
# ---------------------------------------------------------------------------
def _gdn_inputs(rng, B, R, H, dk, dv, unit_keys=True):
    q = rng.standard_normal((B, R, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, R, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, R, H, dv)).astype(np.float32)
    g = -rng.uniform(0.0, 1.0, (B, R, H)).astype(np.float32)
    beta = rng.uniform(0.05, 1.0, (B, R, H)).astype(np.float32)
    s0 = rng.standard_normal((B, H, dv, dk)).astype(np.float32)
    return q, k.astype(np.float32), v, g, beta, s0


def test_gdn_pure_decay_closed_form(oracle_mod):
    """beta = 0: the state only decays, S_t = exp(g_0 + ... + g_t) S_0, and o_t = S_t (scale q_t)."""
    rng = np.random.default_rng(70)
    B, R, H, dk, dv = 2, 4, 3, 8, 5
    q, k, v, g, beta, s0 = _gdn_inputs(rng, B, R, H, dk, dv)
    beta[:] = 0
    snaps, out, _ = oracle_mod.gdn_verify(q, k, v, g, beta, s0, scale=0.25)
    decay = np.exp(np.cumsum(g.astype(np.float64), axis=1))  # [B,R,H]
    expect = decay[:, :, :, None, None] * s0.astype(np.float64)[:, None]
    np.testing.assert_allclose(snaps, expect, rtol=1e-6, atol=1e-7)
    o = np.einsum("brhij,brhj->brhi", expect, 0.25 * q.astype(np.float64))
    np.testing.assert_allclose(out, o, rtol=1e-5, atol=1e-6)


def test_gdn_delta_rule_on_the_key_direction(oracle_mod):
    """With unit keys the update moves S k_t to (1 - beta) alpha S_{t-1} k_t + beta v_t
    and only decays every direction orthogonal to k_t (the rule's rank-one form)."""
    rng = np.random.default_rng(71)
    B, R, H, dk, dv = 3, 5, 2, 16, 12
    q, k, v, g, beta, s0 = _gdn_inputs(rng, B, R, H, dk, dv)
    snaps, _, _ = oracle_mod.gdn_verify(q, k, v, g, beta, s0, scale=1.0)
    for b in range(B):
        for h in range(H):
            prev = s0[b, h].astype(np.float64)
            for t in range(R):
                kt = k[b, t, h].astype(np.float64)
                a, bt = np.exp(float(g[b, t, h])), float(beta[b, t, h])
                cur = snaps[b, t, h].astype(np.float64)
                np.testing.assert_allclose(cur @ kt, (1 - bt) * a * (prev @ kt) + bt * v[b, t, h], rtol=1e-5,
                                           atol=1e-5)
                w = rng.standard_normal(dk)
                w -= (w @ kt) * kt  # orthogonal to k_t
                np.testing.assert_allclose(cur @ w, a * (prev @ w), rtol=1e-5, atol=1e-5)
                prev = cur


def test_gdn_orthonormal_keys_store_outer_products(oracle_mod):
    """From S_0 = 0 with alpha = beta = 1 and orthonormal keys the state is the sum of
    v_t k_t^T, so querying with k_j / scale returns v_j for every j <= t."""
    rng = np.random.default_rng(72)
    B, R, H, dk, dv = 1, 4, 2, 8, 6
    _, _, v, g, beta, s0 = _gdn_inputs(rng, B, R, H, dk, dv)
    basis = np.linalg.qr(rng.standard_normal((H, dk, dk)))[0]  # orthonormal columns per head
    k = np.transpose(basis[:, :, :R], (2, 0, 1))[None].astype(np.float32)  # [1,R,H,dk]
    g[:], beta[:], s0[:] = 0, 1, 0
    scale = 0.5
    q = (k[:, :1].repeat(R, axis=1) / scale).astype(np.float32)  # every token queries k_0
    snaps, out, _ = oracle_mod.gdn_verify(q, k, v, g, beta, s0, scale=scale)
    full = sum(np.einsum("hi,hc->hic", v[0, t].astype(np.float64), k[0, t].astype(np.float64)) for t in range(R))
    np.testing.assert_allclose(snaps[0, R - 1], full, atol=1e-6)
    np.testing.assert_allclose(out[0], np.broadcast_to(v[0, 0], (R, H, dv)), atol=1e-5)


def test_gdn_chain_splits_and_windows(oracle_mod):
    """One call over R tokens equals R one-token calls carrying the state; a window
    wider than the chain holds the same states at slots t (token alignment) or
    W - R + t (last alignment) and leaves its other slots untouched."""
    rng = np.random.default_rng(73)
    B, R, H, dk, dv = 2, 4, 2, 8, 8
    q, k, v, g, beta, s0 = _gdn_inputs(rng, B, R, H, dk, dv, unit_keys=False)
    snaps, out, _ = oracle_mod.gdn_verify(q, k, v, g, beta, s0, scale=0.3)
    state = s0
    for t in range(R):
        sl = slice(t, t + 1)
        s1, o1, _ = oracle_mod.gdn_verify(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], state, scale=0.3)
        np.testing.assert_allclose(s1[:, 0], snaps[:, t], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(o1[:, 0], out[:, t], rtol=1e-5, atol=1e-5)
        state = s1[:, 0]
    W = R + 3
    for alignment, base in ((0, 0), (1, W - R)):
        sw, ow, _ = oracle_mod.gdn_verify(q, k, v, g, beta, s0, scale=0.3, num_slots=W, alignment=alignment)
        assert np.array_equal(sw[:, base:base + R], snaps) and np.array_equal(ow, out)
        rest = np.delete(sw, np.arange(base, base + R), axis=1)
        assert not rest.any()
