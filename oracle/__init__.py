"""CPU oracle of the speculative-decoding verify step (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never does: the two
share no code, and the CUDA path fails loudly when its extension is missing
instead of falling back to anything here.

The arithmetic lives in ``spec_oracle.c`` (plain C, double precision, OpenMP
over independent units); this module compiles it with gcc on first use and
wraps it for numpy arrays. Each function states the definition it follows;
the C file cites the pages for each step.

Readings of the pages that the oracle fixes (the pages leave them open):
ctx_lens counts the verify tokens; row i sits at absolute position
ctx - (k+1) + i; GQA groups are contiguous; softmax scale 1/sqrt(D); greedy
ties go to the lowest index; acceptance compares u*q < p; the residual falls
back to p when max(0, p-q) is all zero; without draft probabilities q is one-hot
at the drafted token; the correction/bonus draw is an
exponential race keyed by Philox words as documented in spec_verify.h; the
zero-copy commit exchanges the live row with the chosen checkpoint row of a
state pool; the gated delta rule (from the published Gated DeltaNet method,
which the pages name but do not state) takes log-decay gates g and write
strengths beta as inputs, keeps a V-major dv x dk state and scales q by the
given factor.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspec_oracle.so")

_lock = threading.Lock()
_lib = None

ERRORS = {
    0: "ok",
    -1: "invalid argument",
    -5: "block id out of range",
    -6: "context length out of range",
    -7: "accept_len out of range",
    -8: "draft token out of range",
    -9: "temperature not > 0",
    -10: "out of memory",
}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned {code} ({ERRORS.get(code, 'unknown')})")
        self.code = code


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into oracle/_build/libspec_oracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_uniform.argtypes = [ctypes.c_uint32]
        lib.oracle_uniform.restype = ctypes.c_double
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        lib.oracle_verify_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                                i32, P, i32, P, i32]
        lib.oracle_verify_attention.restype = i32
        lib.oracle_accept.argtypes = [P, P, P, u64, P, P, i32, i32, i32, P, P, P, P, i32]
        lib.oracle_accept.restype = i32
        lib.oracle_commit_state.argtypes = [P, P, P, i32, i32, i32, i64, i32]
        lib.oracle_commit_state.restype = i32
        lib.oracle_commit_state_aligned.argtypes = [P, P, P, i32, i32, i32, i64, i32, i32, i32]
        lib.oracle_commit_state_aligned.restype = i32
        lib.oracle_commit_select.argtypes = [P, P, P, i32, i32, i32, i32, i32]
        lib.oracle_commit_select.restype = i32
        lib.oracle_gdn_verify.argtypes = [P, P, P, P, P, ctypes.c_double, P, P, P, i32, i32, i32, i32, i32, i32,
                                          i32, i32]
        lib.oracle_gdn_verify.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().oracle_max_threads())


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 block function (Salmon et al., SC'11) on one counter/key."""
    lib = _load()
    c = _c(counter, np.uint32)
    k = _c(key, np.uint32)
    assert c.shape == (4,) and k.shape == (2,)
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(word: int) -> float:
    """((word >> 9) + 0.5) * 2^-23, a uniform in (0, 1)."""
    return float(_load().oracle_uniform(int(word) & 0xFFFFFFFF))


def verify_attention(q_bits, k_bits, v_bits, block_table, ctx_lens, *, seqs=None,
                     n_threads: int = 0, check: bool = True) -> np.ndarray:
    """Paged GQA verify attention, double precision.

    q_bits [B,R,Hq,D] and k_bits/v_bits [num_blocks,bs,Hkv,D] hold bf16 bit
    patterns (uint16). Returns out [len(seqs) or B, R, Hq, D] float64 for the
    listed sequences. Row i of sequence b attends keys t <= ctx_b - R + i.
    """
    lib = _load()
    q = _c(q_bits, np.uint16)
    kc = _c(k_bits, np.uint16)
    vc = _c(v_bits, np.uint16)
    bt = _c(block_table, np.int32)
    cl = _c(ctx_lens, np.int32)
    B, R, Hq, D = q.shape
    nb, bs, Hkv, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape and bt.shape[0] == B and cl.shape == (B,)
    s = None if seqs is None else _c(seqs, np.int32)
    n = B if s is None else len(s)
    out = np.zeros((n, R, Hq, D), dtype=np.float64)
    rc = lib.oracle_verify_attention(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), B, R, Hq, Hkv,
                                     D, bs, nb, bt.shape[1], _ptr(s), n, _ptr(out), n_threads)
    if check and rc != 0:
        raise OracleError(rc)
    return out


def accept(target_logits, draft_tokens, draft_probs, seed: int, mode, temperature, *,
           n_threads: int = 0, check: bool = True):
    """Greedy / speculative-sampling acceptance, double precision.

    draft_probs may be None: sampling rows then take the draft distribution as
    one-hot at each drafted token (accept iff u < p(d); the residual is p with
    the rejected token removed).

    Returns (out_tokens [B,k+1] int32, accept_len [B] int32, accept_margin [B],
    race_gap [B], status). accept_margin is the smallest |u - p/q| among the
    drafts tested; race_gap the relative gap between the two largest race keys.
    """
    lib = _load()
    L = _c(target_logits, np.float32)
    d = _c(draft_tokens, np.int32)
    qp = None if draft_probs is None else _c(draft_probs, np.float32)
    md = _c(mode, np.int32)
    tp = _c(temperature, np.float32)
    B, R, V = L.shape
    k = R - 1
    assert d.shape == (B, k) and md.shape == (B,) and tp.shape == (B,)
    if qp is not None:
        assert qp.shape == (B, k, V)
    tok = np.zeros((B, R), dtype=np.int32)
    alen = np.zeros(B, dtype=np.int32)
    margin = np.zeros(B, dtype=np.float64)
    gap = np.zeros(B, dtype=np.float64)
    rc = lib.oracle_accept(_ptr(L), _ptr(d), _ptr(qp), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(md),
                           _ptr(tp), B, k, V, _ptr(tok), _ptr(alen), _ptr(margin), _ptr(gap),
                           n_threads)
    if check and rc != 0:
        raise OracleError(rc)
    return tok, alen, margin, gap, rc


def commit_state(snapshots, accept_len, live, *, n_threads: int = 0, check: bool = True):
    """live[l,b,:] = snapshots[l,b,accept_len[b],:] (in place on `live`); returns the status."""
    lib = _load()
    sn = _c(snapshots, np.float32)
    al = _c(accept_len, np.int32)
    assert live.dtype == np.float32 and live.flags.c_contiguous
    L, B, S, E = sn.shape
    assert live.shape == (L, B, E) and al.shape == (B,)
    rc = lib.oracle_commit_state(_ptr(sn), _ptr(al), _ptr(live), L, B, S, E, n_threads)
    if check and rc != 0:
        raise OracleError(rc)
    return rc


def commit_state_aligned(snapshots, accept_len, live, n_tokens: int, alignment: int, *, n_threads: int = 0,
                         check: bool = True):
    """Windowed checkpoints: snapshots [L,B,W,E] for a step of n_tokens <= W tokens.

    alignment 0: slot j holds the state after token j (slot = accept_len);
    alignment 1: slot W-1 holds the state after the last token
    (slot = W - n_tokens + accept_len). In place on `live`; returns the status.
    """
    lib = _load()
    sn = _c(snapshots, np.float32)
    al = _c(accept_len, np.int32)
    assert live.dtype == np.float32 and live.flags.c_contiguous
    L, B, W, E = sn.shape
    assert live.shape == (L, B, E) and al.shape == (B,)
    rc = lib.oracle_commit_state_aligned(_ptr(sn), _ptr(al), _ptr(live), L, B, W, E, int(n_tokens),
                                         int(alignment), n_threads)
    if check and rc != 0:
        raise OracleError(rc)
    return rc


def commit_select(accept_len, live_row, ckpt_rows, n_tokens: int, alignment: int, *, check: bool = True):
    """Commit by row selection in a state pool: live_row [L,B] and ckpt_rows [L,B,W]
    int32 pool-row indices, updated in place.

    The slot of the accepted prefix (as in commit_state_aligned) trades places
    with the live row: live_row[l,b] <-> ckpt_rows[l,b,slot]. Returns the status.
    """
    lib = _load()
    al = _c(accept_len, np.int32)
    for t in (live_row, ckpt_rows):
        assert t.dtype == np.int32 and t.flags.c_contiguous
    L, B = live_row.shape
    assert ckpt_rows.shape[:2] == (L, B) and al.shape == (B,)
    W = ckpt_rows.shape[2]
    rc = lib.oracle_commit_select(_ptr(al), _ptr(live_row), _ptr(ckpt_rows), L, B, W, int(n_tokens), int(alignment))
    if check and rc != 0:
        raise OracleError(rc)
    return rc


def gdn_verify(q, k, v, g, beta, state_in, *, scale: float, num_slots: int = 0, alignment: int = 0,
               n_threads: int = 0, check: bool = True):
    """Gated delta rule over a verify chain (double precision).

    q, k [B,R,H,dk]; v [B,R,H,dv]; g (log decay), beta [B,R,H]; state_in [B,H,dv,dk]
    (V-major). Token t: S = exp(g) S + beta (v - exp(g) S k) k^T, o = S (scale q).
    Returns (snapshots [B,W,H,dv,dk] with slot base+t = state after token t, out
    [B,R,H,dv], status); W = num_slots (default R), base 0 (alignment 0) or W - R.
    Slots outside the written range are zero.
    """
    lib = _load()
    q, k, v, g, beta, s0 = (_c(x, np.float32) for x in (q, k, v, g, beta, state_in))
    B, R, H, dk = q.shape
    dv = v.shape[3]
    assert k.shape == q.shape and v.shape == (B, R, H, dv) and g.shape == (B, R, H) and beta.shape == (B, R, H)
    assert s0.shape == (B, H, dv, dk)
    W = int(num_slots) if num_slots else R
    snaps = np.zeros((B, W, H, dv, dk), np.float32)
    out = np.zeros((B, R, H, dv), np.float32)
    rc = lib.oracle_gdn_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(s0), _ptr(snaps),
                               _ptr(out), B, R, H, dk, dv, W, int(alignment), n_threads)
    if check and rc != 0:
        raise OracleError(rc)
    return snaps, out, rc
