"""spec_verify_attention_noalloc: the allocation-free form of verify attention.

Some callers may not allocate device memory when they call the library (an
engine's per-step enqueue path, a runtime plugin whose enqueue contract
forbids allocation, a process that reserved all device memory up front).
For them the library keeps its attention scratch in a fixed array and offers
this entry point without a workspace argument. The tests call it through the
C ABI three times in a row on two alternating inputs of the same shapes (each
call reuses the array the previous one left behind) and require every result
to equal, bit for bit, the workspace form of the same call (same kernel, same
grid, same split plan), and the oracle within the attention tolerance.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import ATTN_MAX_ABS, ATTN_REL_L2, attention_errors, oracle_attention_for
from speculative_decoding_verification_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _call_noalloc(sv, lib, a, w, out, err):
    d = sv._attn_desc(a["q"], a["k_cache"], a["block_table"])
    return lib.spec_verify_attention_noalloc(
        ctypes.c_void_p(a["q"].data_ptr()), ctypes.c_void_p(a["k_cache"].data_ptr()),
        ctypes.c_void_p(a["v_cache"].data_ptr()), ctypes.c_void_p(a["block_table"].data_ptr()),
        ctypes.c_void_p(a["ctx_lens"].data_ptr()), w.k_draft, ctypes.c_void_p(out.data_ptr()), ctypes.byref(d),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _ragged(name):
    """Ragged context mixes, so that units split across CTAs and partial slots are used."""
    w = wl.WORKLOADS[name]
    if name == "llama8b_eagle3":  # mma.sync, 16 packed rows
        return w.replace(batch=12, ctx_lens=(2048, 17, 4, 700, 64, 65, 1999, 2048, 130, 5, 1024, 333))
    if name == "hybrid_gdn":  # D = 256, 24 packed rows: the largest partial slots per CTA
        return w.replace(batch=6, ctx_lens=(4100, 4, 1500, 63, 2049, 777), ctx_range=None)
    if name == "longctx":  # D = 128 with 64 packed rows: the tcgen05 kernel
        return w.replace(batch=2, ctx_lens=(3000, 700), ctx_range=None)
    return w


@pytest.mark.parametrize("name", ["llama8b_eagle3", "tiny", "hybrid_gdn", "longctx"])
def test_noalloc_matches_workspace_calls_alternating_inputs(sv, oracle_mod, name):
    """Three allocation-free calls, on inputs A, B, A of the same shapes (so the same plan and
    the same scratch slots): each equals, bit for bit, the workspace form on its own input, so
    no call reads counters or partials that the previous call left in the scratch."""
    lib = sv.load_library()
    assert lib.spec_verify_attention_noalloc_limit() == 32 << 20
    w = _ragged(name)
    inputs = [wl.make_attention_inputs(w, device=DEV), wl.make_attention_inputs(w, device=DEV, seed=w.seed + 1)]
    shape = (w.batch, w.rows, w.num_q_heads, w.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    refs = []
    for a in inputs:
        ref = torch.empty(shape, dtype=torch.float32, device=DEV)
        sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft,
                                 ref, dev_err=err)
        refs.append(ref)
    outs = []
    for i in (0, 1, 0):
        out = torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)
        rc = _call_noalloc(sv, lib, inputs[i], w, out, err)
        assert rc == 0, sv.status_string(rc)
        outs.append((i, out))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not torch.equal(refs[0], refs[1])
    for i, out in outs:
        assert torch.equal(out, refs[i]), i
    for i in (0, 1):
        mx, rel = attention_errors(refs[i].cpu().numpy(), oracle_attention_for(oracle_mod, inputs[i]))
        assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (i, mx, rel)


@pytest.mark.parametrize("name", ["llama8b_eagle3", "longctx"])
def test_noalloc_small_batch_then_workspace_large_batch(sv, oracle_mod, name):
    """A small allocation-free call, then a larger workspace call of the same kernel
    instance: the first must not leave the kernel's shared-memory limit below what
    the second needs."""
    lib = sv.load_library()
    big = _ragged(name)
    small = big.replace(batch=1, ctx_lens=big.ctx_lens[:1])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    a_s = wl.make_attention_inputs(small, device=DEV)
    out_s = torch.empty((small.batch, small.rows, small.num_q_heads, small.head_dim), device=DEV)
    assert _call_noalloc(sv, lib, a_s, small, out_s, err) == 0
    a_b = wl.make_attention_inputs(big, device=DEV, seed=big.seed + 5)
    out_b = torch.empty((big.batch, big.rows, big.num_q_heads, big.head_dim), device=DEV)
    sv.spec_verify_attention(a_b["q"], a_b["k_cache"], a_b["v_cache"], a_b["block_table"], a_b["ctx_lens"],
                             big.k_draft, out_b, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for a, out in ((a_s, out_s), (a_b, out_b)):
        mx, rel = attention_errors(out.cpu().numpy(), oracle_attention_for(oracle_mod, a))
        assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)
    assert np.isfinite(out_b.cpu().numpy()).all()


def test_noalloc_rejects_shapes_beyond_its_scratch(sv):
    lib = sv.load_library()
    # 4096 sequences x 4096 kv heads: the arrival counters alone (64 MiB) exceed the
    # scratch, so the call is rejected on the host before anything reaches the GPU
    d = sv._AttnDesc(4096, 4096, 4096, 128, 64, 4, 1 << 16)
    fake = ctypes.c_void_p(256)
    rc = lib.spec_verify_attention_noalloc(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(d), None, None)
    assert rc == -5 and "fixed scratch" in sv.status_string(rc)
