"""spec_verify_attention_noalloc: the allocation-free form of verify attention.

Some callers may not allocate device memory when they call the library (an
engine's per-step enqueue path, a runtime plugin whose enqueue contract
forbids allocation, a process that reserved all device memory up front).
For them the library keeps its attention scratch in a fixed array and offers
this entry point without a workspace argument. The test calls it through the
C ABI twice in a row (the second call reuses the array the first left behind)
and checks both results against the workspace form of the same call.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import pytest
import torch

from helpers import ATTN_MAX_ABS, ATTN_REL_L2, attention_errors
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


@pytest.mark.parametrize("name", ["llama8b_eagle3", "tiny"])
def test_noalloc_matches_workspace_call_twice(sv, name):
    lib = sv.load_library()
    assert lib.spec_verify_attention_noalloc_limit() == 32 << 20
    w = wl.WORKLOADS[name]
    if name == "llama8b_eagle3":  # ragged lengths so that units split across CTAs
        w = w.replace(batch=12, ctx_lens=(2048, 17, 4, 700, 64, 65, 1999, 2048, 130, 5, 1024, 333))
    a = wl.make_attention_inputs(w, device=DEV)
    shape = (w.batch, w.rows, w.num_q_heads, w.head_dim)
    ref = torch.empty(shape, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft, ref,
                             dev_err=err)
    outs = []
    for _ in range(2):
        out = torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)
        rc = _call_noalloc(sv, lib, a, w, out, err)
        assert rc == 0, sv.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for out in outs:
        mx, rel = attention_errors(out.cpu().numpy(), ref.cpu().double().numpy())
        assert mx <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (mx, rel)


def test_noalloc_rejects_shapes_beyond_its_scratch(sv):
    lib = sv.load_library()
    # 4096 sequences x 4096 kv heads: the arrival counters alone (64 MiB) exceed the
    # scratch, so the call is rejected on the host before anything reaches the GPU
    d = sv._AttnDesc(4096, 4096, 4096, 128, 64, 4, 1 << 16)
    fake = ctypes.c_void_p(256)
    rc = lib.spec_verify_attention_noalloc(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(d), None, None)
    assert rc == -5 and "fixed scratch" in sv.status_string(rc)
