"""GB300-native verify step of chain speculative decoding.

A thin ctypes binding over ``libspecverify.so`` (C ABI in ``include/spec_verify.h``).
Every function here only checks shapes and dtypes, then passes device pointers,
sizes and the current CUDA stream to the library of the same name; all of the
step's arithmetic runs in the library's kernels. There is no fallback: if the
library is missing, calls raise.

    spec_verify_attention(q, k_cache, v_cache, block_table, ctx_lens, k_draft, out)
    spec_accept(target_logits, draft_tokens, draft_probs, philox_seed, mode,
                temperature, out_tokens, accept_len)
    spec_commit_state(snapshots, accept_len, live_state)
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import buildlib as _build_mod

__all__ = [
    "SpecError", "build", "library_path", "load_library", "spec_verify_attention",
    "spec_verify_attention_workspace", "new_attention_workspace", "spec_verify_attention_noalloc",
    "spec_verify_attention_plan",
    "spec_accept", "spec_commit_state", "spec_commit_state_aligned", "spec_commit_select", "spec_gdn_verify",
    "spec_gdn_verify_pooled", "status_string",
    "DEVERR", "MODE_GREEDY", "MODE_SAMPLE", "ALIGN_TOKEN", "ALIGN_LAST",
]

MODE_GREEDY = 0
MODE_SAMPLE = 1
DEVERR = {
    "block_id": 1, "token": 2, "accept_len": 4, "ctx_len": 8, "temperature": 16,
    "timeout": 32, "mode": 64, "pool_row": 128,
}

_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({status_string(code)})")
        self.code = code


class _AttnPlan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in
                ("kernel", "m_tiles", "keys_per_tile", "stages", "p_buffers", "ctas_per_sm")]


_ATTN_KERNELS = {1: "mma", 2: "tc"}


class _AttnDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
    ]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libspecverify.so for sm_103a (in-tree)."""
    return _build_mod.build(force=force, verbose=verbose)


def library_path() -> str:
    return _build_mod.LIB


def load_library():
    """Load libspecverify.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build_mod.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(speculative_decoding_verification_paged_gb300.build())")
        lib = ctypes.CDLL(path)
        P, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
        lib.spec_status_string.argtypes = [ctypes.c_int]
        lib.spec_status_string.restype = ctypes.c_char_p
        lib.spec_verify_attention_workspace.argtypes = [ctypes.POINTER(_AttnDesc), i32]
        lib.spec_verify_attention_workspace.restype = sz
        lib.spec_verify_attention.argtypes = [P, P, P, P, P, i32, P, ctypes.POINTER(_AttnDesc), P, sz, P, P]
        lib.spec_verify_attention.restype = ctypes.c_int
        lib.spec_verify_attention_noalloc.argtypes = [P, P, P, P, P, i32, P, ctypes.POINTER(_AttnDesc), P, P]
        lib.spec_verify_attention_noalloc.restype = ctypes.c_int
        lib.spec_verify_attention_noalloc_limit.argtypes = []
        lib.spec_verify_attention_noalloc_limit.restype = sz
        lib.spec_verify_attention_plan.argtypes = [ctypes.POINTER(_AttnDesc), i32, ctypes.POINTER(_AttnPlan)]
        lib.spec_verify_attention_plan.restype = ctypes.c_int
        lib.spec_accept.argtypes = [P, P, P, u64, P, P, P, P, i32, i32, i32, P, P]
        lib.spec_accept.restype = ctypes.c_int
        lib.spec_commit_state.argtypes = [P, P, P, i32, i32, i32, i64, P, P]
        lib.spec_commit_state.restype = ctypes.c_int
        lib.spec_commit_state_aligned.argtypes = [P, P, P, i32, i32, i32, i64, i32, i32, P, P]
        lib.spec_commit_state_aligned.restype = ctypes.c_int
        lib.spec_commit_select.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P]
        lib.spec_commit_select.restype = ctypes.c_int
        lib.spec_gdn_verify.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                         P, P]
        lib.spec_gdn_verify.restype = ctypes.c_int
        lib.spec_gdn_verify_pooled.argtypes = [P, P, P, P, P, ctypes.c_float, P, i64, P, P, P, i32, i32, i32, i32,
                                                i32, i32, i32, P, P]
        lib.spec_gdn_verify_pooled.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().spec_status_string(int(code)).decode()


def _check(fn: str, rc: int):
    if rc != 0:
        raise SpecError(fn, rc)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    """The stream to launch on; it must belong to the current device (the one the
    library launches on)."""
    s = torch.cuda.current_stream() if stream is None else stream
    if s.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {s.device}, the current device is cuda:{torch.cuda.current_device()}")
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the call runs on the current device "
                         f"cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _err_ptr(dev_err: Optional[torch.Tensor]):
    """The optional device error word: an int32 CUDA tensor of at least one element."""
    if dev_err is None:
        return None
    if not isinstance(dev_err, torch.Tensor) or not dev_err.is_cuda or dev_err.dtype != torch.int32 \
            or dev_err.numel() < 1:
        raise ValueError("dev_err must be an int32 CUDA tensor with at least one element")
    if dev_err.device.index != torch.cuda.current_device():
        raise ValueError(f"dev_err is on {dev_err.device}, the call runs on cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(dev_err.data_ptr())


def _attn_desc(q, k_cache, block_table) -> _AttnDesc:
    B, R, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and cache differ")
    return _AttnDesc(B, Hq, Hkv, D, bs, block_table.shape[1], nb)


def spec_verify_attention_workspace(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                                    k_draft: int) -> int:
    """Workspace bytes spec_verify_attention needs for these shapes."""
    d = _attn_desc(q, k_cache, block_table)
    return int(load_library().spec_verify_attention_workspace(ctypes.byref(d), int(k_draft)))


def spec_verify_attention_plan(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                               k_draft: int) -> dict:
    """Which kernel spec_verify_attention launches for these shapes on the current
    device, and its tile settings. Only the tensors' shapes are read (meta tensors
    do); D = 128 with 17 or more packed rows queries the current device."""
    d = _attn_desc(q, k_cache, block_table)
    plan = _AttnPlan()
    _check("spec_verify_attention_plan",
           load_library().spec_verify_attention_plan(ctypes.byref(d), int(k_draft), ctypes.byref(plan)))
    out = {name: int(getattr(plan, name)) for name, _ in _AttnPlan._fields_}
    out["kernel"] = _ATTN_KERNELS[out["kernel"]]
    return out


def new_attention_workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace for spec_verify_attention: zero-filled once, reusable by later calls on one stream."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def spec_verify_attention(q, k_cache, v_cache, block_table, ctx_lens, k_draft: int, out,
                          workspace: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Paged GQA verify attention into `out` [B, k+1, Hq, D] fp32 (see spec_verify.h)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(out, "out", torch.float32, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    B, R, Hq, D = q.shape
    if R != k_draft + 1 or out.shape != q.shape or block_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("inconsistent verify-attention shapes")
    d = _attn_desc(q, k_cache, block_table)
    need = int(lib.spec_verify_attention_workspace(ctypes.byref(d), int(k_draft)))
    if workspace is None:
        workspace = new_attention_workspace(need, q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    rc = lib.spec_verify_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens),
                                   int(k_draft), _ptr(out), ctypes.byref(d), _ptr(workspace),
                                   workspace.numel(), _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_verify_attention", rc)
    return out


def spec_verify_attention_noalloc(q, k_cache, v_cache, block_table, ctx_lens, k_draft: int, out,
                                  dev_err: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """spec_verify_attention without a workspace argument, for callers that may not
    allocate device memory at call time; its scratch is a fixed array inside the
    library (see spec_verify.h for the limit and the rules on overlapping calls)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(out, "out", torch.float32, 4)
    B, R, Hq, D = q.shape
    if v_cache.shape != k_cache.shape or R != k_draft + 1 or out.shape != q.shape \
            or block_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("inconsistent verify-attention shapes")
    d = _attn_desc(q, k_cache, block_table)
    rc = lib.spec_verify_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                           _ptr(ctx_lens), int(k_draft), _ptr(out), ctypes.byref(d),
                                           _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_verify_attention_noalloc", rc)
    return out


def spec_accept(target_logits, draft_tokens, draft_probs, philox_seed: int, mode, temperature, out_tokens,
                accept_len, dev_err: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None):
    """Greedy / speculative-sampling acceptance (see spec_verify.h)."""
    lib = load_library()
    _need(target_logits, "target_logits", torch.float32, 3)
    _need(draft_tokens, "draft_tokens", torch.int32, 2)
    if draft_probs is not None:
        _need(draft_probs, "draft_probs", torch.float32, 3)
    _need(mode, "mode", torch.int32, 1)
    _need(temperature, "temperature", torch.float32, 1)
    _need(out_tokens, "out_tokens", torch.int32, 2)
    _need(accept_len, "accept_len", torch.int32, 1)
    B, R, V = target_logits.shape
    k = R - 1
    if draft_tokens.shape != (B, k) or out_tokens.shape != (B, R) or accept_len.shape != (B,) \
            or mode.shape != (B,) or temperature.shape != (B,):
        raise ValueError("inconsistent acceptance shapes")
    if draft_probs is not None and draft_probs.shape != (B, k, V):
        raise ValueError("draft_probs must be [B, k, V]")
    rc = lib.spec_accept(_ptr(target_logits), _ptr(draft_tokens), _ptr(draft_probs),
                         int(philox_seed) & 0xFFFFFFFFFFFFFFFF, _ptr(mode), _ptr(temperature),
                         _ptr(out_tokens), _ptr(accept_len), B, k, V, _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_accept", rc)
    return out_tokens, accept_len


def spec_commit_state(snapshots, accept_len, live_state, dev_err: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None):
    """live_state[l, b] = snapshots[l, b, accept_len[b]] (see spec_verify.h)."""
    lib = load_library()
    _need(snapshots, "snapshots", torch.float32, 4)
    _need(accept_len, "accept_len", torch.int32, 1)
    _need(live_state, "live_state", torch.float32, 3)
    L, B, S, E = snapshots.shape
    if live_state.shape != (L, B, E) or accept_len.shape != (B,):
        raise ValueError("inconsistent commit shapes")
    rc = lib.spec_commit_state(_ptr(snapshots), _ptr(accept_len), _ptr(live_state), L, B, S, E,
                               _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_commit_state", rc)
    return live_state


ALIGN_TOKEN, ALIGN_LAST = 0, 1


def spec_commit_state_aligned(snapshots, accept_len, live_state, num_tokens: int, alignment: int,
                              dev_err: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Commit from a checkpoint window [L, B, W, E] of a num_tokens-token step (see spec_verify.h):
    slot accept_len[b] (ALIGN_TOKEN) or W - num_tokens + accept_len[b] (ALIGN_LAST)."""
    lib = load_library()
    _need(snapshots, "snapshots", torch.float32, 4)
    _need(accept_len, "accept_len", torch.int32, 1)
    _need(live_state, "live_state", torch.float32, 3)
    L, B, W, E = snapshots.shape
    if live_state.shape != (L, B, E) or accept_len.shape != (B,):
        raise ValueError("inconsistent commit shapes")
    rc = lib.spec_commit_state_aligned(_ptr(snapshots), _ptr(accept_len), _ptr(live_state), L, B, W, E,
                                       int(num_tokens), int(alignment), _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_commit_state_aligned", rc)
    return live_state


def spec_commit_select(accept_len, live_row, ckpt_rows, num_tokens: int, alignment: int,
                       dev_err: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Zero-copy commit over a state pool (see spec_verify.h): exchange live_row[l, b] [L, B] with
    the window slot ckpt_rows[l, b, s] [L, B, W] of the accepted prefix, in place; no state moves."""
    lib = load_library()
    _need(accept_len, "accept_len", torch.int32, 1)
    _need(live_row, "live_row", torch.int32, 2)
    _need(ckpt_rows, "ckpt_rows", torch.int32, 3)
    L, B = live_row.shape
    W = ckpt_rows.shape[2]
    if ckpt_rows.shape[:2] != (L, B) or accept_len.shape != (B,):
        raise ValueError("inconsistent commit shapes")
    rc = lib.spec_commit_select(_ptr(accept_len), _ptr(live_row), _ptr(ckpt_rows), L, B, W, int(num_tokens),
                                int(alignment), _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_commit_select", rc)
    return live_row, ckpt_rows


def _gdn_shapes(q, k, v, g, beta, out):
    _need(q, "q", torch.float32, 4)
    _need(k, "k", torch.float32, 4)
    _need(v, "v", torch.float32, 4)
    _need(g, "g", torch.float32, 3)
    _need(beta, "beta", torch.float32, 3)
    _need(out, "out", torch.float32, 4)
    B, R, H, dk = q.shape
    dv = v.shape[3]
    if k.shape != q.shape or v.shape != (B, R, H, dv) or g.shape != (B, R, H) or beta.shape != (B, R, H) \
            or out.shape != (B, R, H, dv):
        raise ValueError("inconsistent gated-delta-rule shapes")
    return B, R, H, dk, dv


def spec_gdn_verify(q, k, v, g, beta, state_in, snapshots, out, scale: float, alignment: int = ALIGN_TOKEN,
                    dev_err: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Gated delta rule over the verify chain for one layer (see spec_verify.h): state_in [B,H,dv,dk],
    snapshots [B,W,H,dv,dk] (slot base+t = state after token t), out [B,R,H,dv]."""
    lib = load_library()
    B, R, H, dk, dv = _gdn_shapes(q, k, v, g, beta, out)
    _need(state_in, "state_in", torch.float32, 4)
    _need(snapshots, "snapshots", torch.float32, 5)
    W = snapshots.shape[1]
    if state_in.shape != (B, H, dv, dk) or snapshots.shape != (B, W, H, dv, dk):
        raise ValueError("inconsistent state shapes")
    rc = lib.spec_gdn_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(state_in),
                             _ptr(snapshots), _ptr(out), B, R, H, dk, dv, W, int(alignment), _err_ptr(dev_err),
                             _stream_handle(stream))
    _check("spec_gdn_verify", rc)
    return snapshots, out


def spec_gdn_verify_pooled(q, k, v, g, beta, pool, live_row, ckpt_rows, out, scale: float,
                           alignment: int = ALIGN_TOKEN, dev_err: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None):
    """The same step over a state pool [P, H*dv*dk]: reads pool[live_row[b]], writes checkpoint slot s to
    pool[ckpt_rows[b, s]] (the tables of one layer: live_row [B], ckpt_rows [B, W])."""
    lib = load_library()
    B, R, H, dk, dv = _gdn_shapes(q, k, v, g, beta, out)
    _need(pool, "pool", torch.float32, 2)
    _need(live_row, "live_row", torch.int32, 1)
    _need(ckpt_rows, "ckpt_rows", torch.int32, 2)
    W = ckpt_rows.shape[1]
    if pool.shape[1] != H * dv * dk or live_row.shape != (B,) or ckpt_rows.shape != (B, W):
        raise ValueError("inconsistent pool shapes")
    rc = lib.spec_gdn_verify_pooled(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(pool),
                                    pool.shape[0], _ptr(live_row), _ptr(ckpt_rows), _ptr(out), B, R, H, dk, dv, W,
                                    int(alignment), _err_ptr(dev_err), _stream_handle(stream))
    _check("spec_gdn_verify_pooled", rc)
    return out
