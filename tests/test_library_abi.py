"""The C-ABI library builds, loads and exports every entry point of spec_verify.h (CPU only).

Also checks the host-side argument validation, which returns before any CUDA
call and so needs no GPU.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_verification_paged_gb300 as sv
    sv.build()
    return sv.load_library()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("spec_verify_attention", "spec_accept", "spec_commit_state"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    import speculative_decoding_verification_paged_gb300 as sv
    assert sv.status_string(0) == "ok"
    assert sv.status_string(-4) == "workspace missing or too small"


def _desc(**kw):
    import speculative_decoding_verification_paged_gb300 as sv
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=64, max_blocks_per_seq=4,
                num_blocks=8)
    base.update(kw)
    return sv._AttnDesc(**base)


def test_attention_host_validation(lib):
    fake = ctypes.c_void_p(256)
    d = _desc()
    ws = lib.spec_verify_attention_workspace(ctypes.byref(d), 3)
    assert ws > 0
    # workspace grows with batch and head count
    assert lib.spec_verify_attention_workspace(ctypes.byref(_desc(batch=64)), 3) > ws
    # invalid descriptor
    assert lib.spec_verify_attention_workspace(None, 3) == 0
    assert lib.spec_verify_attention_workspace(ctypes.byref(_desc(num_q_heads=7)), 3) == 0
    call = lambda dd, kd=3, wsb=ws, q=fake, w=fake: lib.spec_verify_attention(
        q, fake, fake, fake, fake, kd, fake, ctypes.byref(dd), w, wsb, None, None)
    assert call(_desc(), q=None) == -1
    assert call(_desc(num_q_heads=7)) == -1
    assert call(_desc(), kd=0) == -1
    assert call(_desc(head_dim=96)) == -2
    assert call(_desc(block_size=48)) == -2
    assert call(_desc(num_q_heads=36, num_kv_heads=2)) == -2  # (k+1)*G = 72 > 64 rows
    assert call(_desc(), wsb=ws - 1) == -4
    assert call(_desc(), w=None) == -4
    assert call(_desc(batch=0)) == 0


def _plan(lib, kd=3, **kw):
    import speculative_decoding_verification_paged_gb300 as sv
    plan = sv._AttnPlan()
    rc = lib.spec_verify_attention_plan(ctypes.byref(_desc(**kw)), kd, ctypes.byref(plan))
    return rc, {name: getattr(plan, name) for name, _ in sv._AttnPlan._fields_}


def test_attention_plan_without_a_device(lib, monkeypatch):
    """Plans that need no device query: the mma.sync instances, whose tile settings
    follow from the shared-memory arithmetic of their configuration (16 rows at
    D = 128: 64-key stages of 32 KB, three stages, two CTAs per SM; 24 rows at
    D = 256, forced onto mma.sync: 32-key stages, one CTA per SM, so a fourth
    stage). Head dims 128 and 256 with 17 or more rows take the tcgen05 kernel
    when its shared-memory plan fits, which asks the device: no device here."""
    monkeypatch.delenv("SPEC_ATTN_KERNEL", raising=False)
    rc, p = _plan(lib, num_q_heads=32, num_kv_heads=8)  # (3+1) * 4 = 16 rows
    assert rc == 0
    assert p == dict(kernel=1, m_tiles=1, keys_per_tile=64, stages=3, p_buffers=0, ctas_per_sm=2)
    rc, p = _plan(lib, num_q_heads=4, num_kv_heads=1, head_dim=64)
    assert rc == 0 and p["kernel"] == 1 and p["m_tiles"] == 1 and p["keys_per_tile"] == 64
    assert _plan(lib, kd=7, num_q_heads=64, num_kv_heads=8)[0] == -3
    assert _plan(lib, num_q_heads=24, num_kv_heads=4, head_dim=256)[0] == -3
    monkeypatch.setenv("SPEC_ATTN_KERNEL", "mma")
    rc, p = _plan(lib, kd=7, num_q_heads=64, num_kv_heads=8)  # 64 rows, forced onto mma.sync
    assert rc == 0 and p["kernel"] == 1 and p["m_tiles"] == 4
    rc, p = _plan(lib, num_q_heads=24, num_kv_heads=4, head_dim=256)  # 24 rows, forced onto mma.sync
    assert rc == 0
    assert p == dict(kernel=1, m_tiles=2, keys_per_tile=32, stages=4, p_buffers=0, ctas_per_sm=1)
    monkeypatch.delenv("SPEC_ATTN_KERNEL")
    assert lib.spec_verify_attention_plan(ctypes.byref(_desc()), 3, None) == -1
    assert _plan(lib, num_q_heads=7)[0] == -1
    assert _plan(lib, kd=0)[0] == -1
    assert _plan(lib, head_dim=96)[0] == -2
    assert _plan(lib, num_q_heads=36, num_kv_heads=2)[0] == -2


def test_accept_and_commit_host_validation(lib):
    fake = ctypes.c_void_p(256)
    acc = lambda B=2, k=3, V=100, logits=fake: lib.spec_accept(logits, fake, fake, 1, fake, fake, fake, fake,
                                                               B, k, V, None, None)
    assert acc(k=0) == -1
    assert acc(V=0) == -1
    assert acc(logits=None) == -1
    assert acc(k=32) == -2
    assert acc(B=0) == 0
    com = lambda L=2, B=2, S=4, E=16, snaps=fake: lib.spec_commit_state(snaps, fake, fake, L, B, S, E, None, None)
    assert com(S=0) == -1
    assert com(snaps=None) == -1
    assert com(L=0) == 0
    assert com(L=1000, B=1000) == -2
    al = lambda n=3, a=1, W=4, L=2, snaps=fake: lib.spec_commit_state_aligned(snaps, fake, fake, L, 2, W, 16, n, a,
                                                                               None, None)
    assert al(n=5) == -1      # step longer than the window
    assert al(n=0) == -1
    assert al(a=2) == -1      # unknown alignment
    assert al(snaps=None) == -1
    assert al(L=0) == 0
    sel = lambda n=3, a=1, W=4, L=2, B=2, live=fake: lib.spec_commit_select(fake, live, fake, L, B, W, n, a, None,
                                                                              None)
    assert sel(n=5) == -1     # step longer than the window
    assert sel(n=0) == -1
    assert sel(W=0) == -1
    assert sel(a=2) == -1     # unknown alignment
    assert sel(L=-1) == -1
    assert sel(live=None) == -1
    assert sel(L=0) == 0      # nothing to do: no launch
    assert sel(B=0, live=None) == 0


def test_gdn_host_validation(lib):
    fake = ctypes.c_void_p(256)
    gv = lambda B=2, R=4, H=2, dk=16, dv=16, W=4, a=0, state=fake: lib.spec_gdn_verify(
        fake, fake, fake, fake, fake, ctypes.c_float(0.25), state, fake, fake, B, R, H, dk, dv, W, a, None, None)
    assert gv(R=0) == -1
    assert gv(R=33) == -1     # longer than a verify chain can be
    assert gv(W=3) == -1      # window shorter than the chain
    assert gv(a=2) == -1
    assert gv(H=0) == -1
    assert gv(dk=0) == -1
    assert gv(state=None) == -1
    assert gv(B=0) == 0       # nothing to do: no launch
    assert gv(dk=512, dv=512) == -2  # state too large for either kernel
    gp = lambda B=2, rows=10, live=fake, a=0: lib.spec_gdn_verify_pooled(
        fake, fake, fake, fake, fake, ctypes.c_float(0.25), fake, rows, live, fake, fake, B, 4, 2, 16, 16, 4, a,
        None, None)
    assert gp(rows=0) == -1
    assert gp(live=None) == -1
    assert gp(a=5) == -1
    assert gp(B=0) == 0


def test_plain_c_program_uses_the_boundary(lib, tmp_path):
    """A C program built with gcc against the header alone links the library and
    exercises its host-side paths (no GPU needed)."""
    import shutil
    import subprocess

    import speculative_decoding_verification_paged_gb300 as sv

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    libdir = os.path.dirname(sv.library_path())
    exe = str(tmp_path / "c_abi_host_checks")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_host_checks.c"), "-L", libdir, "-lspecverify",
                        "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    env = {k: v for k, v in os.environ.items() if k != "SPEC_ATTN_KERNEL"}  # the default kernel choice
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120, env=env)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
