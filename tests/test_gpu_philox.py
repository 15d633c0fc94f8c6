"""Philox4x32-10 three ways on a counter sweep: the library's device generator
(the one the acceptance kernel draws its uniforms and race keys from), cuRAND's
Philox4_32_10 device API, and the oracle; all must agree bit for bit."""

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_philox_device_matches_curand_and_oracle(sv, oracle_mod, tmp_path):
    lib_path = str(tmp_path / "libphilox_probe.so")
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "speculative_decoding_verification_paged_gb300", "csrc"),
           os.path.join(ROOT, "tests", "philox_probe.cu"), "-o", lib_path]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    probe = ctypes.CDLL(lib_path)
    probe.philox_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    probe.philox_probe.restype = ctypes.c_int

    rng = np.random.default_rng(11)
    n = 4096
    words = rng.integers(0, 2**32, size=(n, 6), dtype=np.uint64)
    words[:, 1] >>= 2  # c1 < 2^30 for the cuRAND offset
    words[0] = 0
    words[1] = [0xFFFFFFFF, 0x3FFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF]
    words[2] = [0xFFFFFFFF] * 6  # all ones: library and oracle only
    words = words.astype(np.uint32)
    dev_in = torch.from_numpy(words.view(np.int32).copy()).cuda()
    lib_out = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    cur_out = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    assert probe.philox_probe(dev_in.data_ptr(), lib_out.data_ptr(), cur_out.data_ptr(), n) == 0
    lib = lib_out.cpu().numpy().view(np.uint32)
    cur = cur_out.cpu().numpy().view(np.uint32)
    has_curand = words[:, 1] < (1 << 30)
    assert has_curand.sum() == n - 1
    assert np.array_equal(lib[has_curand], cur[has_curand])
    for i in range(n):
        want = oracle_mod.philox4x32_10([int(x) for x in words[i, :4]], [int(words[i, 4]), int(words[i, 5])])
        assert [int(x) for x in want] == [int(x) for x in lib[i]], i
