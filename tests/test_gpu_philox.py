"""Philox4x32-10: three-way agreement between the oracle, the library's device
generator and CUDA's curand_Philox4x32_10 (the published algorithm of Salmon
et al., SC'11), on random and edge-case counters and keys."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    import serving_vocab_wide_gb300 as svw
    B = __import__("serving_vocab_wide_gb300.build", fromlist=["ARCH"])
    out = str(tmp_path_factory.mktemp("philox") / "philox_check.so")
    subprocess.run([B._nvcc(), B.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-o", out,
                    os.path.join(HERE, "philox_check.cu")], check=True)
    lib = ctypes.CDLL(out)
    P = ctypes.c_void_p
    lib.philox_check.argtypes = [P, P, ctypes.c_int, P, P, P]
    lib.philox_check.restype = ctypes.c_int
    return lib


def test_three_way(harness):
    rng = np.random.default_rng(2024)
    n = 4096
    ctr = rng.integers(0, 2**32, size=(n, 3), dtype=np.uint64).astype(np.uint32)
    seed = rng.integers(0, 2**63, size=n, dtype=np.uint64) * 2 + rng.integers(0, 2, size=n, dtype=np.uint64)
    # edge cases: zero and all-ones counters and keys, small request / position indices
    ctr[:4] = [[0, 0, 0], [0xFFFFFFFF] * 3, [1, 2, 1], [255, 31, 0]]
    seed[:4] = [0, 2**64 - 1, 1234567, 0x0123456789ABCDEF]
    ctr = np.ascontiguousarray(ctr)
    seed = np.ascontiguousarray(seed.astype(np.uint64))
    w0 = np.zeros(n, np.uint32)
    u = np.zeros(n, np.float32)
    cur = np.zeros((n, 4), np.uint32)
    rc = harness.philox_check(ctr.ctypes.data, seed.ctypes.data, n, w0.ctypes.data, u.ctypes.data, cur.ctypes.data)
    assert rc == 0
    # library == CUDA's generator
    assert np.array_equal(w0, cur[:, 0])
    for i in range(0, n, 37):
        key = [int(seed[i]) & 0xFFFFFFFF, int(seed[i]) >> 32]
        ref = oracle.philox4x32_10([ctr[i, 0], ctr[i, 1], ctr[i, 2], 0], key)
        assert np.array_equal(ref, cur[i]), i            # oracle == CUDA's generator, all four words
        assert oracle.uniform(int(seed[i]), int(ctr[i, 0]), int(ctr[i, 1]), int(ctr[i, 2])) == float(u[i])
    assert np.all((u >= 0) & (u < 1))
