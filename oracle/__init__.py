"""CPU oracle for batched speculative verification and the OPD loss.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; the product path never imports it.

The arithmetic lives in ``svw_oracle.c`` (plain C, binary64, sequential sums in
vocabulary order); this module only compiles it with the host C compiler and
marshals numpy arrays through ctypes.  See the header of ``svw_oracle.c`` for
the passages each function follows and the readings taken where the pages are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "svw_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32 = 0
BF16 = 1

FLAG_NEAR_ACCEPT = 1
FLAG_NEAR_CDF = 2
FLAG_DEGENERATE = 4
FLAG_BAD = 8
FLAG_NEAR_CLIP = 16
FLAG_NEAR_FLOOR = 32
FLAG_NEAR_FILTER = 64

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32,
                                           ctypes.c_uint32, ctypes.c_uint32]
            lib.oracle_uniform.restype = ctypes.c_double
            lib.oracle_spec_verify.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, P, P,
                ctypes.c_double, ctypes.c_uint64, ctypes.c_int32, P, P, P, P, P, P, P]
            lib.oracle_spec_verify.restype = ctypes.c_int
            lib.oracle_spec_verify_filtered.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, P, P,
                ctypes.c_double, ctypes.c_int32, ctypes.c_double, ctypes.c_uint64, ctypes.c_int32,
                P, P, P, P]
            lib.oracle_spec_verify_filtered.restype = ctypes.c_int
            lib.oracle_opd_loss.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, P,
                ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                ctypes.c_double, ctypes.c_double, P, P, P]
            lib.oracle_opd_loss.restype = ctypes.c_int
            lib.oracle_length_head.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                P, P, ctypes.c_float, ctypes.c_double, P, P, P]
            lib.oracle_length_head.restype = ctypes.c_int
            lib.oracle_length_label.argtypes = [P, P, P, ctypes.c_int32, P, P]
            lib.oracle_length_label.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """(array, dtype code): uint16 arrays are bf16 bit patterns, float32 is fp32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {a.dtype}")


def philox4x32_10(counter, key):
    """Philox4x32-10 block: four 32-bit counter words, two key words -> 4 words."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, i: int, j: int, s: int) -> float:
    """U(seed, i, j, s): 24-bit uniform in [0, 1) from Philox word 0."""
    return _load().oracle_uniform(seed, i, j, s)


def spec_verify(target, draft, cu_draft, tokens, temperature, seed, max_len=32,
                req_ids=None, want_thr=False, alt_next=None):
    """Verify a ragged batch.  Returns dict(accept_len, next_token, flags[, thr]
    [, alt_dist]).

    target: [total_rows + N, V], draft: [total_rows, V] (uint16 bf16 bits or
    float32); cu_draft: int32 [N + 1]; tokens: int32 [total_rows].
    alt_next: optional int32 [N], another implementation's next tokens; then
    alt_dist[n] is the distance (fraction of Z) from w Z to that token's CDF
    interval in the distribution the oracle drew from (0: the same draw).
    """
    lib = _load()
    t, dt = _logits(target)
    d, dd = _logits(draft)
    assert dt == dd, "target and draft must share a dtype"
    V = t.shape[-1]
    cu = np.ascontiguousarray(cu_draft, dtype=np.int32)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    N = cu.shape[0] - 1
    rid = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int32)
    acc = np.zeros(N, dtype=np.int32)
    nxt = np.zeros(N, dtype=np.int32)
    flg = np.zeros(N, dtype=np.int32)
    thr = np.full(max(1, tok.shape[0]), np.nan) if want_thr else None
    alt = None if alt_next is None else np.ascontiguousarray(alt_next, dtype=np.int32)
    adist = None if alt is None else np.zeros(N, dtype=np.float64)
    rc = lib.oracle_spec_verify(_ptr(t), _ptr(d), dt, V, N, _ptr(cu), _ptr(tok),
                                float(temperature), int(seed), int(max_len), _ptr(rid),
                                _ptr(acc), _ptr(nxt), _ptr(flg), _ptr(thr), _ptr(alt), _ptr(adist))
    if rc != 0:
        raise MemoryError("oracle_spec_verify failed to allocate")
    out = dict(accept_len=acc, next_token=nxt, flags=flg)
    if want_thr:
        out["thr"] = thr[: tok.shape[0]]
    if alt is not None:
        out["alt_dist"] = adist
    return out


def spec_verify_filtered(target, draft, cu_draft, tokens, temperature, top_k, top_p, seed, max_len=32,
                         req_ids=None):
    """Verification with both distributions top-k / top-p filtered (same T,
    top_k, top_p); tokens drawn from the filtered draft distribution.
    Returns dict(accept_len, next_token, flags)."""
    lib = _load()
    t, dt = _logits(target)
    d, dd = _logits(draft)
    assert dt == dd, "target and draft must share a dtype"
    V = t.shape[-1]
    cu = np.ascontiguousarray(cu_draft, dtype=np.int32)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    N = cu.shape[0] - 1
    rid = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int32)
    acc = np.zeros(N, dtype=np.int32)
    nxt = np.zeros(N, dtype=np.int32)
    flg = np.zeros(N, dtype=np.int32)
    rc = lib.oracle_spec_verify_filtered(_ptr(t), _ptr(d), dt, V, N, _ptr(cu), _ptr(tok), float(temperature),
                                         int(top_k), float(top_p), int(seed), int(max_len), _ptr(rid),
                                         _ptr(acc), _ptr(nxt), _ptr(flg))
    if rc != 0:
        raise MemoryError("oracle_spec_verify_filtered failed to allocate")
    return dict(accept_len=acc, next_token=nxt, flags=flg)


def opd_loss(target, draft, temperature=1.0, clip_c=1.0, lambda_ce=0.1, grad_scale=1.0,
             cu_draft=None, has_bonus=False, want_grad=True):
    """Clipped reverse-KL + lambda * CE per draft row and its gradient.

    Returns dict(loss [R] f64, dlogits [R, V] f64 or None, flags [R]).
    """
    lib = _load()
    t, dt = _logits(target)
    d, dd = _logits(draft)
    assert dt == dd, "target and draft must share a dtype"
    R, V = d.shape
    if has_bonus:
        cu = np.ascontiguousarray(cu_draft, dtype=np.int32)
        N = cu.shape[0] - 1
    else:
        cu, N = None, 0
    loss = np.zeros(R, dtype=np.float64)
    grad = np.zeros((R, V), dtype=np.float64) if want_grad else None
    flg = np.zeros(R, dtype=np.int32)
    rc = lib.oracle_opd_loss(_ptr(t), _ptr(d), dt, V, N, _ptr(cu), R, int(bool(has_bonus)),
                             float(temperature), float(clip_c), float(lambda_ce),
                             float(grad_scale), _ptr(loss), _ptr(grad), _ptr(flg))
    if rc != 0:
        raise MemoryError("oracle_opd_loss failed to allocate")
    return dict(loss=loss, dlogits=grad, flags=flg)


def length_head(hidden, w1, b1, w2, b2, gamma=1.0):
    """Adaptive length head forward.  hidden: [N, k, H] (uint16 bf16 bits or
    float32), w1: [H', H] same dtype, b1: [H'], w2: [H'] float32, b2 scalar.
    Returns dict(a_hat [N] float64, k_hat [N] int32, flags [N])."""
    lib = _load()
    h, dt = _logits(hidden)
    w, dt2 = _logits(w1)
    if dt != dt2:
        raise TypeError("hidden and w1 must have the same dtype")
    N, k, H = h.shape
    Hp = w.shape[0]
    assert w.shape == (Hp, H)
    b1 = np.ascontiguousarray(b1, dtype=np.float32)
    w2 = np.ascontiguousarray(w2, dtype=np.float32)
    a_hat = np.zeros(N, np.float64)
    k_hat = np.zeros(N, np.int32)
    flags = np.zeros(N, np.int32)
    rc = lib.oracle_length_head(_ptr(h), _ptr(w), dt, N, k, H, Hp, _ptr(b1), _ptr(w2), float(b2),
                                float(gamma), _ptr(a_hat), _ptr(k_hat), _ptr(flags))
    if rc != 0:
        raise ValueError(f"oracle_length_head failed ({rc})")
    return {"a_hat": a_hat, "k_hat": k_hat, "flags": flags}


def length_label(accept_len, cu_draft, a_hat):
    """a* = accept_len / L per request and the MSE (a_hat - a*)^2."""
    lib = _load()
    acc = np.ascontiguousarray(accept_len, dtype=np.int32)
    cu = np.ascontiguousarray(cu_draft, dtype=np.int32)
    ah = np.ascontiguousarray(a_hat, dtype=np.float64)
    N = acc.shape[0]
    a_star = np.zeros(N, np.float64)
    loss = np.zeros(N, np.float64)
    lib.oracle_length_label(_ptr(acc), _ptr(cu), _ptr(ah), N, _ptr(a_star), _ptr(loss))
    return {"a_star": a_star, "loss": loss}
