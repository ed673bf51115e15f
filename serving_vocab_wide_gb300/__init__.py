"""serving_vocab_wide_gb300 -- batched speculative verification and the OPD
loss over full-vocabulary logits, as hand-written CUDA for GB300 (sm_103a).

This module is a thin ctypes binding over the C ABI in ``include/svw.h``:
it only marshals PyTorch CUDA tensors (data pointers, sizes, the current
stream) into the library's entry points.  Every step of the computation runs
in the library's kernels; there is no CPU or PyTorch fallback -- if the shared
library is missing the calls raise.

Build the library with ``serving_vocab_wide_gb300.build()`` (nvcc, sm_103a).
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH, build  # noqa: F401

SVW_F32 = 0
SVW_BF16 = 1
SVW_DEV_BAD_INPUT = 1
SVW_DEV_TIMEOUT = 2
SVW_ERR_BAD_INPUT = 6
SVW_ERR_TIMEOUT = 7
SVW_MAX_LEN = 32

_lib = None
_lock = threading.Lock()


class SvwError(RuntimeError):
    pass


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise SvwError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run serving_vocab_wide_gb300.build())")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, I64, F, U64, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t)
            L.svw_verify_workspace_size.argtypes = [I32, I64, I32, ctypes.c_int]
            L.svw_verify_workspace_size.restype = SZ
            L.svw_workspace_size.argtypes = [I32, I64, I32, I32]
            L.svw_workspace_size.restype = SZ
            L.svw_device_status.argtypes = [I32]
            L.svw_device_status.restype = ctypes.c_int
            L.spec_verify.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, P, F, U64,
                                      P, P, P, P, SZ, P]
            L.spec_verify.restype = ctypes.c_int
            L.svw_verify_early_workspace_size.argtypes = [I32, I64, I32, ctypes.c_int]
            L.svw_verify_early_workspace_size.restype = SZ
            L.spec_verify_early.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, P, F, U64,
                                            P, P, P, P, P, SZ, P]
            L.spec_verify_early.restype = ctypes.c_int
            L.svw_verify_filtered_workspace_size.argtypes = [I32, I64, I32, ctypes.c_int]
            L.svw_verify_filtered_workspace_size.restype = SZ
            L.spec_verify_filtered.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, P, F, I32, F, U64,
                                               P, P, P, P, SZ, P]
            L.spec_verify_filtered.restype = ctypes.c_int
            L.svw_opd_workspace_size.argtypes = [I64]
            L.svw_opd_workspace_size.restype = SZ
            L.opd_loss.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, F, F, F, F,
                                   P, P, P, P, SZ, P]
            L.opd_loss.restype = ctypes.c_int
            L.spec_verify_noalloc.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, P, F, U64,
                                              P, P, P, P]
            L.svw_verify_opd_workspace_size.argtypes = [I32, I64, I32, ctypes.c_int]
            L.svw_verify_opd_workspace_size.restype = SZ
            L.spec_verify_opd.argtypes = [P, P, ctypes.c_int, I32, I32, P, I64, I32, P, F, F, U64, F, F, F,
                                          P, P, P, P, P, P, SZ, P]
            L.spec_verify_opd.restype = ctypes.c_int
            L.spec_verify_noalloc.restype = ctypes.c_int
            L.svw_length_head_workspace_size.argtypes = [I32, I32, I32]
            L.svw_length_head_workspace_size.restype = SZ
            L.length_head.argtypes = [P, P, P, P, F, I32, I32, I32, I32, F, P, P, P, SZ, P]
            L.length_head.restype = ctypes.c_int
            L.length_head_label.argtypes = [P, P, P, I32, P, P, P]
            L.length_head_label.restype = ctypes.c_int
            L.svw_time_next_launch.argtypes = [ctypes.c_char_p, P, P]
            L.svw_time_next_launch.restype = ctypes.c_int
            L.svw_set_wait_limit.argtypes = [I64]
            L.svw_set_wait_limit.restype = ctypes.c_int
            L.svw_set_fault.argtypes = [I32]
            L.svw_set_fault.restype = ctypes.c_int
            L.svw_status_string.argtypes = [ctypes.c_int]
            L.svw_status_string.restype = ctypes.c_char_p
            L.svw_version.argtypes = []
            L.svw_version.restype = I32
            _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise SvwError(lib().svw_status_string(rc).decode())


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return SVW_BF16
    if t.dtype == torch.float32:
        return SVW_F32
    raise SvwError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise SvwError("tensors must be contiguous CUDA tensors")


def time_next_launch(kernel: str | None, begin=None, end=None):
    """Arm the library's one-shot timer: the next launch of `kernel` from this
    thread records the torch.cuda.Event `begin` before it and `end` after it
    on the launch stream (measurement only)."""
    if kernel is None:
        _check(lib().svw_time_next_launch(None, None, None))
        return
    for ev in (begin, end):
        if not ev.cuda_event:  # torch creates the CUDA event at its first record
            ev.record()
    _check(lib().svw_time_next_launch(kernel.encode(), ctypes.c_void_p(begin.cuda_event),
                                      ctypes.c_void_p(end.cuda_event)))


DEFAULT_WAIT_CYCLES = 4_000_000_000


def set_wait_limit(cycles: int = DEFAULT_WAIT_CYCLES):
    """Test hook: the deadline (SM cycles) of every bounded wait in the
    library's kernels on the current device."""
    _check(lib().svw_set_wait_limit(int(cycles)))


def set_fault(kind: int = 0):
    """Test hook: 1 = the next calls' stats / OPD fast kernels leave one CTA
    (cluster) without its copies, so that its first wait runs out; 0 = none."""
    _check(lib().svw_set_fault(int(kind)))


def workspace_size(n_requests: int, total_draft_rows: int, V: int, max_len: int = SVW_MAX_LEN) -> int:
    """One workspace size that serves every entry point on this batch shape."""
    return int(lib().svw_workspace_size(n_requests, total_draft_rows, V, max_len))


def device_status(word: int) -> int:
    """svw_status code of a device status word (SVW_ERR_TIMEOUT, SVW_ERR_BAD_INPUT or 0)."""
    return int(lib().svw_device_status(int(word)))


def verify_workspace_size(n_requests: int, total_draft_rows: int, V: int, dtype_code: int) -> int:
    return int(lib().svw_verify_workspace_size(n_requests, total_draft_rows, V, dtype_code))


def opd_workspace_size(total_draft_rows: int) -> int:
    return int(lib().svw_opd_workspace_size(total_draft_rows))


def spec_verify(target, draft, cu_draft, draft_tokens, temperature: float, seed: int,
                max_len: int = SVW_MAX_LEN, total_draft_rows: int | None = None,
                accept_len=None, next_token=None, status=None, workspace=None, stream=None):
    """Verify a ragged batch.  Returns (accept_len, next_token) int32 CUDA tensors.

    target: [total_draft_rows + N, V], draft: [total_draft_rows, V] (bf16 or
    fp32); cu_draft: int32 [N + 1] CSR offsets; draft_tokens: int32
    [total_draft_rows].  Output / workspace / status tensors may be passed in
    to avoid allocation; `total_draft_rows` (= cu_draft[-1]) may be passed to
    avoid a device read.
    """
    import torch
    _need_cuda(target, draft, cu_draft, draft_tokens)
    N = cu_draft.numel() - 1
    V = target.shape[-1]
    R = int(cu_draft[-1].item()) if total_draft_rows is None else int(total_draft_rows)
    code = _dtype_code(target)
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(N, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, verify_workspace_size(N, R, V, code)), dtype=torch.uint8,
                                device=dev)
    _need_cuda(accept_len, next_token, workspace, status)
    rc = lib().spec_verify(_ptr(target), _ptr(draft), code, V, N, _ptr(cu_draft), R, max_len,
                           _ptr(draft_tokens), float(temperature), int(seed) & (2**64 - 1),
                           _ptr(accept_len), _ptr(next_token), _ptr(status), _ptr(workspace),
                           workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return accept_len, next_token


def verify_early_workspace_size(n_requests: int, total_draft_rows: int, V: int, dtype_code: int) -> int:
    return int(lib().svw_verify_early_workspace_size(n_requests, total_draft_rows, V, dtype_code))


def spec_verify_early(target, draft, cu_draft, draft_tokens, temperature: float, seed: int,
                      max_len: int = SVW_MAX_LEN, total_draft_rows: int | None = None,
                      accept_len=None, next_token=None, status=None, bytes_read=None, workspace=None,
                      stream=None):
    """spec_verify that stops reading each request at its first rejection.
    Same (accept_len, next_token); `bytes_read` (int64 CUDA scalar, optional)
    receives the logit bytes the call streamed."""
    import torch
    _need_cuda(target, draft, cu_draft, draft_tokens)
    N = cu_draft.numel() - 1
    V = target.shape[-1]
    R = int(cu_draft[-1].item()) if total_draft_rows is None else int(total_draft_rows)
    code = _dtype_code(target)
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(N, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, verify_early_workspace_size(N, R, V, code)), dtype=torch.uint8,
                                device=dev)
    _need_cuda(accept_len, next_token, workspace, status, bytes_read)
    if bytes_read is not None and (bytes_read.dtype != torch.int64 or bytes_read.numel() != 1):
        raise SvwError("bytes_read must be a one-element int64 tensor")
    rc = lib().spec_verify_early(_ptr(target), _ptr(draft), code, V, N, _ptr(cu_draft), R, max_len,
                                 _ptr(draft_tokens), float(temperature), int(seed) & (2**64 - 1),
                                 _ptr(accept_len), _ptr(next_token), _ptr(status), _ptr(bytes_read),
                                 _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return accept_len, next_token


SVW_FILTER_MAX_K = 1024


def verify_filtered_workspace_size(n_requests: int, total_draft_rows: int, V: int, dtype_code: int) -> int:
    return int(lib().svw_verify_filtered_workspace_size(n_requests, total_draft_rows, V, dtype_code))


def spec_verify_filtered(target, draft, cu_draft, draft_tokens, temperature: float, top_k: int, top_p: float,
                         seed: int, max_len: int = SVW_MAX_LEN, total_draft_rows: int | None = None,
                         accept_len=None, next_token=None, status=None, workspace=None, stream=None):
    """spec_verify with both distributions top-k / top-p filtered (draft tokens
    drawn from the filtered draft distribution).  Returns (accept_len, next_token)."""
    import torch
    _need_cuda(target, draft, cu_draft, draft_tokens)
    N = cu_draft.numel() - 1
    V = target.shape[-1]
    R = int(cu_draft[-1].item()) if total_draft_rows is None else int(total_draft_rows)
    code = _dtype_code(target)
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(N, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, verify_filtered_workspace_size(N, R, V, code)), dtype=torch.uint8,
                                device=dev)
    _need_cuda(accept_len, next_token, workspace, status)
    rc = lib().spec_verify_filtered(_ptr(target), _ptr(draft), code, V, N, _ptr(cu_draft), R, max_len,
                                    _ptr(draft_tokens), float(temperature), int(top_k), float(top_p),
                                    int(seed) & (2**64 - 1), _ptr(accept_len), _ptr(next_token), _ptr(status),
                                    _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return accept_len, next_token


def spec_verify_noalloc(target, draft, cu_draft, draft_tokens, temperature: float, seed: int,
                        max_len: int = SVW_MAX_LEN, total_draft_rows: int | None = None,
                        accept_len=None, next_token=None, status=None, stream=None):
    """spec_verify on the library's fixed per-GPU scratch instead of a caller
    workspace (for callers that cannot allocate).  Calls that may overlap on
    the GPU share that scratch and must be serialised on one stream."""
    import torch
    _need_cuda(target, draft, cu_draft, draft_tokens)
    N = cu_draft.numel() - 1
    V = target.shape[-1]
    R = int(cu_draft[-1].item()) if total_draft_rows is None else int(total_draft_rows)
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(N, dtype=torch.int32, device=dev)
    _need_cuda(accept_len, next_token, status)
    # the library uses the current device's scratch: make the inputs' device current
    with torch.cuda.device(dev):
        rc = lib().spec_verify_noalloc(_ptr(target), _ptr(draft), _dtype_code(target), V, N,
                                       _ptr(cu_draft), R, max_len, _ptr(draft_tokens),
                                       float(temperature), int(seed) & (2**64 - 1), _ptr(accept_len),
                                       _ptr(next_token), _ptr(status), _stream_ptr(stream))
    _check(rc)
    return accept_len, next_token


def verify_opd_workspace_size(n_requests: int, total_draft_rows: int, V: int, dtype_code: int) -> int:
    return int(lib().svw_verify_opd_workspace_size(n_requests, total_draft_rows, V, dtype_code))


def spec_verify_opd(target, draft, cu_draft, draft_tokens, temperature: float, seed: int,
                    opd_temperature: float | None = None, clip_c: float = 1.0, lambda_ce: float = 0.1,
                    grad_scale: float = 1.0, max_len: int = SVW_MAX_LEN,
                    total_draft_rows: int | None = None, want_grad: bool = True, accept_len=None,
                    next_token=None, loss=None, dlogits=None, status=None, workspace=None, stream=None):
    """Verification and the OPD loss on the same batch in one pass.  Returns
    (accept_len, next_token, loss, dlogits or None).  opd_temperature
    defaults to temperature (or 1.0 when greedy)."""
    import torch
    _need_cuda(target, draft, cu_draft, draft_tokens)
    N = cu_draft.numel() - 1
    V = target.shape[-1]
    R = int(cu_draft[-1].item()) if total_draft_rows is None else int(total_draft_rows)
    code = _dtype_code(target)
    dev = target.device
    if opd_temperature is None:
        opd_temperature = temperature if temperature > 0 else 1.0
    if accept_len is None:
        accept_len = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(N, dtype=torch.int32, device=dev)
    if loss is None:
        loss = torch.empty(R, dtype=torch.float32, device=dev)
    if want_grad and dlogits is None:
        dlogits = torch.empty((R, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, verify_opd_workspace_size(N, R, V, code)), dtype=torch.uint8,
                                device=dev)
    _need_cuda(accept_len, next_token, loss, dlogits, status, workspace)
    rc = lib().spec_verify_opd(_ptr(target), _ptr(draft), code, V, N, _ptr(cu_draft), R, max_len,
                               _ptr(draft_tokens), float(temperature), float(opd_temperature),
                               int(seed) & (2**64 - 1), float(clip_c), float(lambda_ce),
                               float(grad_scale), _ptr(accept_len), _ptr(next_token), _ptr(loss),
                               _ptr(dlogits) if want_grad else None, _ptr(status), _ptr(workspace),
                               workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return accept_len, next_token, loss, (dlogits if want_grad else None)


def length_head(hidden, w1, b1, w2, b2: float, gamma: float = 1.0, a_hat=None, k_hat=None, workspace=None,
                stream=None):
    """Adaptive length head forward.  hidden: bf16 [N, k, H], w1: bf16 [H', H],
    b1, w2: float32 [H'].  Returns (a_hat float32 [N], k_hat int32 [N])."""
    import torch
    _need_cuda(hidden, w1, b1, w2)
    if hidden.dtype != torch.bfloat16 or w1.dtype != torch.bfloat16:
        raise SvwError("hidden states and W1 must be bfloat16")
    N, k, H = hidden.shape
    Hp = w1.shape[0]
    dev = hidden.device
    if a_hat is None:
        a_hat = torch.empty(N, dtype=torch.float32, device=dev)
    if k_hat is None:
        k_hat = torch.empty(N, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, int(lib().svw_length_head_workspace_size(N, k, Hp))), dtype=torch.uint8,
                                device=dev)
    _need_cuda(a_hat, k_hat, workspace)
    rc = lib().length_head(_ptr(hidden), _ptr(w1), _ptr(b1), _ptr(w2), float(b2), N, k, H, Hp, float(gamma),
                           _ptr(a_hat), _ptr(k_hat), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return a_hat, k_hat


def length_head_label(accept_len, cu_draft, a_hat=None, a_star=None, loss=None, stream=None):
    """a* = accept_len / L per request and, with a_hat, the MSE (a_hat - a*)^2."""
    import torch
    _need_cuda(accept_len, cu_draft, a_hat)
    N = accept_len.numel()
    dev = accept_len.device
    if a_star is None:
        a_star = torch.empty(N, dtype=torch.float32, device=dev)
    if a_hat is not None and loss is None:
        loss = torch.empty(N, dtype=torch.float32, device=dev)
    _need_cuda(a_star, loss)
    rc = lib().length_head_label(_ptr(accept_len), _ptr(cu_draft), _ptr(a_hat), N, _ptr(a_star), _ptr(loss),
                                 _stream_ptr(stream))
    _check(rc)
    return a_star, loss


def opd_loss(target, draft, temperature: float = 1.0, clip_c: float = 1.0,
             lambda_ce: float = 0.1, grad_scale: float = 1.0, cu_draft=None,
             has_bonus: bool = False, want_grad: bool = True, loss=None, dlogits=None,
             status=None, workspace=None, exact_only: bool = False, stream=None):
    """Clipped reverse-KL + lambda*CE per draft row, and its gradient wrt the
    draft logits.  Returns (loss [R] fp32, dlogits [R, V] fp32 or None).

    A workspace (uint8, >= opd_workspace_size(R) bytes) is allocated when not
    given; exact_only=True passes none, so that every row takes the exact
    three-pass kernel."""
    import torch
    _need_cuda(target, draft, cu_draft)
    R, V = draft.shape
    code = _dtype_code(draft)
    N = (cu_draft.numel() - 1) if has_bonus else 0
    dev = draft.device
    if loss is None:
        loss = torch.empty(R, dtype=torch.float32, device=dev)
    if want_grad and dlogits is None:
        dlogits = torch.empty((R, V), dtype=torch.float32, device=dev)
    if exact_only:
        workspace = None
    elif workspace is None:
        workspace = torch.empty(max(1, opd_workspace_size(R)), dtype=torch.uint8, device=dev)
    _need_cuda(loss, dlogits, status, workspace)
    rc = lib().opd_loss(_ptr(target), _ptr(draft), code, V, N, _ptr(cu_draft) if has_bonus else None,
                        R, 1 if has_bonus else 0, float(temperature), float(clip_c),
                        float(lambda_ce), float(grad_scale), _ptr(loss),
                        _ptr(dlogits) if want_grad else None, _ptr(status), _ptr(workspace),
                        0 if workspace is None else workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return loss, (dlogits if want_grad else None)
