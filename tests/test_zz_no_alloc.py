"""The allocation-free verification entry point (spec_verify_noalloc).

It serves callers that cannot allocate device memory, by running the regular
verification kernels on a fixed scratch area the library keeps on each GPU.
Its results must equal those of spec_verify with a caller workspace.  The file
is named so that pytest collects it last; it passes on its own in a fresh
process as well as after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu


def _both(b, T):
    import torch
    import serving_vocab_wide_gb300 as svw
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)
    cu, tok = to_torch_i32(b.cu), to_torch_i32(b.tokens[float(T)])
    acc, nxt = svw.spec_verify(t, d, cu, tok, T, b.seed, total_draft_rows=b.total_rows)
    # the new entry point, called directly through the C ABI
    L = svw.lib()
    acc2 = torch.full((b.N,), -7, dtype=torch.int32, device="cuda")
    nxt2 = torch.full((b.N,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    rc = L.spec_verify_noalloc(P(t.data_ptr()), P(d.data_ptr()), svw._dtype_code(t), b.V, b.N,
                               P(cu.data_ptr()), b.total_rows, 32, P(tok.data_ptr()), float(T),
                               b.seed, P(acc2.data_ptr()), P(nxt2.data_ptr()),
                               P(status.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.svw_status_string(rc)
    return (acc.cpu().numpy(), nxt.cpu().numpy(), acc2.cpu().numpy(), nxt2.cpu().numpy(),
            int(status.item()))


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    import torch
    torch.cuda.set_device(0)
    b1 = synth.config(3, N=24, seed=31)
    b2 = synth.config(5, N=12, seed=32)
    b2.tokens[1.0] = synth.sample_tokens(b2.draft, 1.0, 32)
    for b, T in ((b1, 1.0), (b2, 0.0), (b2, 1.0)):
        acc, nxt, acc2, nxt2, st = _both(b, T)
        # same kernels on the same inputs: identical outputs, bit for bit
        assert np.array_equal(acc, acc2) and np.array_equal(nxt, nxt2), (T, acc, acc2)
        assert st == 0 and np.all(acc >= 0)


def test_noalloc_rejects_batches_beyond_its_scratch():
    import torch
    import serving_vocab_wide_gb300 as svw
    L = svw.lib()
    N, R, V = 4096, 65536, 151936
    assert svw.verify_workspace_size(N, R, V, svw.SVW_BF16) > (32 << 20)
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p(dummy.data_ptr())
    rc = L.spec_verify_noalloc(P, P, svw.SVW_BF16, V, N, P, R, 16, P, 1.0, 0, P, P, None, None)
    assert rc == 2  # SVW_ERR_UNSUPPORTED, nothing launched


def test_noalloc_python_wrapper_reports_bad_requests_like_spec_verify():
    """The Python binding of the allocation-free call, with a status word and
    one bad request (a token out of range): status and outputs equal
    spec_verify's."""
    import torch
    import serving_vocab_wide_gb300 as svw
    b = synth.config(3, N=16, seed=33)
    tok_np = b.tokens[1.0].copy()
    tok_np[int(b.cu[5]) + 1] = b.V + 3          # request 5 has an out-of-range token
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)
    cu, tok = to_torch_i32(b.cu), to_torch_i32(tok_np)
    s1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    s2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    a1, n1 = svw.spec_verify(t, d, cu, tok, 1.0, b.seed, status=s1)
    a2, n2 = svw.spec_verify_noalloc(t, d, cu, tok, 1.0, b.seed, status=s2)   # R derived from cu_draft
    assert int(s1.item()) == int(s2.item()) == svw.SVW_DEV_BAD_INPUT
    assert svw.device_status(int(s2.item())) == 6
    assert np.array_equal(a1.cpu().numpy(), a2.cpu().numpy())
    assert np.array_equal(n1.cpu().numpy(), n2.cpu().numpy())
    assert int(a2[5].item()) == -1 and int(n2[5].item()) == -1
    assert int((a2 >= 0).sum().item()) == b.N - 1


def test_noalloc_rejects_a_stream_of_another_device():
    import torch
    import serving_vocab_wide_gb300 as svw
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    b = synth.config(3, N=4, seed=34)
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)
    cu, tok = to_torch_i32(b.cu), to_torch_i32(b.tokens[1.0])
    acc = torch.full((b.N,), -7, dtype=torch.int32, device="cuda")
    other = torch.cuda.Stream(device=1)
    P = ctypes.c_void_p
    with torch.cuda.device(0):
        rc = svw.lib().spec_verify_noalloc(P(t.data_ptr()), P(d.data_ptr()), svw.SVW_BF16, b.V, b.N,
                                           P(cu.data_ptr()), b.total_rows, 32, P(tok.data_ptr()), 1.0, 0,
                                           P(acc.data_ptr()), P(acc.data_ptr()), None, P(other.cuda_stream))
    assert rc == 1                           # SVW_ERR_INVALID_ARG, nothing launched
    torch.cuda.synchronize()
    assert int((acc == -7).sum().item()) == b.N
