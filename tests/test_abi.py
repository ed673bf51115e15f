"""The C-ABI library loads and exports every symbol its header declares, and
host-side validation rejects bad arguments without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "svw.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = "\n".join(l for l in src.splitlines() if not l.lstrip().startswith("#"))
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", src)
    skip = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in skip})


@pytest.fixture(scope="module")
def lib():
    import serving_vocab_wide_gb300 as svw
    svw.build()
    return svw.lib()


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert {"spec_verify", "opd_loss", "svw_verify_workspace_size", "svw_opd_workspace_size",
            "svw_status_string", "svw_version", "spec_verify_noalloc", "spec_verify_early",
            "svw_verify_early_workspace_size", "spec_verify_filtered",
            "svw_verify_filtered_workspace_size", "svw_workspace_size",
            "svw_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in svw.h but not exported"


def test_no_unresolved_internal_symbols(lib):
    """Every internal function the library calls is defined in it: the library
    loads with immediate binding (as a loader that resolves everything at
    load time requires), and no symbol of its own namespace is undefined."""
    import serving_vocab_wide_gb300 as svw
    ctypes.CDLL(svw.LIB_PATH, mode=os.RTLD_NOW | os.RTLD_LOCAL)
    import shutil
    import subprocess
    if shutil.which("nm"):
        out = subprocess.run(["nm", "-D", "--undefined-only", svw.LIB_PATH], capture_output=True, text=True).stdout
        assert "_ZN3svw" not in out, [l for l in out.splitlines() if "_ZN3svw" in l]


def test_test_hooks_validate(lib):
    """The wait-limit and fault hooks reject bad values on the host."""
    assert lib.svw_set_wait_limit(0) == 1      # SVW_ERR_INVALID_ARG
    assert lib.svw_set_wait_limit(-5) == 1
    assert lib.svw_set_fault(2) == 1
    assert lib.svw_set_fault(-1) == 1
    assert lib.svw_set_fault(0) == 0


def test_version_and_status_strings(lib):
    assert lib.svw_version() == 100
    for code in range(8):
        assert lib.svw_status_string(code).startswith(b"SVW_")
    assert lib.svw_status_string(6).startswith(b"SVW_ERR_BAD_INPUT")
    assert lib.svw_status_string(7).startswith(b"SVW_ERR_TIMEOUT")


def test_status_codes_match_the_contract():
    """The status enum's values: the sizing call's and the host codes' names
    and numbers, and the two device-detected codes."""
    src = open(os.path.join(ROOT, "include", "svw.h"), encoding="utf-8").read()
    want = {"SVW_OK": "0", "SVW_ERR_INVALID_ARG": "1", "SVW_ERR_UNSUPPORTED": "2",
            "SVW_ERR_UNSUPPORTED_DTYPE": "SVW_ERR_UNSUPPORTED", "SVW_ERR_MISALIGNED": "3",
            "SVW_ERR_WORKSPACE": "4", "SVW_ERR_CUDA": "5", "SVW_ERR_BAD_INPUT": "6",
            "SVW_ERR_TIMEOUT": "7"}
    for name, val in want.items():
        assert re.search(rf"\b{name}\s*=\s*{val}\b", src), name


def test_device_status_word(lib):
    import serving_vocab_wide_gb300 as svw
    assert lib.svw_device_status(0) == 0
    assert lib.svw_device_status(svw.SVW_DEV_BAD_INPUT) == 6
    assert lib.svw_device_status(svw.SVW_DEV_TIMEOUT) == 7
    assert lib.svw_device_status(svw.SVW_DEV_TIMEOUT | svw.SVW_DEV_BAD_INPUT) == 7   # a timeout voids the call
    assert svw.device_status(svw.SVW_DEV_BAD_INPUT) == 6


def test_one_workspace_size_for_every_entry_point(lib):
    import serving_vocab_wide_gb300 as svw
    for N, R, V in ((256, 1964, 151936), (4, 64, 1024), (32, 512, 151936), (2, 4, 64)):
        need = svw.workspace_size(N, R, V, 16)
        parts = [svw.opd_workspace_size(R)]
        for dt in (svw.SVW_F32, svw.SVW_BF16):
            parts += [svw.verify_workspace_size(N, R, V, dt), svw.verify_early_workspace_size(N, R, V, dt),
                      svw.verify_filtered_workspace_size(N, R, V, dt),
                      svw.verify_opd_workspace_size(N, R, V, dt)]
        assert need == max(parts) > 0
    assert svw.workspace_size(4, 64, 1024, 0) == 0
    assert svw.workspace_size(4, 64, 1024, 33) == 0
    assert svw.workspace_size(0, 64, 1024, 16) == 0
    assert svw.workspace_size(4, 64, 0, 16) == 0


def test_workspace_size(lib):
    import serving_vocab_wide_gb300 as svw
    big = svw.verify_workspace_size(256, 1920, 151936, svw.SVW_BF16)
    small = svw.verify_workspace_size(4, 64, 1024, svw.SVW_F32)
    assert big > small > 0
    assert big % 256 == 0
    assert svw.verify_workspace_size(0, 10, 100, svw.SVW_BF16) == 0
    assert svw.verify_workspace_size(4, 10, 0, svw.SVW_BF16) == 0
    assert svw.verify_workspace_size(4, 10, 1 << 21, svw.SVW_BF16) == 0
    assert svw.opd_workspace_size(0) == 0
    # flags and row constants (256-byte aligned), then 128 float2 partial sums per row
    assert svw.opd_workspace_size(1) == 512 + 1024
    assert svw.opd_workspace_size(1920) == 7680 + 30720 + 1920 * 1024


def _fake(n):
    # aligned host addresses: validation rejects before any pointer is used
    buf = ctypes.create_string_buffer(n + 256)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    return buf, ctypes.c_void_p(addr)


def test_verify_argument_validation(lib):
    keep, p = _fake(4096)
    ok_args = dict(t=p, d=p, dt=1, V=64, N=2, cu=p, R=4, ml=16, tok=p, T=1.0, seed=0,
                   acc=p, nxt=p, st=None, ws=p, wsb=1 << 30)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spec_verify(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"],
                               a["ml"], a["tok"], a["T"], a["seed"], a["acc"], a["nxt"],
                               a["st"], a["ws"], a["wsb"], None)

    assert call(dt=7) == 2                  # unsupported dtype
    assert call(V=0) == 1
    assert call(N=0) == 1
    assert call(ml=0) == 1
    assert call(ml=33) == 2                 # above SVW_MAX_LEN
    assert call(t=None) == 1
    assert call(ws=None) == 4
    assert call(wsb=16) == 4                # workspace too small
    assert call(T=-1.0) == 1
    assert call(T=float("nan")) == 1
    assert call(T=float("inf")) == 1
    assert call(T=1e-45) == 1               # log2(e)/T overflows
    mis = ctypes.c_void_p(p.value + 1)
    assert call(t=mis) == 3
    assert call(ws=ctypes.c_void_p(p.value + 16)) == 3


def test_verify_early_argument_validation(lib):
    import serving_vocab_wide_gb300 as svw
    keep, p = _fake(4096)
    ok_args = dict(t=p, d=p, dt=1, V=64, N=2, cu=p, R=4, ml=16, tok=p, T=1.0, seed=0,
                   acc=p, nxt=p, st=None, nb=None, ws=p, wsb=1 << 30)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spec_verify_early(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"], a["ml"],
                                     a["tok"], a["T"], a["seed"], a["acc"], a["nxt"], a["st"], a["nb"],
                                     a["ws"], a["wsb"], None)

    assert call(dt=7) == 2
    assert call(V=0) == 1
    assert call(ml=33) == 2
    assert call(tok=None) == 1
    assert call(ws=None) == 4
    assert call(T=float("nan")) == 1
    assert call(nb=ctypes.c_void_p(p.value + 4)) == 3       # bytes_read must be 8-byte aligned
    need = svw.verify_early_workspace_size(2, 4, 64, svw.SVW_BF16)
    assert call(wsb=need - 1) == 4
    # the early-exit state comes after spec_verify's workspace
    for args in ((2, 4, 64, svw.SVW_BF16), (256, 1964, 151936, svw.SVW_BF16), (4, 64, 1024, svw.SVW_F32)):
        assert svw.verify_early_workspace_size(*args) > svw.verify_workspace_size(*args)
    assert svw.verify_early_workspace_size(0, 4, 64, svw.SVW_BF16) == 0


def test_verify_filtered_argument_validation(lib):
    import serving_vocab_wide_gb300 as svw
    keep, p = _fake(4096)
    ok_args = dict(t=p, d=p, dt=1, V=64, N=2, cu=p, R=4, ml=16, tok=p, T=1.0, k=20, tp=0.9, seed=0,
                   acc=p, nxt=p, st=None, ws=p, wsb=1 << 30)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spec_verify_filtered(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"], a["ml"],
                                        a["tok"], a["T"], a["k"], a["tp"], a["seed"], a["acc"], a["nxt"], a["st"],
                                        a["ws"], a["wsb"], None)

    assert call(dt=7) == 2
    assert call(k=0) == 1
    assert call(k=1025) == 2                # above SVW_FILTER_MAX_K
    assert call(tp=0.0) == 1
    assert call(tp=1.5) == 1
    assert call(tp=float("nan")) == 1
    assert call(T=-1.0) == 1
    assert call(ws=None) == 4
    assert call(t=ctypes.c_void_p(p.value + 1)) == 3
    need = svw.verify_filtered_workspace_size(2, 4, 64, svw.SVW_BF16)
    assert call(wsb=need - 1) == 4
    for args in ((2, 4, 64, svw.SVW_BF16), (256, 1964, 151936, svw.SVW_BF16)):
        assert svw.verify_filtered_workspace_size(*args) >= svw.verify_workspace_size(*args)


def test_opd_argument_validation(lib):
    keep, p = _fake(4096)

    def call(**kw):
        a = dict(t=p, d=p, dt=1, V=64, N=0, cu=None, R=4, hb=0, T=1.0, c=1.0, lam=0.1, gs=1.0,
                 loss=p, g=p, st=None, ws=None, wsb=0)
        a.update(kw)
        return lib.opd_loss(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"], a["hb"],
                            a["T"], a["c"], a["lam"], a["gs"], a["loss"], a["g"], a["st"],
                            a["ws"], a["wsb"], None)

    assert call(dt=3) == 2
    assert call(R=0) == 1
    assert call(hb=1) == 1                  # bonus layout needs N and cu
    assert call(T=0.0) == 1
    assert call(c=0.0) == 1
    assert call(c=float("nan")) == 1
    assert call(lam=float("inf")) == 1
    assert call(loss=None) == 1
    assert call(g=ctypes.c_void_p(p.value + 4)) == 3   # dlogits must be 16-byte aligned
    assert call(V=1 << 22, dt=0) == 2       # row too wide for the on-chip slices
    assert call(ws=p, wsb=16) == 4          # workspace smaller than svw_opd_workspace_size
    assert call(ws=ctypes.c_void_p(p.value + 16), wsb=4096) == 3


def test_verify_opd_argument_validation(lib):
    keep, p = _fake(4096)

    def call(**kw):
        a = dict(t=p, d=p, dt=1, V=64, N=2, cu=p, R=4, ml=16, tok=p, T=1.0, To=1.0, seed=0, c=1.0,
                 lam=0.1, gs=1.0, acc=p, nxt=p, loss=p, g=p, st=None, ws=p, wsb=1 << 30)
        a.update(kw)
        return lib.spec_verify_opd(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"], a["ml"],
                                   a["tok"], a["T"], a["To"], a["seed"], a["c"], a["lam"], a["gs"],
                                   a["acc"], a["nxt"], a["loss"], a["g"], a["st"], a["ws"], a["wsb"],
                                   None)

    assert call(dt=5) == 2
    assert call(N=0) == 1
    assert call(R=0) == 1
    assert call(ml=33) == 2
    assert call(loss=None) == 1
    assert call(ws=None) == 4
    assert call(wsb=64) == 4
    assert call(To=0.0) == 1                # the reverse-KL temperature must be positive
    assert call(T=0.6, To=1.0) == 1         # sampling softmaxes are shared with the loss
    assert call(T=-1.0) == 1
    assert call(c=0.0) == 1
    assert call(t=ctypes.c_void_p(p.value + 2)) == 3   # bases must be 16-byte aligned
    assert call(V=63) == 2                  # 126-byte rows are not 16-byte pitched
    assert lib.svw_verify_opd_workspace_size(4, 640, 151936, 1) > lib.svw_verify_opd_workspace_size(4, 64, 151936, 1) > 0
    assert lib.svw_verify_opd_workspace_size(0, 64, 1024, 1) == 0


def test_time_next_launch_arming(lib):
    keep, p = _fake(64)
    assert lib.svw_time_next_launch(None, None, None) == 0          # disarm
    assert lib.svw_time_next_launch(b"opd_fast_kernel", None, p) == 1
    assert lib.svw_time_next_launch(b"x" * 80, p, p) == 1             # name too long
    assert lib.svw_time_next_launch(b"opd_fast_kernel", p, p) == 0
    assert lib.svw_time_next_launch(None, None, None) == 0          # and disarm again


def test_length_head_argument_validation(lib):
    keep, p = _fake(4096)

    def call(**kw):
        a = dict(h=p, w1=p, b1=p, w2=p, b2=0.0, N=4, k=16, H=64, Hp=8, g=1.0, a=p, kh=p, ws=p, wsb=1 << 30)
        a.update(kw)
        return lib.length_head(a["h"], a["w1"], a["b1"], a["w2"], a["b2"], a["N"], a["k"], a["H"], a["Hp"],
                               a["g"], a["a"], a["kh"], a["ws"], a["wsb"], None)

    assert call(N=0) == 1
    assert call(k=40) == 2                  # above SVW_MAX_LEN
    assert call(h=None) == 1
    assert call(ws=None) == 4
    assert call(wsb=128) == 4               # needs 64 positions x 4 bytes, rounded up to 256
    assert call(g=0.0) == 1
    assert call(H=60) == 2                  # rows must be 16-byte pitched
    assert call(h=ctypes.c_void_p(p.value + 8)) == 3
    # one fp32 dot per position and 256-wide column tile of W1, rounded up to 256 bytes
    assert lib.svw_length_head_workspace_size(256, 16, 256) == 4096 * 4
    assert lib.svw_length_head_workspace_size(3, 5, 300) == 256
    assert lib.svw_length_head_workspace_size(5, 16, 40) == 512
    assert lib.svw_length_head_workspace_size(40, 13, 600) == 6400  # 3 tiles x 520 x 4 = 6240
    assert lib.svw_length_head_workspace_size(0, 16, 256) == 0
    # at most 2^20 positions (N k)
    assert lib.svw_length_head_workspace_size(1 << 15, 32, 256) == (1 << 20) * 4
    assert lib.svw_length_head_workspace_size((1 << 15) + 1, 32, 256) == 0


def test_noalloc_argument_checks_come_before_the_size_check(lib):
    """spec_verify_noalloc gives spec_verify's codes for bad arguments, even on a
    batch too large for its scratch (which alone gives SVW_ERR_UNSUPPORTED)."""
    keep, p = _fake(4096)
    big = dict(t=p, d=p, dt=1, V=151936, N=4096, cu=p, R=65536, ml=16, tok=p, T=1.0, seed=0,
               acc=p, nxt=p, st=None)

    def call(**kw):
        a = dict(big, **kw)
        return lib.spec_verify_noalloc(a["t"], a["d"], a["dt"], a["V"], a["N"], a["cu"], a["R"], a["ml"],
                                       a["tok"], a["T"], a["seed"], a["acc"], a["nxt"], a["st"], None)

    assert call(t=None) == 1
    assert call(T=float("nan")) == 1
    assert call(cu=ctypes.c_void_p(p.value + 2)) == 3
    assert call(st=ctypes.c_void_p(p.value + 1)) == 3
    assert call(dt=9) == 2
    assert call() == 2                      # valid arguments, batch beyond the scratch
