"""Host-side checks of the C ABI (CPU only, no CUDA call is made).

The library must load, export every function include/li.h declares, and
reject bad arguments with the documented status *before* touching CUDA --
so these run on a machine without a GPU.  Fake device addresses are plain
integers that are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "li.h")

LI_OK, LI_ERR_INVALID_ARG, LI_ERR_ALIGNMENT, LI_ERR_UNSUPPORTED, LI_ERR_WORKSPACE = 0, -1, -2, -3, -4
F32, BF16, FP8 = 0, 1, 2
A = 0x10000      # a fake, 16-byte aligned "device" address (never dereferenced)
MIS = 0x10004    # misaligned


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(li_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L(li):
    return li.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("li_absorb_queries", "li_score_group", "li_topk", "li_hs_select",
              "li_native_score", "li_hs_workspace_size", "li_device_status", "li_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in li.h but not exported"


def test_exports_are_c_symbols(li):
    so = os.path.join(ROOT, "shared_latent_key_cache_b300", "libli_b300.so")
    lib = ctypes.CDLL(so)
    for n in declared_functions():
        getattr(lib, n)   # unmangled lookup succeeds only for extern "C" symbols


def test_selftest_limit_checked_before_any_cuda_call(L):
    for bad in (0, 1_000_001, 4_000_000_000):
        assert L.li_selftest_wait_timeout(bad, None) == -1


def test_version_and_status_strings(L):
    assert L.li_version() >= 100
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert L.li_status_string(s).startswith(b"LI_")
    assert L.li_status_string(12345) == b"unknown status"


def _score(lib, **kw):
    a = dict(latent=A, lat_t=BF16, lat_scale=None, q_abs=A, abs_t=BF16, q_abs_scale=None, w=A,
             beta=None, q_pos=None, B=1, T=1, G=4, H=64, r=192, Lc=1000, scores=A)
    a.update(kw)
    return lib.li_score_group(a["latent"], a["lat_t"], a["lat_scale"], a["q_abs"], a["abs_t"],
                            a["q_abs_scale"], a["w"], a["beta"], a["q_pos"], a["B"], a["T"], a["G"],
                            a["H"], a["r"], a["Lc"], a["scores"], None)


def test_score_group_argument_errors(L):
    assert _score(L, latent=None) == LI_ERR_INVALID_ARG
    assert _score(L, scores=None) == LI_ERR_INVALID_ARG
    assert _score(L, w=None) == LI_ERR_INVALID_ARG
    assert _score(L, lat_t=7) == LI_ERR_INVALID_ARG
    assert _score(L, Lc=0) == LI_ERR_INVALID_ARG
    assert _score(L, H=-1) == LI_ERR_INVALID_ARG
    assert _score(L, lat_t=FP8, abs_t=FP8, q_abs_scale=A) == LI_ERR_INVALID_ARG  # fp8 needs lat_scale
    assert _score(L, lat_t=FP8, abs_t=FP8, lat_scale=A) == LI_ERR_INVALID_ARG    # and q_abs_scale
    assert _score(L, latent=MIS) == LI_ERR_ALIGNMENT
    assert _score(L, beta=MIS) == LI_ERR_ALIGNMENT
    assert _score(L, r=512) == LI_ERR_UNSUPPORTED
    assert _score(L, G=64, H=128, r=256) == LI_ERR_UNSUPPORTED   # too big for either kernel


def test_absorb_argument_errors(L):
    f = L.li_absorb_queries
    assert f(None, BF16, A, BF16, 1, 1, 4, 64, 128, 192, A, BF16, None, None) == LI_ERR_INVALID_ARG
    assert f(A, FP8, A, BF16, 1, 1, 4, 64, 128, 192, A, BF16, None, None) == LI_ERR_INVALID_ARG
    assert f(A, BF16, None, BF16, 1, 1, 4, 64, 128, 192, A, BF16, None, None) == LI_ERR_INVALID_ARG  # D=NULL needs r==d
    assert f(A, BF16, A, BF16, 1, 1, 4, 64, 128, 192, A, FP8, None, None) == LI_ERR_INVALID_ARG     # fp8 needs scale
    assert f(A, BF16, MIS, BF16, 1, 1, 4, 64, 128, 192, A, BF16, None, None) == LI_ERR_ALIGNMENT
    assert f(A, BF16, A, BF16, 1, 1, 4, 64, 128, 300, A, BF16, None, None) == LI_ERR_UNSUPPORTED


def test_topk_argument_errors(L):
    f = L.li_topk
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert f(None, 4, 100, None, 10, A, None, None, 0, None) == LI_ERR_INVALID_ARG
    assert f(A, 4, 100, None, 0, A, None, None, 0, None) == LI_ERR_INVALID_ARG
    assert f(A, -1, 100, None, 10, A, None, None, 0, None) == LI_ERR_INVALID_ARG
    assert f(MIS, 4, 100, None, 10, A, None, None, 0, None) == LI_ERR_ALIGNMENT
    assert f(A, 4, 100, None, 10, A, None, MIS, 1 << 20, None) == LI_ERR_ALIGNMENT
    assert f(A, 0, 100, None, 10, A, None, None, 0, None) == LI_OK   # nothing to do, no CUDA call


def test_topk_workspace_size(L):
    f = L.li_topk_workspace_size
    f.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    f.restype = ctypes.c_size_t
    # rows of 131,072 in four 32,768-score segments: candidates (value + index) per row and segment
    assert f(32, 131072, 2048) == 2 * 32 * 4 * 2048 * 4
    assert f(8, 131072, 8192) == 2 * 8 * 4 * 8192 * 4
    assert f(3, 40000, 100) == 2 * 2560                # 3 rows x 2 segments x 100 x 4 B, 256-aligned
    assert f(32, 32768, 2048) == 0                     # one segment: one pass
    assert f(4, 131072, 16384) == 0                    # candidates exceed one register-resident row
    assert f(0, 131072, 2048) == 0


def test_hs_workspace_size_and_errors(L):
    ws = L.li_hs_workspace_size(8, 4, 131072, 8192, 2048)
    # anchor scores, every layer's candidate scores, anchor top-m in two passes
    assert ws == 8 * 131072 * 4 + 8 * 4 * 8192 * 4 + 2 * 8 * 4 * 8192 * 4
    assert L.li_hs_workspace_size(0, 4, 10, 10, 10) == 0
    f = L.li_hs_select
    args = [A, FP8, A, A, FP8, A, A, None, 2, 4, 64, 192, 1000, 256, 64, A, A, A, ws, None]
    bad_mk = list(args); bad_mk[13] = 32          # m < k
    assert f(*bad_mk) == LI_ERR_INVALID_ARG
    no_ws = list(args); no_ws[17] = None
    assert f(*no_ws) == LI_ERR_WORKSPACE
    small = list(args); small[18] = 16
    assert f(*small) == LI_ERR_WORKSPACE
    mis_ws = list(args); mis_ws[17] = A + 16
    assert f(*mis_ws) == LI_ERR_ALIGNMENT


def test_native_argument_errors(L):
    f = L.li_native_score
    assert f(None, FP8, A, A, FP8, A, A, 1, 64, 128, 100, A, None) == LI_ERR_INVALID_ARG
    assert f(A, FP8, None, A, FP8, A, A, 1, 64, 128, 100, A, None) == LI_ERR_INVALID_ARG
    assert f(A, FP8, A, A, FP8, A, A, 1, 64, 128, 0, A, None) == LI_ERR_INVALID_ARG


def test_append_argument_errors(L):
    f = L.li_append_latent
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    ok = [A, BF16, A, BF16, A, 4, 7168, 192, 64, 10000.0, A, FP8, A, 1024, None]

    def call(**kw):
        args = list(ok)
        names = ["x", "x_t", "P", "P_t", "pos", "B", "dm", "r", "rR", "base", "lat", "lat_t", "sc", "L", "s"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return f(*args)

    assert call(x=None) == LI_ERR_INVALID_ARG
    assert call(pos=None) == LI_ERR_INVALID_ARG
    assert call(rR=63) == LI_ERR_INVALID_ARG          # RoPE pairs
    assert call(rR=194) == LI_ERR_INVALID_ARG         # rR > r
    assert call(r=300, rR=64) == LI_ERR_INVALID_ARG
    assert call(sc=None) == LI_ERR_INVALID_ARG        # fp8 cache needs its scales
    assert call(base=0.0) == LI_ERR_INVALID_ARG
    assert call(lat_t=7) == LI_ERR_INVALID_ARG
    assert call(x=MIS) == LI_ERR_ALIGNMENT
    assert call(B=0) == LI_OK                         # nothing to do, no CUDA call


def test_hs_profiled_needs_its_events(L):
    ws = L.li_hs_workspace_size(2, 4, 1000, 256, 64)
    assert L.li_hs_select_profiled(A, FP8, A, A, FP8, A, A, None, 2, 4, 64, 192, 1000, 256, 64,
                                   A, A, A, ws, None, None) == LI_ERR_INVALID_ARG


def test_hs_noalloc_reports_argument_errors_like_hs_select(L):
    """The no-allocation entry point runs li_hs_select's argument checks before
    its scratch-size limit: a call that is both malformed and too large gets
    the argument error, as li_hs_select would give it."""
    f = L.li_hs_select_noalloc
    big = [A, FP8, A, A, FP8, A, A, None, 64, 4, 64, 192, 131072, 8192, 2048, A, A, None]
    assert f(*big) == LI_ERR_WORKSPACE                          # valid, but more than 8 MiB of scratch
    mis = list(big); mis[0] = MIS
    assert f(*mis) == LI_ERR_ALIGNMENT
    bad_t = list(big); bad_t[1] = 9
    assert f(*bad_t) == LI_ERR_INVALID_ARG
    no_scale = list(big); no_scale[2] = None                    # fp8 latent without its scales
    assert f(*no_scale) == LI_ERR_INVALID_ARG
    bad_mk = list(big); bad_mk[13] = 1024                       # m < k
    assert f(*bad_mk) == LI_ERR_INVALID_ARG
