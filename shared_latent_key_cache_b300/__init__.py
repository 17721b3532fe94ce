"""Python binding of libli_b300.so -- the LatentIndex indexer scan on B300.

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions named ``li_*`` mirror the C ABI of ``include/li.h`` one to one
and take torch tensors (device memory) plus an optional stream; the
lower-case helpers (``absorb_queries``, ``score_group``, ``topk``,
``hs_select``, ``native_score``) allocate the outputs with torch and call
them.  There is no fallback: if the CUDA library cannot be loaded, importing
this package raises.

Storage types: torch.float32 -> LI_F32, torch.bfloat16 -> LI_BF16, and
torch.uint8 / torch.float8_e4m3fn (E4M3 codes, with a separate fp32
per-row scale tensor) -> LI_FP8_E4M3.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "LI_F32", "LI_BF16", "LI_FP8_E4M3", "LiError", "lib", "library_path",
    "li_version", "li_status_string", "li_absorb_queries", "li_score_group", "li_topk",
    "li_topk_workspace_size",
    "li_hs_workspace_size", "li_hs_select", "li_hs_select_profiled", "li_hs_select_noalloc",
    "li_native_score",
    "li_device_status", "li_selftest_wait_timeout", "li_append_latent", "append_latent",
    "absorb_queries", "score_group", "topk", "hs_select", "native_score", "device_status",
]

LI_F32, LI_BF16, LI_FP8_E4M3 = 0, 1, 2
LI_OK = 0

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libli_b300.so")


class LiError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.li_status_string(status).decode()} ({status})")


def _load():
    if not os.path.exists(library_path):
        raise ImportError(
            f"{library_path} is missing: build it with "
            "`python shared_latent_key_cache_b300/_build.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(library_path)
    P, I, I64, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.li_version.restype = I
    L.li_status_string.argtypes = [I]
    L.li_status_string.restype = ctypes.c_char_p
    L.li_absorb_queries.argtypes = [P, I, P, I, I, I, I, I, I, I, P, I, P, P]
    L.li_score_group.argtypes = [P, I, P, P, I, P, P, P, P, I, I, I, I, I, I, P, P]
    L.li_topk.argtypes = [P, I64, I, P, I, P, P, P, S, P]
    L.li_topk_workspace_size.argtypes = [I64, I, I]
    L.li_topk_workspace_size.restype = S
    L.li_hs_workspace_size.argtypes = [I, I, I, I, I]
    L.li_hs_workspace_size.restype = S
    L.li_hs_select.argtypes = [P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, P, P, P, S, P]
    L.li_native_score.argtypes = [P, I, P, P, I, P, P, I, I, I, I, P, P]
    L.li_hs_select_noalloc.argtypes = [P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, P, P, P]
    L.li_hs_select_profiled.argtypes = [P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, P, P, P, S, P, P]
    L.li_device_status.argtypes = [P]
    L.li_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
    L.li_append_latent.argtypes = [P, I, P, I, P, I, I, I, I, ctypes.c_float, P, I, P, I, P]
    for f in ("li_absorb_queries", "li_score_group", "li_topk", "li_hs_select", "li_hs_select_profiled",
              "li_native_score", "li_device_status", "li_hs_select_noalloc",
              "li_selftest_wait_timeout", "li_append_latent"):
        getattr(L, f).restype = I
    return L


_lib = _load()


def lib():
    """The loaded ctypes library."""
    return _lib


# ---------------------------------------------------------------- marshalling

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LI_F32
    if t.dtype == torch.bfloat16:
        return LI_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return LI_FP8_E4M3
    raise TypeError(f"unsupported storage dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, what: str):
    if status != LI_OK:
        raise LiError(status, what)


# ------------------------------------------------------- one-to-one C entries

def li_version() -> int:
    return _lib.li_version()


def li_status_string(status: int) -> str:
    return _lib.li_status_string(status).decode()


def li_absorb_queries(q, D, q_abs, q_abs_scale=None, stream=None) -> int:
    """q [B][T][G][H][d], D [G][r][d] or None (identity) -> q_abs [B][T][G][H][r] (+ scale)."""
    B, T, G, H, d = q.shape
    r = q_abs.shape[-1]
    return _lib.li_absorb_queries(
        _ptr(q), _dtype_code(q), _ptr(D), _dtype_code(D) if D is not None else LI_F32,
        B, T, G, H, d, r, _ptr(q_abs), _dtype_code(q_abs), _ptr(q_abs_scale), _stream(stream))


def li_score_group(latent, lat_scale, q_abs, q_abs_scale, w, scores, beta=None, q_pos=None,
                   stream=None) -> int:
    """latent [B][L][r], q_abs [B][T][G][H][r], w [B][T][G][H] -> scores [B][T][G][L]."""
    B, L, r = latent.shape
    _, T, G, H, _ = q_abs.shape
    return _lib.li_score_group(
        _ptr(latent), _dtype_code(latent), _ptr(lat_scale), _ptr(q_abs), _dtype_code(q_abs),
        _ptr(q_abs_scale), _ptr(w), _ptr(beta), _ptr(q_pos), B, T, G, H, r, L, _ptr(scores),
        _stream(stream))


def li_topk_workspace_size(rows: int, L: int, k: int) -> int:
    return _lib.li_topk_workspace_size(rows, L, k)


def li_topk(scores, k: int, idx, vals=None, valid_len=None, ws=None, stream=None) -> int:
    """scores [..., L] -> idx [..., k] int32 (+ vals [..., k]); ws: optional uint8 workspace."""
    L = scores.shape[-1]
    rows = scores.numel() // L if L else 0
    return _lib.li_topk(_ptr(scores), rows, L, _ptr(valid_len), k, _ptr(idx), _ptr(vals),
                        _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
                        _stream(stream))


def li_hs_workspace_size(B: int, G: int, L: int, m: int, k: int) -> int:
    return _lib.li_hs_workspace_size(B, G, L, m, k)


def li_hs_select(latent, lat_scale, q_abs, q_abs_scale, w, m: int, k: int, cand, idx, ws,
                 beta=None, stream=None) -> int:
    """latent [B][L][r], q_abs [B][1][G][H][r] -> cand [B][m], idx [B][G][k] (ws: uint8 workspace)."""
    B, L, r = latent.shape
    _, T, G, H, _ = q_abs.shape
    assert T == 1
    return _lib.li_hs_select(
        _ptr(latent), _dtype_code(latent), _ptr(lat_scale), _ptr(q_abs), _dtype_code(q_abs),
        _ptr(q_abs_scale), _ptr(w), _ptr(beta), B, G, H, r, L, m, k, _ptr(cand), _ptr(idx),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def li_hs_select_profiled(latent, lat_scale, q_abs, q_abs_scale, w, m: int, k: int, cand, idx, ws,
                          events, beta=None, stream=None) -> int:
    """li_hs_select with five torch.cuda.Event objects recorded around its four launches.
    torch creates an event's CUDA handle on its first record, so each event is
    recorded once here (on the same stream) before the library records it again."""
    B, L, r = latent.shape
    _, _, G, H, _ = q_abs.shape
    st = stream if stream is not None else torch.cuda.current_stream()
    for e in events:
        e.record(st)
    arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return _lib.li_hs_select_profiled(
        _ptr(latent), _dtype_code(latent), _ptr(lat_scale), _ptr(q_abs), _dtype_code(q_abs),
        _ptr(q_abs_scale), _ptr(w), _ptr(beta), B, G, H, r, L, m, k, _ptr(cand), _ptr(idx),
        _ptr(ws), ws.numel() * ws.element_size(), arr, _stream(stream))


def li_hs_select_noalloc(latent, lat_scale, q_abs, q_abs_scale, w, m: int, k: int, cand, idx,
                         beta=None, stream=None) -> int:
    """As li_hs_select, with the library's built-in 8 MiB scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, L, r = latent.shape
    _, T, G, H, _ = q_abs.shape
    assert T == 1
    return _lib.li_hs_select_noalloc(
        _ptr(latent), _dtype_code(latent), _ptr(lat_scale), _ptr(q_abs), _dtype_code(q_abs),
        _ptr(q_abs_scale), _ptr(w), _ptr(beta), B, G, H, r, L, m, k, _ptr(cand), _ptr(idx),
        _stream(stream))


def li_native_score(keys, key_scale, q, q_scale, w, scores, stream=None) -> int:
    """keys [B][L][d], q [B][H][d], w [B][H] -> scores [B][L]."""
    B, L, d = keys.shape
    H = q.shape[1]
    return _lib.li_native_score(
        _ptr(keys), _dtype_code(keys), _ptr(key_scale), _ptr(q), _dtype_code(q), _ptr(q_scale),
        _ptr(w), B, H, d, L, _ptr(scores), _stream(stream))


def li_device_status(stream=None) -> int:
    return _lib.li_device_status(_stream(stream))


def li_append_latent(x, P, pos, rR: int, latent, lat_scale=None, rope_base: float = 10000.0,
                     stream=None) -> int:
    """x [B][dm], P [r][dm] (rows < rR: P_R^T), pos [B] int32 -> row pos[b] of latent [B][L][r]."""
    B, dm = x.shape
    r = P.shape[0]
    L = latent.shape[1]
    return _lib.li_append_latent(_ptr(x), _dtype_code(x), _ptr(P), _dtype_code(P), _ptr(pos), B, dm, r,
                                 rR, float(rope_base), _ptr(latent), _dtype_code(latent),
                                 _ptr(lat_scale), L, _stream(stream))


def li_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    """Launch the watchdog test kernel (a bounded wait that is never satisfied)."""
    return _lib.li_selftest_wait_timeout(int(limit_us), _stream(stream))


# ------------------------------------------------------- allocating helpers

def absorb_queries(q, D, abs_dtype: str = "bf16", stream=None):
    """Eq. (6) of the summary page: returns (q_abs, q_abs_scale or None)."""
    B, T, G, H, d = q.shape
    r = D.shape[1] if D is not None else d
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[abs_dtype]
    q_abs = torch.empty(B, T, G, H, r, dtype=dt, device=q.device)
    scale = torch.empty(B, T, G, H, dtype=torch.float32, device=q.device) if abs_dtype == "fp8" else None
    _check(li_absorb_queries(q, D, q_abs, scale, stream), "li_absorb_queries")
    return q_abs, scale


def score_group(latent, lat_scale, q_abs, q_abs_scale, w, beta=None, q_pos=None, out=None,
                stream=None):
    """Eq. (8) for all layers of the group: returns scores [B][T][G][L] (fp32)."""
    B, L, _ = latent.shape
    _, T, G, _, _ = q_abs.shape
    if out is None:
        out = torch.empty(B, T, G, L, dtype=torch.float32, device=latent.device)
    _check(li_score_group(latent, lat_scale, q_abs, q_abs_scale, w, out, beta, q_pos, stream),
           "li_score_group")
    return out


def topk(scores, k: int, valid_len=None, with_vals: bool = False, out=None, ws=None, stream=None):
    """Per-row TopK: returns idx [..., k] int32 (and vals when asked).  Long rows
    get a workspace (allocated here unless `ws` is given) for the two-pass path."""
    shape = scores.shape[:-1] + (k,)
    idx = out if out is not None else torch.empty(shape, dtype=torch.int32, device=scores.device)
    vals = torch.empty(shape, dtype=torch.float32, device=scores.device) if with_vals else None
    if ws is None and scores.shape[-1] > 0:
        n = li_topk_workspace_size(scores.numel() // scores.shape[-1], scores.shape[-1], k)
        if n > 0:
            ws = torch.empty(n, dtype=torch.uint8, device=scores.device)
    _check(li_topk(scores, k, idx, vals, valid_len, ws, stream), "li_topk")
    return (idx, vals) if with_vals else idx


def hs_select(latent, lat_scale, q_abs, q_abs_scale, w, m: int, k: int, beta=None, ws=None,
              stream=None):
    """Hierarchical selection: returns (cand [B][m], idx [B][G][k])."""
    B, L, _ = latent.shape
    G = q_abs.shape[2]
    cand = torch.empty(B, m, dtype=torch.int32, device=latent.device)
    idx = torch.empty(B, G, k, dtype=torch.int32, device=latent.device)
    if ws is None:
        ws = torch.empty(li_hs_workspace_size(B, G, L, m, k), dtype=torch.uint8, device=latent.device)
    _check(li_hs_select(latent, lat_scale, q_abs, q_abs_scale, w, m, k, cand, idx, ws, beta, stream),
           "li_hs_select")
    return cand, idx


def native_score(keys, key_scale, q, q_scale, w, out=None, stream=None):
    """Native per-layer DSA indexer: returns scores [B][L]."""
    B, L, _ = keys.shape
    if out is None:
        out = torch.empty(B, L, dtype=torch.float32, device=keys.device)
    _check(li_native_score(keys, key_scale, q, q_scale, w, out, stream), "li_native_score")
    return out


def append_latent(x, P, pos, rR: int, latent, lat_scale=None, rope_base: float = 10000.0,
                  stream=None):
    """Eqs. (1)-(2): writes the new tokens' latents into the cache (in place)."""
    _check(li_append_latent(x, P, pos, rR, latent, lat_scale, rope_base, stream), "li_append_latent")


def device_status(stream=None) -> int:
    return li_device_status(stream)
