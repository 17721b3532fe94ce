"""CPU oracle of the LatentIndex indexer scan -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never does,
and this package never imports the product: the two share no code.

Layers:

* ``li_oracle.c`` (built to ``liboracle.so``): plain fp64 loops with OpenMP,
  written from the equations of the LatentIndex pages (see that file's header
  for the citations).  This is the oracle the GPU path is checked against.
* ``twin.py``: a second, independent fp64 implementation of the same
  definitions in numpy, for small cases.  The two are cross-checked.
* this module: ctypes marshalling, plus the storage arithmetic of the
  explainer page and the HS position count of the summary page.

Parity pins (tests/test_oracle_pins.py) tie the oracle to what the pages and
the mathematics fix: a hand-worked example, the exact dot-product identity
of eq. (7), library decoders for fp8/bf16, brute-force sorts, the HS limits
and the pages' storage numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "li_oracle.c")

OR_F32, OR_BF16, OR_FP8, OR_F64 = 0, 1, 2, 3

_lib = None


def build(force: bool = False) -> str:
    """Compile li_oracle.c with gcc (-O2 -fopenmp) into liboracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
                        "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.or_e4m3_decode.restype = D
        L.or_bf16_decode.argtypes = [ctypes.c_uint16]
        L.or_bf16_decode.restype = D
        L.or_decode_rows.argtypes = [P, I, P, I64, I64, P]
        L.or_absorb.argtypes = [P, I, P, I, I64, I, I, I, I, P, I]
        L.or_reconstruct_keys.argtypes = [P, I, P, P, I, I, I, I, I, I, P, I]
        L.or_score.argtypes = [P, I, P, P, P, P, P, I, I, I, I, I, I, P, I]
        L.or_topk.argtypes = [P, I64, I, P, I, P, P, I]
        L.or_hs.argtypes = [P, I, I, I, I, I, P, P, I]
        L.or_native_score.argtypes = [P, I, P, P, P, I, I, I, I, P, I]
        L.or_append_latent.argtypes = [P, I, P, I, I, I, I, I, ctypes.c_double, P, P, I]
        L.or_rope_rotate.argtypes = [P, I64, I, I, ctypes.c_double, P]
        L.or_rotary_decoder.argtypes = [P, P, I, I, P]
        L.or_rope_keys.argtypes = [P, I, P, I, I, I, I, I, P, P, P, I, I, I, ctypes.c_double, P, P, I]
        for f in ("or_decode_rows", "or_absorb", "or_reconstruct_keys", "or_score", "or_topk",
                  "or_hs", "or_native_score", "or_append_latent", "or_rope_rotate",
                  "or_rotary_decoder", "or_rope_keys"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- marshalling

def _np(x):
    """Host numpy view of a tensor/array (torch tensors are moved to the CPU)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def _code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return OR_F32
    if a.dtype == np.uint16:
        return OR_BF16
    if a.dtype == np.uint8:
        return OR_FP8
    if a.dtype == np.float64:
        return OR_F64
    raise TypeError(f"unsupported storage dtype {a.dtype}")


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(_np(a), dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(_np(a), dtype=np.float64)


# ------------------------------------------------------------------ functions

def e4m3_decode(code: int) -> float:
    return lib().or_e4m3_decode(code)


def bf16_decode(bits: int) -> float:
    return lib().or_bf16_decode(bits)


def decode_rows(x, scale=None) -> np.ndarray:
    """fp64 values of stored rows (last dim = row), times the per-row scale if given."""
    a = np.ascontiguousarray(_np(x))
    s = _f32(scale)
    cols = a.shape[-1] if a.ndim else 1
    rows = a.size // cols if cols else 0
    out = np.empty(a.shape, dtype=np.float64)
    lib().or_decode_rows(_p(a), _code(a), _p(s), rows, cols, _p(out))
    return out


def absorb(q, D, nthreads: int | None = None) -> np.ndarray:
    """Eq. (6): q~ = D_l q.  q [..., G, H, d], D [G, r, d] -> [..., G, H, r] fp64."""
    qa, Da = np.ascontiguousarray(_np(q)), np.ascontiguousarray(_np(D))
    G, H, d = qa.shape[-3:]
    r = Da.shape[1]
    N = qa.size // (G * H * d)
    out = np.empty(qa.shape[:-1] + (r,), dtype=np.float64)
    lib().or_absorb(_p(qa), _code(qa), _p(Da), _code(Da), N, G, H, d, r, _p(out),
                    nthreads or default_threads())
    return out


def reconstruct_keys(latent, lat_scale, D, nthreads: int | None = None) -> np.ndarray:
    """Eq. (3) (no bias): k^l_t = D_l^T c_t.  -> [G][B][L][d] fp64."""
    la, Da = np.ascontiguousarray(_np(latent)), np.ascontiguousarray(_np(D))
    s = _f32(lat_scale)
    B, L, r = la.shape
    G, _, d = Da.shape
    out = np.empty((G, B, L, d), dtype=np.float64)
    lib().or_reconstruct_keys(_p(la), _code(la), _p(s), _p(Da), _code(Da), B, L, G, r, d,
                              _p(out), nthreads or default_threads())
    return out


def score(latent, lat_scale, qabs, w, beta=None, q_pos=None,
          nthreads: int | None = None) -> np.ndarray:
    """Eq. (8) for every query, layer and token -> scores [B][T][G][L] fp64 (-inf outside V).

    latent [B][L][r] stored (f32/bf16/fp8 codes) or fp64; lat_scale [B][L] or None;
    qabs [B][T][G][H][r] (fp64 values); w [B][T][G][H]; beta same or None; q_pos [T] or None.
    """
    la = np.ascontiguousarray(_np(latent))
    s = _f32(lat_scale)
    qa = _f64(qabs)
    wa = _f64(w)
    ba = _f64(beta)
    pa = None if q_pos is None else np.ascontiguousarray(_np(q_pos), dtype=np.int32)
    B, L, r = la.shape
    _, T, G, H, r2 = qa.shape
    assert r2 == r and r <= 1024
    out = np.empty((B, T, G, L), dtype=np.float64)
    lib().or_score(_p(la), _code(la), _p(s), _p(qa), _p(wa), _p(ba), _p(pa), B, T, G, H, r, L,
                   _p(out), nthreads or default_threads())
    return out


def topk(scores, k: int, valid_len=None, nthreads: int | None = None):
    """TopK per row of scores [..., L]: (idx [..., k] int32 -1 padded, vals [..., k] fp64)."""
    sa = _f64(scores)
    L = sa.shape[-1]
    rows = sa.size // L if L else 0
    va = None if valid_len is None else np.ascontiguousarray(_np(valid_len), dtype=np.int32).reshape(-1)
    idx = np.empty(sa.shape[:-1] + (k,), dtype=np.int32)
    vals = np.empty(sa.shape[:-1] + (k,), dtype=np.float64)
    lib().or_topk(_p(sa), rows, L, _p(va), k, _p(idx), _p(vals), nthreads or default_threads())
    return idx, vals


def hs(scores, m: int, k: int, nthreads: int | None = None):
    """Hierarchical selection from per-layer score rows [B][G][L]: (cand [B][m], idx [B][G][k])."""
    sa = _f64(scores)
    B, G, L = sa.shape
    cand = np.empty((B, m), dtype=np.int32)
    idx = np.empty((B, G, k), dtype=np.int32)
    lib().or_hs(_p(sa), B, G, L, m, k, _p(cand), _p(idx), nthreads or default_threads())
    return cand, idx


def append_latent(x, P, rR: int, pos, base: float = 10000.0, nthreads: int | None = None) -> np.ndarray:
    """Eqs. (1)-(2): c = [Q_t P_R^T x ; P_N^T x] per sequence.  x [B][dm],
    P [r][dm] (rows < rR: P_R^T), pos [B] -> c [B][r] fp64 (before storage)."""
    xa, Pa = np.ascontiguousarray(_np(x)), np.ascontiguousarray(_np(P))
    B, dm = xa.shape
    r = Pa.shape[0]
    pa = np.ascontiguousarray(_np(pos), dtype=np.int32).reshape(-1)
    out = np.empty((B, r), dtype=np.float64)
    lib().or_append_latent(_p(xa), _code(xa), _p(Pa), _code(Pa), B, dm, r, rR, float(base), _p(pa),
                           _p(out), nthreads or default_threads())
    return out


def rope_rotate(v, nR: int, pos, base: float = 10000.0) -> np.ndarray:
    """Rotary encoding of the first nR entries of each row of v [n][dim] by its
    position pos [n] (R_t of eq. (4) on a key's RoPE part; Q_t on a latent's
    RoPE branch).  Returns a new fp64 array."""
    out = np.array(_f64(v), dtype=np.float64, copy=True, order="C")
    n, dim = out.shape
    pa = np.ascontiguousarray(_np(pos), dtype=np.int32).reshape(-1)
    assert pa.size == n and nR % 2 == 0 and nR <= dim
    lib().or_rope_rotate(_p(out), n, dim, nR, float(base), _p(pa))
    return out


def rotary_decoder(a_re, a_im, dR: int, rR: int) -> np.ndarray:
    """RoPE part D^R [dR][rR] of a decoder under eq. (4), R_t D^R = D^R Q_t:
    key pair j and latent pair i are coupled by the complex number
    a_re[j][i] + i a_im[j][i] when their rotary frequencies are equal
    (j * rR == i * dR), and not at all otherwise.  a_re, a_im [dR/2][rR/2]."""
    ar = np.ascontiguousarray(_f64(a_re)).reshape(dR // 2, rR // 2)
    ai = np.ascontiguousarray(_f64(a_im)).reshape(dR // 2, rR // 2)
    out = np.empty((dR, rR), dtype=np.float64)
    lib().or_rotary_decoder(_p(ar), _p(ai), dR, rR, _p(out))
    return out


def rope_keys(x, P, rR: int, DR, DN, pos, bias=None, base: float = 10000.0,
              nthreads: int | None = None) -> np.ndarray:
    """Eq. (3) the native way: per-layer keys [R_t D^R_l P_R^T x ; D^N_l P_N^T x + b_l]
    of the token of each sequence at position pos [B].  x [B][dm], P [r][dm],
    DR [G][dR][rR], DN [G][dN][r - rR], bias [G][dN] or None -> keys [G][B][dR + dN]."""
    xa, Pa = np.ascontiguousarray(_np(x)), np.ascontiguousarray(_np(P))
    B, dm = xa.shape
    r = Pa.shape[0]
    DRa, DNa = _f64(DR), _f64(DN)
    G, dR, rR2 = DRa.shape
    _, dN, rN = DNa.shape
    assert rR2 == rR and rN == r - rR and r <= 1024
    ba = _f64(bias)
    pa = np.ascontiguousarray(_np(pos), dtype=np.int32).reshape(-1)
    out = np.empty((G, B, dR + dN), dtype=np.float64)
    lib().or_rope_keys(_p(xa), _code(xa), _p(Pa), _code(Pa), B, dm, r, rR, _p(DRa), _p(DNa), _p(ba),
                       G, dR, dN, float(base), _p(pa), _p(out), nthreads or default_threads())
    return out


def native_score(keys, key_scale, q, w, nthreads: int | None = None) -> np.ndarray:
    """Native per-layer DSA indexer: keys [B][L][d] (+scale), q [B][H][d], w [B][H] -> [B][L]."""
    ka = np.ascontiguousarray(_np(keys))
    s = _f32(key_scale)
    qa, wa = _f64(q), _f64(w)
    B, L, d = ka.shape
    H = qa.shape[1]
    out = np.empty((B, L), dtype=np.float64)
    lib().or_native_score(_p(ka), _code(ka), _p(s), _p(qa), _p(wa), B, H, d, L, _p(out),
                          nthreads or default_threads())
    return out


def decode_queries(q, scale=None) -> np.ndarray:
    """fp64 values of stored (absorbed) query rows, with optional per-row scale."""
    return decode_rows(q, scale)


# ------------------------------------------------- arithmetic fixed by the pages

def indexer_cache_bytes_per_token(n_layers: int, group: int, native_key_bytes: int,
                                  latent_bytes: int, native_layers: int = 1) -> tuple[int, int]:
    """Indexer side-cache bytes per token: (native DSA, LatentIndex).

    Explainer page, storage paragraph: native DSA keeps one key per layer
    (n_layers * native_key_bytes); LatentIndex keeps the first `native_layers`
    layers native and turns the rest into groups of `group` layers that each
    store one latent of `latent_bytes`.
    """
    native = n_layers * native_key_bytes
    shared = n_layers - native_layers
    assert shared % group == 0
    latent = native_layers * native_key_bytes + (shared // group) * latent_bytes
    return native, latent


def payload_ratio(d_c: int, group: int, d_i: int) -> float:
    """Summary page, "Storage Efficiency": one d_C latent instead of m keys of d_I -> d_C/(m d_I)."""
    return d_c / (group * d_i)


def hs_scored_positions(L: int, group: int, m: int) -> int:
    """Summary page, "Hierarchical Selection": scored positions per query per group,
    L + (G-1) min(m, L), against G*L for the full scan."""
    return L + (group - 1) * min(m, L)
