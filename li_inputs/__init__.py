"""Seeded synthetic inputs for the LatentIndex indexer scan.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle's tests.  It holds none of the method's arithmetic (no absorption,
scoring, selection or candidate logic): it only draws random tensors with the
shapes and value distributions of the indexer workloads and stores them in
the storage formats the scan reads:

* ``f32``  -- float32 values;
* ``bf16`` -- torch.bfloat16 values (round-to-nearest-even from float32);
* ``fp8``  -- OCP FP8 E4M3 ("fn") codes as torch.uint8, plus one float32
  scale per stored row, value = scale * decode(code).  The scale of a row is
  its absolute maximum / 448 (the largest finite E4M3 magnitude).

Shapes follow the layouts of the C ABI:

* latent ``[B][L][r]`` (+ ``lat_scale [B][L]``)
* decoders ``D [G][r][d]`` (layer l maps a d-dim query to the r-dim latent
  space: q~ = D_l q; the per-layer key is k = D_l^T c)
* queries ``q [B][T][G][H][d]``, head weights ``w [B][T][G][H]``
* causal positions ``q_pos [T]`` (prefill only)
* native per-layer key caches ``keys [G][B][L][d]`` fp8 + ``key_scale [G][B][L]``

The native keys are built as fp8(D_l^T c) from the *stored* latent, as the
DSA-shaped workload asks; they are an input of the native scan only and the
parity of that scan does not depend on how they were made.

Distributions (the indexer workloads of the LatentIndex pages: DeepSeek-V3.2
shaped, H=64 indexer heads, d=128, a 192-value latent, top-2048):
c ~ N(0,1) with floor(0.01 L) "heavy" tokens per sequence (a seeded
permutation) scaled x4 before quantisation; D ~ N(0, 1/r); q ~ N(0, 1/d);
w ~ U(0,1).  The 128K HS workload mixes q = 0.7 q_shared + 0.3 q_own.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "spec", "make_workload", "make_latent",
           "make_absorbed_queries", "make_rotary_decoders", "quantize_rows_fp8", "FP8_MAX"]

FP8_MAX = 448.0

# Per-tensor stream ids: each tensor gets its own generator seeded from
# (seed, stream id) so adding a tensor never shifts another one's values.
_S_LATENT, _S_HEAVY, _S_D, _S_Q, _S_QSHARED, _S_W, _S_QABS, _S_QABS_SCALE, _S_BETA = range(9)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7919 + 17) & 0x7FFF_FFFF_FFFF)
    return g


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    G: int
    H: int
    d: int
    r: int
    L: int
    k: int
    lat_dtype: str          # "f32" | "bf16" | "fp8"
    q_dtype: str            # dtype of q and D: "f32" | "bf16"
    m: int = 0              # HS candidate budget (0: no HS)
    pos0: int = -1          # first causal position for prefill (-1: decode, all L valid)
    mix_shared: float = 0.0 # q = mix*q_shared + (1-mix)*q_own when > 0
    native: bool = False    # also build per-layer fp8 key caches
    description: str = ""


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=1, T=1, G=4, H=8, d=64, r=32, L=4096, k=256,
                         lat_dtype="f32", q_dtype="f32",
                         description="Tiny CPU-checkable group, fp32, L=4096, top-256"),
    "dsa_bf16_8k": Workload("dsa_bf16_8k", B=1, T=1, G=4, H=64, d=128, r=192, L=8192, k=2048,
                            lat_dtype="bf16", q_dtype="bf16", native=True,
                            description="DSA-shaped decode, bf16 latent, 8K context, batch 1"),
    "fp8_32k_b32": Workload("fp8_32k_b32", B=32, T=1, G=4, H=64, d=128, r=192, L=32768, k=2048,
                            lat_dtype="fp8", q_dtype="bf16", native=True,
                            description="Batched decode, 32 sequences x 32K, fp8 latent + per-token scale"),
    "fp8_128k_hs": Workload("fp8_128k_hs", B=8, T=1, G=4, H=64, d=128, r=192, L=131072, k=2048,
                            lat_dtype="fp8", q_dtype="bf16", m=8192, mix_shared=0.7,
                            description="128K decode, batch 8, full scan vs HS (m=8192)"),
    "prefill_bf16_128k": Workload("prefill_bf16_128k", B=1, T=4096, G=4, H=64, d=128, r=192,
                                  L=131072, k=2048, lat_dtype="bf16", q_dtype="bf16",
                                  pos0=131072 - 4096,
                                  description="Chunked prefill, 4096 queries at 126976..131071, causal"),
}


def spec(name: str, **overrides) -> Workload:
    """The named workload, optionally with some fields replaced (smaller test shapes)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


def quantize_rows_fp8(x: torch.Tensor):
    """Per-row FP8 E4M3 storage of a float tensor: returns (codes uint8, scale f32).

    The row is the last dimension; scale = amax(|row|)/448, codes = RNE(x/scale)
    saturated to +-448.  A zero row gets scale 0 and zero codes.
    """
    x = x.float()
    amax = x.abs().amax(dim=-1)
    scale = amax / FP8_MAX
    inv = torch.where(scale > 0, 1.0 / scale, torch.zeros_like(scale))
    y = (x * inv.unsqueeze(-1)).clamp_(-FP8_MAX, FP8_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.contiguous()


def _store(x: torch.Tensor, dtype: str):
    if dtype == "f32":
        return x.float().contiguous(), None
    if dtype == "bf16":
        return x.to(torch.bfloat16).contiguous(), None
    if dtype == "fp8":
        return quantize_rows_fp8(x)
    raise ValueError(dtype)


def _dequant(stored: torch.Tensor, scale, dtype: str) -> torch.Tensor:
    """Float32 view of stored values (used only to build native key caches)."""
    if dtype == "fp8":
        return stored.view(torch.float8_e4m3fn).float() * scale.unsqueeze(-1)
    return stored.float()


def make_latent(B: int, L: int, r: int, dtype: str, seed: int = 0, device="cpu"):
    """Shared latent cache c[B][L][r] ~ N(0,1) with floor(0.01 L) heavy tokens x4.

    Returns (latent, lat_scale or None, heavy index tensor [B][n_heavy]).
    """
    g = _gen(seed, _S_LATENT, device)
    c = torch.randn(B, L, r, generator=g, device=device, dtype=torch.float32)
    n_heavy = (L * 1) // 100
    gh = _gen(seed, _S_HEAVY, device)
    heavy = torch.stack([torch.randperm(L, generator=gh, device=device)[:n_heavy] for _ in range(B)]) \
        if n_heavy > 0 else torch.zeros(B, 0, dtype=torch.long, device=device)
    if n_heavy > 0:
        bidx = torch.arange(B, device=device).unsqueeze(1).expand_as(heavy)
        c[bidx, heavy] *= 4.0
    lat, scale = _store(c, dtype)
    return lat, scale, heavy


def make_absorbed_queries(B: int, T: int, G: int, H: int, r: int, dtype: str, seed: int = 0,
                          device="cpu", std: float | None = None):
    """Random absorbed-query rows q~[B][T][G][H][r] stored in `dtype` (+ per-row scale for fp8).

    Used to exercise the scoring step on its own.  Default std 1/sqrt(r).
    """
    g = _gen(seed, _S_QABS, device)
    s = (1.0 / math.sqrt(r)) if std is None else std
    x = torch.randn(B, T, G, H, r, generator=g, device=device) * s
    return _store(x, dtype)


def make_beta(B: int, T: int, G: int, H: int, seed: int = 0, device="cpu", std: float = 0.5):
    g = _gen(seed, _S_BETA, device)
    return (torch.randn(B, T, G, H, generator=g, device=device) * std).contiguous()


def make_append_inputs(B: int, dm: int, r: int, dtype: str = "bf16", seed: int = 0, device="cpu"):
    """Inputs of the latent append: the anchor layer's hidden states x [B][dm]
    ~ N(0, 1) and the stacked projections P [r][dm] ~ N(0, 1/dm) (rows < rR
    are P_R^T), stored as `dtype` ("f32" or "bf16")."""
    x = torch.randn(B, dm, generator=_gen(seed, 21, "cpu"))
    P = torch.randn(r, dm, generator=_gen(seed, 22, "cpu")) / dm ** 0.5
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    return x.to(dt).to(device), P.to(dt).to(device)


def make_rotary_decoders(G: int, r: int, rR: int, d: int, dR: int, seed: int = 0):
    """Random decoders whose RoPE part obeys the rotary-structure constraint
    (summary page, eqs. (3)-(4)), as raw draws plus their storage.

    Key RoPE pair j (of dR/2) and latent RoPE pair i (of rR/2) are coupled by
    one complex number (a_re + i a_im)[l][j][i] when j * rR == i * dR (their
    rotary frequencies are equal) and not at all otherwise; the NoPE block maps
    the r - rR latent NoPE values to the d - dR key NoPE values.  Draws:
    a_re, a_im, DN ~ N(0, 1/r), rounded to bfloat16 so that the f32 and bf16
    storages hold exactly the drawn values.

    Returns a dict with a_re, a_im [G][dR/2][rR/2], DN [G][d - dR][r - rR]
    (float64 tensors) and D [G][r][d] float32, the decoders in the library's
    storage orientation (k = D_l^T c): rows < rR / columns < dR carry the
    2 x 2 blocks [[a, -b], [b, a]] transposed, rows >= rR / columns >= dR
    carry DN transposed, the rest is zero."""
    g = torch.Generator().manual_seed((int(seed) * 1_000_003 + 31 * 7919 + 17) & 0x7FFF_FFFF_FFFF)
    s = 1.0 / math.sqrt(r)
    bf = lambda t: t.to(torch.bfloat16).double()
    a_re = bf(torch.randn(G, dR // 2, rR // 2, generator=g) * s)
    a_im = bf(torch.randn(G, dR // 2, rR // 2, generator=g) * s)
    DN = bf(torch.randn(G, d - dR, r - rR, generator=g) * s)
    D = torch.zeros(G, r, d, dtype=torch.float64)
    for j in range(dR // 2):
        for i in range(rR // 2):
            if j * rR != i * dR:
                continue
            a, b = a_re[:, j, i], a_im[:, j, i]
            # key rows (2j, 2j+1) x latent columns (2i, 2i+1) = [[a, -b], [b, a]],
            # stored transposed: D[latent][key]
            D[:, 2 * i, 2 * j], D[:, 2 * i + 1, 2 * j] = a, -b
            D[:, 2 * i, 2 * j + 1], D[:, 2 * i + 1, 2 * j + 1] = b, a
    D[:, rR:, dR:] = DN.transpose(1, 2)
    return {"a_re": a_re, "a_im": a_im, "DN": DN, "D": D.float().contiguous()}


def make_workload(w: Workload | str, seed: int = 0, device="cpu") -> dict:
    """All inputs of one workload as a dict of tensors on `device` (see module doc)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    out = {"spec": w}
    lat, lat_scale, heavy = make_latent(w.B, w.L, w.r, w.lat_dtype, seed, device)
    out["latent"], out["lat_scale"], out["heavy"] = lat, lat_scale, heavy

    gd = _gen(seed, _S_D, device)
    D = torch.randn(w.G, w.r, w.d, generator=gd, device=device) / math.sqrt(w.r)
    out["D"] = _store(D, w.q_dtype)[0]

    gq = _gen(seed, _S_Q, device)
    q_own = torch.randn(w.B, w.T, w.G, w.H, w.d, generator=gq, device=device) / math.sqrt(w.d)
    if w.mix_shared > 0:
        gs = _gen(seed, _S_QSHARED, device)
        q_sh = torch.randn(w.B, w.T, 1, w.H, w.d, generator=gs, device=device) / math.sqrt(w.d)
        q = w.mix_shared * q_sh + (1.0 - w.mix_shared) * q_own
    else:
        q = q_own
    out["q"] = _store(q, w.q_dtype)[0]

    gw = _gen(seed, _S_W, device)
    out["w"] = torch.rand(w.B, w.T, w.G, w.H, generator=gw, device=device).contiguous()

    if w.pos0 >= 0:
        out["q_pos"] = torch.arange(w.pos0, w.pos0 + w.T, dtype=torch.int32, device=device)
    else:
        out["q_pos"] = None

    if w.native:
        cf = _dequant(lat, lat_scale, w.lat_dtype)                     # [B][L][r]
        Df = out["D"].float()                                          # [G][r][d]
        keys, kscale = [], []
        for l in range(w.G):
            kl = torch.matmul(cf, Df[l])                               # [B][L][d] = c^T D_l
            codes, s = quantize_rows_fp8(kl)
            keys.append(codes)
            kscale.append(s)
            del kl
        out["keys"] = torch.stack(keys).contiguous()                   # [G][B][L][d]
        out["key_scale"] = torch.stack(kscale).contiguous()            # [G][B][L]
    return out
