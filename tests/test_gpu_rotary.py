"""GPU parity of the latent path under rotary-constrained decoders (summary
page, Methodology, eqs. (1)-(4) and (6)-(8)).

Tokens are appended to the shared latent cache with the rotary encoding of
their position (li_append_latent, eqs. (1)-(2)); decoders whose RoPE block
commutes with the rotation (eq. (4): complex numbers per rotary frequency)
are absorbed into the queries (li_absorb_queries, eq. (6)); the whole cache
is scanned (li_score_group, eq. (8)) and each layer takes its top-k.  The
oracle scores the same tokens the way a native indexer would: per-layer keys
[R_t D^R z^R ; D^N z^N] decoded first and rotated after, scored with the raw
queries.  Eqs. (4) and (7) make the two equal; nothing on the GPU side sees
the per-layer keys."""
import numpy as np
import pytest
import torch

import li_inputs
from parity import RTOL, assert_scores_close, assert_topk_row

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
B, DM, R, RR, D_KEY, DR, G, L = 2, 512, 192, 64, 128, 64, 4, 131072


def _positions(n, seed):
    """Distinct cache positions per sequence: the ends of the cache, a tile
    boundary and seeded random ones."""
    g = torch.Generator().manual_seed(seed)
    fixed = [0, 1, 2, 127, 128, 129, L - 2, L - 1]
    out = []
    for _ in range(B):
        rest = torch.randperm(L - 3, generator=g)[: 4 * n] + 3
        pos = fixed + [int(p) for p in rest.tolist() if int(p) not in fixed][: n - len(fixed)]
        out.append(pos)
    return np.array(out, dtype=np.int32)                       # [B][n]


@pytest.mark.parametrize("x_dt,lat_dt,abs_dt,H", [("f32", "f32", "f32", 8), ("bf16", "bf16", "bf16", 64),
                                                  ("bf16", "fp8", "fp8", 64)])
def test_append_absorb_scan_with_rotary_decoders(li, orc, x_dt, lat_dt, abs_dt, H):
    """fp32 runs on the CUDA-core scorer (G * H * r <= 8192, so 8 heads); bf16
    and fp8 on the tensor cores with the workloads' 64 heads."""
    n = 600
    pos = _positions(n, seed=61)
    x, P = li_inputs.make_append_inputs(n * B, DM, R, x_dt, seed=62)       # token (j, b) = row j * B + b
    dec = li_inputs.make_rotary_decoders(G, R, RR, D_KEY, DR, seed=63)
    qw = li_inputs.make_workload(li_inputs.spec("tiny_f32", B=B, G=G, H=H, d=D_KEY, r=R, L=8,
                                                q_dtype=x_dt, lat_dtype="f32"), seed=64)
    q, w = qw["q"], qw["w"]
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}
    Dst = dec["D"].to(tdt[x_dt])

    # ---- GPU: append every token at its position, absorb, scan, top-k
    lat = torch.zeros(B, L, R, dtype=tdt[lat_dt], device=DEV)
    sc = torch.zeros(B, L, dtype=torch.float32, device=DEV) if lat_dt == "fp8" else None
    xg, Pg = x.to(DEV), P.to(DEV)
    # one 16-byte aligned position row per append call
    pos_g = torch.zeros(n, 4, dtype=torch.int32)
    pos_g[:, :B] = torch.from_numpy(pos.T.copy())
    pos_g = pos_g.to(DEV)
    for j in range(n):
        li.append_latent(xg[j * B:(j + 1) * B], Pg, pos_g[j, :B], RR, lat, sc)
    q_abs, q_scale = li.absorb_queries(q.to(DEV), Dst.to(DEV), abs_dt)
    scores = li.score_group(lat, sc, q_abs, q_scale, w.to(DEV))
    k = 64
    idx = li.topk(scores, k)
    assert li.device_status() == 0
    g_scores = scores.cpu().numpy()[:, 0]                      # [B][G][L]

    # ---- oracle: per-layer keys decoded then rotated (the native form)
    DRs = np.stack([orc.rotary_decoder(dec["a_re"][l], dec["a_im"][l], DR, RR) for l in range(G)])
    keys = orc.rope_keys(x, P, RR, DRs, dec["DN"], pos.T.reshape(-1))      # [G][n*B][d]
    keys = keys.reshape(G, n, B, D_KEY)
    q64 = orc.decode_rows(q)                                   # exact values of the stored queries
    o = np.zeros((B, G, n))
    for b in range(B):
        for l in range(G):
            o[b, l] = orc.native_score(keys[l, :, b][None], None, q64[b, 0, l][None], w[b, 0, l][None])[0]

    rtol = RTOL[abs_dt]
    for b in range(B):
        assert_scores_close(g_scores[b][:, pos[b]], o[b], rtol, f"{lat_dt} rotary scores, sequence {b}")
        rest = np.ones(L, dtype=bool)
        rest[pos[b]] = False
        assert (g_scores[b][:, rest] == 0).all(), "rows never appended must score 0"
        for l in range(G):
            full = np.zeros(L)
            full[pos[b]] = o[b, l]
            assert_topk_row(idx[b, 0, l].cpu().numpy(), full, k, L, rtol, f"{lat_dt} rotary top-k")
