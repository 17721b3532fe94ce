"""GPU parity of the latent-cache append (eqs. 1-2 of the summary page)
against the fp64 oracle: projection, rotary encoding of the RoPE branch,
storage (fp32 / bf16 / fp8 with the row scale) at the token's position."""
import numpy as np
import pytest
import torch

import li_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(li, orc, B, dm, r, rR, L, pos, x_dtype, lat_dtype, seed):
    x, P = li_inputs.make_append_inputs(B, dm, r, x_dtype, seed=seed)
    pos_t = torch.tensor(pos, dtype=torch.int32)
    esz = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[lat_dtype]
    lat = torch.full((B, L, r), 0x5A if lat_dtype == "fp8" else 7, dtype=esz, device=DEV)
    sc = torch.full((B, L), -1.0, dtype=torch.float32, device=DEV) if lat_dtype == "fp8" else None
    st = li.li_append_latent(x.to(DEV), P.to(DEV), pos_t.to(DEV), rR, lat, sc)
    assert st == 0
    status = li.li_device_status()
    o = orc.append_latent(x, P, rR, pos_t)
    return lat, sc, o, status


def _check_row(lat_dtype, row, scale, o):
    amax = np.abs(o).max()
    if lat_dtype == "f32":
        g = row.double().numpy()
        assert (np.abs(g - o) <= 1e-5 * np.abs(o) + 2e-6 * amax).all()
    elif lat_dtype == "bf16":
        g = row.float().double().numpy()
        assert (np.abs(g - o) <= 2.0 ** -8 * np.abs(o) + 2e-6 * amax).all()
    else:
        np.testing.assert_allclose(scale, amax / 448.0, rtol=1e-5)
        g = row.view(torch.float8_e4m3fn).double().numpy() * scale
        # one E4M3 rounding (a code step either side where fp32 and fp64 straddle a
        # rounding boundary), the subnormal step of the scale, fp32 accumulation
        tol = 2.0 ** -3 * np.abs(o) + scale * 2.0 ** -9 + 2e-6 * amax
        assert (np.abs(g - o) <= tol).all()


@pytest.mark.parametrize("lat_dtype", ["f32", "bf16", "fp8"])
def test_append_matches_oracle(li, orc, lat_dtype):
    B, dm, r, rR, L = 5, 1024, 192, 64, 2048
    pos = [0, 1, 777, 2046, 2047]
    lat, sc, o, status = _run(li, orc, B, dm, r, rR, L, pos, "bf16", lat_dtype, seed=41)
    assert status == 0
    for b in range(B):
        _check_row(lat_dtype, lat[b, pos[b]].cpu(), None if sc is None else float(sc[b, pos[b]]), o[b])
    # nothing else of the cache was written
    mask = torch.ones(B, L, dtype=torch.bool)
    mask[torch.arange(B), torch.tensor(pos)] = False
    fill = 0x5A if lat_dtype == "fp8" else 7
    assert (lat.cpu()[mask] == torch.tensor(fill, dtype=lat.dtype)).all()
    if sc is not None:
        assert (sc.cpu()[mask] == -1.0).all()


@pytest.mark.parametrize("r,rR", [(32, 0), (100, 32), (256, 128), (40, 40)])
def test_append_shapes_and_scalar_path(li, orc, r, rR):
    """Odd dm (scalar loads), fp32 inputs, r not a multiple of 32, all-RoPE and all-NoPE."""
    B, dm, L = 3, 1001, 64
    pos = [5, 63, 0]
    lat, sc, o, status = _run(li, orc, B, dm, r, rR, L, pos, "f32", "fp8", seed=r + rR)
    assert status == 0
    for b in range(B):
        _check_row("fp8", lat[b, pos[b]].cpu(), float(sc[b, pos[b]]), o[b])


def test_append_large_positions_rotate_accurately(li, orc):
    """Angles up to 1.3e5 rad: formed and reduced in double precision."""
    B, dm, r, rR, L = 4, 512, 192, 64, 131072
    pos = [131071, 100000, 65536, 12345]
    lat, sc, o, status = _run(li, orc, B, dm, r, rR, L, pos, "bf16", "f32", seed=43)
    assert status == 0
    for b in range(B):
        _check_row("f32", lat[b, pos[b]].cpu(), None, o[b])


def test_append_position_outside_cache_is_skipped_and_reported(li, orc):
    B, dm, r, rR, L = 3, 256, 64, 32, 16
    pos = [3, 16, -1]
    lat, sc, o, status = _run(li, orc, B, dm, r, rR, L, pos, "bf16", "fp8", seed=44)
    assert status == -7                                 # LI_ERR_DEVICE_BOUNDS
    _check_row("fp8", lat[0, 3].cpu(), float(sc[0, 3]), o[0])
    assert (lat[1:].cpu() == 0x5A).all() and (sc[1:].cpu() == -1.0).all()
    assert li.li_device_status() == 0


@pytest.mark.parametrize("B,lat_dtype", [(9, "fp8"), (32, "fp8"), (32, "bf16")])
def test_append_full_hidden_size(li, orc, B, lat_dtype):
    """The decode size (hidden 7168, r 192, RoPE 64): the hidden dimension is
    split over a 16-CTA cluster and summed across it; 9 tokens leave a ragged
    last group of the 4 tokens a cluster takes."""
    dm, r, rR, L = 7168, 192, 64, 4096
    pos = [(977 * b) % L for b in range(B)]
    lat, sc, o, status = _run(li, orc, B, dm, r, rR, L, pos, "bf16", lat_dtype, seed=45 + B)
    assert status == 0
    for b in range(B):
        _check_row(lat_dtype, lat[b, pos[b]].cpu(), None if sc is None else float(sc[b, pos[b]]), o[b])


def test_scan_right_after_append_sees_the_new_rows(li, orc):
    """A decode scan queued right after an append on the same stream, with no
    synchronisation between them, scores the appended rows: the scan issues
    its first cache-tile loads before waiting for the preceding kernel, and
    the append lets dependents start only after its stores.  4 sequences of
    4,096 tokens give every CTA a single tile, all loaded before the wait."""
    from parity import RTOL, assert_scores_close
    w = li_inputs.spec("fp8_32k_b32", B=4, L=4096, native=False)
    x = li_inputs.make_workload(w, seed=53)
    xa, P = li_inputs.make_append_inputs(w.B, 1024, w.r, "bf16", seed=54)
    pos = torch.tensor([4095, 0, 2000, 128], dtype=torch.int32)
    lat, lsc = x["latent"].to(DEV), x["lat_scale"].to(DEV)
    qa, qs = li.absorb_queries(x["q"].to(DEV), x["D"].to(DEV), "fp8")
    assert li.li_append_latent(xa.to(DEV), P.to(DEV), pos.to(DEV), 64, lat, lsc) == 0
    s = li.score_group(lat, lsc, qa, qs, x["w"].to(DEV))
    torch.cuda.synchronize()
    assert li.li_device_status() == 0
    lat_h, lsc_h = lat.cpu(), lsc.cpu()
    for b in range(w.B):                      # the rows did change
        assert not torch.equal(lat_h[b, pos[b]], x["latent"][b, pos[b]])
    o = orc.score(lat_h, lsc_h, orc.absorb(x["q"], x["D"]), x["w"])
    assert_scores_close(s.cpu().numpy(), o, RTOL["fp8"])
