"""GPU parity of each kernel against the CPU oracle on small seeded cases.

Every call goes through the C ABI (ctypes binding); inputs come from
li_inputs, expected values from the oracle only.  Sizes span several
128-token tiles plus a ragged tail and stay small enough for the oracle to
finish in seconds.
"""
import numpy as np
import pytest
import torch

import li_inputs
from parity import RTOL, assert_scores_close, assert_topk_row, exact_sets_equal, max_rel_err

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _dev(x):
    return None if x is None else x.to(DEV)


def _sync_ok(li):
    assert li.li_device_status() == 0


# ------------------------------------------------------------------ absorption

@pytest.mark.parametrize("abs_dtype", ["f32", "bf16", "fp8"])
@pytest.mark.parametrize("q_dtype", ["f32", "bf16"])
def test_absorb_matches_oracle(li, orc, q_dtype, abs_dtype):
    w = li_inputs.spec("dsa_bf16_8k", B=3, T=2, L=8, q_dtype=q_dtype, native=False)
    x = li_inputs.make_workload(w, seed=1)
    q_abs, scale = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), abs_dtype)
    _sync_ok(li)
    o = orc.absorb(x["q"], x["D"])                                     # fp64
    if abs_dtype == "fp8":
        g = orc.decode_rows(q_abs.cpu(), scale.cpu())
        amax = np.abs(o).max(axis=-1)
        np.testing.assert_allclose(scale.cpu().numpy(), amax / 448.0, rtol=1e-5)
        # one E4M3 rounding: |err| <= 2^-4 |o| (normal range) or half the
        # subnormal spacing (2^-10 of the scale * 448... = s * 2^-10), plus fp32 accumulation
        s = scale.cpu().numpy()[..., None]
        tol = 2.0 ** -4 * np.abs(o) + s * 2.0 ** -10 + 1e-5 * amax[..., None]
        assert (np.abs(g - o) <= tol).all()
    elif abs_dtype == "bf16":
        g = q_abs.float().cpu().double().numpy()
        assert (np.abs(g - o) <= 2.0 ** -8 * np.abs(o) + 1e-6 * np.abs(o).max()).all()
    else:
        g = q_abs.cpu().double().numpy()
        np.testing.assert_allclose(g, o, rtol=1e-5, atol=1e-6 * np.abs(o).max())


def test_absorb_identity_decoder_is_a_conversion(li):
    q = torch.randn(2, 1, 1, 64, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    q_abs, _ = li.absorb_queries(q.to(DEV), None, "bf16")
    assert torch.equal(q_abs.cpu(), q)
    q32, _ = li.absorb_queries(q.float().to(DEV), None, "f32")
    assert torch.equal(q32.cpu(), q.float())
    q8, s8 = li.absorb_queries(q.to(DEV), None, "fp8")
    ref_codes, ref_scale = li_inputs.quantize_rows_fp8(q.float())
    np.testing.assert_allclose(s8.cpu().numpy(), ref_scale.numpy(), rtol=1e-6)
    # same RNE rounding of the same quotient, up to a one-ulp difference in x/s
    d = (q8.cpu().view(torch.float8_e4m3fn).float() - ref_codes.view(torch.float8_e4m3fn).float()).abs()
    assert (d <= ref_codes.view(torch.float8_e4m3fn).float().abs() * 2.0 ** -3 + 1e-6).all()


# --------------------------------------------------------------------- scoring

def _score_case(li, orc, lat_dtype, B, T, G, H, r, L, seed=0, beta=False, q_pos=None):
    lat, lsc, _ = li_inputs.make_latent(B, L, r, lat_dtype, seed=seed)
    qa, qs = li_inputs.make_absorbed_queries(B, T, G, H, r, lat_dtype if lat_dtype != "f32" else "f32",
                                             seed=seed)
    w = torch.rand(B, T, G, H, generator=torch.Generator().manual_seed(seed + 7))
    bt = li_inputs.make_beta(B, T, G, H, seed=seed) if beta else None
    g = li.score_group(_dev(lat), _dev(lsc), _dev(qa), _dev(qs), _dev(w), beta=_dev(bt),
                       q_pos=_dev(q_pos))
    _sync_ok(li)
    o = orc.score(lat, lsc, orc.decode_rows(qa, qs), w, beta=bt, q_pos=q_pos)
    return g.cpu().double().numpy(), o


@pytest.mark.parametrize("L", [1, 127, 128, 129, 1000])
def test_score_f32_simt(li, orc, L):
    g, o = _score_case(li, orc, "f32", B=2, T=1, G=4, H=8, r=32, L=L)
    assert_scores_close(g, o, RTOL["f32"])


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
@pytest.mark.parametrize("L", [1, 127, 128, 129, 1000, 3000])
def test_score_tensor_core(li, orc, dt, L):
    g, o = _score_case(li, orc, dt, B=2, T=1, G=4, H=64, r=192, L=L, seed=L)
    assert_scores_close(g, o, RTOL[dt])
    # both sides consume identical operands: only fp32 accumulation order differs
    assert max_rel_err(g, o) < 1e-4


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
@pytest.mark.parametrize("G,H,r", [(1, 64, 192), (3, 64, 128), (2, 128, 64), (4, 32, 256), (8, 16, 64),
                                   (8, 64, 192), (5, 64, 128), (3, 128, 64)])
def test_score_tensor_core_shapes(li, orc, dt, G, H, r):
    g, o = _score_case(li, orc, dt, B=3, T=1, G=G, H=H, r=r, L=777, seed=G * 100 + H)
    assert_scores_close(g, o, RTOL[dt])
    assert max_rel_err(g, o) < 1e-4


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_score_with_beta(li, orc, dt):
    g, o = _score_case(li, orc, dt, B=2, T=1, G=4, H=64, r=192, L=600, seed=5, beta=True)
    assert_scores_close(g, o, RTOL[dt])
    assert max_rel_err(g, o) < 1e-4


def test_score_f32_with_beta(li, orc):
    g, o = _score_case(li, orc, "f32", B=2, T=1, G=4, H=8, r=32, L=300, seed=6, beta=True)
    assert_scores_close(g, o, RTOL["f32"])


@pytest.mark.parametrize("dt", ["bf16", "fp8", "f32"])
def test_score_causal_prefill(li, orc, dt):
    """Query t sees s <= q_pos[t]; entries past the limit are left untouched."""
    B, T, L = 2, 5, 700
    G, H, r = (4, 64, 192) if dt != "f32" else (4, 8, 32)
    q_pos = torch.tensor([0, 127, 128, 400, 699], dtype=torch.int32)
    lat, lsc, _ = li_inputs.make_latent(B, L, r, dt, seed=9)
    qa, qs = li_inputs.make_absorbed_queries(B, T, G, H, r, dt, seed=9)
    w = torch.rand(B, T, G, H, generator=torch.Generator().manual_seed(2))
    out = torch.full((B, T, G, L), float("nan"), device=DEV)
    li.score_group(_dev(lat), _dev(lsc), _dev(qa), _dev(qs), _dev(w), q_pos=_dev(q_pos), out=out)
    _sync_ok(li)
    o = orc.score(lat, lsc, orc.decode_rows(qa, qs), w, q_pos=q_pos)
    g = out.cpu().double().numpy()
    for t, p in enumerate(q_pos.tolist()):
        assert_scores_close(g[:, t, :, :p + 1], o[:, t, :, :p + 1], RTOL[dt], f"query {t}")
        assert np.isnan(g[:, t, :, p + 1:]).all(), "wrote past the causal limit"


def test_score_mixed_dtypes_fall_back_to_cuda_cores(li, orc):
    """bf16 latent with fp8 absorbed queries (no tensor-core form) still scores exactly."""
    B, L, G, H, r = 1, 300, 2, 16, 64
    lat, _, _ = li_inputs.make_latent(B, L, r, "bf16", seed=4)
    qa, qs = li_inputs.make_absorbed_queries(B, 1, G, H, r, "fp8", seed=4)
    w = torch.rand(B, 1, G, H, generator=torch.Generator().manual_seed(4))
    g = li.score_group(_dev(lat), None, _dev(qa), _dev(qs), _dev(w)).cpu().double().numpy()
    o = orc.score(lat, None, orc.decode_rows(qa, qs), w)
    assert_scores_close(g, o, 1e-5)


# ---------------------------------------------------------------------- top-k

def _topk_gpu(li, s, k, valid_len=None):
    idx, vals = li.topk(s.to(DEV), k, valid_len=_dev(valid_len), with_vals=True)
    _sync_ok(li)
    return idx.cpu().numpy(), vals.cpu().numpy()


@pytest.mark.parametrize("L,k", [(1, 1), (5, 3), (100, 100), (100, 250), (4096, 256),
                                 (8192, 2048), (32768, 2048), (131072, 8192)])
def test_topk_bit_exact_random(li, orc, L, k):
    s = torch.randn(3, L, generator=torch.Generator().manual_seed(L + k)) * 5 + 10
    gi, gv = _topk_gpu(li, s, k)
    oi, ov = orc.topk(s.double().numpy(), k)
    exact_sets_equal(gi, oi)
    n = min(k, L)
    np.testing.assert_array_equal(np.sort(gv[:, :n], axis=1), np.sort(ov[:, :n].astype(np.float32), axis=1))


def test_topk_ties_take_lowest_positions(li, orc):
    g = torch.Generator().manual_seed(11)
    s = torch.randint(-3, 4, (8, 5000), generator=g).float()          # massive ties
    s[1] = 2.0                                                        # all equal
    s[2, ::7] = -0.0
    for k in (1, 17, 1024, 4999):
        gi, _ = _topk_gpu(li, s, k)
        oi, _ = orc.topk(s.double().numpy(), k)
        exact_sets_equal(gi, oi)


def test_topk_short_threshold_list_with_ties(li, orc):
    """Decode-length rows whose threshold bin holds a short candidate list with
    exact ties at the k-th score: the list is ranked by counting, ties by position."""
    g = torch.Generator().manual_seed(21)
    s = torch.randn(6, 32768, generator=g) * 5 + 10
    for r in range(6):
        v = s[r].sort(descending=True).values[2047 - 3 * r]
        pos = torch.randperm(32768, generator=g)[:2 + 7 * r]
        s[r, pos] = v
    s[5, 100:140] = s[5].max()                       # ties among the sure keys too
    for k in (1, 2000, 2048, 2100):
        gi, gv = _topk_gpu(li, s, k)
        oi, ov = orc.topk(s.double().numpy(), k)
        exact_sets_equal(gi, oi)
        np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_two_pass_equals_one_pass(li, orc):
    """Rows longer than 32,768 with a workspace take the two-pass path (segment
    top-k, then top-k of the candidates): same sets and values as one pass and
    as the oracle, including ties that straddle segments."""
    g = torch.Generator().manual_seed(22)
    s = torch.randn(5, 131072, generator=g) * 4 + 10
    s[1] = torch.randint(0, 9, (131072,), generator=g).float()     # ties across segments
    s[2, 40000:100000] = s[2].max() + 1.0                           # one value over two segments
    s[3, ::3] = float("-inf")
    sd = s.to(DEV)
    for k in (1, 100, 2048, 8192):
        n = li.li_topk_workspace_size(5, 131072, k)
        assert n > 0
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        i1 = torch.empty(5, k, dtype=torch.int32, device=DEV)
        v1 = torch.empty(5, k, dtype=torch.float32, device=DEV)
        i2 = torch.empty_like(i1)
        v2 = torch.empty_like(v1)
        assert li.li_topk(sd, k, i1, v1, ws=ws) == 0
        assert li.li_topk(sd, k, i2, v2) == 0
        _sync_ok(li)
        oi, ov = orc.topk(s.double().numpy(), k)
        exact_sets_equal(i1.cpu().numpy(), oi)
        exact_sets_equal(i2.cpu().numpy(), oi)
        np.testing.assert_array_equal(np.sort(v1.cpu().numpy(), axis=1), np.sort(v2.cpu().numpy(), axis=1))


@pytest.mark.parametrize("L", [8193, 16384, 20000, 24577, 32768])
def test_topk_rows_8k_to_32k_ragged_ties_and_valid_lengths(li, orc, L):
    """Rows of 8K-32K scores: lengths off the 8K multiples, valid lengths
    around 8K borders, and ties at the threshold across those borders (taken
    by lowest position) are all bit-exact."""
    g = torch.Generator().manual_seed(L)
    s = torch.randn(8, L, generator=g) * 3 + 5
    s[1] = torch.randint(0, 3, (L,), generator=g).float()               # heavy ties everywhere
    s[2] = 7.0                                                          # one value
    s[3, 8000:8400] = 50.0                                              # ties across the rank-0/1 border
    s[4, ::2] = -0.0
    s[5] = torch.rand(L, generator=g) * 1e-3 + 1.0                      # one narrow binade
    vl = torch.tensor([L, L, 5000, 8192, 8191, L - 1, 3, 0], dtype=torch.int32)
    for k in (1, 100, 2048, 8200):
        for v in (None, vl):
            gi, gv = _topk_gpu(li, s, k, v)
            oi, ov = orc.topk(s.double().numpy(), k, valid_len=None if v is None else v.numpy())
            exact_sets_equal(gi, oi)
            np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_long_rows_with_valid_lengths_and_workspace(li, orc):
    """Causal rows (a valid prefix per row) longer than 32,768 with a
    workspace given: lengths at and around 32K segment borders, empty and
    one-element prefixes, and ties across segment borders."""
    g = torch.Generator().manual_seed(23)
    L = 131072
    s = torch.randn(8, L, generator=g) * 4 + 10
    s[2] = torch.randint(0, 6, (L,), generator=g).float()
    s[5, 30000:70000] = 99.0
    vl = torch.tensor([L, 0, 1, 100, 32768, 32769, 70000, L - 1], dtype=torch.int32)
    sd, vd = s.to(DEV), vl.to(DEV)
    for k in (1, 2048, 8192):
        ws = torch.empty(li.li_topk_workspace_size(8, L, k), dtype=torch.uint8, device=DEV)
        i1 = torch.empty(8, k, dtype=torch.int32, device=DEV)
        v1 = torch.empty(8, k, dtype=torch.float32, device=DEV)
        assert li.li_topk(sd, k, i1, v1, vd, ws) == 0
        _sync_ok(li)
        oi, ov = orc.topk(s.double().numpy(), k, valid_len=vl.numpy())
        gi, gv = i1.cpu().numpy(), v1.cpu().numpy()
        exact_sets_equal(gi, oi)
        np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_threshold_bin_overflows_shared_memory(li, orc):
    """Scores sharing their top 12 key bits (one exponent, same 3 mantissa bits) force the
    re-read path; a narrower cluster forces the second-digit re-read too."""
    g = torch.Generator().manual_seed(12)
    wide = 1.0 + torch.rand(2, 100000, generator=g) * 0.12
    narrow = 1.0 + torch.rand(2, 100000, generator=g) * 1e-4
    for s in (wide, narrow):
        for k in (10, 5000, 60000):
            gi, _ = _topk_gpu(li, s, k)
            oi, _ = orc.topk(s.double().numpy(), k)
            exact_sets_equal(gi, oi)


def test_topk_valid_len_and_padding(li, orc):
    s = torch.randn(6, 3000, generator=torch.Generator().manual_seed(13))
    vl = torch.tensor([0, 1, 100, 2999, 3000, 5000], dtype=torch.int32)
    gi, gv = _topk_gpu(li, s, 200, vl)
    oi, _ = orc.topk(s.double().numpy(), 200, valid_len=vl.numpy())
    exact_sets_equal(gi, oi)
    assert (gi[0] == -1).all() and np.isneginf(gv[0]).all()
    assert gi[1, 0] == 0 and (gi[1, 1:] == -1).all()


def test_topk_negative_and_infinite_scores(li, orc):
    s = torch.randn(4, 2000, generator=torch.Generator().manual_seed(14)) - 50
    s[0, :1500] = float("-inf")
    s[1, 100] = float("inf")
    gi, _ = _topk_gpu(li, s, 700)
    oi, _ = orc.topk(s.double().numpy(), 700)
    exact_sets_equal(gi, oi)


# ---------------------------------------------------------------- pipelines

@pytest.mark.parametrize("name", ["tiny_f32", "dsa_bf16_8k"])
def test_pipeline_full_workload(li, orc, name):
    """absorb -> score -> top-k on the GPU vs the oracle's fp64 absorb -> score -> TopK."""
    x = li_inputs.make_workload(name, seed=0)
    w = x["spec"]
    absd = {"f32": "f32", "bf16": "bf16", "fp8": "fp8"}[w.lat_dtype]
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), absd)
    s = li.score_group(_dev(x["latent"]), _dev(x["lat_scale"]), qa, qs, _dev(x["w"]))
    idx = li.topk(s, w.k)
    _sync_ok(li)
    o = orc.score(x["latent"], x["lat_scale"], orc.absorb(x["q"], x["D"]), x["w"])
    rt = RTOL[w.lat_dtype]
    assert_scores_close(s.cpu().numpy(), o, rt)
    gi = idx.cpu().numpy()
    for b in range(w.B):
        for l in range(w.G):
            assert_topk_row(gi[b, 0, l], o[b, 0, l], w.k, w.L, rt, f"b{b} l{l}")


def test_pipeline_fp8_reduced_batch(li, orc):
    w = li_inputs.spec("fp8_32k_b32", B=3, L=5000, native=False)
    x = li_inputs.make_workload(w, seed=2)
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), "fp8")
    s = li.score_group(_dev(x["latent"]), _dev(x["lat_scale"]), qa, qs, _dev(x["w"]))
    idx = li.topk(s, w.k)
    _sync_ok(li)
    o = orc.score(x["latent"], x["lat_scale"], orc.absorb(x["q"], x["D"]), x["w"])
    assert_scores_close(s.cpu().numpy(), o, RTOL["fp8"])
    gi = idx.cpu().numpy()
    for b in range(w.B):
        for l in range(w.G):
            assert_topk_row(gi[b, 0, l], o[b, 0, l], w.k, w.L, RTOL["fp8"], f"b{b} l{l}")


# ------------------------------------------------------------------- native

def test_native_scan_matches_oracle(li, orc):
    x = li_inputs.make_workload(li_inputs.spec("dsa_bf16_8k", B=2, L=3000), seed=3)
    w = x["spec"]
    for l in range(w.G):
        q8, s8 = li.absorb_queries(_dev(x["q"][:, :, l:l + 1]), None, "fp8")
        g = li.native_score(_dev(x["keys"][l]), _dev(x["key_scale"][l]), q8.view(w.B, w.H, w.d),
                            s8.view(w.B, w.H), _dev(x["w"][:, 0, l]))
        _sync_ok(li)
        o = orc.native_score(x["keys"][l], x["key_scale"][l], orc.decode_rows(x["q"][:, 0, l]),
                             x["w"][:, 0, l])
        assert_scores_close(g.cpu().numpy(), o, RTOL["fp8"])


# ----------------------------------------------------------------------- HS

def _hs_check(li, orc, x, m, k, dt):
    w = x["spec"]
    absd = "fp8" if dt == "fp8" else "bf16"
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), absd)
    cand, idx = li.hs_select(_dev(x["latent"]), _dev(x["lat_scale"]), qa, qs, _dev(x["w"]), m, k)
    _sync_ok(li)
    o = orc.score(x["latent"], x["lat_scale"], orc.absorb(x["q"], x["D"]), x["w"])[:, 0]  # [B][G][L]
    c = cand.cpu().numpy()
    gi = idx.cpu().numpy()
    rt = RTOL[dt]
    nc = min(m, w.L)
    for b in range(w.B):
        assert_topk_row(c[b], o[b, 0], m, w.L, rt, f"cand b{b}")
        C = set(c[b, :nc].tolist())
        for l in range(w.G):
            assert_topk_row(gi[b, l], o[b, l], k, w.L if l == 0 else w.L, rt, f"b{b} l{l}",
                            allowed=C)
    return c, gi, o


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_hs_matches_oracle(li, orc, dt):
    w = li_inputs.spec("fp8_128k_hs", B=2, L=3000, m=512, k=128, lat_dtype=dt)
    x = li_inputs.make_workload(w, seed=4)
    _hs_check(li, orc, x, 512, 128, dt)


def test_hs_profiled_equals_hs_and_times_its_stages(li, orc):
    """li_hs_select_profiled does the same work as li_hs_select (identical
    candidates and selections, both checked against the oracle) and records
    its five events in stream order."""
    w = li_inputs.spec("fp8_128k_hs", B=2, L=40000, m=1024, k=256)
    x = li_inputs.make_workload(w, seed=13)
    c, gi, _ = _hs_check(li, orc, x, 1024, 256, "fp8")
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), "fp8")
    cand = torch.empty(2, 1024, dtype=torch.int32, device=DEV)
    idx = torch.empty(2, 4, 256, dtype=torch.int32, device=DEV)
    ws = torch.empty(li.li_hs_workspace_size(2, 4, 40000, 1024, 256), dtype=torch.uint8, device=DEV)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    assert li.li_hs_select_profiled(_dev(x["latent"]), _dev(x["lat_scale"]), qa, qs, _dev(x["w"]),
                                    1024, 256, cand, idx, ws, ev) == 0
    _sync_ok(li)
    np.testing.assert_array_equal(np.sort(cand.cpu().numpy(), axis=-1), np.sort(c, axis=-1))
    np.testing.assert_array_equal(np.sort(idx.cpu().numpy(), axis=-1), np.sort(gi, axis=-1))
    stages = [ev[i].elapsed_time(ev[i + 1]) for i in range(4)]
    assert all(t >= 0 for t in stages) and sum(stages) > 0


def test_hs_eight_layer_group(li, orc):
    """G = 8 at H = 64: the group scan and the followers' rescoring exceed one
    tensor-core tile (256 columns) and run in chunks of four layers."""
    w = li_inputs.spec("fp8_128k_hs", B=2, L=2500, G=8, m=512, k=128)
    x = li_inputs.make_workload(w, seed=12)
    _hs_check(li, orc, x, 512, 128, "fp8")
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), "fp8")
    s = li.score_group(_dev(x["latent"]), _dev(x["lat_scale"]), qa, qs, _dev(x["w"]))
    _sync_ok(li)
    o = orc.score(x["latent"], x["lat_scale"], orc.absorb(x["q"], x["D"]), x["w"])
    assert_scores_close(s.cpu().numpy(), o, RTOL["fp8"])


def test_hs_budget_at_least_context_is_full_latentindex(li, orc):
    w = li_inputs.spec("fp8_128k_hs", B=2, L=900, m=1024, k=100)
    x = li_inputs.make_workload(w, seed=5)
    c, gi, o = _hs_check(li, orc, x, 1024, 100, "fp8")
    assert (c[:, 900:] == -1).all()
    for b in range(2):
        assert sorted(c[b, :900].tolist()) == list(range(900))
        for l in range(w.G):
            assert_topk_row(gi[b, l], o[b, l], 100, 900, RTOL["fp8"], f"full b{b} l{l}")


def test_hs_budget_equal_k_gives_candidates(li, orc):
    w = li_inputs.spec("fp8_128k_hs", B=2, L=2000, m=256, k=256)
    x = li_inputs.make_workload(w, seed=6)
    c, gi, _ = _hs_check(li, orc, x, 256, 256, "fp8")
    for b in range(2):
        for l in range(w.G):
            assert set(gi[b, l].tolist()) == set(c[b].tolist())


def _hs_exact_vs_scan(li, orc, lat, sc, x, m, k):
    """HS against the oracle's selection on the scan's own fp32 scores (the HS
    kernels score with the same arithmetic), so tied scores are exactly tied."""
    w = x["spec"]
    qa, qs = li.absorb_queries(_dev(x["q"]), _dev(x["D"]), "fp8")
    s = li.score_group(_dev(lat), _dev(sc), qa, qs, _dev(x["w"]))
    cand, idx = li.hs_select(_dev(lat), _dev(sc), qa, qs, _dev(x["w"]), m, k)
    _sync_ok(li)
    oc, oi = orc.hs(s[:, 0].cpu().double().numpy(), m, k)
    exact_sets_equal(cand.cpu().numpy(), oc)
    exact_sets_equal(idx.cpu().numpy(), oi)


def test_hs_ties_taken_by_lowest_token_position(li, orc):
    """Every latent row appears twice, so every score is tied with another
    token's: anchor candidates and follower selections must take the lower
    token positions (the candidate list's own order is arbitrary)."""
    w = li_inputs.spec("fp8_128k_hs", B=2, L=4000, m=600, k=150)
    x = li_inputs.make_workload(w, seed=8)
    lat, sc = x["latent"].clone(), x["lat_scale"].clone()
    lat[:, 2000:] = lat[:, :2000]
    sc[:, 2000:] = sc[:, :2000]
    _hs_exact_vs_scan(li, orc, lat, sc, x, 600, 150)


def test_hs_many_ties_at_the_follower_threshold(li, orc):
    """Zero latent rows score exactly 0 in every layer: with k above the number
    of positive scores, thousands of candidates tie at the threshold and the
    lowest token positions among them are taken."""
    w = li_inputs.spec("fp8_128k_hs", B=1, L=12000, m=8192, k=5000)
    x = li_inputs.make_workload(w, seed=9)
    lat, sc = x["latent"].clone(), x["lat_scale"].clone()
    lat[:, 3000:] = 0
    _hs_exact_vs_scan(li, orc, lat, sc, x, 8192, 5000)


def test_hs_long_anchor_row_two_pass_with_ties(li, orc):
    """An anchor row longer than 32,768 takes its top-m in two passes from the
    HS workspace; duplicated latent rows make ties straddle the segments."""
    w = li_inputs.spec("fp8_128k_hs", B=1, L=40000, m=8192, k=2048)
    x = li_inputs.make_workload(w, seed=10)
    lat, sc = x["latent"].clone(), x["lat_scale"].clone()
    lat[:, 20000:] = lat[:, :20000]
    sc[:, 20000:] = sc[:, :20000]
    _hs_exact_vs_scan(li, orc, lat, sc, x, 8192, 2048)


@pytest.mark.parametrize("d,r", [(40, 64), (36, 100), (128, 256)])
def test_absorb_odd_widths(li, orc, d, r):
    """Key widths that are not multiples of the 32-wide staging chunk (d = 40) or
    of the 16-byte load (d = 36), and output widths that are not multiples of 4."""
    g = torch.Generator().manual_seed(d + r)
    q = torch.randn(2, 3, 2, 16, d, generator=g).to(torch.bfloat16)
    D = (torch.randn(2, r, d, generator=g) / r ** 0.5).to(torch.bfloat16)
    o = orc.absorb(q, D)
    for abs_dtype in ("f32", "bf16", "fp8"):
        q_abs, scale = li.absorb_queries(q.to(DEV), D.to(DEV), abs_dtype)
        _sync_ok(li)
        if abs_dtype == "fp8":
            gv = orc.decode_rows(q_abs.cpu(), scale.cpu())
            s = scale.cpu().numpy()[..., None]
            tol = 2.0 ** -4 * np.abs(o) + s * 2.0 ** -10 + 1e-5 * np.abs(o).max()
        elif abs_dtype == "bf16":
            gv = q_abs.float().cpu().double().numpy()
            tol = 2.0 ** -8 * np.abs(o) + 1e-6 * np.abs(o).max()
        else:
            gv = q_abs.cpu().double().numpy()
            tol = 1e-5 * np.abs(o) + 1e-6 * np.abs(o).max()
        assert (np.abs(gv - o) <= tol).all(), abs_dtype


def test_topk_long_rows_with_heavy_ties(li, orc):
    """Long rows of a few distinct values: the sampled thresholds see thousands of
    ties, so the shared-memory tie ranking and the in-order tie pass both run."""
    g = torch.Generator().manual_seed(15)
    s = torch.randint(0, 7, (4, 50000), generator=g).float()
    s[3] = torch.where(torch.rand(50000, generator=g) < 0.01, 9.0, 1.0)   # 1% on top, rest tied
    for k in (1, 300, 2048, 7000, 12000):
        gi, _ = _topk_gpu(li, s, k)
        oi, _ = orc.topk(s.double().numpy(), k)
        exact_sets_equal(gi, oi)


def test_topk_many_long_rows_valid_len(li, orc):
    """Prefill-shaped rows: long, with per-row valid lengths around the causal limit."""
    g = torch.Generator().manual_seed(16)
    rows, L = 24, 131072
    s = torch.randn(rows, L, generator=g) * 3 + 20
    vl = torch.randint(L - 5000, L + 1, (rows,), generator=g, dtype=torch.int32)
    vl[0] = 8191
    vl[1] = 8192
    gi, _ = _topk_gpu(li, s, 2048, vl)
    oi, _ = orc.topk(s.double().numpy(), 2048, valid_len=vl.numpy())
    exact_sets_equal(gi, oi)


def test_topk_prefill_rows_two_ctas_per_sm(li, orc):
    """Causal prefill rows (128K, valid lengths near the causal limit) in a
    number that puts two 512-thread CTAs on each SM: eight 16K passes per
    row, a ragged last pass, one row of ties across the threshold."""
    g = torch.Generator().manual_seed(33)
    rows, L = 320, 131072
    s = torch.randn(rows, L, generator=g) * 3 + 20
    s[7] = torch.randint(0, 5, (L,), generator=g).float()
    vl = torch.randint(L - 5000, L + 1, (rows,), generator=g, dtype=torch.int32)
    vl[0] = L
    vl[1] = 16385
    gi, gv = _topk_gpu(li, s, 2048, vl)
    oi, ov = orc.topk(s.double().numpy(), 2048, valid_len=vl.numpy())
    exact_sets_equal(gi, oi)
    np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_unaligned_rows(li, orc):
    """Row starts that are not 16-byte aligned take the scalar load paths."""
    g = torch.Generator().manual_seed(17)
    base = torch.randn(5 * 30001 + 16, generator=g).to(DEV)
    s = base[4:4 + 5 * 30001].view(5, 30001)     # 16-byte aligned start, odd row length
    idx = torch.empty(5, 1000, dtype=torch.int32, device=DEV)
    st = li.li_topk(s, 1000, idx)
    assert st == 0 and li.li_device_status() == 0
    oi, _ = orc.topk(s.cpu().double().numpy(), 1000)
    exact_sets_equal(idx.cpu().numpy(), oi)


# ------------------------------------------------- top-k: row spread over a cluster

def _cluster_rows(L, g):
    """Rows built to reach each step of the cluster select: a random row
    (prefix-sharing list ranked in the first CTA), an exact count at the
    level-1 and level-2 digits, exact ties at the k-th key (third level and
    the per-CTA tie quota), one value, and negative / infinite scores."""
    s = torch.randn(9, L, generator=g) * 3 + 10
    s[1] = 1.0
    s[1, torch.randperm(L, generator=g)[:2048]] = 100.0          # level-1 bin holds exactly k
    s[2] = 1.0
    s[2, torch.randperm(L, generator=g)[:2048]] = 1.0 + 2.0 ** -12  # same level-1 bin, level 2 exact
    s[3] = torch.randint(0, 3, (L,), generator=g).float()          # exact ties at the threshold
    s[4] = 7.0                                                     # one value
    s[5] = torch.rand(L, generator=g) * 1e-5 + 1.0                 # one narrow binade: level 3
    s[6, ::3] = float("-inf")
    s[6, 5] = float("inf")
    s[7] = -torch.rand(L, generator=g) - 2.0                       # all negative
    v = s[8].sort(descending=True).values[2047]
    s[8, torch.randperm(L, generator=g)[:40]] = v                  # a short list of exact ties at k
    return s


@pytest.mark.parametrize("L", [8193, 32768, 50001, 131072])
def test_topk_cluster_rows_every_branch(li, orc, L):
    """Few rows longer than 8,192 scores are spread over a thread-block
    cluster: every branch of its threshold search is bit-exact against the
    oracle's full sort, with and without valid lengths at CTA borders."""
    g = torch.Generator().manual_seed(L + 1)
    s = _cluster_rows(L, g)
    vl = torch.tensor([L, 8192, 8193, 0, 1, L - 1, 2049, 16383, L], dtype=torch.int32)
    for k in (1, 100, 2048, 2049, 8192):
        for v in (None, vl):
            gi, gv = _topk_gpu(li, s, k, v)
            oi, ov = orc.topk(s.double().numpy(), k, valid_len=None if v is None else v.numpy())
            exact_sets_equal(gi, oi)
            np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


@pytest.mark.parametrize("L", [100001, 131072])
def test_topk_wide_cluster_rows_every_branch(li, orc, L):
    """More rows than 256-thread clusters fit on the SMs (36 rows), few enough
    for clusters of 1,024-thread CTAs (32K keys each, 4 per row): every
    branch of the threshold search, bit-exact, with valid lengths at CTA
    borders."""
    g = torch.Generator().manual_seed(L + 7)
    s = torch.cat([_cluster_rows(L, g) for _ in range(4)])
    vl = torch.tensor([L, 32768, 32769, 0, 1, L - 1, 2049, 16383, L] * 4, dtype=torch.int32)
    for k in (1, 2048, 2049, 8192):
        for v in (None, vl):
            gi, gv = _topk_gpu(li, s, k, v)
            oi, ov = orc.topk(s.double().numpy(), k, valid_len=None if v is None else v.numpy())
            exact_sets_equal(gi, oi)
            np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_cluster_decode_and_anchor_shapes(li, orc):
    """Decode shapes on scores of the indexer's distribution (non-negative,
    heavy tail), bit-exact: 128 rows of 32K (top-2048, one CTA per row), 32
    rows of 128K (top-2048, clusters of four 1,024-thread CTAs) and the
    anchor's 8 rows of 128K (top-8192, clusters of sixteen 256-thread CTAs)."""
    g = torch.Generator().manual_seed(31)
    for rows, L, k in ((128, 32768, 2048), (32, 131072, 2048), (8, 131072, 8192)):
        s = (torch.randn(rows, L, generator=g).clamp_min(0) * 4) ** 2
        s[:, torch.randperm(L, generator=g)[: L // 100]] *= 16.0
        gi, gv = _topk_gpu(li, s, k)
        oi, ov = orc.topk(s.double().numpy(), k)
        exact_sets_equal(gi, oi)
        np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))


def test_topk_many_long_rows_take_the_per_row_paths(li, orc):
    """With as many long rows as twice the SMs or more, rows are not spread
    over clusters: one CTA per row (sampled thresholds, the exact fallback
    and its shared-memory overflow), or the two-pass path with a workspace.
    Ties across 32K segment borders and valid lengths included."""
    g = torch.Generator().manual_seed(32)
    rows, L = 320, 40000
    s = torch.randn(rows, L, generator=g) * 3 + 10
    s[1] = torch.randint(0, 7, (L,), generator=g).float()
    s[2, 30000:36000] = s[2].max() + 1.0
    s[3] = 1.0 + torch.rand(L, generator=g) * 1e-4             # threshold bin overflows
    s[4] = 5.0
    vl = torch.randint(0, L + 1, (rows,), generator=g, dtype=torch.int32)
    vl[:8] = L
    sd = s.to(DEV)
    for k in (1, 2048, 9000):
        for v in (None, vl):
            gi, gv = _topk_gpu(li, s, k, v)
            oi, ov = orc.topk(s.double().numpy(), k, valid_len=None if v is None else v.numpy())
            exact_sets_equal(gi, oi)
            np.testing.assert_array_equal(np.sort(gv, axis=1), np.sort(ov.astype(np.float32), axis=1))
        n = li.li_topk_workspace_size(rows, L, k)
        if n > 0:
            ws = torch.empty(n, dtype=torch.uint8, device=DEV)
            i1 = torch.empty(rows, k, dtype=torch.int32, device=DEV)
            assert li.li_topk(sd, k, i1, None, ws=ws) == 0
            _sync_ok(li)
            oi, _ = orc.topk(s.double().numpy(), k)
            exact_sets_equal(i1.cpu().numpy(), oi)


def test_topk_two_pass_full_segments(li, orc):
    """Many rows of exactly two 32K segments with a workspace (the two-pass
    path: more rows than the cluster path takes): ties across the segment
    border and a one-value row, bit-exact."""
    g = torch.Generator().manual_seed(33)
    rows, L = 300, 65536
    s = torch.randn(rows, L, generator=g) * 3 + 10
    s[1] = torch.randint(0, 5, (L,), generator=g).float()
    s[2, 30000:40000] = s[2].max() + 1.0
    s[3] = 2.5
    sd = s.to(DEV)
    for k in (1, 2048, 9000):
        n = li.li_topk_workspace_size(rows, L, k)
        assert n > 0
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        idx = torch.empty(rows, k, dtype=torch.int32, device=DEV)
        vals = torch.empty(rows, k, dtype=torch.float32, device=DEV)
        assert li.li_topk(sd, k, idx, vals, ws=ws) == 0
        _sync_ok(li)
        oi, ov = orc.topk(s.double().numpy(), k)
        exact_sets_equal(idx.cpu().numpy(), oi)
        np.testing.assert_array_equal(np.sort(vals.cpu().numpy(), axis=1), np.sort(ov.astype(np.float32), axis=1))
