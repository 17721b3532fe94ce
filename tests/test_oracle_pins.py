"""Pins of the CPU oracle to what the pages and the mathematics fix (CPU only).

Each test ties one oracle function to something other than itself: a
hand-worked example, a library decoder, the exact identity of eq. (7), a
brute-force sort, the HS limits of the summary page or the storage numbers
of the explainer page.  A plausible mistake in the oracle (a dropped term, a
wrong sign or index, a transposed operand) fails at least one of them; the
"planted mistake" tests at the end show that for a few such mistakes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import li_inputs
from oracle import twin

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def hand():
    h = _load("hand_worked_example.json")
    G, H, d, r, L = h["G"], h["H"], h["d"], h["r"], h["L"]
    h["D_np"] = np.array(h["D"], dtype=np.float64).reshape(G, r, d)
    h["q_np"] = np.array(h["q"], dtype=np.float64).reshape(1, 1, G, H, d)
    h["w_np"] = np.array(h["w"], dtype=np.float64).reshape(1, 1, G, H)
    h["c_np"] = np.array(h["latent"], dtype=np.float64).reshape(1, L, r)
    return h


# ----------------------------------------------------------- format decoders

def test_e4m3_decode_all_codes_match_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_decode_spec_points(orc):
    # OCP FP8 E4M3: bias 7, max normal 1.75*2^8 = 448, min normal 2^-6,
    # min subnormal 2^-9, S.1111.111 NaN, negative zero.
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0xB8) == -1.0
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_decode(0x70) == 128.0
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))
    z = orc.e4m3_decode(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def test_bf16_decode_matches_torch(orc):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4096, generator=g) * 100
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_decode(int(v)) for v in bits[:512]])
    np.testing.assert_array_equal(got, b.double().numpy()[:512])
    np.testing.assert_array_equal(orc.decode_rows(b), b.double().numpy())


def test_twin_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = twin.e4m3_values()
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert np.isnan(got[~ok]).all()


def test_decode_rows_applies_per_row_scale(orc):
    codes = torch.tensor([[0x38, 0x40], [0x38, 0xB8]], dtype=torch.uint8)  # 1, 2 ; 1, -1
    out = orc.decode_rows(codes, torch.tensor([0.5, 3.0]))
    np.testing.assert_array_equal(out, [[0.5, 1.0], [3.0, -3.0]])


# ------------------------------------------------------- hand-worked example

def test_hand_example_absorption(orc, hand):
    got = orc.absorb(hand["q_np"], hand["D_np"])
    np.testing.assert_array_equal(got[0, 0], np.array(hand["qabs"], dtype=np.float64))


def test_hand_example_key_reconstruction(orc, hand):
    keys = orc.reconstruct_keys(hand["c_np"], None, hand["D_np"])
    np.testing.assert_array_equal(keys[:, 0], np.array(hand["keys"], dtype=np.float64))


def test_hand_example_scores(orc, hand):
    qabs = orc.absorb(hand["q_np"], hand["D_np"])
    u = orc.score(hand["c_np"], None, qabs, hand["w_np"])
    np.testing.assert_array_equal(u[0, 0], np.array(hand["scores"]))


def test_hand_example_scores_with_beta(orc, hand):
    qabs = orc.absorb(hand["q_np"], hand["D_np"])
    beta = np.array(hand["beta"], dtype=np.float64).reshape(1, 1, 2, 2)
    u = orc.score(hand["c_np"], None, qabs, hand["w_np"], beta=beta)
    np.testing.assert_array_equal(u[0, 0], np.array(hand["scores_beta"]))


def test_hand_example_fp8_latent(orc, hand):
    f = hand["fp8_latent"]
    codes = np.array(f["codes"], dtype=np.uint8).reshape(1, 4, 3)
    scale = np.array(f["scale"], dtype=np.float32).reshape(1, 4)
    qabs = orc.absorb(hand["q_np"], hand["D_np"])
    u = orc.score(codes, scale, qabs, hand["w_np"])
    np.testing.assert_array_equal(u[0, 0], np.array(hand["scores"]))


def test_hand_example_topk(orc, hand):
    scores = np.array(hand["scores"])
    for k, want in hand["topk"].items():
        idx, vals = orc.topk(scores, int(k))
        np.testing.assert_array_equal(idx, np.array(want))
        n = min(int(k), 4)
        np.testing.assert_array_equal(vals[:, :n], np.take_along_axis(scores, idx[:, :n], 1))
        assert np.all(np.isneginf(vals[:, n:]))


def test_hand_example_hs(orc, hand):
    scores = np.array(hand["scores"]).reshape(1, 2, 4)
    for key, want in hand["hs"].items():
        m = int(key[1]); k = int(key.split("_k")[1])
        cand, idx = orc.hs(scores, m, k)
        np.testing.assert_array_equal(cand[0], want["cand"])
        np.testing.assert_array_equal(idx[0], want["idx"])


# ------------------------------------------------ eq. (7): the exact identity

@pytest.mark.parametrize("lat_dtype", ["f32", "bf16", "fp8"])
def test_absorbed_scoring_equals_reconstructed_key_scoring(orc, lat_dtype):
    """Eq. (7) with b = 0: q . (D_l^T c) = (D_l q) . c, so scoring the shared latent
    with absorbed queries equals the native per-layer scorer run on the keys the
    decoders reconstruct (two different oracle code paths)."""
    w = li_inputs.spec("tiny_f32", L=300, G=3, H=5, d=24, r=40, lat_dtype=lat_dtype,
                       q_dtype="bf16" if lat_dtype != "f32" else "f32", B=2)
    x = li_inputs.make_workload(w, seed=11)
    qabs = orc.absorb(x["q"], x["D"])
    u = orc.score(x["latent"], x["lat_scale"], qabs, x["w"])          # [B][1][G][L]
    keys = orc.reconstruct_keys(x["latent"], x["lat_scale"], x["D"])  # [G][B][L][d]
    qd = orc.decode_rows(x["q"])                                       # [B][1][G][H][d]
    wd = x["w"].double().numpy()
    for l in range(w.G):
        nat = orc.native_score(keys[l], None, qd[:, 0, l], wd[:, 0, l])
        np.testing.assert_allclose(u[:, 0, l], nat, rtol=1e-12, atol=1e-12)


def test_identity_decoder_reduces_to_native_scan(orc):
    """G=1 with D = I (r = d): the latent scan is the native scan on the same keys."""
    B, L, d, H = 2, 257, 32, 6
    keys, kscale, _ = li_inputs.make_latent(B, L, d, "fp8", seed=3)
    q = torch.randn(B, 1, 1, H, d, generator=torch.Generator().manual_seed(4))
    w = torch.rand(B, 1, 1, H, generator=torch.Generator().manual_seed(6))
    eye = torch.eye(d).reshape(1, d, d)
    qabs = orc.absorb(q, eye)
    np.testing.assert_array_equal(qabs, q.double().numpy())
    u = orc.score(keys, kscale, qabs, w)
    nat = orc.native_score(keys, kscale, q[:, 0, 0], w[:, 0, 0])
    np.testing.assert_array_equal(u[:, 0, 0], nat)


def test_single_head_unit_weight_is_relu_gemv(orc):
    """H = 1, w = 1, beta = 0: u_t = ReLU(q~ . c_t), a plain GEMV (numpy matmul)."""
    g = np.random.default_rng(9)
    c = g.standard_normal((1, 333, 48))
    qa = g.standard_normal((1, 1, 1, 1, 48))
    u = orc.score(c, None, qa, np.ones((1, 1, 1, 1)))
    ref = np.maximum(c[0] @ qa[0, 0, 0, 0], 0.0)
    np.testing.assert_allclose(u[0, 0, 0], ref, rtol=1e-13, atol=1e-13)


def test_relu_homogeneity_in_latent_scale(orc):
    """beta = 0 and s > 0: ReLU(s x) = s ReLU(x), so doubling every token scale doubles u."""
    lat, sc, _ = li_inputs.make_latent(1, 500, 64, "fp8", seed=21)
    qa = np.random.default_rng(2).standard_normal((1, 1, 2, 4, 64))
    w = np.random.default_rng(3).random((1, 1, 2, 4))
    u1 = orc.score(lat, sc, qa, w)
    u2 = orc.score(lat, sc * 2, qa, w)
    np.testing.assert_array_equal(u2, 2 * u1)


def test_causal_valid_set(orc):
    """V_s = {t <= pos}: positions past a query's position score -inf, the rest match the
    decode scan (q_pos NULL)."""
    lat, _, _ = li_inputs.make_latent(1, 64, 16, "f32", seed=1)
    qa = np.random.default_rng(0).standard_normal((1, 3, 2, 2, 16))
    w = np.random.default_rng(1).random((1, 3, 2, 2))
    pos = np.array([0, 31, 63], dtype=np.int32)
    u = orc.score(lat, None, qa, w, q_pos=pos)
    full = orc.score(lat, None, qa, w)
    for i, p in enumerate(pos):
        np.testing.assert_array_equal(u[0, i, :, :p + 1], full[0, i, :, :p + 1])
        assert np.isneginf(u[0, i, :, p + 1:]).all()


# ---------------------------------------------------------------- selection

def _brute_topk(row, k, V=None):
    V = len(row) if V is None else V
    order = sorted(range(V), key=lambda t: (-row[t], t))
    return order[:k] + [-1] * max(0, k - V)


def test_topk_brute_force_with_ties(orc):
    rng = np.random.default_rng(7)
    for trial in range(60):
        L = int(rng.integers(1, 65))
        row = rng.integers(-3, 4, size=L).astype(np.float64)   # many ties
        for k in (1, max(1, L // 3), L, L + 5):
            V = int(rng.integers(0, L + 1))
            idx, _ = orc.topk(row[None], k, valid_len=np.array([V]))
            assert idx[0].tolist() == _brute_topk(row.tolist(), k, V)


def test_topk_invariants_random(orc):
    rng = np.random.default_rng(8)
    s = rng.standard_normal((6, 1000))
    idx, vals = orc.topk(s, 100)
    for r in range(6):
        S = set(idx[r].tolist())
        assert len(S) == 100 and min(S) >= 0 and max(S) < 1000
        rest = np.setdiff1d(np.arange(1000), idx[r])
        assert s[r, idx[r]].min() >= s[r, rest].max()
        assert np.all(np.diff(vals[r]) <= 0)


def test_twin_matches_c_oracle_tiny_workload(orc):
    """The two independent oracle implementations agree on the tiny fp32 workload."""
    x = li_inputs.make_workload("tiny_f32", seed=0)
    w = x["spec"]
    qabs = orc.absorb(x["q"], x["D"])
    qabs_t = twin.absorb(twin.decode(x["q"].numpy()), twin.decode(x["D"].numpy()))
    np.testing.assert_allclose(qabs, qabs_t, rtol=1e-12, atol=1e-14)
    u = orc.score(x["latent"], None, qabs, x["w"])
    u_t = twin.score(twin.decode(x["latent"].numpy()), qabs_t, x["w"].double().numpy())
    np.testing.assert_allclose(u, u_t, rtol=1e-11, atol=1e-12)
    idx, _ = orc.topk(u[0, 0], w.k)
    np.testing.assert_array_equal(idx, twin.topk(u[0, 0], w.k))


def test_twin_matches_c_oracle_fp8_causal_beta(orc):
    lat, sc, _ = li_inputs.make_latent(2, 300, 64, "fp8", seed=5)
    qa_codes, qa_scale = li_inputs.make_absorbed_queries(2, 3, 2, 4, 64, "fp8", seed=5)
    qa = orc.decode_rows(qa_codes, qa_scale)
    w = torch.rand(2, 3, 2, 4, generator=torch.Generator().manual_seed(1))
    beta = li_inputs.make_beta(2, 3, 2, 4, seed=5)
    pos = np.array([10, 200, 299], dtype=np.int32)
    u = orc.score(lat, sc, qa, w, beta=beta, q_pos=pos)
    u_t = twin.score(twin.decode(lat.numpy(), sc.numpy()), twin.decode(qa_codes.numpy(), qa_scale.numpy()),
                     w.double().numpy(), beta=beta.double().numpy(), q_pos=pos)
    np.testing.assert_allclose(u, u_t, rtol=1e-11, atol=1e-12)


# --------------------------------------------------- hierarchical selection

def test_hs_with_budget_at_least_L_is_full_latentindex(orc):
    """Summary page, HS paragraph: with B >= L every position is a candidate, so each
    follower's selection is its full LatentIndex TopK."""
    rng = np.random.default_rng(12)
    s = rng.standard_normal((3, 4, 700))
    for m in (700, 1000):
        cand, idx = orc.hs(s, m, 50)
        full, _ = orc.topk(s, 50)
        np.testing.assert_array_equal(idx, full)


def test_hs_budget_equal_k_gives_candidate_set(orc):
    rng = np.random.default_rng(13)
    s = rng.standard_normal((2, 4, 900))
    cand, idx = orc.hs(s, 64, 64)
    for b in range(2):
        for l in range(4):
            assert set(idx[b, l].tolist()) == set(cand[b].tolist())


def test_hs_matches_twin_and_anchor_subset(orc):
    rng = np.random.default_rng(14)
    s = np.round(rng.standard_normal((3, 4, 500)), 1)          # ties
    cand, idx = orc.hs(s, 128, 40)
    cand_t, idx_t = twin.hs(s, 128, 40)
    np.testing.assert_array_equal(cand, cand_t)
    np.testing.assert_array_equal(idx, idx_t)
    for b in range(3):
        assert set(idx[b, 0].tolist()) <= set(cand[b].tolist())
        for l in range(1, 4):
            assert set(idx[b, l].tolist()) <= set(cand[b].tolist())


def test_hs_pads_when_budget_exceeds_context(orc):
    s = np.random.default_rng(1).standard_normal((1, 2, 10))
    cand, idx = orc.hs(s, 16, 12)
    assert (cand[0, 10:] == -1).all() and sorted(cand[0, :10].tolist()) == list(range(10))
    assert (idx[0, :, 10:] == -1).all()


def test_hs_scored_positions_formula(orc):
    g = _load("storage_arithmetic.json")
    L, m = g["tokens_128k"]["value"], g["hs_candidates"]["value"]
    assert orc.hs_scored_positions(L, 4, m) == L + 3 * m == 155648
    assert L // m == g["hs_follower_reduction"]["value"]
    assert orc.hs_scored_positions(L, 4, 2 * L) == 4 * L     # B >= L: the full scan


# ------------------------------------------------------- storage arithmetic

def test_storage_numbers_of_the_pages(orc):
    g = _load("storage_arithmetic.json")
    nat, lat = orc.indexer_cache_bytes_per_token(
        g["indexer_layers"]["value"], g["groups"]["group_size"],
        g["native_key_bytes_per_layer"]["value"], g["latent_bytes_per_group"]["value"])
    assert nat == g["native_bytes_per_token"]["value"]
    assert lat == g["latentindex_bytes_per_token"]["value"]
    assert round(100 * (1 - lat / nat), 1) == g["reduction_percent"]["value"]
    n = g["tokens_128k"]["value"]
    assert round(nat * n / 1e9, 2) == g["native_gb_at_128k"]["value"]
    assert round(lat * n / 1e9, 2) == g["latentindex_gb_at_128k"]["value"]
    assert orc.payload_ratio(g["latent_values"]["value"], 4, 128) == 0.375


def test_storage_of_this_library_layout(orc):
    """The library stores the fp8 latent as 192 codes + one fp32 scale = 196 B per token
    per group (the pages' 200 B leave 8 B for scales); native keys 128 + 4 = 132 B."""
    nat, lat = orc.indexer_cache_bytes_per_token(61, 4, 128 + 4, 192 + 4)
    assert nat == 8052 and lat == 132 + 15 * 196
    assert round(100 * (1 - lat / nat), 2) == 61.85


# ------------------------------------------- planted mistakes fail the pins

def test_planted_transposed_decoder_fails_identity(orc):
    """Absorbing with D_l^T instead of D_l (square, non-symmetric decoders) breaks the
    eq. (7) pin: absorbed scoring no longer equals reconstructed-key scoring."""
    rng = np.random.default_rng(31)
    d = 16
    D = rng.standard_normal((2, d, d))
    q = rng.standard_normal((1, 1, 2, 3, d))
    w = rng.random((1, 1, 2, 3))
    c = rng.standard_normal((1, 50, d))
    keys = orc.reconstruct_keys(c, None, D)
    good = orc.score(c, None, orc.absorb(q, D), w)
    bad = orc.score(c, None, np.einsum("gdr,...ghd->...ghr", D, q), w)
    for l in range(2):
        nat = orc.native_score(keys[l], None, q[:, 0, l], w[:, 0, l])
        np.testing.assert_allclose(good[:, 0, l], nat, rtol=1e-12, atol=1e-12)
        assert not np.allclose(bad[:, 0, l], nat, rtol=1e-6)


def test_planted_dropped_relu_or_weight_fails_hand_example(hand):
    qabs = twin.absorb(hand["q_np"], hand["D_np"])
    dots = np.einsum("btghr,blr->btghl", qabs, hand["c_np"])
    no_relu = np.einsum("btgh,btghl->btgl", hand["w_np"], dots)[0, 0]
    no_w = np.maximum(dots, 0).sum(axis=3)[0, 0]
    want = np.array(hand["scores"])
    assert not np.array_equal(no_relu, want)
    assert not np.array_equal(no_w, want)
    np.testing.assert_array_equal(twin.score(hand["c_np"], qabs, hand["w_np"])[0, 0], want)


def test_planted_wrong_tie_break_fails_brute_force():
    row = [1.0, 2.0, 2.0, 0.0]
    assert _brute_topk(row, 2) == [1, 2]
    wrong = sorted(range(4), key=lambda t: (-row[t], -t))[:2]
    assert wrong != _brute_topk(row, 2)


# ------------------------------------------------- latent append, eqs. (1)-(2)

def _append_case(B=3, dm=48, r=24, rR=8, seed=31):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, dm, generator=g, dtype=torch.float64)
    P = torch.randn(r, dm, generator=g, dtype=torch.float64) / math.sqrt(dm)
    return x.numpy(), P.numpy(), rR


def test_append_at_position_zero_is_the_projection(orc):
    x, P, rR = _append_case()
    c = orc.append_latent(x, P, rR, np.zeros(3, dtype=np.int32))
    np.testing.assert_allclose(c, x @ P.T, rtol=1e-12, atol=1e-12)


def test_append_rotation_keeps_pair_norms_and_leaves_nope_alone(orc):
    x, P, rR = _append_case()
    pos = np.array([1, 777, 131071], dtype=np.int32)
    c = orc.append_latent(x, P, rR, pos)
    raw = x @ P.T
    n_c = np.hypot(c[:, 0:rR:2], c[:, 1:rR:2])
    n_raw = np.hypot(raw[:, 0:rR:2], raw[:, 1:rR:2])
    np.testing.assert_allclose(n_c, n_raw, rtol=1e-12)
    np.testing.assert_allclose(c[:, rR:], raw[:, rR:], rtol=1e-12, atol=1e-15)


def test_append_rope_scores_depend_only_on_relative_position(orc):
    """<Q_t a, Q_s b> = <Q_{t-s} a, b> on the RoPE branch: the property rotary
    encoding is for (a wrong sign or frequency index breaks it)."""
    x, P, rR = _append_case(B=2)
    def rope_part(pos):
        return orc.append_latent(x, P, rR, np.asarray(pos, dtype=np.int32))[:, :rR]
    for t, s in ((5, 2), (1000, 37), (40000, 39999)):
        a_t, b_s = rope_part([t, s])
        a_d, b_0 = rope_part([t - s, 0])
        lhs = float(a_t @ b_s)             # token 0 at t, token 1 at s
        rhs = float(a_d @ b_0)             # token 0 at t - s, token 1 at 0
        assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + 1.0)


def test_append_frequency_schedule_on_unit_vectors(orc):
    """A unit input on RoPE pair i comes out as (cos t.theta_i, sin t.theta_i),
    theta_i = 10000^(-2i/rR): the first pair turns by t radians, the last
    pair slowest."""
    rR, r, dm = 8, 8, 8
    P = np.eye(r, dm)
    for i in range(rR // 2):
        x = np.zeros((1, dm))
        x[0, 2 * i] = 1.0
        for t in (1, 3, 100):
            c = orc.append_latent(x, P, rR, np.array([t], dtype=np.int32))[0]
            ang = t * 10000.0 ** (-2.0 * i / rR)
            np.testing.assert_allclose(c[2 * i:2 * i + 2], [math.cos(ang), math.sin(ang)], atol=1e-12)
            assert np.abs(np.delete(c, [2 * i, 2 * i + 1])).max() < 1e-15


def test_append_twin_matches_c_oracle(orc):
    x, P, rR = _append_case(B=4, dm=64, r=40, rR=16, seed=32)
    pos = np.array([0, 9, 4096, 131071], dtype=np.int32)
    np.testing.assert_allclose(orc.append_latent(x, P, rR, pos), twin.append_latent(x, P, rR, pos),
                               rtol=1e-11, atol=1e-12)


def test_planted_reversed_rotation_fails_frequency_schedule():
    """A rotation by -t.theta (a sign slip in Q_t) keeps norms and relative
    positions but fails the unit-vector schedule."""
    rR = dm = 4
    P = np.eye(rR, dm)
    x = np.zeros((1, dm))
    x[0, 0] = 1.0
    good = twin.append_latent(x, P, rR, [3])[0]
    bad = twin.append_latent(x, P, rR, [-3])[0]          # same as rotating by -3 theta_0
    np.testing.assert_allclose(good[:2], [math.cos(3.0), math.sin(3.0)], atol=1e-12)
    assert abs(bad[1] - math.sin(3.0)) > 0.1


def test_two_pass_selection_equals_one_pass(orc):
    """The long-row top-k of the GPU library selects in two passes: the exact
    top-k of each segment, then the top-k of the segments' candidates with
    ties by position.  On the oracle, with heavy ties across segments, the
    two passes give the one-pass set (the row's top-k lies inside the union
    of its segments' top-k)."""
    g = torch.Generator().manual_seed(51)
    L, seg = 1000, 256
    rows = [torch.randint(0, 6, (L,), generator=g).double(),
            torch.randn(L, generator=g, dtype=torch.float64),
            torch.full((L,), 2.0, dtype=torch.float64)]
    for s in rows:
        s = s.numpy()
        for k in (1, 7, 100, 256):
            want, _ = orc.topk(s[None], k)
            cand_pos, cand_val = [], []
            for a in range(0, L, seg):
                i, v = orc.topk(s[None, a:a + seg], k)
                n = min(k, min(seg, L - a))
                cand_pos.append(i[0, :n] + a)
                cand_val.append(v[0, :n])
            cp, cv = np.concatenate(cand_pos), np.concatenate(cand_val)
            order = np.argsort(cp, kind="stable")        # candidates in position order,
            cp, cv = cp[order], cv[order]                 # so ties resolve by position
            j, _ = orc.topk(cv[None], k)
            got = cp[j[0][j[0] >= 0]]
            assert sorted(got.tolist()) == sorted(want[0][want[0] >= 0].tolist())


# --------------------------------- rotary-constrained decoders, eqs. (3)-(4)

def _rot_matrix(orc, n, t):
    """The rotation of `orc.rope_rotate` at position t as an n x n matrix M with M v = rotated v."""
    rows = orc.rope_rotate(np.eye(n), n, np.full(n, t, dtype=np.int32))   # row i = (M e_i)^T
    return rows.T


@pytest.mark.parametrize("dR,rR", [(8, 8), (8, 16), (64, 64)])
def test_rotary_decoder_commutes_with_rotation(orc, dR, rR):
    """Eq. (4): R_t D^R = D^R Q_t for every position t, with R_t the key's and
    Q_t the latent's rotary encoding (each with its own width)."""
    rng = np.random.default_rng(41)
    DR = orc.rotary_decoder(rng.standard_normal((dR // 2, rR // 2)),
                            rng.standard_normal((dR // 2, rR // 2)), dR, rR)
    assert np.abs(DR).sum() > 0
    for t in (1, 7, 1000, 131071):
        lhs = _rot_matrix(orc, dR, t) @ DR
        rhs = DR @ _rot_matrix(orc, rR, t)
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_rotation_matrix_is_the_frequency_schedule(orc):
    """Pair j of an n-wide rotary encoding turns by t * 10000^(-2j/n): the
    matrix form used by the eq. (4) pins, checked entry by entry."""
    n, t = 6, 5
    M = _rot_matrix(orc, n, t)
    want = np.zeros((n, n))
    for j in range(n // 2):
        a = t * 10000.0 ** (-2.0 * j / n)
        want[2 * j:2 * j + 2, 2 * j:2 * j + 2] = [[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]]
    np.testing.assert_allclose(M, want, atol=1e-13)


def test_planted_real_block_fails_rotary_constraint(orc):
    """A decoder block that is a real 2 x 2 matrix but not a complex number
    ([[a, b], [b, -a]], a reflection) breaks eq. (4)."""
    a, b = 0.7, -0.4
    DR = np.array([[a, b], [b, -a]])
    t = 3
    lhs = _rot_matrix(orc, 2, t) @ DR
    rhs = DR @ _rot_matrix(orc, 2, t)
    assert np.abs(lhs - rhs).max() > 0.1


def test_input_generator_rotary_decoders_match_oracle_builder(orc):
    """The decoders the GPU tests store (li_inputs) have, in their RoPE block,
    the oracle's eq. (4) decoder of the same draws, and in their NoPE block the
    drawn DN; the cross blocks are zero."""
    G, r, rR, d, dR = 3, 40, 16, 24, 8
    dec = li_inputs.make_rotary_decoders(G, r, rR, d, dR, seed=5)
    D = dec["D"].double().numpy()
    for l in range(G):
        DR = orc.rotary_decoder(dec["a_re"][l], dec["a_im"][l], dR, rR)
        np.testing.assert_array_equal(D[l, :rR, :dR], DR.T)
        np.testing.assert_array_equal(D[l, rR:, dR:], dec["DN"][l].numpy().T)
        assert not D[l, :rR, dR:].any() and not D[l, rR:, :dR].any()


def _rotary_case(orc, B=3, dm=40, r=24, rR=8, d=20, dR=8, G=2, H=3, seed=43):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, dm))
    P = rng.standard_normal((r, dm)) / math.sqrt(dm)
    DR = np.stack([orc.rotary_decoder(rng.standard_normal((dR // 2, rR // 2)),
                                      rng.standard_normal((dR // 2, rR // 2)), dR, rR) for _ in range(G)])
    DN = rng.standard_normal((G, d - dR, r - rR)) / math.sqrt(r)
    bias = rng.standard_normal((G, d - dR))
    q = rng.standard_normal((B, 1, G, H, d)) / math.sqrt(d)
    w = rng.random((B, 1, G, H))
    D = np.zeros((G, r, d))
    D[:, :rR, :dR] = DR.transpose(0, 2, 1)
    D[:, rR:, dR:] = DN.transpose(0, 2, 1)
    return dict(x=x, P=P, DR=DR, DN=DN, bias=bias, q=q, w=w, D=D, rR=rR, dR=dR, G=G)


def _latent_route(orc, c, k, pos, with_bias=True):
    """Eqs. (1)-(2), (6), (8): score the rotated latent with absorbed queries (+ beta)."""
    lat = orc.append_latent(c["x"], c["P"], c["rR"], pos)           # [B][r]
    qabs = orc.absorb(c["q"], c["D"])                               # [B][1][G][H][r]
    beta = np.einsum("btghn,gn->btgh", c["q"][..., c["dR"]:], c["bias"]) if with_bias else None
    B = lat.shape[0]
    # one cached token per sequence: score it with its own sequence's queries
    return np.stack([orc.score(lat[b:b + 1, None], None, qabs[b:b + 1], c["w"][b:b + 1],
                               None if beta is None else beta[b:b + 1])[0, 0, :, 0] for b in range(B)])


def _key_route(orc, c, pos):
    """Eq. (3) with eq. (4): per-layer keys rotated after decoding, scored natively."""
    keys = orc.rope_keys(c["x"], c["P"], c["rR"], c["DR"], c["DN"], pos, bias=c["bias"])  # [G][B][d]
    B = keys.shape[1]
    return np.stack([[orc.native_score(keys[l, b:b + 1, None], None, c["q"][b:b + 1, 0, l],
                                       c["w"][b:b + 1, 0, l])[0, 0] for l in range(c["G"])]
                     for b in range(B)])


@pytest.mark.parametrize("shape", [dict(), dict(r=48, rR=16, d=24, dR=8), dict(r=32, rR=8, d=24, dR=16)])
def test_rotary_latent_scoring_equals_rope_key_scoring(orc, shape):
    """Eqs. (1), (3), (4), (6)-(8) end to end: scoring the cached latent, which
    is rotated once by Q_t, with decoder-absorbed queries and beta gives the
    scores of the per-layer keys [R_t D^R z^R ; D^N z^N + b] that the native
    indexer would cache."""
    c = _rotary_case(orc, **shape)
    for pos in ([0, 1, 2], [5, 131071, 4096]):
        pos = np.array(pos, dtype=np.int32)
        got = _latent_route(orc, c, 0, pos)
        want = _key_route(orc, c, pos)
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
        assert (want > 0).any()


def test_planted_reversed_latent_rotation_fails_key_identity(orc):
    """Rotating the latent by -t (the conjugate of Q_t) breaks the identity."""
    c = _rotary_case(orc)
    pos = np.array([9, 300, 77], dtype=np.int32)
    want = _key_route(orc, c, pos)
    bad = _latent_route(orc, c, 0, -pos)
    assert np.abs(bad - want).max() > 1e-3 * np.abs(want).max()


def test_planted_dropped_bias_fails_key_identity(orc):
    c = _rotary_case(orc)
    pos = np.array([9, 300, 77], dtype=np.int32)
    assert np.abs(_latent_route(orc, c, 0, pos, with_bias=False) - _key_route(orc, c, pos)).max() > 1e-6


def test_rope_key_scores_depend_only_on_relative_position(orc):
    """With the query's RoPE part rotated by R_s, the score of a key at t
    depends on s - t only: shifting both positions leaves it unchanged."""
    c = _rotary_case(orc, B=1)
    dR = c["dR"]
    q0 = c["q"].copy()

    def score_at(s, t):
        q = q0.copy()
        flat = q.reshape(-1, q.shape[-1])
        flat[:] = orc.rope_rotate(flat, dR, np.full(flat.shape[0], s, dtype=np.int32))
        keys = orc.rope_keys(c["x"], c["P"], c["rR"], c["DR"], c["DN"], np.array([t], dtype=np.int32),
                             bias=c["bias"])
        return np.array([orc.native_score(keys[l, :, None], None, q[:, 0, l], c["w"][:, 0, l])[0, 0]
                         for l in range(c["G"])])
    for s, t, shift in ((10, 3, 1000), (5000, 4999, 77), (0, 0, 131000)):
        np.testing.assert_allclose(score_at(s, t), score_at(s + shift, t + shift), rtol=1e-9, atol=1e-12)
