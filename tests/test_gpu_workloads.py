"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times, on sampled outputs the oracle computes one sequence / query at
a time.  Inputs are generated on the GPU (seeded) and copied to the host for
the oracle.
"""
import numpy as np
import pytest
import torch

import li_inputs
from parity import RTOL, assert_scores_close, assert_topk_row

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _slice(x, b):
    return None if x is None else x[b:b + 1].cpu()


def test_batched_decode_fp8_32k_full_size(li, orc):
    x = li_inputs.make_workload(li_inputs.spec("fp8_32k_b32", native=False), seed=0, device=DEV)
    w = x["spec"]
    qa, qs = li.absorb_queries(x["q"], x["D"], "fp8")
    s = li.score_group(x["latent"], x["lat_scale"], qa, qs, x["w"])
    idx = li.topk(s, w.k)
    assert li.li_device_status() == 0
    D = x["D"].cpu()
    for b in (0, 13, w.B - 1):
        o = orc.score(_slice(x["latent"], b), _slice(x["lat_scale"], b),
                      orc.absorb(_slice(x["q"], b), D), _slice(x["w"], b))
        assert_scores_close(s[b:b + 1].cpu().numpy(), o, RTOL["fp8"], f"seq {b}")
        gi = idx[b, 0].cpu().numpy()
        for l in range(w.G):
            assert_topk_row(gi[l], o[0, 0, l], w.k, w.L, RTOL["fp8"], f"seq {b} layer {l}")


def test_hs_fp8_128k_full_size(li, orc):
    x = li_inputs.make_workload("fp8_128k_hs", seed=0, device=DEV)
    w = x["spec"]
    qa, qs = li.absorb_queries(x["q"], x["D"], "fp8")
    cand, idx = li.hs_select(x["latent"], x["lat_scale"], qa, qs, x["w"], w.m, w.k)
    s = li.score_group(x["latent"], x["lat_scale"], qa, qs, x["w"])
    full = li.topk(s, w.k)
    assert li.li_device_status() == 0
    D = x["D"].cpu()
    for b in (0, w.B - 1):
        o = orc.score(_slice(x["latent"], b), _slice(x["lat_scale"], b),
                      orc.absorb(_slice(x["q"], b), D), _slice(x["w"], b))[0, 0]   # [G][L]
        assert_scores_close(s[b, 0].cpu().numpy(), o, RTOL["fp8"], f"full scan seq {b}")
        c = cand[b].cpu().numpy()
        assert_topk_row(c, o[0], w.m, w.L, RTOL["fp8"], f"candidates seq {b}")
        C = set(c.tolist())
        gi = idx[b].cpu().numpy()
        fi = full[b, 0].cpu().numpy()
        for l in range(w.G):
            assert_topk_row(gi[l], o[l], w.k, w.L, RTOL["fp8"], f"HS seq {b} layer {l}", allowed=C)
            assert_topk_row(fi[l], o[l], w.k, w.L, RTOL["fp8"], f"full seq {b} layer {l}")


def test_prefill_bf16_128k_full_size_sampled_queries(li, orc):
    x = li_inputs.make_workload("prefill_bf16_128k", seed=0, device=DEV)
    w = x["spec"]
    qa, qs = li.absorb_queries(x["q"], x["D"], "bf16")
    s = li.score_group(x["latent"], None, qa, None, x["w"], q_pos=x["q_pos"])
    vl = (x["q_pos"] + 1).repeat_interleave(w.G)                 # rows are (query, layer)
    idx = li.topk(s, w.k, valid_len=vl)
    assert li.li_device_status() == 0
    lat = x["latent"].cpu()
    D = x["D"].cpu()
    for t in (0, 1777, w.T - 1):
        p = int(x["q_pos"][t])
        qt = x["q"][:, t:t + 1].cpu()
        o = orc.score(lat, None, orc.absorb(qt, D), x["w"][:, t:t + 1].cpu(),
                      q_pos=x["q_pos"][t:t + 1].cpu())[0, 0]      # [G][L]
        assert_scores_close(s[0, t, :, :p + 1].cpu().numpy(), o[:, :p + 1], RTOL["bf16"], f"query {t}")
        gi = idx[0, t].cpu().numpy()
        for l in range(w.G):
            assert_topk_row(gi[l], o[l], w.k, p + 1, RTOL["bf16"], f"query {t} layer {l}")


def test_native_dsa_8k_full_size(li, orc):
    x = li_inputs.make_workload("dsa_bf16_8k", seed=0, device=DEV)
    w = x["spec"]
    for l in range(w.G):
        q8, s8 = li.absorb_queries(x["q"][:, :, l:l + 1].contiguous(), None, "fp8")
        g = li.native_score(x["keys"][l], x["key_scale"][l], q8.view(w.B, w.H, w.d),
                            s8.view(w.B, w.H), x["w"][:, 0, l].contiguous())
        idx = li.topk(g, w.k)
        assert li.li_device_status() == 0
        o = orc.native_score(x["keys"][l].cpu(), x["key_scale"][l].cpu(),
                             orc.decode_rows(x["q"][:, 0, l].cpu()), x["w"][:, 0, l].cpu())
        assert_scores_close(g.cpu().numpy(), o, RTOL["fp8"], f"layer {l}")
        assert_topk_row(idx[0].cpu().numpy(), o[0], w.k, w.L, RTOL["fp8"], f"layer {l}")
