"""li_hs_select_noalloc: hierarchical selection for callers that cannot
allocate device memory (for example a plugin whose host engine owns all device
memory, or a decode loop that must not call cudaMalloc).  Its scratch is the
library's fixed 8 MiB device array; the test checks, through the C ABI, that
two calls in a row give the same candidates and selections as li_hs_select
with a caller workspace, and that both meet the fp64 oracle's hierarchical
selection under the band rule.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import li_inputs
from parity import RTOL, assert_topk_row, exact_sets_equal

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(seed):
    w = li_inputs.spec("fp8_128k_hs", B=3, L=20000, m=2048, k=512)
    xc = li_inputs.make_workload(w, seed=seed)
    x = {n: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for n, v in xc.items()}
    return w, x, xc


def _check_against_oracle(orc, w, xc, cand, idx):
    """The candidates are the anchor's top-m and each layer's selection its
    top-k inside them, against fp64 oracle scores (band rule at fp8's rtol)."""
    o = orc.score(xc["latent"], xc["lat_scale"], orc.absorb(xc["q"], xc["D"]), xc["w"])[:, 0]
    c, gi = cand.cpu().numpy(), idx.cpu().numpy()
    nc = min(w.m, w.L)
    for b in range(w.B):
        assert_topk_row(c[b], o[b, 0], w.m, w.L, RTOL["fp8"], f"noalloc cand b{b}")
        C = set(c[b, :nc].tolist())
        for l in range(w.G):
            assert_topk_row(gi[b, l], o[b, l], w.k, w.L, RTOL["fp8"], f"noalloc b{b} l{l}", allowed=C)


def test_noalloc_matches_workspace_version_twice(li, orc):
    w, x, xc = _inputs(7)
    qa, qs = li.absorb_queries(x["q"], x["D"], "fp8")
    ref_c, ref_i = li.hs_select(x["latent"], x["lat_scale"], qa, qs, x["w"], w.m, w.k)
    assert li.li_device_status() == 0
    for call in range(2):
        cand = torch.full((w.B, w.m), -7, dtype=torch.int32, device=DEV)
        idx = torch.full((w.B, w.G, w.k), -7, dtype=torch.int32, device=DEV)
        st = li.li_hs_select_noalloc(x["latent"], x["lat_scale"], qa, qs, x["w"], w.m, w.k, cand, idx)
        assert st == 0, li.li_status_string(st)
        assert li.li_device_status() == 0
        # identical kernels on identical inputs: the same sets (slot order may differ)
        exact_sets_equal(cand.cpu().numpy(), ref_c.cpu().numpy())
        exact_sets_equal(idx.cpu().numpy(), ref_i.cpu().numpy())
    _check_against_oracle(orc, w, xc, cand, idx)


def test_noalloc_rejects_sizes_beyond_its_scratch(li):
    # B = 16, L = 131072 needs 8 MiB of anchor scores alone, more than the array
    need = li.li_hs_workspace_size(16, 4, 131072, 8192, 2048)
    assert need > 8 << 20
    lat = torch.empty(16, 131072, 192, dtype=torch.uint8, device=DEV)
    sc = torch.empty(16, 131072, dtype=torch.float32, device=DEV)
    qa = torch.empty(16, 1, 4, 64, 192, dtype=torch.uint8, device=DEV)
    qs = torch.empty(16, 1, 4, 64, dtype=torch.float32, device=DEV)
    wt = torch.empty(16, 1, 4, 64, dtype=torch.float32, device=DEV)
    cand = torch.empty(16, 8192, dtype=torch.int32, device=DEV)
    idx = torch.empty(16, 4, 2048, dtype=torch.int32, device=DEV)
    st = li.li_hs_select_noalloc(lat, sc, qa, qs, wt, 8192, 2048, cand, idx)
    assert st == -4            # LI_ERR_WORKSPACE, reported before anything runs
