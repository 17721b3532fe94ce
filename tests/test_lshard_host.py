"""The L-sharded exchange protocol (shared_latent_key_cache_b300.lshard) on
two gloo ranks on CPU: each rank takes the oracle's top-k of its shard of
every score row, the ranks all-gather the (score, global position) lists and
merge them with the oracle's top-k (ties to the lower position); the merged
set must equal the one-pass oracle set, with ties across shards.  The module
is pure bookkeeping, so it is imported by path without loading the CUDA
library."""
import importlib.util
import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lshard():
    spec = importlib.util.spec_from_file_location(
        "li_lshard", os.path.join(ROOT, "shared_latent_key_cache_b300", "lshard.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rows():
    g = torch.Generator().manual_seed(71)
    L = 1000
    return L, [torch.randint(0, 5, (L,), generator=g).double(),          # heavy ties everywhere
               torch.randn(L, generator=g, dtype=torch.float64),
               torch.full((L,), 3.0, dtype=torch.float64),               # all equal
               torch.cat([torch.full((500,), 1.0), torch.full((500,), 2.0)]).double()]


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    ls = _lshard()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        L, rows = _rows()
        out = []
        for k in (1, 17, 256, 500):
            ls.check_shards(L, ws, k)
            a, b = ls.shard_range(L, ws, rank)
            for s in rows:
                li, lv = oracle.topk(s[a:b].numpy()[None], k)              # this rank's shard
                pos = ls.to_global(torch.from_numpy(li[0]).long(), a)
                cv, cp = ls.gather_candidates(torch.from_numpy(lv[0]), pos)
                order = torch.argsort(cp, stable=True)                      # position order, so the
                cv, cp = cv[order], cp[order]                               # merge's ties go by position
                j, _ = oracle.topk(cv.numpy()[None], k)
                out.append(sorted(cp[torch.from_numpy(j[0]).long()].tolist()))
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_rank_shard_exchange_merge_equals_one_pass(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29300 + os.getpid() % 150
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    L, rows = _rows()
    want = []
    for k in (1, 17, 256, 500):
        for s in rows:
            i, _ = orc.topk(s.numpy()[None], k)
            want.append(sorted(i[0].tolist()))
    assert got[0] == want and got[1] == want


def test_shard_ranges_cover_the_row_in_order():
    ls = _lshard()
    for L, world in ((1000, 2), (131072, 8), (10, 3), (7, 7)):
        spans = [ls.shard_range(L, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == L
        assert all(spans[r][1] == spans[r + 1][0] for r in range(world - 1))
        sizes = [b - a for a, b in spans]
        assert max(sizes) - min(sizes) <= 1


def test_short_shards_are_rejected():
    ls = _lshard()
    with pytest.raises(ValueError):
        ls.check_shards(1000, 8, 256)
    with pytest.raises(ValueError):
        ls.to_global(torch.tensor([3, -1]), 100)
