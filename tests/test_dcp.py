"""Decode context parallelism: shard construction, the rank-major gather of
the per-rank candidates (2 gloo ranks on CPU), and, on the GPU, the sharded
step emulated on one device (every rank's logits and top-k on its shard,
then the pack and merge kernels) against the unsharded step and the oracle."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W

MIXED = dict(request_lens=[300, 517, 70, 1000, 129], rows_per_request=[1, 3, 2, 2, 5])


# ---------------------------------------------------------------------------
# CPU
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kv_format", [W.KV_FP8, W.KV_FP4, W.KV_MXFP4])
def test_shard_holds_the_ranks_tokens(kv_format):
    wl = W.build("dcp", **MIXED, kv_format=kv_format, topk=32, seed=3)
    src = W._page_views(wl.kv_cache, kv_format)
    ctx = wl.context_lens.numpy()
    for world, inter in ((2, 1), (3, 64), (4, 7)):
        for r in range(world):
            sh = W.dcp_shard(wl, r, world, inter)
            dst = W._page_views(sh.kv_cache, kv_format)
            for t in range(wl.num_rows):
                n = int(sh.context_lens[t])
                assert n == oracle.dcp_local_len(int(ctx[t]), r, world, inter)
                local = torch.arange(n)
                g = torch.tensor([oracle.dcp_global_id(l, r, world, inter) for l in range(n)], dtype=torch.int64)
                gp, gs = wl.block_table[t].long()[g // 64], g % 64
                lp, ls = sh.block_table[t].long()[local // 64], local % 64
                for key in src:
                    assert torch.equal(src[key][gp, gs], dst[key][lp, ls]), (world, inter, r, t, key)


def test_oracle_logits_of_a_shard_are_the_global_columns():
    wl = W.build("dcp", **MIXED, topk=32, seed=4)
    glob, _ = oracle.workload_logits(wl)
    ctx = wl.context_lens.numpy()
    for world, inter in ((2, 1), (3, 5)):
        for r in range(world):
            sh = W.dcp_shard(wl, r, world, inter)
            loc, _ = oracle.workload_logits(sh)
            for t in range(wl.num_rows):
                n = oracle.dcp_local_len(int(ctx[t]), r, world, inter)
                cols = [oracle.dcp_global_id(l, r, world, inter) for l in range(n)]
                assert np.array_equal(loc[t, :n], glob[t, cols])


def _gather_worker(rank, world, port, rows, k, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(7)
        sc = np.round(rng.standard_normal((rows, 211)) * 2) / 2   # the same rows on every rank, many ties
        ends = np.array([211, 150, 3][:rows], dtype=np.int32)
        inter = 3
        packs = []
        for r in range(world):                                     # every rank's pack, computed locally
            cols = [g for g in range(sc.shape[1]) if (g // inter) % world == r]
            loc = sc[:, cols]
            loc_ends = np.array([sum(1 for g in cols if g < e) for e in ends], dtype=np.int32)
            lidx = oracle.top_k_per_row(loc, loc_ends, k)
            packs.append(torch.from_numpy(oracle.dcp_pack(loc, lidx, k, r, world, inter)).float())
        gathered = dsa.dcp_gather_candidates(packs[rank], world)
        rank_major = torch.equal(gathered, torch.stack(packs))
        merged = oracle.dcp_merge(gathered.double().numpy(), k)
        want = oracle.top_k_per_row(sc, ends, k)
        q.put((rank, bool(rank_major), bool(np.array_equal(merged, want))))
    finally:
        torch.distributed.destroy_process_group()


def test_gather_is_rank_major_and_merge_is_exact_gloo():
    world, port = 2, 29513
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, 3, 16, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rank_major, merge_ok in res:
        assert rank_major, f"rank {rank}: the gather is not rank-major"
        assert merge_ok, f"rank {rank}: the merge differs from the global top-k"


# ---------------------------------------------------------------------------
# GPU (one device emulates the ranks)
# ---------------------------------------------------------------------------

def _emulated(wl, world, inter):
    from gpu_helpers import run_path
    glob = run_path(wl)
    assert int(glob["status"].item()) == 0
    packs, locs = [], []
    for r in range(world):
        out = run_path(W.dcp_shard(wl, r, world, inter))
        assert int(out["status"].item()) == 0
        packs.append(dsa.dcp_pack_topk(out["logits"], out["idx"], wl.topk, r, world, inter))
        locs.append(out)
    gathered = torch.stack(packs).contiguous()
    merged = dsa.dcp_merge_topk(gathered, wl.topk)
    torch.cuda.synchronize()
    return glob, locs, gathered, merged


@pytest.mark.gpu
@pytest.mark.parametrize("world,inter", [(2, 1), (3, 64), (4, 7), (8, 1)])
def test_dcp_emulated_equals_unsharded_step(world, inter):
    wl = W.build("dcp", **MIXED, topk=64, seed=11)
    glob, locs, gathered, merged = _emulated(wl, world, inter)
    # exact: every rank computes the same logit for a (row, token) as the unsharded step
    assert torch.equal(merged.cpu(), glob["idx"].cpu())
    # the merge kernel agrees with the oracle merge of the same packs
    want = oracle.dcp_merge(gathered.cpu().double().numpy(), wl.topk)
    assert np.array_equal(merged.cpu().numpy(), want)
    # the pack kernel agrees with the oracle pack of the same local logits and indices
    for r, out in enumerate(locs):
        ref = oracle.dcp_pack(out["logits"].float().cpu().double().numpy(), out["idx"].cpu().numpy(),
                              wl.topk, r, world, inter)
        assert np.array_equal(gathered[r].cpu().double().numpy(), ref)


@pytest.mark.gpu
@pytest.mark.parametrize("kv_format", [W.KV_FP4, W.KV_MXFP4])
def test_dcp_emulated_fp4_bf16_logits(kv_format):
    wl = W.build("dcp", **MIXED, kv_format=kv_format, logits_dtype=W.LOGITS_BF16, topk=48, seed=12)
    glob, _, gathered, merged = _emulated(wl, 3, 2)
    assert torch.equal(merged.cpu(), glob["idx"].cpu())
    assert np.array_equal(merged.cpu().numpy(), oracle.dcp_merge(gathered.cpu().double().numpy(), wl.topk))


def _synthetic_gathered(world, rows, k, order, seed, id_range=None):
    """[world, rows, k, 2] candidates with heavy score ties, NaN scores, padded
    slots, a row with fewer than k candidates and an all-padded row.  `order`
    "ascending" keeps every rank's valid candidates first and in ascending id
    order (the order the top-k and pack calls produce); "random" does not."""
    rng = np.random.default_rng(seed)
    g = np.zeros((world, rows, k, 2))
    span = world * rows * k * 3 if id_range is None else id_range
    ids = rng.choice(span, size=world * rows * k, replace=False).reshape(world, rows, k)
    g[..., 0] = rng.integers(0, 4, size=(world, rows, k)) / 2.0
    g[..., 1] = ids
    g[min(1, world - 1), 0, ::3, 0] = np.nan
    g[world - 1, 1, 5:, :] = (-np.inf, -1.0)
    g[:, 3, 2:, :] = (-np.inf, -1.0)
    g[:, 4, :, :] = (-np.inf, -1.0)
    g[0, 2, :, 0] = -0.0
    if order == "ascending":
        for r in range(world):
            for t in range(rows):
                valid = g[r, t, g[r, t, :, 1] >= 0]
                valid = valid[np.argsort(valid[:, 1])]
                g[r, t, : len(valid)] = valid
                g[r, t, len(valid):] = (-np.inf, -1.0)
    return g


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["ascending", "random"])
@pytest.mark.parametrize("world,k", [(1, 40), (3, 40), (8, 2048), (5, 1), (2, 777)])
def test_dcp_merge_ties_nan_and_padding(world, k, order):
    g = _synthetic_gathered(world, 6, k, order, seed=world * 31 + k)
    gathered = torch.from_numpy(g).float().cuda().contiguous()
    merged = dsa.dcp_merge_topk(gathered, k)
    torch.cuda.synchronize()
    assert np.array_equal(merged.cpu().numpy(), oracle.dcp_merge(g, k))


@pytest.mark.gpu
def test_dcp_merge_ids_across_the_whole_fp32_exact_range():
    # ids up to 2^24 - 1: the merge's id bitmap covers them in several chunks
    g = _synthetic_gathered(4, 6, 512, "random", seed=9, id_range=(1 << 24))
    g[0, 0, 0, 1] = (1 << 24) - 1
    g[1, 0, 0, 1] = 0
    gathered = torch.from_numpy(g).float().cuda().contiguous()
    merged = dsa.dcp_merge_topk(gathered, 512)
    torch.cuda.synchronize()
    assert np.array_equal(merged.cpu().numpy(), oracle.dcp_merge(g, 512))


@pytest.mark.gpu
def test_dcp_merge_pad_between_candidates():
    g = _synthetic_gathered(3, 6, 64, "ascending", seed=5)
    g[1, 0, 10] = (-np.inf, -1.0)            # a padded slot before valid ones
    g[2, 2, [3, 4]] = g[2, 2, [4, 3]]         # two ids out of order
    gathered = torch.from_numpy(g).float().cuda().contiguous()
    merged = dsa.dcp_merge_topk(gathered, 64)
    torch.cuda.synchronize()
    assert np.array_equal(merged.cpu().numpy(), oracle.dcp_merge(g, 64))


@pytest.mark.gpu
def test_dcp_topk_single_rank_is_the_local_topk():
    from gpu_helpers import run_path
    wl = W.build("dcp", **MIXED, topk=64, seed=13)
    out = run_path(wl)
    merged = dsa.dcp_topk(out["logits"], out["idx"], wl.topk, 0, 1, 1)
    torch.cuda.synchronize()
    assert torch.equal(merged.cpu(), out["idx"].cpu())
