"""The multi-GPU path's host logic, on CPU processes with the gloo backend.

Tokens are independent at tp = 1, so a batch shards by contiguous row blocks
with no collective on the data path; each process writes its own tokens into its
own KV-cache replica.  Two gloo ranks check, with the oracle standing in for each
rank's device work, that: the row blocks cover every row once; the projection
rows of the two shards, put side by side, are the unsharded result exactly; the
two cache replicas, merged on the slots each one wrote, are the unsharded
caches exactly; and the timing reduction gives every rank the slowest rank's
time, from which the whole-job rate is computed.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist_pg
import torch.multiprocessing as mp

import oracle
from rope_attention_gb300 import dist, synth

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gather(x: np.ndarray) -> list:
    t = torch.from_numpy(np.ascontiguousarray(x))
    out = [torch.empty_like(t) for _ in range(WORLD)]
    dist_pg.all_gather(out, t)
    return [o.numpy() for o in out]


def _worker(rank: int, port: int, errq):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(WORLD),
                          RANK=str(rank), LOCAL_RANK=str(rank))
        dist_pg.init_process_group("gloo", rank=rank, world_size=WORLD)
        e = dist.env()
        assert (e.world, e.rank) == (WORLD, rank)

        # projection: each rank computes its contiguous block of token rows
        c = synth.make_qkv("mp", 5, S=37, H=256, num_heads=2, num_kv_heads=2, head_dim=64)
        b, en = dist.shard_rows(c.T, WORLD, rank)
        sel = np.arange(b, en)
        mine = oracle.qkv_cte_mx(c.a[sel], c.a_scale[sel], c.w, c.w_block_exp, num_heads=c.num_heads,
                                 num_kv_heads=c.num_kv_heads, head_dim=c.head_dim, bias=c.bias,
                                 q_gamma=c.q_gamma, k_gamma=c.k_gamma, eps=c.eps, fused_rope=True,
                                 cos=c.cos[sel], sin=c.sin[sel])
        width = max(dist.shard_rows(c.T, WORLD, r)[1] - dist.shard_rows(c.T, WORLD, r)[0] for r in range(WORLD))
        padded = np.zeros((width, c.I))
        padded[: en - b] = mine
        parts = _gather(padded)
        got = np.concatenate([parts[r][: dist.shard_rows(c.T, WORLD, r)[1] - dist.shard_rows(c.T, WORLD, r)[0]]
                              for r in range(WORLD)])
        full = oracle.qkv_cte_mx(c.a, c.a_scale, c.w, c.w_block_exp, num_heads=c.num_heads,
                                 num_kv_heads=c.num_kv_heads, head_dim=c.head_dim, bias=c.bias,
                                 q_gamma=c.q_gamma, k_gamma=c.k_gamma, eps=c.eps, fused_rope=True,
                                 cos=c.cos, sin=c.sin)
        assert np.array_equal(got, full)

        # KV cache: each rank scatters its batches' tokens into its own cache replica
        k = synth.make_kv("mp", 6, variant=2, B=4, N=2, S=9, Dkv=64, Dv=32, rope_size=16,
                          block_size=32, block_num=2, quant_k=True, quant_v=True, skip_frac=0.2)
        kb, ke = dist.shard_rows(k.B, WORLD, rank)
        assert ke > kb
        kw = dict(variant=2, rope_size=k.rope_size, block_size=k.block_size, cache_mode=k.cache_mode,
                  epsilon=k.eps, k_scale=k.k_scale, k_offset=k.k_offset, v_scale=k.v_scale,
                  v_offset=k.v_offset, is_output_kv=False)
        r = oracle.kv_rms_norm_rope_cache(k.kv[kb:ke], k.gamma, k.cos[kb:ke], k.sin[kb:ke],
                                          k.index[kb * k.S: ke * k.S], k.k_cache.copy(), k.ckv_cache.copy(),
                                          v=k.v[kb:ke], **kw)
        full = oracle.kv_rms_norm_rope_cache(k.kv, k.gamma, k.cos, k.sin, k.index, k.k_cache.copy(),
                                             k.ckv_cache.copy(), v=k.v, **kw)
        merged = {}
        for name, mask in (("k_cache", "k_written"), ("ckv_cache", "ckv_written")):
            caches, masks = _gather(r[name]), _gather(r[mask].astype(np.uint8))
            assert not np.any(np.logical_and(masks[0], masks[1])), "replicas wrote the same slot"
            m = getattr(k, name).copy()
            for rr in range(WORLD):
                m[masks[rr].astype(bool)] = caches[rr][masks[rr].astype(bool)]
            merged[name] = m
            assert np.array_equal(m, full[name]), name

        # timing: every rank learns the slowest rank's time; the job rate uses it
        slowest = dist.max_over_ranks(1.0 + rank)
        assert slowest == 1.0 + (WORLD - 1)
        assert dist.job_rate(100.0, WORLD, slowest) == 100.0 * WORLD / slowest
        dist_pg.barrier()
        dist_pg.destroy_process_group()
    except BaseException as ex:  # report to the parent, which fails the test
        errq.put(f"rank {rank}: {type(ex).__name__}: {ex}")
        raise


def test_shard_rows_cover_each_row_once():
    for total in (0, 1, 7, 32760, 75600):
        for world in (1, 2, 3, 8):
            blocks = [dist.shard_rows(total, world, r) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == total
            assert all(blocks[i][1] == blocks[i + 1][0] for i in range(world - 1))
            sizes = [e - b for b, e in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        dist.shard_rows(10, 2, 2)


def test_two_gloo_ranks_match_the_unsharded_result():
    ctx = mp.get_context("spawn")
    errq = ctx.SimpleQueue()
    mp.start_processes(_worker, args=(_free_port(), errq), nprocs=WORLD, join=True, start_method="spawn")
    assert errq.empty(), errq.get()
