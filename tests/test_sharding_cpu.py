"""Multi-process (gloo, world_size 2, CPU) test of the row-sharded path:
each rank verifies its contiguous share of the rows with the global row
numbers, then shifts its packed-token offsets by the lower ranks' totals;
the concatenation equals the unsplit batch.  The CPU oracle stands in for
the per-device verify."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_logits_gb300.sharding import global_offsets, shard_rows


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, path):
    import oracle
    import sd_workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = W.synth(7, 3, 301, "bf16", kind="normal", temperature=[0, 0.7, 1, 1.3, 0.9, 0, 1],
                  seed=5)
    base, n = shard_rows(inp.B, world, rank)
    sl = slice(base, base + n)
    r = oracle.verify(W.to_numpy_logits(inp.target[sl]), W.to_numpy_logits(inp.draft[sl]),
                      inp.tokens[sl].numpy(), inp.temperature[sl].numpy(), inp.seed,
                      row_base=base)
    offs, packed = oracle.compact(r["out_tokens"], r["tau"])
    goffs, total = global_offsets(torch.from_numpy(offs))
    np.savez(f"{path}/rank{rank}.npz", out=r["out_tokens"], offs=goffs.numpy(), packed=packed,
             total=total, base=base)
    dist.barrier()
    dist.destroy_process_group()


def test_shard_rows_partition():
    for B in (0, 1, 7, 256):
        for world in (1, 2, 3, 8):
            spans = [shard_rows(B, world, r) for r in range(world)]
            assert sum(n for _, n in spans) == B
            assert all(spans[i][0] + spans[i][1] == spans[i + 1][0] for i in range(world - 1))


def test_two_rank_gloo_sharding_matches_unsplit(tmp_path, oracle_lib):
    import sd_workloads as W
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    inp = W.synth(7, 3, 301, "bf16", kind="normal", temperature=[0, 0.7, 1, 1.3, 0.9, 0, 1],
                  seed=5)
    full = oracle_lib.verify(W.to_numpy_logits(inp.target), W.to_numpy_logits(inp.draft),
                             inp.tokens.numpy(), inp.temperature.numpy(), inp.seed)
    offs, packed = oracle_lib.compact(full["out_tokens"], full["tau"])
    np.testing.assert_array_equal(np.concatenate([p["out"] for p in parts]), full["out_tokens"])
    g_offs = np.concatenate([parts[0]["offs"][:-1], parts[1]["offs"]])
    np.testing.assert_array_equal(g_offs, offs)
    np.testing.assert_array_equal(np.concatenate([p["packed"] for p in parts]), packed)
    assert all(int(p["total"]) == offs[-1] for p in parts)
