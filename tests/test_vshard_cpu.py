"""Multi-process (gloo, world_size 2, CPU) test of the vocabulary-sharded
verify's exchanges: each rank holds half of the vocabulary's columns; the
stats and mass blocks are all-gathered in rank order and the outputs
all-reduced with a maximum.  The per-shard kernels need a GPU, so here the
three phases are stand-ins built on the CPU oracle that keep the kernels'
contract (a stats block per shard, a mass block per shard, outputs written
everywhere except a sampled row's token and hit flag, which only the shard
owning the token writes); the test checks that the exchanges put every
rank's blocks in place and that every rank ends with the unsharded result."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_logits_gb300 import verify_vsharded_dist, vshard_bounds

B, K, V = 6, 3, 401
TEMPS = [0.0, 0.7, 1.0, 1.3, 0.0, 0.9]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    import sd_workloads as W
    return W.synth(B, K, V, "f32", kind="normal", temperature=TEMPS, seed=17)


def _phases(rank, world, full):
    """Stand-ins for sd_vshard_stats / _mass / _pick on this rank's columns,
    checking what the exchanges handed them."""
    v0, vs = vshard_bounds(V, world)[rank]

    def stats(t, d, tok, temp, seed, *, S, shard, **kw):
        assert (S, shard) == (world, rank)
        blk = torch.full((64,), 0, dtype=torch.uint8)
        blk[0] = shard + 1
        blk[1:9] = torch.frombuffer(bytearray(np.int64(kw["v0"]).tobytes()), dtype=torch.uint8)
        return blk

    def mass(t, d, tok, temp, seed, stats_all, *, S, shard, **kw):
        blocks = stats_all.view(S, 64)
        for s_ in range(S):   # every shard's block, in rank order
            assert int(blocks[s_, 0]) == s_ + 1
            assert np.frombuffer(blocks[s_, 1:9].numpy().tobytes(), np.int64)[0] == \
                vshard_bounds(V, S)[s_][0]
        return torch.full((B * 32,), shard + 1, dtype=torch.uint8)

    def pick(t, d, tok, temp, seed, stats_all, mass_all, out, *, S, shard, **kw):
        assert [int(mass_all[s_ * B * 32]) for s_ in range(S)] == list(range(1, S + 1))
        for b in range(B):
            m = int(full["num_accepted"][b])
            token = int(full["out_tokens"][b, m])
            owner = next(s_ for s_, (a, n) in enumerate(vshard_bounds(V, S)) if a <= token < a + n)
            out.num_accepted[b] = m
            out.tau[b] = m + 1
            out.out_tokens[b, :m] = torch.from_numpy(full["out_tokens"][b, :m])
            if TEMPS[b] == 0 or owner == shard:   # a sampled row's token: its owner only
                out.out_tokens[b, m] = token
                out.hit[b] = 1 if b % 2 else 0
        return out

    return (stats, mass, pick), v0, vs


def _worker(rank, world, port, path):
    import oracle
    import sd_workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = _inputs()
    full = oracle.verify(W.to_numpy_logits(inp.target), W.to_numpy_logits(inp.draft),
                         inp.tokens.numpy(), inp.temperature.numpy(), inp.seed)
    phases, v0, vs = _phases(rank, world, full)
    t = inp.target[:, :, v0:v0 + vs].contiguous()
    d = inp.draft[:, :, v0:v0 + vs].contiguous()
    r = verify_vsharded_dist(t, d, inp.tokens, inp.temperature, inp.seed, V=V, v0=v0,
                             phases=phases)
    np.savez(f"{path}/rank{rank}.npz", out=r.out_tokens.numpy(), tau=r.tau.numpy(),
             hit=r.hit.numpy(), ref=full["out_tokens"], ref_tau=full["tau"])
    dist.barrier()
    dist.destroy_process_group()


def test_vshard_bounds_cover_the_vocabulary():
    for V_, S in ((401, 2), (128256, 4), (151936, 3), (7, 7)):
        b = vshard_bounds(V_, S)
        assert b[0][0] == 0 and sum(n for _, n in b) == V_
        assert all(b[i][0] + b[i][1] == b[i + 1][0] for i in range(S - 1))
        assert max(n for _, n in b) - min(n for _, n in b) <= 1


def test_two_rank_gloo_vshard_exchanges(tmp_path, oracle_lib):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    for p in parts:   # every rank holds the unsharded result after the exchanges
        np.testing.assert_array_equal(p["out"], p["ref"])
        np.testing.assert_array_equal(p["tau"], p["ref_tau"])
        np.testing.assert_array_equal(p["hit"], np.arange(B) % 2)
    np.testing.assert_array_equal(parts[0]["out"], parts[1]["out"])
