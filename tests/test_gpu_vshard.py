"""The vocabulary-sharded verify on one GPU (S shards' column blocks, the
exchanges as blocks laid side by side) against the CPU oracle on the
unsharded logits: exact outside the guard band, keys exact, over every row,
at S = 2 and 4 on the peaked and zipf workloads and on small shapes whose
shards start off the 16-byte grid."""
import numpy as np
import pytest
import torch

import oracle
import sd_workloads as W
from tests.parity import compare_verify

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_logits_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oracle.build()
    return torch.device("cuda:0")


def _split(x, bounds):
    return [x[..., a:a + n].contiguous() for a, n in bounds] if x is not None else None


def _run(inp, S, fan=None, check_finite=False):
    bounds = sd.vshard_bounds(inp.V, S)
    return sd.verify_vsharded(_split(inp.target, bounds), _split(inp.draft, bounds), inp.tokens,
                              inp.temperature, inp.seed, V=inp.V, fanout=fan,
                              draft_bonus=_split(inp.draft_bonus, bounds) if fan else None,
                              check_finite=check_finite)


def _np(t):
    return W.to_numpy_logits(t)


def _check_against_oracle(inp, r, fan=None):
    keys = None
    if fan is not None:
        keys = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus) if inp.draft_bonus is not None else None)
        np.testing.assert_array_equal(r.keys.cpu().numpy(), keys)
    o = oracle.verify(_np(inp.target), _np(inp.draft), inp.tokens.cpu().numpy(),
                      inp.temperature.cpu().numpy(), inp.seed, keys=keys)
    stats, bad = compare_verify(r, o, inp.temperature.cpu().numpy(), check_stats=False)
    assert not bad, bad[:5]
    assert stats["mismatch_outside_guard"] == 0
    if fan is None:   # without keys there is no hit test: hit stays 0
        assert not r.hit.any()
    return stats


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("name", ["peaked", "zipf"])
def test_workload_sharded_matches_oracle(dev, name, S):
    for rd in (0, 1):
        inp = W.workload(name, round_idx=10 + rd, device=dev)
        r = _run(inp, S)
        torch.cuda.synchronize()
        _check_against_oracle(inp, r)
        assert int(r.status.item()) == 0


@pytest.mark.parametrize("S", [2, 3, 4])
def test_saguaro_keys_and_hits_sharded(dev, S):
    inp = W.workload("saguaro", round_idx=7, device=dev)
    fan = W.WORKLOADS["saguaro"]["fanout"]
    r = _run(inp, S, fan)
    torch.cuda.synchronize()
    _check_against_oracle(inp, r, fan)
    # the same outputs as the unsharded verify
    u = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), u.keys.cpu().numpy())


@pytest.mark.parametrize("B,K,V,dt,S", [(5, 4, 20011, "bf16", 3), (4, 3, 9001, "f32", 4),
                                        (3, 6, 77, "bf16", 5), (3, 0, 1001, "bf16", 2),
                                        (6, 5, 50021, "bf16", 7)])
def test_small_shapes_sharded(dev, B, K, V, dt, S):
    # odd shard widths: every shard but the first starts off the 16-byte grid
    temps = [0.0, 0.8, 1.3, 0.6, 0.0, 1.0][:B]
    fan = [2] * K + [1]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=5,
                  temperature=temps, seed=B * 100 + V + S, device=dev, bonus_row=True)
    r = _run(inp, S, fan)
    torch.cuda.synchronize()
    _check_against_oracle(inp, r, fan)


def test_sharded_check_finite_and_invalid_rows(dev):
    B, K, V, S = 6, 3, 4001, 3
    inp = W.synth(B, K, V, "f32", kind="normal", temperature=[1.0, 0.0, 0.7, 1.0, -1.0, 0.9],
                  seed=44, device=dev)
    inp.target[0, 1, 2100] = float("nan")      # a NaN in the second shard
    inp.draft[2, 0, 5] = float("inf")         # +inf in the first shard's draft row
    inp.tokens[3, 1] = V + 3                  # a token outside the vocabulary
    r = _run(inp, S, check_finite=True)
    torch.cuda.synchronize()
    tau = r.tau.cpu().numpy()
    assert list(np.nonzero(tau == 0)[0]) == [0, 2, 3, 4]
    st = int(r.status.item())
    assert st & sd.SD_STATUS_NONFINITE and st & sd.SD_STATUS_BAD_TOKEN and st & sd.SD_STATUS_BAD_TEMP
    o = oracle.verify(_np(inp.target), _np(inp.draft), inp.tokens.cpu().numpy(),
                      inp.temperature.cpu().numpy(), inp.seed, check_finite=True)
    np.testing.assert_array_equal(tau, o["tau"])
    for b in (1, 5):
        if o["guard_pos"][b] < 0:
            np.testing.assert_array_equal(r.out_tokens.cpu().numpy()[b], o["out_tokens"][b])
