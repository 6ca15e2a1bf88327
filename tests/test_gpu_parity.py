"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small shapes that span several CTA slices and ragged tails are compared in
full; the five workloads at full size are compared on sampled rows (rows
are independent, so the oracle recomputes a row alone with its global row
number), in the launch configuration the benchmark uses.
"""
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


@pytest.fixture(params=["split", "cluster"])
def path(request, monkeypatch):
    """Both launch paths: the flat streaming grid + per-sequence finish (the
    default when scratch is given), and the single cluster kernel."""
    monkeypatch.setenv("SDV_SPLIT", "1" if request.param == "split" else "0")
    return request.param


def _np(t):
    return W.to_numpy_logits(t)


def _oracle_for(inp, rows=None, keys=None):
    t, d = inp.target, inp.draft
    tok, temps = inp.tokens, inp.temperature
    if rows is None:
        return oracle.verify(_np(t), _np(d), tok.cpu().numpy(), temps.cpu().numpy(), inp.seed,
                             keys=keys, stats=True)
    outs = []
    for b in rows:
        k = None if keys is None else keys[b:b + 1]
        outs.append(oracle.verify(_np(t[b:b + 1]), _np(d[b:b + 1]), tok[b:b + 1].cpu().numpy(),
                                  temps[b:b + 1].cpu().numpy(), inp.seed, row_base=int(b),
                                  keys=k, stats=True))
    return {k: np.concatenate([o[k] for o in outs]) if isinstance(outs[0][k], np.ndarray)
            else sum(o[k] for o in outs) for k in outs[0]}


def _check(stats, bad):
    assert not bad, bad[:10]
    assert stats["mismatch_outside_guard"] == 0


# ----------------------------------------------------------------- uniforms --
def test_uniforms_bit_exact_with_oracle(dev):
    rng = np.random.default_rng(1)
    n = 4096
    row = torch.from_numpy(rng.integers(0, 2 ** 31 - 1, n).astype(np.int32)).to(dev)
    pos = torch.from_numpy(rng.integers(0, 33, n).astype(np.int32)).to(dev)
    slot = torch.from_numpy(rng.integers(0, 2, n).astype(np.int32)).to(dev)
    for seed in (0, 1234, 2 ** 63 + 12345, 0xFFFFFFFFFFFFFFFF):
        u = sd.uniforms(seed, row, pos, slot).cpu().numpy()
        ro, po, so = row.cpu().numpy(), pos.cpu().numpy(), slot.cpu().numpy()
        ref = np.array([oracle.uniform(seed, int(ro[i]), int(po[i]), int(so[i])) for i in range(n)])
        np.testing.assert_array_equal(u, ref)


# ----------------------------------------------------------- worked example --
def test_worked_example_greedy(dev):
    from tests.test_oracle_pins import _worked_example_inputs
    g, ids, target, draftl, tokens = _worked_example_inputs()
    K = tokens.size
    r = sd.verify(torch.from_numpy(target[None]).to(dev), torch.from_numpy(draftl[None]).to(dev),
                  torch.from_numpy(tokens[None]).to(dev), torch.zeros(1, device=dev), seed=1,
                  compact=True)
    assert int(r.num_accepted[0]) == int(g["expect_n_accepted"][0])
    assert int(r.tau[0]) == int(g["expect_tau"][0])
    assert r.packed[: int(r.offsets[1])].tolist() == [ids[w] for w in g["expect_packed"]]
    assert r.out_tokens[0, K - 1].item() == -1


# ------------------------------------------------- small shapes, full compare --
SHAPES = [
    # (B, K, V, dtype)
    (3, 4, 1000, "f32"),
    (4, 3, 4099, "bf16"),      # odd V: rows start off the 16-byte grid
    (5, 5, 20000, "bf16"),
    (2, 2, 32001, "f32"),
    (3, 6, 1, "bf16"),         # one-token vocabulary
    (4, 2, 17, "f32"),
    (2, 0, 777, "bf16"),       # K = 0: a plain sampling step
    (6, 8, 151936, "bf16"),    # largest vocabulary of the workloads
]


@pytest.mark.parametrize("B,K,V,dt", SHAPES)
@pytest.mark.parametrize("kind", ["normal", "peaked"])
def test_small_shapes_full_parity(dev, path, B, K, V, dt, kind):
    temps = [0.0, 0.6, 1.0, 1.7, 0.3, 1.0][:B]
    inp = W.synth(B, K, V, dt, kind=kind, sigma=2.0, draft_sigma=0.7, peaks=3 if V > 8 else 0,
                  temperature=temps, seed=B * 1000 + K * 10 + V, device=dev)
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, stats=True,
                  compact=True)
    torch.cuda.synchronize()
    o = _oracle_for(inp)
    stats, bad = compare_verify(r, o, temps)
    _check(stats, bad)
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.offsets.cpu().numpy(), offs)
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)
    assert int(r.status.item()) == 0


def test_zipf_and_ties_and_neg_inf(dev, path):
    B, K, V = 4, 3, 3001
    inp = W.synth(B, K, V, "bf16", kind="zipf", temperature=[1.0, 0.0, 0.6, 1.0], seed=77,
                  device=dev)
    # ties and -inf logits: quantise some rows and knock out a block of tokens
    t = inp.target.float()
    t[1] = torch.round(t[1] * 2) / 2
    t[2, :, 100:400] = float("-inf")
    inp.target = t.to(torch.bfloat16).contiguous()
    d = inp.draft.float()
    d[2, :, 500:700] = float("-inf")
    inp.draft = d.to(torch.bfloat16).contiguous()
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, stats=True)
    o = _oracle_for(inp)
    _check(*compare_verify(r, o, inp.temperature.cpu().numpy()))


# ------------------------------------------------------ outcome prediction ----
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_outcome_keys_standalone_and_fused(dev, path, dt):
    B, K, V = 5, 6, 12007
    fan = [4, 3, 2, 1, 1, 1, 1]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=20,
                  temperature=[0.7, 0.0, 1.0, 0.7, 0.7], seed=5, device=dev, bonus_row=True)
    # ties in the draft logits of one row
    d = inp.draft.float()
    d[3] = torch.round(d[3])
    inp.draft = d.to(inp.target.dtype).contiguous()
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    keys = sd.outcome_predict(inp.draft, inp.tokens, fan, inp.draft_bonus)
    np.testing.assert_array_equal(keys.cpu().numpy(), keys_ref)
    keys_nb = sd.outcome_predict(inp.draft, inp.tokens, fan, None)
    np.testing.assert_array_equal(
        keys_nb.cpu().numpy(), oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan))
    # fused into the verify pass, and the hit test on both paths
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    r2 = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, cache_keys=keys)
    o = _oracle_for(inp, keys=keys_ref)
    _check(*compare_verify(r, o, inp.temperature.cpu().numpy()))
    _check(*compare_verify(r2, o, inp.temperature.cpu().numpy(), check_stats=False))


@pytest.mark.parametrize("cs", [1, 3, 7, 16])
def test_forced_cluster_sizes(dev, path, cs, monkeypatch):
    # every cluster size streams the same rows: slices off the 16-byte grid
    # (odd V, bf16), fan-outs up to the largest key count, greedy and sampled;
    # on the split path the size is the finish's (the draw's slices)
    monkeypatch.setenv("SDV_CS", str(cs))
    B, K, V = 3, 5, 50021
    fan = [8, 2, 1, 0, 3, 1]
    temps = [0.7, 0.0, 1.3]
    inp = W.synth(B, K, V, "bf16", kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=20,
                  temperature=temps, seed=40 + cs, device=dev, bonus_row=True)
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True, compact=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    o = _oracle_for(inp, keys=keys_ref)
    _check(*compare_verify(r, o, temps))
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.offsets.cpu().numpy(), offs)
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)


@pytest.mark.parametrize("rs,cs,V,dt", [(0, 5, 50021, "bf16"), (1, 5, 50021, "bf16"),
                                        (1, 2, 50021, "f32"), (1, 16, 3001, "bf16"),
                                        (1, 16, 3001, "f32"), (1, 7, 131072, "bf16")])
def test_stream_split_modes(dev, rs, cs, V, dt, monkeypatch):
    # both ways of dividing a sequence's rows among the cluster's CTAs: a
    # vocabulary slice of every row, or row pieces cut at whole streaming
    # steps (pieces that start mid-row, rows off the 16-byte grid for odd V,
    # and CTAs left with no piece at all when the rows hold fewer steps than
    # the cluster has CTAs)
    monkeypatch.setenv("SDV_SPLIT", "0")
    monkeypatch.setenv("SDV_CS", str(cs))
    monkeypatch.setenv("SDV_ROWSPLIT", str(rs))
    B, K = 3, 5
    fan = [4, 3, 2, 1, 1, 2]
    temps = [0.9, 0.0, 0.6]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=20,
                  temperature=temps, seed=70 + cs + rs, device=dev, bonus_row=True)
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True, compact=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    o = _oracle_for(inp, keys=keys_ref)
    _check(*compare_verify(r, o, temps))
    # the same without keys: greedy rows stream the target only
    r2 = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, stats=True)
    _check(*compare_verify(r2, _oracle_for(inp), temps))


@pytest.mark.parametrize("G,V,dt", [(1, 50021, "bf16"), (5, 50021, "bf16"), (37, 50021, "f32"),
                                    (300, 50021, "bf16"), (64, 3001, "bf16"),
                                    (300, 131072, "f32")])
def test_split_grid_sizes(dev, G, V, dt, monkeypatch):
    # the flat streaming grid at several sizes: one CTA streaming every row,
    # ranges that cut rows at arbitrary steps, rows spread over many CTAs
    # (up to the limit of pieces per row), rows of a single step (V = 3001)
    monkeypatch.setenv("SDV_SPLIT", "1")
    monkeypatch.setenv("SDV_GRID", str(G))
    B, K = 4, 5
    fan = [4, 3, 2, 1, 0, 2]
    temps = [0.9, 0.0, 0.6, 1.4]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=20,
                  temperature=temps, seed=90 + G, device=dev, bonus_row=True)
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True, compact=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    _check(*compare_verify(r, _oracle_for(inp, keys=keys_ref), temps))
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.offsets.cpu().numpy(), offs)
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)
    r2 = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, stats=True)
    _check(*compare_verify(r2, _oracle_for(inp), temps))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_largest_k_with_keys(dev, path, dt):
    B, K, V = 2, 32, 3001
    fan = [2] * K + [1]
    temps = [1.0, 0.0]
    inp = W.synth(B, K, V, dt, kind="normal", sigma=1.0, draft_sigma=0.1, temperature=temps,
                  seed=32, device=dev, bonus_row=True)
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True, compact=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    o = _oracle_for(inp, keys=keys_ref)
    _check(*compare_verify(r, o, temps))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_maximum_sizes(dev, path, dt):
    """The header's limits at once: SD_MAX_V, SD_MAX_K and SD_MAX_FANOUT keys
    at every position plus the bonus row; every row against the oracle."""
    B, K, V = 2, sd.SD_MAX_K, sd.SD_MAX_V
    fan = [sd.SD_MAX_FANOUT] * (K + 1)
    temps = [0.8, 0.0]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=2.0, draft_sigma=0.5, peaks=20,
                  temperature=temps, seed=262, device=dev, bonus_row=True)
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, stats=True, compact=True)
    np.testing.assert_array_equal(r.keys.cpu().numpy(), keys_ref)
    o = _oracle_for(inp, keys=keys_ref)
    _check(*compare_verify(r, o, temps))
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)


@pytest.mark.parametrize("B,K,V", [(4096, 2, 300), (1500, 4, 1024)])
def test_large_batches_of_short_rows(dev, path, B, K, V):
    """Many sequences of short rows: a streaming CTA covers dozens of rows,
    the finish launches thousands of clusters; every row against the oracle."""
    g = torch.Generator().manual_seed(B + K)
    temps = torch.where(torch.rand(B, generator=g) < 0.7, torch.rand(B, generator=g) + 0.3,
                        torch.zeros(B)).tolist()
    inp = W.synth(B, K, V, "bf16", kind="normal", sigma=2.0, draft_sigma=0.7,
                  temperature=temps, seed=B, device=dev)
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, compact=True)
    o = _oracle_for(inp)
    stats, bad = compare_verify(r, o, temps, check_stats=False)
    _check(stats, bad)
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.offsets.cpu().numpy(), offs)
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)


def test_d3d_key_counts(dev, path):
    B, K, V = 2, 15, 4096
    inp = W.synth(B, K, V, "bf16", kind="normal", temperature=0.0, seed=9, device=dev,
                  bonus_row=True)
    for positions, cands, tokens_prepared in [(11, 2, 384), (15, 2, 512), (11, 5, 912)]:
        fan = [cands] * positions + [0] * (K - positions) + [1]
        keys = sd.outcome_predict(inp.draft, inp.tokens, fan, inp.draft_bonus)
        assert (keys.shape[1] + 1) * 16 == tokens_prepared
        ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                     _np(inp.draft_bonus))
        np.testing.assert_array_equal(keys.cpu().numpy(), ref)


# --------------------------------------------------------------- edge cases ----
def test_invalid_rows_set_status_and_empty_batch(dev, path):
    B, K, V = 4, 3, 999
    inp = W.synth(B, K, V, "f32", temperature=[1.0, 1.0, 1.0, 0.0], seed=3, device=dev)
    inp.tokens[1, 2] = V
    inp.temperature[2] = -1.0
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, compact=True)
    st = int(r.status.item())
    assert st & sd.SD_STATUS_BAD_TOKEN and st & sd.SD_STATUS_BAD_TEMP
    assert r.tau[1].item() == 0 and r.tau[2].item() == 0
    assert (r.out_tokens[1] == -1).all() and (r.out_tokens[2] == -1).all()
    o = _oracle_for(inp)
    _check(*compare_verify(r, o, inp.temperature.cpu().numpy(), check_stats=False))
    # empty batch
    e = torch.empty((0, K + 1, V), device=dev)
    r0 = sd.verify(e, torch.empty((0, K, V), device=dev), torch.empty((0, K), dtype=torch.int32,
                   device=dev), torch.empty(0, device=dev), 1, compact=True)
    assert r0.offsets.tolist() == [0]


def test_repeated_calls_and_scratch(dev, monkeypatch, capfd):
    # back-to-back calls on one stream give identical results on both paths;
    # with scratch and SDV_SPLIT=1 the split path runs (SDV_VERBOSE names it);
    # scratch is never read before it is written in the same call (it starts
    # filled with garbage here); scratch below sd_verify_workspace_size is
    # refused
    B, K, V = 8, 5, 5000
    inp = W.synth(B, K, V, "bf16", kind="peaked", peaks=4, temperature=0.8, seed=21, device=dev)
    ws = torch.full((sd.workspace_bytes(B, K),), 0xAB, dtype=torch.uint8, device=dev)
    monkeypatch.setenv("SDV_SPLIT", "1")
    monkeypatch.setenv("SDV_VERBOSE", "1")
    a = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, ws=ws,
                  compact=True)
    torch.cuda.synchronize()
    assert "sd_verify split:" in capfd.readouterr().err
    b = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, ws=ws,
                  compact=True)
    monkeypatch.setenv("SDV_SPLIT", "0")
    c = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, compact=True)
    torch.cuda.synchronize()
    assert "sd_verify: mode=0" in capfd.readouterr().err
    n = int(a.offsets[-1])
    assert torch.equal(a.out_tokens, b.out_tokens) and torch.equal(a.tau, b.tau)
    assert torch.equal(a.packed[:n], b.packed[:n])
    # the two paths group the sums differently: both against the oracle
    o = _oracle_for(inp)
    for x in (a, c):
        _check(*compare_verify(x, o, inp.temperature.cpu().numpy(), check_stats=False))
    monkeypatch.setenv("SDV_SPLIT", "1")
    with pytest.raises(sd.SDError):
        sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed,
                  ws=torch.zeros(64, dtype=torch.uint8, device=dev))
    monkeypatch.delenv("SDV_VERBOSE")
    # then a smaller batch with another K and dtype
    inp2 = W.synth(3, 2, 777, "f32", temperature=[0.0, 1.0, 0.5], seed=2, device=dev)
    c = sd.verify(inp2.target, inp2.draft, inp2.tokens, inp2.temperature, inp2.seed)
    o = _oracle_for(inp2)
    _check(*compare_verify(c, o, inp2.temperature.cpu().numpy(), check_stats=False))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_check_finite_flags_rows_read(dev, path, dt):
    # SD_FLAG_CHECK_FINITE: a NaN or +inf, or a row of only -inf, in any row
    # the call reads makes that sequence invalid with SD_STATUS_NONFINITE; a
    # single -inf is a valid logit; every other sequence is exact against the
    # oracle (which applies the same rule to the same rows)
    B, K, V = 24, 4, 9001
    fan = [2, 0, 1, 0, 1]                      # keys at positions 0, 2 and K
    temps = [0.0 if b % 3 == 0 else 0.8 for b in range(B)]
    inp = W.synth(B, K, V, dt, kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=10,
                  temperature=temps, seed=606, device=dev, bonus_row=True)
    t, d, bo = inp.target.float(), inp.draft.float(), inp.draft_bonus.float()
    rng = np.random.default_rng(606)
    planted = [float("nan"), float("inf"), "allneg", float("-inf"), None]
    for b in range(B):
        kind = planted[b % 5]
        if kind is None:
            continue
        where = (b // 5) % 3
        arr = t[b] if where == 0 else d[b] if where == 1 else bo[b:b + 1]
        r = int(rng.integers(0, arr.shape[0]))
        if kind == "allneg":
            arr[r, :] = float("-inf")
        else:
            arr[r, int(rng.integers(0, V))] = kind
    dtype = inp.target.dtype
    inp.target, inp.draft = t.to(dtype).contiguous(), d.to(dtype).contiguous()
    inp.draft_bonus = bo.to(dtype).contiguous()
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, check_finite=True, compact=True)
    torch.cuda.synchronize()
    o = oracle.verify(_np(inp.target), _np(inp.draft), inp.tokens.cpu().numpy(),
                      inp.temperature.cpu().numpy(), inp.seed, check_finite=True, fanout=fan,
                      draft_bonus=_np(inp.draft_bonus))
    flagged = o["nonfinite"].astype(bool)
    assert 5 < flagged.sum() < B
    np.testing.assert_array_equal(r.tau.cpu().numpy() == 0, flagged)
    assert int(r.status.item()) & sd.SD_STATUS_NONFINITE
    assert (r.out_tokens.cpu().numpy()[flagged] == -1).all()
    assert (r.hit.cpu().numpy()[flagged] == 0).all()
    keys_ref = oracle.outcome_predict(_np(inp.draft), inp.tokens.cpu().numpy(), fan,
                                      _np(inp.draft_bonus))
    ok = ~flagged
    np.testing.assert_array_equal(r.keys.cpu().numpy()[ok], keys_ref[ok])
    o2 = _oracle_for(inp, keys=keys_ref)
    rows = list(np.nonzero(ok)[0])
    stats, bad = compare_verify(r, {k: (v[rows] if isinstance(v, np.ndarray) else v)
                                    for k, v in o2.items()}, np.asarray(temps)[rows],
                                check_stats=False, rows=rows)
    _check(stats, bad)
    # without the flag the same call faults nothing and flags nothing
    r2 = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                   draft_bonus=inp.draft_bonus, compact=True)
    torch.cuda.synchronize()
    assert not int(r2.status.item()) & sd.SD_STATUS_NONFINITE


def test_row_base_splits_batch_identically(dev, path):
    B, K, V = 10, 4, 9000
    inp = W.synth(B, K, V, "bf16", kind="normal", temperature=0.9, seed=31, device=dev)
    full = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed)
    h = B // 2
    lo = sd.verify(inp.target[:h].contiguous(), inp.draft[:h].contiguous(),
                   inp.tokens[:h].contiguous(), inp.temperature[:h].contiguous(), inp.seed)
    hi = sd.verify(inp.target[h:].contiguous(), inp.draft[h:].contiguous(),
                   inp.tokens[h:].contiguous(), inp.temperature[h:].contiguous(), inp.seed,
                   row_base=h)
    assert torch.equal(full.out_tokens, torch.cat([lo.out_tokens, hi.out_tokens]))


def test_second_device_in_the_same_process(dev, path):
    """The library's host state (SM count, kernel attributes, cluster
    occupancy) is kept per device: one process calling on cuda:1 after
    cuda:0, and on cuda:0 again, gets the same results on each."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two visible devices")
    B, K, V = 12, 5, 50021
    inp = W.synth(B, K, V, "bf16", kind="normal", temperature=0.8, seed=77, device=dev)
    fan = [2] * (K + 1)

    def run(d):
        with torch.cuda.device(d):
            r = sd.verify(inp.target.to(d), inp.draft.to(d), inp.tokens.to(d),
                          inp.temperature.to(d), inp.seed, fanout=fan, compact=True)
            torch.cuda.synchronize(d)
        return {k: getattr(r, k).cpu() for k in ("out_tokens", "tau", "keys", "packed",
                                                  "status")}

    first = run(torch.device("cuda:0"))
    second = run(torch.device("cuda:1"))
    again = run(torch.device("cuda:0"))
    for k in first:
        assert torch.equal(first[k], second[k]), k
        assert torch.equal(first[k], again[k]), k


def test_compact_standalone(dev):
    rng = np.random.default_rng(4)
    B, K = 3000, 5
    tau = rng.integers(0, K + 2, B).astype(np.int32)
    out = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        out[b, : tau[b]] = rng.integers(0, 10 ** 6, tau[b])
    offs, packed = sd.compact(torch.from_numpy(out).to(dev), torch.from_numpy(tau).to(dev))
    ro, rp = oracle.compact(out, tau)
    np.testing.assert_array_equal(offs.cpu().numpy(), ro)
    np.testing.assert_array_equal(packed.cpu().numpy()[: ro[-1]], rp)


# ------------------------------------------- workloads at full size, sampled --
@pytest.mark.parametrize("name", W.ORDER)
def test_workload_full_size_sampled_rows(dev, path, name):
    inp = W.workload(name, round_idx=3, device=dev)
    spec = W.WORKLOADS[name]
    fan = spec.get("fanout")
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, fanout=fan,
                  draft_bonus=inp.draft_bonus, compact=True, stats=True)
    torch.cuda.synchronize()
    B = inp.B
    rng = np.random.default_rng(hash(name) % 2 ** 32)
    rows = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, 6), replace=False))))
    keys_ref = None
    if fan is not None:
        keys_ref = oracle.outcome_predict(_np(inp.draft[rows]), inp.tokens[rows].cpu().numpy(),
                                          fan, _np(inp.draft_bonus[rows]))
        np.testing.assert_array_equal(r.keys.cpu().numpy()[rows], keys_ref)
        full_keys = np.zeros((B,) + keys_ref.shape[1:], np.int32)
        full_keys[rows] = keys_ref
        keys_ref = full_keys
    o = _oracle_for(inp, rows=rows, keys=keys_ref)
    stats, bad = compare_verify(r, o, inp.temperature.cpu().numpy()[rows], rows=rows)
    _check(stats, bad)
    # compaction over every row (integer work: exact)
    offs, packed = oracle.compact(r.out_tokens.cpu().numpy(), r.tau.cpu().numpy())
    np.testing.assert_array_equal(r.offsets.cpu().numpy(), offs)
    np.testing.assert_array_equal(r.packed.cpu().numpy()[: offs[-1]], packed)
    # properties that hold for every row
    tau = r.tau.cpu().numpy()
    na = r.num_accepted.cpu().numpy()
    assert ((tau >= 1) & (tau <= inp.K + 1)).all() and (tau == na + 1).all()
    ot = r.out_tokens.cpu().numpy()
    tok = inp.tokens.cpu().numpy()
    for b in range(B):
        assert (ot[b, : na[b]] == tok[b, : na[b]]).all()
        assert 0 <= ot[b, na[b]] < inp.V and (ot[b, na[b] + 1:] == -1).all()
        if na[b] < inp.K and inp.temperature[b].item() > 0:
            assert ot[b, na[b]] != tok[b, na[b]]     # the residual excludes a rejected draft
    assert int(r.status.item()) == 0


@pytest.mark.parametrize("name,rounds", [("small", 200), ("peaked", 40)])
def test_many_rounds_mismatch_count(dev, path, name, rounds):
    """Every sampled row compared in full over many rounds: no difference
    outside the guard band; guarded rows counted."""
    tot = dict(rows=0, positions=0, guarded=0, guarded_mismatch=0, mismatch_outside_guard=0)
    for rd in range(rounds):
        inp = W.workload(name, round_idx=rd, device=dev)
        r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed, stats=True)
        o = _oracle_for(inp)
        stats, bad = compare_verify(r, o, inp.temperature.cpu().numpy())
        assert not bad, (rd, bad[:5])
        for k in tot:
            tot[k] += stats[k]
    print(f"{name}: {tot}")
    assert tot["mismatch_outside_guard"] == 0
    assert tot["guarded_mismatch"] <= max(1, 1e-4 * tot["positions"])


# ------------------------------------------------------------ D3D packing --
@pytest.mark.parametrize("B,K,n_keys", [(1, 15, 23), (16, 15, 23), (300, 7, 13), (5, 32, 40),
                                        (3, 0, 2), (4, 5, 0), (7, 15, 56)])
def test_d3d_pack_matches_oracle(dev, B, K, n_keys):
    # keys as sd_outcome_predict writes them, plus empty slots and positions
    # outside [0, K]; integer layout work: exact
    rng = np.random.default_rng(1000 + B + K + n_keys)
    keys = np.stack([rng.integers(-1, K + 2, size=(B, n_keys)),
                     rng.integers(0, 50000, size=(B, n_keys))], -1).astype(np.int32)
    keys[rng.random((B, n_keys)) < 0.2] = -1
    tok = rng.integers(0, 50000, size=(B, K)).astype(np.int32)
    anchor = rng.integers(0, 50000, size=B).astype(np.int32)
    pos = rng.integers(0, 100000, size=B).astype(np.int32)
    t_ref, p_ref, c_ref = oracle.d3d_pack(keys, tok, anchor, pos, 50001)
    g = lambda a: torch.from_numpy(a).to(dev)
    t, p, c = sd.d3d_pack(g(keys), g(tok), g(anchor), g(pos), 50001)
    np.testing.assert_array_equal(t.cpu().numpy(), t_ref)
    np.testing.assert_array_equal(p.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(c.cpu().numpy(), c_ref)


def test_d3d_workload_pack_after_verify(dev, path):
    # the D3D round at full size: verify with fused keys, then the pack from
    # the kernel's own keys; the pack equals the oracle's for those keys, and
    # on every hit row the block of the real outcome continues the confirmed
    # text exactly
    inp = W.workload("d3d", round_idx=2, device=dev)
    m = inp.meta
    r = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed,
                  fanout=inp.fanout, draft_bonus=inp.draft_bonus, compact=True)
    t, p, c = sd.d3d_pack(r.keys, inp.tokens, m["anchor"], m["anchor_pos"], m["mask_token"])
    torch.cuda.synchronize()
    keys = r.keys.cpu().numpy()
    assert keys.shape[1] == 23 and t.shape[1:] == (24, 16)     # 24 blocks x 16 = 384 tokens
    t_ref, p_ref, c_ref = oracle.d3d_pack(keys, inp.tokens.cpu().numpy(),
                                          m["anchor"].cpu().numpy(),
                                          m["anchor_pos"].cpu().numpy(), m["mask_token"])
    np.testing.assert_array_equal(t.cpu().numpy(), t_ref)
    np.testing.assert_array_equal(p.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(c.cpu().numpy(), c_ref)
    tau, na, out = r.tau.cpu().numpy(), r.num_accepted.cpu().numpy(), r.out_tokens.cpu().numpy()
    hit = r.hit.cpu().numpy()
    anchor = m["anchor"].cpu().numpy()
    for b in range(inp.B):
        blocks = [i for i in range(1, 24) if c_ref[b, i] == tau[b] and t_ref[b, i, 0] == out[b, na[b]]]
        assert bool(blocks) == bool(hit[b])
        for i in blocks:
            assert list(t_ref[b, 0, :tau[b]]) + [t_ref[b, i, 0]] == [anchor[b]] + list(out[b, :tau[b]])
    # then the target's KV cache rolled back to the round's tau
    bt = m["block_table"].clone()
    n, f, o = sd.kv_rollback(bt, m["kv_len"], r.tau, m["page_size"], inp.K + 1)
    bt_ref, n_ref, f_ref, o_ref = oracle.kv_rollback(m["block_table"].cpu().numpy(),
                                                     m["kv_len"].cpu().numpy(), tau,
                                                     m["page_size"], inp.K + 1)
    np.testing.assert_array_equal(bt.cpu().numpy(), bt_ref)
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(f.cpu().numpy()[: o_ref[-1]], f_ref)
    assert (n_ref == m["anchor_pos"].cpu().numpy() + tau).all()   # the prefix plus tau


# ------------------------------------------------ n-gram / prompt lookup --
@pytest.mark.parametrize("B,L,K,n_max,n_min,vocab", [(300, 80, 5, 4, 1, 6), (7, 1000, 8, 3, 3, 4),
                                                     (64, 513, 0, 6, 2, 3), (5, 1, 4, 2, 1, 2),
                                                     (40, 2048, 32, 16, 1, 2), (33, 300, 4, 4, 1, 50000)])
def test_ngram_draft_matches_oracle(dev, B, L, K, n_max, n_min, vocab):
    # small vocabularies give many and long matches, a large one almost none;
    # lengths cover 0, 1 and the full row; exact
    rng = np.random.default_rng(7 * B + L + K)
    h = rng.integers(0, vocab, size=(B, L)).astype(np.int32)
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    lens[0], lens[-1] = L, min(1, L)
    ref = oracle.ngram_draft(h, lens, K, n_max, n_min)
    out = sd.ngram_draft(torch.from_numpy(h).to(dev), torch.from_numpy(lens).to(dev), K, n_max,
                         n_min)
    for x, y in zip(out, ref):
        np.testing.assert_array_equal(x.cpu().numpy(), y)


def test_ngram_workload_full_size(dev):
    # the benchmark's histories (256 rows up to 16384 tokens): every row exact
    for rd in (0, 3):
        h, lens, s = W.ngram_inputs(rd, device=dev)
        ref = oracle.ngram_draft(h.cpu().numpy(), lens.cpu().numpy(), s["K"], s["n_max"],
                                 s["n_min"])
        out = sd.ngram_draft(h, lens, s["K"], s["n_max"], s["n_min"])
        for x, y in zip(out, ref):
            np.testing.assert_array_equal(x.cpu().numpy(), y)
        assert (ref[3] >= 0).mean() > 0.8      # the histories repeat themselves


# ------------------------------------------------------- KV-cache rollback --
@pytest.mark.parametrize("B,page,maxp,appended", [(50, 16, 40, 6), (3000, 16, 8, 16), (7, 1, 64, 9),
                                                  (1, 32, 3, 33), (1100, 7, 20, 5)])
def test_kv_rollback_matches_oracle(dev, B, page, maxp, appended):
    rng = np.random.default_rng(B + page + maxp)
    bt = rng.permutation(B * maxp).astype(np.int32).reshape(B, maxp)
    kv = rng.integers(0, page * maxp + page, size=B).astype(np.int32)   # some past the table
    tau = rng.integers(0, appended + 3, size=B).astype(np.int32)
    bt_ref, n_ref, f_ref, o_ref = oracle.kv_rollback(bt, kv, tau, page, appended)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    btd = g(bt)
    n, f, o = sd.kv_rollback(btd, g(kv), g(tau), page, appended)
    np.testing.assert_array_equal(btd.cpu().numpy(), bt_ref)
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(o.cpu().numpy(), o_ref)
    np.testing.assert_array_equal(f.cpu().numpy()[: o_ref[-1]], f_ref)
