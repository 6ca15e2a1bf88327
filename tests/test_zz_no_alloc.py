"""sd_verify_noalloc: the verify step for callers that cannot allocate device
memory while they verify (a runtime whose memory all belongs to its own pool,
a plugin handed only its tensors).  It keeps the split launch's scratch in an
array inside the library instead of a caller buffer.

The GPU test calls it through the C ABI on two different batches in a row
and checks every output against sd_verify on the same inputs, with the
tolerance the parity tests use for probabilities (1e-5 relative) and exact
equality for tokens, counts, keys and offsets.  It runs in a fresh process
and after the other tests alike (the library's state is per device and
set up on first use).  The host-side refusals need no GPU.
"""
import ctypes

import numpy as np
import pytest
import torch

import sd_workloads as W

sd = pytest.importorskip("speculative_decoding_verification_logits_gb300")


def _noalloc_args(inp, r, fanout, n_keys):
    """sd_verify_args for inp / outputs r, filled field by field."""
    a = sd.VerifyArgs()
    B, K, V = inp.B, inp.K, inp.V
    a.B, a.K, a.V = B, K, V
    a.dtype = sd.SD_BF16 if inp.target.dtype == torch.bfloat16 else sd.SD_F32
    a.flags = sd.SD_FLAG_COMPACT | (sd.SD_FLAG_PREDICT if fanout else 0)
    a.seed, a.row_base = int(inp.seed) & (2 ** 64 - 1), 0
    a.target_logits, a.draft_logits = inp.target.data_ptr(), inp.draft.data_ptr()
    a.draft_tokens, a.temperature = inp.tokens.data_ptr(), inp.temperature.data_ptr()
    keep = None
    if fanout:
        keep = (ctypes.c_int32 * (K + 1))(*fanout)
        a.fanout_host = ctypes.cast(keep, ctypes.c_void_p)
        a.draft_bonus_logits = inp.draft_bonus.data_ptr() if inp.draft_bonus is not None else None
        a.keys_out = r.keys.data_ptr()
    a.num_accepted, a.out_tokens, a.tau = (r.num_accepted.data_ptr(), r.out_tokens.data_ptr(),
                                          r.tau.data_ptr())
    a.hit = r.hit.data_ptr() if r.hit is not None else None
    a.offsets, a.packed = r.offsets.data_ptr(), r.packed.data_ptr()
    a.accept_ratio, a.p_draft, a.q_draft = (r.accept_ratio.data_ptr(), r.p_draft.data_ptr(),
                                            r.q_draft.data_ptr())
    a.target_argmax = r.target_argmax.data_ptr()
    a.status = r.status.data_ptr()
    a.workspace, a.workspace_bytes = None, 0
    return a, keep


def _same(r, ref):
    for k in ("num_accepted", "out_tokens", "tau", "hit", "keys", "target_argmax"):
        x, y = getattr(r, k), getattr(ref, k)
        if y is not None:
            assert torch.equal(x, y), k
    n = int(ref.offsets[-1])
    assert torch.equal(r.offsets, ref.offsets) and torch.equal(r.packed[:n], ref.packed[:n])
    for k in ("accept_ratio", "p_draft", "q_draft"):
        np.testing.assert_allclose(getattr(r, k).cpu().numpy(), getattr(ref, k).cpu().numpy(),
                                   rtol=1e-5, equal_nan=True)
    assert int(r.status.item()) == int(ref.status.item()) == 0


@pytest.mark.gpu
def test_noalloc_matches_sd_verify_on_two_calls(monkeypatch, capfd):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # both batches are small enough (B times the cluster size below the SM
    # count) that the split launch, the one that keeps records in the static
    # array, is the one chosen; SDV_VERBOSE names the launch taken
    monkeypatch.delenv("SDV_SPLIT", raising=False)
    monkeypatch.setenv("SDV_VERBOSE", "1")
    dev = torch.device("cuda:0")
    L = sd.lib()
    stream = torch.cuda.current_stream(dev)
    cases = [
        # keys with a bonus row, bf16, sampled rows at two temperatures and a greedy row
        (W.synth(8, 6, 50021, "bf16", kind="peaked", sigma=3.0, draft_sigma=1.0, peaks=20,
                 temperature=[0.7, 0.0, 1.0, 0.7, 0.7, 0.0, 1.3, 0.7], seed=5, device=dev,
                 bonus_row=True), [4, 3, 2, 1, 1, 1, 1]),
        # then a different batch shape: fp32, no keys
        (W.synth(5, 3, 9001, "f32", temperature=[0.0, 1.0, 0.5, 0.9, 1.0], seed=6, device=dev),
         None),
    ]
    for inp, fan in cases:
        n_keys = sum(fan) if fan else 0
        ref = sd.verify(inp.target, inp.draft, inp.tokens, inp.temperature, inp.seed,
                        fanout=fan, draft_bonus=inp.draft_bonus if fan else None,
                        compact=True, stats=True)
        r = sd.alloc_outputs(inp.B, inp.K, dev, hit=bool(fan), compact=True, stats=True,
                             n_keys=n_keys)
        a, keep = _noalloc_args(inp, r, fan, n_keys)
        capfd.readouterr()
        rc = L.sd_verify_noalloc(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream))
        assert rc == sd.SD_OK, L.sd_status_string(rc)
        torch.cuda.synchronize(dev)
        assert "sd_verify split:" in capfd.readouterr().err
        _same(r, ref)
        del keep


def test_noalloc_refuses_caller_scratch_and_oversized_batches():
    # host-side checks, before any device work: a caller buffer is not
    # accepted, and a batch whose records exceed the 2 MiB array is refused
    L = sd.lib()
    a = sd.VerifyArgs()
    a.B, a.K, a.V, a.dtype = 4, 2, 100, sd.SD_F32
    a.workspace, a.workspace_bytes = 4096, 4096
    assert L.sd_verify_noalloc(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG
    a.workspace, a.workspace_bytes = None, 0
    a.B, a.K = 4096, 32     # (1024 + 4096 * 66) records of 96 bytes: about 26 MB
    assert L.sd_verify_noalloc(ctypes.byref(a), None) == sd.SD_ERR_UNSUPPORTED
    a.B, a.K = 4, sd.SD_MAX_K + 1
    assert L.sd_verify_noalloc(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_verify_noalloc(None, None) == sd.SD_ERR_INVALID_ARG
