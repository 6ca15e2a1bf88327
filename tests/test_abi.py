"""The C-ABI library loads and exports every symbol the headers declare
(host-side checks only: no CUDA compute is called here)."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_verification_logits_gb300 as sd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(sd_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    L = sd.lib()
    names = _declared_functions()
    assert "sd_verify" in names and "sd_outcome_predict" in names and "sd_compact" in names
    for n in names:
        assert hasattr(L, n), n


def test_struct_layout_and_strings():
    L = sd.lib()
    assert L.sd_verify_args_size() == ctypes.sizeof(sd.VerifyArgs)
    assert "sm_103a" in sd.version()
    assert L.sd_status_string(sd.SD_ERR_INVALID_ARG) == b"SD_ERR_INVALID_ARG"


def test_workspace_size():
    # the split launch keeps one 96-byte record per row piece: at most one per
    # logit row of the batch (2K+2 per sequence) plus one per streaming CTA
    # (at most 1024); 0 for arguments out of range
    L = sd.lib()
    for B, K in [(8, 5), (256, 5), (1, 0), (4, sd.SD_MAX_K), (0, 3)]:
        assert L.sd_verify_workspace_size(B, K) == (1024 + B * (2 * K + 2)) * 96
    assert L.sd_verify_workspace_size(4, sd.SD_MAX_K + 1) == 0
    assert L.sd_verify_workspace_size(-1, 5) == 0
    assert L.sd_verify_workspace_size(3, -1) == 0


def test_host_argument_checks_reject_bad_requests():
    L = sd.lib()
    assert L.sd_verify(None, None) == sd.SD_ERR_INVALID_ARG
    a = sd.VerifyArgs()
    a.B, a.K, a.V = 4, sd.SD_MAX_K + 1, 100
    assert L.sd_verify(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG
    a.K, a.V = 4, 0
    assert L.sd_verify(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG
    a.V, a.dtype = 100, 7
    assert L.sd_verify(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG
    a.dtype = sd.SD_BF16
    assert L.sd_verify(ctypes.byref(a), None) == sd.SD_ERR_INVALID_ARG   # null pointers
    assert L.sd_compact(-1, 2, None, None, None, None, None, None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_uniforms(1, -1, None, None, None, None, None) == sd.SD_ERR_INVALID_ARG
    fan = (ctypes.c_int32 * 3)(1, 9, 1)
    assert L.sd_outcome_predict(2, 2, 10, sd.SD_BF16, None, None, None,
                                ctypes.cast(fan, ctypes.c_void_p), None, None, None,
                                None) == sd.SD_ERR_INVALID_ARG


def test_next_row_entry_points_refuse_bad_requests():
    # host-side checks only: every call below is refused before any launch
    L = sd.lib()
    P = ctypes.c_void_p
    fake = P(1 << 20)   # a non-null address never dereferenced: the checks fail first
    # D3D pack: K, n_keys out of range, null outputs, keys not 8-byte aligned
    assert L.sd_d3d_pack(2, sd.SD_MAX_K + 1, 3, fake, fake, fake, fake, 0, fake, fake, fake,
                         None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_d3d_pack(2, 4, -1, fake, fake, fake, fake, 0, fake, fake, fake,
                         None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_d3d_pack(2, 4, 3, fake, fake, fake, fake, 0, None, fake, fake,
                         None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_d3d_pack(2, 4, 3, P((1 << 20) + 4), fake, fake, fake, 0, fake, fake, fake,
                         None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_d3d_pack(0, 4, 3, None, None, None, None, 0, None, None, None, None) == sd.SD_OK
    # KV rollback: page size, negative sizes, null inputs
    assert L.sd_kv_rollback(2, 0, 4, 5, fake, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_kv_rollback(2, 16, -1, 5, fake, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_kv_rollback(2, 16, 4, 5, None, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_kv_rollback(2, 16, 4, 5, fake, fake, fake, fake, fake, None,
                            None) == sd.SD_ERR_INVALID_ARG
    # n-gram drafter: n range, K range, history length beyond the packed key
    for n_max, n_min in [(4, 0), (2, 3), (17, 1)]:
        assert L.sd_ngram_draft(2, 64, 4, n_max, n_min, fake, fake, fake, fake, fake, fake,
                                None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_ngram_draft(2, 64, sd.SD_MAX_K + 1, 4, 1, fake, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_ngram_draft(2, 1 << 26, 4, 4, 1, fake, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_ngram_draft(2, 64, 4, 4, 1, None, fake, fake, fake, fake, fake,
                            None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_ngram_draft(0, 64, 4, 4, 1, None, None, None, None, None, None,
                            None) == sd.SD_OK


def test_vshard_entry_points_refuse_bad_requests():
    # host-side checks of the sharded verify: shard index and count, columns
    # outside the vocabulary, flags, null or unaligned blocks; nothing launched
    L = sd.lib()
    P = ctypes.c_void_p
    fake = P(1 << 20)
    assert L.sd_vshard_stats_bytes(4, 3) == 4 * 8 * 96 + 4 * 3 * 16
    assert L.sd_vshard_stats_bytes(-1, 3) == 0 and L.sd_vshard_mass_bytes(4) == 4 * 128
    good = dict(B=4, K=3, V=100, S=2, shard=1, v0=50, vs=50, dtype=sd.SD_BF16)
    for bad in (dict(S=0), dict(S=33), dict(shard=2), dict(shard=-1), dict(v0=60),
                dict(vs=0), dict(K=sd.SD_MAX_K + 1), dict(dtype=7), dict(flags=0x2)):
        a = sd.VShardArgs(**{**good, **bad})
        a.target_logits = a.draft_logits = a.draft_tokens = a.temperature = 1 << 20
        assert L.sd_vshard_stats(ctypes.byref(a), fake, None) == sd.SD_ERR_INVALID_ARG, bad
    a = sd.VShardArgs(**good)
    assert L.sd_vshard_stats(ctypes.byref(a), fake, None) == sd.SD_ERR_INVALID_ARG  # null logits
    a.target_logits = a.draft_logits = a.draft_tokens = a.temperature = 1 << 20
    assert L.sd_vshard_stats(ctypes.byref(a), None, None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_vshard_stats(ctypes.byref(a), P((1 << 20) + 8), None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_vshard_mass(ctypes.byref(a), fake, None, None) == sd.SD_ERR_INVALID_ARG
    assert L.sd_vshard_pick(ctypes.byref(a), fake, fake, None) == sd.SD_ERR_INVALID_ARG  # outputs
    a.flags = sd.SD_FLAG_PREDICT   # keys without fanout
    assert L.sd_vshard_stats(ctypes.byref(a), fake, None) == sd.SD_ERR_INVALID_ARG
    a = sd.VShardArgs(**{**good, "B": 0})
    assert L.sd_vshard_stats(ctypes.byref(a), None, None) == sd.SD_OK


def test_python_binding_refuses_cpu_tensors():
    import torch
    t = torch.zeros(2, 3, 10)
    with pytest.raises(ValueError):
        sd.verify(t, t[:, :2], torch.zeros(2, 2, dtype=torch.int32), torch.zeros(2), 1)


def test_python_wrappers_of_next_rows_refuse_bad_tensors():
    # the bindings refuse host tensors before calling the library
    import torch
    i32 = torch.zeros(4, 3, 2, dtype=torch.int32)
    with pytest.raises(ValueError):   # CPU tensors
        sd.d3d_pack(i32, torch.zeros(4, 5, dtype=torch.int32), torch.zeros(4, dtype=torch.int32),
                    torch.zeros(4, dtype=torch.int32), 0)
    with pytest.raises(ValueError):
        sd.kv_rollback(torch.zeros(4, 8, dtype=torch.int32), torch.zeros(4, dtype=torch.int32),
                       torch.zeros(4, dtype=torch.int32), 16, 6)
    with pytest.raises(ValueError):
        sd.ngram_draft(torch.zeros(4, 64, dtype=torch.int32), torch.zeros(4, dtype=torch.int32),
                       4, 4, 1)
