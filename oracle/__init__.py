"""CPU oracle for the speculative-decoding verify step (test infrastructure).

This package is TEST INFRASTRUCTURE: only ``tests/``, the package smoke
check in ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The product path (the CUDA library and its
Python binding) never imports, links or executes anything here.

The arithmetic lives in ``sd_oracle.cpp`` (plain single-threaded C++ in
double precision); this module only compiles it with g++ and marshals numpy
arrays through ctypes.  See the header of ``sd_oracle.cpp`` for the method,
its sources and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.cpp")
_LIB = os.path.join(_HERE, "libsdoracle.so")
_lock = threading.Lock()
_lib = None

DT_F32 = 0
DT_BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``sd_oracle.cpp`` into ``libsdoracle.so`` (g++, no fast-math,
    no FMA contraction so x86 and Arm hosts round identically)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Bind the oracle's functions from an explicitly named build of
    ``sd_oracle.cpp`` (tests use this to load deliberately broken copies)."""
    global _lib
    with _lock:
        _lib = None
        _lib = _bind(ctypes.CDLL(path))
    return _lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(L):
    P = ctypes.c_void_p
    i32, i64, u32, u64, dbl = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                               ctypes.c_uint64, ctypes.c_double)
    L.oracle_philox4x32_10.argtypes = [P, P, P]
    L.oracle_philox4x32_10.restype = None
    L.oracle_uniform.argtypes = [u64, u32, u32, u32]
    L.oracle_uniform.restype = dbl
    L.oracle_verify_row_u.argtypes = [i32, i32, i32, P, P, P, dbl, P, P, P, P, P,
                                      P, P, P, P]
    L.oracle_verify_row_u.restype = i32
    L.oracle_verify.argtypes = [i32, i32, i32, i32, P, P, P, P, u64, i64, P, i32,
                                P, P, P, P, P, P, P, P, P, P, P]
    L.oracle_verify.restype = i32
    L.oracle_verify_checked.argtypes = [i32, i32, i32, i32, P, P, P, P, u64, i64, P, i32,
                                        P, P, P, P, P, P, P, P, P, P, P, i32, P, P, P]
    L.oracle_verify_checked.restype = i32
    L.oracle_outcome_predict.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
    L.oracle_outcome_predict.restype = i32
    L.oracle_compact.argtypes = [i32, i32, P, P, P, P]
    L.oracle_d3d_pack.argtypes = [i32, i32, i32, P, P, P, P, i32, P, P, P]
    L.oracle_d3d_pack.restype = None
    L.oracle_ngram_draft.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P]
    L.oracle_ngram_draft.restype = None
    L.oracle_kv_rollback.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P]
    L.oracle_kv_rollback.restype = None
    L.oracle_compact.restype = None
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """numpy float32 or bf16-as-uint16 array -> (contiguous array, dtype code)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, DT_F32
    if a.dtype == np.uint16:
        return a, DT_BF16
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {a.dtype}")


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, row: int, pos: int, slot: int) -> float:
    return lib().oracle_uniform(seed, row, pos, slot)


def verify_row_u(target, draft, tokens, T, u_accept, u_sample):
    """One sequence with explicit uniforms.  target [K+1][V], draft [K][V]
    (float32 or bf16 bits), tokens [K].  Returns a dict."""
    target, dt = _logits(target)
    K = target.shape[0] - 1
    V = target.shape[1]
    if K > 0:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape == (K, V)
    else:
        draft = np.zeros((0, V), dtype=target.dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    ua = np.ascontiguousarray(np.asarray(u_accept, dtype=np.float64).reshape(-1))
    us = np.ascontiguousarray(np.asarray(u_sample, dtype=np.float64).reshape(-1))
    assert ua.size >= K and us.size >= K + 1
    out = np.full(K + 1, -1, dtype=np.int32)
    n_acc = np.zeros(1, dtype=np.int32)
    guard = np.zeros(1, dtype=np.int32)
    ratio = np.full(max(K, 1), np.nan)
    ptok = np.full(max(K, 1), np.nan)
    qtok = np.full(max(K, 1), np.nan)
    amax = np.zeros(K + 1, dtype=np.int32)
    tau = lib().oracle_verify_row_u(K, V, dt, _ptr(target), _ptr(draft), _ptr(tokens),
                                    float(T), _ptr(ua), _ptr(us), _ptr(out), _ptr(n_acc),
                                    _ptr(guard), _ptr(ratio), _ptr(ptok), _ptr(qtok),
                                    _ptr(amax))
    return dict(tau=int(tau), n_acc=int(n_acc[0]), out_tokens=out, guard_pos=int(guard[0]),
                ratio=ratio[:K], p_tok=ptok[:K], q_tok=qtok[:K], argmax=amax)


def verify(target, draft, tokens, temperature, seed: int, row_base: int = 0, keys=None,
           stats: bool = False, check_finite: bool = False, fanout=None, draft_bonus=None):
    """Batch verify with Philox uniforms.  target [B][K+1][V], draft
    [B][K][V], tokens [B][K], temperature [B].  keys: optional
    [B][n_keys][2] int32.  check_finite: also check the rows the step reads
    (draft rows of positions with fanout > 0 and, with fanout[K] > 0, the
    draft_bonus rows count as read); 'nonfinite' [B] marks the sequences it
    made invalid.  Returns a dict of numpy arrays."""
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    if K > 0:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape == (B, K, V)
    else:
        draft = np.zeros((B, 0, V), dtype=target.dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    temps = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    n_keys = 0
    if keys is not None:
        keys = np.ascontiguousarray(keys, dtype=np.int32)
        n_keys = keys.shape[1]
    r = dict(
        num_accepted=np.zeros(B, np.int32),
        out_tokens=np.full((B, K + 1), -1, np.int32),
        tau=np.zeros(B, np.int32),
        hit=np.zeros(B, np.uint8),
        guard_pos=np.full(B, -1, np.int32),
    )
    if stats:
        r.update(ratio=np.full((B, K), np.nan), p_tok=np.full((B, K), np.nan),
                 q_tok=np.full((B, K), np.nan), argmax=np.zeros((B, K + 1), np.int32),
                 Zt=np.full((B, K + 1), np.nan), Zd=np.full((B, K), np.nan))
    g = r.get
    fan = None
    if fanout is not None:
        fan = np.ascontiguousarray(fanout, dtype=np.int32).reshape(K + 1)
    bonus = None
    if draft_bonus is not None:
        bonus, dt3 = _logits(draft_bonus)
        assert dt3 == dt and bonus.shape == (B, V)
    r["nonfinite"] = np.zeros(B, np.uint8)
    invalid = lib().oracle_verify_checked(
        B, K, V, dt, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(temps), seed, row_base,
        _ptr(keys), n_keys, _ptr(r["num_accepted"]), _ptr(r["out_tokens"]), _ptr(r["tau"]),
        _ptr(r["hit"]), _ptr(r["guard_pos"]), _ptr(g("ratio")), _ptr(g("p_tok")),
        _ptr(g("q_tok")), _ptr(g("argmax")), _ptr(g("Zt")), _ptr(g("Zd")),
        1 if check_finite else 0, _ptr(fan), _ptr(bonus), _ptr(r["nonfinite"]))
    r["invalid_rows"] = int(invalid)
    return r


def outcome_predict(draft, tokens, fanout, draft_bonus=None):
    """Speculation-cache keys [B][sum(fanout)][2] (position, token)."""
    draft, dt = _logits(draft)
    B, K, V = draft.shape
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    fanout = np.ascontiguousarray(fanout, dtype=np.int32).reshape(K + 1)
    if draft_bonus is not None:
        draft_bonus, dt2 = _logits(draft_bonus)
        assert dt2 == dt and draft_bonus.shape == (B, V)
    n_keys = int(fanout.sum())
    keys = np.zeros((B, n_keys, 2), np.int32)
    n = lib().oracle_outcome_predict(B, K, V, dt, _ptr(draft), _ptr(tokens),
                                     _ptr(draft_bonus), _ptr(fanout), _ptr(keys))
    assert n == n_keys
    return keys


def compact(out_tokens, tau):
    out_tokens = np.ascontiguousarray(out_tokens, dtype=np.int32)
    B, K1 = out_tokens.shape
    tau = np.ascontiguousarray(tau, dtype=np.int32).reshape(B)
    offsets = np.zeros(B + 1, np.int32)
    packed = np.full(max(int(tau.sum()), 1), -1, np.int32)
    lib().oracle_compact(B, K1 - 1, _ptr(out_tokens), _ptr(tau), _ptr(offsets), _ptr(packed))
    return offsets, packed[: int(tau.sum())]


def d3d_pack(keys, draft_tokens, anchor, anchor_pos, mask_token: int):
    """The drafter's packed next pass: (tokens, positions) [B][1+n_keys][K+1]
    and ctx [B][1+n_keys] (block-0 tokens each block sees)."""
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    B, n_keys, _ = keys.shape
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    K = draft_tokens.shape[1]
    anchor = np.ascontiguousarray(anchor, dtype=np.int32).reshape(B)
    anchor_pos = np.ascontiguousarray(anchor_pos, dtype=np.int32).reshape(B)
    nb = 1 + n_keys
    tokens = np.zeros((B, nb, K + 1), np.int32)
    positions = np.zeros((B, nb, K + 1), np.int32)
    ctx = np.zeros((B, nb), np.int32)
    lib().oracle_d3d_pack(B, K, n_keys, _ptr(keys), _ptr(draft_tokens), _ptr(anchor),
                          _ptr(anchor_pos), int(mask_token), _ptr(tokens), _ptr(positions),
                          _ptr(ctx))
    return tokens, positions, ctx


def ngram_draft(history, lengths, K: int, n_max: int, n_min: int):
    """Prompt-lookup drafts: (drafts [B][K], count [B], match_pos [B],
    match_n [B]) from history [B][L] int32 and lengths [B]."""
    history = np.ascontiguousarray(history, dtype=np.int32)
    B, L = history.shape
    lengths = np.ascontiguousarray(lengths, dtype=np.int32).reshape(B)
    drafts = np.zeros((B, K), np.int32)
    count, pos, n = (np.zeros(B, np.int32) for _ in range(3))
    lib().oracle_ngram_draft(B, L, K, n_max, n_min, _ptr(history), _ptr(lengths), _ptr(drafts),
                             _ptr(count), _ptr(pos), _ptr(n))
    return drafts, count, pos, n


def kv_rollback(block_table, kv_len, tau, page_size: int, appended: int):
    """(block_table after, new_len [B], freed page ids, free_offsets [B+1])."""
    bt = np.array(block_table, dtype=np.int32, copy=True)
    B, max_pages = bt.shape
    kv_len = np.ascontiguousarray(kv_len, dtype=np.int32).reshape(B)
    tau = np.ascontiguousarray(tau, dtype=np.int32).reshape(B)
    new_len = np.zeros(B, np.int32)
    freed = np.full(max(B * max_pages, 1), -1, np.int32)
    offs = np.zeros(B + 1, np.int32)
    lib().oracle_kv_rollback(B, page_size, max_pages, appended, _ptr(kv_len), _ptr(tau), _ptr(bt),
                             _ptr(new_len), _ptr(freed), _ptr(offs))
    return bt, new_len, freed[: int(offs[-1])], offs
