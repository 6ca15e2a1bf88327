"""GB300-native speculative-decoding verify step (Python binding).

Thin ctypes binding of ``libsdverify.so`` (C ABI in ``include/sd_verify.h``).
This module only marshals arguments: it checks tensor dtypes, devices and
shapes, allocates outputs with torch, and passes raw device pointers and the
current CUDA stream to the library.  Every step of the verify path runs in
the library's CUDA kernels; there is no CPU fallback, and importing or calling
without the built library raises.

Entry points (same names as the C ABI):
  verify(...)            sd_verify
  outcome_predict(...)   sd_outcome_predict
  compact(...)           sd_compact
  uniforms(...)          sd_uniforms
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading
from dataclasses import dataclass

import torch

from . import _build

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_CUDA = 0, 1, 2, 3
SD_STATUS_BAD_TOKEN, SD_STATUS_BAD_TEMP, SD_STATUS_NONFINITE = 0x1, 0x2, 0x4
SD_F32, SD_BF16 = 0, 1
SD_FLAG_PREDICT, SD_FLAG_COMPACT, SD_FLAG_CHECK_FINITE = 0x1, 0x2, 0x4
SD_MAX_K, SD_MAX_V, SD_MAX_FANOUT = 32, 262144, 8

_P = ctypes.c_void_p


class VerifyArgs(ctypes.Structure):
    """Mirror of ``sd_verify_args`` in include/sd_verify.h."""
    _fields_ = [
        ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("seed", ctypes.c_uint64), ("row_base", ctypes.c_int64),
        ("target_logits", _P), ("draft_logits", _P), ("draft_tokens", _P),
        ("temperature", _P), ("cache_keys", _P), ("n_keys", ctypes.c_int32),
        ("fanout_host", _P), ("draft_bonus_logits", _P), ("keys_out", _P),
        ("num_accepted", _P), ("out_tokens", _P), ("tau", _P),
        ("hit", _P), ("offsets", _P), ("packed", _P),
        ("accept_ratio", _P), ("p_draft", _P), ("q_draft", _P), ("target_argmax", _P),
        ("status", _P), ("workspace", _P), ("workspace_bytes", ctypes.c_size_t),
    ]


class VShardArgs(ctypes.Structure):
    """Mirror of ``sd_vshard_args`` in include/sd_verify.h."""
    _fields_ = [
        ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("S", ctypes.c_int32), ("shard", ctypes.c_int32), ("v0", ctypes.c_int32),
        ("vs", ctypes.c_int32), ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("seed", ctypes.c_uint64), ("row_base", ctypes.c_int64),
        ("target_logits", _P), ("draft_logits", _P), ("draft_tokens", _P),
        ("temperature", _P), ("fanout_host", _P), ("draft_bonus_logits", _P),
        ("keys_out", _P), ("num_accepted", _P), ("out_tokens", _P), ("tau", _P),
        ("hit", _P), ("status", _P),
    ]


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib():
    """Load (building first if the sources are newer) libsdverify.so."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if _build.stale():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError("libsdverify.so is missing; run __graft_entry__.build()")
            L = ctypes.CDLL(_build.LIB)
            i32, u64, sz = ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
            L.sd_verify_workspace_size.argtypes = [i32, i32]
            L.sd_verify_workspace_size.restype = sz
            L.sd_verify.argtypes = [ctypes.POINTER(VerifyArgs), _P]
            L.sd_verify.restype = ctypes.c_int
            L.sd_verify_noalloc.argtypes = [ctypes.POINTER(VerifyArgs), _P]
            L.sd_verify_noalloc.restype = ctypes.c_int
            L.sd_outcome_predict.argtypes = [i32, i32, i32, ctypes.c_int, _P, _P, _P, _P, _P, _P,
                                             _P, _P]
            L.sd_outcome_predict.restype = ctypes.c_int
            L.sd_compact.argtypes = [i32, i32, _P, _P, _P, _P, _P, _P]
            L.sd_compact.restype = ctypes.c_int
            L.sd_d3d_pack.argtypes = [i32, i32, i32, _P, _P, _P, _P, i32, _P, _P, _P, _P]
            L.sd_d3d_pack.restype = ctypes.c_int
            L.sd_ngram_draft.argtypes = [i32, i32, i32, i32, i32, _P, _P, _P, _P, _P, _P, _P]
            L.sd_ngram_draft.restype = ctypes.c_int
            L.sd_kv_rollback.argtypes = [i32, i32, i32, i32, _P, _P, _P, _P, _P, _P, _P]
            L.sd_kv_rollback.restype = ctypes.c_int
            L.sd_uniforms.argtypes = [u64, i32, _P, _P, _P, _P, _P]
            L.sd_uniforms.restype = ctypes.c_int
            L.sd_vshard_stats_bytes.argtypes = [i32, i32]
            L.sd_vshard_stats_bytes.restype = sz
            L.sd_vshard_mass_bytes.argtypes = [i32]
            L.sd_vshard_mass_bytes.restype = sz
            L.sd_vshard_stats.argtypes = [ctypes.POINTER(VShardArgs), _P, _P]
            L.sd_vshard_stats.restype = ctypes.c_int
            L.sd_vshard_mass.argtypes = [ctypes.POINTER(VShardArgs), _P, _P, _P]
            L.sd_vshard_mass.restype = ctypes.c_int
            L.sd_vshard_pick.argtypes = [ctypes.POINTER(VShardArgs), _P, _P, _P]
            L.sd_vshard_pick.restype = ctypes.c_int
            L.sd_verify_args_size.argtypes = []
            L.sd_verify_args_size.restype = sz
            if L.sd_verify_args_size() != ctypes.sizeof(VerifyArgs):
                raise RuntimeError("sd_verify_args layout differs between library and binding")
            L.sd_version.argtypes = []
            L.sd_version.restype = ctypes.c_char_p
            L.sd_status_string.argtypes = [ctypes.c_int]
            L.sd_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


class SDError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != SD_OK:
        raise SDError(f"{what} failed: {lib().sd_status_string(rc).decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _on_stream(fn):
    """Run a wrapper with `stream` (when given) as the current stream, so the
    tensors it allocates belong to the stream its launches are queued on: the
    caching allocator reuses a freed block in the order of the stream that
    allocated it, and a block allocated on another stream could still be in
    use by work queued there."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        s = kwargs.get("stream")
        if s is None:
            return fn(*args, **kwargs)
        with torch.cuda.stream(s):
            return fn(*args, **kwargs)
    return call


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SD_F32
    if t.dtype == torch.bfloat16:
        return SD_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, dtype=None, shape=None, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


_ws = {}
_ws_lock = threading.Lock()


def workspace_bytes(B: int, K: int) -> int:
    return int(lib().sd_verify_workspace_size(B, K))


def workspace(B: int, K: int, device=None, stream=None):
    """Scratch for sd_verify's split launch (sd_verify_workspace_size bytes:
    one 96-byte record per row piece), cached per (device, stream) so that
    calls ordered on one stream share it; None for sizes out of range."""
    need = workspace_bytes(B, K)
    if need == 0:
        return None
    device = torch.device(device if device is not None else torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    with _ws_lock:
        buf = _ws.get(key)
        if buf is None or buf.numel() < need:
            with torch.cuda.stream(s):   # the block belongs to the stream it serves
                buf = torch.zeros(need, dtype=torch.uint8, device=device)
            _ws[key] = buf
    return buf


@dataclass
class VerifyResult:
    num_accepted: torch.Tensor      # [B] int32
    out_tokens: torch.Tensor        # [B][K+1] int32
    tau: torch.Tensor               # [B] int32
    hit: torch.Tensor | None = None           # [B] uint8
    offsets: torch.Tensor | None = None       # [B+1] int32
    packed: torch.Tensor | None = None        # [B*(K+1)] int32
    keys: torch.Tensor | None = None          # [B][n_keys][2] int32
    accept_ratio: torch.Tensor | None = None  # [B][K] float32
    p_draft: torch.Tensor | None = None
    q_draft: torch.Tensor | None = None
    target_argmax: torch.Tensor | None = None  # [B][K+1] int32
    status: torch.Tensor | None = None        # [1] int32


def alloc_outputs(B, K, device, *, hit=False, compact=False, stats=False, n_keys=0,
                  status=True) -> VerifyResult:
    e = lambda *s, dt=torch.int32: torch.empty(s, dtype=dt, device=device)
    r = VerifyResult(e(B), e(B, K + 1), e(B))
    if hit or n_keys:
        r.hit = e(B, dt=torch.uint8)
    if compact:
        r.offsets, r.packed = e(B + 1), e(max(B * (K + 1), 1))
    if n_keys:
        r.keys = e(B, n_keys, 2)
    if stats:
        r.accept_ratio = torch.full((B, K), float("nan"), device=device)
        r.p_draft = torch.full((B, K), float("nan"), device=device)
        r.q_draft = torch.full((B, K), float("nan"), device=device)
        r.target_argmax = e(B, K + 1)
    if status:
        r.status = torch.zeros(1, dtype=torch.int32, device=device)
    return r


@_on_stream
def verify(target, draft, tokens, temperature, seed: int, *, row_base: int = 0,
           cache_keys=None, fanout=None, draft_bonus=None, compact: bool = False,
           stats: bool = False, check_finite: bool = False, out: VerifyResult | None = None,
           ws=None, stream=None) -> VerifyResult:
    """Run sd_verify on the current (or given) stream.

    target [B][K+1][V], draft [B][K][V] (float32 or bfloat16, CUDA,
    contiguous), tokens [B][K] int32, temperature [B] float32.  cache_keys:
    [B][n_keys][2] int32 keys to test the outcome against.  fanout ([K+1]
    ints) asks for the outcome-prediction keys to be built in the same pass
    (draft_bonus [B][V] optional).  compact=True also packs the tokens.
    check_finite=True sets SD_FLAG_CHECK_FINITE: a sequence whose rows hold
    NaN or +inf (or only -inf) comes back invalid with SD_STATUS_NONFINITE."""
    _need(target, "target")
    dev = target.device
    B, K1, V = target.shape
    K = K1 - 1
    dt = _dtype_code(target)
    if K > 0:
        _need(draft, "draft", target.dtype, (B, K, V), dev)
        _need(tokens, "tokens", torch.int32, (B, K), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    n_keys = 0
    flags = 0
    fan_arr = None
    if fanout is not None:
        fanout = [int(f) for f in fanout]
        if len(fanout) != K + 1:
            raise ValueError("fanout needs K+1 entries")
        n_keys = sum(fanout)
        fan_arr = (ctypes.c_int32 * (K + 1))(*fanout)
        flags |= SD_FLAG_PREDICT
        if draft_bonus is not None:
            _need(draft_bonus, "draft_bonus", target.dtype, (B, V), dev)
    if cache_keys is not None:
        _need(cache_keys, "cache_keys", torch.int32, None, dev)
        if cache_keys.dim() != 3 or cache_keys.shape[0] != B or cache_keys.shape[2] != 2:
            raise ValueError("cache_keys must be [B][n_keys][2]")
    if compact:
        flags |= SD_FLAG_COMPACT
    if check_finite:
        flags |= SD_FLAG_CHECK_FINITE
    r = out or alloc_outputs(B, K, dev, hit=cache_keys is not None or n_keys > 0,
                             compact=compact, stats=stats, n_keys=n_keys)
    w = ws if ws is not None else workspace(B, K, dev, stream)
    a = VerifyArgs()
    a.B, a.K, a.V, a.dtype, a.flags = B, K, V, dt, flags
    a.seed, a.row_base = int(seed) & (2 ** 64 - 1), int(row_base)
    a.target_logits, a.draft_logits = target.data_ptr(), (draft.data_ptr() if K > 0 else None)
    a.draft_tokens = tokens.data_ptr() if K > 0 else None
    a.temperature = temperature.data_ptr()
    if cache_keys is not None:
        a.cache_keys, a.n_keys = cache_keys.data_ptr(), cache_keys.shape[1]
    if fan_arr is not None:
        a.fanout_host = ctypes.cast(fan_arr, ctypes.c_void_p)
        a.draft_bonus_logits = draft_bonus.data_ptr() if draft_bonus is not None else None
        a.keys_out = r.keys.data_ptr() if n_keys else None
    a.num_accepted, a.out_tokens, a.tau = (r.num_accepted.data_ptr(), r.out_tokens.data_ptr(),
                                          r.tau.data_ptr())
    a.hit = r.hit.data_ptr() if r.hit is not None else None
    if compact:
        a.offsets, a.packed = r.offsets.data_ptr(), r.packed.data_ptr()
    if r.accept_ratio is not None:
        a.accept_ratio, a.p_draft, a.q_draft = (r.accept_ratio.data_ptr(), r.p_draft.data_ptr(),
                                                r.q_draft.data_ptr())
        a.target_argmax = r.target_argmax.data_ptr()
    a.status = r.status.data_ptr() if r.status is not None else None
    if w is not None:
        a.workspace, a.workspace_bytes = w.data_ptr(), w.numel()
    _check(lib().sd_verify(ctypes.byref(a), _stream(dev, stream)), "sd_verify")
    return r


@_on_stream
def outcome_predict(draft, tokens, fanout, draft_bonus=None, *, keys=None, status=None,
                    stream=None) -> torch.Tensor:
    """Speculation-cache keys [B][sum(fanout)][2] (position, token)."""
    _need(draft, "draft")
    B, K, V = draft.shape
    dev = draft.device
    dt = _dtype_code(draft)
    _need(tokens, "tokens", torch.int32, (B, K), dev)
    fanout = [int(f) for f in fanout]
    if len(fanout) != K + 1:
        raise ValueError("fanout needs K+1 entries")
    if draft_bonus is not None:
        _need(draft_bonus, "draft_bonus", draft.dtype, (B, V), dev)
    n = sum(fanout)
    if keys is None:
        keys = torch.empty((B, n, 2), dtype=torch.int32, device=dev)
    fan_arr = (ctypes.c_int32 * (K + 1))(*fanout)
    n_out = ctypes.c_int32(0)
    _check(lib().sd_outcome_predict(B, K, V, dt, _ptr(draft), _ptr(tokens), _ptr(draft_bonus),
                                    ctypes.cast(fan_arr, ctypes.c_void_p), _ptr(keys),
                                    ctypes.cast(ctypes.byref(n_out), ctypes.c_void_p),
                                    _ptr(status), _stream(dev, stream)), "sd_outcome_predict")
    assert n_out.value == n
    return keys


@_on_stream
def d3d_pack(keys, draft_tokens, anchor, anchor_pos, mask_token: int, *, out=None,
             stream=None):
    """The drafter's packed next pass: (tokens, positions) [B][1+n_keys][K+1]
    and ctx [B][1+n_keys] from keys [B][n_keys][2], draft_tokens [B][K],
    anchor [B] and anchor_pos [B] (int32, CUDA)."""
    _need(keys, "keys", torch.int32)
    B, n_keys, two = keys.shape
    if two != 2:
        raise ValueError("keys must be [B][n_keys][2]")
    dev = keys.device
    _need(draft_tokens, "draft_tokens", torch.int32, None, dev)
    if draft_tokens.dim() != 2 or draft_tokens.shape[0] != B:
        raise ValueError("draft_tokens must be [B][K]")
    K = draft_tokens.shape[1]
    _need(anchor, "anchor", torch.int32, (B,), dev)
    _need(anchor_pos, "anchor_pos", torch.int32, (B,), dev)
    if out is None:
        out = (torch.empty((B, 1 + n_keys, K + 1), dtype=torch.int32, device=dev),
               torch.empty((B, 1 + n_keys, K + 1), dtype=torch.int32, device=dev),
               torch.empty((B, 1 + n_keys), dtype=torch.int32, device=dev))
    t, p, c = out
    _check(lib().sd_d3d_pack(B, K, n_keys, _ptr(keys), _ptr(draft_tokens), _ptr(anchor),
                             _ptr(anchor_pos), int(mask_token), _ptr(t), _ptr(p), _ptr(c),
                             _stream(dev, stream)), "sd_d3d_pack")
    return t, p, c


@_on_stream
def ngram_draft(history, lengths, K: int, n_max: int, n_min: int, *, out=None, stream=None):
    """Prompt-lookup drafts (drafts [B][K], count, match_pos, match_n [B])
    from history [B][L] and lengths [B] (int32, CUDA)."""
    _need(history, "history", torch.int32)
    B, L = history.shape
    dev = history.device
    _need(lengths, "lengths", torch.int32, (B,), dev)
    if out is None:
        e = lambda *s: torch.empty(s, dtype=torch.int32, device=dev)
        out = (e(B, K), e(B), e(B), e(B))
    d, c, p, n = out
    _check(lib().sd_ngram_draft(B, L, K, n_max, n_min, _ptr(history), _ptr(lengths), _ptr(d),
                                _ptr(c), _ptr(p), _ptr(n), _stream(dev, stream)),
           "sd_ngram_draft")
    return d, c, p, n


@_on_stream
def kv_rollback(block_table, kv_len, tau, page_size: int, appended: int, *, out=None,
                stream=None):
    """Roll row caches back after a round: block_table [B][max_pages] is
    updated in place; returns (new_len [B], freed [B*max_pages], free_offsets
    [B+1]) -- freed[:free_offsets[-1]] are the freed page ids."""
    _need(block_table, "block_table", torch.int32)
    B, max_pages = block_table.shape
    dev = block_table.device
    _need(kv_len, "kv_len", torch.int32, (B,), dev)
    _need(tau, "tau", torch.int32, (B,), dev)
    if out is None:
        e = lambda *s: torch.empty(s, dtype=torch.int32, device=dev)
        out = (e(B), e(max(B * max_pages, 1)), e(B + 1))
    n, f, o = out
    _check(lib().sd_kv_rollback(B, page_size, max_pages, appended, _ptr(kv_len), _ptr(tau),
                                _ptr(block_table), _ptr(n), _ptr(f), _ptr(o),
                                _stream(dev, stream)), "sd_kv_rollback")
    return n, f, o


@_on_stream
def compact(out_tokens, tau, *, offsets=None, packed=None, status=None, stream=None):
    """(offsets [B+1], packed [B*(K+1)]) from out_tokens [B][K+1] and tau [B]."""
    _need(out_tokens, "out_tokens", torch.int32)
    B, K1 = out_tokens.shape
    dev = out_tokens.device
    _need(tau, "tau", torch.int32, (B,), dev)
    if offsets is None:
        offsets = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if packed is None:
        packed = torch.empty(max(B * K1, 1), dtype=torch.int32, device=dev)
    _check(lib().sd_compact(B, K1 - 1, _ptr(out_tokens), _ptr(tau), _ptr(offsets), _ptr(packed),
                            _ptr(status), _stream(dev, stream)), "sd_compact")
    return offsets, packed


@_on_stream
def uniforms(seed: int, row, pos, slot, *, stream=None) -> torch.Tensor:
    """The verify step's uniforms u(seed, row, pos, slot) (float64)."""
    _need(row, "row", torch.int32)
    dev = row.device
    _need(pos, "pos", torch.int32, tuple(row.shape), dev)
    _need(slot, "slot", torch.int32, tuple(row.shape), dev)
    out = torch.empty(row.shape, dtype=torch.float64, device=dev)
    _check(lib().sd_uniforms(int(seed) & (2 ** 64 - 1), row.numel(), _ptr(row), _ptr(pos),
                             _ptr(slot), _ptr(out), _stream(dev, stream)), "sd_uniforms")
    return out


# ------------------------------------------------ vocabulary-sharded verify --
def vshard_bounds(V: int, S: int):
    """Even split of [0, V) into S shards in order: list of (v0, vs)."""
    base, extra = divmod(V, S)
    out, v0 = [], 0
    for s in range(S):
        vs = base + (1 if s < extra else 0)
        out.append((v0, vs))
        v0 += vs
    return out


def _vshard_args(target_s, draft_s, tokens, temperature, seed, *, S, shard, v0, V, row_base,
                 fanout, draft_bonus_s, check_finite, out, status, fan_arr):
    B, K1, vs = target_s.shape
    K = K1 - 1
    a = VShardArgs()
    a.B, a.K, a.V, a.S, a.shard, a.v0, a.vs = B, K, V, S, shard, v0, vs
    a.dtype = _dtype_code(target_s)
    a.flags = (SD_FLAG_PREDICT if fanout is not None else 0) | (
        SD_FLAG_CHECK_FINITE if check_finite else 0)
    a.seed, a.row_base = int(seed) & (2 ** 64 - 1), int(row_base)
    a.target_logits = target_s.data_ptr()
    a.draft_logits = draft_s.data_ptr() if K > 0 else None
    a.draft_tokens = tokens.data_ptr() if K > 0 else None
    a.temperature = temperature.data_ptr()
    if fan_arr is not None:
        a.fanout_host = ctypes.cast(fan_arr, ctypes.c_void_p)
        a.draft_bonus_logits = draft_bonus_s.data_ptr() if draft_bonus_s is not None else None
    if out is not None:
        a.keys_out = out.keys.data_ptr() if out.keys is not None else None
        a.num_accepted, a.out_tokens, a.tau = (out.num_accepted.data_ptr(),
                                              out.out_tokens.data_ptr(), out.tau.data_ptr())
        a.hit = out.hit.data_ptr() if out.hit is not None else None
    a.status = status.data_ptr() if status is not None else None
    return a


@_on_stream
def vshard_stats(target_s, draft_s, tokens, temperature, seed, *, S, shard, v0, V, row_base=0,
                 fanout=None, draft_bonus_s=None, check_finite=False, stats=None, stream=None):
    """sd_vshard_stats: this shard's stats block (uint8 tensor)."""
    _need(target_s, "target_s")
    dev = target_s.device
    B, K1, vs = target_s.shape
    K = K1 - 1
    if K > 0:
        _need(draft_s, "draft_s", target_s.dtype, (B, K, vs), dev)
        _need(tokens, "tokens", torch.int32, (B, K), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    fan_arr = None
    if fanout is not None:
        fan_arr = (ctypes.c_int32 * (K + 1))(*[int(f) for f in fanout])
        if draft_bonus_s is not None:
            _need(draft_bonus_s, "draft_bonus_s", target_s.dtype, (B, vs), dev)
    n = int(lib().sd_vshard_stats_bytes(B, K))
    if stats is None:
        stats = torch.empty(n, dtype=torch.uint8, device=dev)
    a = _vshard_args(target_s, draft_s, tokens, temperature, seed, S=S, shard=shard, v0=v0, V=V,
                     row_base=row_base, fanout=fanout, draft_bonus_s=draft_bonus_s,
                     check_finite=check_finite, out=None, status=None, fan_arr=fan_arr)
    _check(lib().sd_vshard_stats(ctypes.byref(a), _ptr(stats), _stream(dev, stream)),
           "sd_vshard_stats")
    return stats


@_on_stream
def vshard_mass(target_s, draft_s, tokens, temperature, seed, stats_all, *, S, shard, v0, V,
                row_base=0, fanout=None, draft_bonus_s=None, check_finite=False, mass=None,
                stream=None):
    """sd_vshard_mass: this shard's mass block (uint8 tensor) from all
    shards' stats blocks (stats_all: S blocks in shard order)."""
    dev = target_s.device
    B, K1, _ = target_s.shape
    K = K1 - 1
    fan_arr = (ctypes.c_int32 * (K + 1))(*[int(f) for f in fanout]) if fanout is not None else None
    if mass is None:
        mass = torch.empty(int(lib().sd_vshard_mass_bytes(B)), dtype=torch.uint8, device=dev)
    a = _vshard_args(target_s, draft_s, tokens, temperature, seed, S=S, shard=shard, v0=v0, V=V,
                     row_base=row_base, fanout=fanout, draft_bonus_s=draft_bonus_s,
                     check_finite=check_finite, out=None, status=None, fan_arr=fan_arr)
    _check(lib().sd_vshard_mass(ctypes.byref(a), _ptr(stats_all), _ptr(mass),
                                _stream(dev, stream)), "sd_vshard_mass")
    return mass


@_on_stream
def vshard_pick(target_s, draft_s, tokens, temperature, seed, stats_all, mass_all, out, *, S,
                shard, v0, V, row_base=0, fanout=None, draft_bonus_s=None, check_finite=False,
                stream=None):
    """sd_vshard_pick into `out` (a VerifyResult whose out_tokens start at -1
    and hit at 0)."""
    dev = target_s.device
    K = target_s.shape[1] - 1
    fan_arr = (ctypes.c_int32 * (K + 1))(*[int(f) for f in fanout]) if fanout is not None else None
    a = _vshard_args(target_s, draft_s, tokens, temperature, seed, S=S, shard=shard, v0=v0, V=V,
                     row_base=row_base, fanout=fanout, draft_bonus_s=draft_bonus_s,
                     check_finite=check_finite, out=out, status=out.status, fan_arr=fan_arr)
    _check(lib().sd_vshard_pick(ctypes.byref(a), _ptr(stats_all), _ptr(mass_all),
                                _stream(dev, stream)), "sd_vshard_pick")
    return out


def _vshard_out(B, K, device, n_keys):
    r = alloc_outputs(B, K, device, hit=True, n_keys=n_keys)
    r.out_tokens.fill_(-1)
    r.hit.fill_(0)
    return r


@_on_stream
def verify_vsharded(targets, drafts, tokens, temperature, seed, *, V, fanout=None,
                    draft_bonus=None, check_finite=False, row_base=0, stream=None):
    """The sharded verify on one device: targets / drafts / draft_bonus are
    lists of the S shards' column blocks ([B][K+1][vs_s] ...) in vocabulary
    order.  The exchanges are the stats and mass blocks laid side by side,
    and the shards' picks writing one set of outputs."""
    S = len(targets)
    B, K1, _ = targets[0].shape
    K = K1 - 1
    dev = targets[0].device
    v0s = [0]
    for t in targets[:-1]:
        v0s.append(v0s[-1] + t.shape[2])
    if v0s[-1] + targets[-1].shape[2] != V:
        raise ValueError("the shards must cover [0, V) in order")
    nst = int(lib().sd_vshard_stats_bytes(B, K))
    nma = int(lib().sd_vshard_mass_bytes(B))
    stats_all = torch.empty(S * nst, dtype=torch.uint8, device=dev)
    mass_all = torch.empty(S * max(nma, 16), dtype=torch.uint8, device=dev)
    bon = draft_bonus if draft_bonus is not None else [None] * S
    kw = dict(V=V, row_base=row_base, fanout=fanout, check_finite=check_finite, stream=stream)
    for s in range(S):
        vshard_stats(targets[s], drafts[s], tokens, temperature, seed, S=S, shard=s, v0=v0s[s],
                     draft_bonus_s=bon[s], stats=stats_all[s * nst:(s + 1) * nst], **kw)
    for s in range(S):
        vshard_mass(targets[s], drafts[s], tokens, temperature, seed, stats_all, S=S, shard=s,
                    v0=v0s[s], draft_bonus_s=bon[s], mass=mass_all[s * nma:(s + 1) * nma], **kw)
    out = _vshard_out(B, K, dev, sum(fanout) if fanout is not None else 0)
    for s in range(S):
        vshard_pick(targets[s], drafts[s], tokens, temperature, seed, stats_all, mass_all, out,
                    S=S, shard=s, v0=v0s[s], draft_bonus_s=bon[s], **kw)
    return out


def verify_vsharded_dist(target_s, draft_s, tokens, temperature, seed, *, V, v0, group=None,
                         fanout=None, draft_bonus_s=None, check_finite=False, row_base=0,
                         phases=None):
    """The sharded verify across the ranks of a torch.distributed group, one
    shard per rank (rank order = vocabulary order; v0 = this rank's first
    column).  Exchanges: all-gather of the stats blocks and of the mass
    blocks, all-reduce (max) of the outputs.  `phases` (stats, mass, pick)
    replaces the library calls (tests of the exchange logic)."""
    import torch.distributed as dist
    S = dist.get_world_size(group)
    shard = dist.get_rank(group)
    B, K1, _ = target_s.shape
    K = K1 - 1
    f_stats, f_mass, f_pick = phases or (vshard_stats, vshard_mass, vshard_pick)
    kw = dict(S=S, shard=shard, v0=v0, V=V, row_base=row_base, fanout=fanout,
              draft_bonus_s=draft_bonus_s, check_finite=check_finite)
    def gather(x):   # the S blocks side by side, in rank order
        parts = [torch.empty_like(x) for _ in range(S)]
        dist.all_gather(parts, x, group=group)
        return torch.cat(parts)

    st = f_stats(target_s, draft_s, tokens, temperature, seed, **kw)
    stats_all = gather(st)
    ma = f_mass(target_s, draft_s, tokens, temperature, seed, stats_all, **kw)
    mass_all = gather(ma)
    out = _vshard_out(B, K, target_s.device, sum(fanout) if fanout is not None else 0)
    f_pick(target_s, draft_s, tokens, temperature, seed, stats_all, mass_all, out, **kw)
    for t in (out.out_tokens, out.hit):
        if t is not None:
            x = t.to(torch.int32) if t.dtype != torch.int32 else t
            dist.all_reduce(x, op=dist.ReduceOp.MAX, group=group)
            if x is not t:
                t.copy_(x)
    if out.status is not None:
        dist.all_reduce(out.status, op=dist.ReduceOp.MAX, group=group)
    return out


def version() -> str:
    return lib().sd_version().decode()
