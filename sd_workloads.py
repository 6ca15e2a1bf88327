"""Seeded synthetic inputs for the speculative-decoding verify step.

Shared by the tests, the benchmark and the package smoke check.  This module
holds none of the verify method's arithmetic: it only draws logits with the
shapes, scales and structure of the five workloads below, and plays the
drafter by drawing the draft tokens from the draft distribution with the
Gumbel-max trick (argmax of logits / T plus Gumbel noise; argmax of the
logits for greedy rows).

Workloads (logit layouts: target [B][K+1][V], draft [B][K][V], row-major):

  small     B=1,  K=4, V=32000,  fp32, target ~ N(0, 2^2) iid, draft = target
            + N(0, 0.5^2); half the rounds greedy (T=0), half at T=1.
  peaked    B=8,  K=5, V=128256, bf16, target ~ N(0, 3^2) with 20 distinct
            "peak" ids per position boosted by +8; draft = target + N(0, 1);
            T=0.7.
  zipf      B=64, K=8, V=151936, bf16, target logit_i = -1.1 ln(pi(i)+1) +
            N(0, 0.3^2) for a seeded permutation pi per position row; draft
            the same pi with exponent -0.9 and N(0, 0.5^2) noise; T=1.
  saguaro   B=32, K=6, V=128256, bf16 as "peaked"; plus a draft row for the
            bonus position (target row K + N(0,1)) and the outcome-prediction
            fan-out 4,3,2,1,1,1,1 (F=4).
  mix       B=256, K=4, V=128256, bf16 as "zipf"; per-row temperature drawn
            uniformly from {0, 0.6, 1.0}.
  d3d       B=16, K=15, V=151936, bf16 as "zipf", greedy (T=0); a block of
            16 tokens (anchor + 15 drafts), keys for rejection positions
            1..11 with two candidates each plus the all-accepted bonus key
            (fan-out 2 x 11, 0 x 4, 1: 23 keys, a 24-block pack of 384
            tokens), a bonus draft row, a seeded anchor token and anchor
            position per row for the pack, mask token id V, and the target's
            paged KV cache for the rollback (anchor position + K + 1 entries,
            16-entry pages, a random page table).

The per-round uniforms of the verify step are keyed by ``seed`` (one per
round), which the generator returns with the inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

WORKLOADS = {
    "small": dict(B=1, K=4, V=32000, dtype="f32", kind="normal", sigma=2.0, draft_sigma=0.5,
                  temperature="alt01", rounds=200, base_seed=1235),
    "peaked": dict(B=8, K=5, V=128256, dtype="bf16", kind="peaked", sigma=3.0, draft_sigma=1.0,
                   peaks=20, peak_boost=8.0, temperature=0.7, rounds=10000, base_seed=1236),
    "zipf": dict(B=64, K=8, V=151936, dtype="bf16", kind="zipf", temperature=1.0, rounds=2000,
                 base_seed=1237),
    "saguaro": dict(B=32, K=6, V=128256, dtype="bf16", kind="peaked", sigma=3.0, draft_sigma=1.0,
                    peaks=20, peak_boost=8.0, temperature=0.7, rounds=5000, base_seed=1238,
                    bonus_row=True, fanout=[4, 3, 2, 1, 1, 1, 1]),
    "mix": dict(B=256, K=4, V=128256, dtype="bf16", kind="zipf", temperature="mix",
                rounds=1000, base_seed=1239),
    "d3d": dict(B=16, K=15, V=151936, dtype="bf16", kind="zipf", temperature=0.0,
                rounds=2000, base_seed=1240, bonus_row=True,
                fanout=[2] * 11 + [0] * 4 + [1], pack=True),
}
# the workloads in the order they are usually listed (1..5)
ORDER = ["small", "peaked", "zipf", "saguaro", "mix", "d3d"]


@dataclass
class Inputs:
    target: torch.Tensor            # [B][K+1][V] float32 or bfloat16
    draft: torch.Tensor             # [B][K][V]
    tokens: torch.Tensor            # [B][K] int32
    temperature: torch.Tensor       # [B] float32
    seed: int                       # key of the verify step's uniforms
    draft_bonus: torch.Tensor | None = None   # [B][V] or None
    fanout: list | None = None      # [K+1] or None
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.target.shape[0]

    @property
    def K(self):
        return self.target.shape[1] - 1

    @property
    def V(self):
        return self.target.shape[2]

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)
        return Inputs(mv(self.target), mv(self.draft), mv(self.tokens), mv(self.temperature),
                      self.seed, mv(self.draft_bonus), self.fanout, dict(self.meta))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed & 0x7FFFFFFFFFFFFFFF)
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _draw_tokens(draft_f32: torch.Tensor, temps: torch.Tensor, g, device) -> torch.Tensor:
    """The drafter: d ~ softmax(draft / T) via Gumbel-max for T > 0, argmax
    for T == 0.  draft_f32: [B][K][V] (the logits as the verifier sees
    them), temps: [B]."""
    B, K, V = draft_f32.shape
    if K == 0:
        return torch.zeros((B, 0), dtype=torch.int32, device=device)
    out = torch.empty((B, K), dtype=torch.int64, device=device)
    chunk = max(1, (1 << 24) // max(1, K * V))   # bound the temporary size
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        x = draft_f32[b0:b1]
        t = temps[b0:b1].view(-1, 1, 1)
        u = torch.rand(x.shape, generator=g, device=device, dtype=torch.float32)
        u = u.clamp_(min=1e-12, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        sampled = torch.argmax(x / torch.where(t > 0, t, torch.ones_like(t)) + gumbel, dim=-1)
        greedy = torch.argmax(x, dim=-1)
        out[b0:b1] = torch.where(t.view(-1, 1) > 0, sampled, greedy)
    return out.to(torch.int32)


def _temps(spec, B, g, device, round_idx=0):
    if isinstance(spec, (int, float)):
        return torch.full((B,), float(spec), dtype=torch.float32, device=device)
    if spec == "alt01":          # whole batch greedy on even rounds, T=1 on odd
        return torch.full((B,), 0.0 if round_idx % 2 == 0 else 1.0, dtype=torch.float32,
                          device=device)
    if spec == "mix":
        choice = torch.randint(0, 3, (B,), generator=g, device=device)
        table = torch.tensor([0.0, 0.6, 1.0], dtype=torch.float32, device=device)
        return table[choice]
    t = torch.as_tensor(spec, dtype=torch.float32)
    assert t.numel() == B
    return t.to(device)


def synth(B, K, V, dtype="bf16", *, kind="normal", temperature=1.0, seed=1, device="cpu",
          round_idx=0, sigma=2.0, draft_sigma=0.5, peaks=0, peak_boost=8.0,
          zipf_target=1.1, zipf_draft=0.9, zipf_noise_target=0.3, zipf_noise_draft=0.5,
          bonus_row=False, fanout=None, **_unused) -> Inputs:
    """Draw one round of inputs.  ``kind`` is "normal", "peaked" or "zipf";
    ``temperature`` a number, a length-B list, "alt01" or "mix"."""
    device = torch.device(device)
    g = _gen(seed * 1000003 + round_idx, device)
    temps = _temps(temperature, B, g, device, round_idx)
    if kind in ("normal", "peaked"):
        t = _normal((B, K + 1, V), g, device) * sigma
        if peaks > 0:
            ids = torch.rand((B, K + 1, V), generator=g, device=device).topk(peaks, dim=-1).indices
            t.scatter_add_(-1, ids, torch.full(ids.shape, peak_boost, device=device))
        d = t[:, :K, :] + _normal((B, K, V), g, device) * draft_sigma
        bonus = t[:, K, :] + _normal((B, V), g, device) * draft_sigma if bonus_row else None
    elif kind == "zipf":
        perm = torch.rand((B, K + 1, V), generator=g, device=device).argsort(dim=-1)
        logrank = torch.log(perm.to(torch.float32) + 1.0)
        del perm
        t = -zipf_target * logrank + _normal((B, K + 1, V), g, device) * zipf_noise_target
        d = -zipf_draft * logrank[:, :K, :] + _normal((B, K, V), g, device) * zipf_noise_draft
        bonus = (-zipf_draft * logrank[:, K, :] + _normal((B, V), g, device) * zipf_noise_draft
                 if bonus_row else None)
        del logrank
    else:
        raise ValueError(kind)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = t.to(tdt).contiguous()
    d = d.to(tdt).contiguous()
    if bonus is not None:
        bonus = bonus.to(tdt).contiguous()
    tokens = _draw_tokens(d.to(torch.float32), temps, g, device)
    # one key per round for the verify step's uniforms
    useed = (seed * 0x9E3779B97F4A7C15 + round_idx * 0xBF58476D1CE4E5B9 + 1) % (1 << 64)
    return Inputs(t, d, tokens.contiguous(), temps.contiguous(), int(useed), bonus,
                  list(fanout) if fanout is not None else None,
                  dict(kind=kind, dtype=dtype, round=round_idx))


def workload(name: str, round_idx: int = 0, device="cpu", **override) -> Inputs:
    spec = dict(WORKLOADS[name])
    spec.update(override)
    spec.pop("rounds")
    base = spec.pop("base_seed")
    pack = spec.pop("pack", False)
    inp = synth(seed=base, round_idx=round_idx, device=device, **spec)
    if pack:  # the settled token before each block and its position
        g = _gen(base * 7919 + round_idx, "cpu")
        inp.meta["anchor"] = torch.randint(0, inp.V, (inp.B,), generator=g,
                                           dtype=torch.int32).to(device)
        inp.meta["anchor_pos"] = torch.randint(0, 8192, (inp.B,), generator=g,
                                               dtype=torch.int32).to(device)
        inp.meta["mask_token"] = inp.V
        # the target's paged KV cache: entries up to the anchor, plus the
        # anchor and the K drafts the verify pass appended; 16-entry pages
        page = 16
        max_pages = (8192 + inp.K + 1 + page - 1) // page
        inp.meta["page_size"] = page
        inp.meta["kv_len"] = (inp.meta["anchor_pos"] + inp.K + 1).contiguous()
        inp.meta["block_table"] = torch.randperm(inp.B * max_pages, generator=g).to(
            torch.int32).reshape(inp.B, max_pages).to(device)
    return inp


def logit_bytes(inp: Inputs, algorithmic: bool = True, with_bonus: bool = True) -> int:
    """Bytes of logits one verify round must read.  algorithmic=True skips
    the draft rows of greedy rows (they are never needed); False gives the
    (2K+1) V B formula."""
    B, K, V = inp.B, inp.K, inp.V
    es = inp.target.element_size()
    if algorithmic:
        # sampled rows read every draft row; greedy rows only those with keys
        n_sampled = int((inp.temperature > 0).sum().item())
        fan = inp.fanout or [0] * (K + 1)
        n_keyed = sum(1 for j in range(K) if fan[j] > 0)
        n = B * (K + 1) * V + n_sampled * K * V + (B - n_sampled) * n_keyed * V
    else:
        n = (2 * K + 1) * V * B
    if with_bonus and inp.draft_bonus is not None:
        n += B * V
    return n * es


def to_numpy_logits(t: torch.Tensor):
    """Host numpy view of logits: float32 stays float32, bf16 becomes its
    raw bits as uint16 (the oracle widens them exactly)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


# ------------------------------------------------------- n-gram drafting --
# Token histories for the prompt-lookup drafter: each row is its prompt and
# output so far, built from a per-row phrase book (48 phrases of 8-32 random
# tokens, drawn with replacement) mixed with fresh random text (30 % of the
# pieces, 1-7 tokens), so that the text's ending usually recurs earlier, as
# in the summarising, editing and quoting the pages name.  One seeded base
# set is drawn on the host; round r maps every token t to (t + 7919 r) mod V
# (a bijection: every match stays where it was, the bytes differ).
NGRAM = dict(B=256, L=16384, V=128256, K=4, n_max=4, n_min=1, base_seed=1241)


def ngram_base(B, L, V, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    lens = rng.integers(L // 4, L + 1, size=B).astype(np.int32)
    h = rng.integers(0, V, size=(B, L)).astype(np.int32)   # padding past the length: random
    for b in range(B):
        book = [rng.integers(0, V, size=int(rng.integers(8, 33))) for _ in range(48)]
        pieces, total = [], 0
        while total < lens[b]:
            if rng.random() < 0.3:
                p = rng.integers(0, V, size=int(rng.integers(1, 8)))
            else:
                p = book[int(rng.integers(0, 48))]
            pieces.append(p)
            total += len(p)
        h[b, :lens[b]] = np.concatenate(pieces)[:lens[b]]
    return h, lens


def ngram_inputs(round_idx=0, device="cpu", **override):
    """(history [B][L] int32, lengths [B] int32, spec) of one drafting round."""
    spec = dict(NGRAM)
    spec.update(override)
    h, lens = ngram_base(spec["B"], spec["L"], spec["V"], spec["base_seed"])
    h = torch.from_numpy(h).to(device)
    if round_idx:
        h = ((h.to(torch.int64) + 7919 * round_idx) % spec["V"]).to(torch.int32)
    return h.contiguous(), torch.from_numpy(lens).to(device), spec
