"""Comparison of the CUDA path's results with the CPU oracle's.

Rules (from the method's tolerance statement):
  * greedy rows (T == 0): tau, num_accepted and every emitted token exact;
  * sampled rows: exact unless the oracle flags a decision whose uniform lies
    within 1e-6 of the accept threshold or of an edge of the chosen CDF bin
    (guard_pos >= 0); such rows are compared exactly up to the guarded
    position only, and counted;
  * probabilities p(d), q(d) and p/q within 1e-5 relative;
  * argmax, keys, hit, offsets and packed tokens exact.
"""
from __future__ import annotations

import numpy as np

RTOL_PROB = 1e-5


def compare_verify(gpu, o, temps, *, check_stats=True, rows=None):
    """gpu: VerifyResult (already on host as numpy via .cpu()) or dict of
    numpy arrays; o: oracle.verify(...) output for the same rows."""
    g = {k: (v.cpu().numpy() if hasattr(v, "cpu") else v)
         for k, v in (gpu.__dict__ if hasattr(gpu, "__dict__") else gpu).items() if v is not None}
    temps = np.asarray(temps, np.float32)
    if rows is not None:
        g = {k: (v[rows] if k not in ("status", "offsets", "packed") else v) for k, v in g.items()}
    B = o["tau"].shape[0]
    K = o["out_tokens"].shape[1] - 1
    stats = dict(rows=B, positions=B * max(K, 1), greedy=0, sampled=0, guarded=0,
                 guarded_mismatch=0, mismatch_outside_guard=0, invalid=0)
    bad = []
    for b in range(B):
        T = float(temps[b])
        valid = o["tau"][b] > 0
        same = (g["tau"][b] == o["tau"][b] and g["num_accepted"][b] == o["num_accepted"][b]
                and np.array_equal(g["out_tokens"][b], o["out_tokens"][b]))
        if "hit" in g and "hit" in o and g.get("hit") is not None:
            same = same and (g["hit"][b] == o["hit"][b])
        if not valid:
            stats["invalid"] += 1
            if not same:
                bad.append((b, "invalid row differs"))
            continue
        if T == 0.0:
            stats["greedy"] += 1
            if not same:
                bad.append((b, "greedy row differs", g["out_tokens"][b].tolist(),
                            o["out_tokens"][b].tolist()))
            continue
        stats["sampled"] += 1
        gp = int(o["guard_pos"][b])
        if gp < 0:
            if not same:
                stats["mismatch_outside_guard"] += 1
                bad.append((b, "sampled row differs outside the guard band",
                            dict(T=T, gpu=g["out_tokens"][b].tolist(),
                                 oracle=o["out_tokens"][b].tolist(),
                                 ratio=(o.get("ratio")[b].tolist()
                                        if o.get("ratio") is not None else None),
                                 gpu_ratio=(g["accept_ratio"][b].tolist()
                                            if "accept_ratio" in g else None))))
        else:
            stats["guarded"] += 1
            if not same:
                stats["guarded_mismatch"] += 1
            if not np.array_equal(g["out_tokens"][b][:gp], o["out_tokens"][b][:gp]):
                bad.append((b, "tokens before the guarded position differ"))
    if check_stats and "target_argmax" in g and "argmax" in o:
        for b in range(B):
            if o["tau"][b] == 0:
                continue
            if not np.array_equal(g["target_argmax"][b], o["argmax"][b]):
                bad.append((b, "argmax differs"))
            if float(temps[b]) > 0 and K > 0:
                for name, oname in (("p_draft", "p_tok"), ("q_draft", "q_tok"),
                                    ("accept_ratio", "ratio")):
                    gv = g[name][b].astype(np.float64)
                    ov = o[oname][b]
                    fin = np.isfinite(ov) & (ov > 1e-30)
                    if not np.allclose(gv[fin], ov[fin], rtol=RTOL_PROB, atol=0):
                        err = np.max(np.abs(gv[fin] / ov[fin] - 1))
                        bad.append((b, f"{name} rel err {err:.2e}"))
    return stats, bad
