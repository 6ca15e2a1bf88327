"""Run a few verify rounds of one synthetic workload (for profilers).

    python profile_case.py WORKLOAD [ROUNDS]

Two input sets of the workload alternate; every round is the verify step
(plus the packing launch, and for the D3D workload the drafter pack and the
KV rollback).  Prints the mean tau of the last round.
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import torch  # noqa: E402

import sd_workloads as W  # noqa: E402
import speculative_decoding_verification_logits_gb300 as sd  # noqa: E402


def main():
    name = sys.argv[1] if len(sys.argv) > 1 else "saguaro"
    n = int(sys.argv[2]) if len(sys.argv) > 2 else 4
    dev = torch.device("cuda:0")
    if name == "ngram":   # prompt-lookup drafting rounds over two history sets
        sets = [W.ngram_inputs(r, device=dev) for r in range(2)]
        out = None
        for i in range(n):
            h, lens, s = sets[i % 2]
            out = sd.ngram_draft(h, lens, s["K"], s["n_max"], s["n_min"])
        torch.cuda.synchronize()
        print("ok", float((out[3] >= 0).float().mean().item()))
        return
    spec = W.WORKLOADS[name]
    fan = spec.get("fanout")
    pool = [W.workload(name, round_idx=i, device=dev) for i in range(2)]
    r = None
    for i in range(n):
        p = pool[i % 2]
        r = sd.verify(p.target, p.draft, p.tokens, p.temperature, p.seed + i, fanout=fan,
                      draft_bonus=p.draft_bonus, compact=True)
        if "anchor" in p.meta:   # the D3D round: the drafter pack and the KV rollback
            m = p.meta
            sd.d3d_pack(r.keys, p.tokens, m["anchor"], m["anchor_pos"], m["mask_token"])
            sd.kv_rollback(m["block_table"], m["kv_len"], r.tau, m["page_size"], p.K + 1)
    torch.cuda.synchronize()
    print("ok", r.tau.float().mean().item())
    # logit bytes each input set's round must read (greedy rows skip their
    # draft rows), for the profile summaries' ratio of DRAM to algorithmic bytes
    print("alg_bytes", *[W.logit_bytes(p, algorithmic=True, with_bonus=fan is not None)
                         for p in pool])


if __name__ == "__main__":
    main()
