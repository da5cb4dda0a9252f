"""Fixed single-GPU workloads for kernel profiling and timing.

    python -m conditional_draft_tree_gb300.profile_cases topm  [--reps R] [--cfg C]
        top-M of a workload's base logits (Qwen3-8B batch 32 by default:
        480 rows x 151936 fp32, 292 MB) through dt_select_topm_noalloc. Its
        kernel is dt_build_trees' top-M kernel, and the launch shape is the same
        while the row segments' partial lists fit in the static scratch (true
        for this workload; a larger one, such as the batch-128 M = 256 stress
        configuration, falls back to one block per row segment). Only the
        logits and the outputs live on the device.
    python -m conditional_draft_tree_gb300.profile_cases round [--reps R] [--cfg C] [--flags F]
        R whole dt_build_trees rounds of the workload (weights, prepared table
        and workspace on the device: about 3.5 GB for the default workload);
        F = dt_options flags (default 0).
    python -m conditional_draft_tree_gb300.profile_cases marginal [--reps R] [--cfg C]
        R marginal-score rounds (DT_OPT_MARGINAL): top-M and the marginal tree
        kernel, no weights on the device.
    python -m conditional_draft_tree_gb300.profile_cases verify [--reps R] [--cfg C]
        R launches of one tree-attention layer over the workload's trees
        (32 query heads, 8 key/value heads, dh 128, prefix cache of 1024 keys
        with lengths in [512, 1024]; synthetic bf16 Q/K/V).
    python -m conditional_draft_tree_gb300.profile_cases chain [--reps R] [--cfg C] [--greedy]
        R Domino chain-decoding rounds (dt_decode_chains) of the workload,
        sampled at its temperatures with seeded uniform draws, or greedy: one
        projection launch and one decoding launch per round.

Each case does one untimed launch first, then R timed ones (CUDA events on the
current stream, L2 flushed by a 256 MB write before each), and prints one line
with the mean time. Run it under ncu with -k / -s / -c to capture one launch.
"""
from __future__ import annotations

import argparse

import torch

import conditional_draft_tree_gb300 as dt
import dt_workloads as W

L2_FLUSH_BYTES = 256 << 20


def _timed(fn, reps, dev):
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fn()
    torch.cuda.synchronize()
    ms = []
    for i in range(reps):
        flush.fill_(i & 0xff)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    return sum(ms) / len(ms)


def case_topm(cfg, reps, dev):
    wl = W.make_workload(cfg)
    logits = torch.from_numpy(wl.base_logits).to(dev)
    topm = torch.empty(wl.batch, wl.D, wl.M, dtype=torch.int32, device=dev)
    status = torch.empty(wl.batch, dtype=torch.int32, device=dev)

    def run():
        rc = dt.select_topm_noalloc(logits, wl.M, topm, status)
        if rc != dt.OK:
            raise dt.DtError(dt.status_string(rc))

    ms = _timed(run, reps, dev)
    gbs = logits.numel() * 4 / (ms * 1e-3) / 1e9
    print(f"topm {wl.name}: rows={wl.batch * wl.D} V={wl.V} M={wl.M} "
          f"mean_us={1000 * ms:.1f} GB/s={gbs:.0f}")


def case_round(cfg, reps, dev, flags=0):
    wl = W.make_workload(cfg)
    tb = dt.TreeBuilder.from_numpy(wl, device=dev, flags=flags)
    inp = tb.inputs_to_device(wl)
    out = dt.alloc_outputs(tb.dims, dev)
    ms = _timed(lambda: tb.run(**inp, out=out), reps, dev)
    print(f"round {wl.name}: batch={wl.batch} mean_us={1000 * ms:.1f} "
          f"trees/s={wl.batch / (ms * 1e-3):.0f}")


def case_chain(cfg, reps, dev, greedy=False):
    wl = W.make_workload(cfg)
    dec = dt.ChainDecoder.from_numpy(wl, device=dev)
    inp = dec.inputs_to_device(wl, W.chain_uniforms(wl.batch, wl.D, seed=cfg))
    if greedy:
        inp["temperature"] = torch.zeros_like(inp["temperature"])
    out = dec.alloc_outputs()
    ms = _timed(lambda: dec.run(**inp, out=out), reps, dev)
    if not bool((out["status"] == 0).all()):
        raise dt.DtError("chain decoding reported a non-OK status")
    print(f"chain {wl.name}: batch={wl.batch} D={wl.D} mean_us={1000 * ms:.1f} "
          f"chains/s={wl.batch / (ms * 1e-3):.0f}")


def case_marginal(cfg, reps, dev):
    wl = W.make_workload(cfg)
    mb = dt.MarginalTreeBuilder.from_workload(wl, device=dev)
    inp = mb.inputs_to_device(wl)
    out = dt.alloc_outputs(mb.dims, dev)
    ms = _timed(lambda: mb.run(**inp, out=out), reps, dev)
    print(f"marginal {wl.name}: batch={wl.batch} mean_us={1000 * ms:.1f} "
          f"trees/s={wl.batch / (ms * 1e-3):.0f}")


def case_verify(cfg, reps, dev):
    import numpy as np
    wl = W.make_workload(cfg)
    tb = dt.TreeBuilder.from_numpy(wl, device=dev)
    trees = tb.run(**tb.inputs_to_device(wl))
    q, k, v, plen = W.verify_inputs(wl.batch, 32, 8, wl.N + 1, 1024, 128, seed=cfg,
                                    min_prefix=512)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    qd, kd, vd, pd = t(q), t(k), t(v), torch.from_numpy(plen).to(dev)
    out = torch.empty((wl.batch, 32, wl.N + 1, 128), dtype=torch.float32, device=dev)
    ms = _timed(lambda: dt.tree_attention(qd, kd, vd, trees["mask"], pd, out=out), reps, dev)
    print(f"verify {wl.name}: batch={wl.batch} n1={wl.N + 1} mean_us={1000 * ms:.1f}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["topm", "round", "chain", "marginal", "verify"])
    ap.add_argument("--greedy", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--cfg", type=int, default=3)
    ap.add_argument("--flags", type=int, default=0)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    from conditional_draft_tree_gb300 import build
    build.build()
    if args.case == "round":
        case_round(args.cfg, args.reps, dev, args.flags)
    elif args.case == "chain":
        case_chain(args.cfg, args.reps, dev, args.greedy)
    elif args.case == "marginal":
        case_marginal(args.cfg, args.reps, dev)
    elif args.case == "verify":
        case_verify(args.cfg, args.reps, dev)
    else:
        case_topm(args.cfg, args.reps, dev)


if __name__ == "__main__":
    main()
