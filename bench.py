#!/usr/bin/env python
"""Benchmark of one conditional draft-tree building round (DominoTree).

Metric: draft trees built per second (whole job) and ms per round, on the
Qwen3-8B-shaped serving batch: 32 independent requests, V = 151936, d = 4096,
d_s = 1024, r = 256, B = 16 (D = 15), M = 64, k = 8, node budget N = 64.
Inputs are seeded synthetic tensors of those shapes (dt_workloads).

A step is one dt_build_trees call: top-M over the base logits, the per-depth
projection and the conditional best-first search with tree and mask emission,
from device-resident inputs to device-resident outputs. The prepared weight
table (dt_prepare_weights) is built once, before timing, like any weight
layout transform; its time is reported as config.prepare_ms.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run; every rank builds its own batch of
32 requests (replicas, weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft trees built/sec and µs per tree-build round (Qwen3-8B shape, batch 32)"
UNIT = "trees/s"
CFG = 3
L2_FLUSH_BYTES = 256 << 20          # > 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--spec", type=int, default=0, help="speculative expansions per step (0=default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--no-verify", action="store_true",
                    help="skip the verify-side tree-attention leg")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the Domino chain-decoding leg")
    ap.add_argument("--no-marginal", action="store_true",
                    help="skip the marginal-score (W2 = 0 ablation) leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the legs of the other configurations (0, 1, 2, 4)")
    ap.add_argument("--flags", type=int, default=0,
                    help="dt_options flags (DT_OPT_* bits of include/dt.h)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained",
                                                      d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                sm_max_mhz=2070.0, source="fallback")


class Clocks:
    """nvidia-smi sampler running during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(wl, reqs, threads, keep=False):
    """Seconds the oracle takes for `reqs` on `threads` host threads (and the
    trees when `keep`)."""
    import oracle
    t0 = time.perf_counter()
    trees = oracle.build_trees(wl, reqs, threads=threads, mask=True, topm_out=keep)
    dt_s = time.perf_counter() - t0
    return (dt_s, dict(zip(reqs, trees))) if keep else dt_s


def source_sha(path):
    import hashlib
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(profile, source):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
    kernel from a committed ncu summary, or None when the summary is missing
    or was taken on another version of the kernel's source file."""
    path = os.path.join(ROOT, "profiles", profile)
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    if d.get("source_sha") != source_sha(os.path.join(ROOT, source)):
        return None
    return d.get("dram_bytes_per_launch")


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def parity_block(wl, g, refs):
    """Oracle parity of the GPU trees `g` over the requests of `refs` (the
    build's bar: top-M bit-exact, topology exact outside near ties within 1e-4,
    scores within 1e-5): counts, or the first violation as a string."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import _parity
    try:
        return _parity.parity_summary(wl, g, refs)
    except AssertionError as e:
        return {"violation": str(e)[:300]}


def algorithmic_counts(wl, out_tokens, out_depths):
    """Per-round algorithmic bytes of each phase and useful GEMM flops of the
    search, from the trees actually built (expansions = root + popped nodes
    below depth D that are not the N-th pop)."""
    import numpy as np
    B, D, V, d, ds, r, M, N = wl.batch, wl.D, wl.V, wl.d, wl.d_s, wl.r, wl.M, wl.N
    w = 2 if wl.wdtype == "bf16" else 4
    topm_bytes = B * D * V * 4 + B * D * M * 8
    proj_bytes = B * D * d * 4 + r * d * w + B * D * r * 4
    proj_flops = 2 * B * D * r * d
    n_exp = 0
    depths_touched = 0
    for b in range(B):
        dep = out_depths[b]
        n = int((out_tokens[b] >= 0).sum())
        idx = np.arange(n)
        exp_nodes = 1 + int(((dep[1:n] < D) & (idx[1:] < N)).sum())
        n_exp += exp_nodes
        depths_touched += len(set((dep[:n][(dep[:n] < D) & (idx < N)] + 1).tolist()))
    search_bytes = ((3 * ds * ds + r * ds) * w + n_exp * 3 * ds * 4
                    + depths_touched * (M * r * w + r * 4 + M * 8)
                    + B * (N + 1) * (16 + N + 1))
    search_flops = n_exp * 2 * (3 * ds + r) * ds
    return dict(topm_bytes=topm_bytes, proj_bytes=proj_bytes, proj_flops=proj_flops,
                search_bytes=search_bytes, search_flops=search_flops, expansions=n_exp)


def run_reference(args, rank):
    """The oracle, as it stands, on the host cores: each step a bounded sample."""
    if rank != 0:
        return
    import dt_workloads as W
    wl = W.make_workload(CFG)
    cores = os.cpu_count() or 1
    reqs = list(range(min(wl.batch, cores)))
    for _ in range(args.warmup):
        oracle_sample(wl, reqs[:1], 1)
    total = sum(oracle_sample(wl, reqs, cores) for _ in range(args.steps))
    value = len(reqs) * args.steps / total
    sample = f"{len(reqs)} of the 32 requests per step, {cores} threads, warm-up {args.warmup} single requests"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "qwen3-8b-b32: V=151936 d=4096 d_s=1024 r=256 D=15 M=64 k=8 N=64 batch=32",
                       "parallelism": "oracle on host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(ms, torch, dist, world, dev):
    """The slowest rank's time: every rank ends with the maximum of the ranks'
    `ms` (replicas only, so this reduction of the timer is the one collective)."""
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, batch, K, total_ms):
    """Units all ranks processed per second: world x batch per step, K steps."""
    return world * batch * K / (total_ms / 1000.0)


def e2e_leg(args, tb, wl, dt, np, torch, dist, world, dev, flush, st, K, Wm):
    """Same metric through dt_build_trees_host: pinned host inputs in and the
    trees copied back inside the timed region. The page-locked base logits are
    mapped, so by default the top-M scan reads them in place over the host link;
    the same leg with OPT_STAGE_HOST_LOGITS (a 292 MB copy first) is timed
    beside it."""
    host_ws = torch.empty(dt.host_workspace_bytes(tb.dims, tb.opt), dtype=torch.uint8, device=dev)
    pin = lambda a, tt: torch.from_numpy(np.ascontiguousarray(a, dtype=tt)).pin_memory()
    hin = dict(base_logits=pin(wl.base_logits, np.float32), H=pin(wl.H, np.float32),
               state0=pin(wl.state0, np.float32), anchor_tok=pin(wl.anchor, np.int32),
               temperature=pin(wl.temperature, np.float32))
    hout = dt.alloc_outputs(tb.dims, "cpu", pin=True)
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values() if v is not None)

    def timed(flags):
        opt = dt.options(tb.opt.spec_width, flags=tb.opt.flags | flags)

        def e2e_step():
            dt.build_trees_host(tb.dims, tb.w, tb.prepared, hin["base_logits"], hin["H"],
                                hin["state0"], hin["anchor_tok"], hin["temperature"], host_ws,
                                hout, opt)
        for _ in range(Wm):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = 0.0
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(K):
            flush.fill_(i & 0xff)
            ea.record(st)
            e2e_step()
            eb.record(st)
            eb.synchronize()
            e_ms += ea.elapsed_time(eb)
        ok = bool((hout["status"] == 0).all())
        return whole_job_rate(world, wl.batch, K, max_over_ranks(e_ms, torch, dist, world, dev)), ok

    staged_value, ok_staged = timed(dt.OPT_STAGE_HOST_LOGITS)
    e2e_value, ok_e2e = timed(0)
    extra = {"logits": ("read in place (mapped page-locked memory)"
                        if dt.mapped_host_pointer(hin["base_logits"]) is not None
                        else "copied (not mapped)"),
             "staged_value": staged_value, "staged_ok": ok_staged}
    return e2e_value, h2d, d2h, ok_e2e and ok_staged, extra


def marginal_leg(wl, dt, torch, dev, flush, st, K, Wm, inp):
    """The marginal-score builder (the conditionality ablation) on the same
    workload and inputs: top-M, then one tree kernel; no weights. Device-timed
    like the main leg (phase events, L2 flushed before every round)."""
    mb = dt.MarginalTreeBuilder(dt.dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N,
                                           wl.batch), device=dev)
    out = dt.alloc_outputs(mb.dims, dev)
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(dt.NUM_PHASE_EVENTS)]
          for _ in range(K)]
    for evs in ph:
        for e in evs:
            e.record(st)
    run = lambda opt=None: mb.run(inp["base_logits"], inp["anchor_tok"], inp["temperature"],
                                  out=out, opt=opt)
    for _ in range(Wm):
        flush.fill_(1)
        run()
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xff)
        run(dt.options(0, ph[i], dt.OPT_MARGINAL))
    torch.cuda.synchronize()
    per = [ph[i][0].elapsed_time(ph[i][3]) for i in range(K)]
    topm = [ph[i][0].elapsed_time(ph[i][1]) for i in range(K)]
    tree = [ph[i][2].elapsed_time(ph[i][3]) for i in range(K)]
    ms = statistics.mean(per)
    return {"us_per_round": 1000.0 * ms, "trees_per_s": wl.batch / (ms * 1e-3),
            "topm_us": 1000.0 * statistics.mean(topm),
            "tree_kernel_us": 1000.0 * statistics.mean(tree),
            "kernel_launches_per_round": dt.kernel_launches(mb.dims, dt.F32, mb.opt),
            "ok": bool((out["status"] == 0).all().item())}


def chain_leg(wl, W, dt, torch, dev, flush, st, K, Wm, inp, greedy):
    """Domino chain decoding (dt_decode_chains) on the same workload: D draft
    tokens per request with the correction over the whole vocabulary, sampled
    at the workload's temperatures with seeded uniform draws, or greedy.
    Device-timed per round (L2 flushed before each); block 0's phase split."""
    import numpy as np
    dec = dt.ChainDecoder(dt.dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N, wl.batch),
                          TreeWeights.get(), device=dev)
    u = torch.from_numpy(W.chain_uniforms(wl.batch, wl.D, seed=3)).to(dev)
    T = torch.zeros_like(inp["temperature"]) if greedy else inp["temperature"]
    out = dec.alloc_outputs()
    run = lambda: dec.run(inp["base_logits"], inp["H"], inp["state0"], inp["anchor_tok"], T, u,
                          out=out)
    for _ in range(Wm):
        flush.fill_(1)
        run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xff)
        ev[i][0].record(st)
        run()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    # block 0's phase times of the last round (the control block is zeroed per call)
    t_ns = dec.workspace[32:32 + 8 * 4].view(torch.int64).cpu().tolist()
    split = {k: v / 1000.0 for k, v in zip(["state_gemm", "vocab_gemm", "token_and_gru",
                                            "barriers"], t_ns)}
    flops = 2.0 * wl.V * wl.r * wl.batch * wl.D        # useful W2 h products of one round
    pk = peaks()
    vocab_s = split["vocab_gemm"] * 1e-6 if split["vocab_gemm"] > 0 else None
    return {"us_per_round": 1000.0 * ms, "chains_per_s": wl.batch / (ms * 1e-3),
            "draft_tokens_per_s": wl.batch * wl.D / (ms * 1e-3),
            "block0_us_per_round": split,
            "vocab_gemm_useful_tflops": (flops / vocab_s / 1e12) if vocab_s else None,
            "base_logit_gbs": wl.base_logits.nbytes / (ms * 1e-3) / 1e9,
            "base_logit_hbm_frac": wl.base_logits.nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "kernel_launches_per_round": dt.chain_kernel_launches(dec.dims),
            "ok": bool((out["status"] == 0).all().item()),
            "sampling": "greedy (T = 0)" if greedy else "inverse CDF at the workload's T"}


def verify_leg(W, dt, torch, np, dev, flush, st, K, Wm, mask, pk):
    """Verify-side tree attention (dt_tree_attention) over the trees of the main
    leg: Qwen3-8B attention shape (32 query heads, 8 key/value heads, dh 128),
    one layer, prefix cache padded to 1024 keys with lengths in [512, 1024],
    synthetic bf16 Q/K/V. Device-timed per call, L2 flushed before each."""
    B, n1 = mask.shape[0], mask.shape[1]
    H, Hkv, P, dh = 32, 8, 1024, 128
    q, k, v, plen = W.verify_inputs(B, H, Hkv, n1, P, dh, seed=3, min_prefix=512)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    qd, kd, vd, pd = t(q), t(k), t(v), torch.from_numpy(plen).to(dev)
    out = torch.empty((B, H, n1, dh), dtype=torch.float32, device=dev)
    for _ in range(Wm):
        flush.fill_(1)
        dt.tree_attention(qd, kd, vd, mask, pd, out=out)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xff)
        ev[i][0].record(st)
        dt.tree_attention(qd, kd, vd, mask, pd, out=out)
        ev[i][1].record(st)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    seen = mask.to(torch.int64).sum(-1).cpu().numpy() + plen[:, None]   # visible keys per row
    # useful flops: q.k and p.v over the visible keys, 2 flops per product (the
    # tensor cores also compute masked keys of a chunk, S twice and P.V in two
    # bf16 terms: about 4x as many issued)
    flops = 4.0 * dh * H * float(seen.sum())
    peak = pk["bf16_tflops"]
    ach = flops / (ms * 1e-3) / 1e12
    return {"us_per_layer": 1000.0 * ms, "shape": f"batch {B}, H {H}, Hkv {Hkv}, n1 {n1}, "
            f"prefix <= {P}, dh {dh}", "roofline": {"bound": "tensor", "achieved": ach,
            "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
            "peak_kind": f"bf16 dense burst, {pk['source']}"},
            "finite": bool(torch.isfinite(out).all().item())}


def adaptive_leg(dt, torch, dev, st, K, out, N, c_fixed=1.0, c_node=1.0 / 256):
    """CondAdaptive (dt_adaptive_budget) on copies of the main leg's trees: the
    kept node counts under a round cost c_fixed + c_node n (a verification pass
    whose cost grows by 1/256 of its fixed cost per tree node; the pages give no
    cost figures) and how often the rule runs to the full budget."""
    ms = []
    for _ in range(K):
        o = {k: (v.clone() if v is not None else None) for k, v in out.items()}
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        counts = dt.adaptive_budget(o, N, c_fixed, c_node)
        b.record(st)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    c = counts.cpu()
    return {"us_per_call": 1000.0 * statistics.mean(ms), "c_fixed": c_fixed, "c_node": c_node,
            "mean_nodes_kept": float(c.float().mean()), "budget": N,
            "share_at_full_budget": float((c == N).float().mean())}


def config_leg(c, wl, dt, torch, np, dev, flush, st, K, Wm, with_parity, oracle_reqs):
    """One configuration of the build: device weights and inputs, Wm warm-up
    and K timed rounds (CUDA events on the stream, L2 flushed before each),
    round time, trees/s, the round's algorithmic HBM bytes against the measured
    copy peak, the search GEMM flops against the measured bf16 peak, status of
    every request and, when asked (bench rank 0 at N = 1), oracle parity on
    `oracle_reqs`."""
    tb = dt.TreeBuilder.from_numpy(wl, device=dev)
    inp = tb.inputs_to_device(wl)
    out = dt.alloc_outputs(tb.dims, dev)
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(dt.NUM_PHASE_EVENTS)]
          for _ in range(K)]
    for evs in ph:
        for e in evs:
            e.record(st)
    for _ in range(Wm):
        flush.fill_(1)
        tb.run(**inp, out=out)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xff)
        tb.run(**inp, out=out, opt=dt.options(0, ph[i]))
    torch.cuda.synchronize()
    per = sorted(ph[i][0].elapsed_time(ph[i][3]) for i in range(K))
    # the search starts after the later of [1] (top-M) and [2] (projection)
    search = statistics.median(
        ph[i][0].elapsed_time(ph[i][3])
        - max(ph[i][0].elapsed_time(ph[i][1]), ph[i][0].elapsed_time(ph[i][2]))
        for i in range(K))
    ms = statistics.median(per)
    o = {k: v.cpu().numpy() for k, v in out.items() if v is not None}
    cnt = algorithmic_counts(wl, o["tokens"], o["depths"])
    pk = peaks()
    rb = cnt["topm_bytes"] + cnt["proj_bytes"] + cnt["search_bytes"]
    ctrl = tb.workspace[:32].view(torch.int32).cpu().tolist()
    leg = {"workload": f"{wl.name}: V={wl.V} d={wl.d} d_s={wl.d_s} r={wl.r} D={wl.D} M={wl.M} "
                       f"k={wl.k} N={wl.N} batch={wl.batch} {wl.wdtype}",
           "us_per_round_median": 1000.0 * ms, "us_per_round_min": 1000.0 * per[0],
           "trees_per_s": wl.batch / (ms * 1e-3), "rounds": K,
           "search_us_median": 1000.0 * search, "search_steps": ctrl[4],
           "round_algorithmic_bytes": rb,
           "round_hbm_gbs": rb / (ms * 1e-3) / 1e9,
           "round_hbm_frac": rb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
           "search_gemm_tflops": cnt["search_flops"] / (search * 1e-3) / 1e12,
           "search_tensor_frac_of_sustained": cnt["search_flops"] / (search * 1e-3) / 1e12
           / pk["bf16_tflops_sustained"],
           "all_status_ok": bool((o["status"] == 0).all())}
    if with_parity and oracle_reqs:
        cores = os.cpu_count() or 1
        secs, refs = oracle_sample(wl, oracle_reqs, cores, keep=True)
        leg["parity"] = parity_block(wl, o, refs)
        leg["parity"]["requests"] = f"{len(oracle_reqs)} of {wl.batch}"
        leg["oracle_s"] = secs
    del tb, inp, out
    torch.cuda.empty_cache()
    return leg


class TreeWeights:
    """The device weights of the main leg, shared with the chain leg."""
    w = None

    @classmethod
    def get(cls):
        return cls.w


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import numpy as np
    import torch
    import torch.distributed as dist

    import conditional_draft_tree_gb300 as dt
    import dt_workloads as W
    from conditional_draft_tree_gb300 import build as dtbuild

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        dtbuild.build()
    if world > 1:
        dist.barrier()
    # every configuration's seeded inputs, generated concurrently on the host
    other_cfgs = [] if (args.no_configs or rank != 0) else [0, 1, 2, 4]
    from concurrent.futures import ThreadPoolExecutor
    gen = ThreadPoolExecutor(max_workers=1 + len(other_cfgs))
    wl_f = {c: gen.submit(W.make_workload, c) for c in [CFG] + other_cfgs}
    wl = wl_f[CFG].result()
    dev = torch.device("cuda", local)

    t0 = time.perf_counter()
    tb = dt.TreeBuilder.from_numpy(wl, spec_width=args.spec, device=dev, flags=args.flags)
    TreeWeights.w = tb.w
    torch.cuda.synchronize()
    prep = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prep[0].record()
    dt.prepare_weights(tb.dims, tb.w, tb.prepared)
    prep[1].record()
    torch.cuda.synchronize()
    prepare_ms = prep[0].elapsed_time(prep[1])
    inp = tb.inputs_to_device(wl)
    out = dt.alloc_outputs(tb.dims, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    K, Wm = args.steps, max(3, args.warmup)
    st = torch.cuda.current_stream()

    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(dt.NUM_PHASE_EVENTS)]
          for _ in range(K)]
    for evs in ph:            # torch creates the CUDA event at its first record
        for e in evs:
            e.record(st)
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for _ in range(Wm):
        flush.fill_(1)
        tb.run(**inp, out=out)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk = Clocks(local)
    clk.start()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xff)                       # L2 flush outside the timed interval
        tb.run(**inp, out=out, opt=dt.options(args.spec, ph[i], args.flags))
        ends[i].record(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = clk.stop()
    ctrl = tb.workspace[:32].view(torch.int32).cpu().tolist()   # search counters of the last round
    search_steps, search_expansions = ctrl[4], ctrl[5]
    t_ns = tb.workspace[32:32 + 8 * 32].view(torch.int64).cpu().tolist()
    search_split_us = {k: t_ns[i] / 1000.0 for i, k in enumerate(
        ["gemm", "barrier_after_gemm", "request_score", "request_gather_children",
         "request_pop_select", "request_gru", "gh_sums_after", "barrier_after_request",
         "gru_wait_parent_gh", "gemm_mma", "gemm_epilogue", None, "gemm_wait_mma", "score_h",
         "score_candidates", "score_softmax_sort"]) if k}
    gemm_cycles = dict(zip(["wait_free_buffer", "wait_landed_copy", "copy_issue", "mma_issue",
                            "pop_iterations", "pop_cycles", "select_iterations",
                            "select_cycles"], t_ns[24:32]))
    per = [ph[i][0].elapsed_time(ph[i][3]) for i in range(K)]
    # [1] after the top-M, [2] after the projection: with bf16 weights the
    # projection runs first ([2] before [1]); with fp32 weights beside the top-M
    t1 = [ph[i][0].elapsed_time(ph[i][1]) for i in range(K)]
    t2 = [ph[i][0].elapsed_time(ph[i][2]) for i in range(K)]
    t3 = [ph[i][0].elapsed_time(ph[i][3]) for i in range(K)]
    proj_first = statistics.mean(t2) <= statistics.mean(t1)
    if proj_first:
        projection_ms = t2
        topm_ms = [a - b for a, b in zip(t1, t2)]
        proj_ms = [0.0] * K
        search_ms = [c - a for a, c in zip(t1, t3)]
    else:
        projection_ms = [0.0] * K
        topm_ms = t1
        proj_ms = [b - a for a, b in zip(t1, t2)]
        search_ms = [c - b for b, c in zip(t2, t3)]
    total_ms = max_over_ranks(sum(per), torch, dist, world, dev)
    value = whole_job_rate(world, wl.batch, K, total_ms)
    launches_per_round = dt.kernel_launches(tb.dims, tb.w.wdtype, tb.opt)

    # end to end through the host-buffer entry point: pinned inputs in, results out
    e2e_value, h2d, d2h, ok_e2e, e2e_extra = None, 0, 0, None, {}
    if not args.no_e2e:
        e2e_value, h2d, d2h, ok_e2e, e2e_extra = e2e_leg(args, tb, wl, dt, np, torch, dist, world, dev, flush,
                                               st, K, Wm)
    marginal = None
    if not args.no_marginal:
        marginal = marginal_leg(wl, dt, torch, dev, flush, st, K, Wm, inp)
    adaptive = adaptive_leg(dt, torch, dev, st, K, out, wl.N)
    verify = None
    if not args.no_verify:
        verify = verify_leg(W, dt, torch, np, dev, flush, st, K, Wm, out["mask"], peaks())
    chain = None
    if not args.no_chain:
        chain = {"sampled": chain_leg(wl, W, dt, torch, dev, flush, st, K, Wm, inp, False),
                 "greedy": chain_leg(wl, W, dt, torch, dev, flush, st, K, Wm, inp, True)}
    # the other configurations (rank 0): timing, rooflines, oracle parity
    configs = {}
    for c in other_cfgs:
        wlc = wl_f[c].result()
        reqs = list(range(wlc.batch)) if wlc.batch <= 32 else list(range(0, wlc.batch, 8))
        configs[f"config{c}"] = config_leg(c, wlc, dt, torch, np, dev, flush, st, K, Wm,
                                           world == 1 and not args.no_cpu_baseline, reqs)
        wl_f[c] = None
    gen.shutdown()
    if rank == 0:
        o = {k: v.cpu().numpy() for k, v in out.items() if v is not None}
        cnt = algorithmic_counts(wl, o["tokens"], o["depths"])
        pk = peaks()
        # phase events: the projection when it runs first (tensor cores), the
        # top-M, the rest of the projection when it runs beside the top-M
        # (CUDA cores, fp32 weights), the search
        phases = {"projection": statistics.mean(projection_ms), "topm": statistics.mean(topm_ms),
                  "projection_tail": statistics.mean(proj_ms),
                  "search": statistics.mean(search_ms)}
        # dominant kernel: the search. Its arithmetic is the recurrent GEMM on
        # the tensor cores (bf16 operands, fp32-exact products of three bf16
        # terms); achieved = algorithmic GEMM flops (2 (3 d_s + r) d_s per
        # expansion) / search time, against the measured dense bf16 burst peak.
        ach = cnt["search_flops"] / (phases["search"] * 1e-3) / 1e12
        traffic = ncu_traffic("chain_kernel_qwen3-8b-b32.json",
                              "conditional_draft_tree_gb300/csrc/dt_chain.cu")
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "traffic": traffic,
                "algorithmic_bytes": cnt["search_bytes"],
                "traffic_over_algorithmic": (traffic / cnt["search_bytes"]
                                             if traffic is not None else None),
                "kernel": "dt::chain_kernel",
                "peak_kind": f"bf16 dense burst, {pk['source']}"}
        ach_t = cnt["topm_bytes"] / (phases["topm"] * 1e-3) / 1e9
        roof_topm = {"bound": "hbm", "achieved": ach_t, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": ach_t / pk["hbm_gbs"], "kernel": "dt::topm_kernel",
                     "note": ("the projection runs before it on the tensor cores"
                              if proj_first else
                              "the projection GEMM runs concurrently on a side stream")}
        round_bytes = cnt["topm_bytes"] + cnt["proj_bytes"] + cnt["search_bytes"]
        status_ok = bool((o["status"] == 0).all())
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "qwen3-8b-b32: V=151936 d=4096 d_s=1024 r=256 D=15 M=64 k=8 N=64 batch=32",
                       "us_per_round": 1000.0 * total_ms / K, "global_batch": world * wl.batch,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed (256 MB write) before every timed round",
                       "spec_width": tb.opt.spec_width or 8, "prepare_ms": prepare_ms,
                       "phases_ms": phases, "expansions_per_round": cnt["expansions"],
                       "search_steps": search_steps, "search_expansions": search_expansions,
                       "search_block0_us": search_split_us,
                       "search_block0_gemm_issuer_cycles": gemm_cycles,
                       "roofline_topm": roof_topm,
                       "marginal_mode": marginal,
                       "chain_decoding": chain,
                       "verify_tree_attention": verify,
                       "cond_adaptive": adaptive,
                       "all_status_ok": status_ok,
                       "other_configs": configs or None,
                       "round_algorithmic_bytes": round_bytes,
                       "round_hbm_frac": round_bytes / (total_ms / K * 1e-3) / 1e9 / pk["hbm_gbs"],
                       "peaks": pk["source"], "wall_s": wall},
            "roofline": roof,
            "e2e": ({"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h, "ok": ok_e2e, **e2e_extra}
                    if e2e_value is not None else None),
            "gpu_launches": launches_per_round * K,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            cores = os.cpu_count() or 1
            reqs = list(range(wl.batch))
            secs, refs = oracle_sample(wl, reqs, cores, keep=True)
            secs1 = oracle_sample(wl, [0], 1)
            line["cpu_baseline"] = {"value": len(reqs) / secs, "unit": UNIT, "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"all {len(reqs)} requests of one round, {cores} threads",
                                    "single_thread": {"value": 1.0 / secs1, "unit": UNIT,
                                                      "sample": "request 0, 1 thread"},
                                    "cpu_model": cpu_model()}
            # the timed trees of the last round against the oracle's (every request)
            line["config"]["parity"] = parity_block(wl, o, refs)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
