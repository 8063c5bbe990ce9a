"""Benchmark: batched DDTree draft-tree rounds per second on GB300.

Workload (default): 64 in-flight requests, 15 draft depths, vocabulary
151,936, budget 32 (K = 32, P = 33 tree positions), Qwen3-8B attention
shapes (32 query heads, 8 KV heads, head dim 128), bf16 paged KV cache
with 16-token pages, contexts uniform in [512, 16384] -- seeded synthetic
inputs (synth.py), larger than L2 per round (about 3.2 GB), so no flush is
needed between rounds.

A step is one full round (ddt_round: top-K, tree, mask, attention, target
argmax, walk, compaction). Every step restores ctx_lens first (a 256-byte
device copy) so each step does the same work. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only other implementation
of the round) on the host cores over a bounded sample of the same workload.
Under torchrun each rank runs its own replica of the round (requests shard
across ranks with no exchange); rank 0 prints the aggregate.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree rounds/s at R=64,L=15,V=152K,B=32; achieved HBM GB/s vs GB300 peak"
UNIT = "rounds/s"
WORKLOAD = "batch64"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- replicas
def rank_seed(base, rank):
    """Each rank's replica draws its own inputs: the workload's seed plus the
    rank."""
    return base + rank


def max_over_ranks(ms, dist, device):
    """The slowest rank's time; every rank gets it (a single process keeps
    its own)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, ms):
    """Units per second of the whole job: every rank ran `steps` units in the
    slowest rank's `ms`."""
    return world * steps / (ms / 1e3)


def _workload_desc(cfg):
    if cfg.ctx_kind == "uniform":
        ctx = "ctx~U[%d,%d]" % cfg.ctx_args[:2]
    elif cfg.ctx_kind == "fixed":
        ctx = "ctx=%d" % cfg.ctx_args[0]
    else:
        ctx = "ctx~%s%s" % (cfg.ctx_kind, tuple(cfg.ctx_args))
    return ("%s: R=%d,L=%d,V=%d,B=%d,K=%d,P=%d,Hq=%d,Hkv=%d,d=%d,page=%d,%s,%s"
            % (cfg.name, cfg.R, cfg.L, cfg.V, cfg.B, cfg.K, cfg.P, cfg.Hq, cfg.Hkv, cfg.d, cfg.page,
               ctx, cfg.logit_dtype))


def config_dict(cfg, total_bytes):
    """The JSON line's `config` (the same for both arms)."""
    return {"workload": _workload_desc(cfg),
            "l2": "inputs larger than L2 (%.2f GB algorithmic per round), no flush"
                  % (total_bytes / 1e9),
            "parallelism": "replicas (requests shard by rank, no collective)"}


def round_bytes(cfg, ctx_lens, acc_len=None):
    """Algorithmic HBM bytes of one round, by stage (each tensor once)."""
    R, L, V, K, P = cfg.R, cfg.L, cfg.V, cfg.K, cfg.P
    W = cfg.W
    kv_row = cfg.Hkv * cfg.d * 2  # bytes of one token's K (or V) for all KV heads
    ctx_tot = int(np.sum(ctx_lens))
    b = {}
    b["topk"] = R * L * V * 2 + R * L * K * 8
    b["tree"] = R * L * K * 8 + R * (cfg.B + 3 * P) * 4 + R * P * W * 4
    b["attention"] = (2 * ctx_tot * kv_row          # paged K and V
                      + R * P * cfg.Hq * cfg.d * (2 + 4)  # Q in (bf16), O out (f32)
                      + 2 * R * P * kv_row          # tree K and V
                      + R * P * W * 4 + R * 4)      # mask, ctx_lens
    nacc = int(np.sum(acc_len)) if acc_len is not None else R
    b["accept"] = (R * P * V * 2                    # target logits
                   + R * (P + cfg.B + 2 * L + 4) * 4
                   + 2 * 2 * nacc * kv_row)         # compaction: read + write K and V rows
    b["total"] = sum(b.values())
    return b


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _traffic_for(kernel_file, kernel_key):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel_key]
        src = open(os.path.join(ROOT, "speculative_decoding_draft_depth_gb300", "csrc",
                                kernel_file), "rb").read()
        if rec.get("source_sha1") != hashlib.sha1(src).hexdigest():
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle
def cpu_oracle_round(cfg, inp, reqs):
    """The oracle's round on a subset of requests (host arrays); seconds."""
    import oracle
    sub = {}
    for k in ("draft_logits", "q", "k_tree", "v_tree", "block_table", "ctx_lens"):
        sub[k] = np.ascontiguousarray(inp[k][reqs])
    t0 = time.perf_counter()
    lp, ids, _, _ = oracle.topk_logprobs(sub["draft_logits"], cfg.K)
    tree = oracle.build_tree(lp, ids, cfg.B)
    mask = oracle.build_mask(tree.parents, tree.n_nodes)
    oracle.tree_attention(sub["q"], sub["k_tree"], sub["v_tree"], inp["k_cache"], inp["v_cache"],
                          sub["block_table"], sub["ctx_lens"], mask)
    a, _ = oracle.argmax(inp["target_logits"][reqs])
    acc_len, acc_nodes, _, _ = oracle.walk(a, tree.tokens, tree.parents, tree.n_nodes, cfg.L)
    # compaction writes into scratch copies of only the touched pages' pool
    kc = inp["k_cache"].copy() if inp.get("copy_cache") else inp["k_cache"]
    vc = inp["v_cache"].copy() if inp.get("copy_cache") else inp["v_cache"]
    ctx = sub["ctx_lens"].copy()
    oracle.compact(kc, vc, sub["block_table"], ctx, sub["k_tree"], sub["v_tree"], acc_nodes,
                   acc_len)
    return time.perf_counter() - t0


def cpu_sample(cfg, inp, n_req, repeats=3):
    """The oracle, as it stands, on n_req requests of the round: the median of
    `repeats` passes, scaled to the full batch."""
    import oracle
    rng = np.random.default_rng(12345)
    reqs = np.sort(rng.choice(cfg.R, size=n_req, replace=False))
    runs = [cpu_oracle_round(cfg, inp, reqs) for _ in range(repeats)]
    secs = float(np.median(runs))
    per_round = secs * cfg.R / n_req
    return {"value": 1.0 / per_round, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d of %d requests of the same round (all stages), median of %d passes "
                      "(%s s), scaled to the full batch"
                      % (n_req, cfg.R, repeats, ", ".join("%.2f" % x for x in runs))}


# ----------------------------------------------------------------- inputs
def make_inputs(cfg):
    from speculative_decoding_draft_depth_gb300 import synth
    inp = synth.draw_round_inputs(cfg)
    return inp


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the timing of the NEXT rows (parent-conditioned tree)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-request and wide workloads' lines")
    ap.add_argument("--stage", default="round",
                    choices=["round", "topk", "tree", "attention", "accept", "cond_tree",
                             "markov", "stochastic", "scheduler", "single", "wide256"],
                    help="time one stage alone (small profiling cases); cond_tree: the "
                         "parent-conditioned tree's workload alone")
    ap.add_argument("--requests", type=int, default=0,
                    help="requests per round (default: the workload's 64)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from speculative_decoding_draft_depth_gb300 import synth
    cfg = synth.config(WORKLOAD, seed=rank_seed(synth.config(WORKLOAD).seed, rank))
    if args.requests:
        cfg = synth.config(WORKLOAD, R=args.requests, seed=cfg.seed)

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(cfg, args)
        return

    import torch
    torch.cuda.set_device(local_rank)
    if args.stage in ("cond_tree", "markov", "stochastic", "scheduler", "single", "wide256"):
        from speculative_decoding_draft_depth_gb300 import ddt
        ddt.load()
        fn = {"cond_tree": time_cond_tree, "markov": time_markov,
              "stochastic": time_stochastic, "scheduler": time_scheduler,
              "single": time_single,
              "wide256": lambda dev, reps, cpu: time_wide256(dev, blocks=max(2, reps // 40),
                                                             cpu=cpu)}[args.stage]
        res = fn(torch.device("cuda", local_rank), reps=max(args.steps, 1),
                 cpu=not args.no_cpu_baseline)
        if rank == 0:
            print(json.dumps({"stage": args.stage, **res}))
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from speculative_decoding_draft_depth_gb300 import ddt
    ddt.load()

    inp = make_inputs(cfg)
    dev = torch.device("cuda", local_rank)

    def td(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    c = ddt.make_config(R_max=cfg.R, L=cfg.L, V=cfg.V, B=cfg.B, K=cfg.K, Hq=cfg.Hq, Hkv=cfg.Hkv,
                        d=cfg.d, page_size=cfg.page,
                        max_pages_per_req=inp["block_table"].shape[1],
                        num_pages=inp["k_cache"].shape[0])
    ctx = ddt.Context(c)
    bufs = ctx.alloc_outputs(cfg.R, device=dev)
    d = {k: td(inp[k]) for k in ("draft_logits", "q", "k_tree", "v_tree", "k_cache", "v_cache",
                                 "block_table", "ctx_lens")}
    ctx0 = d["ctx_lens"].clone()
    # target logits follow this round's tree (set-up round, untimed)
    bufs.update(d)
    bufs["target_logits"] = torch.zeros((cfg.R, cfg.P, cfg.V), dtype=torch.int16, device=dev)
    ctx.ddt_round(cfg.R, bufs)
    torch.cuda.synchronize()
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    tl = target.logits_for_tree(bufs["tree_tokens"].cpu().numpy(), bufs["parents"].cpu().numpy(),
                                bufs["n_nodes"].cpu().numpy())
    inp["target_logits"] = tl
    bufs["target_logits"] = td(tl)
    d["ctx_lens"].copy_(ctx0)
    stream = torch.cuda.current_stream()
    R = cfg.R

    def step(att_events=None):
        """One round: ddt_round (a1..a7); with att_events, the library records
        the pair of CUDA events around the attention launch on `stream`."""
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        ctx.ddt_round(R, bufs, stream, att_events=att_events)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set during warm-up")
    if args.stage != "round":
        ms = time_stages(ctx, cfg, bufs, d, ctx0, stream, reps=args.steps, only=args.stage)
        print(json.dumps({"stage": args.stage, "requests": cfg.R, "ms": ms[args.stage],
                          "workload": _workload_desc(cfg)}))
        return
    acc_len = bufs["acc_len"].cpu().numpy()

    # ---------------- timed region: K full rounds
    clocks = Clocks(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    att_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for a_, b_ in att_ev:  # create the events (the library records them)
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        step(att_ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    att_ms_live = float(np.mean([a.elapsed_time(b) for a, b in att_ev]))
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    ms_per_step = ms_total / args.steps
    value = job_throughput(world, args.steps, ms_total)

    # ---------------- per-stage durations (same stream, CUDA events)
    stage_ms = time_stages(ctx, cfg, bufs, d, ctx0, stream, reps=max(20, args.steps // 10))

    peak, peak_kind = _peaks()
    nb = round_bytes(cfg, inp["ctx_lens"], acc_len)
    # the dominant kernel, timed inside the timed region above
    att_gbs = nb["attention"] / (att_ms_live / 1e3) / 1e9
    traffic = _traffic_for("attention_tc.cu", "att_kernel")
    roofline = {"bound": "hbm", "achieved": round(att_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(att_gbs / peak, 4), "traffic": traffic,
                "kernel": "att_tc_kernel (a4, ddt_tree_attention: paged GQA tree attention on tcgen05)",
                "launch_ms": round(att_ms_live, 4),
                "peak_kind": peak_kind}
    round_gbs = nb["total"] * value / world / 1e9
    stages = {k: {"ms": round(v, 4),
                  "GBps": round(nb[k] / (v / 1e3) / 1e9, 1) if k in nb else None}
              for k, v in stage_ms.items()}

    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded numpy generators)",
           "config": config_dict(cfg, nb["total"]),
           "round_hbm": {"bytes_per_round": nb["total"], "achieved_GBps": round(round_gbs, 1),
                         "peak": peak, "frac": round(round_gbs / peak, 4), "peak_kind": peak_kind},
           "stages": stages,
           "roofline": roofline,
           "gpu_launches": launches_per_round(cfg) * args.steps,
           "clocks": clk,
           "acceptance": {"mean_acc_len": float(np.mean(acc_len))}}

    if rank == 0 and not args.no_configs:
        out["configs"] = {"single": time_single(dev, cpu=not args.no_cpu_baseline),
                          "wide256": time_wide256(dev, cpu=not args.no_cpu_baseline)}
    if rank == 0 and not args.no_next:
        out["next_rows"] = {"cond_tree": time_cond_tree(dev, cpu=not args.no_cpu_baseline),
                            "markov_table_tree": time_markov(dev, cpu=not args.no_cpu_baseline),
                            "stochastic_chain": time_stochastic(dev,
                                                                cpu=not args.no_cpu_baseline),
                            "prefix_scheduler": time_scheduler(dev,
                                                               cpu=not args.no_cpu_baseline)}
    if not args.no_e2e:
        out["e2e"] = time_e2e(ctx, cfg, inp, bufs, d, ctx0, stream, dev, world, dist,
                              steps=max(10, min(args.steps, 50)))
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_sample(cfg, inp, n_req=min(32, cfg.R))
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def launches_per_round(cfg):
    """Kernels of this library one ddt_round launches (the ncu launch list in
    profiles/launches_round_batch64.md shows the same set): a1 streaming +
    a1 selection, the a2/a3 tree, a5 argmax, a4 attention and its split
    combine (launched whenever the grid has more than one CTA group, i.e.
    Hkv < SMs / 2), a6/a7 walk + compaction, and the context-length update."""
    return 8


def time_stages(ctx, cfg, bufs, d, ctx0, stream, reps, only=None):
    import torch
    R = cfg.R
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    res = {}

    def run(name, fn):
        if only is not None and name != only:
            return
        fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / reps

    run("topk", lambda: ctx.ddt_topk_logprobs(bufs["draft_logits"], R, bufs["top_lp"],
                                              bufs["top_ids"], stream))
    run("tree", lambda: ctx.ddt_build_tree(bufs["top_lp"], bufs["top_ids"], R, bufs["tree_tokens"],
                                           bufs["parents"], bufs["depths"], bufs["n_nodes"],
                                           bufs["mask"], stream))
    d["ctx_lens"].copy_(ctx0)
    run("attention", lambda: ctx.ddt_tree_attention(bufs["q"], bufs["k_tree"], bufs["v_tree"],
                                                    bufs["k_cache"], bufs["v_cache"],
                                                    bufs["block_table"], bufs["ctx_lens"],
                                                    bufs["mask"], R, bufs["attn_out"], stream))

    def accept():
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        ctx.ddt_accept(bufs["target_logits"], bufs["tree_tokens"], bufs["parents"],
                       bufs["n_nodes"], R, bufs["target_argmax"], bufs["acc_len"],
                       bufs["acc_nodes"], bufs["acc_tokens"], bufs["bonus"], bufs["k_cache"],
                       bufs["v_cache"], bufs["block_table"], bufs["k_tree"], bufs["v_tree"],
                       bufs["ctx_lens"], stream)

    run("accept", accept)
    d["ctx_lens"].copy_(ctx0)
    torch.cuda.synchronize()
    return res


def _td(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def _make_ctx(cfg, block_table, num_pages):
    from speculative_decoding_draft_depth_gb300 import ddt
    c = ddt.make_config(R_max=cfg.R, L=cfg.L, V=cfg.V, B=cfg.B, K=cfg.K, Hq=cfg.Hq, Hkv=cfg.Hkv,
                        d=cfg.d, page_size=cfg.page, max_pages_per_req=block_table.shape[1],
                        num_pages=num_pages)
    return ddt.Context(c)


def time_single(dev, reps=200, cpu=True):
    """The single-request workload (R=1, L=15, V=151936, B=32, Qwen3-8B
    attention at context 4096): a whole round (ddt_round) as device time per
    call over `reps` calls, the stages alone, the algorithmic bytes, and the
    oracle's round on the same inputs. The round is latency-bound at batch 1;
    the pages' DDTree candidate construction (GPU top-K and logsumexp, a copy
    to the host and a CPU heap) took 0.49 ms per round at batch 1 on an
    unstated GPU, which the top-K plus tree stages here compare with."""
    import torch
    from speculative_decoding_draft_depth_gb300 import synth
    cfg = synth.config("single")
    inp = synth.draw_round_inputs(cfg)
    ctx = _make_ctx(cfg, inp["block_table"], inp["k_cache"].shape[0])
    bufs = ctx.alloc_outputs(cfg.R, device=dev)
    d = {k: _td(inp[k], dev) for k in ("draft_logits", "q", "k_tree", "v_tree", "k_cache",
                                       "v_cache", "block_table", "ctx_lens")}
    ctx0 = d["ctx_lens"].clone()
    bufs.update(d)
    bufs["target_logits"] = torch.zeros((cfg.R, cfg.P, cfg.V), dtype=torch.int16, device=dev)
    ctx.ddt_round(cfg.R, bufs)
    torch.cuda.synchronize()
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    tl = target.logits_for_tree(bufs["tree_tokens"].cpu().numpy(), bufs["parents"].cpu().numpy(),
                                bufs["n_nodes"].cpu().numpy())
    inp["target_logits"] = tl
    bufs["target_logits"] = _td(tl, dev)
    stream = torch.cuda.current_stream()

    def step():
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        ctx.ddt_round(cfg.R, bufs, stream)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set in the single-request round")
    acc_len = bufs["acc_len"].cpu().numpy()
    stage_ms = time_stages(ctx, cfg, bufs, d, ctx0, stream, reps=max(20, reps // 4))
    nb = round_bytes(cfg, inp["ctx_lens"], acc_len)
    peak, _ = _peaks()
    res = {"workload": _workload_desc(cfg), "ms_per_round": round(ms, 4),
           "rounds_per_s": round(1e3 / ms, 1),
           "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
           "construction_ms": round(stage_ms["topk"] + stage_ms["tree"], 4),
           "construction_context": "the pages' DDTree candidate construction at batch 1: 0.49 ms "
                                   "per round (GPU top-K + CPU heap, unstated GPU)",
           "algorithmic_bytes": int(nb["total"]),
           "GBps": round(nb["total"] / (ms / 1e3) / 1e9, 1),
           "frac_of_hbm": round(nb["total"] / (ms / 1e3) / 1e9 / peak, 4),
           "bound": "latency (one request: each stage is a short kernel chain)",
           "mean_acc_len": float(np.mean(acc_len))}
    if cpu:
        secs = [cpu_oracle_round(cfg, inp, np.array([0])) for _ in range(3)]
        res["cpu_oracle_ms"] = round(float(np.median(secs)) * 1e3, 1)
        res["cpu_oracle_sample"] = "the whole round (one request), median of 3"
    ctx.close()
    return res


def gpu_wide_inputs(cfg, dev, seed):
    """The wide workload's round inputs drawn on the GPU (a seeded torch
    generator; the numpy generators take minutes at this size): the same
    recipe as synth.draw_round_inputs (draft rows N(0,1) plus the Zipf boost
    on 20 distinct tokens, divided by a temperature U[0.3, 1.5] per request
    and depth; lognormal contexts; a permuted page pool; N(0,1) caches,
    queries and tree keys/values, all bf16). Contexts and the page table come
    from numpy (small)."""
    import torch
    from speculative_decoding_draft_depth_gb300 import synth
    rng = np.random.default_rng(seed)
    ctx_lens = synth.draw_ctx_lens(cfg, rng)
    grow = cfg.rounds * (cfg.L + 1)
    need = [(int(c) + grow + cfg.page - 1) // cfg.page for c in ctx_lens]
    num_pages = sum(need) + cfg.spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((cfg.R, max(need)), -1, np.int32)
    pos = 0
    for r, n in enumerate(need):
        block_table[r, :n] = perm[pos:pos + n]
        pos += n
    g = torch.Generator(device=dev).manual_seed(int(seed))
    R, L, V, P = cfg.R, cfg.L, cfg.V, cfg.P
    z = torch.randn((R * L, V), generator=g, device=dev)
    toks = torch.multinomial(torch.ones((R * L, V), device=dev), 20, replacement=False,
                             generator=g)
    boost = (8.0 * torch.arange(1, 21, device=dev, dtype=torch.float32) ** -1.1).expand(R * L, 20)
    z.scatter_add_(1, toks, boost.contiguous())
    lo, hi = cfg.temp_range
    temp = lo + (hi - lo) * torch.rand((R * L, 1), generator=g, device=dev)
    z = (z / temp).to(torch.bfloat16).view(R, L, V)

    def nrm(shape):
        return torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)

    out = {"draft_logits": z.view(torch.int16), "ctx_lens": ctx_lens, "block_table": block_table,
           "k_cache": nrm((num_pages, cfg.page, cfg.Hkv, cfg.d)).view(torch.int16),
           "v_cache": nrm((num_pages, cfg.page, cfg.Hkv, cfg.d)).view(torch.int16),
           "q": nrm((R, P, cfg.Hq, cfg.d)).view(torch.int16),
           "k_tree": nrm((R, P, cfg.Hkv, cfg.d)).view(torch.int16),
           "v_tree": nrm((R, P, cfg.Hkv, cfg.d)).view(torch.int16), "gen": g}
    return out


def time_wide256(dev, blocks=5, cpu=True):
    """The wide workload (R=256, B=K=64, lognormal contexts up to 32768,
    Qwen3-4B attention): blocks of 8 consecutive rounds (ddt_round) with
    compaction in between, the context lengths growing by each round's
    accepted length; every block restores the first round's contexts. Device
    time per round over `blocks` blocks after one warm-up block, the
    algorithmic bytes of the 8 rounds (contexts as they grew), and the
    oracle's round on two requests scaled to the batch. The 8 rounds of a
    block reuse one set of logits, queries and tree keys/values (the parity
    test draws fresh ones per round); the target agrees with the draft's
    top-1 token at 3 of 4 tree positions, the rest pick a random token."""
    import torch
    from speculative_decoding_draft_depth_gb300 import synth
    cfg = synth.config("wide256")
    gi = gpu_wide_inputs(cfg, dev, cfg.seed)
    g = gi.pop("gen")
    ctx = _make_ctx(cfg, gi["block_table"], gi["k_cache"].shape[0])
    bufs = ctx.alloc_outputs(cfg.R, device=dev)
    d = {k: (v if torch.is_tensor(v) else _td(v, dev)) for k, v in gi.items()}
    ctx0 = d["ctx_lens"].clone()
    bufs.update(d)
    R, P, V, L = cfg.R, cfg.P, cfg.V, cfg.L
    bufs["target_logits"] = torch.zeros((R, P, V), dtype=torch.int16, device=dev)
    ctx.ddt_round(R, bufs)  # set-up round: the tree the target follows
    torch.cuda.synchronize()
    top1 = d["draft_logits"].view(torch.bfloat16).float().argmax(-1)  # [R, L] (construction)
    depth = bufs["depths"].long().clamp(0, L - 1)
    want = torch.gather(top1, 1, depth)
    agree = torch.rand((R, P), generator=g, device=dev) < 0.75
    tok = torch.where(agree, want, torch.randint(0, V, (R, P), generator=g, device=dev))
    tl = torch.randn((R, P, V), generator=g, device=dev)
    tl.scatter_add_(2, tok.unsqueeze(-1), torch.full((R, P, 1), 20.0, device=dev))
    bufs["target_logits"] = tl.to(torch.bfloat16).view(torch.int16)
    del tl
    d["ctx_lens"].copy_(ctx0)
    stream = torch.cuda.current_stream()

    def block():
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        for _ in range(cfg.rounds):
            ctx.ddt_round(R, bufs, stream)

    block()
    torch.cuda.synchronize()
    acc_len = bufs["acc_len"].cpu().numpy()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(blocks):
        block()
    b.record(stream)
    torch.cuda.synchronize()
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set in the wide rounds")
    ms = a.elapsed_time(b) / (blocks * cfg.rounds)
    c0 = gi["ctx_lens"].astype(np.int64)
    nbytes = [round_bytes(cfg, c0 + k * acc_len, acc_len)["total"] for k in range(cfg.rounds)]
    per_round = float(np.mean(nbytes))
    peak, _ = _peaks()
    res = {"workload": _workload_desc(cfg) + ", 8 rounds with compaction",
           "ms_per_round": round(ms, 4), "rounds_per_s": round(1e3 / ms, 1),
           "rounds_per_block": cfg.rounds, "blocks": blocks,
           "bytes_per_round": int(per_round),
           "GBps": round(per_round / (ms / 1e3) / 1e9, 1),
           "frac_of_hbm": round(per_round / (ms / 1e3) / 1e9 / peak, 4),
           "mean_acc_len": float(np.mean(acc_len)),
           "data": "synthetic, drawn on the GPU (seeded torch generator, the synth recipe)"}
    if cpu:
        import oracle
        reqs = np.array([0, 1])
        sub = _host_requests(cfg, d, bufs, reqs)
        secs = cpu_oracle_round(replace_R(cfg, len(reqs)), sub, np.arange(len(reqs)))
        res["cpu_oracle_ms"] = round(secs * R / len(reqs) * 1e3, 1)
        res["cpu_oracle_sample"] = "2 of 256 requests (all stages), scaled to the batch"
    ctx.close()
    return res


def replace_R(cfg, R):
    from dataclasses import replace
    return replace(cfg, R=R)


def _host_requests(cfg, d, bufs, reqs):
    """Host copies of some requests' round inputs, their pages gathered into a
    small pool with a renumbered page table (for the oracle)."""
    import torch
    bt = d["block_table"].cpu().numpy()[reqs]
    pages = sorted({int(p) for p in bt.reshape(-1) if p >= 0})
    remap = {p: i for i, p in enumerate(pages)}
    nbt = np.where(bt >= 0, np.vectorize(lambda p: remap.get(int(p), -1))(bt), -1).astype(np.int32)
    pi = torch.tensor(pages, device=d["k_cache"].device, dtype=torch.long)
    host = lambda t: t.cpu().numpy().view(np.uint16) if t.dtype == torch.int16 else t.cpu().numpy()  # noqa: E731
    ri = torch.tensor(reqs, device=d["k_cache"].device, dtype=torch.long)
    return {"draft_logits": host(d["draft_logits"][ri]), "q": host(d["q"][ri]),
            "k_tree": host(d["k_tree"][ri]), "v_tree": host(d["v_tree"][ri]),
            "block_table": nbt, "ctx_lens": d["ctx_lens"].cpu().numpy()[reqs],
            "k_cache": host(d["k_cache"][pi]), "v_cache": host(d["v_cache"][pi]),
            "target_logits": host(bufs["target_logits"][ri]), "copy_cache": True}


def time_cond_tree(dev, reps=20, cpu=True):
    """The parent-conditioned tree ("Robot2050/TreeSpark", items 1-2) on its own
    workload (8 requests, 7 depths, V=151936, H=256, k=F=4, N=32, Qwen3-4B
    attention at context 2048): the tree alone (ddt_build_tree_conditioned) and
    the whole conditioned round (ddt_round_conditioned: the tree, then a4..a7),
    each as device time per call over `reps` calls after 3 warm-up calls, with
    algorithmic bytes (W and the backbone rows once per depth, then the
    round's verification bytes), and the oracle's tree time for one request
    scaled to the batch."""
    import torch
    from speculative_decoding_draft_depth_gb300 import ddt, synth
    cfg = synth.config("treespark")
    inp = synth.draw_round_inputs(cfg)
    W, E, anchors = synth.draw_markov_head(cfg)
    c = ddt.make_config(R_max=cfg.R, L=cfg.L, V=cfg.V, B=cfg.B, K=cfg.K, Hq=cfg.Hq, Hkv=cfg.Hkv,
                        d=cfg.d, page_size=cfg.page,
                        max_pages_per_req=inp["block_table"].shape[1],
                        num_pages=inp["k_cache"].shape[0], markov_dim=cfg.markov_dim,
                        frontier=cfg.frontier)
    ctx = ddt.Context(c)

    def td(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    ell, Wd, Ed, an = td(inp["draft_logits"]), td(W), td(E), td(anchors)
    R = cfg.R
    bufs = ctx.alloc_outputs(R, device=dev)
    d = {k: td(inp[k]) for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache", "block_table",
                                 "ctx_lens")}
    ctx0 = d["ctx_lens"].clone()
    bufs.update(d)
    bufs["draft_logits"] = ell

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def tree():
        ctx.ddt_build_tree_conditioned(ell, Wd, Ed, an, R, bufs["tree_tokens"], bufs["parents"],
                                       bufs["depths"], bufs["n_nodes"], bufs["mask"])

    ms = timed(tree)
    # the synthetic target follows this tree (set-up, untimed)
    torch.cuda.synchronize()
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    bufs["target_logits"] = td(target.logits_for_tree(
        bufs["tree_tokens"].cpu().numpy(), bufs["parents"].cpu().numpy(),
        bufs["n_nodes"].cpu().numpy()))

    def round_():
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        ctx.ddt_round_conditioned(R, bufs, Wd, Ed, an)

    ms_round = timed(round_)
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set in the conditioned round")
    # W is read at every depth but stays in L2 after the first (evict-last
    # TMA loads): DRAM bytes count it once, L2 bytes once per depth
    w_bytes = cfg.V * cfg.markov_dim * 2
    rows = cfg.L * R * cfg.V * 2 + R * cfg.L * cfg.frontier * cfg.markov_dim * 2
    nbytes = w_bytes + rows
    l2_bytes = cfg.L * w_bytes + rows
    rb = round_bytes(cfg, inp["ctx_lens"], bufs["acc_len"].cpu().numpy())
    nbytes_round = nbytes + rb["attention"] + rb["accept"]
    peak, _ = _peaks()
    res = {"workload": "treespark: R=8, 7 depths, V=151936, H=256, k=4, F=4, N=32, "
                       "Hq=32, Hkv=8, d=128, ctx 2048, bf16",
           "ms": round(ms, 4),
           "bound": "latency: %d dependent depth steps (a GEMM over the L2-resident W, then "
                    "the merge), chained by programmatic dependent launch" % cfg.L,
           "us_per_depth": round(ms * 1e3 / cfg.L, 2),
           "algorithmic_bytes": int(nbytes),
           "dram_bytes_note": "W (%.1f MB) once, the backbone rows and the frontier's E rows "
                              "at every depth" % (w_bytes / 1e6),
           "GBps": round(nbytes / (ms / 1e3) / 1e9, 1),
           "frac_of_hbm": round(nbytes / (ms / 1e3) / 1e9 / peak, 4),
           "l2_bytes": int(l2_bytes),
           "l2_GBps": round(l2_bytes / (ms / 1e3) / 1e9, 1),
           "round": {"ms": round(ms_round, 4), "rounds_per_s": round(1e3 / ms_round, 1),
                     "algorithmic_bytes": int(nbytes_round),
                     "GBps": round(nbytes_round / (ms_round / 1e3) / 1e9, 1),
                     "frac_of_hbm": round(nbytes_round / (ms_round / 1e3) / 1e9 / peak, 4)}}
    if cpu:
        import oracle
        t0 = time.perf_counter()
        oracle.cond_tree(inp["draft_logits"][:1], W, E, anchors[:1], k=cfg.K, F=cfg.frontier,
                         N=cfg.B)
        sec = (time.perf_counter() - t0) * R
        res["cpu_oracle_ms"] = round(sec * 1e3, 1)
        res["cpu_oracle_sample"] = "1 of 8 requests, scaled"
    return res


def time_markov(dev, reps=20, cpu=True):
    """The SparklingTree table tree ("SparklingTree ...", "Solving the
    candidate tree construction") on its workload (R=64, L=15, V=151936,
    C=128, B=64, H=256): the prefilter + table (ddt_markov_table), the tree
    over the table (ddt_build_tree_markov) and the whole round
    (ddt_round_markov: both, then a4..a7), each as device time per call over
    `reps` calls after 3 warm-up calls, with algorithmic bytes; and the
    oracle's table + tree time for one request scaled to the batch."""
    import torch
    from speculative_decoding_draft_depth_gb300 import ddt, synth
    cfg = synth.config("sparkling")
    inp = synth.draw_round_inputs(cfg)
    W, E, anchors = synth.draw_markov_head(cfg)
    c = ddt.make_config(R_max=cfg.R, L=cfg.L, V=cfg.V, B=cfg.B, K=cfg.K, Hq=cfg.Hq, Hkv=cfg.Hkv,
                        d=cfg.d, page_size=cfg.page,
                        max_pages_per_req=inp["block_table"].shape[1],
                        num_pages=inp["k_cache"].shape[0], markov_dim=cfg.markov_dim,
                        prefilter=cfg.prefilter)
    ctx = ddt.Context(c)

    def td(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    R, L, V, C, H, B = cfg.R, cfg.L, cfg.V, cfg.prefilter, cfg.markov_dim, cfg.B
    ell, Wd, Ed, an = td(inp["draft_logits"]), td(W), td(E), td(anchors)
    cand = torch.empty((R, L, C), dtype=torch.int32, device=dev)
    tab = torch.empty((R, L, C, C), dtype=torch.float32, device=dev)
    bufs = ctx.alloc_outputs(R, device=dev)
    d = {k: td(inp[k]) for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache", "block_table",
                                 "ctx_lens")}
    ctx0 = d["ctx_lens"].clone()
    bufs.update(d)
    bufs["draft_logits"] = ell

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    ms_table = timed(lambda: ctx.ddt_markov_table(ell, Wd, Ed, an, R, cand, tab))
    ms_tree = timed(lambda: ctx.ddt_build_tree_markov(
        cand, tab, R, bufs["tree_tokens"], bufs["parents"], bufs["depths"], bufs["n_nodes"],
        bufs["mask"]))
    torch.cuda.synchronize()
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    bufs["target_logits"] = td(target.logits_for_tree(
        bufs["tree_tokens"].cpu().numpy(), bufs["parents"].cpu().numpy(),
        bufs["n_nodes"].cpu().numpy()))

    def round_():
        d["ctx_lens"].copy_(ctx0, non_blocking=True)
        ctx.ddt_round_markov(R, bufs, Wd, Ed, an)

    ms_round = timed(round_)
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set in the table-tree round")
    # algorithmic bytes: the logits once (prefilter), the kept tokens' W rows
    # and the parents' E rows (one parent at depth 0), the table written once;
    # the tree reads the rows of the nodes it expands
    b_table = (R * L * V * 2 + R * L * C * H * 2 + R * (1 + (L - 1) * C) * H * 2
               + R * L * C * 4 + R * L * C * C * 4)
    b_tree = R * L * C * 4 + R * (B + 1) * C * 4 + R * (B + 2 * (B + 1) + 1) * 4
    rb = round_bytes(cfg, inp["ctx_lens"], bufs["acc_len"].cpu().numpy())
    b_round = b_table + b_tree + rb["attention"] + rb["accept"]
    peak, _ = _peaks()

    def rate(nbytes, ms):
        return {"ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                "GBps": round(nbytes / (ms / 1e3) / 1e9, 1),
                "frac_of_hbm": round(nbytes / (ms / 1e3) / 1e9 / peak, 4)}

    res = {"workload": "sparkling: R=64, L=15, V=151936, C=128, B=64, H=256, Hq=32, Hkv=8, "
                       "d=128, ctx~U[512,16384], bf16",
           "table": dict(rate(b_table, ms_table),
                         bound="HBM: the logits once, then gathered W/E rows and the table"),
           "tree": dict(rate(b_tree, ms_tree),
                        bound="latency: %d dependent heap pops per request (one CTA each)" % B,
                        us_per_pop=round(ms_tree * 1e3 / B, 3)),
           "round": dict(rate(b_round, ms_round), rounds_per_s=round(1e3 / ms_round, 1))}
    if cpu:
        import oracle
        t0 = time.perf_counter()
        oc, ot = oracle.markov_table(inp["draft_logits"][:1], W, E, anchors[:1], C)
        oracle.markov_tree(oc, ot, B)
        sec = (time.perf_counter() - t0) * R
        res["cpu_oracle_ms"] = round(sec * 1e3, 1)
        res["cpu_oracle_sample"] = "1 of 64 requests (table + tree), scaled"
    return res


def time_stochastic(dev, reps=20, cpu=True):
    """Stochastic verification of drafted chains ("DSpark Speculative Decoding
    Explained ...", the probability rule) on the batch64 shapes (R=64 chains
    of L=15 guesses, V=151936, bf16 draft [R, L, V] and target [R, L+1, V]
    logits): device time per ddt_accept_stochastic call over `reps` calls
    after 3 warm-up calls (the logits, 603 MB, exceed L2, so no flush is
    needed), with the algorithmic bytes (every logit read once); and the
    oracle's time for the same 64 chains."""
    import torch
    from speculative_decoding_draft_depth_gb300 import ddt, synth
    cfg = synth.config("batch64")
    inp = synth.draw_chain_inputs(cfg)
    R, L, V = cfg.R, cfg.L, cfg.V
    K = cfg.K
    c = ddt.make_config(R_max=R, L=L, V=V, B=K, K=K, Hq=4, Hkv=1, d=64, page_size=16,
                        max_pages_per_req=1, num_pages=1)
    ctx = ddt.Context(c)

    def td(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    dr, tg, tok, u, r = (td(inp[k]) for k in ("draft", "target", "tokens", "u", "r"))
    acc_len = torch.empty(R, dtype=torch.int32, device=dev)
    acc_tok = torch.empty((R, L + 1), dtype=torch.int32, device=dev)

    def call():
        ctx.ddt_accept_stochastic(dr, tg, tok, u, r, R, acc_len, acc_tok)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    if ctx.ddt_device_status() != 0:
        raise RuntimeError("device status flags set in stochastic verification")
    al = acc_len.cpu().numpy()
    nbytes = R * (2 * L + 1) * V * 2 + R * L * 12 + R * 4 + R * (L + 2) * 4
    # the draw re-reads row k* of the target (and of the draft after a rejection)
    redraw = int(sum(V * 2 * (1 + (k - 1 < L)) for k in al))
    peak, _ = _peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"workload": "batch64 chains: R=64, L=15, V=151936, bf16 draft and target logits, "
                       "target = draft + N(0, s^2), s~U[0.2,1.0], guesses sampled from the draft",
           "ms": round(ms, 4), "chains_per_s": round(R * 1e3 / ms, 1),
           "algorithmic_bytes": int(nbytes), "redraw_bytes": redraw,
           "GBps": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
           "mean_acc_len": float(al.mean())}
    if cpu:
        import oracle
        t0 = time.perf_counter()
        oracle.accept_stochastic(inp["draft"], inp["target"], inp["tokens"],
                                 inp["u"].astype(np.float64), inp["r"].astype(np.float64))
        res["cpu_oracle_ms"] = round((time.perf_counter() - t0) * 1e3, 1)
        res["cpu_oracle_sample"] = "all 64 chains"
    return res


def time_scheduler(dev, reps=200, cpu=True):
    """The hardware-aware prefix scheduler ("DSpark Speculative Decoding
    Explained ...", "Picking the budget") on two workloads:
      toy:      128 requests x 5 guesses with the page's toy cost, 25 ms plus
                0.1 ms per token checked (R + n tokens);
      measured: 64 requests x 15 guesses (the batch64 chains) with a cost
                table measured here from this library's own verification
                (ddt_accept_stochastic of the first 1, 2, 4, 8 and 15
                guesses of each chain, interpolated in the number of
                guesses).
    Confidences come from synth.draw_confidences. Reports the device time
    per ddt_schedule_prefix call (CUDA events around one replay of a CUDA
    graph of `reps` calls, after 3 warm-up calls; beside it the same over an
    eager loop of calls, where the host's launch rate can be the bound), the
    chosen budget, its tokens per ms against verifying
    every guess, and the oracle's time for the same decision; for the
    measured workload also the scheduled step (the budget, then verification
    of the kept prefixes with n_keep left on the device) beside verifying
    every guess."""
    import torch
    from speculative_decoding_draft_depth_gb300 import ddt, synth

    def td(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    def events_ms(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    def graph_ms(fn, n):
        # n calls captured in one CUDA graph and replayed: device time per
        # call without the host's launch rate (a call is one kernel)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    # the cost table: our chain verification of the first Lp guesses of every
    # chain (per-request guess counts on one 15-guess context, as a scheduled
    # step runs it)
    cfg = synth.config("batch64")
    R, L, V = cfg.R, cfg.L, cfg.V
    inp = synth.draw_chain_inputs(cfg)
    dr, tg, tok, u, r = (td(inp[k]) for k in ("draft", "target", "tokens", "u", "r"))
    cv = ddt.Context(ddt.make_config(R_max=R, L=L, V=V, B=8, K=8, Hq=4, Hkv=1, d=64,
                                     page_size=16, max_pages_per_req=1, num_pages=1))
    al = torch.empty(R, dtype=torch.int32, device=dev)
    at = torch.empty((R, L + 1), dtype=torch.int32, device=dev)
    points = []
    for Lp in (1, 2, 4, 8, 15):
        ng = torch.full((R,), Lp, dtype=torch.int32, device=dev)
        ms = events_ms(lambda: cv.ddt_accept_stochastic(dr, tg, tok, u, r, R, al, at,
                                                        n_guess=ng), 10)
        points.append((R * Lp, ms))
    xs = np.array([p[0] for p in points], np.float64)
    ys = np.array([p[1] for p in points], np.float64)
    n_all = np.arange(R * L + 1, dtype=np.float64)
    slope0 = (ys[1] - ys[0]) / (xs[1] - xs[0])
    measured = np.where(n_all < xs[0], ys[0] - slope0 * (xs[0] - n_all), np.interp(n_all, xs, ys))
    measured = np.maximum(measured, 1e-3).astype(np.float32)

    out = {}
    for name, Rw, Lw, cost in (
            ("toy", 128, 5, (25.0 + 0.1 * (128 + np.arange(128 * 5 + 1))).astype(np.float32)),
            ("measured", R, L, measured)):
        conf = synth.draw_confidences(Rw, Lw, seed=1)
        c = ddt.make_config(R_max=Rw, L=Lw, V=64, B=8, K=8, Hq=4, Hkv=1, d=64, page_size=16,
                            max_pages_per_req=1, num_pages=1)
        cx = ddt.Context(c)
        conf_d, cost_d = td(conf), td(cost)
        n_keep = torch.empty(Rw, dtype=torch.int32, device=dev)
        n_tot = torch.empty(1, dtype=torch.int32, device=dev)
        stats = torch.empty(2, dtype=torch.float64, device=dev)
        call = lambda: cx.ddt_schedule_prefix(conf_d, Rw, cost_d, n_keep, n_tot, stats)  # noqa: E731
        ms_eager = events_ms(call, reps)
        ms = graph_ms(call, reps)
        if cx.ddt_device_status() != 0:
            raise RuntimeError("device status flags set in the scheduler")
        keep = n_keep.cpu().numpy()
        st = stats.cpu().numpy()
        surv = np.cumprod(conf.astype(np.float64), axis=1)
        theta_all = (Rw + surv.sum()) / float(cost[-1])
        row = {"requests": Rw, "guesses_per_request": Lw, "us_per_call": round(ms * 1e3, 2),
               "us_per_call_eager": round(ms_eager * 1e3, 2),
               "kept": int(n_tot.cpu().numpy()[0]), "of": Rw * Lw,
               "tokens_per_ms": round(float(st[0]), 4),
               "tokens_per_ms_all_verified": round(theta_all, 4),
               "expected_tokens": round(float(st[1]), 3),
               "kept_per_request_histogram": np.bincount(keep, minlength=Lw + 1).tolist()}
        if cpu:
            import oracle
            t0 = time.perf_counter()
            for _ in range(20):
                oracle.schedule_prefix(conf, cost)
            row["cpu_oracle_us"] = round((time.perf_counter() - t0) / 20 * 1e6, 1)
        out[name] = row
        if name == "measured":
            # the scheduled step: the budget, then verification of the kept
            # prefixes (n_keep stays on the device), against verifying all
            n_kv = torch.empty(R, dtype=torch.int32, device=dev)

            def scheduled():
                cv.ddt_schedule_prefix(conf_d, R, cost_d, n_kv)
                cv.ddt_accept_stochastic(dr, tg, tok, u, r, R, al, at, n_guess=n_kv)

            row["scheduled_step_us"] = round(events_ms(scheduled, 20) * 1e3, 2)
            row["verify_all_us"] = round(
                events_ms(lambda: cv.ddt_accept_stochastic(dr, tg, tok, u, r, R, al, at), 20)
                * 1e3, 2)
            if cv.ddt_device_status() != 0:
                raise RuntimeError("device status flags set in the scheduled step")
    out["measured"]["cost_table_points_ms"] = [[int(x), round(y, 4)] for x, y in points]
    out["workload"] = ("toy: 128 x 5, cost 25 ms + 0.1 ms per token checked; measured: 64 x 15 "
                       "(batch64 chains), cost = this library's ddt_accept_stochastic time; "
                       "scheduled_step_us = ddt_schedule_prefix then ddt_accept_stochastic of "
                       "the kept prefixes")
    out["bound"] = "latency (one CTA; a few thousand slots)"
    return out


def time_e2e(ctx, cfg, inp, bufs, d, ctx0, stream, dev, world, dist, steps, n_copy=4):
    """Same metric through the C ABI with the step's inputs in pinned host
    memory: every step copies its inputs host->device, runs ddt_round and
    reads its results back, all inside the timed region. The copies are cut
    into chunks on n_copy streams (several DMA engines), and inputs are
    double-buffered on the device so that step i+1's copies overlap step i's
    round."""
    import torch
    names = ("draft_logits", "target_logits", "q", "k_tree", "v_tree")
    host = {}
    for k in names:
        a = np.ascontiguousarray(inp[k])
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        host[k] = torch.from_numpy(a).pin_memory()
    host_ctx = ctx0.cpu().pin_memory()
    outs = {k: torch.empty(bufs[k].shape, dtype=bufs[k].dtype).pin_memory()
            for k in ("acc_len", "acc_tokens", "bonus")}
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + host_ctx.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    sets = [{k: bufs[k] for k in names}, {k: torch.empty_like(bufs[k]) for k in names}]
    cstreams = [torch.cuda.Stream() for _ in range(n_copy)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    copied = [[ev() for _ in range(n_copy)] for _ in range(2)]
    used = [ev(), ev()]  # the round that last read each input set is done

    def step(i, first):
        cur = sets[i & 1]
        for c, cs in enumerate(cstreams):
            if not first[i & 1]:
                cs.wait_event(used[i & 1])
            with torch.cuda.stream(cs):
                for k in names:
                    src, dst = host[k].view(-1), cur[k].view(-1)
                    n = src.numel()
                    lo, hi = n * c // n_copy, n * (c + 1) // n_copy
                    dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
            copied[i & 1][c].record(cs)
        first[i & 1] = False
        for e in copied[i & 1]:
            stream.wait_event(e)
        d["ctx_lens"].copy_(host_ctx, non_blocking=True)
        rb = dict(bufs)
        rb.update(cur)
        ctx.ddt_round(cfg.R, rb, stream)
        used[i & 1].record(stream)
        for k, t in outs.items():
            t.copy_(bufs[k], non_blocking=True)

    first = [True, True]
    for i in range(3):
        step(i, first)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for cs in cstreams:
        cs.wait_event(a)
    first = [False, False]
    for i in range(steps):
        step(i, first)
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dist, dev)
    d["ctx_lens"].copy_(ctx0)
    return {"value": round(job_throughput(world, steps, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copy_streams": n_copy}


def run_reference(cfg, args):
    """The fp64 CPU oracle as the reference arm, on the host cores: every step
    (warm-up and timed) is the oracle's whole round over all requests, so
    ms_per_step is the measured time of one round."""
    import oracle
    from speculative_decoding_draft_depth_gb300 import synth
    inp = make_inputs(cfg)
    lp, ids, _, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
    tree = oracle.build_tree(lp, ids, cfg.B)
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    inp["target_logits"] = target.logits_for_tree(tree.tokens, tree.parents, tree.n_nodes)
    a, _ = oracle.argmax(inp["target_logits"])
    acc_len, _, _, _ = oracle.walk(a, tree.tokens, tree.parents, tree.n_nodes, cfg.L)
    nb = round_bytes(cfg, inp["ctx_lens"], acc_len)
    reqs = np.arange(cfg.R)
    times = []
    for s in range(max(args.warmup, 3) + args.steps):
        secs = cpu_oracle_round(cfg, inp, reqs)
        if s >= max(args.warmup, 3):
            times.append(secs)
    per_round = float(np.mean(times))
    value = 1.0 / per_round
    out = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": max(args.warmup, 3),
           "ms_per_step": round(per_round * 1e3, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded numpy generators)", "impl": "reference",
           "config": config_dict(cfg, nb["total"]),
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                            "kind": "oracle",
                            "sample": "each step: the oracle's whole round over all %d requests "
                                      "(all stages), mean of %d timed steps" % (cfg.R, args.steps)},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
