"""Benchmark: score-emitting paged decode attention + H2O select on one GB300.

Workload (default): the Llama-2-70B layer shape at 32K context -- batch 8,
64 q / 8 kv heads, head_dim 128, bf16 N(0,1) K/V in 16-token pages placed by
a random permutation of the pool, H2O budget 6553 = 4 sinks + 1024 window +
5525 heavy hitters.  One step = append the new token, attention over every
live key with each key's probability written and the H2O score updated,
then the H2O heavy-hitter selection (keep list, no compaction).  The 128
decode steps of the workload are replayed cyclically (after 128 steps the
sequence lengths return to 32768), so every step attends 32769..32896 keys.

Arms:
  default            the CUDA library (libkvsel.so) through its C ABI.
  --impl reference   the fp64 CPU oracle on the host cores, on a bounded
                     sample of the same workload (one (sequence, kv head)
                     pair per step), scaled to whole steps.

Prints one JSON line (rank 0).  Multi-GPU (torchrun): every rank runs an
independent replica of the workload (the path has no exchange step), value =
all ranks' steps / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s and effective KV GB/s (% of GB300 HBM peak) for attn+H2O select"
CONFIG_NAME = ("paged GQA decode + H2O select, Llama-2-70B layer shape (64 q / 8 kv heads, d=128, bf16), "
               "batch 8, 32K context, 16-token pages randomly permuted, budget 6553 = 4 sinks + 1024 "
               "window + 5525 heavy hitters")
PAGE = 16


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes)
# ---------------------------------------------------------------------------
def kv_bytes(S_list, Hkv, d=128):
    return sum(S_list) * Hkv * d * 2 * 2


def step_kernel_bytes(S_list, Hkv, Hq, d=128, probs=True, cum=True):
    """decode_step: read K,V of every live key; write each (q head, key) probability;
    read+write the H2O score of each (kv head, key); read q and write O (bf16)."""
    keys = sum(S_list)
    return (kv_bytes(S_list, Hkv, d) + (keys * Hq * 4 if probs else 0) + (keys * Hkv * 8 if cum else 0)
            + len(S_list) * Hq * d * 2 * 2)


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [r for (t, r) in self.rows if t0 - 0.06 <= t <= t1 + 0.06] or \
              [r for (t, r) in sorted(self.rows, key=lambda x: abs(x[0] - (t0 + t1) / 2))[:1]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in sel if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sel),
                "power_w_max": max((float(r[3]) for r in sel if r[3].replace(".", "").isdigit()),
                                   default=None)}


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in a fresh interpreter: never forked after CUDA init)
# ---------------------------------------------------------------------------
def oracle_pair_seconds(n_pairs: int, seed: int = 1, keys: int = 32769):
    """Time the oracle on n_pairs (sequence, kv head) pairs of one decode+select step.

    ``keys`` < 32769 times a prefix of the pair's keys (the oracle's cost is
    linear in the key count); the result is scaled back to the full pair.
    """
    import numpy as np
    import workloads
    from oracle.attention import bf16_bits_to_f64, decode_attention, h2o_accumulate
    from oracle.h2o import h2o_keep
    rng = np.random.default_rng(seed)
    Hq, Hkv, d, S0 = 64, 8, 128, 32768
    G = Hq // Hkv
    budget, n_sink, window = int(0.2 * 32768), 4, 1024
    # one pair's inputs, same distribution as the workload (N(0,1) bf16)
    S = min(keys, S0 + 1)
    Kb = bf16_bits_to_f64(workloads.normal_bf16(rng, (1, S, d)))
    Vb = bf16_bits_to_f64(workloads.normal_bf16(rng, (1, S, d)))
    q = bf16_bits_to_f64(workloads.normal_bf16(rng, (G, d)))
    cum = np.zeros((1, S))
    frac = S / (S0 + 1)
    b = max(n_sink + window, int(budget * frac))
    t0 = time.perf_counter()
    for _ in range(n_pairs):
        o, p = decode_attention(q, Kb, Vb, 1 / math.sqrt(d))
        cum = h2o_accumulate(cum, p)
        h2o_keep(cum[0], S, b, n_sink, min(window, b - n_sink))
    return (time.perf_counter() - t0) / n_pairs / frac


def cpu_worker_main(n_pairs):
    t = oracle_pair_seconds(n_pairs)
    print(json.dumps({"pair_seconds": t}))


def run_cpu_baseline(n_pairs: int, pairs_per_step: int):
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(n_pairs)],
                       capture_output=True, text=True, env=env, timeout=900)
    line = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not line:
        return None
    t = json.loads(line[-1])["pair_seconds"]
    return {"value": 1.0 / (t * pairs_per_step), "unit": "steps/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_pairs} (sequence, kv head) pairs of one step at 32769 keys "
                      f"(attention + probabilities + H2O update + select, fp64 numpy), "
                      f"scaled x{pairs_per_step} pairs per step"}


# ---------------------------------------------------------------------------
# reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
def reference_arm(args, rank, world):
    if rank != 0:
        return
    B, Hkv = 8, 8
    ts = []
    cores = len(os.sched_getaffinity(0))
    # size each step's sample so the whole run stays within ~2 minutes
    t_full = oracle_pair_seconds(1, seed=99)
    per_step = 120.0 / (args.warmup + args.steps)
    keys = int(min(32769, max(1024, 32769 * per_step / max(t_full, 1e-6))))
    for i in range(args.warmup + args.steps):
        t = oracle_pair_seconds(1, seed=100 + i, keys=keys) * B * Hkv
        if i >= args.warmup:
            ts.append(t)
    mean = sum(ts) / len(ts)
    value = 1.0 / mean
    line = {"metric": METRIC, "value": value, "unit": "steps/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": CONFIG_NAME},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: one (sequence, kv head) pair of the 70B-shape "
                                       f"step over {keys} of its 32769 keys, scaled to the full "
                                       f"pair and x64 pairs"},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def cuda_arm(args, rank, world):
    import numpy as np
    import torch
    import torch.distributed as dist

    import attention_guided_kv_gb300 as K
    import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K.lib()

    wl = workloads.decode_70b(seed=1 + rank, B=args.batch)
    B, Hq, Hkv, d, S0, T = wl.B, wl.Hq, wl.Hkv, wl.d, wl.S0, wl.steps
    max_len = wl.max_len

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    kpool = bf(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages))
    vpool = bf(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages))
    wl.K = wl.V = None
    kv = K.paged_kv(kpool, vpool, Hq)
    bt = torch.from_numpy(wl.block_table).to(dev)
    seq0 = torch.full((B,), S0, dtype=torch.int32, device=dev)
    seq = seq0.clone()
    q_all, kn_all, vn_all = bf(wl.q), bf(wl.k_new), bf(wl.v_new)
    cum = torch.zeros(B, Hkv, max_len, device=dev)
    probs = torch.zeros(B, Hq, max_len, device=dev) if not args.no_probs else None
    out = torch.zeros(B, Hq, d, device=dev, dtype=torch.bfloat16)
    keep = torch.zeros(B, Hkv, wl.budget, dtype=torch.int32, device=dev)
    ws = K.workspace(K.kvsel_decode_attn_workspace(kv, B, max_len, probs is not None))
    ws_ev = K.workspace(K.kvsel_h2o_evict_workspace(kv, B, wl.budget))
    stream = torch.cuda.current_stream()

    def step(i, q, kn, vn):
        if i % T == 0 and i > 0:
            seq.copy_(seq0)            # replay the 128-step window from 32K again
        K.kvsel_decode_attn(kv, bt, seq, q, out, ws, k_new=kn, v_new=vn, probs=probs, h2o_cum=cum,
                            max_len=max_len)
        K.kvsel_h2o_evict(kv, bt, seq, cum, ws_ev, budget=wl.budget, n_sink=wl.n_sink,
                          window=wl.window, compact=False, keep_out=keep)

    def dev_step(i):
        t = i % T
        step(i, q_all[t], kn_all[t], vn_all[t])

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up
    for i in range(args.warmup):
        dev_step(i)
    torch.cuda.synchronize()
    st0, st1 = K.read_status(ws), K.read_status(ws_ev)
    if st0 or st1:
        raise RuntimeError(f"device status after warm-up: {st0} {st1}")

    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid)
    clocks.start()
    time.sleep(0.3)

    # ---- timed region (device-resident inputs) ----
    n_launch_cap = 3 * args.steps + 8
    trace = K.LaunchTrace(n_launch_cap)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with trace:
        ev0.record(stream)
        for i in range(args.warmup, args.warmup + args.steps):
            dev_step(i)
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    durs = trace.durations()
    launches = len(durs)

    # live step lengths in the timed region (after the append)
    S_steps = [S0 + ((i % T) + 1) for i in range(args.warmup, args.warmup + args.steps)]
    dec = [ms_ for (nm, ms_) in durs if nm == "decode_step"]
    sel = [ms_ for (nm, ms_) in durs if nm == "h2o_select"]
    dec_bytes = sum(step_kernel_bytes([S] * B, Hkv, Hq, d, probs is not None) for S in S_steps) / len(S_steps)
    dec_ms = sum(dec) / len(dec)

    # ---- end to end: host inputs -> device -> host results, every step ----
    e2e_steps = args.steps
    h_q = torch.empty((T, B, Hq, d), dtype=torch.bfloat16, pin_memory=True)
    h_kn = torch.empty((T, B, Hkv, d), dtype=torch.bfloat16, pin_memory=True)
    h_vn = torch.empty((T, B, Hkv, d), dtype=torch.bfloat16, pin_memory=True)
    h_q.copy_(q_all.cpu())
    h_kn.copy_(kn_all.cpu())
    h_vn.copy_(vn_all.cpu())
    h_out = torch.empty((B, Hq, d), dtype=torch.bfloat16, pin_memory=True)
    h_keep = torch.empty((B, Hkv, wl.budget), dtype=torch.int32, pin_memory=True)
    d_q = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=dev)
    d_kn = torch.empty((B, Hkv, d), dtype=torch.bfloat16, device=dev)
    d_vn = torch.empty((B, Hkv, d), dtype=torch.bfloat16, device=dev)
    h2d = (d_q.numel() + d_kn.numel() + d_vn.numel()) * 2
    d2h = h_out.numel() * 2 + h_keep.numel() * 4
    base = args.warmup + args.steps
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(base, base + e2e_steps):
        t = i % T
        d_q.copy_(h_q[t], non_blocking=True)
        d_kn.copy_(h_kn[t], non_blocking=True)
        d_vn.copy_(h_vn[t], non_blocking=True)
        step(i, d_q, d_kn, d_vn)
        h_out.copy_(out, non_blocking=True)
        h_keep.copy_(keep, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    clocks.stop()
    st0, st1 = K.read_status(ws), K.read_status(ws_ev)
    if st0 or st1:
        raise RuntimeError(f"device status after the timed region: {st0} {st1}")

    if rank != 0:
        return
    hbm, peak_kind = peaks()
    if args.batch != 8:
        line_note = f"batch {args.batch}: profiling case, not the measured workload"
    else:
        line_note = None
    steps_per_s = world * args.steps / (ms / 1e3)
    kvb = sum(kv_bytes([S] * B, Hkv, d) for S in S_steps) / len(S_steps)
    eff_kv_gbs = kvb / (ms / args.steps / 1e3) / 1e9
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": CONFIG_NAME, "batch": B, "context": S0, "q_heads": Hq, "kv_heads": Hkv,
                   "head_dim": d, "page": PAGE, "budget": wl.budget, "probs_written": probs is not None,
                   "l2": "inputs larger than L2 (1.07 GB of K/V per step vs 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "effective_kv_gbs": eff_kv_gbs,
        "effective_kv_frac_of_peak": eff_kv_gbs / hbm,
        "kernel_ms": {"decode_step": dec_ms, "h2o_select": sum(sel) / max(1, len(sel))},
        "roofline": {"bound": "hbm", "kernel": "decode_step", "achieved": achieved, "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None},
        "e2e": {"value": world * e2e_steps / (e2e_ms / 1e3), "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "note": line_note,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(args.cpu_pairs, B * Hkv)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3072)
    ap.add_argument("--warmup", type=int, default=128)
    ap.add_argument("--impl", default="kvsel", choices=["kvsel", "reference"])
    ap.add_argument("--no-probs", action="store_true", help="do not keep the probability tensor")
    ap.add_argument("--batch", type=int, default=8, help="sequences (8 = the measured workload; "
                    "smaller only for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=64)
    ap.add_argument("--cpu-worker", type=int, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker is not None:
        cpu_worker_main(args.cpu_worker)
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    cuda_arm(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
