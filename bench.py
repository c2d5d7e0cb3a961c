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



# DRAM bytes (read + write) of one decode_step launch at batch 8 x 32K, from one ncu DRAM-counter
# capture of this kernel (summarised under profiles/); set to None whenever the kernel changes.
DECODE_STEP_TRAFFIC = 1.141956e9

TRACE_EVERY = 8   # launch tracing on one timed step in eight: events between kernels cost time


def slowest_rank(value: float, world: int, device=None) -> float:
    """The largest of the ranks' figures (a replica job takes its slowest rank's
    time); the value itself when running alone."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Units all ranks processed per second over the (slowest rank's) time."""
    return world * units_per_rank / (ms / 1e3)


def replica_seed(base: int, rank: int) -> int:
    """Each replica draws its own synthetic inputs."""
    return base + rank


def timed_steps(step_fn, first, steps, stream, per_step_launches):
    """Run `steps` steps between two events on `stream`; every TRACE_EVERY-th
    step is bracketed by the library's launch trace (events around each of its
    kernels).  Returns (ms, [(kernel, ms)], launches per step)."""
    import attention_guided_kv_gb300 as K
    import torch
    sampled = [i for i in range(first, first + steps) if (i - first) % TRACE_EVERY == 0]
    traces = {i: K.LaunchTrace(per_step_launches + 4) for i in sampled}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(first, first + steps):
        tr = traces.get(i)
        if tr is None:
            step_fn(i)
        else:
            with tr:
                step_fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    durs = [d for tr in traces.values() for d in tr.durations()]
    per_step = max(len(tr.names) for tr in traces.values())
    return e0.elapsed_time(e1), durs, per_step


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# byte model: algorithmic bytes per launch
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
    """The oracle on the host cores, one step at a time.  Each step runs as many of the step's
    64 (sequence, kv head) pairs as fit a ~2-minute budget for the whole --steps/--warmup run:
    all 64 (a whole step, nothing extrapolated) when they fit, else a stated sample scaled to
    the whole step.  ms_per_step is the time the sampled step actually took."""
    if rank != 0:
        return
    B, Hkv = 8, 8
    n_pairs_step = B * Hkv
    cores = len(os.sched_getaffinity(0))
    t_pair = oracle_pair_seconds(1, seed=99)               # one full pair (calibration, untimed)
    per_step = 120.0 / (args.warmup + args.steps)
    pairs = int(min(n_pairs_step, max(1, per_step // max(t_pair, 1e-6))))
    keys = 32769 if per_step >= t_pair else int(max(1024, 32769 * per_step / max(t_pair, 1e-6)))
    frac = (pairs / n_pairs_step) * (min(keys, 32769) / 32769)
    ts = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_pair_seconds(pairs, seed=100 + i, keys=keys)
        t = time.perf_counter() - t0
        if i >= args.warmup:
            ts.append(t)
    mean = sum(ts) / len(ts)                               # seconds the sampled step took
    value = frac / mean                                    # whole steps per second
    sample = (f"each step: {pairs} of the 70B-shape step's {n_pairs_step} (sequence, kv head) pairs over "
              f"{min(keys, 32769)} of their 32769 keys (attention, probabilities, H2O update, select; "
              f"fp64 numpy)" + ("" if frac == 1.0 else f", scaled x{1 / frac:.1f} to the whole step"))
    line = {"metric": METRIC, "value": value, "unit": "steps/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": CONFIG_NAME, "sample_fraction_of_step": frac},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
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

    wl = workloads.decode_70b(seed=replica_seed(1, rank), B=args.batch)
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

    def decode(i, q, kn, vn, o):
        if i % T == 0 and i > 0:
            seq.copy_(seq0)            # replay the 128-step window from 32K again
        K.kvsel_decode_attn(kv, bt, seq, q, o, ws, k_new=kn, v_new=vn, probs=probs, h2o_cum=cum,
                            max_len=max_len, h2o_link=ws_ev)

    def select(kp):
        K.kvsel_h2o_evict(kv, bt, seq, cum, ws_ev, budget=wl.budget, n_sink=wl.n_sink,
                          window=wl.window, compact=False, keep_out=kp)

    def step(i, q, kn, vn):
        decode(i, q, kn, vn, out)
        select(keep)

    def dev_step(i):
        t = i % T
        step(i, q_all[t], kn_all[t], vn_all[t])

    def barrier():
        if world > 1:
            dist.barrier()

    # the clock sampler starts (and settles) before the warm-up, so that the warm-up steps run
    # right before the timed ones with no idle gap between them
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid)
    clocks.start()
    time.sleep(0.3)

    # warm-up
    try:
        for i in range(args.warmup):
            dev_step(i)
        torch.cuda.synchronize()
        st0, st1 = K.read_status(ws), K.read_status(ws_ev)
        if st0 or st1:
            raise RuntimeError(f"device status after warm-up: {st0} {st1}")
    except BaseException:
        clocks.stop()
        raise

    # ---- timed region (device-resident inputs) ----
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms, durs, per_step_launches = timed_steps(dev_step, args.warmup, args.steps, stream, 3)
    barrier()
    t_wall1 = time.time()
    ms = slowest_rank(ms, world, dev)
    launches = per_step_launches * args.steps

    # live step lengths in the timed region (after the append)
    S_steps = [S0 + ((i % T) + 1) for i in range(args.warmup, args.warmup + args.steps)]
    dec = [ms_ for (nm, ms_) in durs if nm == "decode_step"]
    sel = [ms_ for (nm, ms_) in durs if nm == "h2o_select"]
    dec_bytes = sum(step_kernel_bytes([S] * B, Hkv, Hq, d, probs is not None) for S in S_steps) / len(S_steps)
    dec_ms = sum(dec) / len(dec)

    # ---- end to end: host inputs -> device -> host results, every step ----
    # The copies run on two side streams: step i+1's inputs go up and step
    # i-1's results come down while step i computes.  Inputs are double-buffered
    # and results triple-buffered on the device.  Every event operation sits
    # between a decode and its select, so that a decode still starts while the
    # previous select runs.  ev_dec[i] (after decode i) also marks select i-1
    # done, since decode i waits for it before its V pass.
    e2e_steps = args.steps
    import ctypes
    n_q, n_kv = B * Hq * d, B * Hkv * d                  # bf16 elements
    in_bytes = (n_q + 2 * n_kv) * 2                      # one step's q | k_new | v_new
    out_bytes = B * Hq * d * 2
    keep_off = (out_bytes + 255) // 256 * 256
    res_bytes = keep_off + B * Hkv * wl.budget * 4       # one step's O | keep lists
    h_in = torch.empty((T, in_bytes), dtype=torch.uint8, pin_memory=True)
    for t in range(T):
        row = h_in[t]
        row[:n_q * 2].view(torch.bfloat16).copy_(q_all[t].reshape(-1).cpu())
        row[n_q * 2:(n_q + n_kv) * 2].view(torch.bfloat16).copy_(kn_all[t].reshape(-1).cpu())
        row[(n_q + n_kv) * 2:].view(torch.bfloat16).copy_(vn_all[t].reshape(-1).cpu())
    h_res = torch.empty((res_bytes,), dtype=torch.uint8, pin_memory=True)
    d_in = [torch.empty((in_bytes,), dtype=torch.uint8, device=dev) for _ in range(2)]
    d_res = [torch.empty((res_bytes,), dtype=torch.uint8, device=dev) for _ in range(3)]
    h2d, d2h = in_bytes, out_bytes + B * Hkv * wl.budget * 4
    cs_up, cs_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    base = args.warmup + args.steps
    # argument lists marshalled once per buffer (the binding's per-call checks
    # would cost host time that the loop below cannot hide)
    ms_ = ctypes.c_void_p(stream.cuda_stream)
    kvr = ctypes.byref(kv)
    dec_args = {}
    for bi in range(2):
        base_in = d_in[bi].data_ptr()
        for ro in range(3):
            dec_args[bi, ro] = (
                kvr, K._ptr(bt), bt.shape[1], K._ptr(seq), B, ctypes.c_void_p(base_in),
                ctypes.c_void_p(base_in + n_q * 2), ctypes.c_void_p(base_in + (n_q + n_kv) * 2), None, None,
                float(d ** -0.5), ctypes.c_void_p(d_res[ro].data_ptr()), K.KVSEL_BF16, K._ptr(probs), K._ptr(cum),
                int(max_len), 0, None, K._ptr(ws), ws.numel(), K._ptr(ws_ev), ws_ev.numel(), ms_)
    sel_args = [(kvr, K._ptr(bt), bt.shape[1], K._ptr(seq), B, K._ptr(cum), None, int(max_len), int(wl.budget),
                 int(wl.n_sink), int(wl.window), 0, ctypes.c_void_p(d_res[ro].data_ptr() + keep_off), None,
                 K._ptr(ws_ev), ws_ev.numel(), ms_) for ro in range(3)]
    dec_call, sel_call = K.lib().kvsel_decode_attn_ex, K.lib().kvsel_h2o_evict
    ring = 4
    ev_dec = [torch.cuda.Event() for _ in range(ring)]
    ev_up = [torch.cuda.Event() for _ in range(ring)]
    ev_down = [torch.cuda.Event() for _ in range(ring)]

    def e2e_step(i, j):
        if i % T == 0 and i > 0:
            seq.copy_(seq0)            # replay the 128-step window from 32K again
        code = dec_call(*dec_args[j % 2, j % 3])
        if code != K.KVSEL_OK:
            raise RuntimeError(f"kvsel_decode_attn: status {code}")

    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs_up.wait_event(e0)
    with torch.cuda.stream(cs_up):
        d_in[0].copy_(h_in[base % T], non_blocking=True)
    ev_up[0].record(cs_up)
    stream.wait_event(ev_up[0])
    for j in range(e2e_steps):
        i = base + j
        e2e_step(i, j)
        ev_dec[j % ring].record(stream)
        if j + 1 < e2e_steps:             # step j+1's q, k_new, v_new
            # into the buffer decode j-1 read (done once that decode is), so the copy runs during
            # decode j and is in place before select j, which the stream holds until it is
            if j >= 1:
                cs_up.wait_event(ev_dec[(j - 1) % ring])
            with torch.cuda.stream(cs_up):
                d_in[(j + 1) % 2].copy_(h_in[(i + 1) % T], non_blocking=True)
            ev_up[(j + 1) % ring].record(cs_up)
            stream.wait_event(ev_up[(j + 1) % ring])
        if j >= 1:                        # step j-1's O and keep lists
            cs_down.wait_event(ev_dec[j % ring])
            with torch.cuda.stream(cs_down):
                h_res.copy_(d_res[(j - 1) % 3], non_blocking=True)
            ev_down[(j - 1) % ring].record(cs_down)
        if j >= 2:
            stream.wait_event(ev_down[(j - 2) % ring])  # buffers (j+1) % 3 are free again
        code = sel_call(*sel_args[j % 3])
        if code != K.KVSEL_OK:
            raise RuntimeError(f"kvsel_h2o_evict: status {code}")
    ev_dec[0].record(stream)
    cs_down.wait_event(ev_dec[0])
    with torch.cuda.stream(cs_down):
        h_res.copy_(d_res[(e2e_steps - 1) % 3], non_blocking=True)
    ev_down[0].record(cs_down)
    stream.wait_event(ev_down[0])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = slowest_rank(e0.elapsed_time(e1), world, dev)
    clocks.stop()

    # ---- the same step with the per-step top-512 block signal emitted by the decode launch ----
    ws_sig = K.workspace(K.kvsel_decode_attn_ex_workspace(kv, B, max_len, probs is not None, True))
    bscore = torch.zeros(wl.num_pages, device=dev)
    bstep = torch.full((wl.num_pages,), -1, dtype=torch.int32, device=dev)
    btop = torch.zeros(B, 512, dtype=torch.int32, device=dev)

    def sig_step(i):
        t = i % T
        if t == 0 and i > 0:
            seq.copy_(seq0)
        K.kvsel_decode_attn(kv, bt, seq, q_all[t], out, ws_sig, k_new=kn_all[t], v_new=vn_all[t], probs=probs,
                            h2o_cum=cum, max_len=max_len, h2o_link=ws_ev, block_score=bscore, block_step=bstep,
                            signal_topk=512, signal_step=i, signal_topk_out=btop)
        K.kvsel_h2o_evict(kv, bt, seq, cum, ws_ev, budget=wl.budget, n_sink=wl.n_sink,
                          window=wl.window, compact=False, keep_out=keep)
    seq.copy_(seq0)
    for i in range(3):
        sig_step(i)
    torch.cuda.synchronize()
    v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for i in range(3, 3 + 64):
        sig_step(i)
    v1.record(stream)
    torch.cuda.synchronize()
    sig_ms = v0.elapsed_time(v1) / 64
    if K.read_status(ws_sig):
        raise RuntimeError(f"device status after the block-signal steps: {K.read_status(ws_sig)}")
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
    steps_per_s = job_rate(world, args.steps, ms)
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
                   "h2o_scores": ("start at zero and accumulate over the replayed 128-step window; the "
                                  "first tens of steps hand the select longer candidate lists"),
                   "parallelism": f"replicas x{world}"},
        "effective_kv_gbs": eff_kv_gbs,
        "effective_kv_frac_of_peak": eff_kv_gbs / hbm,
        "kernel_ms": {"decode_step": dec_ms, "h2o_select": sum(sel) / max(1, len(sel))},
        "roofline": {"bound": "hbm", "kernel": "decode_step", "achieved": achieved, "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": DECODE_STEP_TRAFFIC if B == 8 else None,
                     "algorithmic_bytes": dec_bytes},
        "e2e": {"value": job_rate(world, e2e_steps, e2e_ms), "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "variants_ms_per_step": {"with_block_signal_top512": sig_ms},
        "note": line_note,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(args.cpu_pairs, B * Hkv)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the other hot-path workloads (one JSON line each)
# ---------------------------------------------------------------------------
WORKLOADS = {
    "decode_70b": None,
    "decode_small": ("decode steps/s with H2O evict + compaction every step",
                     "single seq, 16 q / 8 kv heads, d=128, prompt 1600, 64 decode steps, H2O budget "
                     "256 = 4 sinks + 64 window + 188 heavy hitters, evict and compact every step",
                     "steps/s"),
    "snapkv": ("SnapKV prefill selects/s (all 28 layers)",
               "SnapKV prefill select, Qwen2.5-7B shape (28 layers, 28 q / 4 kv heads, d=128), prompt "
               "32K, obs window 32, sum vote, maxpool 7, keep 2048 per kv head", "selects/s"),
    "block_priority": ("block offload priority passes/s",
                       "block offload priority: 64 requests, lengths log-uniform 4K-128K, Dirichlet "
                       "increments with decay 0.98, 16-token blocks, max aggregation, per-request "
                       "percentile, evict order for 25% of blocks", "passes/s"),
    "sparse_decode": ("sparse decode steps/s",
                      "DSA-style sparse decode, 70B shape (64 q / 8 kv heads, d=128), batch 4, 128K "
                      "context, indexer 4 x 64, top-2048", "steps/s"),
}


def _dev_bf16(bits, dev):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _setup_decode_small(dev, small=False):
    """Evict-every-step loop: append + attention + probabilities + H2O update, then select +
    compaction; the caller's allocator hands the page released at index 16 back for the
    next append (budget 256 = 16 full pages)."""
    import numpy as np
    import torch
    import attention_guided_kv_gb300 as K
    import workloads
    wl = workloads.decode_small()
    kpool = _dev_bf16(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages), dev)
    vpool = _dev_bf16(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages), dev)
    kv = K.paged_kv(kpool, vpool, wl.Hq)
    bt = torch.from_numpy(wl.block_table).to(dev)
    seq = torch.full((1,), wl.S0, dtype=torch.int32, device=dev)
    cum = torch.zeros(1, wl.Hkv, wl.max_len, device=dev)
    probs = torch.zeros(1, wl.Hq, wl.max_len, device=dev)
    pos = torch.from_numpy(np.tile(np.arange(wl.max_len, dtype=np.int32), (1, wl.Hkv, 1))).to(dev)
    nxt = torch.full((1,), wl.S0, dtype=torch.int32, device=dev)
    out = torch.zeros(1, wl.Hq, wl.d, device=dev, dtype=torch.bfloat16)
    keep = torch.zeros(1, wl.Hkv, wl.budget, dtype=torch.int32, device=dev)
    freed = torch.zeros(1, wl.max_pages, dtype=torch.int32, device=dev)
    ws = K.workspace(K.kvsel_decode_attn_workspace(kv, 1, wl.max_len, True))
    ws2 = K.workspace(K.kvsel_h2o_evict_workspace(kv, 1, wl.budget))
    q, kn, vn = _dev_bf16(wl.q, dev), _dev_bf16(wl.k_new, dev), _dev_bf16(wl.v_new, dev)
    page = wl.budget // 16

    def run(i, qi, kni, vni):
        K.kvsel_decode_attn(kv, bt, seq, qi, out, ws, k_new=kni, v_new=vni, pos_map=pos, next_pos=nxt,
                            probs=probs, h2o_cum=cum, max_len=wl.max_len, h2o_link=ws2)
        K.kvsel_h2o_evict(kv, bt, seq, cum, ws2, budget=wl.budget, n_sink=wl.n_sink, window=wl.window,
                          compact=True, pos_map=pos, keep_out=keep, freed_pages=freed)
        bt[:, page].copy_(freed[:, 0])

    def step(i):
        t = i % wl.steps
        run(i, q[t], kn[t], vn[t])

    host_in = [("q", q), ("k_new", kn), ("v_new", vn)]
    outs = [out, keep]
    # bytes of the dominant kernel (decode_step) per launch at the steady length 257
    S = wl.budget + 1
    byts = {"decode_step": S * wl.Hkv * 512 + S * wl.Hq * 4 + S * wl.Hkv * 8 + wl.Hq * wl.d * 4}
    return dict(step=step, run=run, host_in=host_in, outs=outs, bytes=byts, flops={},
                ws=[ws, ws2], per_step_launches=4, graph_cycle=True, config={"batch": 1, "context": wl.S0,
                "q_heads": wl.Hq, "kv_heads": wl.Hkv, "budget": wl.budget, "steps_cycle": wl.steps,
                "l2": "working set (~1 MB) fits in L2: latency-bound"})


def _setup_snapkv(dev, small=False):
    import numpy as np
    import torch
    import attention_guided_kv_gb300 as K
    import workloads
    wl = workloads.snapkv_qwen7b(L=4 if small else 28)
    P = wl.pages
    pool = np.zeros((wl.L * P, wl.Hkv, 16, wl.d), dtype=np.uint16)
    bts = np.zeros((wl.L, P), dtype=np.int32)
    qo = np.zeros((wl.L, wl.Hq, wl.W, wl.d), dtype=np.uint16)
    for l in range(wl.L):
        lay = wl.layer(l)
        pool[l * P:(l + 1) * P] = workloads.paged_pool(lay.K[None], lay.block_table[None], P)
        bts[l] = lay.block_table + l * P
        qo[l] = lay.q_obs
    kpool = _dev_bf16(pool, dev)
    del pool
    kv = K.paged_kv(kpool, kpool, wl.Hq)
    bt = torch.from_numpy(bts).to(dev)
    q = _dev_bf16(qo, dev)
    keep = torch.zeros(wl.L, wl.Hkv, wl.keep_k + wl.W, dtype=torch.int32, device=dev)
    vote = torch.zeros(wl.L, wl.Hkv, wl.S - wl.W, device=dev)
    ws = K.workspace(K.kvsel_snapkv_select_workspace(kv, wl.L, wl.S, wl.W, True))

    def run(i, qi):
        K.kvsel_snapkv_select(kv, bt, qi, keep, ws, seq_len=wl.S, keep_k=wl.keep_k,
                              pool_kernel=wl.pool_kernel, vote_out=vote)

    def step(i):
        run(i, q)

    # the GQA-union keep mode and the cold-start seeds (timed apart, same inputs)
    cap_u = wl.G * wl.keep_k + wl.W
    keep_u = torch.zeros(wl.L, wl.Hkv, cap_u, dtype=torch.int32, device=dev)
    count = torch.zeros(wl.L, wl.Hkv, dtype=torch.int32, device=dev)
    seed = torch.zeros(wl.L, wl.Hkv, cap_u, device=dev)
    ws_u = K.workspace(K.kvsel_snapkv_select_ex_workspace(kv, wl.L, wl.S, wl.W, False, K.KVSEL_SNAP_HEAD_UNION))

    def run_ex(mode, seeds):
        cap = cap_u if mode == K.KVSEL_SNAP_HEAD_UNION else wl.keep_k + wl.W
        so = dict(seed_out=seed, seed_layer_stride=wl.Hkv * cap, seed_head_stride=cap) if seeds else {}
        return lambda i: K.kvsel_snapkv_select_ex(
            kv, bt, q, keep_u if mode == K.KVSEL_SNAP_HEAD_UNION else keep, ws_u, seq_len=wl.S,
            keep_k=wl.keep_k, mode=mode, pool_kernel=wl.pool_kernel, keep_count=count, **so)
    variant_runs = [("group_sum_with_seeds", run_ex(K.KVSEL_SNAP_GROUP_SUM, True)),
                    ("head_union", run_ex(K.KVSEL_SNAP_HEAD_UNION, False)),
                    ("head_union_with_seeds", run_ex(K.KVSEL_SNAP_HEAD_UNION, True))]

    def compact_after():
        """Compaction of the kept prompt cache (kvsel_kv_compact on the group-sum keep lists), timed
        once the selections above are done: it rewrites the pool in place, so every repetition first
        restores the lengths and the block table (outside the timed events) and then moves the same
        rows again (same bytes moved)."""
        vpool = torch.empty_like(kpool)
        kvc = K.paged_kv(kpool, vpool, wl.Hq)
        count_g = torch.zeros(wl.L, wl.Hkv, dtype=torch.int32, device=dev)
        K.kvsel_snapkv_select_ex(kvc, bt, q, keep, ws_u, seq_len=wl.S, keep_k=wl.keep_k,
                                 pool_kernel=wl.pool_kernel, keep_count=count_g)
        bt0 = bt.clone()
        lens = torch.full((wl.L,), wl.S, dtype=torch.int32, device=dev)
        freed = torch.zeros(wl.L, P, dtype=torch.int32, device=dev)
        ws_c = K.workspace(K.kvsel_kv_compact_workspace(wl.L, wl.Hkv))
        times = []
        for rep in range(6):
            bt.copy_(bt0)
            lens.fill_(wl.S)
            torch.cuda.synchronize()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            K.kvsel_kv_compact(kvc, bt, lens, keep, ws_c, keep_count=count_g, freed_pages=freed)
            b2.record()
            torch.cuda.synchronize()
            if rep >= 2:
                times.append(a.elapsed_time(b2) * 1e3)
        if K.read_status(ws_c):
            raise RuntimeError("device status after the compaction")
        bt.copy_(bt0)
        us = sum(times) / len(times)
        moved = wl.L * wl.Hkv * (wl.keep_k + wl.W) * 2 * 512   # K and V rows, read and written
        return {"compact_us": us, "compact_gbs": moved / (us * 1e-6) / 1e9,
                "compact_note": "kvsel_kv_compact of the 28 x 4 x 2080 kept rows (K and V, read + write "
                                "1024 B per row), mean of 4 calls after 2 untimed"}

    pairs = wl.L * wl.Hkv
    rows = wl.G * wl.W
    qk_flops = 2.0 * rows * wl.S * wl.d * pairs
    kbytes = wl.S * wl.d * 2 * pairs
    # one exp2 per (window row, key) in each pass: the special-function unit bounds both
    ex2 = {"snap_stats": float(rows) * wl.S * pairs, "snap_vote": float(rows) * (wl.S - wl.W) * pairs}
    return dict(step=step, run=run, host_in=[("q_obs", q[None])], outs=[keep], ws=[ws, ws_u],
                bytes={"snap_stats": kbytes, "snap_vote": kbytes}, flops={"snap_stats": qk_flops,
                "snap_vote": 2.0 * rows * (wl.S - wl.W) * wl.d * pairs}, ex2=ex2, per_step_launches=3,
                variant_runs=variant_runs, variants_key="variants_us_per_select", after=compact_after,
                config={"layers": wl.L, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "prompt": wl.S,
                        "obs_window": wl.W, "keep": wl.keep_k, "pool_kernel": wl.pool_kernel,
                        "l2": "inputs larger than L2 (940 MB of K per pass)"})


def _setup_block_priority(dev, small=False):
    import numpy as np
    import torch
    import attention_guided_kv_gb300 as K
    import workloads
    wl = workloads.block_priority()
    off = torch.from_numpy(wl.offsets).to(dev)
    tok = torch.from_numpy(wl.increments(0)).to(dev)
    incs = [torch.from_numpy(wl.increments(t)).to(dev) for t in range(1, 5)]
    nblk = int(sum(-(-int(L) // 16) for L in wl.lengths))
    order = torch.zeros(-(-nblk // 4), dtype=torch.int64, device=dev)
    n_out = torch.zeros(2, dtype=torch.int64, device=dev)
    maxb = int(sum(-(-int(L) // 1) for L in wl.lengths))      # bound for every block size
    ws = K.workspace(K.kvsel_block_priority_workspace(wl.R, maxb))
    variant = dict(block_size=16, agg=K.KVSEL_AGG_MAX, norm=K.KVSEL_NORM_PERCENTILE)
    hist = torch.zeros(8, wl.total_tokens, device=dev)   # sliding-window update: 8 steps

    def run(i, inc, **v):
        if v.get("update") == K.KVSEL_UPDATE_WINDOW:
            v = dict(v, history=hist, window=8, step=i)
        opts = dict(variant)
        opts.update(v)
        K.kvsel_block_priority(tok, off, order, n_out, ws, evict_frac=0.25, increment=inc, decay=0.98,
                               top_p=0.1, max_total_blocks=maxb, **opts)

    def step(i):
        run(i, incs[i % 4])

    T = wl.total_tokens
    byts = {"bp_fold": T * 12 + nblk * 4, "bp_rank": nblk * 12, "bp_sort": nblk * 12 * 2 * 8,
            "bp_prefix": wl.R * 16}
    return dict(step=step, run=run, host_in=[("increment", incs[0][None])], outs=[order, n_out], ws=[ws],
                bytes=byts, flops={}, per_step_launches=4, extra_variants=True, nblk=nblk, incs=incs,
                config={"requests": wl.R, "tokens": T, "blocks": nblk, "block_size": 16, "agg": "max",
                        "norm": "percentile", "evict_frac": 0.25,
                        "l2": "~9 MB of token scores per pass (fits in L2): latency-bound"})


class _Rt:
    """The CUDA runtime that torch has loaded, called through ctypes for a loop's per-step copies
    and event operations: torch's Python wrappers cost several microseconds of host time a call,
    more than a short step leaves.  `ok` is False where the library cannot be found."""

    def __init__(self, dev):
        import ctypes
        self.lib = None
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        self.ok = self.lib is not None
        if not self.ok:
            return
        vp = ctypes.c_void_p
        L = self.lib
        L.cudaSetDevice.argtypes = [ctypes.c_int]
        L.cudaMemcpyAsync.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int, vp]
        L.cudaEventRecord.argtypes = [vp, vp]
        L.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
        L.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        L.cudaEventDestroy.argtypes = [vp]
        for f in (L.cudaSetDevice, L.cudaMemcpyAsync, L.cudaEventRecord, L.cudaStreamWaitEvent,
                  L.cudaEventCreateWithFlags, L.cudaEventDestroy):
            f.restype = ctypes.c_int
        self.check(L.cudaSetDevice(dev.index or 0), "cudaSetDevice")

    @staticmethod
    def check(code, what):
        if code != 0:
            raise RuntimeError(f"{what}: CUDA error {code}")

    def events(self, n):
        import ctypes
        out = []
        for _ in range(n):
            h = ctypes.c_void_p()
            self.check(self.lib.cudaEventCreateWithFlags(ctypes.byref(h), 2), "cudaEventCreateWithFlags")  # no timing
            out.append(h)
        return out

    def destroy(self, evs):
        for h in evs:
            self.check(self.lib.cudaEventDestroy(h), "cudaEventDestroy")


def _setup_sparse_decode(dev, small=False):
    import numpy as np
    import torch
    import attention_guided_kv_gb300 as K
    import workloads
    wl = workloads.sparse_decode(B=1 if small else 4)
    kpool = _dev_bf16(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages), dev)
    vpool = _dev_bf16(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages), dev)
    wl.K = wl.V = None
    kv = K.paged_kv(kpool, vpool, wl.Hq)
    bt = torch.from_numpy(wl.block_table).to(dev)
    seq0 = torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev)
    seq = seq0.clone()
    idx = np.zeros((wl.B, wl.max_len, wl.Di), dtype=np.uint16)
    idx[:, :wl.S0] = wl.k_idx
    idx_k = _dev_bf16(idx, dev)
    del idx
    q, kn, vn = _dev_bf16(wl.q, dev), _dev_bf16(wl.k_new, dev), _dev_bf16(wl.v_new, dev)
    qi, kin = _dev_bf16(wl.q_idx, dev), _dev_bf16(wl.k_idx_new, dev)
    wi = torch.from_numpy(wl.w_idx).to(dev)
    out = torch.zeros(wl.B, wl.Hq, wl.d, device=dev, dtype=torch.bfloat16)
    topk = torch.zeros(wl.B, wl.top_k, dtype=torch.int32, device=dev)
    ws = K.workspace(K.kvsel_sparse_decode_workspace(kv, wl.B, wl.max_len, wl.top_k, False))

    def run(i, q_, qi_, wi_, kn_, vn_, kin_):
        if i % wl.steps == 0 and i > 0:
            seq.copy_(seq0)                 # replay the 64-step window from 128K again
        K.kvsel_sparse_decode(kv, bt, seq, q_, qi_, wi_, idx_k, out, ws, top_k=wl.top_k, k_new=kn_,
                              v_new=vn_, idx_k_new=kin_, topk_out=topk)

    # The timed steps call the C ABI with argument lists marshalled once per step of the 64-step
    # window (the binding's per-call checks cost more host time than the GPU spends on a step).
    import ctypes
    Sc = torch.cuda.current_stream()
    fixed = dict(kv=ctypes.byref(kv), bt=K._ptr(bt), mp=bt.shape[1], seq=K._ptr(seq), B=wl.B, idx_k=K._ptr(idx_k),
                 out=K._ptr(out), topk=K._ptr(topk), ws=K._ptr(ws), wsb=ws.numel())
    argsets = [(fixed["kv"], fixed["bt"], fixed["mp"], fixed["seq"], fixed["B"], K._ptr(q[t]), K._ptr(kn[t]),
                K._ptr(vn[t]), K._ptr(qi[t]), K._ptr(wi[t]), fixed["idx_k"], K._ptr(kin[t]), wl.Hi, wl.Di,
                wl.max_len, wl.top_k, float(wl.scale), fixed["out"], K.KVSEL_BF16, fixed["topk"], None,
                fixed["ws"], fixed["wsb"], ctypes.c_void_p(Sc.cuda_stream)) for t in range(wl.steps)]
    call = K.lib().kvsel_sparse_decode

    def step(i):
        t = i % wl.steps
        if t == 0 and i > 0:
            seq.copy_(seq0)                 # replay the 64-step window from 128K again
        code = call(*argsets[t])
        if code != K.KVSEL_OK:
            raise RuntimeError(f"kvsel_sparse_decode: status {code}")

    # Quest page selection on the same cache: top_k / 16 pages (2048 tokens) per q head
    budget_pages = wl.top_k // 16
    meta = torch.zeros(wl.num_pages, wl.Hkv, wl.page // 16, 2, wl.d, dtype=torch.bfloat16, device=dev)
    seq_q = seq0.clone()
    ws_q = K.workspace(K.kvsel_quest_decode_workspace(kv, wl.B, wl.max_pages, budget_pages))
    K.kvsel_quest_page_meta(kv, bt, seq_q, meta, ws_q)
    out_q = torch.zeros_like(out)

    def quest(i):
        t = i % wl.steps
        if t == 0 and i > 0:
            seq_q.copy_(seq0)
        K.kvsel_quest_decode(kv, bt, seq_q, q[t], meta, out_q, ws_q, budget_pages=budget_pages, k_new=kn[t],
                             v_new=vn[t])

    # ---- end to end: one packed upload of a step's six inputs, one packed download of its O and
    # top-k positions, on two side streams.  Inputs are double-buffered and results
    # triple-buffered on the device; the events that order them sit between steps (the three
    # launches of a step come from one call).  Argument lists are marshalled once per buffer.
    def al(n):
        return (n + 255) // 256 * 256
    parts = [("q", q), ("q_idx", qi), ("w_idx", wi), ("k_new", kn), ("v_new", vn), ("k_idx_new", kin)]
    offs, in_bytes = {}, 0
    for nm, t in parts:
        offs[nm] = in_bytes
        in_bytes += al(t[0].numel() * t.element_size())
    h_in = torch.zeros((wl.steps, in_bytes), dtype=torch.uint8, pin_memory=True)
    for nm, t in parts:
        nb = t[0].numel() * t.element_size()
        h_in[:, offs[nm]:offs[nm] + nb].copy_(t.reshape(wl.steps, -1).view(torch.uint8).cpu())
    out_bytes = out.numel() * out.element_size()
    topk_off = al(out_bytes)
    res_bytes = topk_off + topk.numel() * 4
    h_res = torch.empty((res_bytes,), dtype=torch.uint8, pin_memory=True)
    d_in = [torch.empty((in_bytes,), dtype=torch.uint8, device=dev) for _ in range(2)]
    d_res = [torch.empty((res_bytes,), dtype=torch.uint8, device=dev) for _ in range(3)]
    e2e_args = {}
    for bi in range(2):
        a = d_in[bi].data_ptr()
        pv = {nm: ctypes.c_void_p(a + o) for nm, o in offs.items()}
        for ro in range(3):
            r0 = d_res[ro].data_ptr()
            e2e_args[bi, ro] = (fixed["kv"], fixed["bt"], fixed["mp"], fixed["seq"], fixed["B"], pv["q"],
                                pv["k_new"], pv["v_new"], pv["q_idx"], pv["w_idx"], fixed["idx_k"], pv["k_idx_new"],
                                wl.Hi, wl.Di, wl.max_len, wl.top_k, float(wl.scale), ctypes.c_void_p(r0),
                                K.KVSEL_BF16, ctypes.c_void_p(r0 + topk_off), None, fixed["ws"], fixed["wsb"],
                                ctypes.c_void_p(Sc.cuda_stream))

    rt = _Rt(dev)

    def e2e_rt(base, n, cs_up, cs_down, ring):  # the loop below, its copies and events through ctypes
        L, vp = rt.lib, ctypes.c_void_p
        evs = rt.events(3 * ring)
        ev_step, ev_up, ev_down = evs[:ring], evs[ring:2 * ring], evs[2 * ring:]
        sC, sU, sD = vp(Sc.cuda_stream), vp(cs_up.cuda_stream), vp(cs_down.cuda_stream)
        hin0, hres = h_in.data_ptr(), vp(h_res.data_ptr())
        din = [vp(t.data_ptr()) for t in d_in]
        dres = [vp(t.data_ptr()) for t in d_res]
        rec, wait, cp = L.cudaEventRecord, L.cudaStreamWaitEvent, L.cudaMemcpyAsync
        try:
            return e2e_rt_loop(base, n, cs_up, ring, ev_step, ev_up, ev_down, sC, sU, sD, hin0, hres, din, dres,
                               rec, wait, cp)
        finally:
            torch.cuda.synchronize()
            rt.destroy(evs)

    def e2e_rt_loop(base, n, cs_up, ring, ev_step, ev_up, ev_down, sC, sU, sD, hin0, hres, din, dres, rec, wait, cp):
        vp = ctypes.c_void_p
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(Sc)
        cs_up.wait_event(e0)
        err = cp(din[0], vp(hin0 + (base % wl.steps) * in_bytes), in_bytes, 1, sU)
        err |= rec(ev_up[0], sU) | wait(sC, ev_up[0], 0)
        for j in range(n):
            i = base + j
            if i % wl.steps == 0 and i > 0:
                seq.copy_(seq0)             # replay the 64-step window from 128K again
            code = call(*e2e_args[j % 2, j % 3])
            if code != K.KVSEL_OK:
                raise RuntimeError(f"kvsel_sparse_decode: status {code}")
            err |= rec(ev_step[j % ring], sC)
            if j + 1 < n:                   # step j+1's inputs, into the buffer step j-1 read
                if j >= 1:
                    err |= wait(sU, ev_step[(j - 1) % ring], 0)
                err |= cp(din[(j + 1) % 2], vp(hin0 + ((i + 1) % wl.steps) * in_bytes), in_bytes, 1, sU)
                err |= rec(ev_up[(j + 1) % ring], sU) | wait(sC, ev_up[(j + 1) % ring], 0)
            err |= wait(sD, ev_step[j % ring], 0)   # step j's O and top-k down
            err |= cp(hres, dres[j % 3], res_bytes, 2, sD) | rec(ev_down[j % ring], sD)
            if j >= 2:
                err |= wait(sC, ev_down[(j - 2) % ring], 0)  # result buffer (j + 1) % 3 is free again
            if err:
                raise RuntimeError(f"end-to-end loop: CUDA error {err} at step {j}")
        err = wait(sC, ev_down[(n - 1) % ring], 0)
        e1.record(Sc)
        torch.cuda.synchronize()
        rt.check(err, "cudaStreamWaitEvent")
        return e0.elapsed_time(e1), in_bytes, res_bytes

    def e2e(base, n):
        cs_up, cs_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ring = 4
        if rt.ok:
            return e2e_rt(base, n, cs_up, cs_down, ring)
        ev_step = [torch.cuda.Event() for _ in range(ring)]
        ev_up = [torch.cuda.Event() for _ in range(ring)]
        ev_down = [torch.cuda.Event() for _ in range(ring)]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(Sc)
        cs_up.wait_event(e0)
        with torch.cuda.stream(cs_up):
            d_in[0].copy_(h_in[base % wl.steps], non_blocking=True)
        ev_up[0].record(cs_up)
        Sc.wait_event(ev_up[0])
        for j in range(n):
            i = base + j
            if i % wl.steps == 0 and i > 0:
                seq.copy_(seq0)             # replay the 64-step window from 128K again
            code = call(*e2e_args[j % 2, j % 3])
            if code != K.KVSEL_OK:
                raise RuntimeError(f"kvsel_sparse_decode: status {code}")
            ev_step[j % ring].record(Sc)
            if j + 1 < n:                   # step j+1's inputs, into the buffer step j-1 read
                if j >= 1:
                    cs_up.wait_event(ev_step[(j - 1) % ring])
                with torch.cuda.stream(cs_up):
                    d_in[(j + 1) % 2].copy_(h_in[(i + 1) % wl.steps], non_blocking=True)
                ev_up[(j + 1) % ring].record(cs_up)
                Sc.wait_event(ev_up[(j + 1) % ring])
            cs_down.wait_event(ev_step[j % ring])   # step j's O and top-k down
            with torch.cuda.stream(cs_down):
                h_res.copy_(d_res[j % 3], non_blocking=True)
            ev_down[j % ring].record(cs_down)
            if j >= 2:
                Sc.wait_event(ev_down[(j - 2) % ring])  # result buffer (j + 1) % 3 is free again
        Sc.wait_event(ev_down[(n - 1) % ring])
        e1.record(Sc)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), in_bytes, res_bytes

    S = wl.S0 + wl.steps // 2
    byts = {"sd_index": wl.B * S * (wl.Di * 2 + 4), "sd_attn": wl.B * wl.top_k * wl.Hkv * 512,
            "sd_select": wl.B * S * 4}
    host_in = [("q", q), ("q_idx", qi), ("w_idx", wi), ("k_new", kn), ("v_new", vn), ("k_idx_new", kin)]
    return dict(step=step, run=run, host_in=host_in, outs=[out, topk], ws=[ws, ws_q], bytes=byts, flops={},
                per_step_launches=3, steps_cycle=wl.steps, e2e_graph=False, e2e=e2e,
                e2e_launch=("C ABI called eagerly, copies overlapped on side streams"
                            + ("; copies and events through the CUDA runtime" if rt.ok else "")),
                variant_runs=[(f"quest_{budget_pages}_pages_per_head", quest)], variants_key="variants_us_per_step",
                config={"batch": wl.B, "context": wl.S0, "q_heads": wl.Hq, "kv_heads": wl.Hkv,
                        "indexer": f"{wl.Hi} x {wl.Di}", "top_k": wl.top_k,
                        "l2": "inputs larger than L2 (67 MB indexer keys + 33.5 MB gathered K/V per step)"})


SETUPS = {"decode_small": _setup_decode_small, "snapkv": _setup_snapkv,
          "block_priority": _setup_block_priority, "sparse_decode": _setup_sparse_decode}


def _oracle_decode_small():
    import numpy as np
    import workloads
    from oracle.attention import bf16_bits_to_f64
    from oracle.h2o import H2OSequence
    wl = workloads.decode_small()
    seq = H2OSequence(bf16_bits_to_f64(wl.K[0]), bf16_bits_to_f64(wl.V[0]))
    args = [(bf16_bits_to_f64(wl.q[t, 0]), bf16_bits_to_f64(wl.k_new[t, 0]), bf16_bits_to_f64(wl.v_new[t, 0]))
            for t in range(wl.steps)]
    seq.step(*args[0], wl.scale, wl.budget, wl.n_sink, wl.window)       # first step from 1600
    t0 = time.perf_counter()
    for a in args[1:]:
        seq.step(*a, wl.scale, wl.budget, wl.n_sink, wl.window)
    dt = (time.perf_counter() - t0) / (wl.steps - 1)
    return {"seconds_per_unit": dt, "sample": f"{wl.steps - 1} steady-state steps (append, attention, "
            f"H2O update, select, compaction; fp64 numpy)", "scale": 1}


def _oracle_snapkv():
    import workloads
    from oracle import snapkv
    from oracle.attention import bf16_bits_to_f64
    wl = workloads.snapkv_qwen7b()
    lay = wl.layer(0)
    G = wl.G
    t0 = time.perf_counter()
    v = snapkv.snapkv_vote(bf16_bits_to_f64(lay.q_obs[:G]), bf16_bits_to_f64(lay.K[:1]), wl.scale)
    pooled = snapkv.maxpool1d(v, wl.pool_kernel)
    snapkv.snapkv_keep(pooled[0], wl.S, wl.W, wl.keep_k)
    dt = time.perf_counter() - t0
    pairs = wl.L * wl.Hkv
    return {"seconds_per_unit": dt * pairs, "sample": f"one (layer, kv head) of {pairs} (vote, max-pool, "
            f"keep; fp64 numpy), scaled x{pairs}", "scale": pairs}


def _oracle_block_priority():
    import numpy as np
    import workloads
    from oracle import block_priority as BP
    wl = workloads.block_priority()
    tok = wl.increments(0).astype(np.float64)
    inc = wl.increments(1).astype(np.float64)
    t0 = time.perf_counter()
    tok = BP.decay_update(tok, inc, 0.98)
    BP.priority_pass(tok, wl.offsets, 16, BP.AGG_MAX, 0.1, BP.NORM_PERCENTILE, 0.25)
    dt = time.perf_counter() - t0
    return {"seconds_per_unit": dt, "sample": "one full pass (decay update, fold, percentile, global "
            "order) over all 64 requests (fp64 numpy)", "scale": 1}


def _oracle_sparse_decode():
    import numpy as np
    import workloads
    from oracle import dsa
    from oracle.attention import bf16_bits_to_f64
    wl = workloads.sparse_decode(B=1, steps=1)
    Kb, Vb = bf16_bits_to_f64(wl.K[0]), bf16_bits_to_f64(wl.V[0])
    ki = bf16_bits_to_f64(wl.k_idx[0])
    t0 = time.perf_counter()
    dsa.sparse_decode_step(bf16_bits_to_f64(wl.q[0, 0]), Kb, Vb, bf16_bits_to_f64(wl.q_idx[0, 0]),
                           wl.w_idx[0, 0].astype(np.float64), ki, wl.top_k, wl.scale)
    dt = time.perf_counter() - t0
    return {"seconds_per_unit": dt * 4, "sample": "one sequence of the batch of 4 (indexer over 128K "
            "keys, top-2048, attention over the selection; fp64 numpy), scaled x4", "scale": 4}


ORACLE_SAMPLES = {"decode_small": _oracle_decode_small, "snapkv": _oracle_snapkv,
                  "block_priority": _oracle_block_priority, "sparse_decode": _oracle_sparse_decode}


def _oracle_subprocess(name):
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", name],
                       capture_output=True, text=True, env=env, timeout=1200)
    line = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not line:
        return None, cores
    return json.loads(line[-1]), cores


def other_reference(args, world):
    metric, cfg, unit = WORKLOADS[args.workload]
    ts = []
    for i in range(args.warmup + args.steps):
        res = ORACLE_SAMPLES[args.workload]()
        if i >= args.warmup:
            ts.append(res["seconds_per_unit"])
    mean = sum(ts) / len(ts)
    cores = len(os.sched_getaffinity(0))
    line = {"metric": metric, "value": 1.0 / mean, "unit": unit, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg},
            "cpu_baseline": {"value": 1.0 / mean, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": 1.0 / mean, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def other_workload(args, rank, world):
    import torch
    import torch.distributed as dist
    import attention_guided_kv_gb300 as K
    metric, cfg_name, unit = WORKLOADS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K.lib()
    S = SETUPS[args.workload](dev, small=args.small)
    stream = torch.cuda.current_stream()
    steps = args.steps
    # the clock sampler starts (and settles) before the warm-up: no idle gap before the timed steps
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid)
    clocks.start()
    time.sleep(0.3)
    try:
        for i in range(args.warmup):
            S["step"](i)
        torch.cuda.synchronize()
        for w in S["ws"]:
            st = K.read_status(w)
            if st:
                raise RuntimeError(f"device status after warm-up: {st}")
    except BaseException:
        clocks.stop()
        raise
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    ms, durs, per_step_launches = timed_steps(S["step"], args.warmup, steps, stream, S["per_step_launches"])
    tw1 = time.time()
    eager_ms = None
    if S.get("graph_cycle") and not args.no_graph:
        # Launch-bound loop: the same K steps captured once in a CUDA graph and
        # replayed (once untimed, once timed), so the host's per-call overhead
        # does not gate the GPU.  The per-kernel times above come from the
        # eager (traced) steps.
        eager_ms = ms
        base0 = args.warmup + steps
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(base0, base0 + steps):
                S["step"](i)
        g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        tw1 = time.time()
        ms = ga.elapsed_time(gb)
    ms = slowest_rank(ms, world, dev)
    per = {}
    for nm, d in durs:
        per.setdefault(nm, []).append(d)
    kern_ms = {k: sum(v) / len(v) for k, v in per.items()}
    dominant = max(kern_ms, key=lambda k: kern_ms[k] * len(per[k]))

    # end to end: every step copies its inputs from pinned host memory and its results back
    hin = [(n, t.cpu().pin_memory()) for n, t in S["host_in"]]
    dins = [torch.empty_like(t[0]) for _, t in S["host_in"]]
    houts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in S["outs"]]
    h2d = sum(t[0].numel() * t.element_size() for _, t in hin)
    d2h = sum(o.numel() * o.element_size() for o in S["outs"])
    base = args.warmup + steps
    cyc = S.get("steps_cycle", None)

    def e2e_run(i0, n):  # n steps: each one's inputs up, the step through the binding, results down
        for i in range(i0, i0 + n):
            for (nm_, h), d in zip(hin, dins):
                d.copy_(h[i % h.shape[0]], non_blocking=True)
            if args.workload in ("snapkv", "block_priority"):
                S["run"](i, dins[0])
            else:
                S["run"](i, *dins)
            for ho, o in zip(houts, S["outs"]):
                ho.copy_(o, non_blocking=True)

    # Where the workload allows it, the steps, copies included, are captured once as a CUDA graph
    # of one cycle of the workload (64 steps when it has none) and replayed, so the host's per-call
    # overhead (binding checks, the launches and the copies of every step) does not gate the GPU.
    # The sparse decode is not captured (its entry point is documented as not graph-capturable)
    # and runs its steps eagerly.
    cap = cyc or 64
    e2e_graph = None
    e2e_own = None
    if S.get("e2e") is not None:  # the workload's own loop (packed copies overlapped with the steps)
        e2e_own = S["e2e"](base, steps)
    elif S.get("e2e_graph", True) and not args.no_graph:
        gr = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(gr):
            e2e_run(base, cap)
        gr.replay()
        torch.cuda.synchronize()
        e2e_graph = gr
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    if e2e_own is not None:
        e2e_n = steps
        e2e_ms, h2d, d2h = e2e_own
    elif e2e_graph is not None:
        reps = max(1, steps // cap)
        for _ in range(reps):
            e2e_graph.replay()
        e2e_n = reps * cap
    else:
        e2e_run(base, steps)
        e2e_n = steps
    f1.record(stream)
    torch.cuda.synchronize()
    if e2e_own is not None:
        e2e_ms = slowest_rank(e2e_ms, world, dev)
    else:
        e2e_ms = slowest_rank(f0.elapsed_time(f1), world, dev)
    variants = None
    if S.get("variant_runs"):
        variants = {}
        for name, fn in S["variant_runs"]:
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(10):
                fn(i)
            b2.record(stream)
            torch.cuda.synchronize()
            variants[name] = a.elapsed_time(b2) / 10 * 1e3
    if S.get("extra_variants"):
        variants = {}
        for bs in (16, 64, 256):
            for agg, an in ((K.KVSEL_AGG_MAX, "max"), (K.KVSEL_AGG_MEAN, "mean"), (K.KVSEL_AGG_TOPP, "top10%")):
                torch.cuda.synchronize()
                a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for i in range(20):
                    S["run"](i, None, block_size=bs, agg=agg)
                b2.record(stream)
                torch.cuda.synchronize()
                variants[f"bs{bs}_{an}"] = a.elapsed_time(b2) / 20 * 1e3
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(20):
            S["step"](i)
        b2.record(stream)
        torch.cuda.synchronize()
        variants["bs16_max_with_decay_update"] = a.elapsed_time(b2) / 20 * 1e3
        # the other temporal aggregations and the threshold block policies
        for name, kw in (("bs16_max_with_max_update", dict(update=K.KVSEL_UPDATE_MAX)),
                         ("bs16_max_with_window8_update", dict(update=K.KVSEL_UPDATE_WINDOW)),
                         ("bs16_frac_hot", dict(agg=K.KVSEL_AGG_FRAC_HOT, threshold=1e-5)),
                         ("bs16_all_cold", dict(agg=K.KVSEL_AGG_ALL_COLD, threshold=1e-5))):
            upd = "update" in kw
            torch.cuda.synchronize()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(20):
                S["run"](i, S["incs"][i % 4] if upd else None, **kw)
            b2.record(stream)
            torch.cuda.synchronize()
            variants[name] = a.elapsed_time(b2) / 20 * 1e3
    after = S["after"]() if S.get("after") else None
    clocks.stop()
    for w in S["ws"]:
        st = K.read_status(w)
        if st:
            raise RuntimeError(f"device status after the timed region: {st}")
    if rank != 0:
        return
    hbm, peak_kind = peaks()
    kms = kern_ms[dominant]
    if dominant in S.get("ex2", {}):
        # bound by the special-function unit: one exp2 per element, 16 per clock per SM
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                mp = json.load(f)
            tf, clk, tk = float(mp["bf16_tflops"]), float(mp["sm_max_mhz"]), "measured"
        except Exception:
            tf, clk, tk = 1900.0, 2070.0, "fallback"
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mufu = sms * 16 * clk * 1e6 / 1e9  # G exp2 / s
        ach = S["ex2"][dominant] / (kms / 1e3) / 1e9
        tach = S["flops"][dominant] / (kms / 1e3) / 1e12
        roof = {"bound": "alu", "kernel": dominant, "achieved": ach, "peak": mufu, "peak_kind":
                f"derived: {sms} SMs x 16 exp2/clock x {clk:.0f} MHz", "unit": "Gexp2/s", "frac": ach / mufu,
                "traffic": None, "tensor_achieved_tflops": tach, "tensor_frac_of_" + tk + "_bf16": tach / tf,
                "hbm_achieved_gbs": S["bytes"][dominant] / (kms / 1e3) / 1e9}
    elif dominant in S["flops"] and S["flops"][dominant]:
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                tf = float(json.load(f)["bf16_tflops"])
            tk = "measured"
        except Exception:
            tf, tk = 1900.0, "fallback"
        ach = S["flops"][dominant] / (kms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dominant, "achieved": ach, "peak": tf, "peak_kind": tk,
                "unit": "TFLOP/s", "frac": ach / tf, "traffic": None,
                "hbm_achieved_gbs": S["bytes"][dominant] / (kms / 1e3) / 1e9}
    else:
        ach = S["bytes"].get(dominant, 0) / (kms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dominant, "achieved": ach, "peak": hbm, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": ach / hbm, "traffic": None}
    line = {"metric": metric, "value": job_rate(world, steps, ms), "unit": unit, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if args.workload != "block_priority" else "f32",
            "data": "synthetic", "config": dict({"workload": cfg_name}, **S["config"]),
            "kernel_ms": kern_ms, "roofline": roof,
            "e2e": {"value": job_rate(world, e2e_n, e2e_ms), "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_n,
                    "launch": (S["e2e_launch"] if e2e_own is not None else
                               f"CUDA graph of {cap} steps (copies and launches), replayed"
                               if e2e_graph is not None else "eager")},
            "gpu_launches": per_step_launches * steps, "clocks": clocks.summary(tw0, tw1)}
    if eager_ms is not None:
        line["config"]["launch"] = f"CUDA graph of the {steps} timed steps (captured, replayed once untimed, then timed)"
        line["config"]["eager_ms_per_step"] = eager_ms / steps
    if variants:
        line[S.get("variants_key", "variants_us_per_pass")] = variants
    if after:
        line.update(after)
    if args.small:
        line["note"] = "--small profiling case, not the measured workload"
    if not args.no_cpu_baseline:
        res, cores = _oracle_subprocess(args.workload)
        if res:
            line["cpu_baseline"] = {"value": 1.0 / res["seconds_per_unit"], "unit": unit, "cores": cores,
                                    "kind": "oracle", "sample": res["sample"]}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3072)
    ap.add_argument("--warmup", type=int, default=128)
    ap.add_argument("--impl", default="kvsel", choices=["kvsel", "reference"])
    ap.add_argument("--no-probs", action="store_true", help="do not keep the probability tensor")
    ap.add_argument("--no-graph", action="store_true",
                    help="time launch-bound workloads with eager launches instead of a CUDA graph")
    ap.add_argument("--batch", type=int, default=8, help="sequences (8 = the measured workload; "
                    "smaller only for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=64)
    ap.add_argument("--cpu-worker", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--workload", default="decode_70b", choices=list(WORKLOADS),
                    help="decode_70b (the headline) or one of the other hot-path workloads")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--small", action="store_true",
                    help="profiling case (fewer layers / sequences), not the measured workload")
    args = ap.parse_args()
    if args.cpu_worker is not None:
        cpu_worker_main(args.cpu_worker)
        return
    if args.oracle_sample is not None:
        print(json.dumps(ORACLE_SAMPLES[args.oracle_sample]()))
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":  # rank 0 alone; the other ranks exit without work
        if rank == 0:
            if args.workload != "decode_70b":
                other_reference(args, world)
            else:
                reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.workload != "decode_70b":
        other_workload(args, rank, world)
    else:
        cuda_arm(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
