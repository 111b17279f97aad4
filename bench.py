"""Benchmark of the KIVI KV-cache decode path on GB300.

One step = one pass of the whole path over a batch of synthetic input: for
each rotated layer cache, prefill the prompt (quantize + residual), then for
every decode step and layer append one token (flushing the residual when
full) and run decode attention.  The step is replayed as a CUDA graph; the
value is decode-attention KV tokens per second (batch rows x attended tokens,
summed over layers and decode calls) over the whole step time.

Also measured in the same run:
  roofline     decode calls replayed back to back (graph), average duration per
               call, algorithmic bytes per call (codes, steps/zeros, fp16
               residual, q, out) / duration, against the measured HBM copy
               bandwidth;
  e2e          the same step through the Python API with inputs copied from
               pinned host memory each step and outputs copied back;
  cpu_baseline the CPU oracle on a bounded sample of the same workload;
  clocks       nvidia-smi samples taken during the timed region.

--impl reference times the CPU oracle alone (the reference implementation
of the method), on this arm's workload, metric and unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV tokens/s and HBM GB/s vs ~8 TB/s peak (2-bit, Llama-2-7B shape)"
UNIT = "KV tokens/s"

# name -> shape and call sequence (layers = distinct caches rotated in a step)
WORKLOADS = {
    "tiny-b1h1d64": dict(B=1, Hq=1, Hkv=1, D=64, bits=2, G=32, R=32, prompt=256, decode=1, layers=1,
                         outliers="fixed4x20", sink=False, seed=1000),
    "llama2-7b-layer": dict(B=8, Hq=32, Hkv=32, D=128, bits=2, G=32, R=128, prompt=4096, decode=64,
                            layers=4, outliers="range", sink=True, seed=1001),
    "llama2-13b-40layer": dict(B=32, Hq=40, Hkv=40, D=128, bits=2, G=32, R=128, prompt=4096, decode=1,
                               layers=40, outliers="range", sink=True, seed=1002),
    "llama3-8b-gqa": dict(B=64, Hq=32, Hkv=8, D=128, bits=4, G=128, R=128, prompt=8192, decode=20,
                          layers=2, outliers="range", sink=True, seed=1003),
    "llama2-7b-layer-8bit": dict(B=8, Hq=32, Hkv=32, D=128, bits=8, G=32, R=128, prompt=4096, decode=64,
                                 layers=4, outliers="range", sink=True, seed=1005),
    # the 7B layer with the value residual kept as a queue (one value quantized per append)
    "llama2-7b-layer-vqueue": dict(B=8, Hq=32, Hkv=32, D=128, bits=2, G=32, R=128, prompt=4096, decode=64,
                                   layers=4, outliers="range", sink=True, seed=1001, vqueue=True),
    # the 7B layer with ragged prompts (mean 4096) on the paged cache
    "llama2-7b-ragged": dict(B=8, Hq=32, Hkv=32, D=128, bits=2, G=32, R=128, prompt=4096,
                             lengths=[512, 1536, 2560, 3584, 4608, 5632, 6656, 7680], decode=64,
                             layers=4, outliers="range", sink=True, seed=1006, paged=True),
    "long-context": dict(B=2, Hq=32, Hkv=32, D=128, bits=2, G=32, R=128, prompt=131072, decode=512,
                         layers=1, outliers="range", sink=True, seed=1004),
}
DEFAULT = "llama2-7b-layer"
_KERNEL_IDS = {"auto": 0, "cuda-core": 1, "tensor-core": 2}


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _prefill_split(L, G, R):
    over = max(L - R, 0)
    Lq = G * ((over + G - 1) // G)
    return Lq, L - Lq


def _lengths(w):
    """Prompt length of each batch row (sequence)."""
    return list(w.get("lengths") or [w["prompt"]] * w["B"])


def _call_counts(w, L=None):
    """Per decode call: (n_quant, n_resid) after its append, for one sequence
    of prompt L (default: the workload's prompt)."""
    Lq, r = _prefill_split(w["prompt"] if L is None else L, w["G"], w["R"])
    out = []
    for _ in range(w["decode"]):
        if r == w["R"]:
            Lq, r = Lq + w["R"], 0
        r += 1
        out.append((Lq, r))
    return out


def _bytes_last_call(w):
    """Algorithmic bytes of a decode call over the cache as the step leaves it:
    codes + (step, zero) entries of every quantized token, fp16 residual rows,
    the query and the output."""
    half_tok = w["D"] * w["bits"] // 8 + 4 * w["D"] // w["G"]   # codes + (step, zero) of K or of V
    kv = 0
    for L in _lengths(w):
        Lq, r = _call_counts(w, L)[-1]
        # values quantized: with the value queue all but the newest R, else those of the keys
        Lv = max(Lq + r - w["R"], 0) if w.get("vqueue") else Lq
        kv += w["Hkv"] * (Lq * half_tok + Lv * half_tok + r * 2 * w["D"] + (Lq + r - Lv) * 2 * w["D"])
    return kv + 2 * w["B"] * w["Hq"] * w["D"] * 2


def _tokens_last_call(w):
    return sum(sum(_call_counts(w, L)[-1]) for L in _lengths(w))


def _kv_tokens_per_step(w):
    return w["layers"] * sum(Lq + r for L in _lengths(w) for Lq, r in _call_counts(w, L))


# ---- N > 1: each rank runs its own replica of the workload (its own batch) ----
def replica_seed(w, layer, rank):
    """Seed of one rank's layer cache: replicas hold different synthetic batches."""
    return w["seed"] + 7919 * layer + 104729 * rank


def max_over_ranks(ms, device=None):
    """Slowest rank's timed-region milliseconds (all ranks get the same value)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(w, world, steps, t_max_ms):
    """KV tokens/s of all ranks together: every rank processes the same
    per-rank workload (weak scaling), timed by the slowest rank."""
    return world * _kv_tokens_per_step(w) * steps / (t_max_ms / 1e3)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks ----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch
        uid = str(getattr(torch.cuda.get_device_properties(device), "uuid", ""))
        self.dev = uid if uid.startswith("GPU-") else (f"GPU-{uid}" if uid else str(device.index or 0))
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [ln.strip().split(", ") for ln in f if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ oracle (CPU) ----
def oracle_sample(w, n_slots=None, budget_s=15.0, step_seed=0):
    """Run the CPU oracle on whole (batch, kv-head) slots of the workload.

    Each slot: prefill the prompt, then every decode step append + attention
    for the slot's query heads.  Stops after budget_s seconds (at least one
    slot).  Returns (kv_tokens_equivalent, seconds, slots_done).
    One KV token of the metric covers all Hkv heads of a batch row, so a
    single slot contributes its attended tokens / Hkv.
    """
    import numpy as np
    import torch
    from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV
    from oracle.attention import decode_attention
    from oracle.cache import OracleCache, OracleCacheFifo

    outl = FIXED_4_X20 if w["outliers"] == "fixed4x20" else RANGE_2_6_X10_50
    syn = SynthKV(1, w["Hq"] // w["Hkv"], 1, w["D"], seed=w["seed"] + step_seed, outliers=outl,
                  sink=w["sink"], device="cpu")
    lengths = _lengths(w)
    K, V = syn.prompt(max(lengths))
    Kn, Vn = K.numpy(), V.numpy()
    steps = [tuple(t.numpy() for t in syn.step(s)) for s in range(w["decode"])]
    t0 = time.perf_counter()
    done, tokens = 0, 0
    while True:
        oc = (OracleCacheFifo if w.get("vqueue") else OracleCache)(1, 1, w["D"], w["bits"], w["G"], w["R"])
        L = lengths[(done + step_seed) % len(lengths)]     # ragged workloads: the rows' lengths in turn
        oc.prefill(np.ascontiguousarray(Kn[:, :, :L]), np.ascontiguousarray(Vn[:, :, :L]))
        for (q, k, v) in steps:
            oc.append(k, v)
            decode_attention(q, oc.keys_hat(), oc.values_hat())
            tokens += oc.n_quant + oc.n_resid
        done += 1
        el = time.perf_counter() - t0
        if (n_slots is not None and done >= n_slots) or (n_slots is None and el >= budget_s):
            break
    return tokens / w["Hkv"], time.perf_counter() - t0, done


def _oracle_worker(job):
    """One process of the all-cores oracle run: its own slots, its own budget."""
    name, budget_s, idx = job
    t0 = time.time()
    tok, secs, done = oracle_sample(WORKLOADS[name], budget_s=budget_s, step_seed=idx)
    return tok, done, t0 + 0.0, time.time()


def host_cores():
    """Cores of this host: os.cpu_count() and the ones this process may run on (nproc)."""
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count() or 1
    return {"cpu_count": os.cpu_count(), "nproc": usable}


def oracle_all_cores(name, workers, budget_s):
    """The oracle on every usable core at once: one process per core (spawned,
    single-threaded numpy), each on its own (batch, kv-head) slots for about
    budget_s seconds of work.  KV tokens of all processes / the wall time from
    the first start to the last finish."""
    import multiprocessing as mp
    env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            res = pool.map(_oracle_worker, [(name, budget_s, 1 + i) for i in range(workers)])
    finally:
        for k, v in env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    tok = sum(r[0] for r in res)
    wall = max(r[3] for r in res) - min(r[2] for r in res)
    return tok / wall, wall, sum(r[1] for r in res)


def sink_mass_sample(w, n_slots=8):
    """Attention weight of the sink token (token 0) at the first decode step,
    from the oracle, over n_slots (batch, kv-head) slots of the workload's
    generator: (median, all).  None for workloads without a sink."""
    if not w["sink"]:
        return None
    import math
    import numpy as np
    from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV
    from oracle.attention import decode_attention
    from oracle.cache import OracleCache
    outl = FIXED_4_X20 if w["outliers"] == "fixed4x20" else RANGE_2_6_X10_50
    L = min(_lengths(w))
    masses = []
    for j in range(n_slots):
        syn = SynthKV(1, 1, 1, w["D"], seed=w["seed"] * 1000 + j, outliers=outl, sink=True, device="cpu")
        K, V = syn.prompt(L)
        oc = OracleCache(1, 1, w["D"], w["bits"], w["G"], w["R"])
        oc.prefill(K.numpy(), V.numpy())
        q, k, v = (t.numpy() for t in syn.step(0))
        oc.append(k, v)
        Kh = oc.keys_hat()
        _, lse = decode_attention(q, Kh, oc.values_hat())
        l0 = (Kh[0, 0, 0] * q[0, 0].astype(np.float64)).sum() / math.sqrt(w["D"])
        masses.append(float(np.exp(l0 - lse[0, 0])))
    return float(np.median(masses)), masses


def run_reference(args, w):
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(w, n_slots=1)
    tok, secs = 0.0, 0.0
    for s in range(args.steps):
        t, sec, _ = oracle_sample(w, n_slots=1, step_seed=s)
        tok += t
        secs += sec
    value = tok / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w, args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "threads": 1, "host_cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"per step one (batch, kv-head) slot of {args.workload}: prefill "
                                   f"{w['prompt']} + {w['decode']} x (append + attention); "
                                   f"KV tokens counted per slot / {w['Hkv']} heads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, name):
    c = {"workload": name, "batch": w["B"], "q_heads": w["Hq"], "kv_heads": w["Hkv"],
         "head_dim": w["D"], "bits": w["bits"], "group": w["G"], "residual": w["R"],
         "prompt": w["prompt"], "decode_steps": w["decode"], "layers_rotated": w["layers"]}
    if w.get("lengths"):
        c["prompt_lengths"] = list(w["lengths"])
    if w.get("paged"):
        c["cache"] = "paged (page pool + block tables)"
    if w.get("vqueue"):
        c["value_residual"] = "queue (one value token quantized per append)"
    return c


# --------------------------------------------------------------- GPU arm ----
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    from bit_kivi_kv_gb300 import build as _b
    _b.build()
    from bit_kivi_kv_gb300 import kivi as K
    from bit_kivi_kv_gb300.kivi import KiviCache
    from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV

    outl = FIXED_4_X20 if w["outliers"] == "fixed4x20" else RANGE_2_6_X10_50
    NL, S = w["layers"], w["decode"]
    paged = bool(w.get("paged") or args.paged)
    eng = (_PagedEngine if paged else _DenseEngine)(args, w, dev, rank, outl, SynthKV, torch)
    step, decode_only = eng.step, eng.decode_only

    # eager warm-up (also the first device query), then capture
    step()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    g_step, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g_step, stream=stream):
            step()
        decode_only()
        torch.cuda.synchronize()
        with torch.cuda.graph(g_dec, stream=stream):
            for _ in range(8):
                decode_only()
    launches_per_step = None

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        g_step.replay()
    barrier()
    n0 = K.kivi_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                g_step.replay()
        ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1)
    # kernels launched per step = the launches the captured step issued
    launches_per_step = _launches_in(step, K, stream, torch)
    gpu_launches = launches_per_step * args.steps
    clocks = clk.summary()
    t_max = max_over_ranks(ms, dev) if world > 1 else ms
    value = whole_job_value(w, world, args.steps, t_max)

    # ---- roofline: decode calls back to back (graph), rotated across layers ----
    reps = max(4, int(200 / max(NL * 8, 1)))
    for _ in range(3):
        g_dec.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g_dec.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    calls = reps * 8 * NL
    dec_ms = e0.elapsed_time(e1) / calls
    bytes_call = _bytes_last_call(w)
    achieved = bytes_call / (dec_ms / 1e3) / 1e9
    peak, peak_kind = _peaks()
    traffic = _profile_traffic(args.workload + ("-paged" if paged and not w.get("paged") else ""))

    # ---- the other workloads' decode calls, measured the same way (1 GPU only) ----
    configs = None
    if world == 1 and args.configs and args.workload in FIVE:
        configs = {args.workload: {"us": dec_ms * 1e3, "bytes": bytes_call, "gbs": achieved,
                                   "frac": achieved / peak, "context": "after the step's decode calls",
                                   "note": "the headline: same numbers as decode_call / roofline"}}
        for name in FIVE:
            if name != args.workload:
                configs[name] = decode_call_config(name, dev, torch, peak)

    # ---- e2e through the Python API from pinned host memory ----
    barrier()
    e2e = eng.e2e(max(3, min(args.steps, 10)))
    if world > 1:
        # whole job: every rank runs its replica's step; the slowest rank sets the time
        e2e_ms = max_over_ranks(e2e["ms_per_step"], dev)
        e2e["ms_per_step"] = e2e_ms
        e2e["value"] = world * _kv_tokens_per_step(w) / (e2e_ms / 1e3)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; key outlier channels, attention sink)",
        "config": dict(_config(w, args.workload), parallelism=f"replicas x{world}",
                       step_calls=("kivi_paged_add + kivi_paged_append_decode" if paged else
                                   "kivi_append + kivi_decode_attn" if args.separate_append else
                                   "kivi_append_decode"),
                       l2="inputs larger than L2: each step rotates layer caches "
                          f"({NL} x ~{bytes_call / 1e6:.0f} MB read per decode round)"),
        "decode_call": {"us": dec_ms * 1e3, "bytes": bytes_call, "gbs": achieved,
                        "kv_tokens_per_s": _tokens_last_call(w) / (dec_ms / 1e3),
                        "steps_per_s": 1e3 / dec_ms},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "kernel": "decode attention call: " + (
                         "decode_split_kernel + combine_kernel" if args.decode_kernel == "cuda-core" and not paged
                         else "decode_mma_kernel (paged) + finish_paged_kernel (tensor cores)" if paged
                         else "decode_mma_kernel + finish_kernel (tensor cores)")},
        "e2e": e2e, "clocks": clocks, "gpu_launches": gpu_launches,
    }
    if configs is not None:
        result["configs"] = {"peak_gbs": peak, "how": "decode call: CUDA-graph replay over rotated caches, "
                                                      "CUDA events; frac of the measured copy bandwidth",
                             **configs}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sm = sink_mass_sample(w)
        if sm is not None:
            result["sink_mass"] = {"median": sm[0], "slots": len(sm[1]),
                                   "how": "oracle attention weight of token 0 at the first decode step, "
                                          "one head per slot, prompt of the workload's shortest length"}
        tok, secs, done = oracle_sample(w, budget_s=args.cpu_budget)
        hc = host_cores()
        result["cpu_baseline"] = {
            "value": tok / secs, "unit": UNIT, "cores": 1, "threads": 1, "host_cores": hc, "kind": "oracle",
            "sample": f"{done} (batch, kv-head) slot(s) of {args.workload}: prefill {w['prompt']} + "
                      f"{w['decode']} x (append + fp64 attention), {secs:.1f} s on one core; KV tokens per slot "
                      f"counted / {w['Hkv']} heads"}
        if args.cpu_all_cores and hc["nproc"] > 1:
            v_all, wall, n_all = oracle_all_cores(args.workload, hc["nproc"], args.cpu_budget / 2)
            result["cpu_baseline"]["all_cores"] = {
                "value": v_all, "unit": UNIT, "cores": hc["nproc"], "slots": n_all,
                "how": f"{hc['nproc']} spawned single-threaded oracle processes, one per usable core, each on "
                       f"its own slots for ~{args.cpu_budget / 2:.0f} s; all their KV tokens / {wall:.1f} s wall"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# the method's five workloads (the headline is measured by run_ours itself)
FIVE = ("tiny-b1h1d64", "llama2-7b-layer", "llama2-13b-40layer", "llama3-8b-gqa", "long-context")


def decode_call_config(name, dev, torch, peak):
    """One workload's decode call, measured as the headline's is: caches built once
    (prefill of the prompt, then one append, which flushes where the residual is
    full), then decode calls replayed back to back from a CUDA graph over rotated
    caches (each call of the large workloads reads more than L2 holds), timed with
    CUDA events.  Returns {us, bytes, gbs, frac, kv_tokens_per_s, calls}."""
    from bit_kivi_kv_gb300.kivi import KiviCache
    from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV
    w = dict(WORKLOADS[name], decode=1)
    outl = FIXED_4_X20 if w["outliers"] == "fixed4x20" else RANGE_2_6_X10_50
    nl = {"tiny-b1h1d64": 4, "long-context": 1}.get(name, 2)
    caches, qs, outs = [], [], []
    for li in range(nl):
        syn = SynthKV(w["B"], w["Hq"], w["Hkv"], w["D"], seed=replica_seed(w, li, 0), outliers=outl,
                      sink=w["sink"], device=dev)
        Kp, Vp = syn.prompt(w["prompt"])
        q, k, v = syn.step(0)
        c = KiviCache(w["B"], w["Hq"], w["Hkv"], w["D"], w["bits"], w["G"], w["R"], w["prompt"] + 1, device=dev)
        c.prefill(Kp, Vp)
        c.append(k, v)
        torch.cuda.synchronize()
        del Kp, Vp
        caches.append(c)
        qs.append(q)
        outs.append(torch.empty_like(q))
    rounds = max(1, 16 // nl)
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c, q, o in zip(caches, qs, outs):
            c.decode_attn(q, out=o)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(rounds):
                for c, q, o in zip(caches, qs, outs):
                    c.decode_attn(q, out=o)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = 40 if name == "tiny-b1h1d64" else 8
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    calls = reps * rounds * nl
    us = e0.elapsed_time(e1) * 1e3 / calls
    nbytes = _bytes_last_call(w)
    gbs = nbytes / (us * 1e-6) / 1e9
    out = {"us": us, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak,
           "kv_tokens_per_s": _tokens_last_call(w) / (us * 1e-6), "calls": calls,
           "caches_rotated": nl, "context": w["prompt"] + 1}
    if name == "tiny-b1h1d64":
        out["note"] = "latency-bound (12.8 KB per call): no roofline claim"
    del caches, qs, outs, g
    torch.cuda.empty_cache()
    return out


def _launches_in(step, K, stream, torch):
    """Kernel launches one eager step issues (the captured graph holds the same kernels)."""
    n0 = K.kivi_launch_count()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    return K.kivi_launch_count() - n0


def _decode_source_sha1():
    import hashlib
    h = hashlib.sha1()
    for f in ("kivi_decode.cu", "kivi_common.cuh", "kivi_decode_mma.cuh", "kivi_decode_mma_launch.cuh",
              "kivi_decode_mma_d128.cu", "kivi_decode_mma_d64.cu", "kivi_decode_mma_d128p.cu",
              "kivi_decode_mma_d64p.cu"):
        with open(os.path.join(ROOT, "bit_kivi_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _profile_traffic(name):
    """DRAM bytes per decode call from the committed ncu summary, if it was taken
    on the decode kernel as it is now (same source hash); else None."""
    p = os.path.join(ROOT, "profiles", f"decode_{name}.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("decode_source_sha1") == _decode_source_sha1():
            return d.get("traffic_bytes_per_call")
    return None


def run_profile(args, w):
    """Small eager run for ncu: the bench's step on at most 2 layers (2 x decode
    calls of decode kernels: appends + decodes), then profile_calls rounds of
    decode-only calls at the state the step leaves (no graphs, e2e or oracle)."""
    import torch
    from bit_kivi_kv_gb300 import build as _b
    _b.build()
    from bit_kivi_kv_gb300.synth import FIXED_4_X20, RANGE_2_6_X10_50, SynthKV
    dev = torch.device("cuda", 0)
    outl = FIXED_4_X20 if w["outliers"] == "fixed4x20" else RANGE_2_6_X10_50
    w2 = dict(w, layers=min(w["layers"], 2))
    paged = bool(w.get("paged") or args.paged)
    eng = (_PagedEngine if paged else _DenseEngine)(args, w2, dev, 0, outl, SynthKV, torch)
    eng.step()
    for _ in range(args.profile_calls):
        eng.decode_only()
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": args.workload, "paged": paged, "decode_source_sha1": _decode_source_sha1()}))


class _DenseEngine:
    """The workload on dense caches (one KiviCache per layer, all rows of equal length)."""

    def __init__(self, args, w, dev, rank, outl, SynthKV, torch):
        from bit_kivi_kv_gb300.kivi import KiviCache
        self.args, self.w, self.dev, self.torch = args, w, dev, torch
        NL, S = w["layers"], w["decode"]
        self.caches, self.prompts, self.steps = [], [], []
        for li in range(NL):
            syn = SynthKV(w["B"], w["Hq"], w["Hkv"], w["D"], seed=replica_seed(w, li, rank),
                          outliers=outl, sink=w["sink"], device=dev)
            self.prompts.append(syn.prompt(w["prompt"]))
            self.steps.append([syn.step(s) for s in range(S)])
            c = KiviCache(w["B"], w["Hq"], w["Hkv"], w["D"], w["bits"], w["G"], w["R"], w["prompt"] + S, device=dev)
            c.set_decode_kernel(_KERNEL_IDS[args.decode_kernel])
            if w.get("vqueue"):
                c.set_value_residual(1)
            self.caches.append(c)
        self.outs = [torch.empty(w["B"], w["Hq"], w["D"], dtype=torch.float16, device=dev) for _ in range(NL)]

    def step(self):
        w, sep = self.w, self.args.separate_append
        for li, c in enumerate(self.caches):
            c.reset()
            c.prefill(*self.prompts[li])
        for s in range(w["decode"]):
            for li, c in enumerate(self.caches):
                q, k, v = self.steps[li][s]
                if sep:
                    c.append(k, v)
                    c.decode_attn(q, out=self.outs[li])
                else:
                    c.append_decode(k, v, q, out=self.outs[li])

    def decode_only(self):
        for li, c in enumerate(self.caches):
            c.decode_attn(self.steps[li][-1][0], out=self.outs[li])

    # ---- end to end: the step's inputs from pinned host memory, outputs back ----
    def host_inputs(self):
        torch = self.torch
        pin = lambda t: t.cpu().pin_memory()
        ins = []
        for K_, V_ in self.prompts:
            ins += [pin(K_), pin(V_)]
        for layer in self.steps:    # the step's 64 (q, k, v), stacked per layer
            ins += [pin(torch.stack([st[j] for st in layer])) for j in range(3)]
        return ins

    def run_from(self, bufs, outs):
        NL, sep = len(self.caches), self.args.separate_append
        for li, c in enumerate(self.caches):
            c.reset()
            c.prefill(bufs[2 * li], bufs[2 * li + 1])
        for s in range(self.w["decode"]):
            for li, c in enumerate(self.caches):
                q, k, v = (bufs[2 * NL + 3 * li + j][s] for j in range(3))
                if sep:
                    c.append(k, v)
                    c.decode_attn(q, out=outs[li][s])
                else:
                    c.append_decode(k, v, q, out=outs[li][s])

    def new_outputs(self):
        w = self.w
        return [self.torch.empty(w["decode"], w["B"], w["Hq"], w["D"], dtype=self.torch.float16, device=self.dev)
                for _ in self.caches]

    def e2e(self, n):
        return _pipelined_e2e(self, n, self.w, self.dev, self.torch)


class _PagedEngine:
    """The workload on paged caches (one KiviPagedCache per layer): every step
    releases the rows' sequences and adds them again with their prompts (the
    allocator hands out the pages), then appends + decodes all of them."""

    def __init__(self, args, w, dev, rank, outl, SynthKV, torch):
        from bit_kivi_kv_gb300.kivi import KiviPagedCache
        self.args, self.w, self.dev, self.torch = args, w, dev, torch
        NL, S = w["layers"], w["decode"]
        lengths = _lengths(w)
        blocks = [_call_counts(w, L)[-1][0] // w["G"] for L in lengths]
        self.caches, self.prompts, self.steps, self.seqs = [], [], [], []
        for li in range(NL):
            # the dense workload's generator: row b's prompt is the first L_b tokens
            # of its row, its queries carry the row's attention-sink direction
            syn = SynthKV(len(lengths), w["Hq"], w["Hkv"], w["D"], seed=replica_seed(w, li, rank),
                          outliers=outl, sink=w["sink"], device=dev)
            K_, V_ = syn.prompt(max(lengths))
            self.prompts.append([(K_[b, :, :L].contiguous(), V_[b, :, :L].contiguous())
                                 for b, L in enumerate(lengths)])
            del K_, V_
            self.steps.append([syn.step(s) for s in range(S)])
            self.caches.append(KiviPagedCache(len(lengths), w["Hq"], w["Hkv"], w["D"], w["bits"], w["G"], w["R"],
                                              max(blocks) + 1, sum(blocks) + len(lengths), device=dev))
            self.seqs.append([])
        self.outs = [torch.empty(len(lengths), w["Hq"], w["D"], dtype=torch.float16, device=dev) for _ in range(NL)]

    def _readd(self, li, prompts):
        c = self.caches[li]
        for s in self.seqs[li]:
            c.release(s)
        self.seqs[li] = [c.add(K_, V_) for K_, V_ in prompts]

    def step(self):
        for li in range(len(self.caches)):
            self._readd(li, self.prompts[li])
        for s in range(self.w["decode"]):
            for li, c in enumerate(self.caches):
                q, k, v = self.steps[li][s]
                c.append_decode(self.seqs[li], k, v, q, out=self.outs[li])

    def decode_only(self):
        for li, c in enumerate(self.caches):
            c.append_decode(self.seqs[li], None, None, self.steps[li][-1][0], out=self.outs[li])

    def host_inputs(self):
        torch = self.torch
        pin = lambda t: t.cpu().pin_memory()
        ins = []
        for rows in self.prompts:
            for K_, V_ in rows:
                ins += [pin(K_), pin(V_)]
        for layer in self.steps:
            ins += [pin(torch.stack([st[j] for st in layer])) for j in range(3)]
        return ins

    def run_from(self, bufs, outs):
        NL, nb = len(self.caches), len(self.prompts[0])
        for li in range(NL):
            self._readd(li, [(bufs[2 * (li * nb + b)], bufs[2 * (li * nb + b) + 1]) for b in range(nb)])
        base = 2 * NL * nb
        for s in range(self.w["decode"]):
            for li, c in enumerate(self.caches):
                q, k, v = (bufs[base + 3 * li + j][s] for j in range(3))
                c.append_decode(self.seqs[li], k, v, q, out=outs[li][s])

    def new_outputs(self):
        w, nb = self.w, len(self.prompts[0])
        return [self.torch.empty(w["decode"], nb, w["Hq"], w["D"], dtype=self.torch.float16, device=self.dev)
                for _ in self.caches]

    def e2e(self, n):
        return _pipelined_e2e(self, n, self.w, self.dev, self.torch)


def _pipelined_e2e(eng, n, w, dev, torch):
    """The step end to end through the Python binding: every step uploads all of
    its inputs (prompts and the decode steps' q, k, v) from pinned host memory
    and reads all of its outputs back.  A copy stream uploads step i+1's inputs
    into a second buffer set while step i computes (copies overlapped with
    compute); every copy of every step is inside the timed region."""
    h_in = eng.host_inputs()
    bufs = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(2)]
    d_out = eng.new_outputs()
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in d_out]
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    free = [torch.cuda.Event(), torch.cuda.Event()]

    def upload(b):
        with torch.cuda.stream(cp):
            cp.wait_event(free[b])          # the step that read buffer b has finished with it
            for d, h in zip(bufs[b], h_in):
                d.copy_(h, non_blocking=True)
            ready[b].record(cp)

    def compute(b):
        comp.wait_event(ready[b])
        eng.run_from(bufs[b], d_out)
        free[b].record(comp)
        for h, d in zip(h_out, d_out):
            h.copy_(d, non_blocking=True)

    for b in (0, 1):
        free[b].record(comp)
    upload(0)                               # untimed warm-up step
    compute(0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    upload(0)
    for i in range(n):
        if i + 1 < n:
            upload((i + 1) % 2)
        compute(i % 2)
    torch.cuda.synchronize()
    secs = (time.perf_counter() - t0) / n
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    return {"value": _kv_tokens_per_step(w) / secs, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": secs * 1e3, "steps": n,
            "how": "eager calls through bit_kivi_kv_gb300.kivi; each step's inputs uploaded from pinned host "
                   "memory on a copy stream (step i+1's during step i) and its outputs read back; host-timed"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-all-cores", type=int, default=1,
                    help="also time the oracle on every usable core (1, default) or not (0)")
    ap.add_argument("--configs", type=int, default=1,
                    help="also measure the decode call of the other workloads of the method's five (1, default)")
    ap.add_argument("--profile", action="store_true", help="small eager run for ncu captures")
    ap.add_argument("--separate-append", action="store_true",
                    help="decode steps as kivi_append + kivi_decode_attn instead of kivi_append_decode")
    ap.add_argument("--decode-kernel", choices=["auto", "cuda-core", "tensor-core"], default="auto")
    ap.add_argument("--profile-calls", type=int, default=4)
    ap.add_argument("--paged", action="store_true",
                    help="run the workload on the paged cache (ragged workloads always are)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.profile:
        run_profile(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
