"""Benchmark of the paged decode step on GB300.

A step is one pass of the whole hot path over one batch: copy-on-write block
copies (when the step has any), the scatter of the new tokens into their
slots, and paged decode attention (single pass, split-context partitions plus
log-sum-exp reduce, or the shared-prefix kernel plus its merge).

Default line: the largest workload that fits one GPU, the long-context decode
(batch 16, 64 query / 8 kv heads, head_dim 128, block 16, contexts of 16K-32K
tokens whose blocks are scattered over a ~60 GB pool, 512-token partitions).
At one GPU the same line carries ``per_config``: every workload -- Llama-7B
fp16, Llama-13B continuous batching, parallel sampling with shared prefixes,
the long-context decode at block sizes 8 / 16 / 32, and cached system prompts
-- each over its own step count, with the same figures as the headline.

Figures (rank 0 prints ONE JSON line):
  value      algorithmic bytes of the steps / device time of the steps, every
             input resident in HBM; L2 is flushed (256 MiB read) before every
             step, outside the timed events.
  roofline   the decode's own algorithmic bytes per launch / its mean
             event-timed duration, against the measured HBM copy bandwidth.
  e2e        the same metric with the step's inputs copied from pinned host
             memory and the output read back inside the device-timed region.
  host_e2e   a serving loop's steps timed by the host's wall clock: block-pool
             bookkeeping, the shared-prefix planner, packing, copies, library
             calls and a stream synchronise.
  cpu_baseline  the CPU oracle on a bounded sample of the same steps.

--impl reference times the oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import CONFIGS, PagedDecodeWorkload, get  # noqa: E402
from workloads.runner import DeviceState, algorithmic_bytes  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak); seq-steps/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
SEED_BASE = 311 * 100


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--op", default="decode", choices=["decode", "swap_blocks", "host_step"],
                    help="swap_blocks: time the block swap of a preempted tenth of the batch; "
                         "host_step: time a step's host bookkeeping (no GPU)")
    ap.add_argument("--config", default=HEADLINE[0])
    ap.add_argument("--block-size", type=int, default=0)
    ap.add_argument("--num-seqs", type=int, default=0, help="override the batch (profiling cases)")
    ap.add_argument("--pool-gb", type=float, default=0.0,
                    help="cap the pool of byte-sized presets (profiling cases)")
    ap.add_argument("--partition-size", type=int, default=-1, help="-1: the preset's choice")
    ap.add_argument("--engine", default="auto", choices=["auto", "cuda_core", "tensor_core", "tcgen05"])
    ap.add_argument("--no-shared", action="store_true",
                    help="shared-prefix workloads: use the per-sequence entry point")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-host-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="only the headline workload (per_config is on by default at one GPU)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--per-config-cpu-seconds", type=float, default=4.0)
    ap.add_argument("--identity-tables", action="store_true",
                    help="place every sequence's blocks contiguously (gather-overhead comparison)")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def local_device():
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(lr)
    return torch.device("cuda", lr)


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def run_native(args):
    dist, rank, world = dist_setup()
    dev = local_device()
    head = measure(args, args.config, args.block_size, args.steps, args.warmup, dist, rank, world,
                   dev, cpu_seconds=args.cpu_seconds)
    per_config = None
    if world == 1 and not args.no_per_config and args.op == "decode":
        per_config = {}
        for name, bs in PER_CONFIG:
            key = name if name != "long_context_bf16" else f"{name}/bs{bs}"
            if (name, bs or get(name).block_size) == (head["config"]["workload"],
                                                      head["config"]["block_size"]):
                per_config[key] = _compact(head)
                continue
            cfg = get(name)
            r = measure(args, name, bs, cfg.steps - PER_CONFIG_WARMUP if cfg.steps > 10 else cfg.steps,
                        PER_CONFIG_WARMUP, None, 0, 1, dev, cpu_seconds=args.per_config_cpu_seconds,
                        engine="auto", shared_default=True)
            per_config[key] = _compact(r)
    if rank == 0:
        line = {"metric": METRIC, **{k: head[k] for k in (
            "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "seq_steps_per_s", "step_ms",
            "decode_ms", "unflushed", "pct_of_peak", "roofline", "clocks", "gpu_launches", "e2e",
            "host_e2e", "cpu_baseline", "kv_memory")}}
        if per_config is not None:
            line["per_config"] = per_config
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


# The headline line: the largest configuration that fits one GPU -- the
# long-context decode (batch 16, 64 q / 8 kv heads, 16K-32K tokens) over a
# ~60 GB pool, split-context partitions and their merge.  per_config: every
# workload of the survey at one GPU, each over its own step count.
HEADLINE = ("long_context_bf16", 16)
PER_CONFIG = [("llama7b_f16", 0), ("llama13b_cb_bf16", 0), ("shared_prefix_bf16", 0),
              ("long_context_bf16", 8), ("long_context_bf16", 16), ("long_context_bf16", 32),
              ("system_prompt_bf16", 0)]
PER_CONFIG_WARMUP = 3


def _compact(r):
    """A per_config entry: the measured figures of one workload."""
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "seq_steps_per_s", "decode_ms",
            "roofline", "clocks", "gpu_launches", "e2e", "host_e2e", "cpu_baseline", "kv_memory")
    out = {k: r[k] for k in keep}
    c = r["config"]
    out["config"] = {k: c[k] for k in ("workload", "kv_dtype", "num_seqs", "num_heads",
                                       "num_kv_heads", "block_size", "partition_size",
                                       "decode_launches_per_step", "engine", "pool_gb", "path")}
    return out


def measure(args, name, block_size, steps, warmup, dist, rank, world, dev, cpu_seconds,
            engine=None, shared_default=None):
    """One workload: device-timed steps, the unflushed repeat, e2e through
    the C ABI with host buffers, the wall-clock host_e2e serving loop, the
    CPU oracle on a bounded sample, and memory accounting."""
    import paged_kv_cache_311_gb300 as pkv
    cfg = get(name)
    if block_size:
        cfg = cfg.with_(block_size=block_size)
    engine = args.engine if engine is None else engine
    no_shared = args.no_shared if shared_default is None else not shared_default
    seed = SEED_BASE + CONFIGS.index(get(name)) + 1000 * rank
    total = warmup + steps
    w = PagedDecodeWorkload(cfg, seed, total_steps=max(total, cfg.steps),
                            contiguous=args.identity_tables and name == args.config,
                            num_seqs=(args.num_seqs or None) if name == args.config else None,
                            pool_blocks=_pool_blocks(cfg, dev, args.pool_gb if name == args.config
                                                     else 0.0))
    P = cfg.partition_size if (args.partition_size < 0 or name != args.config) else args.partition_size
    out_dtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[cfg.dtype]
    state = DeviceState(cfg, w, seed, device=dev, out_dtype=out_dtype)
    host_inputs = [w.next_step() for _ in range(total)]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and cpu_seconds > 0:
        cpu = cpu_baseline(cfg, state, host_inputs, cpu_seconds, seed)

    shared = cfg.kind in ("shared_prefix", "system_prompt") and not no_shared
    if shared and (args.partition_size < 0 or name != args.config):
        P = 0   # the shared-prefix planner's own default partition
    pkv.set_decode_engine(engine)   # before planning: the automatic plan follows the kernel
    steps_dev = [state.to_device(inp, shared=shared, partition_size=P) for inp in host_inputs]
    for s in steps_dev:
        state.ensure_workspace(s.max_context_len, P, s.plan)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    out_bytes = torch.tensor([], dtype=out_dtype).element_size()

    # warm-up
    for s in steps_dev[:warmup]:
        state.run_step(s, partition_size=P)
    torch.cuda.synchronize()
    state.status.zero_()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    launches = 0
    decode_launches = []
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if rank == 0 else None
    gc.collect()      # no collector pass inside the timed steps
    gc.disable()
    torch.cuda.nvtx.range_push("timed_steps")
    for i, s in enumerate(steps_dev[warmup:]):
        _flush_l2(flush)
        _preroll()
        e0, e1, e2 = ev[i]
        e0.record(stream)
        if s.cow_pairs is not None:
            pkv.copy_blocks([state.k_cache], [state.v_cache], s.cow_pairs,
                            device_status=state.status)
            launches += 1
        pkv.reshape_and_cache(s.key, s.value, state.k_cache, state.v_cache, s.slot_mapping,
                              device_status=state.status)
        launches += 1
        e1.record(stream)
        _decode(pkv, state, s, s.q, s.block_tables, s.context_lens, s.plan_device, P)
        n = pkv.last_decode_launches()
        decode_launches.append(n)
        engine_used = pkv.last_decode_engine()
        launches += n
        e2.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    gc.enable()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if state.status.item() != 0:
        raise RuntimeError(f"{cfg.name}: device status {state.status.item()} during the timed steps")

    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    tot_ms = sum(step_ms)
    bytes_step, bytes_dec, seqs = 0, 0, 0
    dec_bytes = []
    for s, n in zip(steps_dev[warmup:], decode_launches):
        ab = _step_bytes(cfg, s.host, w.num_seqs, out_bytes, s.plan, P, n)
        bytes_step += ab["total"]
        bytes_dec += ab["attention"]
        dec_bytes.append(ab["attention"])
        seqs += w.num_seqs
    plan_s = sum(s.plan_seconds for s in steps_dev[warmup:])
    t_max = max_over_ranks(dist, tot_ms / 1e3)
    bytes_all = sum_over_ranks(dist, bytes_step)
    seqs_all = sum_over_ranks(dist, seqs)
    value = bytes_all / t_max / 1e9
    dec_mean_ms = sum(dec_ms) / len(dec_ms)
    achieved = bytes_dec / len(dec_ms) / (dec_mean_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    main_kernel = (("pa_cascade_tc05_kernel" if engine_used == "tcgen05" else "pa_cascade_kernel")
                   if shared else "pa_decode_kernel")

    unflushed = _unflushed_decode(pkv, state, steps_dev[-1], P, dec_bytes[-1], peak)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(state, steps_dev[warmup:], host_inputs[warmup:], P, flush, bytes_step)
    # memory accounting of the paged cache at the first timed step
    first = host_inputs[warmup]
    use = pkv.kv_cache_usage(first.block_tables, first.context_lens, cfg.block_size, w.num_blocks)
    kv_memory = {"block_size": cfg.block_size, "tokens": use.tokens, "blocks": use.blocks,
                 "paged_waste": round(use.paged_waste, 4),
                 "reserve_longest_waste": round(use.reserved_waste(int(first.context_lens.max())), 4)}
    host = None
    if not args.no_host_e2e and world == 1:
        # last: it writes its own prefill into the same cache
        host = run_host_e2e(cfg, w, state, shared, P, engine, flush, seed,
                            steps=min(steps, HOST_E2E_STEPS), warmup=min(warmup, 3))
    pkv.set_decode_engine("auto")

    pool_gb = round(2 * w.num_blocks * cfg.block_bytes / 1e9, 3)
    res = {
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": round(t_max * 1e3 / steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "kv_dtype": cfg.dtype, "num_seqs": w.num_seqs,
                   "num_heads": cfg.num_heads, "num_kv_heads": cfg.num_kv_heads,
                   "head_dim": cfg.head_dim, "block_size": cfg.block_size,
                   "partition_size": P, "decode_launches_per_step": decode_launches[0],
                   "engine": engine_used,
                   "path": "shared prefix" if shared else (
                       "split-context + merge" if decode_launches[0] == 2 else "single pass"),
                   "pool_gb": pool_gb,
                   "parallelism": f"replicas x{world} (sequences sharded, no collective)",
                   "l2": "flushed (256 MiB read) before every timed step, outside the events",
                   "block_placement": "contiguous" if args.identity_tables and name == args.config
                   else "random",
                   "timed_steps": f"steps {warmup}..{warmup + steps - 1} of the workload"},
        # shared paths: the host planner's time for each step counts too
        "seq_steps_per_s": round(seqs_all / (t_max + max_over_ranks(dist, plan_s)), 1),
        "step_ms": _spread(step_ms),
        "decode_ms": _spread(dec_ms),
        "unflushed": unflushed,
        "pct_of_peak": round(100 * value / peak, 2),
        "roofline": {"bound": "hbm",
                     "kernel": main_kernel + ("+pa_cascade_merge_kernel" if shared else
                                              "+pa_merge_kernel" if decode_launches[0] == 2 else ""),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": traffic_for(cfg, main_kernel, bytes_dec / len(dec_ms)),
                     "algorithmic_bytes_per_launch": int(bytes_dec / len(dec_ms)),
                     "mean_launch_ms": round(dec_mean_ms, 5)},
        "clocks": clk,
        "gpu_launches": launches,
        "e2e": e2e,
        "host_e2e": host,
        "cpu_baseline": cpu,
        "kv_memory": kv_memory,
    }
    if shared:
        res["config"]["planner_ms_per_step"] = round(plan_s * 1e3 / steps, 4)
    del state, steps_dev, flush
    gc.collect()
    torch.cuda.empty_cache()
    return res


def _step_bytes(cfg, inp, num_seqs, out_bytes, plan, P, launches):
    """Algorithmic bytes of one step (attention, scatter, copies)."""
    if plan is not None:
        expected = plan.host[8:8 + num_seqs]
        return algorithmic_bytes(cfg, inp, num_seqs, out_bytes=out_bytes, partials=expected)
    return algorithmic_bytes(cfg, inp, num_seqs, split_partition=_split_partition(P, 0, launches),
                             out_bytes=out_bytes)


def _decode(pkv, state, s, q, bt, cl, plan_dev, P):
    """The step's attention call: the shared-prefix entry point when the step
    carries a plan, the per-sequence one otherwise."""
    cfg = state.cfg
    if s.plan is not None:
        pkv.paged_attention_decode_shared(state.out, q, state.k_cache, state.v_cache, bt, cl,
                                          cfg.softmax_scale, s.plan, plan_dev,
                                          max_context_len=s.max_context_len,
                                          workspace=state.workspace, device_status=state.status)
    else:
        pkv.paged_attention_decode(state.out, q, state.k_cache, state.v_cache, bt, cl,
                                   cfg.softmax_scale, max_context_len=s.max_context_len,
                                   partition_size=P, workspace=state.workspace,
                                   device_status=state.status)


def _spread(ms):
    """p10 / median / p90 of per-step times (ms)."""
    a = np.sort(np.asarray(ms, dtype=np.float64))
    return {"p10": round(float(np.percentile(a, 10)), 5), "median": round(float(np.median(a)), 5),
            "p90": round(float(np.percentile(a, 90)), 5)}


def _unflushed_decode(pkv, state, s, P, algo_bytes, peak, reps=5):
    """The last timed step's attention again, `reps` times back to back with
    no L2 flush in between (it only reads the cache and rewrites its output):
    what L2 reuse across launches adds when nothing else runs between them."""
    stream = torch.cuda.current_stream()
    _decode(pkv, state, s, s.q, s.block_tables, s.context_lens, s.plan_device, P)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    _preroll()
    for a, b in evs:
        a.record(stream)
        _decode(pkv, state, s, s.q, s.block_tables, s.context_lens, s.plan_device, P)
        b.record(stream)
    torch.cuda.synchronize()
    ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
    gbs = algo_bytes / (ms / 1e3) / 1e9
    return {"decode_ms_median": round(ms, 5), "achieved": round(gbs, 2), "unit": "GB/s",
            "frac": round(gbs / peak, 4), "launches": reps}


def _flush_l2(buf):
    """Evicts the decode step's data from L2 by reading a 256 MiB buffer (twice
    the L2).  A read leaves clean lines behind, so the timed kernels do not pay
    for writing flush data back to DRAM."""
    torch.sum(buf)


def _preroll():
    """Keeps the GPU busy for ~0.3 ms before a timed step so that the host has
    enqueued the whole step before its first event is reached: the events
    then time the kernels, not Python's launch overhead."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(600_000)


def _pool_blocks(cfg, dev, cap_gb=0.0):
    """Pools given in bytes (the long-context preset, ~60 GB) shrink to 80% of
    the free device memory when the GPU has less room, or to cap_gb."""
    if cfg.pool != "bytes":
        return None
    free = torch.cuda.mem_get_info(dev)[0]
    want = min(cfg.pool_value, 0.8 * free)
    if cap_gb > 0:
        want = min(want, cap_gb * 1e9)
    return int(want // (2 * cfg.block_bytes))


def _split_partition(P, max_len, launches):
    if launches != 2:
        return 0
    return P if P > 0 else 512


# the sources each timed decode kernel is compiled from (its own file and
# every header it includes): a traffic figure stays valid while these are
# unchanged, whatever else in the library changes
_COMMON_SOURCES = ("pa_decode.cuh", "pa_merge.cuh", "pkv_device.cuh")
KERNEL_SOURCES = {
    "pa_decode_kernel": _COMMON_SOURCES,
    "pa_cascade_kernel": _COMMON_SOURCES + ("pa_cascade.cuh", "cascade_plan.h"),
    "pa_cascade_tc05_kernel": _COMMON_SOURCES + ("pa_cascade.cuh", "cascade_plan.h",
                                                 "pa_cascade_tc05.cuh"),
}


def kernel_source_sha(kernel):
    """sha256 prefix over one decode kernel's sources: a traffic figure taken
    on other sources is stale."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_311_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(cfg, kernel, algo_bytes):
    """Per-launch DRAM traffic (read + write) of the decode kernel, from the
    committed ncu capture's traffic / algorithmic-bytes ratio scaled to this
    run's launches; None unless that capture was taken on this workload, with
    this kernel, on its current sources."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(cfg.name, {}).get(kernel)   # {workload: {kernel: figure}}
    if not e or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return int(e["traffic_per_algorithmic_byte"] * algo_bytes)


_PACK_ALIGN = 256   # every piece of a packed step starts on a 256-byte boundary


def _pack_pinned(tensors, pin=True):
    """One host buffer (pinned unless `pin` is false) holding the given CPU
    tensors back to back (each 256-byte aligned), and where each one sits:
    the step's inputs then cross to the device in one copy instead of one
    per tensor."""
    layout, off = {}, 0
    for name, t in tensors.items():
        t = t.contiguous()
        nbytes = t.numel() * t.element_size()
        layout[name] = (off, tuple(t.shape), t.dtype, nbytes)
        off += -(-nbytes // _PACK_ALIGN) * _PACK_ALIGN
    buf = torch.empty(max(off, _PACK_ALIGN), dtype=torch.uint8)
    if pin and torch.cuda.is_available():
        buf = buf.pin_memory()
    for name, t in tensors.items():
        o, shape, dtype, nbytes = layout[name]
        if nbytes:
            buf[o:o + nbytes].copy_(t.contiguous().reshape(-1).view(torch.uint8))
    return buf, layout


def _unpack(dev_buf, layout):
    """Device views of a packed step's tensors."""
    out = {}
    for name, (o, shape, dtype, nbytes) in layout.items():
        out[name] = dev_buf[o:o + nbytes].view(dtype).view(shape)
    return out


def run_e2e(state, steps, host_inputs, P, flush, bytes_step):
    """Same step, inputs from pinned host memory, output read back, all timed.
    Each step's inputs (q, new K/V, slot mapping, block tables, lengths,
    copy-on-write pairs, the shared-prefix plan) were packed into one buffer
    when the step was prepared; before the step they are placed in the one
    pinned staging buffer the loop reuses (as a serving loop reuses its
    own), so a step makes one host-to-device copy and one device-to-host
    copy of the output.  As in the device-timed
    loop, the GPU is kept busy while the host enqueues a step (a serving loop
    prepares step n + 1 while step n runs), so the events time the copies and
    kernels rather than Python's launch latency."""
    import paged_kv_cache_311_gb300 as pkv
    stream = torch.cuda.current_stream()
    dev = state.device
    packed = []
    for s in steps:
        d = {k: getattr(s, k).cpu() for k in
             ("q", "key", "value", "slot_mapping", "block_tables", "context_lens")}
        if s.cow_pairs is not None:
            d["cow_pairs"] = s.cow_pairs.cpu()
        if s.plan is not None:
            d["plan"] = torch.from_numpy(s.plan.host)
        packed.append(_pack_pinned(d, pin=False))
    stage_bytes = max(b.numel() for b, _ in packed)
    dev_buf = torch.empty(stage_bytes, dtype=torch.uint8, device=dev)
    stage = torch.empty(stage_bytes, dtype=torch.uint8)
    if torch.cuda.is_available():
        stage = stage.pin_memory()
    # each step's device views of the staging buffer, made with the step
    views = [_unpack(dev_buf, layout) for _, layout in packed]
    out_host = torch.empty(state.out.shape, dtype=state.out.dtype).pin_memory()
    h2d = d2h = 0
    total_ms = 0.0
    gc.collect()      # no collector pass inside the timed steps
    gc.disable()
    for s, (pbuf, _), t in zip(steps, packed, views):
        hbuf = stage[:pbuf.numel()]
        hbuf.copy_(pbuf)   # the previous step's copies are done (its end event was waited for)
        dst = dev_buf[:hbuf.numel()]
        _flush_l2(flush)
        _preroll()    # the host enqueues the step while the GPU is busy, as in a pipelined loop
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(hbuf, non_blocking=True)
        if "cow_pairs" in t:
            pkv.copy_blocks([state.k_cache], [state.v_cache], t["cow_pairs"], device_status=state.status)
        pkv.reshape_and_cache(t["key"], t["value"], state.k_cache, state.v_cache, t["slot_mapping"],
                              device_status=state.status)
        _decode(pkv, state, s, t["q"], t["block_tables"], t["context_lens"], t.get("plan"), P)
        out_host.copy_(state.out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        total_ms += e0.elapsed_time(e1)
        h2d += hbuf.numel()
        d2h += out_host.numel() * out_host.element_size()
    gc.enable()
    n = len(steps)
    return {"value": round(bytes_step / (total_ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d / n), "d2h_bytes_per_step": int(d2h / n),
            "ms_per_step": round(total_ms / n, 5), "h2d_copies_per_step": 1}


# ----------------------------------------------------- wall-clock serving loop
HOST_E2E_STEPS = 20


def _host_cpu():
    """Host core model and count, for the wall-clock figures."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu part") and not model:
                    model = line.split(":", 1)[1].strip()
    except OSError:
        pass
    parts = {"0xd4f": "Neoverse-V2", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1"}
    return {"machine": platform.machine(), "cores": os.cpu_count(),
            "model": parts.get(model.lower(), model)}


class _Staging:
    """A pinned host buffer and its device twin for one step's small inputs
    (tables, lengths, slots, copy pairs, plan), packed 256-byte aligned so
    that they cross in one copy."""

    def __init__(self, nbytes, dev):
        self.host = torch.empty(nbytes, dtype=torch.uint8)
        if torch.cuda.is_available():
            self.host = self.host.pin_memory()
        self.hnp = self.host.numpy()
        self.dev = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def pack(self, arrays):
        off, views = 0, {}
        for name, a in arrays:
            a = np.ascontiguousarray(a)
            n = a.nbytes
            if off + n > self.hnp.size:
                raise ValueError("staging buffer too small")
            self.hnp[off:off + n] = a.reshape(-1).view(np.uint8)
            views[name] = (off, a.shape, a.dtype, n)
            off += -(-n // _PACK_ALIGN) * _PACK_ALIGN
        return off, views

    def device_views(self, views):
        tdt = {np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}
        return {k: self.dev[o:o + n].view(tdt[dt]).view(shape) for k, (o, shape, dt, n) in views.items()}


def run_host_e2e(cfg, w, state, shared, P, engine, flush, seed, steps, warmup):
    """A serving loop's decode steps through the public API, timed by the
    host's wall clock (time.perf_counter) with no GPU pre-roll: each step's
    block bookkeeping on the product's block pool (continuous batching: the
    finished sequences' release and the new requests' prompt blocks; then
    every sequence's next slot and the copy-on-write pairs, DecodeBatch.step
    -> pkv_block_pool_append_slots), the shared-prefix planner for the shared
    paths, packing the step's tables, lengths, slots, pairs and plan into one
    pinned buffer, its host-to-device copy and those of q and the new K/V
    (prepared beforehand: in a model they come from the layers before), the
    library calls (copy_blocks, reshape_and_cache, decode), the copy of the
    output back to pinned memory and a stream synchronise.  The batch has
    the workload's shapes (lengths, prompts shared or forked as the workload
    shares them), but its blocks are the ones the pool hands out: their
    K/V is written by a prefill scatter before the timed steps."""
    import paged_kv_cache_311_gb300 as pkv
    from paged_kv_cache_311_gb300.batch import DecodeBatch
    from workloads.gen import StepInputs
    dev = state.device
    bs, B, Hk, D, H = cfg.block_size, w.num_seqs, cfg.num_kv_heads, cfg.head_dim, cfg.num_heads
    dt = state.k_cache.dtype
    rng = np.random.default_rng(seed + 77)
    total = warmup + steps
    n_rep = int(round(cfg.replace_fraction * B)) if cfg.kind == "continuous" else 0
    longest = int(max(int(np.max(w.init_lens)), cfg.new_len_hi if n_rep else 0)) + total + bs
    MB = -(-longest // bs)
    pool = pkv.BlockPool(w.num_blocks, bs)
    batch = DecodeBatch(pool, B, MB)

    # the batch's requests, shaped as the workload's
    prefill = []
    if cfg.kind == "shared_prefix":
        S = cfg.samples_per_prompt
        for p, lp in enumerate(w.prompt_lens):
            prefill.append(batch.add_prompt(p * S, rng.integers(0, 32000, int(lp)))[0])
            for k in range(1, S):
                batch.fork(p * S, p * S + k)
    elif cfg.kind == "system_prompt":
        sys_toks = [rng.integers(0, 32000, int(lp)) for lp in w.prompt_lens]
        for i in range(B):
            toks = np.concatenate([sys_toks[int(w.prompt_of[i])],
                                   rng.integers(0, 32000, int(w.own_lens[i]))])
            prefill.append(batch.add_prompt(i, toks)[0])
            batch.commit(i, toks)
    else:
        for i in range(B):
            prefill.append(batch.add_prompt(i, rng.integers(0, 32000, int(w.init_lens[i])))[0])
    pre = np.concatenate(prefill)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 78)
    chunk = max(1, (64 << 20) // (Hk * D * 4))
    for c in range(0, pre.size, chunk):
        sl = torch.from_numpy(pre[c:c + chunk]).to(dev)
        k = torch.randn((sl.numel(), Hk, D), generator=gen, device=dev).to(dt)
        v = torch.randn((sl.numel(), Hk, D), generator=gen, device=dev).to(dt)
        pkv.reshape_and_cache(k, v, state.k_cache, state.v_cache, sl, device_status=state.status)
    torch.cuda.synchronize()

    # per step: the replaced rows and their prompts (continuous batching)
    plans = []
    for _ in range(total):
        rows = rng.choice(B, size=n_rep, replace=False) if n_rep else []
        plans.append([(int(r), rng.integers(0, 32000, int(rng.integers(cfg.new_len_lo,
                                                                          cfg.new_len_hi + 1))))
                      for r in rows])
    t_max = B + n_rep * (cfg.new_len_hi if n_rep else 0)
    hq = _normal_pinned((B, H, D), dt, gen)
    hk = _normal_pinned((t_max, Hk, D), dt, gen)
    hv = _normal_pinned((t_max, Hk, D), dt, gen)
    dq = torch.empty_like(hq, device=dev)
    dk = torch.empty_like(hk, device=dev)
    dv = torch.empty_like(hv, device=dev)
    out_host = torch.empty(state.out.shape, dtype=state.out.dtype).pin_memory()
    meta_bytes = B * MB * 4 + B * 4 + t_max * 8 + B * 16 + 8 * _PACK_ALIGN
    if shared:
        meta_bytes += 4 * int(pkv.load_library().pkv_shared_plan_max_ints(
            B, H, Hk, longest, 0))
    stage = _Staging(meta_bytes, dev)
    stream = torch.cuda.current_stream()
    ws = state.workspace
    pkv.set_decode_engine(engine)

    wall, book, plan_t, bytes_ = [], [], [], []
    h2d = d2h = 0
    gc.collect()
    gc.disable()
    for i in range(total):
        _flush_l2(flush)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pre_slots = []
        for row, toks in plans[i]:
            batch.release(row)
            pre_slots.append(batch.add_prompt(row, toks)[0])
        dec_slots, pairs = batch.step(B)
        slots = np.concatenate(pre_slots + [dec_slots]) if pre_slots else dec_slots
        tables, lens = batch.tables[:B], batch.lens[:B]
        max_len = int(lens.max())
        t1 = time.perf_counter()
        plan = None
        arrays = [("bt", tables), ("cl", lens), ("slots", slots)]
        if pairs.shape[0]:
            arrays.append(("pairs", pairs))
        if shared:
            plan = pkv.plan_shared_prefix(tables, lens, H, Hk, D, bs, max_len, 0)
            arrays.append(("plan", plan.host))
        t2 = time.perf_counter()
        nbytes, views = stage.pack(arrays)
        T = slots.size
        stage.dev[:nbytes].copy_(stage.host[:nbytes], non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dk[:T].copy_(hk[:T], non_blocking=True)
        dv[:T].copy_(hv[:T], non_blocking=True)
        d = stage.device_views(views)
        need = (plan.workspace_bytes if shared else
                pkv.paged_attention_workspace_bytes(B, H, max_len, D, P))
        if need and (ws is None or ws.numel() < need):
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
        if pairs.shape[0]:
            pkv.copy_blocks([state.k_cache], [state.v_cache], d["pairs"], device_status=state.status)
        pkv.reshape_and_cache(dk[:T], dv[:T], state.k_cache, state.v_cache, d["slots"],
                              device_status=state.status)
        if shared:
            pkv.paged_attention_decode_shared(state.out, dq, state.k_cache, state.v_cache, d["bt"],
                                              d["cl"], cfg.softmax_scale, plan, d["plan"],
                                              max_context_len=max_len, workspace=ws,
                                              device_status=state.status)
        else:
            pkv.paged_attention_decode(state.out, dq, state.k_cache, state.v_cache, d["bt"], d["cl"],
                                       cfg.softmax_scale, max_context_len=max_len,
                                       partition_size=P, workspace=ws, device_status=state.status)
        launches = pkv.last_decode_launches()
        out_host.copy_(state.out, non_blocking=True)
        stream.synchronize()
        t3 = time.perf_counter()
        if i >= warmup:
            wall.append(t3 - t0)
            book.append(t1 - t0)
            plan_t.append(t2 - t1)
            inp = StepInputs(step=i, slot_mapping=slots, token_seq=np.zeros(T, np.int64),
                             token_pos=np.zeros(T, np.int64), context_lens=lens.copy(),
                             block_tables=tables.copy(), cow_pairs=pairs, max_context_len=max_len)
            bytes_.append((inp, plan, launches))
            h2d += nbytes + dq.numel() * dq.element_size() + 2 * T * Hk * D * dk.element_size()
            d2h += out_host.numel() * out_host.element_size()
    gc.enable()
    pkv.set_decode_engine("auto")
    if state.status.item() != 0:
        raise RuntimeError(f"{cfg.name}: device status {state.status.item()} in the host_e2e steps")
    out_bytes = state.out.element_size()
    nb = sum(_step_bytes(cfg, inp, B, out_bytes, plan, P, n)["total"] for inp, plan, n in bytes_)
    tot = sum(wall)
    n = len(wall)
    return {"value": round(nb / tot / 1e9, 2), "unit": "GB/s", "steps": n, "warmup": warmup,
            "ms_per_step": round(1e3 * tot / n, 4), "seq_steps_per_s": round(B * n / tot, 1),
            "h2d_bytes_per_step": int(h2d / n), "d2h_bytes_per_step": int(d2h / n),
            "host_ms": {"bookkeeping_median": round(1e3 * statistics.median(book), 4),
                        "planner_median": round(1e3 * statistics.median(plan_t), 4),
                        "step_median": round(1e3 * statistics.median(wall), 4)},
            "host": _host_cpu(),
            "timed": "wall clock per step: pool bookkeeping, planner, packing, copies in and out, "
                     "library calls, stream synchronise; no GPU pre-roll, L2 flushed before each"}


def _normal_pinned(shape, dt, gen):
    x = torch.randn(shape, generator=gen, device=gen.device).to(dt)
    return x.cpu().pin_memory()


# ------------------------------------------------------------- CPU oracle
def _raw(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


class _OracleStepper:
    """Host copy of the blocks that `seqs` touch over `inputs`, advanced step
    by step with the oracle's own copy-on-write copies and scatter, and the
    oracle's attention for those sequences."""

    def __init__(self, cfg, num_blocks, seqs, inputs, k_blocks_fn, v_blocks_fn):
        bs = cfg.block_size
        blocks = set()
        for inp in inputs:
            for s in seqs:
                L = int(inp.context_lens[s])
                blocks.update(int(b) for b in inp.block_tables[s][:-(-L // bs)])
            for a, b in inp.cow_pairs:
                if int(b) in blocks or int(a) in blocks:
                    blocks.update((int(a), int(b)))
        self.blocks = np.array(sorted(blocks), dtype=np.int64)
        self.local = np.full(num_blocks, -1, dtype=np.int64)
        self.local[self.blocks] = np.arange(self.blocks.size)
        self.k = k_blocks_fn(self.blocks)
        self.v = v_blocks_fn(self.blocks)
        self.cfg, self.seqs = cfg, np.array(seqs, dtype=np.int64)

    def step(self, inp, q, key, value, nthreads):
        import oracle
        bs = self.cfg.block_size
        if inp.cow_pairs.shape[0]:
            loc = self.local[inp.cow_pairs]
            loc = loc[loc[:, 1] >= 0]
            if loc.shape[0]:
                oracle.copy_blocks([self.k], [self.v], loc)
        sm = inp.slot_mapping
        lb = self.local[sm // bs]
        slots = np.where(lb >= 0, lb * bs + sm % bs, -1)
        oracle.reshape_and_cache(key, value, self.k, self.v, slots)
        t = inp.block_tables[self.seqs]
        tables = np.where(t >= 0, self.local[np.maximum(t, 0)], -1).astype(np.int32)
        out, st = oracle.paged_attention(q[self.seqs], self.k, self.v, self.cfg.dtype, tables,
                                         inp.context_lens[self.seqs], self.cfg.num_kv_heads,
                                         float(np.float32(self.cfg.softmax_scale)),
                                         nthreads=nthreads)
        return out


def _sample_bytes(cfg, inp, seqs):
    """Algorithmic bytes of the oracle's share of one step (its sequences)."""
    sub = _restrict(inp, seqs)
    return algorithmic_bytes(cfg, sub, len(seqs))["total"]


def _restrict(inp, seqs):
    from workloads.gen import StepInputs
    seqs = np.asarray(seqs)
    keep = np.isin(inp.token_seq, seqs)
    pairs = inp.cow_pairs
    if pairs.shape[0]:
        mine = set()
        for s in seqs:
            mine.update(int(b) for b in inp.block_tables[s] if b >= 0)
        pairs = pairs[[int(b) in mine for b in pairs[:, 1]]].reshape(-1, 2)
    return StepInputs(step=inp.step, slot_mapping=inp.slot_mapping[keep],
                      token_seq=inp.token_seq[keep], token_pos=inp.token_pos[keep],
                      context_lens=inp.context_lens[seqs], block_tables=inp.block_tables[seqs],
                      cow_pairs=pairs, max_context_len=int(inp.context_lens[seqs].max()))


def cpu_baseline(cfg, state, host_inputs, budget_s, seed):
    """The oracle, as it stands, on whole steps of this workload (copies,
    scatter and attention over every sequence, the same values as the GPU
    run) until about budget_s seconds of it are spent."""
    from workloads import step_values
    nthreads = os.cpu_count() or 1
    seqs = list(range(state.w.num_seqs))

    def take(cache):
        def f(blocks):
            idx = torch.as_tensor(blocks, device=cache.device)
            return _raw(cache.index_select(0, idx))
        return f

    st = _OracleStepper(cfg, state.w.num_blocks, seqs, host_inputs, take(state.k_cache),
                        take(state.v_cache))
    done, t_used, nbytes = 0, 0.0, 0
    for inp in host_inputs:
        q, k, v = step_values(cfg, seed, inp, state.w.num_seqs, device=state.device)
        q, k, v = _raw(q), _raw(k), _raw(v)
        t0 = time.perf_counter()
        st.step(inp, q, k, v, nthreads)
        t_used += time.perf_counter() - t0
        nbytes += algorithmic_bytes(cfg, inp, state.w.num_seqs)["total"]
        done += 1
        if t_used >= budget_s:
            break
    return {"value": round(nbytes / t_used / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "kind": "oracle", "seconds": round(t_used, 2),
            "sample": f"steps 0..{done - 1} of {cfg.name}: all {state.w.num_seqs} sequences, "
                      f"copy-on-write + scatter + fp64 attention (C, {nthreads} threads)"}


# -------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as the reference arm: each step runs the oracle (as it
    stands, all host cores) on a fixed sample of the step's sequences, sized
    so that warm-up plus timed steps end within about three minutes."""
    dist, rank, world = dist_setup()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    from workloads import TAG_CACHE_K, TAG_CACHE_V, normal, step_values
    cfg = get(args.config)
    if args.block_size:
        cfg = cfg.with_(block_size=args.block_size)
    seed = SEED_BASE + CONFIGS.index(get(args.config))
    total = args.warmup + args.steps
    w = PagedDecodeWorkload(cfg, seed, total_steps=max(total, cfg.steps))
    inputs = [w.next_step() for _ in range(total)]
    nthreads = os.cpu_count() or 1
    shape = (cfg.num_kv_heads, cfg.block_size, cfg.head_dim)

    def fill(tag):
        def f(blocks):
            x = normal((blocks.size,) + shape, cfg.dtype, seed, tag, 0, device="cpu")
            return _raw(x)
        return f

    def stepper(seqs):
        return _OracleStepper(cfg, w.num_blocks, seqs, inputs, fill(TAG_CACHE_K), fill(TAG_CACHE_V))

    def values(inp):
        q, k, v = step_values(cfg, seed, inp, w.num_seqs, device="cpu")
        return _raw(q), _raw(k), _raw(v)

    # calibrate: one thread's time for one sequence, then size the sample
    probe = stepper([0])
    q, k, v = values(inputs[0])
    t0 = time.perf_counter()
    probe.step(inputs[0], q, k, v, 1)
    t1 = max(time.perf_counter() - t0, 1e-4)
    per_step = 150.0 / max(total, 1)
    n = int(max(1, min(w.num_seqs, per_step * nthreads / t1)))
    n = max(1, (n // nthreads) * nthreads) if n >= nthreads else n
    seqs = list(range(n))
    st = stepper(seqs)
    times, nbytes = [], 0
    for i, inp in enumerate(inputs):
        q, k, v = values(inp)
        t0 = time.perf_counter()
        st.step(inp, q, k, v, nthreads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes += _sample_bytes(cfg, inp, seqs)
    tot = sum(times)
    value = nbytes / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot * 1e3 / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "kv_dtype": cfg.dtype, "num_seqs": w.num_seqs,
                       "sampled_seqs": n, "num_heads": cfg.num_heads,
                       "num_kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
                       "block_size": cfg.block_size},
            "seq_steps_per_s": round(n * len(times) / tot, 2),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                             "kind": "oracle",
                             "sample": f"sequences 0..{n - 1} of {w.num_seqs} of every step: "
                                       "copy-on-write + scatter + fp64 attention"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_swap(args):
    """Swap-out and swap-in of every block of about a tenth of the workload's
    sequences (preemption), against the host link's own copy bandwidth
    measured in the same run (one pinned cudaMemcpyAsync of the same bytes
    each way) and against one copy per block (the many small transfers the
    pages name as the cost of swapping small blocks)."""
    import paged_kv_cache_311_gb300 as pkv
    dev = local_device()
    cfg = get(args.config)
    if args.block_size:
        cfg = cfg.with_(block_size=args.block_size)
    seed = SEED_BASE + CONFIGS.index(get(args.config))
    w = PagedDecodeWorkload(cfg, seed, total_steps=max(args.warmup + args.steps, 1),
                            pool_blocks=_pool_blocks(cfg, dev, args.pool_gb))
    state = DeviceState(cfg, w, seed, device=dev)
    inp = w.next_step()
    n_out = max(1, w.num_seqs // 10)
    blocks = []
    for s in range(n_out):
        nb = -(-int(inp.context_lens[s]) // cfg.block_size)
        blocks += [int(b) for b in inp.block_tables[s][:nb]]
    blocks = sorted(set(blocks))
    n = len(blocks)
    pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int64, device=dev)
    shape = (n,) + tuple(state.k_cache.shape[1:])
    hk = torch.empty(shape, dtype=state.k_cache.dtype).pin_memory()
    hv = torch.empty(shape, dtype=state.k_cache.dtype).pin_memory()
    nbytes = 2 * n * cfg.block_bytes
    stream = torch.cuda.current_stream()
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(fn, reps):
        ms = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return sorted(ms)[len(ms) // 2]

    out = lambda: pkv.swap_blocks([state.k_cache], [state.v_cache], [hk], [hv], pairs, pkv.SWAP_OUT,
                                  device_status=st)
    inn = lambda: pkv.swap_blocks([state.k_cache], [state.v_cache], [hk], [hv], pairs, pkv.SWAP_IN,
                                  device_status=st)
    for _ in range(args.warmup):
        out(); inn()
    torch.cuda.synchronize()
    reps = max(args.steps, 3)
    t_out, t_in = timed(out, reps), timed(inn, reps)
    # the link: one contiguous copy of the same bytes each way
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    t_d2h = timed(lambda: hbuf.copy_(dbuf, non_blocking=True), reps)
    t_h2d = timed(lambda: dbuf.copy_(hbuf, non_blocking=True), reps)
    # one copy per block and cache (copy engines, no gather kernel)
    idx = pairs[:, 0].tolist()
    def per_block():
        for i, b in enumerate(idx):
            hk[i].copy_(state.k_cache[b], non_blocking=True)
            hv[i].copy_(state.v_cache[b], non_blocking=True)
    t_small = timed(per_block, max(3, reps // 3))
    if st.item() != 0:
        raise RuntimeError(f"device status {st.item()} during the swaps")
    gbs = lambda t: nbytes / (t / 1e3) / 1e9
    line = {"metric": "swap_blocks: block bytes moved per second between the GPU pool and pinned host memory",
            "value": round(gbs(t_out), 2), "unit": "GB/s", "n_gpus": 1, "steps": reps,
            "warmup": args.warmup, "ms_per_step": round(t_out, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": cfg.name, "block_size": cfg.block_size, "blocks": n,
                       "sequences_swapped": n_out, "bytes": nbytes, "block_bytes": cfg.block_bytes},
            "swap_in": {"value": round(gbs(t_in), 2), "unit": "GB/s", "ms": round(t_in, 5)},
            "roofline": {"bound": "host link", "unit": "GB/s",
                         "out": {"achieved": round(gbs(t_out), 2), "peak": round(gbs(t_d2h), 2),
                                 "frac": round(t_d2h / t_out, 4)},
                         "in": {"achieved": round(gbs(t_in), 2), "peak": round(gbs(t_h2d), 2),
                                "frac": round(t_h2d / t_in, 4)},
                         "peak_source": "one pinned cudaMemcpyAsync of the same bytes, same run"},
            "one_copy_per_block": {"value": round(gbs(t_small), 2), "unit": "GB/s",
                                   "ms": round(t_small, 5)},
            "gpu_launches": 1}
    print(json.dumps(line))


def run_host_step(args):
    """A decode step's host bookkeeping for the workload's batch, timed on the
    host cores (no GPU): the block pool giving every sequence its next slot
    in one call (append_slots) and one call per sequence, and, for workloads
    with shared prompts, the shared-prefix planner on the step's tables.
    Prints one JSON line of medians in microseconds per step."""
    import paged_kv_cache_311_gb300 as pkv
    cfg = get(args.config)
    if args.block_size:
        cfg = cfg.with_(block_size=args.block_size)
    seed = SEED_BASE + CONFIGS.index(get(args.config))
    steps = max(args.steps, 3)
    w = PagedDecodeWorkload(cfg, seed, total_steps=max(steps + args.warmup, 2),
                            num_seqs=args.num_seqs or None, pool_blocks=None if cfg.pool != "bytes" else 1 << 20)
    inputs = [w.next_step() for _ in range(args.warmup + steps)]
    bs, B = cfg.block_size, w.num_seqs
    res = {}
    # the pool: the batch's first-step lengths, then one token per sequence per step
    first = inputs[0]
    MB = int(first.block_tables.shape[1]) + steps + 2
    nb_total = int(sum(-(-int(L) // bs) + steps // bs + 2 for L in first.context_lens))
    for mode in ("append_slots", "per_sequence"):
        pool = pkv.BlockPool(nb_total + B, bs)
        rows = np.full((B, MB), -1, np.int32)
        lens = np.asarray(first.context_lens, np.int32).copy()
        for s in range(B):
            t = pool.allocate(-(-int(lens[s]) // bs))
            rows[s, :t.size] = t
        ts = []
        for i in range(args.warmup + steps):
            t0 = time.perf_counter()
            if mode == "append_slots":
                pool.append_slots(rows, lens)
            else:
                for s in range(B):
                    j, off = divmod(int(lens[s]), bs)
                    if off == 0:
                        rows[s, j] = pool.allocate(1)[0]
                    else:
                        pool.prepare_write(rows[s], j)
            ts.append(time.perf_counter() - t0)
            lens += 1
        res[f"pool_{mode}_us"] = round(1e6 * statistics.median(ts[args.warmup:]), 1)
    if cfg.kind in ("shared_prefix", "system_prompt"):
        ts = []
        for inp in inputs:
            t0 = time.perf_counter()
            pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads, cfg.num_kv_heads,
                                   cfg.head_dim, bs, int(inp.context_lens.max()), 0)
            ts.append(time.perf_counter() - t0)
        res["plan_shared_prefix_us"] = round(1e6 * statistics.median(ts[args.warmup:]), 1)
    import platform
    print(json.dumps({"metric": "host bookkeeping per decode step (median us)", "op": "host_step",
                      "unit": "us", "higher_is_better": False, "steps": steps, "warmup": args.warmup,
                      "config": {"workload": cfg.name, "num_seqs": B, "block_size": bs},
                      "host": {"machine": platform.machine(), "cores": os.cpu_count()},
                      **res}))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "swap_blocks":
        run_swap(args)
    elif args.op == "host_step":
        run_host_step(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
