"""Benchmark: paged decode attention on one Llama-3-8B-shaped layer.

One step = the decode-step KV-append of one new token per sequence followed
by paged GQA decode attention (partition kernel + split-K merge) over
64 sequences with context lengths uniform in [512, 4096] (seeded), 32 query /
8 KV heads, head dim 128, bf16, 16-token blocks from a 40,000-block pool in
seeded random order.  The metric is decode-attention KV bytes per second
(4,096 bytes per token per layer: K and V, 8 heads x 128 x 2 bytes).

Prints ONE JSON line.  Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
N > 1 runs under torch.distributed.run, one rank per GPU; every rank decodes
its own batch (weak scaling, no collective on the data path; the barrier and
the max-over-ranks of the elapsed time are the only cross-rank calls).
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

WORKLOAD = "llama3_8b_b64"
METRIC = "decode-attention KV GB/s and % of GB300 HBM peak; sequences/s per layer"
KV_BYTES_PER_TOKEN = 2 * 8 * 128 * 2  # K and V, 8 KV heads, head dim 128, bf16
L2_BYTES = 129 * 10 ** 6
NOMINAL_HBM_GBS = 8000.0
DECODE_SOURCES = ["paged_kv_cache_13_gb300/csrc/decode.cu", "paged_kv_cache_13_gb300/csrc/common.cuh"]
TRAFFIC_FILE = "profiles/paged_decode_bf16_llama3_8b_b64_traffic.txt"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--partition-size", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool-blocks", type=int, default=0,
                    help="override the pool size (blocks); 0 keeps the workload's 40,000")
    ap.add_argument("--cpu-worker", type=float, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


# ----------------------------------------------------------------- helpers
def shard(n, world, rank):
    """Contiguous share [lo, hi) of n independent units for one rank."""
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (the job ends with its slowest rank)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world / seconds


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_digest():
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kv_bytes_per_launch):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, scaled to this launch; None if the kernel changed since."""
    p = os.path.join(ROOT, TRAFFIC_FILE)
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != source_digest():
        return None
    try:
        per_kv_byte = float(vals["dram_bytes_per_launch"]) / float(vals["kv_bytes_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None
    return per_kv_byte * kv_bytes_per_launch


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        self.path = os.path.join("/tmp", "pkv_clocks_%d_%d.csv" % (os.getpid(), device_index))

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- device setup
class Layer:
    """The workload's cache, built with the library's own entry points."""

    def __init__(self, pkv, torch, device, partition_size, headroom_tokens, pool_blocks=0):
        import synthetic as syn
        self.pkv, self.torch, self.dev = pkv, torch, device
        w = syn.workload(WORKLOAD, **({"num_blocks": pool_blocks} if pool_blocks else {}))
        self.w = w
        NB, BS, Hkv, D, Hq = w["num_blocks"], w["block_size"], w["hkv"], w["d"], w["hq"]
        dt = w["torch_dtype"]
        self.pool = pkv.pkv_pool_create(NB, BS, syn.free_order(w))
        self.k_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
        self.v_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
        ops, decoded = syn.prefill_schedule(w)
        self.seqs = np.array(decoded, dtype=np.int64)
        B = len(decoded)
        rows = {}
        for op in ops:
            if op[0] == "create":
                pkv.pkv_seq_create(self.pool)
            elif op[0] == "append":
                _, h, n = op
                slots, pairs = pkv.pkv_seq_append(self.pool, h, n)
                assert not pairs
                k, v = syn.sequence_kv(w, h)
                rows[h] = (k, v)
                pkv.pkv_kv_append(k[:n].to(device), v[:n].to(device),
                                  torch.from_numpy(slots).to(device), self.k_pool, self.v_pool)
        # the decode step's append: token L-1 of every sequence
        slots, pairs = pkv.pkv_seq_append_batch(self.pool, self.seqs, 1)
        self.new_k = torch.stack([rows[h][0][-1] for h in decoded]).to(device)
        self.new_v = torch.stack([rows[h][1][-1] for h in decoded]).to(device)
        self.slots = torch.from_numpy(slots.copy()).to(device)
        lens = syn.context_lengths(w)
        self.max_blocks = -(-max(lens) // BS)  # exact: the timed decode reads these tables
        self.max_blocks_grown = -(-(max(lens) + headroom_tokens) // BS)  # for the e2e loop
        tables, ctx = pkv.pkv_build_block_tables(self.pool, self.seqs, self.max_blocks)
        self.tables = torch.from_numpy(tables.copy()).to(device)
        self.lens = torch.from_numpy(ctx.copy()).to(device)
        self.ctx_host = ctx.copy()
        self.q = syn.query(w).to(device)
        self.out = torch.empty((B, Hq, D), dtype=dt, device=device)
        self.partition_size = partition_size
        ws = pkv.pkv_decode_workspace_bytes(B, Hq, D, self.max_blocks, BS, partition_size)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.B = B
        torch.cuda.synchronize()

    def kv_bytes(self, ctx=None):
        return int(np.sum(self.ctx_host if ctx is None else ctx)) * KV_BYTES_PER_TOKEN

    # one step, device-resident inputs: one kernel appends the new rows and
    # attends (split-K partials merged by the last CTA of each sequence/head)
    def step(self):
        self.pkv.pkv_paged_attention_decode_append(
            self.q, self.new_k, self.new_v, self.slots, self.k_pool, self.v_pool, self.tables,
            self.lens, self.w["scale"], self.out, self.ws, self.partition_size)


def run_device(args, rank, world, dist):
    import torch
    import paged_kv_cache_13_gb300 as pkv

    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    device = torch.device("cuda", dev_index)
    e2e_steps = max(1, min(args.steps, 200))
    layer = Layer(pkv, torch, device, args.partition_size, headroom_tokens=e2e_steps + args.warmup + 8,
                  pool_blocks=args.pool_blocks)
    stream = torch.cuda.current_stream()
    kv_bytes = layer.kv_bytes()

    # ---------- device-resident timed region
    for _ in range(args.warmup):
        layer.step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev_index)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        layer.step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    assert pkv.pkv_device_status() == 0
    elapsed_ms = max_over_ranks(elapsed_ms, dist, device)
    ms_per_step = elapsed_ms / args.steps

    # ---------- end to end through the public API, host buffers
    e2e = run_e2e(pkv, torch, layer, e2e_steps, dist, device)

    return dict(ms_per_step=ms_per_step, kern_ms=kern_ms, kv_bytes=kv_bytes, clocks=clk, e2e=e2e,
                B=layer.B, launches=2 * args.steps)  # partials + merge per step


def run_e2e(pkv, torch, layer, steps, dist, device):
    """Every step: host allocator append + tables, H2D of q / new K,V / slots /
    tables / lens from pinned memory, KV-append + decode, D2H of the output."""
    import synthetic as syn
    w = layer.w
    B, Hq, Hkv, D = layer.B, w["hq"], w["hkv"], w["d"]
    dt = w["torch_dtype"]
    pin = dict(pin_memory=True)
    h_q = torch.empty((B, Hq, D), dtype=dt, **pin)
    h_k = torch.empty((B, Hkv, D), dtype=dt, **pin)
    h_v = torch.empty((B, Hkv, D), dtype=dt, **pin)
    h_slots = torch.empty(B, dtype=torch.int64, **pin)
    h_pairs = torch.empty(2 * B, dtype=torch.int32, **pin)
    mb = layer.max_blocks_grown
    h_tab = torch.empty((B, mb), dtype=torch.int32, **pin)
    h_lens = torch.empty(B, dtype=torch.int32, **pin)
    h_out = torch.empty((B, Hq, D), dtype=dt, **pin)
    d_q = torch.empty_like(h_q, device=device)
    d_k = torch.empty_like(h_k, device=device)
    d_v = torch.empty_like(h_v, device=device)
    d_slots = torch.empty_like(h_slots, device=device)
    d_tab = torch.empty_like(h_tab, device=device)
    d_lens = torch.empty_like(h_lens, device=device)
    d_out = torch.empty_like(h_out, device=device)
    ws = torch.empty(max(16, pkv.pkv_decode_workspace_bytes(B, Hq, D, mb, 16, layer.partition_size)),
                     dtype=torch.uint8, device=device)
    # fresh per-step inputs, generated before the timed region
    inputs = []
    for s in range(steps):
        k, v = syn.new_token_kv(w, s)
        inputs.append((k, v))
    h_q.copy_(syn.query(w))
    stream = torch.cuda.current_stream()
    h2d = (h_q.numel() * 2 + h_k.numel() * 2 + h_v.numel() * 2 + h_slots.numel() * 8
           + h_tab.numel() * 4 + h_lens.numel() * 4)
    d2h = h_out.numel() * 2
    total_kv = 0
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    for s in range(steps):
        h_k.copy_(inputs[s][0])
        h_v.copy_(inputs[s][1])
        slots, pairs = pkv.pkv_seq_append_batch(layer.pool, layer.seqs, 1, h_slots.numpy(), h_pairs.numpy())
        assert len(pairs) == 0
        pkv.pkv_build_block_tables(layer.pool, layer.seqs, mb, h_tab.numpy(), h_lens.numpy())
        total_kv += int(h_lens.numpy().sum()) * KV_BYTES_PER_TOKEN
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_slots.copy_(h_slots, non_blocking=True)
        d_tab.copy_(h_tab, non_blocking=True)
        d_lens.copy_(h_lens, non_blocking=True)
        pkv.pkv_paged_attention_decode_append(d_q, d_k, d_v, d_slots, layer.k_pool, layer.v_pool,
                                              d_tab, d_lens, w["scale"], d_out, ws,
                                              layer.partition_size, stream)
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()
    elapsed = max_over_ranks(time.perf_counter() - t_start, dist, device)
    assert torch.isfinite(h_out.float()).all()
    return dict(gbs=total_kv / elapsed / 1e9, h2d=h2d, d2h=d2h, steps=steps)


# -------------------------------------------------------------- CPU oracle
def cpu_worker(min_seconds):
    """Times the oracle's paged decode on a sample of the workload (16 of
    the 64 sequences, all 32 query heads), repeated until min_seconds."""
    import synthetic as syn
    from oracle import allocator, attention, kvcache
    w = syn.workload(WORKLOAD)
    S = 16
    q = syn.kv_rows_to_numpy(syn.query(w))[:S]
    ks, vs = [], []
    for i in range(S):
        k, v = syn.sequence_kv(w, i)
        ks.append(syn.kv_rows_to_numpy(k))
        vs.append(syn.kv_rows_to_numpy(v))
    nb = sum(-(-k.shape[0] // 16) for k in ks)
    m = allocator.KVCacheManager(nb, 16, syn.free_order(dict(w, num_blocks=nb)))
    kp = np.zeros((nb, w["hkv"], 16, w["d"]), np.float32)
    vp = np.zeros_like(kp)
    sids = []
    for i in range(S):
        s = m.create()
        slots, _ = m.append(s, ks[i].shape[0])
        kvcache.kv_append(ks[i], vs[i], slots, kp, vp)
        sids.append(s)
    tables, ctx = m.block_tables(sids, max(len(m.table(s)) for s in sids))
    reps, t0 = 0, time.perf_counter()
    while True:
        attention.paged_attention_decode(q, kp, vp, tables, ctx, w["scale"])
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    kv = int(np.sum(ctx)) * KV_BYTES_PER_TOKEN * reps
    print(json.dumps({"seconds": dt, "reps": reps, "kv_bytes": kv, "seqs": S * reps}))


def cpu_baseline(min_seconds):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(min_seconds)],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        return None
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return {
        "value": res["kv_bytes"] / res["seconds"] / 1e9,
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": "float64 NumPy oracle paged decode of 16 of the 64 sequences (all 32 query "
                  "heads), repeated %d times in %.1f s, single thread" % (res["reps"], res["seconds"]),
        "seq_per_s": res["seqs"] / res["seconds"],
    }


def config_block(B, kv_bytes, partition_size):
    return {
        "workload": "%s: one Llama-3-8B-shaped layer, %d sequences, context uniform in [512, 4096] "
                    "(seeded), 32 q / 8 KV heads, head dim 128, bf16, 16-token blocks, 40,000-block "
                    "pool in seeded random order; step = KV-append of 1 token per sequence + paged "
                    "decode attention (split-K partials with the append fused, then a merge launched with programmatic dependent launch; %d-token partitions)" % (WORKLOAD, B, partition_size),
        "batch": B,
        "kv_bytes_per_step": kv_bytes,
        "partition_size": partition_size,
        "l2": "inputs larger than L2 (%.0f MB of KV read per step vs 129 MB L2), no flush" % (kv_bytes / 1e6),
    }


def main():
    args = parse_args()
    if args.cpu_worker is not None:
        cpu_worker(args.cpu_worker)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, world)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    res = run_device(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return
    value = whole_job_rate(res["kv_bytes"], world, res["ms_per_step"] * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = res["kv_bytes"] / (res["kern_ms"] * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(10.0)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_block(res["B"], res["kv_bytes"], args.partition_size),
        "seq_per_s_per_layer": round(res["B"] * world / (res["ms_per_step"] * 1e-3), 1),
        "pct_of_8tbs_nominal": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100.0 * value / world / peak, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "paged_decode_kernel<bf16, 128, split-K partials, fused append> + merge_kernel (programmatic dependent launch)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy burst)" if peak_kind == "measured" else peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(res["kv_bytes"]),
            "algorithmic_bytes_per_launch": res["kv_bytes"],
            "avg_launch_ms": res["kern_ms"],
        },
        "e2e": {
            "value": round(res["e2e"]["gbs"] * world, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": res["e2e"]["h2d"],
            "d2h_bytes_per_step": res["e2e"]["d2h"],
            "steps": res["e2e"]["steps"],
        },
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))


def run_reference(args, world):
    """The oracle, as it stands, on the host cores: each step is the oracle's
    paged decode of a bounded sample (2 of the 64 sequences, all heads)."""
    import synthetic as syn
    from oracle import allocator, attention, kvcache
    w = syn.workload(WORKLOAD)
    S = 2
    q = syn.kv_rows_to_numpy(syn.query(w))[:S]
    ks, vs = [], []
    for i in range(S):
        k, v = syn.sequence_kv(w, i)
        ks.append(syn.kv_rows_to_numpy(k))
        vs.append(syn.kv_rows_to_numpy(v))
    nb = sum(-(-k.shape[0] // 16) for k in ks)
    m = allocator.KVCacheManager(nb, 16, syn.free_order(dict(w, num_blocks=nb)))
    kp = np.zeros((nb, w["hkv"], 16, w["d"]), np.float32)
    vp = np.zeros_like(kp)
    sids = []
    for i in range(S):
        s = m.create()
        slots, _ = m.append(s, ks[i].shape[0])
        kvcache.kv_append(ks[i], vs[i], slots, kp, vp)
        sids.append(s)
    tables, ctx = m.block_tables(sids, max(len(m.table(s)) for s in sids))
    for _ in range(args.warmup):
        attention.paged_attention_decode(q, kp, vp, tables, ctx, w["scale"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attention.paged_attention_decode(q, kp, vp, tables, ctx, w["scale"])
    dt = time.perf_counter() - t0
    kv = int(np.sum(ctx)) * KV_BYTES_PER_TOKEN
    value = kv * args.steps / dt / 1e9
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    cores = int(threads) if threads and threads.isdigit() else len(os.sched_getaffinity(0))
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": config_block(64, kv, args.partition_size),
        "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": cores,
                         "sample": "float64 NumPy oracle paged decode of 2 of the 64 sequences "
                                   "(%d tokens, all 32 query heads) per step" % int(np.sum(ctx))},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
