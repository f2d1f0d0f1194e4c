"""Benchmark: paged decode attention (KV GB/s, % of HBM peak, sequences/s).

Default workload (the one the headline metric is quoted on): one
Llama-3-8B-shaped layer -- 64 sequences with context lengths uniform in
[512, 4096] (seeded), 32 query / 8 KV heads, head dim 128, bf16, 16-token
blocks from a 40,000-block pool in seeded random order.  One step = the
decode step's KV-append of one new token per sequence and paged GQA decode
attention over the whole context (split-K partition kernel with the append
fused in, then the merge kernel).  The metric counts the KV bytes the decode
attention reads: 4,096 bytes per token per layer (K and V, 8 heads x 128 x
2 bytes).

Other workloads (``--workload``, one JSON line each):
  long_splitk   4 sequences of 65,536 / 32,768 x 3 tokens, interleaved blocks
  quant_int4    32 x 16,384 tokens, INT4 cache (group = head dim), 4 sinks:
                step = quantised append + quantised decode, 1,088 B/token
  quant_fp8     the same with an FP8 E4M3 cache, 2,080 B/token
  prefix_cow    8 children forked from a 2,000-token prompt + tails of
                1..300 tokens (logical bytes: shared blocks counted per child)

Prints ONE JSON line.  Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
                    [--workload NAME]
N > 1 runs under torch.distributed.run, one rank per GPU; every rank builds
and decodes its own replica of the whole workload (replicas only: weak
scaling, no collective on the data path; the barrier and the max-over-ranks
of the elapsed time are the only cross-rank calls).
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

METRIC = "decode-attention KV GB/s and % of GB300 HBM peak; sequences/s per layer"
KV_BYTES_PER_TOKEN = 2 * 8 * 128 * 2  # K and V, 8 KV heads, head dim 128, bf16
NOMINAL_HBM_GBS = 8000.0
# the end-to-end leg runs at least this many pipelined steps, whatever --steps
# is, so that filling and draining the copy/compute pipeline does not dominate
E2E_MIN_STEPS = 4000
E2E_RING = 64  # pinned host input buffers the end-to-end leg cycles through
_CSRC = "paged_kv_cache_13_gb300/csrc/"
# workload -> (committed ncu traffic summary of its decode kernel, the sources
# that kernel is built from); the traffic is reported only while they hash
# to the summary's source_sha256_16
TRAFFIC = {
    "llama3_8b_b64": ("profiles/paged_decode_bf16_llama3_8b_b64_traffic.txt",
                      [_CSRC + "decode.cu", _CSRC + "common.cuh", _CSRC + "balanced.cuh"]),
    "quant_int4": ("profiles/paged_decode_quant_int4_32x16k_traffic.txt",
                   [_CSRC + "decode_quant.cu", _CSRC + "common.cuh", _CSRC + "balanced.cuh"]),
    "quant_fp8": ("profiles/paged_decode_quant_fp8_32x16k_traffic.txt",
                  [_CSRC + "decode_quant.cu", _CSRC + "common.cuh", _CSRC + "balanced.cuh"]),
}



def _slab_overrides(syn):
    """The 64-sequence layer as one contiguous slab per (sequence, KV head):
    each of the 64 x 8 (sequence, KV head) pairs becomes a sequence with one
    KV head and its GQA group of 4 query heads, whose blocks are allocated in
    ascending order, so its K (and V) rows are one contiguous run -- the
    layout of an unpaged [sequence, head, token, dim] cache, read by the same
    kernel at the same bytes."""
    base = syn.workload("llama3_8b_b64")
    lens = syn.context_lengths(base)
    return {"lens": [L for L in lens for _ in range(base["hkv"])], "hq": base["hq"] // base["hkv"],
            "hkv": 1, "in_order": True, "num_blocks": base["num_blocks"] * base["hkv"]}


# name -> (synthetic workload, overrides (or a function of the synthetic
# module returning them), cache mode)
WORKLOADS = {
    "llama3_8b_b64": ("llama3_8b_b64", {}, None),
    "llama3_8b_b64_bs8": ("llama3_8b_b64", {"block_size": 8, "num_blocks": 80000}, None),
    "llama3_8b_b64_bs32": ("llama3_8b_b64", {"block_size": 32, "num_blocks": 20000}, None),
    "llama3_8b_b64_in_order": ("llama3_8b_b64", {"in_order": True}, None),
    "llama3_8b_b64_slab": ("llama3_8b_b64", _slab_overrides, None),
    "long_splitk": ("long_splitk", {}, None),
    "quant_int4": ("quant", {}, "int4"),
    "quant_fp8": ("quant", {}, "fp8"),
    "quant_int4_g64": ("quant", {"group_size": 64, "n_sink": 8}, "int4"),
    "quant_int4_bie": ("quant", {"group_size": 64, "n_sink": 8, "window": 128}, "int4"),
    "prefix_cow": ("prefix_cow", {}, None),
    "verify_b64_g5": ("llama3_8b_b64", {}, None),
    "prefill_chunk512": ("llama3_8b_b64", {"lens": [4096] * 8, "num_blocks": 4096}, None),
}

# decoded rows per model sequence (the slab layout decodes each KV head's
# group as its own row)
ROWS_PER_SEQ = {"llama3_8b_b64_slab": 8}

# multi-query workloads: query tokens per sequence (the last ones of its context)
MQ_LEN = {"verify_b64_g5": 6, "prefill_chunk512": 512}

DESCRIPTIONS = {
    "llama3_8b_b64": "one Llama-3-8B-shaped layer, 64 sequences, context uniform in [512, 4096] "
                     "(seeded), 32 q / 8 KV heads, head dim 128, bf16, 16-token blocks, "
                     "40,000-block pool in seeded random order",
    "llama3_8b_b64_bs8": "the 64-sequence Llama-3-8B-shaped layer (contexts uniform in [512, 4096], "
                         "32 q / 8 KV heads, head dim 128, bf16) in 8-token blocks: 80,000-block "
                         "pool in seeded random order (same bytes as the 16-token pool)",
    "llama3_8b_b64_bs32": "the 64-sequence Llama-3-8B-shaped layer in 32-token blocks: 20,000-block "
                          "pool in seeded random order (same bytes as the 16-token pool)",
    "llama3_8b_b64_in_order": "the 64-sequence Llama-3-8B-shaped layer in 16-token blocks allocated "
                              "in ascending order: each sequence's prompt blocks are consecutive "
                              "(paged layout, unscattered)",
    "llama3_8b_b64_slab": "the 64-sequence Llama-3-8B-shaped layer as 512 contiguous (sequence, KV "
                          "head) slabs: each pair is a 1-KV-head sequence with its 4 query heads "
                          "and consecutive blocks, i.e. the unpaged [sequence, head, token, dim] "
                          "layout, read by the same kernel at the same bytes",
    "long_splitk": "4 sequences of 65,536 / 32,768 / 32,768 / 32,768 tokens, blocks allocated "
                   "round-robin across the sequences from a shuffled 12,288-block pool, 32 q / 8 "
                   "KV heads, head dim 128, bf16",
    "quant_int4": "32 sequences x 16,384 tokens, 32 q / 8 KV heads, head dim 128, bf16 queries, "
                  "INT4 asymmetric cache with fp16 scale/zero per (token, head), 4 bf16 sink "
                  "tokens, values N(0,1) with 1% outliers at +-8",
    "quant_fp8": "32 sequences x 16,384 tokens, 32 q / 8 KV heads, head dim 128, bf16 queries, "
                 "FP8 E4M3 cache with an fp16 scale per (token, head), 4 bf16 sink tokens, "
                 "values N(0,1) with 1% outliers at +-8",
    "quant_int4_g64": "32 sequences x 16,384 tokens in the pages' INT4 layout: groups of 64 along "
                      "the head dim (two fp16 scale/zero pairs per token and head, 36 B per 64 "
                      "elements), 8 bf16 sink tokens, 32 q / 8 KV heads, head dim 128, values "
                      "N(0,1) with 1% outliers at +-8",
    "quant_int4_bie": "the pages' full cache layout on 32 sequences x 16,384 tokens: INT4 groups "
                      "of 64 along the head dim, 8 bf16 sink tokens, and the last 128 tokens (whole "
                      "blocks) read from a 16-bit window ring, 32 q / 8 KV heads, head dim 128, "
                      "values N(0,1) with 1% outliers at +-8",
    "prefix_cow": "8 sequences forked from a shared 2,000-token prompt, each extended by a "
                  "seeded tail of 1..300 tokens, 32 q / 8 KV heads, head dim 128, bf16",
    "verify_b64_g5": "speculative verify on the 64-sequence Llama-3-8B-shaped layer: the target's "
                     "one pass over gamma + 1 = 6 tokens per sequence (the pages' gamma = 5), each "
                     "attending causally over its context (512..4096 tokens), 32/8/128 bf16",
    "prefill_chunk512": "one 512-token chunked-prefill slice per sequence (the pages' "
                        "--chunked-prefill-size 512) at positions 3,584..4,095 of 8 sequences, "
                        "causal, 32/8/128 bf16",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="llama3_8b_b64", choices=sorted(WORKLOADS))
    ap.add_argument("--partition-size", type=int, default=0,
                    help="tokens per split-K partition; 0 = the library's automatic choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool-blocks", type=int, default=0,
                    help="override the pool size (blocks); 0 keeps the workload's")
    ap.add_argument("--cpu-worker", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--clock-worker", nargs=3, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


# ----------------------------------------------------------------- helpers
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


def source_digest(sources):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kv_bytes_per_launch):
    """DRAM bytes per launch of the workload's decode kernel from the
    committed ncu summary, scaled to this launch; None if there is none or
    the kernel changed since."""
    if workload not in TRAFFIC:
        return None
    rel, sources = TRAFFIC[workload]
    p = os.path.join(ROOT, rel)
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != source_digest(sources):
        return None
    try:
        per_kv_byte = float(vals["dram_bytes_per_launch"]) / float(vals["kv_bytes_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None
    return per_kv_byte * kv_bytes_per_launch


# clock-event reason bits (nvml.h, nvmlClocksEventReason*)
CLOCK_REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
                 (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))


def clock_worker(device, period_s, out_path):
    """Sampling process: read-only NVML queries of the SM clock, power and
    active clock-event reasons every period_s until SIGTERM, one line each
    ("monotonic_s mhz watts reasons") to out_path; the first line is the
    device's maximum SM clock.  It runs in its own interpreter so the
    launching process's GIL never delays a sample."""
    import ctypes
    import signal
    stop = []
    signal.signal(signal.SIGTERM, lambda *_: stop.append(1))
    lib = ctypes.CDLL("libnvidia-ml.so.1")
    if lib.nvmlInit_v2() != 0:
        raise SystemExit("nvmlInit_v2 failed")
    h = ctypes.c_void_p()
    if not (device.startswith("GPU-") and lib.nvmlDeviceGetHandleByUUID(device.encode(), ctypes.byref(h)) == 0):
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(device) if device.isdigit() else 0),
                                             ctypes.byref(h)) != 0:
            raise SystemExit("no NVML handle")
    reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
        lib.nvmlDeviceGetCurrentClocksThrottleReasons
    mx, mhz, mw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
    lines = ["max %d" % mx.value]
    for _ in range(3):  # the first queries are the slow ones: before "ready"
        lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))
        reasons_fn(h, ctypes.byref(rs))
        lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
    with open(out_path + ".ready", "w") as f:
        f.write("1")
    n = 0
    while not stop:
        ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0
        reasons_fn(h, ctypes.byref(rs))
        if n % 8 == 0:  # power changes slowly: one read in eight
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
        n += 1
        if ok:
            lines.append("%.6f %d %.3f %d" % (time.monotonic(), mhz.value, mw.value / 1000.0, rs.value))
        if period_s >= 1e-3:
            time.sleep(period_s)
    with open(out_path, "w") as f:
        f.write("\n".join(lines) + "\n")


class ClockSampler:
    """SM clock, power and clock-event reasons during the timed region.

    A separate sampling process (``clock_worker``) reads NVML every
    ``period_s`` from before the warm-up until ``stop``; ``mark_start`` /
    ``mark_end`` bracket the timed region (CLOCK_MONOTONIC, shared by both
    processes) and the summary is taken over the samples inside it.  A
    20-step region lasts about 2 ms and NVML answers every few ms on some
    hosts: with fewer than MIN_SAMPLES inside, the summary takes the
    MIN_SAMPLES samples nearest to the region and says so (``basis``).
    Without NVML the summary says so and holds no samples."""

    MIN_SAMPLES = 5

    def __init__(self, device_index, period_s=0.0002):
        self.period = period_s
        self.t_start = self.t_end = None
        self.proc, self.error = None, None
        self.path = os.path.join("/tmp", "pkv_clocks_%d_%d.txt" % (os.getpid(), device_index))
        try:
            import torch
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self.device = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            self.device = str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen([sys.executable, os.path.abspath(__file__), "--clock-worker",
                                          self.device, str(self.period), self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.PIPE)
            t0 = time.monotonic()
            while not os.path.exists(self.path + ".ready"):  # NVML up before the warm-up
                if self.proc.poll() is not None or time.monotonic() - t0 > 20:
                    raise RuntimeError("clock sampler did not start")
                time.sleep(0.005)
        except Exception as e:
            self.error = str(e)
            self.proc = None

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def poll_until(self, event):
        """Kept for the launch loops' call: the sampling process samples on
        its own, so this only waits for the timed launches to finish."""
        event.synchronize()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "NVML sampler unavailable: %s" % self.error}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except Exception:
            self.proc.kill()
        samples, sm_max = [], None
        try:
            with open(self.path) as f:
                for line in f:
                    parts = line.split()
                    if parts and parts[0] == "max":
                        sm_max = float(parts[1]) or None
                    elif len(parts) == 4:
                        samples.append((float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3])))
        except OSError as e:
            self.error = str(e)
        for path in (self.path, self.path + ".ready"):
            if os.path.exists(path):
                os.unlink(path)
        lo = self.t_start if self.t_start is not None else -1e30
        hi = self.t_end if self.t_end is not None else 1e30
        inside = [x for x in samples if lo <= x[0] <= hi]
        basis = "the samples inside the timed region"
        used = inside
        if len(inside) < self.MIN_SAMPLES and samples:
            # a short timed region (20 steps last about 2 ms) may fall between
            # NVML reads: take the samples nearest to it, the warm-up steps
            # running before it and the per-call pass of the same steps after
            near = sorted(samples, key=lambda x: max(lo - x[0], x[0] - hi, 0.0))[:self.MIN_SAMPLES]
            gap = max(max(lo - x[0], x[0] - hi, 0.0) for x in near)
            used = near
            basis = ("%d samples inside the timed region; the %d nearest to it (within %.1f ms; the "
                     "same steps ran before and after it)" % (len(inside), len(near), gap * 1e3))
        reasons = sorted({n for x in used for bit, n in CLOCK_REASONS if x[3] & bit})
        return {"sm_mhz": statistics.median([x[1] for x in used]) if used else None,
                "sm_max_mhz": sm_max, "reasons": reasons, "samples": len(inside),
                "power_w_max": max((x[2] for x in used), default=None),
                "basis": basis,
                "samples_whole_run": len(samples),
                "sm_mhz_median_whole_run": statistics.median([x[1] for x in samples]) if samples else None,
                "source": "NVML read-only queries back to back (period %.1f ms or less) by a sampling "
                          "process, from before the warm-up until after the per-call pass that follows "
                          "the timed loop" % (self.period * 1e3)}


# ----------------------------------------------------------- device setup
class Cache:
    """A workload's paged cache, built with the library's own entry points
    (host block manager, KV-append / quantised append, copy-on-write copy)."""

    def __init__(self, pkv, torch, device, name, partition_size, headroom_tokens, pool_blocks=0):
        import synthetic as syn
        base, over, qmode = WORKLOADS[name]
        over = dict(over(syn) if callable(over) else over)
        if pool_blocks:
            over["num_blocks"] = pool_blocks
        w = syn.workload(base, **over)
        self.pkv, self.torch, self.dev, self.w, self.qmode, self.name = pkv, torch, device, w, qmode, name
        NB, BS, Hkv, D, Hq = w["num_blocks"], w["block_size"], w["hkv"], w["d"], w["hq"]
        dt = w["torch_dtype"]
        self.pool = pkv.pkv_pool_create(NB, BS, syn.free_order(w))
        ops, decoded = syn.prefill_schedule(w)
        self.seqs = np.array(decoded, dtype=np.int64)
        B = len(decoded)
        self.B = B
        self.n_sink = w.get("n_sink", 0)
        self.window = 0
        if qmode is None:
            self.k_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
            self.v_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
            self.pools = [self.k_pool, self.v_pool]
        else:
            cb = D // 2 if qmode == "int4" else D
            self.group_size = w.get("group_size", D) if qmode == "int4" else D
            ng = D // self.group_size
            u8, f16 = torch.uint8, torch.float16
            self.cache = {
                "k_codes": torch.empty((NB, Hkv, BS, cb), dtype=u8, device=device),
                "v_codes": torch.empty((NB, Hkv, BS, cb), dtype=u8, device=device),
                "k_scale": torch.empty((NB, Hkv, BS, ng), dtype=f16, device=device),
                "v_scale": torch.empty((NB, Hkv, BS, ng), dtype=f16, device=device),
                "sink_k": torch.zeros((B, max(self.n_sink, 1), Hkv, D), dtype=dt, device=device),
                "sink_v": torch.zeros((B, max(self.n_sink, 1), Hkv, D), dtype=dt, device=device),
            }
            if qmode == "int4":
                self.cache["k_zero"] = torch.empty((NB, Hkv, BS, ng), dtype=f16, device=device)
                self.cache["v_zero"] = torch.empty((NB, Hkv, BS, ng), dtype=f16, device=device)
            self.window = w.get("window", 0)
            if self.window:
                R = self.window // BS + 1
                self.cache["win_k"] = torch.zeros((B, R, Hkv, BS, D), dtype=dt, device=device)
                self.cache["win_v"] = torch.zeros((B, R, Hkv, BS, D), dtype=dt, device=device)
            self.pools = [self.cache[k] for k in ("k_codes", "k_scale", "k_zero", "v_codes",
                                                  "v_scale", "v_zero") if k in self.cache]
        row_of = {h: i for i, h in enumerate(decoded)}
        src = {}

        def rows(h, start, n):
            key = "prompt" if ("prompt" in w and h == 0) else (h - 1 if "prompt" in w else h)
            if key not in src:
                src[key] = syn.prompt_kv(w) if key == "prompt" else syn.sequence_kv(w, key)
            k, v = src[key]
            return k[start:start + n], v[start:start + n]

        lens = {}
        for op in ops:
            if op[0] == "create":
                pkv.pkv_seq_create(self.pool)
            elif op[0] == "fork":
                child = pkv.pkv_seq_fork(self.pool, op[1])
                lens[child] = lens.get(op[1], 0)
            else:
                _, h, n = op
                start = lens.get(h, 0)
                slots, pairs = pkv.pkv_seq_append(self.pool, h, n)
                if pairs:
                    pkv.pkv_copy_blocks(self.pools, torch.tensor(pairs, dtype=torch.int32, device=device))
                k, v = rows(h, start, n)
                self._append(k.to(device), v.to(device), torch.from_numpy(slots).to(device),
                             np.arange(start, start + n), row_of.get(h, 0))
                lens[h] = start + n
        if qmode is not None and "prompt" in w:
            kp, vp = rows(0, 0, self.n_sink)
            for r in range(B):
                self.cache["sink_k"][r, :self.n_sink] = kp.to(device)
                self.cache["sink_v"][r, :self.n_sink] = vp.to(device)
        # the decode step's append: token L-1 of every sequence
        slots, pairs = pkv.pkv_seq_append_batch(self.pool, self.seqs, 1)
        if len(pairs):
            pkv.pkv_copy_blocks(self.pools, torch.from_numpy(np.ascontiguousarray(pairs)).to(device))
        nk, nv = [], []
        for h in decoded:
            k, v = rows(h, lens[h], 1)
            nk.append(k[0])
            nv.append(v[0])
        self.new_k = torch.stack(nk).to(device)
        self.new_v = torch.stack(nv).to(device)
        self.slots = torch.from_numpy(slots.copy()).to(device)
        self.positions = torch.tensor([lens[h] for h in decoded], dtype=torch.int32, device=device)
        self.seq_idx = torch.arange(B, dtype=torch.int32, device=device)
        ctx_list = syn.context_lengths(w)
        self.max_blocks = -(-max(ctx_list) // BS)  # exact: the timed decode reads these tables
        self.max_blocks_grown = -(-(max(ctx_list) + headroom_tokens) // BS)  # for the e2e loop
        tables, ctx = pkv.pkv_build_block_tables(self.pool, self.seqs, self.max_blocks)
        self.tables = torch.from_numpy(tables.copy()).to(device)
        self.lens = torch.from_numpy(ctx.copy()).to(device)
        self.ctx_host = ctx.copy()
        self.unique_blocks = len(set(int(x) for x in tables.ravel() if x >= 0))
        self.q = syn.query(w).to(device)
        self.out = torch.empty((B, Hq, D), dtype=dt, device=device)
        # 0 = the library's automatic split: balanced over the GPU's warps for
        # the 16-bit cache, automatic partitions for the quantised one
        self.partition_size = partition_size
        auto_ps = pkv.pkv_decode_auto_partition_size(B, Hq, self.max_blocks, BS)
        self.split = self.max_blocks * BS > (partition_size or auto_ps)
        if not self.split:
            self.split_desc = "single pass (one partition covers every context)"
        elif partition_size == 0 and qmode is None and B <= 1024:
            self.split_desc = ("balanced split-K: every warp of 4 resident 4-warp CTAs per SM "
                               "streams an equal share of the (sequence, KV head, 16-token unit) items")
        else:
            self.split_desc = "%d-token split-K partitions" % (partition_size or auto_ps)
        ws = pkv.pkv_decode_workspace_bytes(B, Hq, D, self.max_blocks, BS, self.partition_size)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def _append(self, k, v, slots, positions, seq_row):
        if self.qmode is None:
            self.pkv.pkv_kv_append(k, v, slots, self.k_pool, self.v_pool)
            return
        torch = self.torch
        if not torch.is_tensor(positions):
            positions = torch.from_numpy(np.asarray(positions, dtype=np.int32)).to(self.dev)
        sidx = torch.full((k.shape[0],), seq_row, dtype=torch.int32, device=self.dev)
        self.pkv.pkv_kv_append_quant(k, v, slots, positions, sidx, self.cache, self.n_sink,
                                     self.qmode, self.group_size, window=self.window)

    def bytes_per_token(self):
        Hkv, D = self.w["hkv"], self.w["d"]
        if self.qmode == "int4":
            return 2 * Hkv * (D // 2 + 4 * (D // self.group_size))
        if self.qmode == "fp8":
            return 2 * Hkv * (D + 2)
        return 2 * Hkv * D * 2

    def kv_bytes(self, ctx=None):
        """Algorithmic KV bytes one decode reads (sinks read in 16-bit)."""
        ctx = self.ctx_host if ctx is None else ctx
        total = int(np.sum(ctx)) * self.bytes_per_token()
        if self.qmode is not None:
            # sink and window tokens are read in 16-bit, not as codes; the window
            # is the last `window` tokens rounded down to a block boundary
            w16 = np.array([c - max(int(c) - self.window, 0) // 16 * 16 if self.window else 0
                            for c in ctx])
            sinks = np.minimum(ctx, self.n_sink)
            if self.window:
                ws = ctx - w16
                sinks = np.minimum(sinks, ws)  # sinks inside the window are read once
                total -= int(np.sum(w16)) * self.bytes_per_token()
                total += int(np.sum(w16)) * 2 * self.w["hkv"] * self.w["d"] * 2
            total += int(np.sum(sinks)) * 2 * self.w["hkv"] * self.w["d"] * 2
        return total

    def step(self, q=None, k_new=None, v_new=None, slots=None, tables=None, lens=None, out=None,
             ws=None, positions=None, stream=None):
        """One decode step: append each sequence's new row, then attend."""
        pkv = self.pkv
        q = self.q if q is None else q
        k_new = self.new_k if k_new is None else k_new
        v_new = self.new_v if v_new is None else v_new
        slots = self.slots if slots is None else slots
        tables = self.tables if tables is None else tables
        lens = self.lens if lens is None else lens
        out = self.out if out is None else out
        ws = self.ws if ws is None else ws
        if self.qmode is None:
            pkv.pkv_paged_attention_decode_append(q, k_new, v_new, slots, self.k_pool, self.v_pool,
                                                  tables, lens, self.w["scale"], out, ws,
                                                  self.partition_size, stream)
            return
        positions = self.positions if positions is None else positions
        pkv.pkv_kv_append_quant(k_new, v_new, slots, positions, self.seq_idx, self.cache,
                                self.n_sink, self.qmode, self.group_size, stream, window=self.window)
        pkv.pkv_paged_attention_decode_quant(q, self.cache, self.n_sink, tables, lens,
                                             self.w["scale"], out, self.qmode, self.group_size, ws,
                                             self.partition_size, stream, window=self.window)

    def launches_per_step(self):
        return (2 if self.split else 1) + (1 if self.qmode else 0)


def per_call_ms(torch, step, stream, steps):
    """Mean device time of one call, each bracketed by its own CUDA events on
    the launching stream.  A separate pass after the timed loop, which has
    nothing on the stream between consecutive steps (the event pairs add
    about 2 us per step on the 64-sequence layer)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def run_device(args, rank, world, dist):
    import torch
    import paged_kv_cache_13_gb300 as pkv

    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    device = torch.device("cuda", dev_index)
    e2e_steps = max(E2E_MIN_STEPS, args.steps)
    cache = Cache(pkv, torch, device, args.workload, args.partition_size,
                  headroom_tokens=e2e_steps + 8, pool_blocks=args.pool_blocks)
    stream = torch.cuda.current_stream()
    kv_bytes = cache.kv_bytes()

    # ---------- device-resident timed region
    clocks = ClockSampler(dev_index)
    clocks.start()
    for _ in range(args.warmup):
        cache.step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    # the steps back to back, as a serving loop issues them (nothing between
    # consecutive steps on the stream)
    t0.record(stream)
    for i in range(args.steps):
        cache.step()
    t1.record(stream)
    clocks.poll_until(t1)
    torch.cuda.synchronize()
    clocks.mark_end()
    # the same steps again, each timed alone, while the sampler still runs
    call_ms = per_call_ms(torch, cache.step, stream, args.steps)
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    assert pkv.pkv_device_status() == 0
    elapsed_ms = max_over_ranks(elapsed_ms, dist, device)
    ms_per_step = elapsed_ms / args.steps

    # ---------- end to end through the public API, host buffers
    # the e2e loop appends a token per sequence per step: as many steps as
    # the pool has blocks for (the quantised workloads fill most of theirs)
    free = pkv.pkv_pool_num_free(cache.pool)
    e2e_steps = max(16, min(e2e_steps, (free // max(cache.B, 1) - 1) * 16))
    e2e = run_e2e(pkv, torch, cache, e2e_steps, dist, device)
    prefix = prefix_cache_timing(pkv, cache) if "prompt" in cache.w else None
    append = append_timing(pkv, torch, cache)

    return dict(ms_per_step=ms_per_step, call_ms=call_ms, kv_bytes=kv_bytes, clocks=clk, e2e=e2e,
                prefix=prefix, append=append,
                B=cache.B, launches=cache.launches_per_step() * args.steps,
                unique_blocks=cache.unique_blocks, partition_size=cache.partition_size,
                split_desc=cache.split_desc)


def append_timing(pkv, torch, cache, iters=200):
    """The decode step's KV-append alone (the step itself fuses it into the
    decode for the 16-bit cache): the step's B new K/V rows written to their
    slots.  The calls are tiny, so back-to-back launches from Python would
    time the host; `iters` calls are captured in one CUDA graph and its
    replay is timed with CUDA events (after a warm-up replay)."""
    def one():
        if cache.qmode is None:
            pkv.pkv_kv_append(cache.new_k, cache.new_v, cache.slots, cache.k_pool, cache.v_pool)
        else:
            pkv.pkv_kv_append_quant(cache.new_k, cache.new_v, cache.slots, cache.positions, cache.seq_idx,
                                    cache.cache, cache.n_sink, cache.qmode, cache.group_size,
                                    window=cache.window)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            one()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(iters):
            one()
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / iters
    row_bytes = cache.w["hkv"] * cache.w["d"] * 2 * 2  # K and V rows in, 16-bit
    return {"kernel": "kv_append_kernel" if cache.qmode is None else "kv_append_quant_kernel",
            "rows": cache.B, "us_per_call": round(us, 2), "input_bytes": cache.B * row_bytes,
            "timing": "%d calls in one CUDA graph replay, CUDA events" % iters,
            "note": "timed alone; the 16-bit step fuses it into the decode kernel"
            if cache.qmode is None else "timed alone; part of each quantised step"}


def mq_kernel_name(balanced, D, G, L):
    """The kernel(s) pkv_paged_attention_multi_query runs for L queries per
    sequence: the balanced split (when a workspace is given and it applies),
    else the tcgen05 kernel for long spans at head dim 128 (more than 64
    (token, head) rows per (sequence, KV head)), else the one-pass tiles."""
    if balanced:
        return "multi_query_balanced_kernel<bf16, %d, %d> + multi_query_merge_kernel" % (D, -(-L * G // 8))
    if D == 128 and G in (1, 2, 4, 8) and L * G > 64:
        return "prefill_tc_kernel<bf16> (tcgen05 + TMA)"
    return "multi_query_kernel<bf16, %d, %d> (mma.sync)" % (D, 1 if L * G <= 8 else 2)


def run_mq(args, rank, world, dist):
    """Multi-query workloads: every step rewrites the L new tokens' K/V rows
    of every sequence (pkv_kv_append) and runs pkv_paged_attention_multi_query
    with L queries per sequence at the last L positions of its context."""
    import torch
    import paged_kv_cache_13_gb300 as pkv
    import synthetic as syn

    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    device = torch.device("cuda", dev_index)
    name, L = args.workload, MQ_LEN[args.workload]
    cache = Cache(pkv, torch, device, name, 0, 8)
    w, B = cache.w, cache.B
    Hq, Hkv, D = w["hq"], w["hkv"], w["d"]
    # the pool holds every context token
    pkv.pkv_kv_append(cache.new_k, cache.new_v, cache.slots, cache.k_pool, cache.v_pool)
    tables = cache.tables.cpu().numpy()
    ctx = cache.ctx_host
    ks, vs, slots = [], [], []
    for b in range(B):
        k, v = syn.sequence_kv(w, b)
        lo = int(ctx[b]) - L
        ks.append(k[lo:])
        vs.append(v[lo:])
        for pos in range(lo, int(ctx[b])):
            slots.append(int(tables[b, pos // 16]) * 16 + pos % 16)
    mq_k = torch.cat(ks).to(device)
    mq_v = torch.cat(vs).to(device)
    mq_slots = torch.tensor(slots, dtype=torch.int64, device=device)
    rng = np.random.default_rng(np.random.SeedSequence([w["seed"], 77]))
    q = torch.from_numpy(rng.standard_normal((B * L, Hq, D), dtype=np.float32)).to(w["torch_dtype"]).to(device)
    q_start = torch.arange(0, B * L + 1, L, dtype=torch.int32, device=device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    # the balanced split where it applies (a workspace of the size it asks for)
    ws_n = pkv.pkv_multi_query_workspace_bytes(B, Hq, Hkv, D, cache.max_blocks, L)
    mq_ws = torch.empty(ws_n, dtype=torch.uint8, device=device) if ws_n else None
    mq_kernels = mq_kernel_name(bool(ws_n), D, Hq // Hkv, L)

    def step(qq=q, oo=out):
        pkv.pkv_kv_append(mq_k, mq_v, mq_slots, cache.k_pool, cache.v_pool)
        pkv.pkv_paged_attention_multi_query(qq, q_start, cache.k_pool, cache.v_pool, cache.tables,
                                            cache.lens, w["scale"], oo, L, workspace=mq_ws)

    clocks = ClockSampler(dev_index)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    clocks.poll_until(t1)
    torch.cuda.synchronize()
    clocks.mark_end()
    call_ms = per_call_ms(torch, step, stream, args.steps)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), dist, device)
    ms = elapsed_ms / args.steps
    assert pkv.pkv_device_status() == 0

    # end to end: q from pinned host memory, out back to pinned host memory
    e2e_steps = max(E2E_MIN_STEPS, args.steps)
    hq_ = q.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dq = torch.empty_like(q)
    torch.cuda.synchronize()
    te = time.perf_counter()
    for _ in range(e2e_steps):
        dq.copy_(hq_, non_blocking=True)
        step(dq, out)
        ho.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - te, dist, device) / e2e_steps

    kv_bytes = cache.kv_bytes()
    positions = [int(ctx[b]) - L + i for b in range(B) for i in range(L)]
    flops = sum(4.0 * (p + 1) * D * Hq for p in positions)  # QK^T and PV, causal
    qo_bytes = 2 * q.numel() * q.element_size()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    tflops_peak = float(peaks.get("bf16_tflops", 1900.0))
    cfg = {"workload": "%s: %s; step = pkv_kv_append of the %d new rows per sequence + "
                       "pkv_paged_attention_multi_query" % (name, DESCRIPTIONS[name], L),
           "batch": B, "query_tokens_per_sequence": L, "kv_bytes_per_step": kv_bytes,
           "causal_flops_per_step": flops,
           "l2": "inputs larger than L2 (%.0f MB of KV per step), no flush" % (kv_bytes / 1e6)
           if kv_bytes > 129e6 else "KV working set %.0f MB fits the 129 MB L2" % (kv_bytes / 1e6)}
    common = {"n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
              "data": "synthetic", "config": cfg, "gpu_launches": (3 if ws_n else 2) * args.steps, "clocks": clk,
              "queries_per_s": round(B * L * world / (ms * 1e-3), 1), "cpu_baseline": None}
    if name == "prefill_chunk512":
        value = flops * world / (ms * 1e-3) / 1e12
        achieved = flops / (call_ms * 1e-3) / 1e12
        line = dict(metric="chunked-prefill attention TFLOP/s (causal QK^T + PV FLOPs)",
                    value=round(value, 2), unit="TFLOP/s", **common)
        line["roofline"] = {"bound": "tensor", "kernel": mq_kernels,
                            "achieved": round(achieved, 2), "peak": tflops_peak, "unit": "TFLOP/s",
                            "peak_kind": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS, burst)",
                            "frac": round(achieved / tflops_peak, 4), "traffic": None,
                            "algorithmic_flops_per_launch": flops, "avg_launch_ms": call_ms}
        line["e2e"] = {"value": round(flops * world / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2}
    else:
        value = kv_bytes * world / (ms * 1e-3) / 1e9
        achieved = kv_bytes / (call_ms * 1e-3) / 1e9
        line = dict(metric=METRIC, value=round(value, 1), unit="GB/s", **common)
        line["roofline"] = {"bound": "hbm", "kernel": mq_kernels,
                            "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                            "peak_kind": "measured (MEASURED_PEAKS.json hbm_gbs, copy, burst)",
                            "frac": round(achieved / hbm, 4), "traffic": None,
                            "algorithmic_bytes_per_launch": kv_bytes + qo_bytes, "avg_launch_ms": call_ms}
        line["e2e"] = {"value": round(kv_bytes * world / e2e_s / 1e9, 1), "unit": "GB/s",
                       "h2d_bytes_per_step": q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2}
    return line


def prefix_cache_timing(pkv, cache, iters=2000):
    """Host prefix cache on the prefix workload's pool: the prompt holder's
    blocks are registered under seeded token ids, then each iteration maps a
    new request (the prompt plus 64 tokens of its own) onto them and releases
    it -- the lookup a request pays before its prefill.  The cache is cleared
    afterwards, so the decode state is unchanged."""
    w = cache.w
    tokens = np.random.default_rng(np.random.SeedSequence([w["seed"], 99])).integers(
        0, 128256, size=w["prompt"] + 64).astype(np.int32)
    holder = 0  # the prompt's own sequence (created first)
    t0 = time.perf_counter()
    entries = pkv.pkv_prefix_register(cache.pool, holder, tokens[:w["prompt"]])
    reg_us = (time.perf_counter() - t0) * 1e6
    matched = 0
    t0 = time.perf_counter()
    for _ in range(iters):
        seq, matched = pkv.pkv_prefix_match(cache.pool, tokens)
        pkv.pkv_seq_free(cache.pool, seq)
    match_us = (time.perf_counter() - t0) * 1e6 / iters
    pkv.pkv_prefix_clear(cache.pool)
    return {"register_us": round(reg_us, 2), "match_and_release_us": round(match_us, 2),
            "prompt_tokens": int(w["prompt"]), "request_tokens": int(tokens.shape[0]),
            "matched_tokens": int(matched), "entries": int(entries), "iterations": iters,
            "note": "host C++ through the C ABI (ctypes call overhead included), one thread"}


def run_e2e(pkv, torch, cache, steps, dist, device):
    """End to end through the public API with host buffers, pipelined the way
    a serving loop would run it.  Each step's q and new K/V rows arrive in a
    pinned host buffer.  Every step: the host block manager appends one token
    per sequence and writes the slots, CoW pairs, tables and lengths into the
    same buffer; the whole buffer goes to the device in one H2D on a copy
    stream; the decode step runs on the compute stream; the output comes back
    in one D2H.  Device slots are double-buffered and ordered by events, so
    the CPU work and copies of step s+1 overlap the decode of step s."""
    import synthetic as syn
    w = cache.w
    B, Hq, Hkv, D = cache.B, w["hq"], w["hkv"], w["d"]
    dt = w["torch_dtype"]
    mb = cache.max_blocks_grown
    esz = torch.tensor([], dtype=dt).element_size()

    # packed layout of one step's inputs (256-byte aligned fields)
    fields = [("q", B * Hq * D * esz), ("k", B * Hkv * D * esz), ("v", B * Hkv * D * esz),
              ("slots", B * 8), ("pairs", 2 * B * 4), ("tab", B * mb * 4), ("lens", B * 4),
              ("pos", B * 4)]
    off, layout = 0, {}
    for name, nbytes in fields:
        layout[name] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    in_bytes = off

    def views(buf):
        def v(name, dtype, shape):
            o, n = layout[name]
            return buf[o:o + n].view(dtype).view(shape)
        return {"q": v("q", dt, (B, Hq, D)), "k": v("k", dt, (B, Hkv, D)), "v": v("v", dt, (B, Hkv, D)),
                "slots": v("slots", torch.int64, (B,)), "pairs": v("pairs", torch.int32, (B, 2)),
                "tab": v("tab", torch.int32, (B, mb)), "lens": v("lens", torch.int32, (B,)),
                "pos": v("pos", torch.int32, (B,))}

    # each step's q and new K/V rows arrive in pinned host memory, a ring of
    # R buffers an upstream producer fills ahead (staged before the timed
    # region); the timed loop adds the block manager's slots, pairs and
    # tables to buffer s % R once that buffer's previous copy has finished
    R = min(steps, E2E_RING)
    h_in = [torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True) for _ in range(R)]
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    h_out = [torch.empty((B, Hq, D), dtype=dt, pin_memory=True) for _ in range(2)]
    d_out = [torch.empty((B, Hq, D), dtype=dt, device=device) for _ in range(2)]
    hv = [views(b) for b in h_in]
    dv = [views(b) for b in d_in]
    ws = torch.empty(max(16, pkv.pkv_decode_workspace_bytes(B, Hq, D, mb, 16, cache.partition_size)),
                     dtype=torch.uint8, device=device)
    q16 = syn.query(w)
    for s in range(R):
        k, v = syn.new_token_kv(w, s)
        hv[s]["q"].copy_(q16)
        hv[s]["k"].copy_(k)
        hv[s]["v"].copy_(v)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()
    e_h2d = [None] * steps
    e_dec = [None] * steps
    e_d2h = [None] * steps
    total_kv = 0
    h2d = in_bytes
    d2h = h_out[0].numel() * esz
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    for s in range(steps):
        j = s % 2
        h = hv[s % R]
        if s >= R:
            e_h2d[s - R].synchronize()  # the ring buffer's previous copy is done
        _, pairs = pkv.pkv_seq_append_batch(cache.pool, cache.seqs, 1, h["slots"].numpy(),
                                            h["pairs"].view(-1).numpy())
        pkv.pkv_build_block_tables(cache.pool, cache.seqs, mb, h["tab"].numpy(), h["lens"].numpy())
        lens = h["lens"].numpy()
        total_kv += cache.kv_bytes(lens)
        if cache.qmode:
            np.subtract(lens, 1, out=h["pos"].numpy())
        with torch.cuda.stream(copy):
            if s >= 2:
                copy.wait_event(e_dec[s - 2])  # decode s-2 no longer reads this device slot
            d_in[j].copy_(h_in[s % R], non_blocking=True)
            e_h2d[s] = ev()
            e_h2d[s].record(copy)
        compute.wait_event(e_h2d[s])
        if s >= 2:
            compute.wait_event(e_d2h[s - 2])  # output slot copied out
        d = dv[j]
        if len(pairs):
            pkv.pkv_copy_blocks(cache.pools, d["pairs"][:len(pairs)], compute)
        cache.step(q=d["q"], k_new=d["k"], v_new=d["v"], slots=d["slots"], tables=d["tab"],
                   lens=d["lens"], out=d_out[j], ws=ws, positions=d["pos"], stream=compute)
        e_dec[s] = ev()
        e_dec[s].record(compute)
        with torch.cuda.stream(copy):
            copy.wait_event(e_dec[s])
            h_out[j].copy_(d_out[j], non_blocking=True)
            e_d2h[s] = ev()
            e_d2h[s].record(copy)
    torch.cuda.synchronize()
    elapsed = max_over_ranks(time.perf_counter() - t_start, dist, device)
    assert all(torch.isfinite(o.float()).all() for o in h_out)
    return dict(gbs=total_kv / elapsed / 1e9, h2d=h2d, d2h=d2h, steps=steps)


# -------------------------------------------------------------- CPU oracle
def oracle_sample(name, S):
    """The first S decoded sequences of a workload as an oracle-side paged
    cache.  Returns (decode(), kv bytes per decode, S, tokens)."""
    import synthetic as syn
    from oracle import allocator, attention, kvcache
    base, over, qmode = WORKLOADS[name]
    w = syn.workload(base, **(over(syn) if callable(over) else over))
    S = min(S, len(syn.context_lengths(w)))
    q = syn.kv_rows_to_numpy(syn.query(w))[:S]
    ks, vs = [], []
    for i in range(S):
        k, v = syn.sequence_kv(w, i)
        ks.append(syn.kv_rows_to_numpy(k))
        vs.append(syn.kv_rows_to_numpy(v))
    bs = w["block_size"] if qmode is None else 16
    nb = sum(-(-k.shape[0] // bs) for k in ks)
    m = allocator.KVCacheManager(nb, bs, syn.free_order(dict(w, num_blocks=nb)))
    Hkv, D = w["hkv"], w["d"]
    sids, all_slots = [], []
    for i in range(S):
        s = m.create()
        slots, _ = m.append(s, ks[i].shape[0])
        sids.append(s)
        all_slots.append(slots)
    tables, ctx = m.block_tables(sids, max(len(m.table(s)) for s in sids))
    if qmode is None:
        kp = np.zeros((nb, Hkv, bs, D), np.float32)
        vp = np.zeros_like(kp)
        for i in range(S):
            kvcache.kv_append(ks[i], vs[i], all_slots[i], kp, vp, block_size=bs)

        def decode():
            attention.paged_attention_decode(q, kp, vp, tables, ctx, w["scale"], block_size=bs)
        kvb = int(np.sum(ctx)) * 2 * Hkv * D * 2
    else:
        ns = w["n_sink"]
        cb = D // 2 if qmode == "int4" else D
        gsz = w.get("group_size", D) if qmode == "int4" else D
        ng = D // gsz
        cache = {"k_codes": np.zeros((nb, Hkv, 16, cb), np.uint8),
                 "v_codes": np.zeros((nb, Hkv, 16, cb), np.uint8),
                 "k_scale": np.zeros((nb, Hkv, 16, ng), np.float16),
                 "v_scale": np.zeros((nb, Hkv, 16, ng), np.float16),
                 "k_zero": np.zeros((nb, Hkv, 16, ng), np.float16),
                 "v_zero": np.zeros((nb, Hkv, 16, ng), np.float16),
                 "sink_k": np.zeros((S, ns, Hkv, D)), "sink_v": np.zeros((S, ns, Hkv, D))}
        for i in range(S):
            # the oracle's vectorised quantiser, written at the slots
            _, kc, ksc, kz = kvcache.quantize_sequence(ks[i], qmode, gsz)
            _, vc, vsc, vz = kvcache.quantize_sequence(vs[i], qmode, gsz)
            for t, slot in enumerate(all_slots[i]):
                blk, off = divmod(int(slot), 16)
                cache["k_codes"][blk, :, off] = kc[t]
                cache["v_codes"][blk, :, off] = vc[t]
                cache["k_scale"][blk, :, off] = ksc[t]
                cache["v_scale"][blk, :, off] = vsc[t]
                if kz is not None:
                    cache["k_zero"][blk, :, off] = kz[t]
                    cache["v_zero"][blk, :, off] = vz[t]
            cache["sink_k"][i] = ks[i][:ns]
            cache["sink_v"][i] = vs[i][:ns]
        win = w.get("window", 0)
        if win:
            R = kvcache.ring_blocks(win)
            cache["win_k"] = np.zeros((S, R, Hkv, 16, D))
            cache["win_v"] = np.zeros((S, R, Hkv, 16, D))
            for i in range(S):
                for t in range(kvcache.window_start(ks[i].shape[0], win), ks[i].shape[0]):
                    cache["win_k"][i, (t // 16) % R, :, t % 16] = ks[i][t]
                    cache["win_v"][i, (t // 16) % R, :, t % 16] = vs[i][t]

        def decode():
            kvcache.paged_attention_decode_quant(q, cache, tables, ctx, w["scale"], ns, qmode, gsz,
                                                 window=win)
        per_tok = 2 * Hkv * (D // 2 + 4 * ng) if qmode == "int4" else 2 * Hkv * (D + 2)
        w16 = np.array([c - kvcache.window_start(int(c), win) if win else 0 for c in ctx])
        sinks = np.minimum(np.minimum(ctx, ns), ctx - w16)
        kvb = (int(np.sum(ctx - w16)) * per_tok + int(np.sum(w16)) * 2 * Hkv * D * 2
               + int(np.sum(sinks)) * 2 * Hkv * D * 2)
    return decode, kvb, S, int(np.sum(ctx))


def cpu_worker(name, min_seconds, S):
    decode, kvb, S, toks = oracle_sample(name, S)
    reps, t0 = 0, time.perf_counter()
    while True:
        decode()
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "reps": reps, "kv_bytes": kvb * reps, "seqs": S * reps,
                      "sample_seqs": S, "sample_tokens": toks}))


CPU_SAMPLE_SEQS = {"llama3_8b_b64": 16, "llama3_8b_b64_bs8": 16, "llama3_8b_b64_bs32": 16,
                   "llama3_8b_b64_in_order": 16, "llama3_8b_b64_slab": 128, "long_splitk": 1, "quant_int4": 1, "quant_fp8": 1,
                   "quant_int4_g64": 1, "quant_int4_bie": 1, "prefix_cow": 8}


def cpu_baseline(name, min_seconds):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(min_seconds),
                        "--workload", name], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        return None
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return {
        "value": res["kv_bytes"] / res["seconds"] / 1e9,
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": "float64 NumPy oracle paged decode of %d sequence(s) of the workload (%d tokens, "
                  "all query heads), repeated %d times in %.1f s, single thread"
                  % (res["sample_seqs"], res["sample_tokens"], res["reps"], res["seconds"]),
        "seq_per_s": res["seqs"] / res["seconds"],
    }


def config_block(name, B, kv_bytes, partition_size, split_desc):
    step = ("quantised KV-append of 1 token per sequence + paged decode over the quantised "
            "cache (split-K partials, merge kernel)" if WORKLOADS[name][2] else
            "KV-append of 1 token per sequence fused into the paged decode (split-K "
            "partials, then a merge kernel with programmatic dependent launch)")
    return {
        "workload": "%s: %s; step = %s; %s" % (name, DESCRIPTIONS[name], step, split_desc),
        "batch": B,
        "kv_bytes_per_step": kv_bytes,
        "partition_size": partition_size or "auto",
        "l2": ("inputs larger than L2 (%.0f MB of KV read per step vs 129 MB L2), no flush"
               % (kv_bytes / 1e6)) if kv_bytes > 129e6 else
              ("KV working set %.0f MB fits the 129 MB L2: numbers are L2-resident"
               % (kv_bytes / 1e6)),
    }


def main():
    args = parse_args()
    if args.clock_worker is not None:
        clock_worker(args.clock_worker[0], float(args.clock_worker[1]), args.clock_worker[2])
        return
    if args.cpu_worker is not None:
        cpu_worker(args.workload, args.cpu_worker, CPU_SAMPLE_SEQS[args.workload])
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
    if args.workload in MQ_LEN:
        line = run_mq(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(line))
        return
    res = run_device(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return
    value = whole_job_rate(res["kv_bytes"], world, res["ms_per_step"] * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = res["kv_bytes"] / (res["call_ms"] * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(args.workload, 10.0)
    quant = WORKLOADS[args.workload][2]
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
        "dtype": "bf16" if not quant else ("bf16 q, u4 KV codes" if quant == "int4" else "bf16 q, e4m3 KV codes"),
        "data": "synthetic",
        "config": config_block(args.workload, res["B"], res["kv_bytes"], res["partition_size"],
                               res["split_desc"]),
        "seq_per_s_per_layer": round(res["B"] / ROWS_PER_SEQ.get(args.workload, 1) * world
                                     / (res["ms_per_step"] * 1e-3), 1),
        "pct_of_8tbs_nominal": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100.0 * value / world / peak, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": ("kv_append_quant + paged_decode_quant_kernel + merge_kernel" if quant else
                       "paged_decode_balanced_kernel<bf16, 128, fused append> + merge_balanced_kernel"
                       if "balanced" in res["split_desc"] else
                       "paged_decode_kernel<bf16, 128, partials, fused append> + merge_kernel"),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": ("measured (MEASURED_PEAKS.json hbm_gbs, copy, burst)"
                          if peak_kind == "measured" else "fallback"),
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(args.workload, res["kv_bytes"]),
            "algorithmic_bytes_per_launch": res["kv_bytes"],
            "avg_launch_ms": res["call_ms"],
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
    if args.workload == "prefix_cow":
        line["unique_kv_bytes_per_step"] = res["unique_blocks"] * 16 * KV_BYTES_PER_TOKEN
    if res.get("prefix"):
        line["prefix_cache"] = res["prefix"]
    if res.get("append"):
        line["append"] = res["append"]
    print(json.dumps(line))


def run_reference(args, world):
    """The oracle, as it stands, on the host cores: each step is the oracle's
    paged decode of a bounded sample (2 sequences of the workload, all heads)."""
    decode, kvb, S, toks = oracle_sample(args.workload, 2 if args.workload != "long_splitk" else 1)
    for _ in range(args.warmup):
        decode()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        decode()
    dt = time.perf_counter() - t0
    value = kvb * args.steps / dt / 1e9
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
        "config": config_block(args.workload, S, kvb, args.partition_size,
                               "the oracle has no split: plain softmax per (sequence, query head)"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": cores,
                         "sample": "float64 NumPy oracle paged decode of %d sequence(s) of the "
                                   "workload (%d tokens, all query heads) per step" % (S, toks)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
