"""Workload definitions and seeded generators.

Five workloads, shaped like the pages' setting (an 8B GQA model: 32 query
heads, 8 KV heads, head dim 128, blocks of 16 tokens -- "The 8GB VRAM
Breakthrough", §2 and §3):

``tiny``             3 sequences of 25, 47 and 12 tokens (the worked example
                     of "PagedAttention aplica memória virtual ao cache KV de
                     LLMs"), pool of 64 blocks in seeded random order,
                     8 query / 2 KV heads, head dim 64, fp16, scale 1/8.
``llama3_8b_b64``    one Llama-3-8B-shaped layer: 64 sequences, lengths
                     uniform in [512, 4096], 32/8 heads, dim 128, bf16,
                     40,000-block pool in seeded random order.
``long_splitk``      4 sequences of 65,536 / 32,768 / 32,768 / 32,768 tokens,
                     blocks handed out round-robin across the sequences from
                     a shuffled pool (randomly interleaved), bf16, 32/8/128.
``quant``            32 sequences of 16,384 tokens, 32/8/128, bf16 inputs,
                     N(0,1) values with 1% replaced by +-8, 4 sink tokens,
                     INT4 (group = head dim) or FP8 E4M3 cache.
``prefix_cow``       a 2,000-token prompt forked 8 times, each child extended
                     by a seeded tail of 1..300 tokens; ``prefix_cow_2008``
                     is the same with a 2,008-token prompt so that the shared
                     tail block is partially filled at the fork.

Every length counts the token appended by the decode step: a sequence of
length L is prefilled with L-1 tokens, then one decode step appends one token
per sequence and attends over all L.

Random values come from NumPy's PCG64 streams (platform-independent bit
streams), drawn as float32 N(0,1) and rounded to the 16-bit dtype with
round-to-nearest-even.  Each sequence has its own stream, so any one of them
can be regenerated alone.
"""

import math

import numpy as np
import torch

__all__ = [
    "WORKLOADS", "workload", "context_lengths", "free_order", "query",
    "sequence_kv", "prompt_kv", "new_token_kv", "prefill_schedule", "tails",
    "kv_rows_to_numpy",
]

WORKLOADS = {
    "tiny": dict(seed=1, lens=[25, 47, 12], num_blocks=64, hq=8, hkv=2, d=64,
                 dtype="fp16", block_size=16, scale=1.0 / 8.0),
    "llama3_8b_b64": dict(seed=2, batch=64, len_lo=512, len_hi=4096, num_blocks=40000,
                          hq=32, hkv=8, d=128, dtype="bf16", block_size=16),
    "long_splitk": dict(seed=3, lens=[65536, 32768, 32768, 32768], num_blocks=12288,
                        hq=32, hkv=8, d=128, dtype="bf16", block_size=16,
                        partition_size=512, interleave=True),
    "quant": dict(seed=4, batch=32, ctx=16384, num_blocks=40000, hq=32, hkv=8, d=128,
                  dtype="bf16", block_size=16, n_sink=4, group_size=128,
                  outlier_frac=0.01, outlier_mag=8.0),
    "prefix_cow": dict(seed=5, prompt=2000, n_fork=8, tail_lo=1, tail_hi=300,
                       num_blocks=4096, hq=32, hkv=8, d=128, dtype="bf16", block_size=16),
    "prefix_cow_2008": dict(seed=5, prompt=2008, n_fork=8, tail_lo=1, tail_hi=300,
                            num_blocks=4096, hq=32, hkv=8, d=128, dtype="bf16", block_size=16),
}

_TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}

# stream ids within one workload seed
_S_LENS, _S_FREE, _S_Q, _S_KV, _S_PROMPT, _S_TAILS, _S_NEW = range(7)


def workload(name, **overrides):
    w = dict(WORKLOADS[name])
    w.update(overrides)
    w["name"] = name
    w.setdefault("scale", 1.0 / math.sqrt(w["d"]))
    w["torch_dtype"] = _TORCH_DTYPES[w["dtype"]]
    return w


def _rng(w, *stream):
    return np.random.default_rng(np.random.SeedSequence([w["seed"], *stream]))


def _to16(x32, w):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(w["torch_dtype"])


def _values(rng, shape, w):
    x = rng.standard_normal(shape, dtype=np.float32)
    frac = w.get("outlier_frac", 0.0)
    if frac:
        hit = rng.random(shape) < frac
        sign = np.where(rng.random(shape) < 0.5, -1.0, 1.0).astype(np.float32)
        x = np.where(hit, sign * np.float32(w["outlier_mag"]), x).astype(np.float32)
    return x


def tails(w):
    """Per-child tail lengths of a prefix workload (uniform, inclusive)."""
    rng = _rng(w, _S_TAILS)
    return [int(t) for t in rng.integers(w["tail_lo"], w["tail_hi"] + 1, size=w["n_fork"])]


def context_lengths(w):
    """Context length of every decoded sequence (including the new token)."""
    if "lens" in w:
        return list(w["lens"])
    if "ctx" in w:
        return [w["ctx"]] * w["batch"]
    if "prompt" in w:
        return [w["prompt"] + t for t in tails(w)]
    rng = _rng(w, _S_LENS)
    return [int(x) for x in rng.integers(w["len_lo"], w["len_hi"] + 1, size=w["batch"])]


def free_order(w):
    """The pool's allocation order: a seeded permutation of the block ids,
    or, for a workload with ``in_order``, the ids in ascending order (each
    sequence prefilled in one go then owns consecutive blocks)."""
    if w.get("in_order"):
        return np.arange(w["num_blocks"], dtype=np.int32)
    rng = _rng(w, _S_FREE)
    return rng.permutation(w["num_blocks"]).astype(np.int32)


def query(w):
    """q [B, Hq, D] in the workload's 16-bit dtype (CPU)."""
    B = len(context_lengths(w))
    rng = _rng(w, _S_Q)
    return _to16(rng.standard_normal((B, w["hq"], w["d"]), dtype=np.float32), w)


def sequence_kv(w, i):
    """Logical K, V rows [ctx_i, Hkv, D] of decoded sequence i (CPU, 16-bit).

    For a prefix workload, rows 0..prompt-1 are the shared prompt's.
    """
    ctx = context_lengths(w)[i]
    shape_row = (w["hkv"], w["d"])
    if "prompt" in w:
        pr = _rng(w, _S_PROMPT)
        P = w["prompt"]
        kp = _values(pr, (P,) + shape_row, w)
        vp = _values(pr, (P,) + shape_row, w)
        rng = _rng(w, _S_KV, i)
        kt = _values(rng, (ctx - P,) + shape_row, w)
        vt = _values(rng, (ctx - P,) + shape_row, w)
        return _to16(np.concatenate([kp, kt]), w), _to16(np.concatenate([vp, vt]), w)
    rng = _rng(w, _S_KV, i)
    k = _values(rng, (ctx,) + shape_row, w)
    v = _values(rng, (ctx,) + shape_row, w)
    return _to16(k, w), _to16(v, w)


def prompt_kv(w):
    """Shared prompt rows [prompt, Hkv, D] of a prefix workload."""
    pr = _rng(w, _S_PROMPT)
    shape = (w["prompt"], w["hkv"], w["d"])
    return _to16(_values(pr, shape, w), w), _to16(_values(pr, shape, w), w)


def new_token_kv(w, step):
    """Fresh K, V [B, Hkv, D] for repeated decode steps of a benchmark loop."""
    B = len(context_lengths(w))
    rng = _rng(w, _S_NEW, step)
    shape = (B, w["hkv"], w["d"])
    return _to16(_values(rng, shape, w), w), _to16(_values(rng, shape, w), w)


def prefill_schedule(w):
    """Order of operations that builds the cache before the decode step.

    Returns a list of ("create",), ("append", seq, n) and ("fork", parent)
    tuples over local sequence handles 0, 1, 2, ... (handles are numbered in
    creation order, forks included), plus the list of handles that are
    decoded, in batch order.  The decode step then appends one token to every
    decoded handle.
    """
    lens = context_lengths(w)
    bs = w["block_size"]
    ops = []
    if "prompt" in w:
        ops.append(("create",))
        ops.append(("append", 0, w["prompt"]))
        decoded = []
        for j in range(w["n_fork"]):
            ops.append(("fork", 0))
            decoded.append(1 + j)
        for j, L in enumerate(lens):
            n = L - 1 - w["prompt"]
            if n > 0:
                ops.append(("append", 1 + j, n))
        return ops, decoded
    B = len(lens)
    for _ in range(B):
        ops.append(("create",))
    if w.get("interleave"):
        remaining = [L - 1 for L in lens]
        while any(r > 0 for r in remaining):
            for i in range(B):
                if remaining[i] > 0:
                    n = min(bs, remaining[i])
                    ops.append(("append", i, n))
                    remaining[i] -= n
    else:
        for i, L in enumerate(lens):
            if L - 1 > 0:
                ops.append(("append", i, L - 1))
    return ops, list(range(B))


def kv_rows_to_numpy(t):
    """16-bit tensor -> float32 NumPy array holding exactly the same values."""
    return t.float().numpy()
