"""GPU parity of multi-query paged attention (speculative verify of gamma + 1
tokens, chunked-prefill slices) against the float64 oracle."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, logical_rows
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


def _queries(w, qlens, seed):
    rng = np.random.default_rng(seed)
    T = int(sum(qlens))
    q32 = rng.standard_normal((T, w["hq"], w["d"]), dtype=np.float32)
    q = torch.from_numpy(q32).to(w["torch_dtype"])
    q_start = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    return q, q_start


def _run(pkv, c, qlens, seed=0, lens=None):
    w = c.w
    q, q_start = _queries(w, qlens, seed)
    dev = c.q.device
    out = torch.full(q.shape, 7.0, dtype=q.dtype, device=dev)
    pkv.pkv_paged_attention_multi_query(q.to(dev), torch.from_numpy(q_start).to(dev), c.k_pool, c.v_pool,
                                        c.tables, c.lens if lens is None else lens, w["scale"], out,
                                        max(max(qlens), 1))
    torch.cuda.synchronize()
    return q, q_start, out.float().cpu().numpy()


def _expected(c, q, q_start, seqs, ctx_override=None):
    qn = q.float().numpy()
    want = {}
    for b in seqs:
        k, v = logical_rows(c, b)
        if ctx_override is not None:
            k, v = k[:ctx_override[b]], v[:ctx_override[b]]
        want[b] = oatt.multi_query_attention(qn[q_start[b]:q_start[b + 1]], k, v, c.w["scale"])
    return want


def _check(c, q, q_start, got, seqs=None, ctx_override=None, what=""):
    seqs = range(len(q_start) - 1) if seqs is None else seqs
    want = _expected(c, q, q_start, seqs, ctx_override)
    for b, wb in want.items():
        if wb.shape[0]:
            assert_close(got[q_start[b]:q_start[b + 1]], wb, what="%s seq %d" % (what, b))


@pytest.mark.parametrize("L", [1, 2, 3, 4, 6, 8, 16, 17, 40])
def test_uniform_query_lengths(pkv, cuda_dev, L):
    w = syn.workload("llama3_8b_b64", batch=5, len_lo=40, len_hi=900, num_blocks=1024)
    c = build(pkv, w, cuda_dev)
    q, q_start, got = _run(pkv, c, [L] * 5, seed=L)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="L %d" % L)


def test_ragged_query_lengths_with_empty(pkv, cuda_dev):
    w = syn.workload("llama3_8b_b64", batch=7, len_lo=20, len_hi=600, num_blocks=1024)
    c = build(pkv, w, cuda_dev)
    qlens = [6, 0, 1, 19, 3, 0, 12]
    q, q_start, got = _run(pkv, c, qlens, seed=3)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="ragged")


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, "bf16"), (64, 8, 64, "fp16"), (16, 2, 64, "bf16"),
                                            (8, 2, 128, "fp16")])
def test_groups_dims_dtypes(pkv, cuda_dev, hq, hkv, d, dtype):
    w = syn.workload("llama3_8b_b64", batch=4, len_lo=30, len_hi=400, num_blocks=512, hq=hq, hkv=hkv,
                     d=d, dtype=dtype)
    c = build(pkv, w, cuda_dev)
    q, q_start, got = _run(pkv, c, [5, 1, 9, 2], seed=hq)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="G %d D %d %s" % (hq // hkv, d, dtype))


def test_whole_prefill_and_short_contexts(pkv, cuda_dev):
    """L = ctx: the whole sequence is new (a prefill from an empty cache),
    including contexts of 1, 15, 16 and 17 tokens."""
    w = syn.workload("llama3_8b_b64", lens=[1, 15, 16, 17, 100, 130], num_blocks=256)
    c = build(pkv, w, cuda_dev)
    lens = syn.context_lengths(w)
    q, q_start, got = _run(pkv, c, lens, seed=11)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="whole prefill")


def test_more_queries_than_context_sets_status(pkv, cuda_dev):
    w = syn.workload("llama3_8b_b64", lens=[5, 40], num_blocks=64)
    c = build(pkv, w, cuda_dev)
    pkv.pkv_device_status()
    q, q_start, got = _run(pkv, c, [8, 3], seed=12)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_CONTEXT
    assert (got[:3] == 0).all()  # queries 0..2 of sequence 0 sit at negative positions
    _check(c, q, q_start, got, seqs=[1], what="valid sequence")
    assert pkv.pkv_device_status() == 0


def test_one_query_agrees_with_decode(pkv, cuda_dev):
    w = syn.workload("llama3_8b_b64", batch=6, num_blocks=2048)
    c = build(pkv, w, cuda_dev)
    B = len(c.decoded)
    q = c.q
    out = torch.empty_like(q)
    q_start = torch.arange(B + 1, dtype=torch.int32, device=cuda_dev)
    pkv.pkv_paged_attention_multi_query(q, q_start, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, 1)
    dec = torch.empty_like(q)
    ws = torch.empty(max(pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0), 16),
                     dtype=torch.uint8, device=cuda_dev)
    pkv.pkv_paged_attention_decode(q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], dec, ws, 0)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), dec.float().cpu().numpy().astype(np.float64), what="vs decode")


def test_speculative_verify_full_layer_sampled(pkv, cuda_dev):
    """The 64-sequence layer with gamma + 1 = 6 query tokens per sequence
    (the pages' gamma = 5): sampled sequences against the oracle."""
    w = syn.workload("llama3_8b_b64")
    c = build(pkv, w, cuda_dev)
    q, q_start, got = _run(pkv, c, [6] * len(c.decoded), seed=5)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, seqs=[0, 17, 63], what="verify")


# ---------------------------------------------------------------- balanced split
def _run_balanced(pkv, c, qlens, seed=0, lens=None, max_q_len=None):
    """The multi-query call with a workspace: the balanced split where it
    applies (asserted)."""
    w = c.w
    B = len(qlens)
    mq = max(max(qlens), 1) if max_q_len is None else max_q_len
    n = pkv.pkv_multi_query_workspace_bytes(B, w["hq"], w["hkv"], w["d"], c.max_blocks, mq)
    assert n > 0, "the balanced split should apply"
    ws = torch.empty(n, dtype=torch.uint8, device=c.q.device)
    q, q_start = _queries(w, qlens, seed)
    dev = c.q.device
    out = torch.full(q.shape, 7.0, dtype=q.dtype, device=dev)
    pkv.pkv_paged_attention_multi_query(q.to(dev), torch.from_numpy(q_start).to(dev), c.k_pool, c.v_pool,
                                        c.tables, c.lens if lens is None else lens, w["scale"], out, mq,
                                        workspace=ws)
    torch.cuda.synchronize()
    return q, q_start, out.float().cpu().numpy()


def test_balanced_verify_full_layer(pkv, cuda_dev):
    """gamma + 1 = 6 queries on the 64-sequence layer (24 rows per KV head):
    every sequence against the oracle, and against the one-pass kernel."""
    w = syn.workload("llama3_8b_b64")
    c = build(pkv, w, cuda_dev)
    q, q_start, got = _run_balanced(pkv, c, [6] * len(c.decoded), seed=5)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="balanced verify")
    _, _, tile = _run(pkv, c, [6] * len(c.decoded), seed=5)
    assert_close(got, tile.astype(np.float64), what="balanced vs one-pass")


def _short(n=640, hi=320, **over):
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(1, hi + 1, size=n)]
    base = dict(lens=lens, num_blocks=sum(-(-L // 16) for L in lens) + n + 64)
    base.update(over)
    return syn.workload("llama3_8b_b64", **base)


@pytest.mark.parametrize("hq,hkv,d,dtype,maxL", [(32, 8, 128, "bf16", 6), (64, 8, 64, "fp16", 3),
                                                 (8, 8, 128, "bf16", 17), (16, 8, 64, "bf16", 8),
                                                 (32, 8, 128, "fp16", 2)])
def test_balanced_many_short_sequences(pkv, cuda_dev, hq, hkv, d, dtype, maxL):
    """640 sequences of 1..320 tokens with ragged query counts 0..maxL (never
    more than the context): runs start and end inside warp ranges, and some
    sequences have no queries at all."""
    w = _short(hq=hq, hkv=hkv, d=d, dtype=dtype)
    c = build(pkv, w, cuda_dev)
    rng = np.random.default_rng(hq + d)
    ctx = syn.context_lengths(w)
    qlens = [int(min(x, L)) for x, L in zip(rng.integers(0, maxL + 1, size=len(ctx)), ctx)]
    q, q_start, got = _run_balanced(pkv, c, qlens, seed=7, max_q_len=maxL)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="balanced short G %d D %d" % (hq // hkv, d))


def test_balanced_bad_table_entry_and_excess_queries(pkv, cuda_dev):
    w = _short()
    c = build(pkv, w, cuda_dev)
    ctx = syn.context_lengths(w)
    qlens = [min(4, L) for L in ctx]
    victim = int(np.argmax(ctx))
    tables = c.tables.clone()
    tables[victim, 1] = 1 << 24
    c.tables = tables
    pkv.pkv_device_status()
    q, q_start, got = _run_balanced(pkv, c, qlens, seed=9)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_BLOCK
    keep = [b for b in range(len(ctx)) if b != victim]
    _check(c, q, q_start, got, seqs=keep, what="other sequences")
    # a sequence with more queries than max_q_len: status, first rows computed
    qlens2 = list(qlens)
    j = next(b for b in range(len(ctx)) if ctx[b] >= 8 and b != victim)
    qlens2[j] = 5
    pkv.pkv_device_status()
    q2, q_start2, got2 = _run_balanced(pkv, c, qlens2, seed=10, max_q_len=4)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_CONTEXT
    _check(c, q2, q_start2, got2, seqs=[b for b in keep if b != j], what="others, excess queries")
    assert pkv.pkv_device_status() == 0


def test_balanced_workspace_too_small(pkv, cuda_dev):
    w = _short()
    c = build(pkv, w, cuda_dev)
    B = len(c.decoded)
    n = pkv.pkv_multi_query_workspace_bytes(B, w["hq"], w["hkv"], w["d"], c.max_blocks, 4)
    ws = torch.empty(n - 16, dtype=torch.uint8, device=cuda_dev)
    q = torch.zeros((B * 4, w["hq"], w["d"]), dtype=w["torch_dtype"], device=cuda_dev)
    q_start = torch.arange(0, B * 4 + 1, 4, dtype=torch.int32, device=cuda_dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attention_multi_query(q, q_start, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"],
                                            torch.empty_like(q), 4, workspace=ws)
    assert e.value.name == "PKV_ERR_WORKSPACE"


# ------------------------------------------------------- tensor-core prefill
# Long query spans (max_q_len x G > 64 at head dim 128) run on the tcgen05
# kernel: 128 (token, head) rows per CTA, K/V tiles of 128 keys by TMA.
@pytest.mark.parametrize("hq,hkv,dtype,qlens", [
    (32, 8, "bf16", [130, 77, 200, 33]),
    (32, 8, "fp16", [130, 77, 200, 33]),
    (8, 8, "bf16", [65, 300, 1, 129]),     # G = 1: 128 tokens per tile
    (16, 8, "fp16", [40, 129, 64, 7]),     # G = 2
    (64, 8, "bf16", [16, 17, 9, 250]),     # G = 8: 16 tokens per tile
])
def test_prefill_tc_groups_dtypes_nan_slots(pkv, cuda_dev, hq, hkv, dtype, qlens):
    """Contexts 300..900 (several 128-key tiles, the last one partial), slots
    past each context filled with NaN: those V rows must not reach O."""
    w = syn.workload("llama3_8b_b64", lens=[900, 511, 640, 301], num_blocks=512, hq=hq, hkv=hkv, d=128,
                     dtype=dtype)
    c = build(pkv, w, cuda_dev, empty_fill=float("nan"))
    q, q_start, got = _run(pkv, c, qlens, seed=hq + len(dtype))
    assert pkv.pkv_device_status() == 0
    assert not np.isnan(got).any()
    _check(c, q, q_start, got, what="tc G %d %s" % (hq // hkv, dtype))


def test_prefill_tc_chunk_of_long_prompts(pkv, cuda_dev):
    """512-token chunked-prefill slices at the end of 4,096-token contexts
    (the benchmark's shape), two sequences sampled in full."""
    w = syn.workload("llama3_8b_b64", lens=[4096, 3000, 4096], num_blocks=1024)
    c = build(pkv, w, cuda_dev)
    q, q_start, got = _run(pkv, c, [512, 512, 300], seed=31)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, seqs=[0, 2], what="512-token slice")


def test_prefill_tc_bad_block_and_short_context(pkv, cuda_dev):
    w = syn.workload("llama3_8b_b64", lens=[700, 40, 500], num_blocks=256)
    c = build(pkv, w, cuda_dev)
    tables = c.tables.clone()
    tables[2, 3] = 1 << 24
    c.tables = tables
    pkv.pkv_device_status()
    # sequence 1 has 40 tokens but 60 queries: queries 0..19 sit at negative positions
    q, q_start, got = _run(pkv, c, [100, 60, 80], seed=32)
    st = pkv.pkv_device_status()
    assert st & pkv.PKV_STATUS_BAD_BLOCK and st & pkv.PKV_STATUS_BAD_CONTEXT
    assert not (st & pkv.PKV_STATUS_COPY_TIMEOUT)
    assert (got[100:120] == 0).all()
    _check(c, q, q_start, got, seqs=[0], what="intact sequence")


@pytest.mark.parametrize("scale", [-0.0884, 0.0])
def test_prefill_tc_non_positive_scale(pkv, cuda_dev, scale):
    """A scale <= 0 takes the kernel's path that scales the scores before the
    max (with a positive scale the max is taken over raw scores): softmax of
    -|s| q.k, and at 0 the plain mean of V up to each query's position."""
    w = syn.workload("llama3_8b_b64", lens=[900, 640], num_blocks=256, hq=32, hkv=8, d=128, dtype="bf16",
                     scale=scale)
    c = build(pkv, w, cuda_dev, empty_fill=float("nan"))
    q, q_start, got = _run(pkv, c, [130, 200], seed=41)
    assert pkv.pkv_device_status() == 0
    assert not np.isnan(got).any()
    _check(c, q, q_start, got, what="tc scale %g" % scale)


def test_prefill_tc_wait_runs_out_and_the_context_stays_usable(pkv, cuda_dev):
    """A K copy that never comes (the test hook drops key tile 1 of every
    CTA): the S issuer's bounded wait runs out, the kernel reports
    PKV_STATUS_COPY_TIMEOUT and every CTA stops (no fault, no hang); the same
    call with the hook off then gives the oracle's outputs and a clean
    status."""
    w = syn.workload("llama3_8b_b64", lens=[700, 500], num_blocks=128)
    c = build(pkv, w, cuda_dev)
    pkv.pkv_device_status()
    try:
        pkv.pkv_debug_prefill_drop_copy(1)
        _run(pkv, c, [100, 80], seed=51)
        st = pkv.pkv_device_status()
    finally:
        pkv.pkv_debug_prefill_drop_copy(-1)
    assert st & pkv.PKV_STATUS_COPY_TIMEOUT
    q, q_start, got = _run(pkv, c, [100, 80], seed=51)
    assert pkv.pkv_device_status() == 0
    _check(c, q, q_start, got, what="after a run-out wait")
