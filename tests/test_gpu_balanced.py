"""GPU parity of the balanced split -- the automatic split of large decode
calls, where every warp streams an equal share of the (sequence, KV head,
block) items -- against the float64 oracle.

Covers runs much shorter than a warp's share (hundreds of short sequences,
lengths 1..320 tokens, so one warp crosses many sequences), runs spread over
a hundred warps (64k contexts), contexts set to zero after the build, fp16
with head dim 64 and GQA groups 1 and 8, the fused KV-append, and the
kernel's own checks (bad table entry, wrong slot)."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, expected

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def _is_balanced(c):
    """The library picks the balanced split for partition_size 0 when the
    tables hold >= 32 items per launched warp (16 warps per SM)."""
    w = c.w
    items = len(c.decoded) * w["hkv"] * c.max_blocks
    return items >= 32 * 16 * _sms() and len(c.decoded) <= 1024


def _short_workload(n=640, hi=320, **over):
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(1, hi + 1, size=n)]
    base = dict(lens=lens, num_blocks=sum(-(-L // 16) for L in lens) + n + 64)
    base.update(over)
    return syn.workload("llama3_8b_b64", **base)


def _decode(pkv, c, lens=None, tables=None):
    w = c.w
    B = len(c.decoded)
    out = torch.full((B, w["hq"], w["d"]), 7.0, dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables if tables is None else tables,
                                   c.lens if lens is None else lens, w["scale"], out, ws, 0)
    torch.cuda.synchronize()
    return out


def test_many_short_sequences(pkv, cuda_dev):
    w = _short_workload()
    c = build(pkv, w, cuda_dev)
    assert _is_balanced(c)
    out = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="640 short sequences")


def test_long_contexts_over_many_warps(pkv, cuda_dev):
    w = syn.workload("long_splitk")
    c = build(pkv, w, cuda_dev)
    assert _is_balanced(c)
    out = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="long contexts, balanced")


def test_zero_contexts_inside_the_batch(pkv, cuda_dev):
    w = _short_workload()
    c = build(pkv, w, cuda_dev)
    zero = [0, 1, 2, 200, 317, 639]  # the first, the last and runs of them
    lens = c.lens.clone()
    lens[zero] = 0
    out = _decode(pkv, c, lens=lens)
    assert pkv.pkv_device_status() == 0
    got = out.float().cpu().numpy()
    assert (got[zero] == 0).all()
    keep = [i for i in range(len(c.decoded)) if i not in zero]
    assert_close(got[keep], expected(c, keep), what="non-zero rows")


@pytest.mark.parametrize("hq,hkv,d,dtype", [(64, 8, 64, "fp16"), (8, 8, 64, "fp16"), (16, 8, 128, "bf16")])
def test_groups_dims_dtypes(pkv, cuda_dev, hq, hkv, d, dtype):
    w = _short_workload(n=700, hi=300, hq=hq, hkv=hkv, d=d, dtype=dtype)
    c = build(pkv, w, cuda_dev)
    assert _is_balanced(c)
    out = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="G %d D %d %s" % (hq // hkv, d, dtype))


def test_bad_table_entry_is_skipped(pkv, cuda_dev):
    w = _short_workload()
    c = build(pkv, w, cuda_dev)
    nblk = (c.lens_host + 15) // 16
    victim = int(np.argmax(nblk))
    tables = c.tables.clone()
    tables[victim, 1] = 1 << 24  # far outside the pool
    pkv.pkv_device_status()
    out = _decode(pkv, c, tables=tables)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_BLOCK
    keep = [i for i in range(len(c.decoded)) if i != victim]
    assert_close(out.float().cpu().numpy()[keep], expected(c, keep), what="other rows")
    assert pkv.pkv_device_status() == 0


def _decode_append(pkv, c, slots):
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode_append(c.q, c.new_k, c.new_v, torch.from_numpy(slots).to(c.q.device),
                                          c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, ws, 0)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", ["short", "llama3_8b_b64"])
def test_fused_append(pkv, cuda_dev, name):
    w = _short_workload() if name == "short" else syn.workload(name)
    c = build(pkv, w, cuda_dev, step_append=False, empty_fill=float("nan"))
    assert _is_balanced(c)
    out = _decode_append(pkv, c, c.step_slots.copy())
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="fused append, balanced")
    for i, slot in enumerate(c.step_slots):
        blk, off = divmod(int(slot), 16)
        assert torch.equal(c.k_pool[blk, :, off], c.new_k[i])
        assert torch.equal(c.v_pool[blk, :, off], c.new_v[i])
    out2 = _decode_append(pkv, c, c.step_slots.copy())
    assert torch.equal(out, out2)


def test_fused_append_rejects_wrong_slot(pkv, cuda_dev):
    w = _short_workload()
    c = build(pkv, w, cuda_dev, step_append=False, empty_fill=0.0)
    slots = c.step_slots.copy()
    i = next(j for j in range(5, len(slots)) if slots[j] % 16 < 15)
    slots[i] += 1  # the next offset of the right block: never written
    pkv.pkv_device_status()
    _decode_append(pkv, c, slots)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_SLOT
    blk, off = divmod(int(slots[i]), 16)
    assert (c.k_pool[blk, :, off] == 0).all()
    assert pkv.pkv_device_status() == 0


def _decode_quant(pkv, c, lens=None):
    w = c.w
    B = len(c.decoded)
    out = torch.full((B, w["hq"], w["d"]), 7.0, dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode_quant(c.q, c.cache, c.n_sink, c.tables, c.lens if lens is None else lens,
                                         w["scale"], out, c.quant, c.group_size, ws, 0,
                                         window=getattr(c, "window", 0))
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _short_quant_workload(n=640, hi=320, **over):
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(1, hi + 1, size=n)]
    base = dict(lens=lens, num_blocks=sum(-(-L // 16) for L in lens) + n + 64)
    base.update(over)
    return syn.workload("quant", **base)


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_quant_many_short_sequences_with_sinks(pkv, cuda_dev, qmode):
    """Hundreds of 1..320-token sequences (many shorter than the 4 sinks):
    runs start and end inside warp ranges, and the sink block of each run is
    taken by whichever warp's range holds it."""
    w = _short_quant_workload()
    c = build(pkv, w, cuda_dev, quant=qmode)
    assert _is_balanced(c)
    got = _decode_quant(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(got, expected(c), what="%s, 640 short sequences" % qmode)


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_quant_zero_contexts_and_head64_group8(pkv, cuda_dev, qmode):
    w = _short_quant_workload(n=700, hi=300, hq=64, hkv=8, d=64, dtype="fp16", group_size=64)
    c = build(pkv, w, cuda_dev, quant=qmode)
    assert _is_balanced(c)
    zero = [0, 5, 6, 699]
    lens = c.lens.clone()
    lens[zero] = 0
    got = _decode_quant(pkv, c, lens)
    assert pkv.pkv_device_status() == 0
    assert (got[zero] == 0).all()
    keep = [i for i in range(len(c.decoded)) if i not in zero]
    assert_close(got[keep], expected(c, keep), what="%s, G 8, D 64" % qmode)


def test_quant_int4_group64_many_short_sequences(pkv, cuda_dev):
    w = _short_quant_workload(group_size=64, n_sink=8)
    c = build(pkv, w, cuda_dev, quant="int4")
    assert _is_balanced(c)
    got = _decode_quant(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(got, expected(c), what="int4 g64, 640 short sequences")


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_quant_window_many_short_sequences(pkv, cuda_dev, qmode):
    """640 sequences of 1..320 tokens with a 128-token 16-bit window: runs
    start and end inside warp ranges, and the window blocks of a run may be
    split between warps."""
    w = _short_quant_workload(group_size=64 if qmode == "int4" else 128, n_sink=8, window=128)
    c = build(pkv, w, cuda_dev, quant=qmode)
    assert _is_balanced(c)
    got = _decode_quant(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(got, expected(c), what="%s window, 640 short sequences" % qmode)


def _runs_pieces(lens, hkv, max_blocks, sms):
    """How many warp ranges meet each non-empty (sequence, KV head) run of
    a balanced call: the split restated on the host (items of the call cut
    into nwt equal contiguous shares, 16 warps per SM at most)."""
    units = [-(-int(L) // 16) for L in lens]
    W = hkv * sum(units)
    nwt_launch = max(1, min(len(lens) * hkv * -(-max_blocks * 16 // 16) // 2, sms * 16))
    nwt = max(min(W // 2, nwt_launch), 1)
    out, cs = [], 0
    for nb in units:
        for k in range(hkv):
            if nb:
                S = cs + k * nb
                out.append(((S + nb) * nwt - 1) // W - ((S + 1) * nwt - 1) // W + 1)
        cs += nb * hkv
    return np.array(out)


def _mixed_workload():
    """400 short sequences and two long ones: runs met by one warp, by a
    few, and by dozens (merged with 4 partial groups per CTA)."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 321, size=400)] + [65536, 40000]
    return syn.workload("llama3_8b_b64", lens=lens,
                        num_blocks=sum(-(-L // 16) for L in lens) + len(lens) + 64)


def test_runs_of_one_few_and_many_pieces_in_one_call(pkv, cuda_dev):
    """One call whose runs are met by one warp range, by a few, and by more
    than 32 (the merge folds each from its consecutive partial slots)."""
    c = build(pkv, _mixed_workload(), cuda_dev)
    assert _is_balanced(c)
    pieces = _runs_pieces(c.lens_host, c.w["hkv"], c.max_blocks, _sms())
    assert (pieces == 1).any() and ((pieces > 1) & (pieces <= 32)).any() and (pieces > 32).any()
    out = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="mixed runs")


def test_back_to_back_calls_share_the_workspace(pkv, cuda_dev):
    """Calls of two shapes alternate on one stream and one workspace (first
    filled with 0xFF bytes) with no synchronisation between them: each call
    finds the other shape's partials in its slots, and gives the same bits
    every time."""
    c = build(pkv, _mixed_workload(), cuda_dev)
    w = c.w
    B, sub = len(c.decoded), 300
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0)
    ws = torch.empty(n, dtype=torch.uint8, device=cuda_dev)
    ws.fill_(0xFF)
    full, part = [], []
    for _ in range(3):
        o = torch.full((B, w["hq"], w["d"]), float("nan"), dtype=w["torch_dtype"], device=cuda_dev)
        pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], o, ws, 0)
        full.append(o)
        p = torch.full((sub, w["hq"], w["d"]), float("nan"), dtype=w["torch_dtype"], device=cuda_dev)
        pkv.pkv_paged_attention_decode(c.q[:sub].contiguous(), c.k_pool, c.v_pool, c.tables[:sub].contiguous(),
                                       c.lens[:sub].contiguous(), w["scale"], p, ws, 0)
        part.append(p)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    want = expected(c)
    for o in full:
        assert torch.equal(o, full[0])  # the same bits every call
    for p in part:
        assert torch.equal(p, part[0])
    assert_close(full[0].float().cpu().numpy(), want, what="full shape")
    assert_close(part[0].float().cpu().numpy(), want[:sub], what="first 300 sequences")


def test_graph_replay_of_the_balanced_call(pkv, cuda_dev):
    """The balanced call (split kernel and its merge, launched with
    programmatic dependent launch) captured in a CUDA graph: every replay
    gives the same bits, within the bound of the oracle."""
    c = build(pkv, syn.workload("llama3_8b_b64"), cuda_dev)
    assert _is_balanced(c)
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=cuda_dev)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 0)
    ws = torch.zeros(n, dtype=torch.uint8, device=cuda_dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, ws, 0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, ws, 0)
    want = expected(c)
    first = None
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() == 0
        got = out.clone()
        first = got if first is None else first
        assert torch.equal(got, first)
    assert_close(first.float().cpu().numpy(), want, what="graph replays")
