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
