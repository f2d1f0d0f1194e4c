"""GPU parity of the 16-bit paged decode at block sizes 8 and 32 (the
16-token default is covered everywhere else) against the float64 oracle.

The kernels tile the context in 16-token units whatever the block size (two
8-token blocks, or half a 32-token block, per unit), and the split-K is cut
in tokens, so the same logical cache must give the same output BITS at
block sizes 8, 16 and 32 -- on every path: single pass, fixed partitions,
the balanced split and the fused append.  Ragged lengths cover a context
ending inside either 8-token half of a unit and an odd number of 8-token
blocks (a unit whose second block does not exist)."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, expected

pytestmark = pytest.mark.gpu

RAGGED = [1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 32, 33, 47, 48, 100, 257, 300, 511, 1000]


def _decode(pkv, c, partition_size=0, append=False, slots=None):
    w = c.w
    B = len(c.decoded)
    out = torch.full((B, w["hq"], w["d"]), 7.0, dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, w["block_size"], partition_size)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    if append:
        s = torch.from_numpy(c.step_slots.copy() if slots is None else slots).to(c.q.device)
        pkv.pkv_paged_attention_decode_append(c.q, c.new_k, c.new_v, s, c.k_pool, c.v_pool, c.tables,
                                              c.lens, w["scale"], out, ws, partition_size)
    else:
        pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, ws,
                                       partition_size)
    torch.cuda.synchronize()
    return out


def _ragged(bs, **over):
    lens = RAGGED
    base = dict(lens=lens, num_blocks=2 * sum(-(-L // bs) for L in lens) + 16, block_size=bs)
    base.update(over)
    return syn.workload("llama3_8b_b64", **base)


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("hq,hkv,d,dtype", [(32, 8, 128, "bf16"), (8, 2, 64, "fp16"), (8, 8, 64, "bf16")])
def test_ragged_lengths_all_paths(pkv, cuda_dev, bs, hq, hkv, d, dtype):
    c = build(pkv, _ragged(bs, hq=hq, hkv=hkv, d=d, dtype=dtype), cuda_dev, empty_fill=float("nan"))
    want = expected(c)
    for ps in (0, 32, 64, 1024):
        got = _decode(pkv, c, ps)
        assert pkv.pkv_device_status() == 0
        assert not torch.isnan(got).any()
        assert_close(got.float().cpu().numpy(), want, what="block %d partition %d" % (bs, ps))


@pytest.mark.parametrize("ps", [0, 32, 1024])
def test_same_bits_at_block_sizes_8_16_32(pkv, cuda_dev, ps):
    outs = {}
    for bs in (8, 16, 32):
        c = build(pkv, _ragged(bs), cuda_dev)
        outs[bs] = _decode(pkv, c, ps)
        assert pkv.pkv_device_status() == 0
    assert torch.equal(outs[8], outs[16])
    assert torch.equal(outs[32], outs[16])


def _short(bs, n=640, hi=320, **over):
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(1, hi + 1, size=n)]
    base = dict(lens=lens, num_blocks=sum(-(-L // bs) for L in lens) + n + 64, block_size=bs)
    base.update(over)
    return syn.workload("llama3_8b_b64", **base)


@pytest.mark.parametrize("bs", [8, 32])
def test_balanced_split_short_sequences(pkv, cuda_dev, bs):
    """640 sequences of 1..320 tokens: the automatic split is balanced (>= 32
    items per launched warp) and runs start and end inside warp ranges."""
    w = _short(bs)
    c = build(pkv, w, cuda_dev)
    items = len(c.decoded) * w["hkv"] * -(-c.max_blocks * bs // 16)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    assert items >= 32 * 16 * sms
    got = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(got.float().cpu().numpy(), expected(c), what="balanced, block %d" % bs)
    ref = _decode(pkv, build(pkv, _short(16), cuda_dev))
    assert torch.equal(got, ref)


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("mode", ["ragged", "balanced"])
def test_fused_append(pkv, cuda_dev, bs, mode):
    w = _ragged(bs) if mode == "ragged" else _short(bs)
    c = build(pkv, w, cuda_dev, step_append=False, empty_fill=float("nan"))
    want = expected(c)
    for ps in ((0, 32) if mode == "ragged" else (0,)):
        got = _decode(pkv, c, ps, append=True)
        assert pkv.pkv_device_status() == 0
        assert_close(got.float().cpu().numpy(), want, what="fused append, block %d, ps %d" % (bs, ps))
    for i, slot in enumerate(c.step_slots):
        blk, off = divmod(int(slot), bs)
        assert torch.equal(c.k_pool[blk, :, off], c.new_k[i])
        assert torch.equal(c.v_pool[blk, :, off], c.new_v[i])


def test_fused_append_wrong_slot_block8(pkv, cuda_dev):
    c = build(pkv, _ragged(8), cuda_dev, step_append=False, empty_fill=0.0)
    slots = c.step_slots.copy()
    i = next(j for j in range(len(slots)) if slots[j] % 8 < 7)
    slots[i] += 1  # the next offset of the right block: never written
    pkv.pkv_device_status()
    _decode(pkv, c, 0, append=True, slots=slots)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_SLOT
    blk, off = divmod(int(slots[i]), 8)
    assert (c.k_pool[blk, :, off] == 0).all()
    assert pkv.pkv_device_status() == 0


@pytest.mark.parametrize("which", [0, 1])
def test_bad_entry_in_either_half_of_a_unit_block8(pkv, cuda_dev, which):
    """At block size 8 a 16-token unit reads two table entries; a bad one in
    either half skips that unit of that sequence only and sets the status."""
    c = build(pkv, _ragged(8), cuda_dev)
    victim = len(RAGGED) - 1  # 1000 tokens: 125 blocks
    tables = c.tables.clone()
    tables[victim, 40 + which] = 1 << 24
    pkv.pkv_device_status()
    w = c.w
    B = len(c.decoded)
    for ps in (0, 64):
        out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=cuda_dev)
        n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 8, ps)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=cuda_dev)
        pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, tables, c.lens, w["scale"], out, ws, ps)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_BLOCK
        keep = [j for j in range(B) if j != victim]
        assert_close(out.float().cpu().numpy()[keep], expected(c, keep), what="other rows, ps %d" % ps)
    assert pkv.pkv_device_status() == 0


@pytest.mark.parametrize("bs", [8, 32])
def test_llama3_layer_full_size(pkv, cuda_dev, bs):
    """The 64-sequence Llama-3-8B-shaped layer (contexts 512..4096) at block
    size 8 / 32, through the automatic split the benchmark times."""
    w = syn.workload("llama3_8b_b64", block_size=bs, num_blocks=40000 * 16 // bs)
    c = build(pkv, w, cuda_dev)
    got = _decode(pkv, c)
    assert pkv.pkv_device_status() == 0
    assert_close(got.float().cpu().numpy(), expected(c), what="llama3 layer, block %d" % bs)
