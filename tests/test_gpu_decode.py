"""GPU parity of the 16-bit paged decode path against the float64 oracle."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, expected
from oracle import attention as oatt
from oracle import kvcache as okv

pytestmark = pytest.mark.gpu


def _decode(pkv, c, partition_size=0, out_dtype=None):
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=c.q.device)
    nbytes = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, partition_size)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out,
                                   workspace=ws, partition_size=partition_size)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    return out


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64", "long_splitk", "prefix_cow", "prefix_cow_2008"])
def test_workload_decode_matches_oracle(pkv, cuda_dev, name):
    w = syn.workload(name)
    c = build(pkv, w, cuda_dev)
    want = expected(c)
    got = _decode(pkv, c, w.get("partition_size", 0)).float().cpu().numpy()
    err = assert_close(got, want, what=name)
    assert err < 2e-3
    if name == "prefix_cow_2008":
        assert len(c.all_pairs) == 8  # each child clones the shared partial block once
    if name == "prefix_cow":
        assert c.all_pairs == []  # the shared tail block is full: nothing to clone


@pytest.mark.parametrize("partition_size", [16, 32, 48, 512, 4096])
def test_partition_sizes_agree(pkv, cuda_dev, partition_size):
    w = syn.workload("llama3_8b_b64", batch=6, num_blocks=2048)
    c = build(pkv, w, cuda_dev)
    want = expected(c)
    got = _decode(pkv, c, partition_size).float().cpu().numpy()
    assert_close(got, want, what="partition %d" % partition_size)


def test_single_partition_equals_split_bitwise(pkv, cuda_dev):
    """partition >= context: the split path (partials + merge) gives the
    same bits as the single-pass path."""
    w = syn.workload("tiny")
    c = build(pkv, w, cuda_dev)
    single = _decode(pkv, c, 0)
    B = len(c.decoded)
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, 16) + 16,
                     dtype=torch.uint8, device=cuda_dev)
    # partials with a partition covering all blocks, then merge
    big = 16 * c.max_blocks
    ws2 = torch.empty(B * w["hq"] * (w["d"] + 2) * 4, dtype=torch.uint8, device=cuda_dev)
    pkv.pkv_paged_attention_decode_partials(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"],
                                            ws2, partition_size=big)
    out2 = torch.empty_like(single)
    pkv.pkv_paged_attention_decode_merge(c.lens, c.max_blocks, ws2, out2, partition_size=big)
    torch.cuda.synchronize()
    assert torch.equal(single, out2)
    del ws


@pytest.mark.parametrize("ctx", [1, 2, 15, 16, 17, 31, 33, 511, 512, 513, 1000])
@pytest.mark.parametrize("G,D,dtype", [(4, 128, torch.bfloat16), (1, 64, torch.float16),
                                       (8, 128, torch.float16), (2, 64, torch.bfloat16)])
def test_edge_lengths_and_groups(pkv, cuda_dev, ctx, G, D, dtype):
    rng = np.random.default_rng(ctx * 10 + G)
    Hkv, bs = 2, 16
    Hq = G * Hkv
    nblk = -(-ctx // bs)
    NB = nblk * 2 + 3
    order = rng.permutation(NB)
    table = np.array(order[:nblk], dtype=np.int32)
    k = torch.from_numpy(rng.standard_normal((ctx, Hkv, D)).astype(np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((ctx, Hkv, D)).astype(np.float32)).to(dtype)
    q = torch.from_numpy(rng.standard_normal((1, Hq, D)).astype(np.float32)).to(dtype)
    kp = torch.full((NB, Hkv, bs, D), float("nan"), dtype=dtype, device=cuda_dev)
    vp = torch.full((NB, Hkv, bs, D), float("nan"), dtype=dtype, device=cuda_dev)
    slots = torch.tensor([int(table[t // bs]) * bs + t % bs for t in range(ctx)], dtype=torch.int64, device=cuda_dev)
    pkv.pkv_kv_append(k.to(cuda_dev), v.to(cuda_dev), slots, kp, vp)
    tables = torch.from_numpy(table[None, :]).to(cuda_dev)
    lens = torch.tensor([ctx], dtype=torch.int32, device=cuda_dev)
    want = oatt.sequence_attention(q[0].float().numpy(), k.float().numpy(), v.float().numpy(), D ** -0.5)
    for ps in (0, 32, 512):
        out = torch.empty((1, Hq, D), dtype=dtype, device=cuda_dev)
        n = pkv.pkv_decode_workspace_bytes(1, Hq, D, nblk, 16, ps)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=cuda_dev)
        pkv.pkv_paged_attention_decode(q.to(cuda_dev), kp, vp, tables, lens, D ** -0.5, out, ws, ps)
        torch.cuda.synchronize()
        assert not torch.isnan(out).any()
        assert_close(out[0].float().cpu().numpy(), want, what="ctx %d ps %d" % (ctx, ps))
    assert pkv.pkv_device_status() == 0


def test_zero_context_gives_zeros(pkv, cuda_dev):
    D, Hkv, G = 128, 2, 4
    kp = torch.randn((4, Hkv, 16, D), dtype=torch.bfloat16, device=cuda_dev)
    q = torch.randn((3, G * Hkv, D), dtype=torch.bfloat16, device=cuda_dev)
    tables = torch.tensor([[0, 1], [2, -1], [-1, -1]], dtype=torch.int32, device=cuda_dev)
    lens = torch.tensor([20, 3, 0], dtype=torch.int32, device=cuda_dev)
    want = oatt.paged_attention_decode(q.float().cpu().numpy(), kp.float().cpu().numpy(),
                                       kp.float().cpu().numpy(), tables.cpu().numpy(),
                                       lens.cpu().numpy(), 0.1)
    assert not want[2].any()
    for ps in (0, 16):
        out = torch.full((3, G * Hkv, D), 7.0, dtype=torch.bfloat16, device=cuda_dev)
        ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_dev)
        pkv.pkv_paged_attention_decode(q, kp, kp, tables, lens, 0.1, out, ws, ps)
        torch.cuda.synchronize()
        assert (out[2] == 0).all()
        assert_close(out.float().cpu().numpy(), want, what="zero context beside 20 and 3, ps %d" % ps)
    assert pkv.pkv_device_status() == 0


def test_bit_identical_across_block_permutations(pkv, cuda_dev):
    """Paging changes layout only: the same logical cache at different
    physical blocks gives the same output bits (the reduction order never
    depends on physical block ids)."""
    rng = np.random.default_rng(3)
    B, Hkv, G, D, bs = 3, 2, 4, 128, 16
    lens = [25, 47, 300]
    ks = [torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16) for L in lens]
    vs = [torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16) for L in lens]
    q = torch.from_numpy(rng.standard_normal((B, G * Hkv, D)).astype(np.float32)).to(torch.bfloat16).to(cuda_dev)
    NB = 64
    outs = []
    for trial in range(8):
        pool = pkv.pkv_pool_create(NB, bs, rng.permutation(NB))
        kp = torch.empty((NB, Hkv, bs, D), dtype=torch.bfloat16, device=cuda_dev)
        vp = torch.empty_like(kp)
        seqs = []
        for i, L in enumerate(lens):
            s = pkv.pkv_seq_create(pool)
            slots, _ = pkv.pkv_seq_append(pool, s, L)
            pkv.pkv_kv_append(ks[i].to(cuda_dev), vs[i].to(cuda_dev), torch.from_numpy(slots).to(cuda_dev), kp, vp)
            seqs.append(s)
        tables, cl = pkv.pkv_build_block_tables(pool, seqs, 19)
        for ps in (0, 64):
            out = torch.empty((B, G * Hkv, D), dtype=torch.bfloat16, device=cuda_dev)
            ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_dev)
            pkv.pkv_paged_attention_decode(q, kp, vp, torch.from_numpy(tables).to(cuda_dev),
                                           torch.from_numpy(cl).to(cuda_dev), D ** -0.5, out, ws, ps)
            outs.append((ps, out.cpu()))
        pkv.pkv_pool_destroy(pool)
    for ps in (0, 64):
        ref = [o for p, o in outs if p == ps]
        for o in ref[1:]:
            assert torch.equal(o, ref[0])


def test_fully_shared_table(pkv, cuda_dev):
    """Every sequence points at the same physical blocks."""
    rng = np.random.default_rng(4)
    Hkv, G, D, bs, L, B = 8, 4, 128, 16, 700, 5
    NB = 64
    k = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    table = rng.permutation(NB)[: -(-L // bs)].astype(np.int32)
    kp = torch.empty((NB, Hkv, bs, D), dtype=torch.bfloat16, device=cuda_dev)
    vp = torch.empty_like(kp)
    slots = torch.tensor([int(table[t // bs]) * bs + t % bs for t in range(L)], device=cuda_dev)
    pkv.pkv_kv_append(k.to(cuda_dev), v.to(cuda_dev), slots, kp, vp)
    q = torch.from_numpy(rng.standard_normal((B, G * Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    tables = torch.from_numpy(np.tile(table, (B, 1))).to(cuda_dev)
    lens = torch.full((B,), L, dtype=torch.int32, device=cuda_dev)
    out = torch.empty((B, G * Hkv, D), dtype=torch.bfloat16, device=cuda_dev)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device=cuda_dev)
    pkv.pkv_paged_attention_decode(q.to(cuda_dev), kp, vp, tables, lens, D ** -0.5, out, ws, 128)
    torch.cuda.synchronize()
    for b in range(B):
        want = oatt.sequence_attention(q[b].float().numpy(), k.float().numpy(), v.float().numpy(), D ** -0.5)
        assert_close(out[b].float().cpu().numpy(), want, what="seq %d" % b)


def test_bad_table_entry_sets_status_and_is_skipped(pkv, cuda_dev):
    """A table entry outside the pool is never dereferenced: the kernel's own
    bounds check skips that block and records PKV_STATUS_BAD_BLOCK."""
    D, Hkv, G = 128, 2, 4
    kp = torch.randn((4, Hkv, 16, D), dtype=torch.bfloat16, device=cuda_dev)
    q = torch.randn((1, G * Hkv, D), dtype=torch.bfloat16, device=cuda_dev)
    tables = torch.tensor([[0, 1000]], dtype=torch.int32, device=cuda_dev)
    lens = torch.tensor([32], dtype=torch.int32, device=cuda_dev)
    out = torch.empty((1, G * Hkv, D), dtype=torch.bfloat16, device=cuda_dev)
    pkv.pkv_device_status()
    pkv.pkv_paged_attention_decode(q, kp, kp, tables, lens, 0.1, out, None, 0)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_BLOCK
    # the result equals attention over the valid first block alone
    want = oatt.sequence_attention(q[0].float().cpu().numpy(), kp[0].float().cpu().numpy().transpose(1, 0, 2),
                                   kp[0].float().cpu().numpy().transpose(1, 0, 2), 0.1)
    assert_close(out[0].float().cpu().numpy(), want)
    assert pkv.pkv_device_status() == 0


def _decode_append(pkv, c, partition_size=0):
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, partition_size)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    slots = torch.from_numpy(c.step_slots.copy()).to(c.q.device)
    pkv.pkv_paged_attention_decode_append(c.q, c.new_k, c.new_v, slots, c.k_pool, c.v_pool, c.tables,
                                          c.lens, w["scale"], out, ws, partition_size)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,ps", [("tiny", 0), ("tiny", 16), ("llama3_8b_b64", 512),
                                     ("long_splitk", 512), ("prefix_cow_2008", 256)])
def test_fused_append_decode(pkv, cuda_dev, name, ps):
    """One kernel writes the step's new rows and attends with them: the
    output matches the oracle and the pool then holds the new rows exactly."""
    w = syn.workload(name)
    c = build(pkv, w, cuda_dev, step_append=False, empty_fill=float("nan"))
    out = _decode_append(pkv, c, ps)
    assert pkv.pkv_device_status() == 0
    assert_close(out.float().cpu().numpy(), expected(c), what="fused %s" % name)
    for i, slot in enumerate(c.step_slots):
        blk, off = divmod(int(slot), 16)
        assert torch.equal(c.k_pool[blk, :, off], c.new_k[i])
        assert torch.equal(c.v_pool[blk, :, off], c.new_v[i])
    # a second call with the rows now in the pool gives the same bits
    out2 = _decode_append(pkv, c, ps)
    assert torch.equal(out, out2)


def test_fused_append_rejects_wrong_slot(pkv, cuda_dev):
    w = syn.workload("tiny")
    c = build(pkv, w, cuda_dev, step_append=False, empty_fill=0.0)
    c.step_slots = c.step_slots.copy()
    good = int(c.step_slots[1])
    c.step_slots[1] = good + 1 if good % 16 < 15 else good - 1  # wrong offset
    pkv.pkv_device_status()
    _decode_append(pkv, c, 0)
    assert pkv.pkv_device_status() & pkv.PKV_STATUS_BAD_SLOT
    blk, off = divmod(int(c.step_slots[1]), 16)
    assert (c.k_pool[blk, :, off] == 0).all()  # nothing written at the wrong slot
    assert pkv.pkv_device_status() == 0
