"""GPU KV-append scatter and copy-on-write copy: bit-exact with the oracle."""

import numpy as np
import pytest
import torch

from oracle import kvcache as okv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float16, 64), (torch.bfloat16, 256)])
def test_kv_append_bit_exact(pkv, cuda_dev, dtype, D):
    rng = np.random.default_rng(D)
    NB, Hkv, bs, T = 40, 4, 16, 300
    k = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32)).to(dtype)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[::7] = -1  # skipped tokens
    init_k = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    init_v = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    kp = torch.from_numpy(init_k).to(dtype).to(cuda_dev)
    vp = torch.from_numpy(init_v).to(dtype).to(cuda_dev)
    pkv.pkv_kv_append(k.to(cuda_dev), v.to(cuda_dev), torch.from_numpy(slots).to(cuda_dev), kp, vp)
    torch.cuda.synchronize()
    want_k = torch.from_numpy(init_k).to(dtype).view(torch.int16).numpy().copy()
    want_v = torch.from_numpy(init_v).to(dtype).view(torch.int16).numpy().copy()
    okv.kv_append(k.view(torch.int16).numpy(), v.view(torch.int16).numpy(), slots, want_k, want_v, bs)
    assert np.array_equal(kp.view(torch.int16).cpu().numpy(), want_k)
    assert np.array_equal(vp.view(torch.int16).cpu().numpy(), want_v)
    assert pkv.pkv_device_status() == 0


def test_kv_append_out_of_range_slot_sets_status(pkv, cuda_dev):
    kp = torch.zeros((2, 1, 16, 64), dtype=torch.float16, device=cuda_dev)
    vp = torch.zeros_like(kp)
    k = torch.ones((2, 1, 64), dtype=torch.float16, device=cuda_dev)
    slots = torch.tensor([3, 32], dtype=torch.int64, device=cuda_dev)  # 32 == 2 blocks * 16
    pkv.pkv_device_status()
    pkv.pkv_kv_append(k, k, slots, kp, vp)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == pkv.PKV_STATUS_BAD_SLOT
    assert kp[0, 0, 3].eq(1).all() and kp.sum().item() == 64


def test_copy_blocks_bit_exact(pkv, cuda_dev):
    rng = np.random.default_rng(1)
    NB = 32
    pools_np = [rng.integers(0, 255, size=(NB, 2, 16, 64), dtype=np.uint8),
                rng.integers(0, 255, size=(NB, 2, 16, 2), dtype=np.uint8).view(np.uint8)]
    pools = [torch.from_numpy(p.copy()).to(cuda_dev) for p in pools_np]
    pairs = np.array([[3, 7], [10, 2], [31, 0]], dtype=np.int32)
    pkv.pkv_copy_blocks(pools, torch.from_numpy(pairs).to(cuda_dev))
    torch.cuda.synchronize()
    okv.copy_blocks(pools_np, pairs)
    for got, want in zip(pools, pools_np):
        assert np.array_equal(got.cpu().numpy(), want)
    bad = torch.tensor([[1, 99]], dtype=torch.int32, device=cuda_dev)
    pkv.pkv_copy_blocks(pools, bad)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == pkv.PKV_STATUS_BAD_PAIR
    for got, want in zip(pools, pools_np):
        assert np.array_equal(got.cpu().numpy(), want)
