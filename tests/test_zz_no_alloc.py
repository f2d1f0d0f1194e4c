"""The allocation-free decode entry point, for callers that cannot allocate a
device workspace (graph capture, host runtimes that own all device memory,
fixed-budget serving loops).  Called through the C ABI, its output must
match the regular entry point's (which gets a torch-allocated workspace),
on two calls in a row -- the second call reuses the library's array with the
first call's partials still in it."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build

pytestmark = pytest.mark.gpu


def _regular(pkv, c, ps):
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, ps)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode(c.q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"], out, ws, ps)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,ps", [("llama3_8b_b64", 512), ("long_splitk", 512), ("tiny", 0)])
def test_static_workspace_matches_regular_twice(pkv, cuda_dev, name, ps):
    w = syn.workload(name)
    c = build(pkv, w, cuda_dev)
    B = len(c.decoded)
    need = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, ps)
    assert need <= pkv.PKV_STATIC_WORKSPACE_BYTES
    want = _regular(pkv, c, ps).float().cpu().numpy()
    for call in range(2):
        out = torch.full((B, w["hq"], w["d"]), float("nan"), dtype=w["torch_dtype"], device=cuda_dev)
        pkv.pkv_paged_attention_decode_static_ws(c.q, c.k_pool, c.v_pool, c.tables, c.lens,
                                                 w["scale"], out, ps)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert_close(got, want, what="%s call %d" % (name, call))
    assert pkv.pkv_device_status() == 0


def test_static_workspace_rejects_oversized_shapes(pkv, cuda_dev):
    # 64 sequences x 32 heads x 128 partitions of 16 tokens x (128 + 2) floats > 16 MiB
    B, Hq, Hkv, D, mb = 64, 32, 8, 128, 2048
    assert pkv.pkv_decode_workspace_bytes(B, Hq, D, mb, 16, 256) > pkv.PKV_STATIC_WORKSPACE_BYTES
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=cuda_dev)
    pool = torch.zeros((4, Hkv, 16, D), dtype=torch.bfloat16, device=cuda_dev)
    tables = torch.zeros((B, mb), dtype=torch.int32, device=cuda_dev)
    lens = torch.zeros(B, dtype=torch.int32, device=cuda_dev)
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attention_decode_static_ws(q, pool, pool, tables, lens, 0.1, out, 256)
    assert e.value.name == "PKV_ERR_WORKSPACE"
