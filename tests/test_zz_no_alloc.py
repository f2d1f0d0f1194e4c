"""The allocation-free decode entry point, for callers that cannot allocate a
device workspace (graph capture, host runtimes that own all device memory,
fixed-budget serving loops).  Called through the C ABI, its output must
match the regular entry point's (which gets a torch-allocated workspace) and
the oracle's, on two calls in a row that follow a call with a different
query -- so every call reuses the library's array with another call's
partials still in it."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, expected

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


def _static(pkv, c, q, ps):
    w = c.w
    B = len(c.decoded)
    out = torch.full((B, w["hq"], w["d"]), float("nan"), dtype=w["torch_dtype"], device=q.device)
    pkv.pkv_paged_attention_decode_static_ws(q, c.k_pool, c.v_pool, c.tables, c.lens, w["scale"],
                                             out, ps)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


# partition 0 is the automatic choice: the balanced split and its merge on
# the two large workloads (partials for every warp's runs in the array), a
# single pass on the tiny one
@pytest.mark.parametrize("name,ps", [("llama3_8b_b64", 0), ("long_splitk", 0),
                                     ("llama3_8b_b64", 512), ("long_splitk", 512), ("tiny", 0)])
def test_static_workspace_matches_regular_twice(pkv, cuda_dev, name, ps):
    w = syn.workload(name)
    c = build(pkv, w, cuda_dev)
    B = len(c.decoded)
    need = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, ps)
    assert need <= pkv.PKV_STATIC_WORKSPACE_BYTES
    want = _regular(pkv, c, ps).float().cpu().numpy()
    oracle = expected(c)
    assert_close(want, oracle, what="%s regular entry point" % name)
    # leave other partials in the shared array first: the same cache with a
    # different query, so a missed write or a stale slot read shows
    other = _static(pkv, c, (c.q.float() * -1.75).to(c.q.dtype), ps)
    assert np.isfinite(other).all()
    assert not np.allclose(other, want)
    for call in range(2):
        got = _static(pkv, c, c.q, ps)
        assert np.isfinite(got).all()
        assert_close(got, want, what="%s call %d vs regular" % (name, call))
        assert_close(got, oracle, what="%s call %d vs oracle" % (name, call))
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
