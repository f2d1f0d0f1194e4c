"""The C-ABI library loads on a host without a GPU and exports every entry
point the header declares; host-side argument checks reject bad calls
before any device work."""

import ctypes
import os
import re

import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_pool_create", "pkv_seq_append", "pkv_seq_fork", "pkv_kv_append",
                     "pkv_paged_attention_decode", "pkv_kv_append_quant",
                     "pkv_paged_attention_decode_quant", "pkv_copy_blocks", "pkv_device_status"):
        assert required in names
    assert len(names) >= 30


def test_every_declared_symbol_is_exported(pkv):
    missing = [n for n in declared_functions() if not hasattr(pkv.lib, n)]
    assert missing == []


def test_every_declared_symbol_has_a_binding(pkv):
    for n in declared_functions():
        assert hasattr(pkv, n) or n == "pkv_status_string" or n in ("pkv_pool_block_size",), n


def test_static_workspace_size_agrees_with_the_header(pkv):
    """The binding's PKV_STATIC_WORKSPACE_BYTES (used to size-check calls of
    the allocation-free decode) is the header's #define, not a separate copy
    that could drift."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+PKV_STATIC_WORKSPACE_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "PKV_STATIC_WORKSPACE_BYTES not found in the header"
    assert pkv.PKV_STATIC_WORKSPACE_BYTES == int(m.group(1)) << int(m.group(2))


def test_status_strings(pkv):
    for code in range(-10, 1):
        s = pkv.lib.pkv_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert pkv.lib.pkv_status_string(0) == b"ok"
    assert pkv.pkv_version() >= 1


def test_host_validation_rejects_before_launch(pkv):
    L = pkv.lib
    # Hq not a multiple of Hkv
    st = L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 6, 4, 128, 10, 16, 4, 1.0, 16, None, 0, 0, 1, None)
    assert st == -1
    # unsupported head dim and block size
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 96, 10, 16, 4, 1.0, 16, None, 0, 0, 1, None) == -8
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 128, 10, 24, 4, 1.0, 16, None, 0, 0, 1, None) == -8
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 128, 10, 64, 4, 1.0, 16, None, 0, 0, 1, None) == -8
    # GQA group above 8
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 32, 2, 128, 10, 16, 4, 1.0, 16, None, 0, 0, 1, None) == -8
    # misaligned query pointer
    assert L.pkv_paged_attention_decode(18, 16, 16, 16, 16, 1, 8, 2, 128, 10, 16, 4, 1.0, 16, None, 0, 0, 1, None) == -10
    # partition not a multiple of the block size
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 128, 10, 16, 4, 1.0, 16, None, 0, 100, 1, None) == -1
    # 8-token blocks: the partition must also be a multiple of the 16-token tile
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 128, 10, 8, 4, 1.0, 16, None, 0, 24, 1, None) == -1
    # 32-token blocks: a 16-token partition is not a multiple of the block
    assert L.pkv_paged_attention_decode(16, 16, 16, 16, 16, 1, 8, 2, 128, 10, 32, 4, 1.0, 16, None, 0, 16, 1, None) == -1
    # bad dtype
    assert L.pkv_kv_append(16, 16, 16, 1, 16, 16, 4, 2, 128, 16, 7, None) == -1
    # empty work is a no-op even without a device
    assert L.pkv_kv_append(16, 16, 16, 0, 16, 16, 4, 2, 128, 16, 1, None) == 0
    # copy_blocks pool count limits
    assert L.pkv_copy_blocks(None, None, 0, None, 1, 4, None) == -1
    # the prefill test hook takes a key tile or -1 (off)
    assert L.pkv_debug_prefill_drop_copy(-2) == -1


def test_workspace_bytes(pkv):
    # 64 sequences, 32 heads, dim 128, 256 blocks of 16, 512-token partitions
    # fp32 partials: o [B, Hq, P, D] and (m, l) [B, Hq, P, 2]
    assert pkv.pkv_decode_workspace_bytes(64, 32, 128, 256, 16, 512) == 64 * 32 * 8 * 130 * 4
    # one partition covers everything: single pass, no workspace
    assert pkv.pkv_decode_workspace_bytes(3, 8, 64, 3, 16, 512) == 0
    assert pkv.pkv_decode_workspace_bytes(1, 3, 64, 64, 16, 512) == 3 * 2 * 66 * 4


def _sms():
    import torch
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 152  # the library's default without a device


def test_workspace_bytes_automatic(pkv):
    # automatic split on tables of >= 32 items per 16 warps per SM (items =
    # batch x Hq x max_blocks bounds batch x Hkv x blocks): room for the
    # balanced split (partial rows for a GQA group of up to 8 per warp, up to
    # 20 warps per SM, one row per (sequence, query head)) and for the
    # automatic partitions, whichever is more
    nwt = 20 * _sms()
    assert 4 * 32 * 4096 >= 32 * 16 * _sms()
    balanced = (nwt * 8 + 4 * 32) * 130 * 4
    fixed = 4 * 32 * 128 * 130 * 4
    assert pkv.pkv_decode_workspace_bytes(4, 32, 128, 4096, 16, 0) == max(balanced, fixed)
    # 300 sequences of 64k tokens: the fixed partitions dominate
    fixed = 300 * 32 * 128 * 130 * 4
    assert pkv.pkv_decode_workspace_bytes(300, 32, 128, 4096, 16, 0) == fixed
    # above 1,024 sequences only the partitions are used
    assert pkv.pkv_decode_workspace_bytes(1025, 32, 128, 64, 16, 0) == \
        pkv.pkv_decode_workspace_bytes(1025, 32, 128, 64, 16, 512)
    # small tables: the automatic partitions only (64 tokens here)
    assert 3 * 8 * 19 < 32 * 16 * _sms()
    assert pkv.pkv_decode_workspace_bytes(3, 8, 128, 19, 16, 0) == 3 * 8 * 5 * 130 * 4
    # one partition covers everything: single pass, no workspace
    assert pkv.pkv_decode_workspace_bytes(3, 8, 64, 3, 16, 0) == 0


def test_auto_partition_size(pkv):
    # enough (query head, partition) items at 512 tokens: keep 512
    assert pkv.pkv_decode_auto_partition_size(64, 32, 256) == 512
    # 8 sequences of ~2,300 tokens: finer splits to fill 152 SMs
    assert pkv.pkv_decode_auto_partition_size(8, 32, 144) == 256
    assert pkv.pkv_decode_auto_partition_size(2, 32, 144) == 64
    # tiny: the smallest size (a single partition then covers it)
    assert pkv.pkv_decode_auto_partition_size(3, 8, 3) == 64
    # the workspace for partition 0 covers the automatic partitions
    assert pkv.pkv_decode_workspace_bytes(8, 32, 128, 144, 16, 0) >= pkv.pkv_decode_workspace_bytes(8, 32, 128, 144, 16, 256)


def test_block_sizes_8_and_32(pkv):
    """Block sizes 8 and 32 keep the same split in tokens: the workspace
    follows the tables' capacity in tokens (max_blocks x block_size), and
    the automatic partition size depends on that capacity alone."""
    for bs, mb in ((8, 512), (32, 128)):  # 4,096 tokens, as 256 blocks of 16
        assert pkv.pkv_decode_workspace_bytes(64, 32, 128, mb, bs, 512) == \
            pkv.pkv_decode_workspace_bytes(64, 32, 128, 256, 16, 512)
        assert pkv.pkv_decode_workspace_bytes(4, 32, 128, mb * 16, bs, 0) == \
            pkv.pkv_decode_workspace_bytes(4, 32, 128, 4096, 16, 0)
        assert pkv.pkv_decode_auto_partition_size(8, 32, 144 * 16 // bs, bs) == 256
    # an odd number of 8-token blocks: 3 blocks = 24 tokens = 2 tiles of 16
    assert pkv.pkv_decode_workspace_bytes(1, 3, 64, 3, 8, 16) == 3 * 2 * 66 * 4
    # 32-token blocks: 48-token partitions are not whole blocks
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_workspace_bytes(1, 3, 64, 4, 32, 48)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_auto_partition_size(8, 32, 144, 24)


def test_multi_query_workspace_bytes(pkv):
    """The balanced multi-query split: (nwt + batch x Hkv) slots of R =
    8 ceil(rows / 8) partial rows of (D + 2) fp32, nwt = min(SMs x warps per
    SM, items / 2) with 8 warps per SM at 17..24 rows (12 at 1..8)."""
    sms = _sms()
    nwt = min(sms * 8, 64 * 8 * 256 // 2)
    assert pkv.pkv_multi_query_workspace_bytes(64, 32, 8, 128, 256, 6) == (nwt + 64 * 8) * 24 * 130 * 4
    nwt1 = min(sms * 12, 64 * 8 * 256 // 2)
    assert pkv.pkv_multi_query_workspace_bytes(64, 32, 8, 128, 256, 2) == (nwt1 + 64 * 8) * 8 * 130 * 4
    # more than 24 rows per KV head, too few items, too many sequences: none
    assert pkv.pkv_multi_query_workspace_bytes(64, 32, 8, 128, 256, 7) == 0
    assert pkv.pkv_multi_query_workspace_bytes(2, 32, 8, 128, 16, 6) == 0
    assert pkv.pkv_multi_query_workspace_bytes(1025, 32, 8, 128, 256, 1) == 0
    with pytest.raises(pkv.PkvError):
        pkv.pkv_multi_query_workspace_bytes(64, 32, 8, 128, 256, 6, block_size=8)
