"""Python binding of libpkv (paged KV-cache decode attention, GB300 / sm_103a).

Argument marshalling only: every function here forwards to the C entry point
of the same name in ``include/pkv.h``.  Tensors are passed by device pointer
(``data_ptr()``), shapes are read off the tensors, the stream defaults to
torch's current CUDA stream, and a negative status raises ``PkvError``.
Every step of the computation runs in the library's kernels; there is no
other implementation to fall back on, and importing this package fails when
``libpkv.so`` has not been built (``python -c "import __graft_entry__ as g;
g.build()"`` or ``python paged_kv_cache_13_gb300/build.py``).
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libpkv.so is not built (expected at %s); build it with "
        "paged_kv_cache_13_gb300/build.py" % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

PKV_OK = 0
PKV_DTYPE_F16 = 0
PKV_DTYPE_BF16 = 1
PKV_QMODE_INT4_ASYM = 1
PKV_QMODE_FP8_E4M3 = 2
STATUS_NAMES = {
    0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_OUT_OF_BLOCKS", -3: "PKV_ERR_BAD_HANDLE",
    -4: "PKV_ERR_BAD_SEQ", -5: "PKV_ERR_DOUBLE_FREE", -6: "PKV_ERR_CUDA",
    -7: "PKV_ERR_DEVICE_BOUNDS", -8: "PKV_ERR_UNSUPPORTED", -9: "PKV_ERR_WORKSPACE",
    -10: "PKV_ERR_MISALIGNED",
}
PKV_STATUS_BAD_BLOCK, PKV_STATUS_BAD_SLOT, PKV_STATUS_BAD_CONTEXT = 1, 2, 4
PKV_STATUS_BAD_PAIR, PKV_STATUS_BAD_SINK, PKV_STATUS_COPY_TIMEOUT = 8, 16, 32

_i32, _i64, _f32, _int = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_int
_vp, _sz = ctypes.c_void_p, ctypes.c_size_t
_p_i32, _p_i64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)

_SIGS = {
    "pkv_status_string": ([_int], ctypes.c_char_p),
    "pkv_version": ([], _int),
    "pkv_pool_create": ([_i32, _i32, _vp, ctypes.POINTER(_vp)], _int),
    "pkv_pool_destroy": ([_vp], _int),
    "pkv_pool_num_free": ([_vp, _p_i32], _int),
    "pkv_pool_num_blocks": ([_vp, _p_i32], _int),
    "pkv_pool_block_size": ([_vp, _p_i32], _int),
    "pkv_block_alloc": ([_vp, _p_i32], _int),
    "pkv_block_incref": ([_vp, _i32], _int),
    "pkv_block_decref": ([_vp, _i32], _int),
    "pkv_block_refcount": ([_vp, _i32, _p_i32], _int),
    "pkv_seq_create": ([_vp, _p_i64], _int),
    "pkv_seq_free": ([_vp, _i64], _int),
    "pkv_seq_fork": ([_vp, _i64, _p_i64], _int),
    "pkv_seq_append": ([_vp, _i64, _i32, _vp, _vp, _p_i32], _int),
    "pkv_seq_append_batch": ([_vp, _vp, _i32, _i32, _vp, _vp, _p_i32], _int),
    "pkv_seq_len": ([_vp, _i64, _p_i64], _int),
    "pkv_seq_num_blocks": ([_vp, _i64, _p_i32], _int),
    "pkv_seq_block_table": ([_vp, _i64, _vp, _i32], _int),
    "pkv_build_block_tables": ([_vp, _vp, _i32, _vp, _i32, _vp], _int),
    "pkv_debug_fail_after": ([_vp, _i64], _int),
    "pkv_debug_prefill_drop_copy": ([_i32], _int),
    "pkv_prefix_register": ([_vp, _i64, _vp, _i32, _p_i32], _int),
    "pkv_prefix_match": ([_vp, _vp, _i32, _p_i64, _p_i32], _int),
    "pkv_prefix_evict": ([_vp, _i32, _p_i32], _int),
    "pkv_prefix_clear": ([_vp], _int),
    "pkv_prefix_stats": ([_vp, _p_i64, _p_i64, _p_i64], _int),
    "pkv_decode_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)], _int),
    "pkv_decode_auto_partition_size": ([_i32, _i32, _i32, _i32, _p_i32], _int),
    "pkv_kv_append": ([_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _int, _vp], _int),
    "pkv_paged_attention_multi_query": (
        [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp,
         _vp, _sz, _int, _vp], _int),
    "pkv_multi_query_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)],
                                        _int),
    "pkv_paged_attention_decode": (
        [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz,
         _i32, _int, _vp], _int),
    "pkv_paged_attention_decode_append": (
        [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
         _vp, _vp, _sz, _i32, _int, _vp], _int),
    "pkv_paged_attention_decode_partials": (
        [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _sz, _i32,
         _int, _vp], _int),
    "pkv_paged_attention_decode_merge": (
        [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp, _int, _vp], _int),
    "pkv_paged_attention_decode_static_ws": (
        [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _i32, _int,
         _vp], _int),
    "pkv_kv_append_quant": (
        [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
         _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _int, _int, _vp], _int),
    "pkv_paged_attention_decode_quant": (
        [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _i32,
         _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, _i32, _int, _int, _vp], _int),
    "pkv_copy_blocks": ([_vp, _vp, _i32, _vp, _i32, _i32, _vp], _int),
    "pkv_device_status": ([_p_i32, _vp], _int),
}

for _name, (_args, _res) in _SIGS.items():
    if hasattr(lib, _name):
        _f = getattr(lib, _name)
        _f.argtypes = _args
        _f.restype = _res


class PkvError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__("%s failed: %s (%s)" % (where, self.name, lib.pkv_status_string(status).decode()))


def _check(st, where):
    if st != PKV_OK:
        raise PkvError(st, where)


# ------------------------------------------------------------ marshalling
def _ptr(x):
    """Device/host address of a tensor or ndarray, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return PKV_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return PKV_DTYPE_BF16
    raise TypeError("16-bit fp16 / bf16 tensor expected, got %s" % t.dtype)


def _qmode_code(qmode):
    if qmode in ("int4", PKV_QMODE_INT4_ASYM):
        return PKV_QMODE_INT4_ASYM
    if qmode in ("fp8", PKV_QMODE_FP8_E4M3):
        return PKV_QMODE_FP8_E4M3
    raise ValueError(qmode)


def pkv_version():
    return lib.pkv_version()


# ------------------------------------------------------------ host manager
def pkv_pool_create(num_blocks, block_size=16, free_order=None):
    h = _vp()
    fo = None
    if free_order is not None:
        fo = np.ascontiguousarray(free_order, dtype=np.int32)
        if fo.shape != (num_blocks,):
            raise ValueError("free_order must have num_blocks entries")
    _check(lib.pkv_pool_create(num_blocks, block_size, _ptr(fo), ctypes.byref(h)), "pkv_pool_create")
    return h


def pkv_pool_destroy(pool):
    _check(lib.pkv_pool_destroy(pool), "pkv_pool_destroy")


def _out_i32(fn, *args):
    v = _i32()
    _check(getattr(lib, fn)(*args, ctypes.byref(v)), fn)
    return v.value


def _out_i64(fn, *args):
    v = _i64()
    _check(getattr(lib, fn)(*args, ctypes.byref(v)), fn)
    return v.value


def pkv_pool_num_free(pool):
    return _out_i32("pkv_pool_num_free", pool)


def pkv_pool_num_blocks(pool):
    return _out_i32("pkv_pool_num_blocks", pool)


def pkv_block_alloc(pool):
    return _out_i32("pkv_block_alloc", pool)


def pkv_block_incref(pool, block):
    _check(lib.pkv_block_incref(pool, block), "pkv_block_incref")


def pkv_block_decref(pool, block):
    _check(lib.pkv_block_decref(pool, block), "pkv_block_decref")


def pkv_block_refcount(pool, block):
    return _out_i32("pkv_block_refcount", pool, block)


def pkv_seq_create(pool):
    return _out_i64("pkv_seq_create", pool)


def pkv_seq_free(pool, seq):
    _check(lib.pkv_seq_free(pool, seq), "pkv_seq_free")


def pkv_seq_fork(pool, parent):
    return _out_i64("pkv_seq_fork", pool, parent)


def pkv_seq_append(pool, seq, n_tokens):
    """Returns (slots int64[n], copy pairs list of (src, dst))."""
    slots = np.empty(max(n_tokens, 1), dtype=np.int64)
    pairs = np.empty(2, dtype=np.int32)
    n = _i32()
    _check(lib.pkv_seq_append(pool, seq, n_tokens, _ptr(slots), _ptr(pairs), ctypes.byref(n)),
           "pkv_seq_append")
    return slots[:n_tokens], [(int(pairs[0]), int(pairs[1]))] if n.value else []


def pkv_seq_append_batch(pool, seqs, n_tokens_each=1, slots_out=None, pairs_out=None):
    """One decode step for many sequences; returns (slots, pairs [n_copies, 2])."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int64)
    n = seqs.shape[0]
    if slots_out is None:
        slots_out = np.empty(max(n * n_tokens_each, 1), dtype=np.int64)
    if pairs_out is None:
        pairs_out = np.empty(max(2 * n, 2), dtype=np.int32)
    nc = _i32()
    _check(lib.pkv_seq_append_batch(pool, _ptr(seqs), n, n_tokens_each, _ptr(slots_out),
                                    _ptr(pairs_out), ctypes.byref(nc)), "pkv_seq_append_batch")
    return slots_out[:n * n_tokens_each], pairs_out[:2 * nc.value].reshape(-1, 2)


def pkv_seq_len(pool, seq):
    return _out_i64("pkv_seq_len", pool, seq)


def pkv_seq_num_blocks(pool, seq):
    return _out_i32("pkv_seq_num_blocks", pool, seq)


def pkv_seq_block_table(pool, seq):
    n = pkv_seq_num_blocks(pool, seq)
    out = np.empty(max(n, 1), dtype=np.int32)
    _check(lib.pkv_seq_block_table(pool, seq, _ptr(out), n), "pkv_seq_block_table")
    return out[:n]


def pkv_build_block_tables(pool, seqs, max_blocks, tables_out=None, lens_out=None):
    """Host int32 tables [n, max_blocks] (-1 padded) and context lengths [n]."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int64)
    n = seqs.shape[0]
    if tables_out is None:
        tables_out = np.empty((n, max_blocks), dtype=np.int32)
    if lens_out is None:
        lens_out = np.empty(n, dtype=np.int32)
    _check(lib.pkv_build_block_tables(pool, _ptr(seqs), n, _ptr(tables_out), max_blocks,
                                      _ptr(lens_out)), "pkv_build_block_tables")
    return tables_out, lens_out


def pkv_debug_fail_after(pool, n_allocs):
    _check(lib.pkv_debug_fail_after(pool, n_allocs), "pkv_debug_fail_after")


def pkv_debug_prefill_drop_copy(tile):
    """Test hook: the tensor-core prefill kernel skips the K copy of key
    tile `tile` (-1: off), so its bounded wait for it runs out."""
    _check(lib.pkv_debug_prefill_drop_copy(int(tile)), "pkv_debug_prefill_drop_copy")


def pkv_prefix_register(pool, seq, tokens):
    """Registers seq's full blocks holding tokens; returns entries added."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = _i32()
    _check(lib.pkv_prefix_register(pool, seq, _ptr(tokens), tokens.shape[0], ctypes.byref(n)),
           "pkv_prefix_register")
    return n.value


def pkv_prefix_match(pool, tokens):
    """New sequence mapped onto the longest cached prefix: (seq, matched tokens)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    seq, m = _i64(), _i32()
    _check(lib.pkv_prefix_match(pool, _ptr(tokens), tokens.shape[0], ctypes.byref(seq),
                                ctypes.byref(m)), "pkv_prefix_match")
    return seq.value, m.value


def pkv_prefix_evict(pool, n_blocks):
    return _out_i32("pkv_prefix_evict", pool, n_blocks)


def pkv_prefix_clear(pool):
    _check(lib.pkv_prefix_clear(pool), "pkv_prefix_clear")


def pkv_prefix_stats(pool):
    """(entries, lookups, matched blocks)."""
    e, l, h = _i64(), _i64(), _i64()
    _check(lib.pkv_prefix_stats(pool, ctypes.byref(e), ctypes.byref(l), ctypes.byref(h)),
           "pkv_prefix_stats")
    return e.value, l.value, h.value


def pkv_decode_workspace_bytes(batch, num_q_heads, head_dim, max_blocks, block_size=16,
                               partition_size=0):
    v = _sz()
    _check(lib.pkv_decode_workspace_bytes(batch, num_q_heads, head_dim, max_blocks, block_size,
                                          partition_size, ctypes.byref(v)),
           "pkv_decode_workspace_bytes")
    return v.value


def pkv_decode_auto_partition_size(batch, num_q_heads, max_blocks, block_size=16):
    return _out_i32("pkv_decode_auto_partition_size", batch, num_q_heads, max_blocks, block_size)


# ------------------------------------------------------------------ device
def pkv_kv_append(k, v, slot_mapping, k_pool, v_pool, stream=None):
    """k, v [T, Hkv, D]; slot_mapping int64 [T]; pools [NB, Hkv, BS, D]."""
    T, Hkv, D = k.shape
    NB, _, BS, _ = k_pool.shape
    _check(lib.pkv_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_pool), _ptr(v_pool),
                             NB, Hkv, D, BS, _dtype_code(k), _stream(stream)), "pkv_kv_append")


def pkv_paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                               workspace=None, partition_size=0, stream=None):
    """q, out [B, Hq, D]; pools [NB, Hkv, BS, D]; tables int32 [B, max_blocks]."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    mb = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D,
        NB, BS, mb, float(scale), _ptr(out), _ptr(workspace), ws_bytes, partition_size,
        _dtype_code(q), _stream(stream)), "pkv_paged_attention_decode")


def pkv_multi_query_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, max_q_len,
                                    block_size=16):
    v = _sz()
    _check(lib.pkv_multi_query_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                               block_size, int(max_q_len), ctypes.byref(v)),
           "pkv_multi_query_workspace_bytes")
    return v.value


def pkv_paged_attention_multi_query(q, q_start, k_pool, v_pool, block_tables, context_lens, scale,
                                    out, max_q_len, workspace=None, stream=None):
    """q, out [T, Hq, D]; q_start int32 [B + 1] (sequence b's queries are rows
    q_start[b] .. q_start[b+1]-1, the last of its context_lens[b] tokens).
    workspace: device bytes (pkv_multi_query_workspace_bytes) for the
    balanced split, or None."""
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    B = q_start.shape[0] - 1
    mb = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_multi_query(
        _ptr(q), _ptr(q_start), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
        B, Hq, Hkv, D, NB, BS, mb, int(max_q_len), float(scale), _ptr(out), _ptr(workspace), ws_bytes,
        _dtype_code(q), _stream(stream)), "pkv_paged_attention_multi_query")


def pkv_paged_attention_decode_append(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                                      context_lens, scale, out, workspace=None, partition_size=0,
                                      stream=None):
    """Fused decode step: write k_new/v_new [B, Hkv, D] at slot_mapping [B]
    and attend over context_lens tokens (the new row being the last)."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool),
        _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D, NB, BS, block_tables.shape[1],
        float(scale), _ptr(out), _ptr(workspace), ws_bytes, partition_size, _dtype_code(q),
        _stream(stream)), "pkv_paged_attention_decode_append")


def pkv_paged_attention_decode_partials(q, k_pool, v_pool, block_tables, context_lens, scale,
                                        workspace, partition_size=0, stream=None):
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    _check(lib.pkv_paged_attention_decode_partials(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D,
        NB, BS, block_tables.shape[1], float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), partition_size, _dtype_code(q),
        _stream(stream)), "pkv_paged_attention_decode_partials")


def pkv_paged_attention_decode_merge(context_lens, max_blocks, workspace, out, block_size=16,
                                     partition_size=0, stream=None):
    B, Hq, D = out.shape
    _check(lib.pkv_paged_attention_decode_merge(
        _ptr(context_lens), B, Hq, D, max_blocks, block_size, partition_size, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _dtype_code(out), _stream(stream)),
        "pkv_paged_attention_decode_merge")


PKV_STATIC_WORKSPACE_BYTES = 16 << 20


def pkv_paged_attention_decode_static_ws(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                                         partition_size=0, stream=None):
    """Decode without a caller workspace: the split-K partials go to a fixed
    array inside the library (PKV_STATIC_WORKSPACE_BYTES per GPU).  For
    callers that cannot allocate device memory on the decode path."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    _check(lib.pkv_paged_attention_decode_static_ws(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D,
        NB, BS, block_tables.shape[1], float(scale), _ptr(out), partition_size, _dtype_code(q),
        _stream(stream)), "pkv_paged_attention_decode_static_ws")


def pkv_kv_append_quant(k, v, slot_mapping, positions, seq_idx, cache, n_sink, qmode,
                        group_size=0, stream=None, window=0):
    """cache: dict with k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, sink_k, sink_v,
    and win_k, win_v [rows, window / block_size + 1, Hkv, block_size, D] when window > 0."""
    T, Hkv, D = k.shape
    kc = cache["k_codes"]
    NB, _, BS, _ = kc.shape
    rows_of = cache.get("sink_k") if cache.get("sink_k") is not None else cache.get("win_k")
    sink_rows = rows_of.shape[0] if rows_of is not None else 0
    _check(lib.pkv_kv_append_quant(
        _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(positions), _ptr(seq_idx), T, _ptr(kc),
        _ptr(cache["k_scale"]), _ptr(cache.get("k_zero")), _ptr(cache["v_codes"]),
        _ptr(cache["v_scale"]), _ptr(cache.get("v_zero")), _ptr(cache.get("sink_k")),
        _ptr(cache.get("sink_v")), n_sink, sink_rows, _ptr(cache.get("win_k")),
        _ptr(cache.get("win_v")), window, NB, Hkv, D, BS, group_size or D,
        _qmode_code(qmode), _dtype_code(k), _stream(stream)), "pkv_kv_append_quant")


def pkv_paged_attention_decode_quant(q, cache, n_sink, block_tables, context_lens, scale, out,
                                     qmode, group_size=0, workspace=None, partition_size=0,
                                     stream=None, window=0):
    B, Hq, D = q.shape
    kc = cache["k_codes"]
    NB, Hkv, BS, _ = kc.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_quant(
        _ptr(q), _ptr(kc), _ptr(cache["k_scale"]), _ptr(cache.get("k_zero")),
        _ptr(cache["v_codes"]), _ptr(cache["v_scale"]), _ptr(cache.get("v_zero")),
        _ptr(cache.get("sink_k")), _ptr(cache.get("sink_v")), n_sink, _ptr(cache.get("win_k")),
        _ptr(cache.get("win_v")), window, _ptr(block_tables),
        _ptr(context_lens), B, Hq, Hkv, D, NB, BS, block_tables.shape[1], group_size or D,
        float(scale), _ptr(out), _ptr(workspace), ws_bytes, partition_size, _qmode_code(qmode),
        _dtype_code(q), _stream(stream)), "pkv_paged_attention_decode_quant")


def pkv_copy_blocks(pools, pairs, stream=None):
    """pools: list of device tensors [NB, ...]; pairs: device int32 [n, 2]."""
    n = pairs.shape[0]
    if n == 0:
        return
    ptrs = (_vp * len(pools))(*[_ptr(p) for p in pools])
    bpb = (_i64 * len(pools))(*[p[0].numel() * p.element_size() for p in pools])
    NB = pools[0].shape[0]
    _check(lib.pkv_copy_blocks(ptrs, bpb, len(pools), _ptr(pairs), n, NB, _stream(stream)),
           "pkv_copy_blocks")


def pkv_device_status(stream=None):
    """Read and clear the device status word; returns the PKV_STATUS_* bits."""
    v = _i32()
    st = lib.pkv_device_status(ctypes.byref(v), _stream(stream))
    if st not in (PKV_OK, -7):
        _check(st, "pkv_device_status")
    return v.value
