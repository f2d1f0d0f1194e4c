"""KV-cache byte accounting (test infrastructure; see ``oracle/__init__``).

The KV-cache equation of "The 8GB VRAM Breakthrough", §2 "First-Principles
Math": total bytes = 2 (K and V) x layers x KV heads x head dim x sequence
length x batch x bytes per element.  The quantised footprints follow §4
"Dynamic KV-Cache Quantization": FP8 stores one byte per element; group-wise
INT4 stores half a byte per element plus an fp16 scale and an fp16 zero point
per group.
"""

GiB = 1 << 30
KiB = 1 << 10


def kv_cache_bytes(n_layers, n_kv_heads, d_head, s_seq, batch, sizeof_dtype):
    """The KV-cache equation (§2): 2 * L * H_kv * d * s * b * sizeof."""
    return 2 * n_layers * n_kv_heads * d_head * s_seq * batch * sizeof_dtype


def kv_bytes_per_token(n_layers, n_kv_heads, d_head, sizeof_dtype):
    """Bytes one token adds to the cache of one sequence (§2, s = b = 1)."""
    return kv_cache_bytes(n_layers, n_kv_heads, d_head, 1, 1, sizeof_dtype)


def int4_group_bytes(group_size):
    """Bytes for one INT4 group: packed nibbles + fp16 s + fp16 z (§4)."""
    assert group_size % 2 == 0
    return group_size * 4 // 8 + 2 + 2


def int4_bytes_per_token(n_layers, n_kv_heads, d_head, group_size):
    """Group-wise INT4 bytes per token across the whole model (§4)."""
    elements = 2 * n_layers * n_kv_heads * d_head
    assert elements % group_size == 0
    return elements // group_size * int4_group_bytes(group_size)


def fp8_code_bytes_per_token(n_layers, n_kv_heads, d_head):
    """FP8 E4M3 code bytes per token, scales not counted (the §4 figure)."""
    return 2 * n_layers * n_kv_heads * d_head


def fp8_bytes_per_token_per_layer_with_scales(n_kv_heads, d_head):
    """FP8 codes plus one fp16 scale per (token, KV head), K and V, one layer."""
    return 2 * n_kv_heads * (d_head + 2)


def int4_bytes_per_token_per_layer(n_kv_heads, d_head, group_size):
    """INT4 codes plus fp16 scale/zero per group, K and V, one layer."""
    return 2 * n_kv_heads * (d_head // group_size) * int4_group_bytes(group_size)
