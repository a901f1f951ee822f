"""Oracle KV-byte accounting (the roofline numerator for decode).

Test infrastructure only (see ``oracle/__init__``).

Source: "SGLang 深度拆解" (chenxutan.com/d/5669.html) §4.3: the KV cache of
one token is 2 (K and V) x layers x KV heads x head_dim x bytes per element;
the page works it for Llama-3.1-70B (80 layers, 8 KV heads, head_dim 128,
bf16) as 327,680 bytes per token and 1.25 GB for a 4096-token prompt.
"""


def kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes, num_layers=1):
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def unique_kv_bytes(groups, num_kv_heads, head_dim, dtype_bytes):
    """Bytes of K and V a shared-aware decode must read: every segment once."""
    tokens = sum(int(e) - int(b) for b, e in zip(groups["seg_begin"], groups["seg_end"]))
    return tokens * kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes)


def unshared_kv_bytes(seq_lens, num_kv_heads, head_dim, dtype_bytes):
    """Bytes read when every request re-reads its whole context."""
    return int(sum(int(x) for x in seq_lens)) * kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes)
