"""Oracle KV-byte accounting (the roofline numerator for decode).

Test infrastructure only (see ``oracle/__init__``).

Source: "SGLang 深度拆解" (chenxutan.com/d/5669.html) §4.3: the KV cache of
one token is 2 (K and V) x layers x KV heads x head_dim x bytes per element;
the page works it for Llama-3.1-70B (80 layers, 8 KV heads, head_dim 128,
bf16) as 327,680 bytes per token and 1.25 GB for a 4096-token prompt.
The CS349D lecture-16 notes §5.1 "DP attention": MLA stores per token and
layer ONE row (a 512-dimensional latent plus a 64-dimensional position part,
read as keys and, its latent part, as values): 1,152 bytes for
DeepSeek-Coder-V2, about 69 KB over its 60 layers against 246 KB for a
60-layer GQA model with 8 KV heads.
"""


def kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes, num_layers=1):
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def mla_kv_bytes_per_token(latent_dim, rope_dim, dtype_bytes, num_layers=1):
    return num_layers * (latent_dim + rope_dim) * dtype_bytes


def unique_kv_bytes(groups, num_kv_heads, head_dim, dtype_bytes):
    """Bytes of K and V a shared-aware decode must read: every segment once."""
    tokens = sum(int(e) - int(b) for b, e in zip(groups["seg_begin"], groups["seg_end"]))
    return tokens * kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes)


def unshared_kv_bytes(seq_lens, num_kv_heads, head_dim, dtype_bytes):
    """Bytes read when every request re-reads its whole context."""
    return int(sum(int(x) for x in seq_lens)) * kv_bytes_per_token(num_kv_heads, head_dim, dtype_bytes)
