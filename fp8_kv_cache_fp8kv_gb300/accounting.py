"""Byte and flop accounting for the fp8 decode path (host-side arithmetic).

bytes_per_token follows the KV sizing formula on gpusmith.com, "FP8 KV Cache
Quantization: Capacity Gains and Accuracy Risk", section "Why the KV cache
sets long-context capacity": 2 (K and V) x layers x kv heads x head_dim x
bytes per element, with 1 byte per element for E4M3 and 2 for bf16 (section
"What FP8 KV changes").  The decode-attention arithmetic intensity of
2g flop/byte with fp8 is the phantomic12 record's "Arithmetic intensity"
paragraph (g flop/byte with bf16, doubled by halving the bytes).
"""
from __future__ import annotations

BF16_BYTES = 2
FP8_BYTES = 1


def bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                    bytes_per_element: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_element


def attended(L: int, window: int) -> int:
    """Number of keys a query of a length-L sequence attends (window<=0: all)."""
    L = max(0, int(L))
    return min(L, window) if window > 0 else L


def decode_bytes(seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 window: int = 0, block_size: int = 16) -> int:
    """Algorithmic HBM bytes of one paged decode call: every attended K and V
    element once (1 byte each), q and out once (bf16), and the block-table
    entries of the attended pages (int32)."""
    kv = 0
    pages = 0
    for L in seq_lens:
        n = attended(L, window)
        kv += 2 * num_kv_heads * n * head_dim * FP8_BYTES
        if n > 0:
            first = (int(L) - n) // block_size
            last = (int(L) - 1) // block_size
            pages += last - first + 1
    B = len(list(seq_lens))
    qo = 2 * B * num_q_heads * head_dim * BF16_BYTES
    return kv + qo + 4 * pages


def decode_flops(seq_lens, num_q_heads: int, head_dim: int, window: int = 0) -> int:
    """4*Hq*d flops per attended key: q.k and p*v, a multiply and an add each."""
    return sum(4 * num_q_heads * head_dim * attended(L, window) for L in seq_lens)


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int) -> int:
    """quant_append: read bf16 K and V rows, write fp8 K and V rows, read the
    int64 slot of each token."""
    elems = 2 * num_tokens * num_kv_heads * head_dim
    return elems * (BF16_BYTES + FP8_BYTES) + 8 * num_tokens
