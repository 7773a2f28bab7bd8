"""KV-size closed form and utilisation estimator -- TEST INFRASTRUCTURE.

* ``kv_cache_bytes``: Bytes = 2 * L * H_kv * d_h * s * b (times the batch).
  "4.6 PagedAttention & KV-Cache Memory Management" (llm-stack-book), section
  "The size formula"; "PagedAttention - Explained" (mohdvasim.com), section
  "Memory Consumption Formula" and Appendix A.
* ``utilisation``: tokens used over tokens reserved, either per request at
  ``max_len`` (contiguous reservation) or rounded up to whole blocks (paging).
  "Paged KV cache" (ai-infra-handbooks), section "Why paging".
"""
from __future__ import annotations

import math


def kv_cache_bytes(num_layers: int, num_kv_heads: int, head_dim: int,
                   seq_len: int, bytes_per_elem: int = 2, batch: int = 1) -> int:
    """Exact KV bytes; the leading 2 is K and V."""
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem * seq_len * batch


def utilisation(lengths, block_size: int | None = None,
                max_len: int | None = None) -> float:
    """Fraction of reserved token slots that hold a token.

    ``max_len`` given: every request reserves ``max_len`` slots.
    ``block_size`` given: every request reserves ceil(len / B) * B slots."""
    used = sum(lengths)
    if max_len is not None:
        return used / (len(lengths) * max_len)
    reserved = sum(math.ceil(n / block_size) * block_size for n in lengths)
    return used / reserved
