"""The Python binding refuses shapes the C ABI cannot check through its raw
pointers (one table row and length per sequence, one key/value row per
slot, q's head_dim), before any device work: a wrong size would otherwise
make a kernel read past a buffer."""
import pytest
import torch

from paged_kv_cache_108_gb300 import ops

H, HKV, D, B, NB = 32, 8, 128, 16, 10


def _cache():
    return (torch.zeros(NB, B, HKV, D, dtype=torch.bfloat16),
            torch.zeros(NB, B, HKV, D, dtype=torch.bfloat16))


def test_cache_write_needs_one_key_and_value_row_per_slot():
    kc, vc = _cache()
    slots = torch.zeros(4, dtype=torch.int32)
    k = torch.zeros(4, HKV, D, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="one row per slot"):
        ops.reshape_and_cache(k, torch.zeros(1, HKV, D, dtype=torch.bfloat16), kc, vc, slots)
    with pytest.raises(ValueError, match="one row per slot"):
        ops.reshape_and_cache(torch.zeros(4, HKV, 64, dtype=torch.bfloat16),
                              torch.zeros(4, HKV, 64, dtype=torch.bfloat16), kc, vc, slots)


def test_decode_needs_one_length_and_table_row_per_sequence():
    kc, vc = _cache()
    q = torch.zeros(3, H, D, dtype=torch.bfloat16)
    out = torch.empty_like(q)
    with pytest.raises(ValueError, match="context_lens needs 3"):
        ops.decode(out, q, kc, vc, torch.zeros(3, 4, dtype=torch.int32),
                   torch.zeros(2, dtype=torch.int32), 0.1)
    with pytest.raises(ValueError, match="block_tables"):
        ops.decode(out, q, kc, vc, torch.zeros(2, 4, dtype=torch.int32),
                   torch.zeros(3, dtype=torch.int32), 0.1)
    q64 = torch.zeros(3, H, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="head_dim"):
        ops.decode(torch.empty_like(q64), q64, kc, vc, torch.zeros(3, 4, dtype=torch.int32),
                   torch.zeros(3, dtype=torch.int32), 0.1)


def test_varlen_multi_and_shared_prefix_check_their_metadata():
    kc, vc = _cache()
    q = torch.zeros(6, H, D, dtype=torch.bfloat16)
    out = torch.empty_like(q)
    with pytest.raises(ValueError, match="block_tables"):
        ops.varlen_attention(out, q, kc, vc, torch.zeros(3, 4, dtype=torch.int32),
                             torch.zeros(2, dtype=torch.int32),
                             torch.tensor([0, 3, 6], dtype=torch.int32), 0.1)
    with pytest.raises(ValueError, match="block_tables"):
        ops.decode_multi(out, q, kc, vc, torch.zeros(2, 4, dtype=torch.int32),
                         torch.zeros(3, dtype=torch.int32), 2, 0.1)
    q3 = torch.zeros(3, H, D, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="context_lens needs 3"):
        ops.decode_shared_prefix(torch.empty_like(q3), q3, kc, vc,
                                 torch.zeros(3, 4, dtype=torch.int32),
                                 torch.zeros(4, dtype=torch.int32), 3, 0.1)


def test_write_and_decode_checks_both_halves():
    kc, vc = _cache()
    q = torch.zeros(2, H, D, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="one row per slot"):
        ops.write_and_decode(torch.zeros(2, HKV, D, dtype=torch.bfloat16),
                             torch.zeros(1, HKV, D, dtype=torch.bfloat16),
                             torch.zeros(2, dtype=torch.int32), torch.empty_like(q), q, kc, vc,
                             torch.zeros(2, 4, dtype=torch.int32),
                             torch.zeros(2, dtype=torch.int32), 0.1)
