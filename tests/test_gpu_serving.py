"""Copy-on-write serving step: groups of 8 sequences share a prefix through
ref-counted blocks, every sequence's first divergent write goes through the
pool's copy-on-write decision ("4.6 PagedAttention & KV-Cache Memory
Management", section "Copy-on-write for shared prefixes"), the device copies
run with pa_copy_blocks, then the suffix and the step's new tokens are
written and all sequences decode.

With a 1024-token prefix and block size 16 the shared prefix ends on a block
boundary, so the first divergent write opens a fresh block and no copy is
needed (the literal workload: 0 pairs); with a 1000-token prefix the last
shared block is half full and the first 7 writers of each group copy it
(the 8th finds ref count 1 and writes in place).

Tables, copy pairs, slots and both caches must equal the oracle's exactly;
outputs must meet the bf16 tolerance."""
import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _run(mix, kernel=0):
    nb = harness.serving_pool_size(mix)
    data = synth.serving_data(mix, nb, harness.serving_unique_tokens(mix))
    got = harness.serving_product(mix, data, nb, kernel=kernel)
    ref = harness.serving_oracle(mix, data, nb)
    if kernel != 1:  # word 0 is the tensor-core kernel's error word
        assert got["err"] == 0
    assert np.array_equal(got["tables"], ref["tables"])
    assert np.array_equal(got["pairs"], ref["pairs"])
    for a, b in zip(got["slots"], ref["slots"]):
        assert np.array_equal(a, b)
    assert np.array_equal(got["k_cache"], ref["k_cache"])
    assert np.array_equal(got["v_cache"], ref["v_cache"])
    harness.assert_close(got["out"], ref["out"], False)
    return got


@requires_gpu
def test_serving_mix_shared_prefix_on_block_boundary():
    got = _run(synth.serving(prefix_len=1024))
    assert got["pairs"].shape[0] == 0  # 1024 % 16 == 0: no shared partial block


@requires_gpu
def test_serving_mix_copy_on_write_partial_prefix_block():
    mix = synth.serving(prefix_len=1000)
    got = _run(mix)
    assert got["pairs"].shape[0] == mix.num_groups * (mix.group_size - 1)


@requires_gpu
def test_serving_mix_small_simt_kernel():
    _run(synth.serving(num_groups=4, prefix_len=1000, max_suffix=300), kernel=1)
