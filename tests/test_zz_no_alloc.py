"""pa_decode_noalloc: the decode entry point that keeps its split-K scratch in
a fixed array inside the library, for callers that cannot hand out device
memory at the call site (for example a plugin whose host application owns
every device allocation, or a serving loop that must not call cudaMalloc
because it can synchronise the device).

Its output must match pa_decode's (the entry point with a caller workspace)
within the tolerance the parity tests use, on two calls in a row (the second
call finds the first call's leftovers in the shared array), on each kernel
the automatic choice can take: the per-head tensor-core kernel (the batch-64
layer, long contexts), the SIMT kernel with split-K partitions longer than
256 tokens because the array caps the partials (head_dim 64, one 32K-token
sequence), and the head-packed kernel (an MHA batch with many units).  The
status word reads zero after good calls, reports an out-of-range block id
(which the tensor-core kernels replace by block 0), and is cleared by the
read.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import _lib, ops, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _call_noalloc(out, dev, w, bt=None):
    lib = _lib.lib()
    desc = ops.cache_desc(dev["k_cache"])
    bt = dev["bt"] if bt is None else bt
    return lib.pa_decode_noalloc(
        out.data_ptr(), dev["q"].data_ptr(), dev["k_cache"].data_ptr(),
        dev["v_cache"].data_ptr(), desc, bt.data_ptr(), int(bt.shape[1]),
        dev["cl"].data_ptr(), w.num_seqs, w.num_heads, ctypes.c_float(w.scale), None, None,
        torch.cuda.current_stream().cuda_stream)


def _read_status():
    """The status word, read (and cleared) through pa_decode_noalloc_error."""
    code = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = _lib.lib().pa_decode_noalloc_error(code.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PA_OK, _lib.lib().pa_last_error().decode()
    torch.cuda.synchronize()
    return int(code.item())


def _two_calls_match(w, ref, dev):
    for call in range(2):
        out = torch.full_like(dev["q"], float("nan"))
        st = _call_noalloc(out, dev, w)
        assert st == _lib.PA_OK, _lib.lib().pa_last_error().decode()
        torch.cuda.synchronize()
        res = out.float().cpu().numpy().astype(np.float64)
        harness.assert_close(res, ref, fp8=False)
    return res


@requires_gpu
@pytest.mark.parametrize("make", [synth.llama8b, synth.longctx], ids=["llama8b", "longctx"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(make):
    w = make()
    got = harness.product_step(w)  # caches written, reference decode through pa_decode
    _read_status()                 # start from a clear word whatever ran before
    _two_calls_match(w, got["out"], got["dev"])
    assert _read_status() == 0


@requires_gpu
def test_noalloc_simt_kernel_with_partitions_capped_by_the_array():
    # head_dim 64 takes the SIMT kernel; a 32K-token table row makes 256-token
    # partitions need 64 MiB of partials, so the array forces longer ones
    lengths = [32768] + [int(x) for x in np.random.default_rng(7).integers(1, 3000, size=63)]
    w = synth.make("noalloc-simt", lengths, 32, 8, 64, 16, seed=4242)
    need256 = _lib.lib().pa_decode_workspace_size_ex(w.num_seqs, w.num_heads, w.head_dim,
                                                     w.max_blocks, w.block_size, 256)
    assert need256 > _lib.PA_DECODE_NOALLOC_SCRATCH_BYTES
    got = harness.product_step(w)
    res = _two_calls_match(w, got["out"], got["dev"])
    harness.assert_close(res, harness.oracle_step(w)["out"], fp8=False)


@requires_gpu
def test_noalloc_head_packed_kernel_on_an_mha_batch():
    # 48 MHA sequences = 96 head-packed units, enough for the automatic choice
    lengths = [int(x) for x in np.random.default_rng(8).integers(64, 600, size=48)]
    w = synth.make("noalloc-hp", lengths, 32, 32, 128, 16, seed=4343)
    got = harness.product_step(w, kernel=3)
    res = _two_calls_match(w, got["out"], got["dev"])
    assert np.array_equal(res, got["out"]), "expected the head-packed kernel's exact output"
    harness.assert_close(res, harness.oracle_step(w)["out"], fp8=False)
    assert _read_status() == 0


@requires_gpu
def test_noalloc_status_word_reports_an_out_of_range_block_id():
    w = synth.llama8b(batch=8)
    got = harness.product_step(w)
    dev = got["dev"]
    _read_status()
    out = torch.empty_like(dev["q"])
    assert _call_noalloc(out, dev, w) == _lib.PA_OK
    assert _read_status() == 0
    bad = dev["bt"].clone()
    bad[0, 0] = w.num_blocks + 7   # the kernel loads block 0 instead and records code 3
    assert _call_noalloc(out, dev, w, bt=bad) == _lib.PA_OK
    assert _read_status() == 3
    assert _read_status() == 0     # the read cleared it
    assert _call_noalloc(out, dev, w) == _lib.PA_OK
    torch.cuda.synchronize()
    harness.assert_close(out.float().cpu().numpy().astype(np.float64), got["out"], fp8=False)
    assert _read_status() == 0


@requires_gpu
def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib.lib()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check comes first
    desc = _lib.CacheDesc(num_blocks=1 << 20, block_size=16, num_kv_heads=8, head_dim=128, dtype=0)
    st = lib.pa_decode_noalloc(fake, fake, fake, fake, desc, fake, 1 << 16, fake, 8192, 64,
                               ctypes.c_float(0.1), None, None, None)
    assert st == _lib.PA_ERR_UNSUPPORTED
    assert "built-in scratch" in lib.pa_last_error().decode()
