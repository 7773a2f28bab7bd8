"""pa_decode_noalloc: the decode entry point that keeps its split-K scratch in
a fixed array inside the library, for callers that cannot hand out device
memory at the call site (for example a plugin whose host application owns
every device allocation, or a serving loop that must not call cudaMalloc
because it can synchronise the device).

Its output must match pa_decode's (the entry point with a caller workspace)
within the tolerance the parity tests use, on two calls in a row (the second
call finds the first call's leftovers in the shared array).  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import _lib, ops, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _call_noalloc(out, dev, w):
    lib = _lib.lib()
    desc = ops.cache_desc(dev["k_cache"])
    return lib.pa_decode_noalloc(
        out.data_ptr(), dev["q"].data_ptr(), dev["k_cache"].data_ptr(),
        dev["v_cache"].data_ptr(), desc, dev["bt"].data_ptr(), int(dev["bt"].shape[1]),
        dev["cl"].data_ptr(), w.num_seqs, w.num_heads, ctypes.c_float(w.scale), None, None,
        torch.cuda.current_stream().cuda_stream)


@requires_gpu
@pytest.mark.parametrize("make", [synth.llama8b, synth.longctx], ids=["llama8b", "longctx"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(make):
    w = make()
    got = harness.product_step(w)  # caches written, reference decode through pa_decode
    ref = got["out"]
    dev = got["dev"]
    for call in range(2):
        out = torch.full_like(dev["q"], float("nan"))
        st = _call_noalloc(out, dev, w)
        assert st == _lib.PA_OK, _lib.lib().pa_last_error().decode()
        torch.cuda.synchronize()
        res = out.float().cpu().numpy().astype(np.float64)
        harness.assert_close(res, ref, fp8=False)


@requires_gpu
def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib.lib()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check comes first
    desc = _lib.CacheDesc(num_blocks=1 << 20, block_size=16, num_kv_heads=8, head_dim=128, dtype=0)
    st = lib.pa_decode_noalloc(fake, fake, fake, fake, desc, fake, 1 << 16, fake, 8192, 64,
                               ctypes.c_float(0.1), None, None, None)
    assert st == _lib.PA_ERR_UNSUPPORTED
    assert "built-in scratch" in lib.pa_last_error().decode()
