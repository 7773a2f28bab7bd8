"""The C-ABI library builds, loads without a GPU, exports every function
include/pa.h declares, and rejects malformed host-visible arguments before
touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_108_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    lib = _lib.lib()
    names = _declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    assert set(names) <= set(_lib.SIGNATURES), "binding lacks a signature"


def test_status_strings_and_version():
    lib = _lib.lib()
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(2) == b"PA_ERR_OOM"
    assert b"sm_103a" in lib.pa_version()


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def _desc(**kw):
    d = dict(num_blocks=32, block_size=16, num_kv_heads=2, head_dim=64, dtype=0)
    d.update(kw)
    return _lib.CacheDesc(**d)


def _decode(desc, num_heads=4, ks=None, vs=None, ws=None, ws_bytes=0, opts=None, out=FAKE):
    return _lib.lib().pa_decode_ex(out, FAKE, FAKE, FAKE, desc, FAKE, 3, FAKE, 4, num_heads,
                                   ctypes.c_float(0.125), ks, vs, ws, ws_bytes,
                                   ctypes.byref(opts) if opts else None, None)


@pytest.mark.parametrize("desc,heads,expect", [
    (_desc(head_dim=96), 4, _lib.PA_ERR_UNSUPPORTED),
    (_desc(block_size=24), 4, _lib.PA_ERR_UNSUPPORTED),
    (_desc(dtype=7), 4, _lib.PA_ERR_INVALID),
    (_desc(num_blocks=0), 4, _lib.PA_ERR_INVALID),
    (_desc(), 5, _lib.PA_ERR_INVALID),          # not a multiple of H_kv
    (_desc(num_kv_heads=1), 3, _lib.PA_ERR_UNSUPPORTED),  # group 3
    (_desc(dtype=1), 4, _lib.PA_ERR_INVALID),   # fp8 without scales
])
def test_decode_rejects_bad_arguments(desc, heads, expect):
    assert _decode(desc, heads) == expect
    assert _lib.lib().pa_last_error().decode().startswith("pa_decode")


def test_decode_rejects_bad_partition_and_null_output():
    opts = _lib.DecodeOpts(96, 0)
    assert _decode(_desc(), opts=opts) == _lib.PA_ERR_INVALID
    assert _decode(_desc(), out=None) == _lib.PA_ERR_INVALID
    assert _decode(_desc(), opts=_lib.DecodeOpts(0, 9)) == _lib.PA_ERR_UNSUPPORTED


def test_write_and_copy_reject_bad_arguments():
    lib = _lib.lib()
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, _desc(dtype=1), FAKE, 4, None, None,
                                    None) == _lib.PA_ERR_INVALID
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, _desc(), FAKE, -1, None, None,
                                    None) == _lib.PA_ERR_INVALID
    assert lib.pa_reshape_and_cache(None, None, None, None, _desc(), None, 0, None, None,
                                    None) == _lib.PA_OK  # nothing to do
    assert lib.pa_copy_blocks(FAKE, FAKE, _desc(), None, 3, None) == _lib.PA_ERR_INVALID
    assert lib.pa_copy_blocks(None, None, _desc(), None, 0, None) == _lib.PA_OK


def test_workspace_size():
    lib = _lib.lib()
    # head_dim 64 (SIMT kernel only): contexts within one partition need none
    assert lib.pa_decode_workspace_size(64, 32, 64, 16, 16) == 0
    # 64 seqs x 32 heads x 14 partitions of 256 tokens (3584 tokens max)
    n = lib.pa_decode_workspace_size(64, 32, 64, 224, 16)
    parts = -(-224 * 16 // 256)
    o = 64 * 32 * parts * 64 * 4
    assert n == -(-o // 256) * 256 + 64 * 32 * parts * 8
    assert lib.pa_decode_workspace_size_ex(64, 32, 128, 224, 16, 96) == 0  # bad partition
    # head_dim 128 also covers the tensor-core kernel's per-CTA partials
    n128 = lib.pa_decode_workspace_size(64, 32, 128, 224, 16)
    assert n128 >= 2 * o and n128 >= 64 * 32 * 28 * 128 * 4 // 28
