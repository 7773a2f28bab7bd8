"""GPU parity of the tensor-core prefill tiles (pa_varlen_attention_ex
method 2) against the fp64 varlen oracle, with the bf16 decode tolerance.

A tile holds 128 / G new tokens of one request for one KV head; the cases
put request lengths on both sides of tile and 128-key chunk boundaries, mix
chunked prefill (a context before the new tokens), full prefill (none) and
single-token requests, and cover every GQA group the tiles serve, several
block sizes, long prefills, many small requests, requests without new
tokens, requests whose count exceeds their context (zero rows), the
kernel's error word, e4m3 caches (the e4m3 tolerance, against the oracle on
the dequantised cache), and the automatic choice on a step that mixes one
prefill with single-token decodes."""
import numpy as np
import pytest
import torch

from oracle import varlen
from paged_kv_cache_108_gb300 import ops
from paged_kv_cache_108_gb300._lib import PaError
from tests import harness
from tests.test_gpu_varlen import _setup

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

TILES = 2


def _run(c, scale, method=TILES):
    q = harness.to_dev_bits(c["q"], "bf16", "cuda")
    out = torch.empty_like(q)
    n = ops.varlen_workspace_size(q.shape[0], c["H"], c["d"], c["tables"].shape[1],
                                  c["kc"].shape[1])
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ws.random_(0, 256)
    ws[:4] = 0
    ops.varlen_attention(out, q, c["kc"], c["vc"], torch.from_numpy(c["tables"]).cuda(),
                         torch.from_numpy(c["seq_lens"]).cuda(), torch.from_numpy(c["qsl"]).cuda(),
                         scale, c["ks"], c["vs"], workspace=ws, method=method)
    torch.cuda.synchronize()
    if method == TILES:
        assert int(ws[:4].view(torch.int32).item()) == 0, "prefill kernel error word"
    return out.float().cpu().numpy().astype(np.float64)


def _check(c, scale, method=TILES):
    got = _run(c, scale, method)
    ref = varlen.varlen_attention(c["q"], harness.bits_from_dev(c["kc"]),
                                  harness.bits_from_dev(c["vc"]), c["tables"], c["seq_lens"],
                                  c["qsl"], scale, c["kscale"], c["vscale"])
    harness.assert_close(got, ref, c["kv"] == "fp8")
    assert np.isfinite(got).all()
    return got


@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 16), (16, 8), (64, 8)])
def test_tiles_mixed_step(hq, hkv):
    # G = 4, 1, 2, 8: tiles of 32, 128, 64, 16 tokens; lengths around them
    g = hq // hkv
    mq = 128 // g
    seq = [700, 300, 1500, 129, mq + 5, 2 * mq, 40]
    new = [200, 300, 1, 129, mq + 1, mq - 1, 40]
    c = _setup(seq, new, hq, hkv, 128, 16, seed=100 + g)
    _check(c, 128 ** -0.5)


@requires_gpu
@pytest.mark.parametrize("block_size", [8, 16, 64, 256])
def test_tiles_block_sizes(block_size):
    seq = [1000, 257, 520, 64]
    new = [333, 257, 100, 64]
    c = _setup(seq, new, 32, 8, 128, block_size, seed=110)
    _check(c, 0.09)


@requires_gpu
def test_tiles_long_prefill_and_long_context_chunk():
    # a 2048-token full prefill and a 512-token chunk after 3000 cached tokens
    c = _setup([2048, 3512], [2048, 512], 32, 8, 128, 16, seed=111)
    _check(c, 128 ** -0.5)


@requires_gpu
def test_tiles_many_small_requests_and_empty_ones():
    rng = np.random.default_rng(112)
    new = [int(x) for x in rng.integers(0, 40, size=200)]
    seq = [n + int(x) for n, x in zip(new, rng.integers(0, 300, size=200))]
    seq = [max(s, 1) for s in seq]
    c = _setup(seq, new, 32, 8, 128, 16, seed=113)
    _check(c, 0.1)


@requires_gpu
def test_tiles_zero_rows_when_new_tokens_exceed_the_context():
    c = _setup([50, 60, 90], [20, 0, 33], 32, 8, 128, 16, seed=114)
    c["seq_lens"][2] = 30  # 33 new tokens, 30 in the context: its rows are zero
    got = _run(c, 0.1)
    assert not got[20:].any()
    ref = varlen.varlen_attention(c["q"][:20], harness.bits_from_dev(c["kc"]),
                                  harness.bits_from_dev(c["vc"]), c["tables"][:1],
                                  c["seq_lens"][:1], c["qsl"][:2], 0.1)
    harness.assert_close(got[:20], ref, False)


@requires_gpu
def test_tiles_agree_with_per_token_decodes():
    c = _setup([900, 450, 77], [300, 450, 20], 32, 8, 128, 16, seed=115)
    tiles = _check(c, 0.08)
    per_token = _run(c, 0.08, method=1)
    harness.assert_close(tiles, per_token, False)


@requires_gpu
def test_tiles_repeatable_bit_for_bit():
    c = _setup([1200, 640], [600, 640], 32, 8, 128, 16, seed=116)
    a = _run(c, 0.09)
    b = _run(c, 0.09)
    assert np.array_equal(a, b)


@requires_gpu
@pytest.mark.parametrize("what", ["head_dim", "block4", "group16"])
def test_tiles_refuse_shapes_they_do_not_serve(what):
    if what == "head_dim":
        c = _setup([40, 20], [10, 20], 8, 2, 64, 16, seed=117)
    elif what == "block4":
        c = _setup([40, 20], [10, 20], 32, 8, 128, 4, seed=117)
    else:
        c = _setup([40, 20], [10, 20], 64, 4, 128, 16, seed=117)
    with pytest.raises(PaError, match="prefill tiles"):
        _run(c, 0.1)


@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 16)])
def test_automatic_choice_on_a_step_mixing_one_prefill_with_decodes(hq, hkv):
    # one 700-token chunked prefill among 40 single-token decodes (average
    # under 16 new tokens per request): the prefill goes to the tiles, the
    # decodes to the decode kernels, in one call
    rng = np.random.default_rng(120)
    seq = [1500] + [int(x) for x in rng.integers(1, 4000, size=40)]
    new = [700] + [1] * 40
    c = _setup(seq, new, hq, hkv, 128, 16, seed=121)
    got = _check(c, 128 ** -0.5, method=0)
    per_token = _run(c, 128 ** -0.5, method=1)
    harness.assert_close(got, per_token, False)


# ---- e4m3 cache: kind::f8f6f4 tiles, q and P split into e4m3 parts ----

@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 16), (16, 8), (64, 8)])
def test_tiles_fp8_mixed_step(hq, hkv):
    g = hq // hkv
    mq = 128 // g
    seq = [700, 300, 1500, 129, mq + 5, 2 * mq, 40]
    new = [200, 300, 1, 129, mq + 1, mq - 1, 40]
    c = _setup(seq, new, hq, hkv, 128, 16, "fp8", seed=130 + g)
    _check(c, 128 ** -0.5)


@requires_gpu
@pytest.mark.parametrize("block_size", [8, 64, 256])
def test_tiles_fp8_block_sizes_and_long_chunks(block_size):
    c = _setup([2048, 3512, 257], [2048, 512, 257], 32, 8, 128, block_size, "fp8",
               seed=140 + block_size)
    _check(c, 128 ** -0.5)


@requires_gpu
def test_tiles_fp8_query_magnitudes_and_per_token_agreement():
    # rows of very different size: each row gets its own power-of-two scale
    c = _setup([900, 450, 77], [300, 450, 20], 32, 8, 128, 16, "fp8", seed=150)
    q = c["q"].astype(np.uint32) << 16
    f = q.view(np.float32)
    f[::3] *= np.float32(40.0)
    f[1::3] *= np.float32(1e-3)
    c["q"] = (f.view(np.uint32) >> 16).astype(np.uint16)
    tiles = _check(c, 0.08)
    per_token = _run(c, 0.08, method=1)
    harness.assert_close(tiles, per_token, True)


@requires_gpu
def test_tiles_fp8_repeatable_bit_for_bit():
    c = _setup([1200, 640], [600, 640], 32, 8, 128, 16, "fp8", seed=151)
    a = _run(c, 0.09)
    b = _run(c, 0.09)
    assert np.array_equal(a, b)


@requires_gpu
def test_automatic_choice_fp8_mixed_step():
    rng = np.random.default_rng(160)
    seq = [1500] + [int(x) for x in rng.integers(1, 4000, size=30)]
    new = [600] + [1] * 30
    c = _setup(seq, new, 32, 8, 128, 16, "fp8", seed=161)
    _check(c, 128 ** -0.5, method=0)
