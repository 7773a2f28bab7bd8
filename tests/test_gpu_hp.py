"""GPU parity of the head-packed tensor-core decode kernel (pa_decode kernel 3:
one TMA copy per block for 8 or 16 KV heads, the heads' query heads as MMA
columns) against the fp64 oracle, and agreement with the per-head kernel.

Same bars as tests/test_gpu_parity.py; the kernel's error word (workspace
word 0: an expired bounded wait or an out-of-range block id) must stay zero.
The cases cover several tiles and ragged tails per unit, units split over
many CTAs (long contexts: merges of dozens of pieces), both tile shapes
(8 heads x 16 tokens for GQA groups 2 and 4, 16 heads x 8 tokens for MHA),
block sizes that hold one or several chunks, blocks smaller than a chunk
(token-major tiles: a chunk of whole blocks, one copy per block, blocks past
the context end not copied), and empty sequences."""
import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import ops, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

HP = 3


def _check(w, **kw):
    got = harness.product_step(w, kernel=HP, **kw)
    assert got["err"] == 0, f"head-packed kernel error word {got['err']}"
    ref = harness.oracle_step(w)
    assert np.array_equal(got["k_cache"], ref["k_cache"])
    assert np.array_equal(got["v_cache"], ref["v_cache"])
    return harness.assert_close(got["out"], ref["out"], w.kv_dtype == "fp8"), got, ref


@requires_gpu
def test_hp_small_length_mix():
    # lengths around the 16-token chunk and the CTA split points
    lens = [1, 2, 15, 16, 17, 31, 33, 127, 128, 129, 255, 257, 1000, 3]
    w = synth.make("hp-small", lens, 32, 8, 128, 16, seed=131)
    _check(w)


@requires_gpu
def test_hp_llama8b_batch64():
    _check(synth.llama8b())


@requires_gpu
def test_hp_long_context_many_pieces():
    # 8 sequences up to 131072 tokens: each unit spans many CTAs
    _check(synth.longctx())


@requires_gpu
@pytest.mark.parametrize("block_size", [16, 64, 256])
def test_hp_block_sizes(block_size):
    _check(synth.sweep(block_size, "bf16"))


@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (64, 16), (16, 16), (32, 32)])
def test_hp_head_groups(hq, hkv):
    # groups 2 and 4: 8 KV heads x 16 tokens per tile; group 1: 16 x 8
    lens = [3, 130, 700, 2000, 64, 1, 9]
    w = synth.make(f"hp-heads-{hq}-{hkv}", lens, hq, hkv, 128, 16, seed=141)
    _check(w)


@requires_gpu
def test_hp_mha_block8():
    # group 1 tiles hold 8 tokens: a block of 8 is one chunk
    lens = [1, 7, 8, 9, 300, 1111]
    w = synth.make("hp-mha-b8", lens, 32, 32, 128, 8, seed=143)
    _check(w)


@requires_gpu
def test_hp_empty_sequences():
    w = synth.make("hp-empty", [0, 300, 0, 5, 0], 32, 8, 128, 16, seed=145)
    _, got, _ = _check(w)
    assert np.all(got["out"][0] == 0) and np.all(got["out"][2] == 0) and np.all(got["out"][4] == 0)


@requires_gpu
def test_hp_many_short_sequences():
    # more units than CTAs, most of them whole in one CTA
    rng = np.random.default_rng(147)
    lens = [int(x) for x in rng.integers(1, 200, size=700)]
    w = synth.make("hp-many", lens, 32, 8, 128, 16, seed=149, num_blocks=12000)
    _check(w)


@requires_gpu
def test_hp_agrees_with_per_head_kernel_and_is_permutation_invariant():
    lens = synth.llama8b_lengths(16)
    a = synth.make("hp-perm-a", lens, 32, 8, 128, 16, seed=151, num_blocks=2000)
    b = synth.make("hp-perm-b", lens, 32, 8, 128, 16, seed=151, num_blocks=2000)
    rng = np.random.default_rng(153)
    perm = rng.permutation(2000).astype(np.int32)
    mask = np.zeros_like(a.block_tables, dtype=bool)
    for i, n in enumerate(lens):
        mask[i, :-(-n // 16)] = True
    b.block_tables = np.where(mask, perm[a.block_tables], 0).astype(np.int32)
    oa = harness.product_step(a, kernel=HP)
    ob = harness.product_step(b, kernel=HP)
    assert oa["err"] == 0 and ob["err"] == 0
    assert np.array_equal(oa["out"], ob["out"])
    per_head = harness.product_step(a, kernel=2)["out"]
    harness.assert_close(oa["out"], per_head, False)


@requires_gpu
def test_hp_workspace_shared_across_shapes_and_repeated_calls():
    """One workspace (arbitrary bytes) serves calls of different shapes and
    both tensor-core kernels back to back, and a repeated call gives
    bit-identical output."""
    big = synth.longctx()
    small = synth.make("hp-reuse", [5000, 300, 9000, 17], 32, 8, 128, 16, seed=155)
    outs = {}
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    ws.random_(0, 256)
    for w, kern in ((big, HP), (small, HP), (big, 2), (big, HP), (small, 2), (small, HP)):
        got = harness.product_step(w, kernel=HP)
        assert got["err"] == 0
        dev = got["dev"]
        ws[:4] = 0
        out = torch.empty_like(dev["q"])
        ops.decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["bt"], dev["cl"], w.scale,
                   workspace=ws, kernel=kern)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).item()) == 0
        res = out.float().cpu().numpy().astype(np.float64)
        if kern == HP:
            assert np.array_equal(res, got["out"]), w.name
            if w.name in outs:
                assert np.array_equal(outs[w.name], res)
            outs[w.name] = res


@requires_gpu
@pytest.mark.parametrize("block_size", [1, 2, 4, 8])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 8), (32, 32), (64, 16)])
def test_hp_blocks_smaller_than_a_chunk(block_size, hq, hkv):
    # token-major tiles (8 heads x 16 tokens for groups 2 and 4, 16 x 8 for
    # MHA, so MHA at block size 8 is head-major); lengths around block,
    # chunk and CTA boundaries
    lens = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 127, 129, 700, 2000, 4]
    w = synth.make(f"hp-small-blocks-{hq}-{hkv}-{block_size}", lens, hq, hkv, 128, block_size,
                   seed=171 + block_size)
    _check(w)


@requires_gpu
def test_hp_block1_llama8b_and_automatic_choice():
    # the batch-64 layer at block size 1 (121,416 single-token blocks): the
    # automatic choice is the head-packed kernel, bit-identical to forcing it
    w = synth.sweep(1, "bf16")
    _, forced, _ = _check(w)
    auto = harness.product_step(w, kernel=0)
    assert auto["err"] == 0
    assert np.array_equal(auto["out"], forced["out"])


@requires_gpu
def test_hp_block1_long_contexts():
    # units split over many CTAs with one-token blocks
    lens = [70000, 5000, 1, 23000, 0, 999]
    w = synth.make("hp-b1-long", lens, 32, 8, 128, 1, seed=181, heavy_frac=0.01, heavy_mult=3.0)
    _check(w)


@requires_gpu
@pytest.mark.parametrize("block_size", [1, 4])
def test_hp_small_blocks_permutation_invariant(block_size):
    lens = synth.llama8b_lengths(8)
    nb = sum(-(-n // block_size) for n in lens) + 500
    a = synth.make("hp-sb-perm-a", lens, 32, 8, 128, block_size, seed=183, num_blocks=nb)
    b = synth.make("hp-sb-perm-b", lens, 32, 8, 128, block_size, seed=183, num_blocks=nb)
    rng = np.random.default_rng(185)
    perm = rng.permutation(nb).astype(np.int32)
    mask = np.zeros_like(a.block_tables, dtype=bool)
    for i, n in enumerate(lens):
        mask[i, :-(-n // block_size)] = True
    b.block_tables = np.where(mask, perm[a.block_tables], 0).astype(np.int32)
    oa = harness.product_step(a, kernel=HP)
    ob = harness.product_step(b, kernel=HP)
    assert oa["err"] == 0 and ob["err"] == 0
    assert np.array_equal(oa["out"], ob["out"])
    harness.assert_close(oa["out"], harness.oracle_step(a)["out"], False)


@requires_gpu
@pytest.mark.parametrize("hq,hkv,bs,kv", [(64, 8, 16, "bf16"), (8, 8, 16, "bf16"),
                                          (8, 8, 1, "fp8")])
def test_hp_unsupported_shapes_are_refused(hq, hkv, bs, kv):
    # group 8, H_kv not a multiple of the tile's heads: kernel 3 refuses
    # instead of launching
    w = synth.make("hp-refuse", [20, 40], hq, hkv, 128, bs, kv_dtype=kv, seed=157)
    from paged_kv_cache_108_gb300._lib import PaError
    with pytest.raises(PaError, match="head-packed"):
        harness.product_step(w, kernel=HP)


@requires_gpu
def test_automatic_choice_takes_head_packed_for_many_units():
    # 700 sequences of 8 KV heads: kernel 0 picks the head-packed kernel; the
    # result must equal the forced choice bit for bit and match the oracle
    rng = np.random.default_rng(159)
    lens = [int(x) for x in rng.integers(1, 300, size=700)]
    w = synth.make("hp-auto", lens, 32, 8, 128, 16, seed=161, num_blocks=16000)
    auto = harness.product_step(w, kernel=0)
    forced = harness.product_step(w, kernel=HP)
    assert auto["err"] == 0 and forced["err"] == 0
    assert np.array_equal(auto["out"], forced["out"])
    harness.assert_close(auto["out"], harness.oracle_step(w)["out"], False)


# ---- e4m3 cache: kind::f8f6f4 MMAs, q in three e4m3 parts, P in two ----

@requires_gpu
@pytest.mark.parametrize("block_size", [1, 2, 4, 8, 16, 64])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 8), (32, 32)])
def test_hp_fp8_block_sizes_and_groups(block_size, hq, hkv):
    # token-major tiles below 16 (8 for MHA) tokens per block, head-major
    # above; lengths around block, chunk and CTA boundaries
    lens = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 127, 129, 700, 2000, 4]
    w = synth.make(f"hp-fp8-{hq}-{hkv}-{block_size}", lens, hq, hkv, 128, block_size,
                   kv_dtype="fp8", seed=191 + block_size)
    _check(w)


@requires_gpu
@pytest.mark.parametrize("block_size", [1, 16])
def test_hp_fp8_llama8b(block_size):
    # the batch-64 layer; at block size 1 the automatic choice is the
    # head-packed kernel, bit-identical to forcing it
    w = synth.sweep(block_size, "fp8")
    _, forced, _ = _check(w)
    if block_size == 1:
        auto = harness.product_step(w, kernel=0)
        assert auto["err"] == 0
        assert np.array_equal(auto["out"], forced["out"])


@requires_gpu
def test_hp_fp8_long_contexts_many_pieces():
    # units split over many CTAs (merges of many pieces), peaked rows
    lens = [70000, 5000, 1, 23000, 0, 999]
    w = synth.make("hp-fp8-long", lens, 32, 8, 128, 1, kv_dtype="fp8", seed=193,
                   heavy_frac=0.01, heavy_mult=3.0)
    _check(w)
    _check(synth.longctx(kv_dtype="fp8"))


@requires_gpu
@pytest.mark.parametrize("qmult", [1e-3, 13.7, 77.3])
def test_hp_fp8_query_magnitudes(qmult):
    # the q warp scales each unit's q by a power of two before splitting it
    # into e4m3 parts; tiny and large q must come out as accurate as unit q
    lens = [5, 129, 600, 1500, 40]
    w = synth.make(f"hp-fp8-q{qmult}", lens, 32, 8, 128, 1, kv_dtype="fp8", seed=197)
    qf = (w.q.astype(np.uint32) << np.uint32(16)).view(np.float32) * np.float32(qmult)
    w.q = synth.bf16_bits(qf)
    _check(w)


@requires_gpu
def test_hp_fp8_permutation_invariant_and_agrees_with_per_head_kernel():
    lens = synth.llama8b_lengths(8)
    nb = sum(lens) + 500
    a = synth.make("hp-fp8-perm-a", lens, 32, 8, 128, 1, kv_dtype="fp8", seed=199, num_blocks=nb)
    b = synth.make("hp-fp8-perm-b", lens, 32, 8, 128, 1, kv_dtype="fp8", seed=199, num_blocks=nb)
    rng = np.random.default_rng(201)
    perm = rng.permutation(nb).astype(np.int32)
    mask = np.zeros_like(a.block_tables, dtype=bool)
    for i, n in enumerate(lens):
        mask[i, :n] = True
    b.block_tables = np.where(mask, perm[a.block_tables], 0).astype(np.int32)
    oa = harness.product_step(a, kernel=HP)
    ob = harness.product_step(b, kernel=HP)
    assert oa["err"] == 0 and ob["err"] == 0
    assert np.array_equal(oa["out"], ob["out"])
    harness.assert_close(oa["out"], harness.oracle_step(a)["out"], True)
    per_head = harness.product_step(a, kernel=2)["out"]
    assert np.max(np.abs(oa["out"] - per_head)) < 6e-2
