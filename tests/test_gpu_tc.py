"""GPU parity of the tensor-core (tcgen05 + TMA) decode kernel against the
fp64 oracle, and agreement with the SIMT kernel.

Same bars as tests/test_gpu_parity.py; additionally the kernel's error word
(workspace word 0: an expired bounded wait or an out-of-range block id) must
stay zero."""
import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

TC = 2


def _check(w, **kw):
    got = harness.product_step(w, kernel=TC, **kw)
    assert got["err"] == 0, f"tensor-core kernel error word {got['err']}"
    ref = harness.oracle_step(w)
    assert np.array_equal(got["k_cache"], ref["k_cache"])
    assert np.array_equal(got["v_cache"], ref["v_cache"])
    return harness.assert_close(got["out"], ref["out"], w.kv_dtype == "fp8"), got, ref


@requires_gpu
def test_tc_small_group_mix():
    lens = [1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 257, 1000]
    w = synth.make("tc-small", lens, 32, 8, 128, 16, seed=31)
    _check(w)


@requires_gpu
def test_tc_llama8b_batch64():
    _check(synth.llama8b())


@requires_gpu
def test_tc_long_context():
    _check(synth.longctx())


@requires_gpu
@pytest.mark.parametrize("block_size", [1, 2, 4, 8, 16, 64, 256])
def test_tc_block_sizes(block_size):
    # below 8 tokens per block the rows are gathered by cp.async, not TMA
    _check(synth.sweep(block_size, "bf16"))


@requires_gpu
@pytest.mark.parametrize("block_size", [1, 2, 4])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_tc_gathered_rows_at_chunk_edges(block_size, kv_dtype):
    # lengths on both sides of the 128-token (bf16) and 256-token (e4m3)
    # chunk ends, single tokens, and long units split over CTAs
    lens = [1, 2, 3, 127, 128, 129, 255, 256, 257, 511, 513, 5000, 20000]
    w = synth.make(f"tc-gather-{block_size}-{kv_dtype}", lens, 32, 8, 128, block_size,
                   kv_dtype=kv_dtype, seed=53 + block_size)
    _check(w)


@requires_gpu
def test_tc_gathered_rows_permutation_invariant_and_agree_with_simt():
    lens = [int(x) for x in np.random.default_rng(61).integers(1, 1500, size=20)]
    a = synth.make("tc-gather-perm-a", lens, 32, 8, 128, 1, seed=62)
    b = synth.make("tc-gather-perm-b", lens, 32, 8, 128, 1, seed=62)
    # same data, blocks placed by another permutation
    perm = np.random.default_rng(63).permutation(a.num_blocks).astype(np.int32)
    b.block_tables = np.where(a.block_tables >= 0, perm[a.block_tables], a.block_tables)
    ga = harness.product_step(a, kernel=TC)
    gb = harness.product_step(b, kernel=TC)
    assert ga["err"] == 0 and gb["err"] == 0
    assert np.array_equal(ga["out"], gb["out"])
    simt = harness.product_step(a, kernel=1)["out"]
    harness.assert_close(ga["out"], simt, False)


@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (64, 8), (4, 2)])
def test_tc_head_groups(hq, hkv):
    lens = [3, 130, 700, 2000, 64, 1]
    w = synth.make(f"tc-heads-{hq}-{hkv}", lens, hq, hkv, 128, 16, seed=41)
    _check(w)


@requires_gpu
def test_tc_empty_sequences():
    w = synth.make("tc-empty", [0, 300, 0, 5], 32, 8, 128, 16, seed=43)
    err, got, ref = _check(w)
    assert np.all(got["out"][0] == 0) and np.all(got["out"][2] == 0)


@requires_gpu
def test_tc_agrees_with_simt_and_is_permutation_invariant():
    lens = synth.llama8b_lengths(16)
    a = synth.make("perm-a", lens, 32, 8, 128, 16, seed=11, num_blocks=2000)
    b = synth.make("perm-b", lens, 32, 8, 128, 16, seed=11, num_blocks=2000)
    rng = np.random.default_rng(99)
    perm = rng.permutation(2000).astype(np.int32)
    mask = np.zeros_like(a.block_tables, dtype=bool)
    for i, n in enumerate(lens):
        mask[i, :-(-n // 16)] = True
    b.block_tables = np.where(mask, perm[a.block_tables], 0).astype(np.int32)
    oa = harness.product_step(a, kernel=TC)
    ob = harness.product_step(b, kernel=TC)
    assert oa["err"] == 0 and ob["err"] == 0
    assert np.array_equal(oa["out"], ob["out"])
    simt = harness.product_step(a, kernel=1)["out"]
    harness.assert_close(oa["out"], simt, False)


@requires_gpu
def test_tc_workspace_shared_across_shapes_and_repeated_calls():
    """One workspace serves calls of different shapes back to back (merge
    counters of one shape land where another shape keeps partials), and a
    repeated call gives bit-identical output."""
    from paged_kv_cache_108_gb300 import ops
    big = synth.longctx()
    small = synth.make("tc-reuse", [5000, 300, 9000, 17], 32, 8, 128, 16, seed=47)
    outs = {}
    ws = None
    for w in (big, small, big, small):
        got = harness.product_step(w, kernel=TC)
        assert got["err"] == 0
        dev = got["dev"]
        if ws is None:
            ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
            ws.random_(0, 256)
        ws[:4] = 0
        out = torch.empty_like(dev["q"])
        ops.decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["bt"], dev["cl"], w.scale,
                   workspace=ws, kernel=TC)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).item()) == 0
        res = out.float().cpu().numpy().astype(np.float64)
        assert np.array_equal(res, got["out"]), w.name
        if w.name in outs:
            assert np.array_equal(outs[w.name], res)
        outs[w.name] = res


@requires_gpu
def test_write_and_decode_matches_separate_calls():
    """The one-call step gives the same caches and bit-identical output as the
    separate write and decode calls (the overlap changes only timing)."""
    from paged_kv_cache_108_gb300 import ops, pool
    w = synth.llama8b()
    got = harness.product_step(w)  # separate calls
    dev = got["dev"]
    kc = harness.to_dev_bits(w.junk_k, "bf16", "cuda")
    vc = harness.to_dev_bits(w.junk_v, "bf16", "cuda")
    seq_idx, pos = harness.ctx_positions(w)
    ops.reshape_and_cache(harness.to_dev_bits(w.ctx_k, "bf16", "cuda"),
                          harness.to_dev_bits(w.ctx_v, "bf16", "cuda"), kc, vc,
                          torch.from_numpy(pool.slot_mapping(w.block_tables, w.block_size, pos, seq_idx)).cuda())
    out = torch.empty_like(dev["q"])
    ws = ops.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_blocks, w.block_size)
    ws.random_(0, 256)
    for _ in range(2):
        ops.write_and_decode(harness.to_dev_bits(w.k_new, "bf16", "cuda"),
                             harness.to_dev_bits(w.v_new, "bf16", "cuda"),
                             torch.from_numpy(got["slots_new"]).cuda(), out, dev["q"], kc, vc,
                             dev["bt"], dev["cl"], w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(harness.bits_from_dev(kc), got["k_cache"])
        assert np.array_equal(harness.bits_from_dev(vc), got["v_cache"])
        assert np.array_equal(out.float().cpu().numpy().astype(np.float64), got["out"])


# ---- e4m3 cache: kind::f8f6f4 MMAs with q and P split into e4m3 parts ----

@requires_gpu
@pytest.mark.parametrize("block_size", [1, 2, 4, 8, 16, 64, 256])
def test_tc_fp8_block_sizes(block_size):
    _check(synth.sweep(block_size, "fp8"))


@requires_gpu
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (4, 2)])
def test_tc_fp8_head_groups(hq, hkv):
    lens = [3, 130, 700, 2000, 64, 1, 257]
    w = synth.make(f"tc-fp8-heads-{hq}-{hkv}", lens, hq, hkv, 128, 16, kv_dtype="fp8", seed=47)
    _check(w)


@requires_gpu
def test_tc_fp8_long_context_split_units():
    _check(synth.longctx(kv_dtype="fp8"))


@requires_gpu
@pytest.mark.parametrize("qmult", [1e-3, 13.7, 77.3])
def test_tc_fp8_query_magnitudes(qmult):
    # the q warp scales each group's q by a power of two before splitting it
    # into e4m3 parts; tiny and large q must come out as accurate as unit q
    lens = [5, 129, 600, 1500, 40]
    w = synth.make(f"tc-fp8-q{qmult}", lens, 32, 8, 128, 16, kv_dtype="fp8", seed=53)
    qf = (w.q.astype(np.uint32) << np.uint32(16)).view(np.float32) * np.float32(qmult)
    w.q = synth.bf16_bits(qf)
    _check(w)


@requires_gpu
def test_tc_fp8_agrees_with_simt():
    w = synth.make("tc-fp8-vs-simt", synth.llama8b_lengths(16), 32, 8, 128, 16,
                   kv_dtype="fp8", seed=59)
    _, got, ref = _check(w)
    simt = harness.product_step(w, kernel=1)["out"]
    harness.assert_close(simt, ref["out"], True)
    assert np.max(np.abs(got["out"] - simt)) < 6e-2
