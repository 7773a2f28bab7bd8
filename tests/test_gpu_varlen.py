"""GPU parity of pa_varlen_attention (multi-token decode, chunked and full
prefill) against the fp64 varlen oracle, with the bf16 / e4m3 tolerances of
the decode tests; and bit-equality with pa_decode when every request adds
exactly one token (same kernels, same work)."""
import numpy as np
import pytest
import torch

from oracle import varlen
from paged_kv_cache_108_gb300 import ops, pool, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _setup(seq_lens, query_lens, H, Hkv, d, B, kv_dtype="bf16", seed=0):
    rng = np.random.default_rng(seed)
    nblk = [-(-s // B) for s in seq_lens]
    num_blocks = int(1.2 * sum(nblk)) + 4
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((len(seq_lens), max(nblk)), dtype=np.int32)
    at = 0
    for i, c in enumerate(nblk):
        tables[i, :c] = perm[at:at + c]
        at += c
    shape = (num_blocks, B, Hkv, d)
    if kv_dtype == "bf16":
        kc = torch.from_numpy(rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)).cuda()
        vc = torch.from_numpy(rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)).cuda()
        kc, vc = kc.view(torch.bfloat16), vc.view(torch.bfloat16)
    else:
        kc = torch.from_numpy(rng.integers(0, 256, size=shape, dtype=np.uint8)).cuda()
        vc = torch.from_numpy(rng.integers(0, 256, size=shape, dtype=np.uint8)).cuda()
    tok = sum(seq_lens)
    k = synth.normal_bf16(rng, (tok, Hkv, d))
    v = synth.normal_bf16(rng, (tok, Hkv, d))
    seq_idx = np.concatenate([np.full(s, i, np.int32) for i, s in enumerate(seq_lens)])
    pos = np.concatenate([np.arange(s, dtype=np.int32) for s in seq_lens])
    slots = pool.slot_mapping(tables, B, pos, seq_idx)
    ks = vs = None
    kscale = vscale = 1.0
    if kv_dtype == "fp8":
        kscale, vscale = synth.per_tensor_scale(k), synth.per_tensor_scale(v)
        ks = torch.tensor([kscale], dtype=torch.float32, device="cuda")
        vs = torch.tensor([vscale], dtype=torch.float32, device="cuda")
    ops.reshape_and_cache(harness.to_dev_bits(k, "bf16", "cuda"),
                          harness.to_dev_bits(v, "bf16", "cuda"), kc, vc,
                          torch.from_numpy(slots).cuda(), ks, vs)
    q = synth.normal_bf16(rng, (sum(query_lens), H, d))
    qsl = np.concatenate([[0], np.cumsum(query_lens)]).astype(np.int32)
    return dict(kc=kc, vc=vc, ks=ks, vs=vs, kscale=kscale, vscale=vscale, tables=tables,
                seq_lens=np.array(seq_lens, np.int32), qsl=qsl, q=q, H=H, d=d, kv=kv_dtype)


def _run(c, scale):
    q = harness.to_dev_bits(c["q"], "bf16", "cuda")
    out = torch.empty_like(q)
    ops.varlen_attention(out, q, c["kc"], c["vc"], torch.from_numpy(c["tables"]).cuda(),
                         torch.from_numpy(c["seq_lens"]).cuda(), torch.from_numpy(c["qsl"]).cuda(),
                         scale, c["ks"], c["vs"])
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _check(c, scale):
    got = _run(c, scale)
    ref = varlen.varlen_attention(c["q"], harness.bits_from_dev(c["kc"]),
                                  harness.bits_from_dev(c["vc"]), c["tables"], c["seq_lens"],
                                  c["qsl"], scale, c["kscale"], c["vscale"])
    harness.assert_close(got, ref, c["kv"] == "fp8")
    return got


@requires_gpu
def test_pages_three_requests_decode_full_and_chunked_prefill():
    c = _setup([37, 5, 20], [1, 5, 8], 8, 2, 64, 4, seed=1)
    _check(c, 64 ** -0.5)


@requires_gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_multi_token_decode_batch(kv_dtype):
    rng = np.random.default_rng(2)
    lens = rng.integers(100, 2500, size=32).tolist()
    c = _setup(lens, [4] * 32, 32, 8, 128, 16, kv_dtype, seed=3)
    _check(c, 128 ** -0.5)


@requires_gpu
def test_chunked_and_full_prefill_mix():
    c = _setup([700, 300, 1500, 129], [200, 300, 1, 129], 32, 8, 128, 16, seed=4)
    _check(c, 128 ** -0.5)


@requires_gpu
def test_requests_without_new_tokens_and_inconsistent_counts():
    c = _setup([50, 60, 10], [3, 0, 4], 8, 8, 128, 16, seed=5)
    c["seq_lens"][2] = 3          # 4 new tokens but only 3 in the context: zero rows
    got = _run(c, 0.1)
    assert not got[3:].any()
    ref = varlen.varlen_attention(c["q"][:3], harness.bits_from_dev(c["kc"]),
                                  harness.bits_from_dev(c["vc"]), c["tables"][:1],
                                  c["seq_lens"][:1], c["qsl"][:2], 0.1)
    harness.assert_close(got[:3], ref, False)


@requires_gpu
def test_one_token_per_request_equals_decode_bit_for_bit():
    rng = np.random.default_rng(6)
    lens = rng.integers(1, 3000, size=40).tolist()
    c = _setup(lens, [1] * 40, 32, 8, 128, 16, seed=7)
    got = _run(c, 0.08)
    q = harness.to_dev_bits(c["q"], "bf16", "cuda")
    out = torch.empty_like(q)
    ws = ops.alloc_workspace(40, 32, 128, c["tables"].shape[1], 16)
    ops.decode(out, q, c["kc"], c["vc"], torch.from_numpy(c["tables"]).cuda(),
               torch.from_numpy(c["seq_lens"]).cuda(), 0.08, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(got, out.float().cpu().numpy().astype(np.float64))


def _check_multi(c, T, scale):
    q = harness.to_dev_bits(c["q"], "bf16", "cuda")
    out = torch.empty_like(q)
    ops.decode_multi(out, q, c["kc"], c["vc"], torch.from_numpy(c["tables"]).cuda(),
                     torch.from_numpy(c["seq_lens"]).cuda(), T, scale, c["ks"], c["vs"])
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = varlen.varlen_attention(c["q"], harness.bits_from_dev(c["kc"]),
                                  harness.bits_from_dev(c["vc"]), c["tables"], c["seq_lens"],
                                  c["qsl"], scale, c["kscale"], c["vscale"])
    harness.assert_close(got, ref, c["kv"] == "fp8")
    return got


@requires_gpu
@pytest.mark.parametrize("T,hq,hkv,kv", [(2, 32, 8, "bf16"), (4, 32, 8, "bf16"),
                                         (2, 64, 8, "bf16"), (8, 8, 8, "bf16"),
                                         (16, 8, 8, "bf16"), (2, 32, 8, "fp8"),
                                         (4, 32, 8, "fp8"), (3, 32, 8, "bf16")])
def test_multi_token_decode_one_pass_and_fallback(T, hq, hkv, kv):
    # group x T columns: 8 and 16 run one tensor-core pass; fp8 with 16
    # columns and T = 3 (12 columns) take the per-token path
    rng = np.random.default_rng(10 + T)
    lens = [int(x) for x in rng.integers(T, 2600, size=24)] + [T, T + 1, 129]
    c = _setup(lens, [T] * len(lens), hq, hkv, 128, 16, kv, seed=11 + T)
    _check_multi(c, T, 128 ** -0.5)


@requires_gpu
def test_multi_token_split_units_with_masked_columns():
    # few long sequences: units split over many CTAs, and pieces near a
    # sequence's end hold keys that some of its tokens must not see
    lens = [4096, 9000, 130, 16384]
    c = _setup(lens, [4] * 4, 32, 8, 128, 16, seed=21)
    got = _check_multi(c, 4, 0.09)
    assert np.isfinite(got).all()


@requires_gpu
@pytest.mark.parametrize("block_size,kv", [(1, "bf16"), (2, "fp8"), (4, "bf16")])
def test_multi_token_decode_on_gathered_rows(block_size, kv):
    # blocks below 8 tokens: the one-pass kernel gathers its rows by cp.async
    rng = np.random.default_rng(30 + block_size)
    lens = [int(x) for x in rng.integers(4, 1800, size=12)] + [4, 5, 260]
    c = _setup(lens, [4] * len(lens), 32, 8, 128, block_size, kv, seed=31 + block_size)
    _check_multi(c, 4, 128 ** -0.5)
