"""Prefix caching end to end on the GPU.

Requests that repeat a system prompt get their blocks from the host pool's
prefix cache ("Paged KV cache", Exercises: the copy-on-write answer -- full
blocks are shared, every request writes in a block of its own; "4.6
PagedAttention & KV-Cache Memory Management", section "Copy-on-write for
shared prefixes").  Each request writes only the tokens the cache did not
already hold, through pa_reshape_and_cache; one request is freed and its
prompt asked for again, so the second copy matches blocks that sat in the
free queue.  Then the batch is decoded with pa_decode and with
pa_decode_shared_prefix.

Checked: the native pool's tables and cached-token counts equal the oracle
model's; the caches equal the oracle's writes bit for bit; both decodes are
within the bf16 tolerance of the fp64 oracle on the oracle's caches."""
import hashlib

import numpy as np
import pytest
import torch

from oracle import core as ocore
from oracle.pool_model import PrefixCachePoolModel
from paged_kv_cache_108_gb300 import ops, pool, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

B, HKV, H, D = 16, 8, 32, 128


def _row(tokens_upto):
    """K and V of the last token of ``tokens_upto``: a function of the whole
    prefix, as in a model, so equal prefixes give equal rows."""
    digest = hashlib.sha256(np.asarray(tokens_upto, np.int64).tobytes()).digest()
    rng = np.random.default_rng(int.from_bytes(digest[:8], "little"))
    return synth.normal_bf16(rng, (2, HKV, D))


@requires_gpu
def test_prefix_cached_batch_decodes_like_the_oracle():
    rng = np.random.default_rng(2024)
    num_blocks = 96
    order = rng.permutation(num_blocks).tolist()
    nat = pool.BlockPool(num_blocks, free_order=order)
    nat.enable_prefix_cache(B)
    mod = PrefixCachePoolModel(num_blocks, B, free_order=order)

    system = [int(x) for x in rng.integers(1000, 2000, size=70)]      # 4 full blocks + 6
    prompts = [system + [int(x) for x in rng.integers(0, 1000, size=int(n))]
               for n in (9, 40, 1, 75, 26)]
    prompts.append(list(system[:48]) + [7, 7, 7])                      # shares 3 blocks

    kc_dev = harness.to_dev_bits(rng.integers(0, 1 << 16, size=(num_blocks, B, HKV, D),
                                              dtype=np.uint16), "bf16", "cuda")
    vc_dev = harness.to_dev_bits(rng.integers(0, 1 << 16, size=(num_blocks, B, HKV, D),
                                              dtype=np.uint16), "bf16", "cuda")
    kc_ref, vc_ref = harness.bits_from_dev(kc_dev), harness.bits_from_dev(vc_dev)

    def admit(tokens):
        got, want = nat.allocate_prefix(tokens), mod.allocate_prefix(tokens)
        assert got == want
        blocks, cached = got
        # write the tokens the cache does not hold, positions cached..n-1
        pos = np.arange(cached, len(tokens), dtype=np.int32)
        if pos.size:
            rows = np.stack([_row(tokens[:p + 1]) for p in pos])           # [n, 2, HKV, D]
            k, v = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
            slots = np.array([blocks[p // B] * B + p % B for p in pos], dtype=np.int32)
            ops.reshape_and_cache(harness.to_dev_bits(k, "bf16", "cuda"),
                                  harness.to_dev_bits(v, "bf16", "cuda"), kc_dev, vc_dev,
                                  torch.from_numpy(slots).cuda())
            ocore.reshape_and_cache(k, v, kc_ref, vc_ref, slots)
        return blocks, cached

    live = [admit(t) + (t,) for t in prompts]
    assert [c for _, c, _ in live] == [0, 64, 64, 64, 64, 48]
    # the fourth request finishes; the same prompt comes again and matches
    # its full blocks while they wait in the free queue
    blocks3, _, tokens3 = live.pop(3)
    nat.free(blocks3)
    mod.free(blocks3)
    assert nat.free_order() == mod.free_order()
    again = admit(tokens3)
    assert again[1] == (len(tokens3) // B) * B and again[0][:len(tokens3) // B] == \
        blocks3[:len(tokens3) // B]
    live.append(again + (tokens3,))
    assert [nat.refcount(i) for i in range(num_blocks)] == \
        [mod.refcount(i) for i in range(num_blocks)]
    torch.cuda.synchronize()
    assert np.array_equal(harness.bits_from_dev(kc_dev), kc_ref)
    assert np.array_equal(harness.bits_from_dev(vc_dev), vc_ref)

    S = len(live)
    lens = np.array([len(t) for _, _, t in live], dtype=np.int32)
    tables = np.zeros((S, max(len(b) for b, _, _ in live)), dtype=np.int32)
    for i, (b, _, _) in enumerate(live):
        tables[i, :len(b)] = b
    q = synth.normal_bf16(rng, (S, H, D))
    scale = D ** -0.5
    ref = ocore.decode(q, kc_ref, vc_ref, tables, lens, scale)
    qd = harness.to_dev_bits(q, "bf16", "cuda")
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    out = torch.empty_like(qd)
    ws = ops.alloc_workspace(S, H, D, tables.shape[1], B)
    ops.decode(out, qd, kc_dev, vc_dev, bt, cl, scale, workspace=ws)
    torch.cuda.synchronize()
    harness.assert_close(out.float().cpu().numpy().astype(np.float64), ref, False)
    out2 = torch.empty_like(qd)
    ops.decode_shared_prefix(out2, qd, kc_dev, vc_dev, bt, cl, 2, scale)
    torch.cuda.synchronize()
    harness.assert_close(out2.float().cpu().numpy().astype(np.float64), ref, False)
