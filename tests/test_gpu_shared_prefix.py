"""pa_decode_shared_prefix: forked groups read their shared prefix once.

The output must equal the fp64 oracle's plain decode (the prefix split and
the log-sum-exp merge change only the rounding), with the decode
tolerances: on the serving mix (1024-token prefix on a block boundary, and
the 1000-token prefix whose last shared block was copied on write), on GQA
and e4m3 groups, on a batch with no sharing at all, and when a member's
context ends exactly at the prefix."""
import numpy as np
import pytest
import torch

from oracle import core as ocore
from paged_kv_cache_108_gb300 import ops, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@requires_gpu
@pytest.mark.parametrize("prefix", [1024, 1000])
def test_serving_mix(prefix):
    mix = synth.serving(prefix_len=prefix)
    nb = harness.serving_pool_size(mix)
    data = synth.serving_data(mix, nb, harness.serving_unique_tokens(mix))
    got = harness.serving_product(mix, data, nb, shared_prefix_group=mix.group_size)
    ref = harness.serving_oracle(mix, data, nb)
    assert np.array_equal(got["k_cache"], ref["k_cache"])
    harness.assert_close(got["out"], ref["out"], False)


def _grouped(group, n_groups, prefix_blocks, suffix_lens, H, Hkv, kv_dtype, seed, B=16):
    """Tables where each group's members share their first prefix_blocks blocks."""
    rng = np.random.default_rng(seed)
    S = group * n_groups
    lens = np.array([prefix_blocks * B + int(s) for s in suffix_lens], dtype=np.int32)
    nblk = [-(-int(n) // B) for n in lens]
    num_blocks = n_groups * prefix_blocks + sum(n - prefix_blocks for n in nblk) + 8
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((S, max(nblk)), dtype=np.int32)
    at = 0
    for gi in range(n_groups):
        shared = perm[at:at + prefix_blocks]
        at += prefix_blocks
        for i in range(gi * group, (gi + 1) * group):
            tables[i, :prefix_blocks] = shared
            own = nblk[i] - prefix_blocks
            tables[i, prefix_blocks:nblk[i]] = perm[at:at + own]
            at += own
    shape = (num_blocks, B, Hkv, 128)
    if kv_dtype == "bf16":
        kc = synth.normal_bf16(rng, shape)
        vc = synth.normal_bf16(rng, shape)
        kd = torch.from_numpy(kc).cuda().view(torch.bfloat16)
        vd = torch.from_numpy(vc).cuda().view(torch.bfloat16)
        ks = vs = None
        kscale = vscale = 1.0
    else:
        kc = rng.integers(0, 0x7f, size=shape, dtype=np.uint8)
        vc = rng.integers(0, 0x7f, size=shape, dtype=np.uint8)
        kd, vd = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
        kscale, vscale = 0.02, 0.03
        ks = torch.tensor([kscale], dtype=torch.float32, device="cuda")
        vs = torch.tensor([vscale], dtype=torch.float32, device="cuda")
    q = synth.normal_bf16(rng, (S, H, 128))
    return dict(kc=kc, vc=vc, kd=kd, vd=vd, ks=ks, vs=vs, kscale=kscale, vscale=vscale,
                tables=tables, lens=lens, q=q, H=H)


def _run_and_check(c, group, fp8):
    q = harness.to_dev_bits(c["q"], "bf16", "cuda")
    out = torch.empty_like(q)
    scale = 128 ** -0.5
    ops.decode_shared_prefix(out, q, c["kd"], c["vd"], torch.from_numpy(c["tables"]).cuda(),
                             torch.from_numpy(c["lens"]).cuda(), group, scale, c["ks"], c["vs"])
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = ocore.decode(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], scale, c["kscale"],
                       c["vscale"], nthreads=8)
    harness.assert_close(got, ref, fp8)
    return got


@requires_gpu
@pytest.mark.parametrize("group,H,Hkv,kv", [(4, 32, 8, "bf16"), (8, 8, 8, "bf16"),
                                           (2, 32, 8, "fp8"), (16, 8, 8, "bf16")])
def test_groups_gqa_and_e4m3(group, H, Hkv, kv):
    rng = np.random.default_rng(group + H)
    suffix = rng.integers(1, 900, size=group * 6)
    c = _grouped(group, 6, 40, suffix, H, Hkv, kv, seed=group * 3 + H)
    _run_and_check(c, group, kv == "fp8")


@requires_gpu
@pytest.mark.parametrize("B", [1, 4])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_small_blocks(B, kv):
    # blocks of fewer than 8 tokens: the suffix pass runs on the head-packed
    # kernel's token-major tiles (e4m3: row gathers) and hands its log2-sum-
    # exp to the merge; the prefix pass gathers rows on the per-head kernel
    rng = np.random.default_rng(11 + B)
    suffix = rng.integers(1, 700, size=4 * 5)
    c = _grouped(4, 5, 480 // B, suffix, 32, 8, kv, seed=13 + B, B=B)
    _run_and_check(c, 4, kv == "fp8")


@requires_gpu
def test_no_sharing_and_member_ending_at_the_prefix():
    rng = np.random.default_rng(4)
    c = _grouped(4, 5, 0, rng.integers(1, 1500, size=20), 32, 8, "bf16", seed=5)
    _run_and_check(c, 4, False)                  # no shared block: pass 1 is empty
    d = _grouped(4, 3, 24, [0, 17, 300, 5] * 3, 32, 8, "bf16", seed=6)
    _run_and_check(d, 4, False)                  # a member whose context is the prefix


@requires_gpu
def test_many_gqa_groups_suffix_pass_on_head_packed_kernel():
    # 320 sequences x 8 KV heads: the suffix pass has 320 units of 8 heads,
    # enough for the automatic choice to take the head-packed kernel (with
    # its log2-sum-exp output) while the prefix pass stays per-head
    rng = np.random.default_rng(21)
    c = _grouped(8, 40, 10, rng.integers(1, 200, size=320), 32, 8, "bf16", seed=22)
    _run_and_check(c, 8, False)
