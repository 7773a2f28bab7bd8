"""pa_swap_blocks: whole-block copies between the device pool and a pinned
host swap space (and between two device pools), bit for bit, in both
directions; pairs naming a block outside either cache are skipped."""
import numpy as np
import pytest
import torch

from paged_kv_cache_108_gb300 import ops

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _cache(n, B, hkv, d, dtype, device, seed):
    g = torch.Generator().manual_seed(seed)
    bits = torch.randint(0, 256 if dtype == torch.uint8 else 1 << 16, (n, B, hkv, d),
                         generator=g, dtype=torch.int32)
    t = bits.to(torch.uint8) if dtype == torch.uint8 else bits.to(torch.int16).view(torch.bfloat16)
    if device == "pinned":
        return t.contiguous().pin_memory()
    return t.to(device)


def _bits(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


@requires_gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.uint8])
@pytest.mark.parametrize("B,hkv,d", [(16, 8, 128), (1, 32, 128), (256, 2, 64)])
def test_swap_out_and_back_in(dtype, B, hkv, d):
    dev_k = _cache(40, B, hkv, d, dtype, "cuda", 1)
    dev_v = _cache(40, B, hkv, d, dtype, "cuda", 2)
    host_k = _cache(25, B, hkv, d, dtype, "pinned", 3)
    host_v = _cache(25, B, hkv, d, dtype, "pinned", 4)
    k0, v0 = _bits(dev_k), _bits(dev_v)
    hk0, hv0 = _bits(host_k), _bits(host_v)
    # swap out device blocks 3, 17, 39 -> host slots 0, 24, 11; (99, 5) and (4, 31) are out of range
    out_pairs = torch.tensor([[3, 0], [17, 24], [39, 11], [99, 5], [4, 31]], dtype=torch.int32,
                             device="cuda")
    ops.swap_blocks(host_k, host_v, dev_k, dev_v, out_pairs)
    torch.cuda.synchronize()
    hk, hv = hk0.copy(), hv0.copy()
    for s, d_ in [(3, 0), (17, 24), (39, 11)]:
        hk[d_], hv[d_] = k0[s], v0[s]
    assert np.array_equal(_bits(host_k), hk) and np.array_equal(_bits(host_v), hv)
    # the device blocks are reused meanwhile, then the swapped blocks come back
    dev_k.zero_()
    dev_v.zero_()
    in_pairs = torch.tensor([[0, 7], [24, 8], [11, 9]], dtype=torch.int32).pin_memory()
    ops.swap_blocks(dev_k, dev_v, host_k, host_v, in_pairs)
    torch.cuda.synchronize()
    k, v = _bits(dev_k), _bits(dev_v)
    for s, d_ in [(3, 7), (17, 8), (39, 9)]:
        assert np.array_equal(k[d_], k0[s]) and np.array_equal(v[d_], v0[s])
    others = [i for i in range(40) if i not in (7, 8, 9)]
    assert not k[others].any() and not v[others].any()


@requires_gpu
def test_swap_between_two_device_pools_and_reject_mismatched_shapes():
    a_k = _cache(8, 16, 4, 128, torch.bfloat16, "cuda", 5)
    a_v = _cache(8, 16, 4, 128, torch.bfloat16, "cuda", 6)
    b_k = _cache(6, 16, 4, 128, torch.bfloat16, "cuda", 7)
    b_v = _cache(6, 16, 4, 128, torch.bfloat16, "cuda", 8)
    pairs = torch.tensor([[5, 0], [2, 5]], dtype=torch.int32, device="cuda")
    ops.swap_blocks(b_k, b_v, a_k, a_v, pairs)
    torch.cuda.synchronize()
    # compare bits: random bf16 bit patterns include NaNs
    assert np.array_equal(_bits(b_k[0]), _bits(a_k[5]))
    assert np.array_equal(_bits(b_v[5]), _bits(a_v[2]))
    with pytest.raises(ValueError):
        ops.swap_blocks(b_k, b_v, _cache(6, 16, 8, 128, torch.bfloat16, "cuda", 9), a_v, pairs)
