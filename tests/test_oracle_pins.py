"""Pins of the fp64 oracle against what the source pages and mathematics fix.

Nothing here touches the product library or a GPU.  Each test names the
passage or identity it checks.  The pins are chosen so that a plausible slip
in the oracle (dropped scale, wrong GQA index, transposed operand, wrong
block/offset split, wrong rounding rule) fails at least one of them.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

from oracle import accounting, core
from paged_kv_cache_108_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- accounting

def test_kv_bytes_llama3_8b():
    g = _golden("kv_sizes.json")["llama3_8b_8192"]
    b = accounting.kv_cache_bytes(g["layers"], g["kv_heads"], g["head_dim"],
                                  g["seq_len"], g["bytes_per_elem"])
    assert b == g["bytes"] == 1073741824
    # 64 streams, the page prints 64 x 1.07 GB = 68.48 (decimal GB, 2 digits)
    assert round(round(b / 1e9, 2) * 64, 2) == g["batch64_gb_decimal_printed"]


def test_kv_bytes_llama2_13b_and_beta():
    g = _golden("kv_sizes.json")["llama2_13b_2048"]
    b = accounting.kv_cache_bytes(g["layers"], g["kv_heads"], g["head_dim"],
                                  g["seq_len"], g["bytes_per_elem"])
    assert f"{b / 2**30:.2f}" == g["gib_printed"]
    beta = accounting.kv_cache_bytes(g["layers"], g["kv_heads"], g["head_dim"], 1)
    assert f"{beta / 2**20:.3f}" == g["beta_mib_printed"]


def test_kv_bytes_small_model_and_per_token():
    g = _golden("kv_sizes.json")
    s = g["stack100m_beta"]
    assert accounting.kv_cache_bytes(s["layers"], s["kv_heads"], s["head_dim"], 1) == s["bytes"]
    l3 = g["llama3_8b_per_token_kib"]
    assert accounting.kv_cache_bytes(l3["layers"], l3["kv_heads"], l3["head_dim"], 1) == l3["bytes"]


def test_concurrency_qwen():
    g = _golden("kv_sizes.json")["qwen25_7b"]
    per_tok = accounting.kv_cache_bytes(g["layers"], g["kv_heads"], g["head_dim"], 1)
    assert per_tok == g["per_token_bytes"]
    budget = g["budget_gib"] * 1024**3
    paged = budget // (math.ceil(g["avg_ctx"] / g["block_size"]) * g["block_size"] * per_tok)
    pre = budget // (g["max_ctx"] * per_tok)
    assert (paged, pre) == (g["paged_concurrent"], g["prealloc_concurrent"])


def test_waste_and_concurrency_exercises():
    g = _golden("kv_sizes.json")
    w = g["waste_exercise"]
    used = accounting.utilisation(w["actual"], max_len=w["reserved_tokens_each"])
    # the page rounds used bytes to 0.244 GiB before subtracting
    assert f"{(1 - round(used, 3)) * 100:.1f}" == w["wasted_pct_printed"]
    c = g["concurrency_exercise"]
    per_req_static = c["max_len"] * c["kib_per_token"]
    per_req_paged = math.ceil(c["avg_len"] / c["block_size"]) * c["block_size"] * c["kib_per_token"]
    pool_kib = c["pool_gib"] * 1024 * 1024
    assert pool_kib // per_req_static == c["static_requests"]
    assert pool_kib // per_req_paged == c["paged_requests"]
    assert c["paged_requests"] // c["static_requests"] == c["multiplier"]


def test_utilisation_request_mix():
    g = _golden("utilisation.json")
    lengths = [p + o for p, o in synth.request_mix(200)]
    assert f"{accounting.utilisation(lengths, max_len=g['max_len']):.1%}" == g["reservation_pct_printed"]
    for bs, printed in g["paged_pct_printed"].items():
        assert f"{accounting.utilisation(lengths, block_size=int(bs)):.1%}" == printed


def test_request_mix_is_the_pages_generator():
    # the page's own statement of the generator, re-run with the stdlib
    random.seed(0)
    reqs = [(random.randint(100, 2000), random.randint(20, 1500)) for _ in range(200)]
    assert reqs == synth.request_mix(200)
    lens = synth.llama8b_lengths(64)
    assert (sum(lens), min(lens), max(lens)) == (121416, 732, 3360)


# ---------------------------------------------------------------- formats

def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_spec_points_and_library():
    dec = core.e4m3_decode(np.arange(256, dtype=np.uint8))
    # spec corner values: largest finite, smallest normal, smallest subnormal, one
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x08] == 2.0**-6 and dec[0x01] == 2.0**-9 and dec[0x38] == 1.0
    assert dec[0x3C] == 1.5 and dec[0x00] == 0.0 and math.copysign(1, dec[0x80]) == -1
    assert math.isnan(dec[0x7F]) and math.isnan(dec[0xFF])
    ref = _torch_e4m3_values()  # library decoding of every code
    finite = ~np.isnan(ref)
    assert np.array_equal(dec[finite], ref[finite])
    assert np.array_equal(np.isnan(dec), np.isnan(ref))


def _all_finite_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << np.uint32(16)).view(np.float32)
    return f[np.isfinite(f)]


def test_e4m3_encode_is_nearest_ties_to_even_exhaustive():
    """Every finite bf16 value: the code is the nearest finite e4m3 value,
    ties going to the even code, magnitudes above 448 saturating."""
    x = _all_finite_bf16_as_f32()
    got = core.e4m3_encode(x)
    vals = _torch_e4m3_values()
    codes = np.array([c for c in range(256) if not np.isnan(vals[c])], dtype=np.int64)
    cv = vals[codes]
    xd = x.astype(np.float64)
    # brute force over all finite codes, chunked to bound memory
    want = np.empty(x.shape, dtype=np.uint8)
    for s in range(0, x.size, 4096):
        xs = xd[s:s + 4096, None]
        dist = np.abs(xs - cv[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # among ties prefer an even mantissa, then the code with x's sign
        score = cand * 4 + cand * ((codes[None, :] & 1) == 0) * 2 \
            + cand * ((codes[None, :] >> 7) == (np.signbit(xs)).astype(np.int64))
        want[s:s + 4096] = codes[np.argmax(score, axis=1)]
    big = np.abs(xd) > 448.0
    want[big] = np.where(np.signbit(x[big]), 0xFE, 0x7E)
    assert np.array_equal(got, want)


def test_e4m3_encode_matches_library_cast_in_range():
    x = _all_finite_bf16_as_f32()
    x = x[np.abs(x) <= 448.0]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = core.e4m3_encode(x)
    zero = x == 0  # sign of zero may differ between conventions; both decode to 0
    assert np.array_equal(got[~zero], lib[~zero])


def test_e4m3_encode_f32_boundaries():
    # halfway cases straddling the subnormal/normal seam and the top binade
    cases = {2.0**-10: 0x00,              # half of the smallest subnormal -> even (0)
             3 * 2.0**-10: 0x02,          # 1.5 steps -> 2 (even)
             15 * 2.0**-10: 0x08,         # 7.5 steps -> 8 = smallest normal
             464.0: 0x7E, 1e30: 0x7E,     # saturation
             -1e30: 0xFE, 0.0: 0x00,
             1.0625: 0x38,                # 1 + 1/16: tie between 1.0 (even) and 1.125
             1.1875: 0x3A}                # 1 + 3/16: tie between 1.125 and 1.25 (even)
    x = np.array(list(cases), dtype=np.float32)
    assert list(core.e4m3_encode(x)) == list(cases.values())


# ---------------------------------------------------------------- cache write

def _empty_cache(nb, B, hkv, d, dtype=np.uint16):
    return np.zeros((nb, B, hkv, d), dtype=dtype)


def test_reshape_and_cache_slot_example():
    g = _golden("pool_traces.json")["fifo_example"]
    B, hkv, d = g["slot_block_size"], 2, 8
    rng = np.random.default_rng(0)
    k = rng.integers(1, 1 << 15, size=(len(g["slots"]), hkv, d), dtype=np.uint16)
    v = rng.integers(1, 1 << 15, size=k.shape, dtype=np.uint16)
    kc, vc = _empty_cache(8, B, hkv, d), _empty_cache(8, B, hkv, d)
    core.reshape_and_cache(k, v, kc, vc, np.array(g["slots"], dtype=np.int32))
    # the page's flat view: pool.view(-1, H_kv, d)[slot] holds token i
    assert np.array_equal(kc.reshape(-1, hkv, d)[g["slots"]], k)
    assert np.array_equal(vc.reshape(-1, hkv, d)[g["slots"]], v)
    # positions 12, 13 live in physical block 0 at offsets 0, 1
    assert np.array_equal(kc[0, 0], k[12]) and np.array_equal(kc[0, 1], k[13])
    untouched = np.ones(8 * B, dtype=bool)
    untouched[g["slots"]] = False
    assert not kc.reshape(-1, hkv, d)[untouched].any()


def test_reshape_and_cache_negative_slot_skips():
    kc, vc = _empty_cache(4, 4, 1, 8), _empty_cache(4, 4, 1, 8)
    k = np.full((3, 1, 8), 7, dtype=np.uint16)
    core.reshape_and_cache(k, k, kc, vc, np.array([-1, 5, -7], dtype=np.int32))
    flat = kc.reshape(-1, 1, 8)
    assert (flat[5] == 7).all() and flat.sum() == 7 * 8


def test_reshape_and_cache_rejects_out_of_pool_slot():
    kc, vc = _empty_cache(2, 4, 1, 8), _empty_cache(2, 4, 1, 8)
    k = np.zeros((1, 1, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        core.reshape_and_cache(k, k, kc, vc, np.array([8], dtype=np.int32))


def test_reshape_and_cache_fp8_is_encode_of_fp32_quotient():
    rng = np.random.default_rng(1)
    k = synth.normal_bf16(rng, (5, 2, 16))
    v = synth.normal_bf16(rng, (5, 2, 16))
    ks = synth.per_tensor_scale(k)
    vs = synth.per_tensor_scale(v)
    kc, vc = _empty_cache(3, 4, 2, 16, np.uint8), _empty_cache(3, 4, 2, 16, np.uint8)
    slots = np.array([0, 3, 4, 9, 11], dtype=np.int32)
    core.reshape_and_cache(k, v, kc, vc, slots, ks, vs)
    kf = core.bf16_to_f64(k).astype(np.float32)
    want = core.e4m3_encode(kf / np.float32(ks))  # numpy fp32 division is IEEE
    assert np.array_equal(kc.reshape(-1, 2, 16)[slots], want)
    # the per-tensor scale maps the largest magnitude onto 448 (code 0x7E)
    assert (kc.reshape(-1, 2, 16)[slots] & 0x7F).max() == 0x7E
    # dequantised values are within half an e4m3 step (2^-4 relative) of the input
    deq = core.e4m3_decode(kc.reshape(-1, 2, 16)[slots]) * ks
    kd = core.bf16_to_f64(k)
    assert np.all(np.abs(deq - kd) <= np.maximum(np.abs(kd) * 2.0**-4, 2.0**-10 * ks) + 1e-12)


def test_copy_blocks():
    rng = np.random.default_rng(2)
    kc = rng.integers(0, 1 << 16, size=(6, 4, 2, 8), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(6, 4, 2, 8), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    core.copy_blocks(kc, vc, np.array([[1, 4], [2, 5]], dtype=np.int32))
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(kc[5], k0[2])
    assert np.array_equal(vc[4], v0[1]) and np.array_equal(vc[5], v0[2])
    for b in (0, 1, 2, 3):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    core.copy_blocks(kc, vc, np.zeros((0, 2), dtype=np.int32))  # no pairs: no-op
    with pytest.raises(ValueError):
        core.copy_blocks(kc, vc, np.array([[0, 6]], dtype=np.int32))


# ---------------------------------------------------------------- decode

def _paged_from_contiguous(K, V, B, nb, rng):
    """Scatter contiguous per-sequence K/V [n, H_kv, d] into a shuffled pool
    with the pages' write path: slot = table[p // B] * B + p % B."""
    hkv, d = K[0].shape[1:]
    perm = rng.permutation(nb).astype(np.int32)
    kc = rng.integers(0, 1 << 16, size=(nb, B, hkv, d), dtype=np.uint16)  # junk
    vc = rng.integers(0, 1 << 16, size=(nb, B, hkv, d), dtype=np.uint16)
    maxb = max(1, max(-(-k.shape[0] // B) for k in K))
    tables = np.zeros((len(K), maxb), dtype=np.int32)
    at = 0
    for i, (k, v) in enumerate(zip(K, V)):
        c = -(-k.shape[0] // B)
        tables[i, :c] = perm[at:at + c]
        at += c
        slots = [tables[i, p // B] * B + p % B for p in range(k.shape[0])]
        kc.reshape(-1, hkv, d)[slots] = k
        vc.reshape(-1, hkv, d)[slots] = v
    return kc, vc, tables


def _sdpa_reference(q, K, V, scale):
    """torch SDPA in fp64 on contiguous K/V, GQA by repeat_interleave."""
    H = q.shape[0]
    hkv = K.shape[1]
    kt = torch.from_numpy(core.bf16_to_f64(K)).repeat_interleave(H // hkv, dim=1)
    vt = torch.from_numpy(core.bf16_to_f64(V)).repeat_interleave(H // hkv, dim=1)
    qt = torch.from_numpy(core.bf16_to_f64(q))
    o = torch.nn.functional.scaled_dot_product_attention(
        qt[:, None, :], kt.transpose(0, 1), vt.transpose(0, 1), scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("H,hkv,d,B", [(4, 4, 16, 4), (8, 2, 64, 4), (4, 2, 64, 16), (32, 8, 128, 16)])
def test_decode_paged_equals_unpaged_sdpa(H, hkv, d, B):
    """Paged attention equals attention on contiguous storage ("Paged KV
    cache", section 'Paged attention', the check against
    F.scaled_dot_product_attention)."""
    rng = np.random.default_rng(H * 100 + d)
    lens = [37, 5, 20, 1, 16, 17]
    K = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    V = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    q = synth.normal_bf16(rng, (len(lens), H, d))
    nb = sum(-(-n // B) for n in lens) + 3
    kc, vc, tables = _paged_from_contiguous(K, V, B, nb, rng)
    scale = d ** -0.5
    out = core.decode(q, kc, vc, tables, np.array(lens, dtype=np.int32), scale)
    for i in range(len(lens)):
        ref = _sdpa_reference(q[i], K[i], V[i], scale)
        assert np.max(np.abs(out[i] - ref)) < 1e-12


def _streaming_decode(q, kc, vc, table, n, B, G, scale):
    """Per-token online softmax exactly as the kernel sketch of "4.6
    PagedAttention & KV-Cache Memory Management" walks it: block by block,
    token by token, running max / denominator / accumulator (pure Python)."""
    H, d = q.shape
    qf = core.bf16_to_f64(q)
    out = [[0.0] * d for _ in range(H)]
    m = [-math.inf] * H
    l = [0.0] * H
    for lb in range(-(-n // B)):
        phys = int(table[lb])
        valid = min(B, n - lb * B)
        for t in range(valid):
            for h in range(H):
                k = core.bf16_to_f64(kc[phys, t, h // G])
                v = core.bf16_to_f64(vc[phys, t, h // G])
                logit = scale * float(np.dot(qf[h], k))
                m_new = max(m[h], logit)
                alpha = math.exp(m[h] - m_new)
                p = math.exp(logit - m_new)
                l[h] = l[h] * alpha + p
                out[h] = [o * alpha + p * vv for o, vv in zip(out[h], v)]
                m[h] = m_new
    return np.array([[o / l[h] for o in out[h]] for h in range(H)])


def test_decode_brute_force_streaming_tiny():
    rng = np.random.default_rng(5)
    H, hkv, d, B = 4, 2, 8, 4
    lens = [1, 4, 5, 11]
    K = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    V = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    q = synth.normal_bf16(rng, (len(lens), H, d))
    kc, vc, tables = _paged_from_contiguous(K, V, B, 12, rng)
    out = core.decode(q, kc, vc, tables, np.array(lens, dtype=np.int32), 0.37)
    for i, n in enumerate(lens):
        ref = _streaming_decode(q[i], kc, vc, tables[i], n, B, H // hkv, 0.37)
        assert np.max(np.abs(out[i] - ref)) < 1e-12


def test_decode_single_token_returns_v_exactly():
    rng = np.random.default_rng(6)
    kc = rng.integers(0, 1 << 16, size=(4, 16, 2, 64), dtype=np.uint16)
    vc = synth.normal_bf16(rng, (4, 16, 2, 64))
    q = synth.normal_bf16(rng, (1, 4, 64))
    kc[2, 0] = synth.normal_bf16(rng, (2, 64))
    out = core.decode(q, kc, vc, np.array([[2]], dtype=np.int32), np.array([1], dtype=np.int32), 0.125)
    want = core.bf16_to_f64(vc[2, 0])
    assert np.array_equal(out[0, 0], want[0]) and np.array_equal(out[0, 1], want[0])
    assert np.array_equal(out[0, 2], want[1]) and np.array_equal(out[0, 3], want[1])


def test_decode_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(7)
    n, B, d = 23, 4, 16
    krow = synth.normal_bf16(rng, (1, 1, d))
    K = np.repeat(krow, n, axis=0)
    V = synth.normal_bf16(rng, (n, 1, d))
    q = synth.normal_bf16(rng, (1, 2, d))
    kc, vc, tables = _paged_from_contiguous([K], [V], B, 8, rng)
    out = core.decode(q, kc, vc, tables, np.array([n], dtype=np.int32), 0.3)
    mean = core.bf16_to_f64(V)[:, 0, :].mean(axis=0)
    assert np.max(np.abs(out[0, 0] - mean)) < 1e-13 and np.max(np.abs(out[0, 1] - mean)) < 1e-13


def test_decode_dominant_key_selects_its_value():
    rng = np.random.default_rng(8)
    n, B, d = 30, 16, 32
    K = synth.normal_bf16(rng, (n, 1, d))
    V = synth.normal_bf16(rng, (n, 1, d))
    q = synth.normal_bf16(rng, (1, 1, d))
    qf = core.bf16_to_f64(q[0, 0])
    K[17, 0] = synth.bf16_bits((np.sign(qf) * 8.0).astype(np.float32))
    kc, vc, tables = _paged_from_contiguous([K], [V], B, 4, rng)
    out = core.decode(q, kc, vc, tables, np.array([n], dtype=np.int32), 1.0)
    assert np.max(np.abs(out[0, 0] - core.bf16_to_f64(V[17, 0]))) < 1e-9


def test_decode_permutation_invariance_bit_identical():
    rng = np.random.default_rng(9)
    H, hkv, d, B = 8, 2, 32, 4
    lens = [13, 1, 8, 21]
    K = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    V = [synth.normal_bf16(rng, (n, hkv, d)) for n in lens]
    q = synth.normal_bf16(rng, (len(lens), H, d))
    cl = np.array(lens, dtype=np.int32)
    a = core.decode(q, *_paged_from_contiguous(K, V, B, 16, np.random.default_rng(1)), cl, 0.2)
    b = core.decode(q, *_paged_from_contiguous(K, V, B, 40, np.random.default_rng(2)), cl, 0.2)
    assert np.array_equal(a, b)


def test_decode_gqa_uses_group_kv_head():
    """Query head h reads KV head h // G: swapping the two KV heads' data
    must swap which query heads see which values."""
    rng = np.random.default_rng(10)
    H, hkv, d, B, n = 4, 2, 16, 4, 9
    K = synth.normal_bf16(rng, (n, hkv, d))
    V = synth.normal_bf16(rng, (n, hkv, d))
    q = synth.normal_bf16(rng, (1, H, d))
    kc, vc, t = _paged_from_contiguous([K], [V], B, 4, rng)
    out = core.decode(q, kc, vc, t, np.array([n], dtype=np.int32), 0.25)
    q_sw = q[:, [2, 3, 0, 1], :].copy()
    kc2, vc2, t2 = _paged_from_contiguous([K[:, ::-1].copy()], [V[:, ::-1].copy()], B, 4, rng)
    out2 = core.decode(q_sw, kc2, vc2, t2, np.array([n], dtype=np.int32), 0.25)
    assert np.max(np.abs(out[0, [2, 3, 0, 1]] - out2[0])) < 1e-13


def test_decode_empty_context_and_unread_padding():
    rng = np.random.default_rng(11)
    kc = synth.normal_bf16(rng, (4, 4, 1, 8))
    vc = synth.normal_bf16(rng, (4, 4, 1, 8))
    q = synth.normal_bf16(rng, (2, 1, 8))
    tables = np.array([[1, 10**6, -5], [10**6, 10**6, 10**6]], dtype=np.int32)
    out = core.decode(q, kc, vc, tables, np.array([3, 0], dtype=np.int32), 0.5, out=np.full((2, 1, 8), 9.0))
    assert np.all(out[1] == 0.0)
    assert np.all(np.isfinite(out[0]))
    with pytest.raises(ValueError):
        core.decode(q, kc, vc, tables, np.array([5, 0], dtype=np.int32), 0.5)


def test_decode_fp8_dequantises_with_scale():
    """An e4m3 cache decodes as code * scale: the fp8 oracle equals the bf16
    oracle on a cache holding exactly those dequantised values (here
    representable in bf16, since e4m3 values are a subset of bf16)."""
    rng = np.random.default_rng(12)
    codes_k = rng.integers(0, 256, size=(5, 4, 2, 16), dtype=np.uint8)
    codes_v = rng.integers(0, 256, size=(5, 4, 2, 16), dtype=np.uint8)
    for c in (codes_k, codes_v):
        c[(c & 0x7F) == 0x7F] = 0x3F  # no NaN codes in used slots
    ks, vs = 0.5, 0.25  # powers of two keep code*scale exact in bf16
    to_bf16 = lambda codes, s: synth.bf16_bits((core.e4m3_decode(codes) * s).astype(np.float32))
    q = synth.normal_bf16(rng, (2, 4, 16))
    tables = np.array([[3, 0, 4], [1, 2, 0]], dtype=np.int32)
    cl = np.array([11, 6], dtype=np.int32)
    a = core.decode(q, codes_k, codes_v, tables, cl, 0.25, k_scale=ks, v_scale=vs)
    b = core.decode(q, to_bf16(codes_k, ks), to_bf16(codes_v, vs), tables, cl, 0.25)
    assert np.array_equal(a, b)


def test_decode_threads_and_units_agree():
    w = synth.tiny()
    kc, vc = w.junk_k.copy(), w.junk_v.copy()
    rng = np.random.default_rng(13)
    kc[:] = synth.normal_bf16(rng, kc.shape)
    vc[:] = synth.normal_bf16(rng, vc.shape)
    a = core.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    b = core.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, nthreads=3)
    c = core.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, units=[(2, 1), (0, 0)])
    assert np.array_equal(a, b)
    assert np.array_equal(c[2, 2:], a[2, 2:]) and np.array_equal(c[0, :2], a[0, :2])
    assert not c[1].any()
