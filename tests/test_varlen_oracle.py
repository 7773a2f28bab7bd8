"""Pins of the fp64 varlen paged-attention oracle (oracle/varlen.py).

Checked against what the pages and the mathematics fix, not against the
oracle itself: the pages' printed three-request block tables, a scalar
brute-force attention loop on tiny inputs, closed forms (q = 0 averages the
visible V rows; the first prefill token sees only itself), equality with the
(separately pinned) decode oracle when each request has one new token,
invariance under any permutation of physical blocks, an E4M3 cache against a
scalar loop over torch's own E4M3 decoding, and the zero-row reading for a
request with more new tokens than context."""
import json
import math
import os

import numpy as np
import pytest

from oracle import core as ocore
from oracle import pool_model
from oracle import varlen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "varlen_example.json")


def _bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _interleaved_tables(seq_lens, B, num_blocks, order=None):
    """The pages' procedure: one block at a time, request by request, in turn."""
    pool = pool_model.BlockPoolModel(num_blocks, order)
    tables = [[] for _ in seq_lens]
    while any(len(t) * B < s for t, s in zip(tables, seq_lens)):
        for t, s in zip(tables, seq_lens):
            if len(t) * B < s:
                t += pool.allocate(1)
    return tables


def _case(seq_lens, query_lens, H, Hkv, d, B, num_blocks, seed, order=None):
    """Contiguous K/V per request written into a pool by the slot formula."""
    rng = np.random.default_rng(seed)
    tables = _interleaved_tables(seq_lens, B, num_blocks, order)
    kc = np.zeros((num_blocks, B, Hkv, d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    ks, vs = [], []
    for t, s in zip(tables, seq_lens):
        k = _bf16(rng.standard_normal((s, Hkv, d)))
        v = _bf16(rng.standard_normal((s, Hkv, d)))
        for p in range(s):
            kc[t[p // B], p % B] = k[p]
            vc[t[p // B], p % B] = v[p]
        ks.append(k)
        vs.append(v)
    q = _bf16(rng.standard_normal((sum(query_lens), H, d)))
    qsl = np.concatenate([[0], np.cumsum(query_lens)]).astype(np.int64)
    padded = np.zeros((len(tables), max(len(t) for t in tables)), dtype=np.int32)
    for i, t in enumerate(tables):
        padded[i, :len(t)] = t
    return dict(q=q, kc=kc, vc=vc, ks=ks, vs=vs, tables=padded, qsl=qsl,
                seq_lens=np.array(seq_lens), H=H, Hkv=Hkv, d=d)


def test_pages_three_request_tables():
    g = json.load(open(GOLDEN))
    got = _interleaved_tables(g["seq_lens"], g["block_size"], g["num_blocks"])
    assert got == g["printed_tables"]


def test_matches_scalar_brute_force_on_tiny_inputs():
    c = _case([7, 3, 9], [2, 3, 4], 4, 2, 8, 2, 16, seed=3)
    out = varlen.varlen_attention(c["q"], c["kc"], c["vc"], c["tables"], c["seq_lens"],
                                  c["qsl"], scale=0.35)
    rep = c["H"] // c["Hkv"]
    for i, s in enumerate(c["seq_lens"]):
        a, b = int(c["qsl"][i]), int(c["qsl"][i + 1])
        n = b - a
        k, v = _f(c["ks"][i]), _f(c["vs"][i])
        for j in range(n):
            pos = s - n + j
            for h in range(c["H"]):
                qv = _f(c["q"][a + j, h])
                logits = [0.35 * sum(qv[e] * k[t, h // rep, e] for e in range(c["d"]))
                          for t in range(pos + 1)]
                mx = max(logits)
                w = [math.exp(x - mx) for x in logits]
                tot = sum(w)
                for e in range(c["d"]):
                    ref = sum(w[t] * v[t, h // rep, e] for t in range(pos + 1)) / tot
                    assert abs(out[a + j, h, e] - ref) < 1e-12


def test_zero_query_averages_the_visible_rows():
    c = _case([37, 5, 20], [1, 5, 8], 8, 2, 64, 4, 32, seed=5)
    q0 = np.zeros_like(c["q"])
    out = varlen.varlen_attention(q0, c["kc"], c["vc"], c["tables"], c["seq_lens"], c["qsl"],
                                  scale=0.125)
    rep = 4
    for i, s in enumerate(c["seq_lens"]):
        a, b = int(c["qsl"][i]), int(c["qsl"][i + 1])
        v = _f(c["vs"][i])
        for j in range(b - a):
            pos = s - (b - a) + j
            want = np.repeat(v[:pos + 1].mean(axis=0), rep, axis=0)
            np.testing.assert_allclose(out[a + j], want, rtol=0, atol=1e-12)


def test_first_prefill_token_sees_only_itself():
    c = _case([5], [5], 8, 2, 64, 4, 8, seed=7)
    out = varlen.varlen_attention(c["q"], c["kc"], c["vc"], c["tables"], c["seq_lens"],
                                  c["qsl"], scale=0.125)
    assert np.array_equal(out[0], np.repeat(_f(c["vs"][0][0]), 4, axis=0))


def test_one_new_token_per_request_is_the_decode_oracle():
    c = _case([37, 5, 20, 1], [1, 1, 1, 1], 8, 2, 64, 4, 32, seed=9)
    out = varlen.varlen_attention(c["q"], c["kc"], c["vc"], c["tables"], c["seq_lens"],
                                  c["qsl"], scale=0.125)
    dec = ocore.decode(c["q"], c["kc"], c["vc"], c["tables"], c["seq_lens"].astype(np.int32),
                       0.125)
    np.testing.assert_allclose(out, dec, rtol=0, atol=1e-12)


def test_any_block_permutation_gives_the_same_output():
    base = _case([37, 5, 20], [1, 5, 8], 8, 2, 64, 4, 32, seed=11)
    perm = np.random.default_rng(1).permutation(32).tolist()
    moved = _case([37, 5, 20], [1, 5, 8], 8, 2, 64, 4, 32, seed=11, order=perm)
    o1 = varlen.varlen_attention(base["q"], base["kc"], base["vc"], base["tables"],
                                 base["seq_lens"], base["qsl"], 0.125)
    o2 = varlen.varlen_attention(moved["q"], moved["kc"], moved["vc"], moved["tables"],
                                 moved["seq_lens"], moved["qsl"], 0.125)
    assert np.array_equal(o1, o2)


def test_e4m3_cache_matches_brute_force_over_torch_decoding():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    B, Hkv, H, d, nb = 4, 2, 4, 16, 12
    kc = rng.integers(0, 256, size=(nb, B, Hkv, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, B, Hkv, d), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x11   # keep NaN codes out of the context
    vc[(vc & 0x7F) == 0x7F] = 0x22
    tables = np.array([[3, 7, 1], [10, 0, 5]], dtype=np.int32)
    seq_lens, qlens = [11, 6], [3, 2]
    qsl = np.array([0, 3, 5])
    q = _bf16(rng.standard_normal((5, H, d)))
    ks, vs = 0.03125, 0.75
    out = varlen.varlen_attention(q, kc, vc, tables, seq_lens, qsl, 0.2, ks, vs)

    def deq(codes, s):
        return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy() * s

    for r in range(2):
        for j in range(qlens[r]):
            last = seq_lens[r] - qlens[r] + j
            for h in range(H):
                g = h // (H // Hkv)
                rows = [(tables[r][t // B], t % B) for t in range(last + 1)]
                kk = np.array([deq(kc[b, o, g], ks) for b, o in rows])
                vv = np.array([deq(vc[b, o, g], vs) for b, o in rows])
                qv = _f(q[qsl[r] + j, h])
                lg = [0.2 * float(np.dot(qv, kk[t])) for t in range(last + 1)]
                mx = max(lg)
                w = np.array([math.exp(x - mx) for x in lg])
                want = (w[:, None] * vv).sum(axis=0) / w.sum()
                np.testing.assert_allclose(out[qsl[r] + j, h], want, rtol=0, atol=1e-12)


def test_more_new_tokens_than_context_gives_zero_rows():
    c = _case([12, 9], [3, 4], 4, 2, 8, 4, 16, seed=17)
    seq_lens = np.array([12, 2])          # request 1: 4 new tokens, 2 in its context
    out = varlen.varlen_attention(c["q"], c["kc"], c["vc"], c["tables"], seq_lens, c["qsl"],
                                  scale=0.3)
    assert not out[3:].any()
    alone = varlen.varlen_attention(c["q"][:3], c["kc"], c["vc"], c["tables"][:1],
                                    seq_lens[:1], c["qsl"][:2], scale=0.3)
    assert np.array_equal(out[:3], alone)
