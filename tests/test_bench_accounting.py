"""The bench's algorithmic counts, pinned by brute force: the visible
(new token, key) pairs behind the prefill line's TFLOP/s, and the decode
line's algorithmic bytes against the figure the hot-path table states for
the batch-64 layer."""
import numpy as np

import bench
from paged_kv_cache_108_gb300 import synth


def _pairs_brute(lens, T):
    total = 0
    for n in lens:
        for j in range(T):
            pos = n - T + j           # the token's position
            total += pos + 1          # keys 0 .. pos
    return total


def test_causal_pairs_match_brute_force():
    rng = np.random.default_rng(5)
    for T in (1, 2, 7, 16, 33):
        lens = [int(x) for x in rng.integers(T, 300, size=9)]
        assert bench.causal_pairs(lens, T) == _pairs_brute(lens, T)


def test_one_token_is_plain_decode():
    lens = [5, 16, 17, 40]
    assert bench.causal_pairs(lens, 1) == sum(lens)


def test_llama8b_decode_bytes_match_the_stated_figure():
    # 121,416 tokens x 8 KV heads x 128 x 2 bytes x (K and V) = 497,319,936;
    # + q and out (64 x 32 x 128 x 2 each) + 7,620 table entries + 64 lengths
    w = synth.llama8b(with_data=False)
    kv = int(np.sum(w.context_lens)) * 8 * 128 * 2 * 2
    assert kv == 497_319_936
    qo = 2 * 64 * 32 * 128 * 2
    table = sum(-(-int(n) // 16) for n in w.context_lens) * 4
    assert kv + qo + table + 64 * 4 == 498_399_248


def test_traffic_record_applies_only_to_the_source_it_was_taken_on(tmp_path, monkeypatch):
    # a record carries the sha-256 of the kernel sources it was captured on;
    # once one of them changes, the bench reports no traffic rather than a
    # figure taken on other code
    import hashlib
    import json
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    (tmp_path / "profiles").mkdir()
    rec = {"sources": ["k.cu"], "sources_sha256": hashlib.sha256(b"kernel v1").hexdigest(),
           "dram_bytes_per_call": 123}
    (tmp_path / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic(0) == 123
    assert bench.recorded_traffic(0, "fp8") is None  # no record for that cache type
    src.write_bytes(b"kernel v2")
    assert bench.recorded_traffic(0) is None


def test_committed_traffic_records_are_well_formed():
    import json
    import os
    for name in ("decode_traffic.json", "decode_traffic_fp8.json"):
        with open(os.path.join(bench.ROOT, "profiles", name)) as f:
            rec = json.load(f)
        assert all(os.path.exists(os.path.join(bench.ROOT, s)) for s in rec["sources"])
        assert rec["dram_bytes_per_call"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert "--clock-control none" in rec["command"]
