"""Block pool and block-table pins.

Each test runs on the oracle's pure-Python pool model and, when the native
library is built, on the product's C pool (through ``paged_kv_cache_108_gb300.pool``)
-- the two share no code.  The expected values are the pages' printed ones
(tests/golden/pool_traces.json)."""
import json
import os

import numpy as np
import pytest

from oracle import pool_model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
with open(os.path.join(GOLDEN, "pool_traces.json")) as f:
    G = json.load(f)


def _native():
    from paged_kv_cache_108_gb300 import pool as native_pool
    native_pool.load()  # raises if the library cannot be built/loaded
    return native_pool


def _impls():
    impls = [("model", pool_model.BlockPoolModel, pool_model.SequenceTablesModel,
              pool_model.slot_of)]
    try:
        npool = _native()

        def native_slot(table, pos, block_size):
            return int(npool.slot_mapping(np.asarray([table], dtype=np.int32), block_size, [pos])[0])

        impls.append(("native", npool.BlockPool, npool.SequenceTables, native_slot))
    except Exception as e:  # noqa: BLE001 -- reported as a skip below
        impls.append(pytest.param(("native", None, None, None),
                                  marks=pytest.mark.skip(reason=f"native pool unavailable: {e}")))
    return impls


IMPLS = _impls()
IDS = ["model", "native"]


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_fifo_free_queue_and_slots(impl):
    _, Pool, _, slot_fn = impl
    g = G["fifo_example"]
    pool = Pool(g["num_blocks"])
    table = pool.allocate(3)
    assert list(table) == g["first_alloc"] and pool.num_free() == g["free_after_first"]
    pool.allocate(g["second_alloc_n"])
    pool.free(table)
    got = pool.allocate(g["third_alloc_n"])
    assert list(got) == g["third_alloc"]
    slots = [slot_fn(got, p, g["slot_block_size"]) for p in range(g["slot_positions"])]
    assert slots == g["slots"]


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_round_robin_tables(impl):
    _, Pool, _, _ = impl
    g = G["round_robin_tables"]
    pool = Pool(g["num_blocks"])
    B = g["block_size"]
    tables = [[] for _ in g["seq_lens"]]
    while any(len(t) * B < s for t, s in zip(tables, g["seq_lens"])):
        for t, s in zip(tables, g["seq_lens"]):
            if len(t) * B < s:
                t += list(pool.allocate(1))
    assert tables == g["tables"]


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_block_boundary_grow_before_write(impl):
    _, Pool, Seqs, _ = impl
    g = G["block_boundary"]
    B = g["block_size"]
    mgr = Seqs(Pool(g["num_blocks"]), B)
    mgr.allocate("s", g["prompt_len"])
    assert len(mgr.tables["s"]) == g["blocks_after_prefill"]
    for cur in range(g["prompt_len"], g["prompt_len"] + g["decode_steps"]):
        mgr.append_token("s", cur)
        slot = mgr.slot_index("s", cur)
        assert slot % B == cur % B
        assert slot // B == mgr.tables["s"][cur // B]
    assert len(mgr.tables["s"]) == g["blocks_after_decode"]


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_growth_trace_with_injected_free_order(impl):
    _, Pool, Seqs, _ = impl
    g = G["growth_trace"]
    B = g["block_size"]
    order = list(g["initial_table"]) + [g["next_free"]] + [b for b in range(16)
                                                          if b not in g["initial_table"] + [g["next_free"]]]
    mgr = Seqs(Pool(16, free_order=order), B)
    mgr.allocate("r", g["initial_tokens"])
    assert list(mgr.tables["r"]) == g["initial_table"]
    for tok in range(g["initial_tokens"], 13):
        mgr.append_token("r", tok)
    assert list(mgr.tables["r"]) == g["table_after_token_12"]
    assert mgr.slot_index("r", 12) == g["next_free"] * B


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_can_allocate_all_or_nothing(impl):
    _, Pool, _, _ = impl
    g = G["can_allocate"]
    for tokens, fits in g["cases"]:
        pool = Pool(g["num_blocks"])
        need = -(-tokens // g["block_size"])
        got = pool.allocate(need)
        assert (got is not None) == fits
        # a refused request leaves the pool untouched
        assert pool.num_free() == (g["num_blocks"] - need if fits else g["num_blocks"])


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_fork_and_copy_on_write(impl):
    _, Pool, Seqs, _ = impl
    B = 4
    pool = Pool(10)
    mgr = Seqs(pool, B)
    mgr.allocate("p", 6)  # blocks [0, 1], last one half full
    mgr.fork("p", "c")
    assert pool.refcount(0) == 2 and pool.refcount(1) == 2
    # child writes position 6: block 1 is shared -> copy to a fresh block
    src, dst = mgr.cow_for_write("c", 6)
    assert (src, dst) == (1, 2)
    assert list(mgr.tables["c"]) == [0, 2] and list(mgr.tables["p"]) == [0, 1]
    assert pool.refcount(1) == 1 and pool.refcount(2) == 1
    # parent now owns block 1 alone: writes in place
    assert mgr.cow_for_write("p", 6) == (1, 1)
    mgr.free_seq("p")
    assert pool.refcount(0) == 1 and pool.refcount(1) == 0
    mgr.free_seq("c")
    assert pool.num_free() == 10


@pytest.mark.parametrize("impl", IMPLS, ids=IDS)
def test_exhaustion(impl):
    _, Pool, Seqs, _ = impl
    pool = Pool(2)
    mgr = Seqs(pool, 4)
    mgr.allocate("a", 8)
    with pytest.raises(Exception):
        mgr.append_token("a", 8)
    assert pool.num_free() == 0 and len(mgr.tables["a"]) == 2


def test_native_matches_model_on_random_ops():
    """Random alloc / fork / cow / free sequences give identical tables and
    free queues on the native pool and the oracle model."""
    try:
        npool = _native()
    except Exception as e:  # noqa: BLE001
        pytest.skip(f"native pool unavailable: {e}")
    rng = np.random.default_rng(3)
    for trial in range(20):
        nb, B = int(rng.integers(8, 64)), int(rng.choice([1, 4, 16]))
        order = rng.permutation(nb).tolist()
        ma = pool_model.SequenceTablesModel(pool_model.BlockPoolModel(nb, order), B)
        mb = npool.SequenceTables(npool.BlockPool(nb, free_order=order), B)
        lens = {}
        for step in range(200):
            op = rng.integers(0, 4)
            live = sorted(lens)
            try:
                if op == 0 or not live:
                    s, n = f"s{step}", int(rng.integers(1, 3 * B + 1))
                    ra = rb = None
                    try:
                        ma.allocate(s, n)
                    except pool_model.PoolExhausted:
                        ra = "oom"
                    try:
                        mb.allocate(s, n)
                    except Exception:  # noqa: BLE001
                        rb = "oom"
                    assert ra == rb
                    if ra is None:
                        lens[s] = n
                elif op == 1:
                    s = live[int(rng.integers(len(live)))]
                    c = f"f{step}"
                    ma.fork(s, c)
                    mb.fork(s, c)
                    lens[c] = lens[s]
                elif op == 2:
                    s = live[int(rng.integers(len(live)))]
                    pos = lens[s]
                    ra = rb = None
                    try:
                        ma.append_token(s, pos)
                        ra = ma.cow_for_write(s, pos)
                    except pool_model.PoolExhausted:
                        ra = "oom"
                    try:
                        mb.append_token(s, pos)
                        rb = mb.cow_for_write(s, pos)
                    except Exception:  # noqa: BLE001
                        rb = "oom"
                    assert ra == (tuple(rb) if rb != "oom" else rb)
                    if ra == "oom":
                        # both refused; drop the sequence to keep going
                        ma.free_seq(s)
                        mb.free_seq(s)
                        del lens[s]
                    else:
                        lens[s] = pos + 1
                else:
                    s = live[int(rng.integers(len(live)))]
                    ma.free_seq(s)
                    mb.free_seq(s)
                    del lens[s]
            finally:
                assert {k: list(v) for k, v in ma.tables.items()} == \
                       {k: list(v) for k, v in mb.tables.items()}
                assert ma.pool.num_free() == mb.pool.num_free()
        assert ma.pool.free_order() == list(mb.pool.free_order())
