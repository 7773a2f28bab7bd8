"""Prefix caching across requests in the host pool (full blocks only).

Pins from the pages: a shared prompt's full blocks are stored once and
reused by later requests (their K/V need not be recomputed), a partly filled
last block is never shared (each request writes into its own block), blocks
are released to the free queue and reused in freeing order.  Every hand
trace runs on the oracle's model and on the native pool, each on its own;
then the two are compared on random request traces."""
import random

import pytest

from oracle.pool_model import PrefixCachePoolModel
from paged_kv_cache_108_gb300 import pool

B = 16


def _native(n, order=None):
    p = pool.BlockPool(n, free_order=order)
    p.enable_prefix_cache(B)
    return p


def _model(n, order=None):
    return PrefixCachePoolModel(n, B, free_order=order)


@pytest.fixture(params=["model", "native"])
def make_pool(request):
    return _model if request.param == "model" else _native


def test_full_prompt_blocks_are_shared_and_the_partial_block_is_not(make_pool):
    p = make_pool(20)
    prompt = list(range(100, 140))                 # 40 tokens: 2 full blocks + 8 tokens
    a, ca = p.allocate_prefix(prompt)
    b, cb = p.allocate_prefix(prompt)
    assert ca == 0 and cb == 32                    # the second request finds 2 full blocks
    assert a[:2] == b[:2] and a[2] != b[2]          # but writes into its own third block
    assert [p.refcount(x) for x in a] == [2, 2, 1] and p.refcount(b[2]) == 1
    assert p.num_free() == 20 - 4


def test_system_prompt_is_stored_once_for_many_requests(make_pool):
    p = make_pool(64)
    system = list(range(64))                       # 4 full blocks
    tables = [p.allocate_prefix(system + [1000 + r] * (r + 1)) for r in range(10)]
    shared = tables[0][0][:4]
    assert all(t[0][:4] == shared for t in tables)
    assert all(t[1] == 64 for t in tables[1:])
    assert [p.refcount(x) for x in shared] == [10] * 4


def test_freed_cached_blocks_are_reused_until_evicted_in_freeing_order(make_pool):
    p = make_pool(6, order=[0, 1, 2, 3, 4, 5])
    prompt = list(range(32))                       # 2 full blocks
    blocks, _ = p.allocate_prefix(prompt)          # blocks 0, 1
    p.free(blocks)                                 # free queue: 2 3 4 5 0 1
    assert p.free_order() == [2, 3, 4, 5, 0, 1] and p.num_cached() == 2
    again, cached = p.allocate_prefix(prompt)      # matched while free: leaves the queue
    assert again == blocks and cached == 32
    assert p.free_order() == [2, 3, 4, 5]
    p.free(again)                                  # 2 3 4 5 0 1
    taken = p.allocate(5)                          # handed out fresh: 2 3 4 5 0
    assert taken == [2, 3, 4, 5, 0]
    assert p.num_cached() == 1                     # block 0's entry went with it
    p.free(taken)                                  # queue: 1 2 3 4 5 0
    third, cached = p.allocate_prefix(prompt)
    assert cached == 0                             # block 1's parent changed: no match
    assert third == [1, 2] and p.num_cached() == 2  # fresh from the head, registered anew


def test_prompts_diverging_after_one_block_share_one_block(make_pool):
    p = make_pool(10)
    a, _ = p.allocate_prefix(list(range(32)))
    b, cb = p.allocate_prefix(list(range(16)) + list(range(50, 66)))
    assert cb == 16 and b[0] == a[0] and b[1] != a[1]


def test_out_of_blocks_leaves_the_pool_unchanged(make_pool):
    p = make_pool(4)
    p.allocate_prefix(list(range(32)))
    before = (p.free_order(), [p.refcount(i) for i in range(4)], p.num_cached())
    assert p.allocate_prefix(list(range(32)) + list(range(200, 260))) is None
    assert (p.free_order(), [p.refcount(i) for i in range(4)], p.num_cached()) == before


def test_registering_a_block_filled_by_decode(make_pool):
    p = make_pool(8)
    a, _ = p.allocate_prefix(list(range(20)))      # block 1 holds tokens 16..19 so far
    tail = list(range(16, 32))                     # decode filled it
    p.register_block(a[1], a[0], tail)
    b, cb = p.allocate_prefix(list(range(32)) + [7])
    assert cb == 32 and b[:2] == a[:2]
    with pytest.raises(Exception):
        p.register_block(a[1], a[0], tail[:5])


@pytest.mark.parametrize("seed", range(6))
def test_native_pool_matches_the_model_on_random_traces(seed):
    rng = random.Random(seed)
    n = rng.choice([24, 40, 80])
    order = list(range(n))
    rng.shuffle(order)
    nat = _native(n, order)
    mod = _model(n, order)
    templates = [[rng.randrange(50) for _ in range(rng.choice([16, 32, 48, 70]))] for _ in range(4)]
    live = []
    for step in range(250):
        op = rng.random()
        if op < 0.45 or not live:
            t = list(rng.choice(templates))
            t = t[:rng.randrange(len(t) + 1)] + [rng.randrange(50) for _ in range(rng.randrange(40))]
            got, want = nat.allocate_prefix(t), mod.allocate_prefix(t)
            assert got == (None if want is None else (want[0], want[1])), (step, t)
            if got is not None:
                live.append(got[0])
        elif op < 0.75:
            blocks = live.pop(rng.randrange(len(live)))
            nat.free(blocks)
            mod.free(blocks)
        elif op < 0.85:
            k = rng.randrange(4)
            assert nat.allocate(k) == mod.allocate(k)
        else:
            # a write into one block of a live sequence: copy-on-write remaps it
            blocks = rng.choice(live)
            if not blocks:  # an empty prompt holds no block
                continue
            i = rng.randrange(len(blocks))
            bk = blocks[i]
            if nat.refcount(bk) == 1 or nat.num_free() > 0:
                got = nat.cow(bk)
                assert got == mod.cow(bk)
                blocks[i] = got[1]
        assert nat.free_order() == mod.free_order()
        assert [nat.refcount(i) for i in range(n)] == [mod.refcount(i) for i in range(n)]
        assert nat.num_cached() == mod.num_cached()
