"""pa_step_prepare: block-table updates, context-length advance and slot
mapping on the device.  Slots must equal the oracle's slot formula bit for
bit; tables and lengths must equal the host bookkeeping model after every
step of a multi-step decode loop."""
import numpy as np
import pytest
import torch

from oracle import pool_model
from paged_kv_cache_108_gb300 import ops, pool

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _expected(tables, lens, B):
    out = np.full(len(lens), -1, dtype=np.int32)
    for i, n in enumerate(lens):
        if n <= 0 or (n - 1) // B >= tables.shape[1] or tables[i, (n - 1) // B] < 0:
            continue
        out[i] = pool_model.slot_of(tables[i], int(n) - 1, B)
    return out


@requires_gpu
@pytest.mark.parametrize("B", [1, 16, 64])
def test_slots_updates_and_advance_match_the_model(B):
    rng = np.random.default_rng(71 + B)
    S, mb = 57, 40
    tables = rng.integers(0, 5000, size=(S, mb)).astype(np.int32)
    tables[3, :] = -1                                  # no blocks at all
    lens = rng.integers(0, mb * B, size=S).astype(np.int32)
    lens[0], lens[1], lens[2] = 0, mb * B, 1           # empty, table full, first token
    # updates: a few entries per sequence, some out of range (skipped)
    ups = []
    for i in rng.choice(S, size=20, replace=False):
        ups.append((int(i), int(rng.integers(0, mb)), int(rng.integers(0, 5000))))
    ups.append((5, mb + 3, 7))   # logical block past the table: skipped
    ups.append((6, -1, 7))       # negative logical block: skipped
    up = np.array(ups, dtype=np.int32)
    for advance in (0, 1, 3):
        t_dev = torch.from_numpy(tables).cuda()
        l_dev = torch.from_numpy(lens).cuda()
        slots = torch.empty(S, dtype=torch.int32, device="cuda")
        ops.step_prepare(t_dev, l_dev, B, slots, torch.from_numpy(up).cuda(), advance)
        torch.cuda.synchronize()
        t_ref = tables.copy()
        for s_, idx, blk in ups:
            if 0 <= idx < mb:
                t_ref[s_, idx] = blk
        l_ref = lens + advance
        assert np.array_equal(t_dev.cpu().numpy(), t_ref)
        assert np.array_equal(l_dev.cpu().numpy(), l_ref)
        assert np.array_equal(slots.cpu().numpy(), _expected(t_ref, l_ref, B))


@requires_gpu
def test_device_slots_equal_host_slot_mapping():
    rng = np.random.default_rng(83)
    S, mb, B = 64, 210, 16
    tables = rng.permutation(S * mb).astype(np.int32).reshape(S, mb)
    lens = rng.integers(1, mb * B, size=S).astype(np.int32)
    host = pool.slot_mapping(tables, B, lens - 1)
    slots = torch.empty(S, dtype=torch.int32, device="cuda")
    ops.step_prepare(torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), B, slots)
    torch.cuda.synchronize()
    assert np.array_equal(slots.cpu().numpy(), host)


@requires_gpu
def test_decode_loop_keeps_device_metadata_in_step_with_the_pool():
    """Ten decode steps: each step the host pool gives a new block to every
    sequence whose next token opens one; the device applies the updates,
    advances the lengths by one and maps the slots."""
    B, S, mb, steps = 16, 12, 16, 10
    model = pool_model.BlockPoolModel(400)
    rng = np.random.default_rng(91)
    lens = rng.integers(1, 8 * B, size=S).astype(np.int32)
    tables = np.full((S, mb), -1, dtype=np.int32)
    for i in range(S):
        blocks = model.allocate(-(-int(lens[i]) // B))
        tables[i, :len(blocks)] = blocks
    t_dev = torch.from_numpy(tables).cuda()
    l_dev = torch.from_numpy(lens).cuda()
    slots = torch.empty(S, dtype=torch.int32, device="cuda")
    for _ in range(steps):
        ups = []
        for i in range(S):
            n_next = int(lens[i]) + 1
            if (n_next - 1) % B == 0:  # the new token opens a block
                blk = model.allocate(1)[0]
                ups.append((i, (n_next - 1) // B, blk))
                tables[i, (n_next - 1) // B] = blk
        lens = lens + 1
        up = torch.tensor(ups, dtype=torch.int32, device="cuda").reshape(-1, 3)
        ops.step_prepare(t_dev, l_dev, B, slots, up, advance=1)
        torch.cuda.synchronize()
        assert np.array_equal(t_dev.cpu().numpy(), tables)
        assert np.array_equal(l_dev.cpu().numpy(), lens)
        assert np.array_equal(slots.cpu().numpy(), _expected(tables, lens, B))
