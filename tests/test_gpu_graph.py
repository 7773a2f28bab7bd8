"""The captured step (ops.StepGraph): host-to-device staging of the step's
inputs, the cache write and the paged decode, and the device-to-host copy of
the output, as one CUDA graph.

A replay must give the same bits as the same calls made eagerly (same
kernels, same inputs), must read its input buffers afresh on every replay,
and must stay correct over many replays (the decode kernel's merge counters
are left at zero by every launch).  Outputs are also checked against the
fp64 oracle with the parity tolerances."""
import numpy as np
import pytest
import torch

from oracle import core as ocore
from paged_kv_cache_108_gb300 import ops, pool, synth
from tests import harness

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _setup(w):
    """Device state with every context token written; returns the step's
    inputs (new K/V, their slots, q, tables, lengths) beside it."""
    dev = harness.product_step(w)["dev"]
    B = w.block_size
    idx = np.arange(w.num_seqs, dtype=np.int32)
    slots = pool.slot_mapping(w.block_tables, B, harness.new_positions(w), idx)
    step = {
        "k": harness.to_dev_bits(w.k_new, "bf16", "cuda"),
        "v": harness.to_dev_bits(w.v_new, "bf16", "cuda"),
        "slots": torch.from_numpy(slots).cuda(),
    }
    return dev, step


def _oracle(w, dev, q_bits):
    kc = harness.bits_from_dev(dev["k_cache"])
    vc = harness.bits_from_dev(dev["v_cache"])
    return ocore.decode(q_bits, kc, vc, w.block_tables, w.context_lens, w.scale,
                        w.k_scale, w.v_scale)


@requires_gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_captured_step_matches_eager_and_oracle(kv_dtype):
    w = synth.make(f"graph-{kv_dtype}", synth.llama8b_lengths(24), 32, 8, 128, 16,
                   kv_dtype=kv_dtype, seed=61)
    dev, st = _setup(w)
    S, H, d = w.num_seqs, w.num_heads, w.head_dim
    # pinned host staging and the device buffers the graph copies into
    h_q = torch.empty((S, H, d), dtype=torch.bfloat16).pin_memory()
    h_out = torch.empty((S, H, d), dtype=torch.bfloat16).pin_memory()
    d_q = torch.empty((S, H, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(d_q)
    h_q.copy_(dev["q"].cpu())
    g = ops.StepGraph(st["k"], st["v"], st["slots"], out, d_q, dev["k_cache"], dev["v_cache"],
                      dev["bt"], dev["cl"], w.scale, dev["ks"], dev["vs"], dev["ws"],
                      h2d=[(d_q, h_q)], d2h=[(h_out, out)])
    rng = np.random.default_rng(5)
    for it in range(3):
        q_bits = synth.normal_bf16(rng, (S, H, d))
        h_q.copy_(torch.from_numpy(q_bits).view(torch.bfloat16))
        for _ in range(7 if it == 2 else 1):  # several replays in a row
            g.replay()
        torch.cuda.synchronize()
        got = h_out.clone()
        # the same calls made eagerly
        eager = torch.empty_like(out)
        ops.write_and_decode(st["k"], st["v"], st["slots"], eager, d_q, dev["k_cache"],
                             dev["v_cache"], dev["bt"], dev["cl"], w.scale, dev["ks"], dev["vs"],
                             dev["ws"])
        torch.cuda.synchronize()
        assert torch.equal(got, eager.cpu()), f"replay {it} differs from the eager step"
        assert int(dev["ws"][:4].view(torch.int32).item()) == 0
        ref = _oracle(w, dev, q_bits)
        harness.assert_close(got.float().numpy().astype(np.float64), ref, kv_dtype == "fp8")


@requires_gpu
def test_captured_step_rejects_pageable_staging():
    w = synth.make("graph-pageable", [40, 17], 8, 2, 128, 16, seed=67)
    dev, st = _setup(w)
    out = torch.empty_like(dev["q"])
    with pytest.raises(ValueError):
        ops.StepGraph(st["k"], st["v"], st["slots"], out, dev["q"], dev["k_cache"],
                      dev["v_cache"], dev["bt"], dev["cl"], w.scale, workspace=dev["ws"],
                      h2d=[(dev["q"], torch.empty_like(dev["q"], device="cpu"))])


@requires_gpu
def test_captured_step_with_device_slots_matches_host_slots():
    """device_slots=True: the graph derives the new tokens' slots from the
    tables and lengths (pa_step_prepare); caches and outputs must equal the
    eager step fed with host-computed slots, bit for bit."""
    w = synth.make("graph-devslots", synth.llama8b_lengths(20), 32, 8, 128, 16, seed=73)
    dev, st = _setup(w)
    eager_k, eager_v = dev["k_cache"].clone(), dev["v_cache"].clone()
    out_e = torch.empty_like(dev["q"])
    ops.write_and_decode(st["k"], st["v"], st["slots"], out_e, dev["q"], eager_k, eager_v,
                         dev["bt"], dev["cl"], w.scale, workspace=dev["ws"])
    slots = torch.full_like(st["slots"], -7)
    out_g = torch.empty_like(dev["q"])
    h_out = torch.empty(out_g.shape, dtype=torch.bfloat16).pin_memory()
    g = ops.StepGraph(st["k"], st["v"], slots, out_g, dev["q"], dev["k_cache"], dev["v_cache"],
                      dev["bt"], dev["cl"], w.scale, workspace=dev["ws"], d2h=[(h_out, out_g)],
                      device_slots=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(slots, st["slots"])
    assert torch.equal(h_out, out_e.cpu())
    assert np.array_equal(harness.bits_from_dev(dev["k_cache"]), harness.bits_from_dev(eager_k))
    assert np.array_equal(harness.bits_from_dev(dev["v_cache"]), harness.bits_from_dev(eager_v))
