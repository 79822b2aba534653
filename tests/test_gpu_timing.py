"""Per-kernel device timing through the C ABI (ulysses_timing_enable / _read)."""
import pytest
import torch

from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_timing_counts_each_kernel_of_a_layer_step(fused):
    import ulysses_sequence_attention_gb300 as u
    sl, hc, hkv, P = 1024, 8, 4, 4
    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 7)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16, fused=fused)
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    q, k, v, do = cu(x["q"]), cu(x["k"]), cu(x["v"]), cu(x["do"])
    o = L.new_seq_shards(hc)
    dq, dk, dv = L.new_seq_shards(hc), L.new_seq_shards(hkv), L.new_seq_shards(hkv)

    u.ulysses_timing_enable(L.h, True)
    for _ in range(2):
        L.forward(q, k, v, o)
        L.backward(do, dq, dk, dv)
    u.ulysses_timing_enable(L.h, False)
    L.forward(q, k, v, o)              # not timed
    got = {name: u.ulysses_timing_read(L.h, i) for i, name in enumerate(u.KERNEL_NAMES)}
    # per step: one launch of each attention kernel; the explicit path adds
    # seq->head of (q, k, v) and of dO, and head->seq of o and of (dq, dk, dv)
    # (the fused one reads and writes the sequence shards inside the
    # attention kernels)
    assert got["seq_to_head"][1] == (0 if fused else 2 * 2)
    assert got["head_to_seq"][1] == (0 if fused else 2 * 2)
    for name in ("attn_fwd", "bwd_prep", "bwd_dkdv", "bwd_dq"):
        assert got[name][1] == 2, name
    for name, (ms, n) in got.items():
        assert (ms > 0.0) == (n > 0), name
    # enabling again clears the totals
    u.ulysses_timing_enable(L.h, True)
    assert u.ulysses_timing_read(L.h, u.ULYSSES_KERNEL_COUNT - 1) == (0.0, 0)
    with pytest.raises(u.UlyssesError):
        u.ulysses_timing_read(L.h, u.ULYSSES_KERNEL_COUNT)
