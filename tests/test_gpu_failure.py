"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait of the tensor-core kernels has a cycle limit. The tests set a short
limit and inject a missing producer signal with the test hook
(ulysses_inject_fault kind 1: no K/V loads are issued in the next forward;
kind 2: no Q/dO loads in the next backward's dK/dV kernel).
The consumers' waits then run out. The kernel sets the status word and
returns, and ulysses_get_status reports ULYSSES_ERR_TIMEOUT. The same handle
and CUDA context then compute a correct result. Nothing faults, traps or hangs.
"""
import math

import pytest
import torch

import oracle
from tests._gpu import assert_close
from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def test_timeout_is_reported_and_the_context_survives(u):
    sl, hc, hkv, P = 128, 2, 1, 1          # one CTA
    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 41, with_grad=False)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16)
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    q, k, v = cu(x["q"]), cu(x["k"]), cu(x["v"])
    o = L.new_seq_shards(hc)
    u.ulysses_set_wait_limit(L.h, 200_000)   # about 0.1 ms per wait
    u.ulysses_inject_fault(L.h, 1)
    L.forward(q, k, v, o)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_ERR_TIMEOUT
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK       # reading clears the word
    # the injection was consumed: the same handle now computes the right answer
    u.ulysses_set_wait_limit(L.h, 4_000_000_000)
    o = L.new_seq_shards(hc)
    L.forward(q, k, v, o)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    O, _ = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=True)
    assert_close("O after recovery", torch.cat([t.cpu() for t in o]), O, torch.bfloat16)


def test_wait_limit_and_fault_kind_are_validated(u):
    h = u.ulysses_create(128, 1, 2, 1, 128, 1, True, None, torch.bfloat16)
    for bad in (0, -5):
        with pytest.raises(u.UlyssesError):
            u.ulysses_set_wait_limit(h, bad)
    with pytest.raises(u.UlyssesError):
        u.ulysses_inject_fault(h, 7)
    h.destroy()


@pytest.mark.parametrize("ds_budget", [None, 0], ids=["stored_ds", "recomputed_dq"])
def test_backward_timeout_is_reported_and_the_context_survives(u, ds_budget):
    """Kind 2: the next backward's dK/dV producer issues no Q/dO loads; its waits run out.

    Both backward paths: with stored dS the dS store thread's wait runs out
    too (the compute warps never stage a tile), and the dQ kernel then reads
    whatever the workspace holds; the status word reports the timeout either
    way, and the next call is right.
    """
    sl, hc, hkv, P = 256, 2, 1, 1          # one CTA pair, two query tiles per query head
    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 42)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16, ds_budget=ds_budget)
    assert L.stores_ds == (ds_budget is None)
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    q, k, v, do = cu(x["q"]), cu(x["k"]), cu(x["v"]), cu(x["do"])
    o = L.new_seq_shards(hc)
    dq, dk, dv = L.new_seq_shards(hc), L.new_seq_shards(hkv), L.new_seq_shards(hkv)
    L.forward(q, k, v, o)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    u.ulysses_set_wait_limit(L.h, 200_000)
    u.ulysses_inject_fault(L.h, 2)
    L.backward(do, dq, dk, dv)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_ERR_TIMEOUT
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    # consumed: the same handle, stream and context now give the right gradients
    u.ulysses_set_wait_limit(L.h, 4_000_000_000)
    L.backward(do, dq, dk, dv)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    qs, ks, vs, dos = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v", "do"))
    g = oracle.ulysses_backward(qs, ks, vs, dos, P, causal=True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(f"{name} after recovery", torch.cat([t.cpu() for t in got]), oracle.unshard_sequence(g[name]),
                     torch.bfloat16)
