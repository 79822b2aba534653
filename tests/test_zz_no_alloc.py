"""The backward entry point that allocates nothing: ulysses_attn_bwd_noalloc.

Some callers of this library cannot allocate device memory. Examples are a
plugin that a host runtime hands only its input and output buffers, a server
that reserves all GPU memory at start-up and must not allocate while it
serves, and a framework whose caching allocator must see every byte. They
cannot provide the workspace that ulysses_attn_bwd takes.
ulysses_attn_bwd_noalloc runs the same backward on a fixed scratch array inside
the library. These tests call it through the C ABI and check it against the
allocating entry point: two calls in a row, because the array keeps the last
call's contents and each call must clear what has to start at zero.

This file is named so that pytest collects it last. A run that stops at the
first failure has then already run every other test.
"""
import ctypes

import pytest
import torch

from tests._gpu import assert_close
from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def _forward(u, sl, hc, hkv, P, seed, offs=None):
    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, seed)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, offs, torch.bfloat16, fused=False)
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    o = L.new_seq_shards(hc)
    L.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
    L._alloc(backward=True)
    b = L.head_buffers
    u.ulysses_seq_to_head(L.h, hc, cu(x["do"]), b["doh"])
    return L, b


def _grads(L, hk_shape):
    P = L.P
    dq = [torch.full_like(t, float("nan")) for t in L.head_buffers["qh"]]
    dk = [torch.full_like(t, float("nan")) for t in L.head_buffers["kh"]]
    dv = [torch.full_like(t, float("nan")) for t in L.head_buffers["vh"]]
    return dq, dk, dv


@pytest.mark.parametrize("sl,hc,hkv,P,offs", [
    (1024, 32, 8, 8, None),                    # Llama-8B heads
    (1000, 8, 2, 4, [0, 333, 334, 1000]),      # ragged tail, packed documents, replicated kv
])
def test_noalloc_matches_the_allocating_entry_point(u, sl, hc, hkv, P, offs):
    L, b = _forward(u, sl, hc, hkv, P, seed=31, offs=offs)
    assert u.ulysses_workspace_size(L.h) <= u.ULYSSES_NOALLOC_SCRATCH_BYTES
    args = (b["qh"], b["kh"], b["vh"], b["oh"], b["doh"], b["lse"])
    ref = _grads(L, None)
    u.ulysses_attn_bwd(L.h, *args, *ref, b["ws"])
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    for call in range(2):
        got = _grads(L, None)
        u.ulysses_attn_bwd_noalloc(L.h, *args, *got)
        torch.cuda.synchronize()
        assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
        for name, gs, rs in zip(("dq", "dk", "dv"), got, ref):
            for r in range(P):
                assert_close(f"{name}[{r}] call {call}", gs[r], rs[r], torch.bfloat16)
        # dK and dV take no atomics: the two entry points agree bit for bit
        for gs, rs in zip(got[1:], ref[1:]):
            for r in range(P):
                assert torch.equal(gs[r], rs[r])


def test_noalloc_call_allocates_no_device_memory(u):
    """A call after set-up leaves the device's free memory and torch's allocator untouched.

    The handle (ulysses_create) sets the scratch array up; the outputs are
    allocated before the measurement. A first call launches every kernel
    once (the driver can size per-kernel resources on a first launch); the
    second is measured.
    """
    sl, hc, hkv, P = 1024, 8, 4, 4
    L, b = _forward(u, sl, hc, hkv, P, seed=32)
    args = (b["qh"], b["kh"], b["vh"], b["oh"], b["doh"], b["lse"])
    first, second = _grads(L, None), _grads(L, None)
    u.ulysses_attn_bwd_noalloc(L.h, *args, *first)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    u.ulysses_attn_bwd_noalloc(L.h, *args, *second)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == alloc0
    for a, c in zip(first, second):
        for r in range(P):
            assert torch.equal(a[r], c[r])


def test_noalloc_rejects_a_layer_beyond_its_scratch(u):
    # The row planes need 8 bytes per (token, query head, batch element):
    # 256 tokens x 2 heads x 65535 batch = 256 MiB > 64 MiB. The size check
    # comes before any pointer is looked at, so no buffers are needed.
    h = u.ulysses_create(256, 65535, 2, 2, 128, 1, True, None, torch.bfloat16)
    assert u.ulysses_workspace_size(h) > u.ULYSSES_NOALLOC_SCRATCH_BYTES
    n0 = u.ulysses_launch_count()
    null = (ctypes.c_void_p * 1)()
    st = u._binding.lib.ulysses_attn_bwd_noalloc(h.ptr, *([ctypes.cast(null, ctypes.POINTER(ctypes.c_void_p))] * 9),
                                                 None)
    assert st == u.ULYSSES_ERR_TOO_LARGE
    assert u.ulysses_launch_count() == n0   # rejected before anything was enqueued
    h.destroy()
