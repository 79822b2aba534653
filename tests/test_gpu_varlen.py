"""Sequences of varying length on one handle (ulysses_create_varlen / ulysses_set_seq).

The pages' default mode re-derives shapes for every batch
(`seq_length_is_variable=True`, ALST guide section 2.1 item (5)). One handle
with a capacity of 4096 tokens takes several sequences in turn: different
lengths, packed and unpacked, one the fused kernels cannot take (shards of
250 tokens) and one empty. Every set_seq and every layer call is enqueued on
the stream before anything synchronises, so the new schedules must reach the
device in stream order. Each result must equal, bit for bit, what a fixed
handle made for that sequence computes; two are also checked against the
oracle.
"""
import pytest
import torch

import oracle
from tests._gpu import assert_close, rounding_sigma
from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu

HC, HKV, P, CAP = 8, 4, 4, 4096
SEQS = [
    (1024, None),
    (4096, [0, 1000, 1001, 4096]),
    (1000, None),                       # shards of 250 tokens: the explicit path
    (0, None),                          # empty: every call is a no-op
    (2048, [0, 512, 2048]),
    (3072, None),
]


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def run(L, x, sl):
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    o = L.new_seq_shards(HC)
    dq, dk, dv = L.new_seq_shards(HC), L.new_seq_shards(HKV), L.new_seq_shards(HKV)
    L.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
    L.backward(cu(x["do"]), dq, dk, dv)
    return {"o": o, "dq": dq, "dk": dk, "dv": dv, "lse": [t.clone() for t in L.lse]}


def test_one_handle_takes_sequences_of_varying_length(u):
    V = u.UlyssesLayer.variable_length(CAP, 1, HC, HKV, 128, P, True, max_docs=4)
    ws0 = u.ulysses_workspace_size(V.h)
    got = []
    for i, (sl, offs) in enumerate(SEQS):
        x = random_inputs(sl, 1, HC, HKV, 128, torch.bfloat16, 300 + i)
        V.set_seq(sl, offs)
        got.append((sl, offs, x, run(V, x, sl)))
    torch.cuda.synchronize()
    assert u.ulysses_get_status(V.h) == u.ULYSSES_OK
    assert u.ulysses_workspace_size(V.h) == ws0          # sized for the capacity, once

    for sl, offs, x, res in got:
        if sl == 0:
            continue
        F = u.UlyssesLayer(sl, 1, HC, HKV, 128, P, True, offs, torch.bfloat16)
        ref = run(F, x, sl)
        torch.cuda.synchronize()
        for name in ("o", "dq", "dk", "dv", "lse"):
            for r in range(P):
                assert torch.equal(res[name][r], ref[name][r]), (sl, name, r)

    for sl, offs, x, res in (got[0], got[4]):
        qs, ks, vs, dos = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v", "do"))
        f = oracle.ulysses_forward(qs, ks, vs, P, causal=True, doc_offsets=offs)
        g = oracle.ulysses_backward(qs, ks, vs, dos, P, causal=True, doc_offsets=offs)
        sig = rounding_sigma(x, True, offs)
        for name, want in (("o", f["o"]), ("dq", g["dq"]), ("dk", g["dk"]), ("dv", g["dv"])):
            gpu = torch.cat([t.cpu() for t in res[name]])
            assert_close(f"{name} sl={sl}", gpu, oracle.unshard_sequence(want), torch.bfloat16, sigma=sig.get(name))


def test_set_seq_checks_each_sequence(u):
    h = u.ulysses_create_varlen(CAP, 1, HC, HKV, 128, P, True, 2, torch.bfloat16)
    cases = [
        (CAP + 4, None, u.ULYSSES_ERR_TOO_LARGE),
        (1026, None, u.ULYSSES_ERR_DIVISIBILITY),        # sl % P != 0
        (1024, [0, 10, 20, 1024], u.ULYSSES_ERR_INVALID_ARG),   # 3 documents > max_docs = 2
        (1024, [0, 600, 1000], u.ULYSSES_ERR_INVALID_ARG),      # offsets do not end at sl
        (1024, [0, 600, 600, 1024], u.ULYSSES_ERR_INVALID_ARG),
    ]
    for sl, offs, want in cases:
        with pytest.raises(u.UlyssesError) as e:
            u.ulysses_set_seq(h, sl, offs)
        assert e.value.status == want, (sl, offs)
    assert h.sl == 0                                       # a failed check changes nothing
    u.ulysses_set_seq(h, 1024, [0, 600, 1024])
    assert h.sl == 1024
    h.destroy()


def test_a_fixed_handle_takes_shorter_sequences_too(u):
    """ulysses_create's capacity is its own length: set_seq may shorten it."""
    x = random_inputs(512, 1, HC, HKV, 128, torch.bfloat16, 77)
    F = u.UlyssesLayer(2048, 1, HC, HKV, 128, P, True, None, torch.bfloat16)
    F.set_seq(512)
    a = run(F, x, 512)
    G = u.UlyssesLayer(512, 1, HC, HKV, 128, P, True, None, torch.bfloat16)
    b = run(G, x, 512)
    torch.cuda.synchronize()
    for name in ("o", "dq", "dk", "dv"):
        for r in range(P):
            assert torch.equal(a[name][r], b[name][r]), name
    with pytest.raises(u.UlyssesError) as e:
        F.set_seq(4096)
    assert e.value.status == u.ULYSSES_ERR_TOO_LARGE
