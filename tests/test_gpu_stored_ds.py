"""Stored dS (ulysses_set_ds_budget): dQ read back from the dS the dK/dV pass wrote.

The backward's dQ_i = s sum_j dS_ij k_j uses the same dS_ij = P_ij (dO_i . v_j
- D_i) as dK. With a dS budget the dK/dV kernel writes bf16 dS to the
workspace and the dQ kernel is one GEMM per block; without one, the dQ
kernel recomputes S and dP. Each case runs the layer both ways on the same
seeded inputs:
* both against the fp64 oracle, at the bf16 bar;
* dK and dV bit for bit the same (the dK/dV kernel's arithmetic does not
  change, it only also stores dS);
* the workspace grows by exactly the reserved stored-dS area, whose size
  follows from the block count of the tile schedule: per (rank, batch,
  head), one 64 KB block per visible (256-key tile, 128-query tile).
The cases cover a block that one CTA of a pair has and the other lacks (a
document across the pair), a pair whose odd query tile is past the sequence,
non-causal documents, replicated kv heads and more ranks than one launch
holds.
"""
import pytest
import torch

import oracle
from tests._gpu import assert_close, cat_cpu, replica_allowance, rounding_sigma
from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu

BIG = 1 << 40


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def run(L, x, P):
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    hc, hkv = x["q"].shape[2], x["k"].shape[2]
    o = L.new_seq_shards(hc)
    dq, dk, dv = L.new_seq_shards(hc), L.new_seq_shards(hkv), L.new_seq_shards(hkv)
    L.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
    L.backward(cu(x["do"]), dq, dk, dv)
    torch.cuda.synchronize()
    return {"o": cat_cpu(o), "dq": cat_cpu(dq), "dk": cat_cpu(dk), "dv": cat_cpu(dv)}


def blocks_per_head(sl, causal, offs):
    """Stored blocks of one (rank, batch, head): per 256-key tile, the 128-query tiles that see a key of it."""
    offs = offs or [0, sl]

    def doc(t):
        return max(i for i in range(len(offs) - 1) if offs[i] <= t)

    n = 0
    for first in range(0, sl, 256):
        last = min(sl, first + 256) - 1
        lo = first if causal else offs[doc(first)]
        hi = offs[doc(last) + 1] - 1
        n += hi // 128 - lo // 128 + 1
    return n


CASES = [
    # sl, bs, hc, hkv, P, causal, doc offsets, fused, seed
    (1000, 1, 4, 2, 2, True, None, False, 41),                    # ragged tail (explicit path)
    (768, 2, 8, 4, 2, True, [0, 200, 768], True, 42),             # batch 2, a document across a pair
    (1536, 1, 8, 4, 4, False, [0, 700, 1536], True, 43),          # non-causal documents
    (640, 1, 10, 5, 5, True, None, True, 44),                     # odd query tile past the sequence
    (384, 1, 8, 2, 8, True, None, False, 45),                     # replicated kv heads
    (4096, 1, 32, 16, 16, True, [0, 1000, 1001, 4096], False, 46),  # 16 ranks: two launches a pass
    (3072, 1, 32, 8, 8, True, [0, 57, 1100, 1101, 2900, 3072], True, 47),  # packed, shards of 384
]


@pytest.mark.parametrize("sl,bs,hc,hkv,P,causal,offs,fused,seed", CASES)
def test_stored_ds_against_the_oracle_and_the_recomputing_dq(u, sl, bs, hc, hkv, P, causal, offs, fused, seed):
    dt = torch.bfloat16
    x = random_inputs(sl, bs, hc, hkv, 128, dt, seed)
    S = u.UlyssesLayer(sl, bs, hc, hkv, 128, P, causal, offs, dt, fused=fused, ds_budget=BIG)
    R = u.UlyssesLayer(sl, bs, hc, hkv, 128, P, causal, offs, dt, fused=fused, ds_budget=0)
    assert S.stores_ds and not R.stores_ds
    # The sequence needs its own blocks; the largest budget reserves what one
    # document of the capacity (the handle's own length) needs.
    need = 32768 + bs * hc * blocks_per_head(sl, causal, offs) * 65536
    cap = 32768 + bs * hc * blocks_per_head(sl, causal, None) * 65536
    assert u.ulysses_ds_bytes(S.h) == (need, cap)
    assert u.ulysses_ds_bytes(R.h) == (need, 0)
    rows = u.ulysses_workspace_size(R.h)
    assert u.ulysses_workspace_size(S.h) == (rows + 1023) // 1024 * 1024 + cap

    got, ref = run(S, x, P), run(R, x, P)
    assert u.ulysses_get_status(S.h) == u.ULYSSES_OK and u.ulysses_get_status(R.h) == u.ULYSSES_OK
    for n in ("o", "dk", "dv"):
        assert torch.equal(got[n], ref[n]), n

    qs, ks, vs, dos = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v", "do"))
    g = oracle.ulysses_backward(qs, ks, vs, dos, P, causal=causal, doc_offsets=offs)
    sig = rounding_sigma(x, causal, offs)
    for n in ("dq", "dk", "dv"):
        want = oracle.unshard_sequence(g[n])
        extra = replica_allowance(g, n, P, hkv, dt)
        assert_close(f"{n} stored", got[n], want, dt, extra=extra, sigma=sig.get(n))
        assert_close(f"{n} recomputed", ref[n], want, dt, extra=extra, sigma=sig.get(n))


def test_budget_reserves_whole_blocks_and_noalloc(u):
    """The budget reserves whole blocks, up to the capacity's need; the no-alloc entry point recomputes dQ."""
    sl, hc, hkv, P = 1024, 8, 4, 4
    h = u.ulysses_create(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16)
    base = u.ulysses_workspace_size(h)
    rounded = (base + 1023) // 1024 * 1024
    nblk = blocks_per_head(sl, True, None)
    need = 32768 + hc * nblk * 65536
    assert u.ulysses_ds_bytes(h) == (need, 0)
    for budget, blocks in ((need - 1, nblk - 1), (need, nblk), (need + 10 * hc * 65536, nblk),
                           (32768 + hc * 65536 - 1, 0), (0, 0)):
        u.ulysses_set_ds_budget(h, budget)
        reserved = 32768 + hc * blocks * 65536 if blocks else 0
        assert u.ulysses_ds_bytes(h) == (need, reserved), budget
        assert u.ulysses_workspace_size(h) == (rounded + reserved if blocks else base), budget
    h.destroy()

    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 48)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16, fused=False, ds_budget=BIG)
    R = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, None, torch.bfloat16, fused=False, ds_budget=0)
    ref = run(R, x, P)
    cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
    o = L.new_seq_shards(hc)
    L.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
    L._alloc(backward=True)
    b = L.head_buffers
    u.ulysses_seq_to_head(L.h, hc, cu(x["do"]), b["doh"])
    dqh = [torch.empty_like(t) for t in b["qh"]]
    dkh = [torch.empty_like(t) for t in b["kh"]]
    dvh = [torch.empty_like(t) for t in b["vh"]]
    u.ulysses_attn_bwd_noalloc(L.h, b["qh"], b["kh"], b["vh"], b["oh"], b["doh"], b["lse"], dqh, dkh, dvh)
    dq = L.new_seq_shards(hc)
    u.ulysses_head_to_seq(L.h, hc, dqh, dq)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    assert torch.equal(cat_cpu(dq), ref["dq"])     # the recomputing dQ, bit for bit


def test_varying_length_with_a_partial_area(u):
    """An area that holds one 2048-token document: sequences that fit store dS, the others recompute dQ.

    Every set_seq and layer call is enqueued before anything synchronises.
    Each result equals, bit for bit, a fixed handle's on the same path.
    """
    hc, hkv, P, cap = 8, 4, 4, 4096
    budget = 32768 + hc * blocks_per_head(2048, True, None) * 65536
    V = u.UlyssesLayer.variable_length(cap, 1, hc, hkv, 128, P, True, max_docs=4, ds_budget=budget)
    ws0 = u.ulysses_workspace_size(V.h)
    seqs = [(2048, [0, 512, 2048], True), (4096, None, False), (1024, [0, 1, 1024], True),
            (3072, [0, 1024, 2048, 3072], True), (3072, None, False)]   # three 1024 documents fit; 3072 does not
    outs = []
    for i, (sl, offs, fits) in enumerate(seqs):
        x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 60 + i)
        V.set_seq(sl, offs)
        assert V.stores_ds == fits, (sl, offs)
        outs.append((sl, offs, fits, x, run(V, x, P)))
    assert u.ulysses_get_status(V.h) == u.ULYSSES_OK
    assert u.ulysses_workspace_size(V.h) == ws0
    for sl, offs, fits, x, got in outs:
        F = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, offs, torch.bfloat16, ds_budget=BIG if fits else 0)
        assert F.stores_ds == fits
        ref = run(F, x, P)
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(got[n], ref[n]), (sl, n)
    sl, offs, _, x, got = outs[1]                 # the recomputed one, against the oracle
    qs, ks, vs, dos = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v", "do"))
    g = oracle.ulysses_backward(qs, ks, vs, dos, P, causal=True, doc_offsets=offs)
    assert_close("dq recomputed in a partial area", got["dq"], oracle.unshard_sequence(g["dq"]), torch.bfloat16)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("budget", [BIG, 0])
def test_backward_repeats_bit_for_bit(u, fused, budget):
    """Twenty backwards of one packed layer give the same dQ, dK and dV, bit for bit.

    The kernels have no atomics and a fixed order of every sum, so any
    difference between repetitions is a race (a buffer read before it is
    written, or overwritten while still in use). This shape (shards of 384
    tokens, documents of 57 and 1 tokens) is the one on which per-lane
    polling loops made the stored-dS dK/dV kernel vary.
    """
    sl, hc, hkv, P, offs = 3072, 32, 8, 8, [0, 57, 1100, 1101, 2900, 3072]
    x = random_inputs(sl, 1, hc, hkv, 128, torch.bfloat16, 47)
    L = u.UlyssesLayer(sl, 1, hc, hkv, 128, P, True, offs, torch.bfloat16, fused=fused, ds_budget=budget)
    assert L.stores_ds == (budget > 0)
    first = run(L, x, P)
    for rep in range(19):
        again = run(L, x, P)
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(again[n], first[n]), (rep, n)
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK


def test_default_budget_of_a_fixed_layer_is_its_own_need(u):
    L = u.UlyssesLayer(2048, 1, 8, 4, 128, 4, True, [0, 700, 2048], torch.bfloat16)
    need, reserved = u.ulysses_ds_bytes(L.h)
    assert L.stores_ds and need == reserved == 32768 + 8 * blocks_per_head(2048, True, [0, 700, 2048]) * 65536
