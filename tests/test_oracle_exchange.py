"""Pins of the oracle's exchanges against what the pages fix (CPU only).

* The 2-GPU layout diagram of the Transformers DeepSpeed-Ulysses guide
  (section "Ulysses 序列并行的核心原理"), checked element by element on an
  index-encoded tensor.
* The second all-to-all reverses the first (HF blog "Ulysses Sequence
  Parallelism: Training with Million-Token Contexts", algorithm step 5), so a
  round trip is the identity, bit for bit.
* Message sizes of 3Nh and Nh (DeepSpeed-Ulysses blog, section "显著的通信量减少").
"""
import json
import os

import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def encoded(sl, bs, H, hs):
    """Every element holds its own (t, b, h, d) index as one integer."""
    t = torch.arange(sl).view(sl, 1, 1, 1)
    b = torch.arange(bs).view(1, bs, 1, 1)
    h = torch.arange(H).view(1, 1, H, 1)
    d = torch.arange(hs).view(1, 1, 1, hs)
    return ((t * 1000 + b) * 1000 + h) * 1000 + d


def decode(v):
    d = v % 1000
    h = (v // 1000) % 1000
    b = (v // 1000000) % 1000
    t = v // 1000000000
    return t, b, h, d


def test_layout_matches_2gpu_diagram():
    g = json.load(open(os.path.join(GOLDEN, "layout_2gpu_diagram.json")))
    N, H, P, hs, bs = g["N"], g["H"], g["P"], 3, 2
    x = encoded(N, bs, H, hs)
    seq = oracle.shard_sequence(x, P)
    for ent in g["seq_sharded"]:
        t, b, h, d = decode(seq[ent["gpu"]])
        assert sorted(set(t.flatten().tolist())) == list(range(*ent["tokens"]))
        assert sorted(set(h.flatten().tolist())) == list(range(*ent["heads"]))
    head = oracle.seq_to_head(seq, P)
    for ent in g["head_sharded"]:
        shard = head[ent["gpu"]]
        t, b, h, d = decode(shard)
        toks = list(range(*ent["tokens"]))
        heads = list(range(*ent["heads"]))
        assert shard.shape == (len(toks), bs, len(heads), hs)
        # element [t, b, j, d] holds token t, batch b, the j-th head of the block, feature d
        assert torch.equal(t, torch.tensor(toks).view(-1, 1, 1, 1).expand_as(t))
        assert torch.equal(h, torch.tensor(heads).view(1, 1, -1, 1).expand_as(h))
        assert torch.equal(b, torch.arange(bs).view(1, -1, 1, 1).expand_as(b))
        assert torch.equal(d, torch.arange(hs).view(1, 1, 1, -1).expand_as(d))


@pytest.mark.parametrize("H,P", [(8, 1), (8, 2), (8, 4), (8, 8), (6, 3), (4, 2)])
def test_round_trip_is_identity(H, P):
    x = encoded(24, 2, H, 5)
    seq = oracle.shard_sequence(x, P)
    back = oracle.head_to_seq(oracle.seq_to_head(seq, P), P, H)
    for a, b in zip(seq, back):
        assert torch.equal(a, b)


def test_p1_exchange_is_identity():
    x = encoded(16, 1, 4, 3)
    (h,) = oracle.seq_to_head(oracle.shard_sequence(x, 1), 1)
    assert torch.equal(h, x)


def test_every_element_lands_exactly_once():
    H, P, sl = 8, 4, 32
    x = encoded(sl, 2, H, 3)
    head = oracle.seq_to_head(oracle.shard_sequence(x, P), P)
    allv = torch.cat([s.flatten() for s in head])
    assert torch.equal(torch.sort(allv).values, torch.sort(x.flatten()).values)


def test_replicated_kv_heads():
    # P > hkv: rank r holds kv head r*hkv//P, all tokens.
    hkv, P, sl = 2, 4, 8
    x = encoded(sl, 1, hkv, 2)
    head = oracle.seq_to_head(oracle.shard_sequence(x, P), P)
    for r in range(P):
        t, b, h, d = decode(head[r])
        assert head[r].shape == (sl, 1, 1, 2)
        assert set(h.flatten().tolist()) == {r * hkv // P}
        assert t[:, 0, 0, 0].tolist() == list(range(sl))
    # gradients of a replicated head add up over its replicas
    ones = [torch.ones(sl, 1, 1, 2) for _ in range(P)]
    g = oracle.head_to_seq(ones, P, hkv, sum_replicas=True)
    for s in g:
        assert torch.all(s == P // hkv)


@pytest.mark.parametrize("sl,bs,H,hs,P,elem", [(24, 2, 8, 3, 4, 2), (12, 3, 6, 5, 3, 4), (16, 1, 4, 7, 1, 2)])
def test_exchange_bytes_counts_what_the_exchange_moves(sl, bs, H, hs, P, elem):
    """exchange_bytes against the oracle's own exchange, block by block.

    An index-encoded tensor tells where every element of every head shard
    came from. The blocks (source rank s -> destination rank r) add up to the
    whole tensor once: exchange_bytes. The DeepSpeed-Ulysses blog (section
    "显著的通信量减少") puts M/P on each GPU's links for an aggregate message
    M: each of the P^2 blocks holds M/P^2, and each rank sends the (P-1)/P of
    its M/P that it does not keep. Sizes are all different, so a dropped or
    repeated factor (batch, head size, element size) fails.
    """
    x = encoded(sl, bs, H, hs)
    n = sl // P
    head = oracle.seq_to_head(oracle.shard_sequence(x, P), P)
    block = torch.zeros(P, P, dtype=torch.int64)      # [source, destination] elements
    for r, shard in enumerate(head):
        t, _, _, _ = decode(shard)
        src = (t // n).flatten()
        block[:, r] += torch.bincount(src, minlength=P)
    M = oracle.exchange_bytes(sl, bs, H, hs, elem)
    assert int(block.sum()) * elem == M
    assert torch.all(block * elem * P * P == M)
    sent = (block.sum(1) - block.diagonal()) * elem     # bytes each rank sends away
    assert torch.all(sent * P * P == M * (P - 1))


def test_message_sizes_3nh_plus_nh():
    """Q, K and V exchange 3Nh elements and the output Nh (hc == hkv, h = hc*hs), per batch element."""
    sl, bs, hc, hs, P = 64, 2, 8, 16, 4
    N, h = sl, hc * hs
    x = encoded(sl, bs, hc, hs)
    moved = sum(s.numel() for s in oracle.seq_to_head(oracle.shard_sequence(x, P), P))
    assert 3 * moved == 3 * N * h * bs
    assert 3 * oracle.exchange_bytes(sl, bs, hc, hs, 1) + oracle.exchange_bytes(sl, bs, hc, hs, 1) == 4 * N * h * bs
