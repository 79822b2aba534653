"""Pins of the oracle's backward (CPU only).

* Central finite differences in fp64 of L = sum(O * dO) through the whole
  Ulysses layer (exchanges included), w.r.t. every element of Q, K and V.
* Library special case: torch autograd through SDPA in fp64.
* Closed forms: a constant V makes O independent of Q and K, so dQ = dK = 0.
  A zero query gives uniform causal weights, so dV_j = sum_{i >= j} dO_i / (i + 1).
* Invariant: the softmax rows sum to one, so the sum of dK over all key
  positions of a head is zero.
"""
import math

import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import random_inputs

F64 = torch.float64


def layer_loss(q, k, v, do, P, offs):
    res = oracle.ulysses_forward(oracle.shard_sequence(q, P), oracle.shard_sequence(k, P),
                                 oracle.shard_sequence(v, P), P, causal=True, doc_offsets=offs)
    return float((oracle.unshard_sequence(res["o"]) * do).sum())


@pytest.mark.parametrize("P,offs", [(1, None), (2, None), (2, [0, 5, 16]), (4, None)])
def test_finite_differences_through_layer(P, offs):
    sl, bs, hc, hkv, hs = 16, 1, 4, 2, 4     # P=4 replicates the kv heads
    x = random_inputs(sl, bs, hc, hkv, hs, torch.float64, seed=21)
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    g = oracle.ulysses_backward(oracle.shard_sequence(q, P), oracle.shard_sequence(k, P),
                                oracle.shard_sequence(v, P), oracle.shard_sequence(do, P),
                                P, causal=True, doc_offsets=offs)
    grads = {"q": oracle.unshard_sequence(g["dq"]), "k": oracle.unshard_sequence(g["dk"]),
             "v": oracle.unshard_sequence(g["dv"])}
    eps = 1e-6
    for name in ("q", "k", "v"):
        base = {"q": q, "k": k, "v": v}
        fd = torch.zeros_like(base[name])
        flat = fd.view(-1)
        for idx in range(flat.numel()):
            plus = {n: t.clone() for n, t in base.items()}
            minus = {n: t.clone() for n, t in base.items()}
            plus[name].view(-1)[idx] += eps
            minus[name].view(-1)[idx] -= eps
            lp = layer_loss(plus["q"], plus["k"], plus["v"], do, P, offs)
            lm = layer_loss(minus["q"], minus["k"], minus["v"], do, P, offs)
            flat[idx] = (lp - lm) / (2 * eps)
        err = (fd - grads[name]).abs().max() / grads[name].abs().max()
        assert err < 1e-6, (name, float(err))


@pytest.mark.parametrize("hc,hkv", [(4, 4), (8, 2)])
def test_backward_matches_sdpa_autograd(hc, hkv):
    x = random_inputs(40, 2, hc, hkv, 8, torch.float32, seed=22)
    q = x["q"].to(F64).requires_grad_()
    k = x["k"].to(F64).requires_grad_()
    v = x["v"].to(F64).requires_grad_()
    g = hc // hkv
    o = F.scaled_dot_product_attention(
        q.permute(1, 2, 0, 3), k.repeat_interleave(g, 2).permute(1, 2, 0, 3),
        v.repeat_interleave(g, 2).permute(1, 2, 0, 3), is_causal=True).permute(2, 0, 1, 3)
    (o * x["do"].to(F64)).sum().backward()
    dq, dk, dv = oracle.unsharded_backward(x["q"], x["k"], x["v"], x["do"], causal=True)
    assert torch.allclose(dq, q.grad, atol=1e-12)
    assert torch.allclose(dk, k.grad, atol=1e-12)
    assert torch.allclose(dv, v.grad, atol=1e-12)


def test_constant_values_zero_query_key_gradients():
    x = random_inputs(24, 1, 4, 2, 8, torch.float32, seed=23)
    v = torch.full_like(x["v"], -1.25)
    dq, dk, dv = oracle.unsharded_backward(x["q"], x["k"], v, x["do"], causal=True,
                                           doc_offsets=[0, 11, 24])
    assert dq.abs().max() < 1e-13
    assert dk.abs().max() < 1e-13
    assert dv.abs().max() > 0.1


def test_zero_query_value_gradient_closed_form():
    sl, hs = 18, 5
    x = random_inputs(sl, 1, 1, 1, hs, torch.float32, seed=24)
    q = torch.zeros_like(x["q"])
    _, _, dv = oracle.unsharded_backward(q, x["k"], x["v"], x["do"], causal=True)
    do = x["do"].to(F64)[:, 0, 0]
    w = do / torch.arange(1, sl + 1, dtype=F64)[:, None]
    expect = torch.flip(torch.cumsum(torch.flip(w, [0]), 0), [0])   # sum over i >= j
    assert torch.allclose(dv[:, 0, 0], expect, atol=1e-13)


def test_key_gradient_sums_to_zero_per_head():
    x = random_inputs(32, 2, 4, 1, 8, torch.float32, seed=25)
    _, dk, _ = oracle.unsharded_backward(x["q"], x["k"], x["v"], x["do"], causal=True,
                                         doc_offsets=[0, 13, 32])
    assert dk.sum(dim=0).abs().max() < 1e-12
