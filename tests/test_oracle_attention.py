"""Pins of the oracle's attention forward (CPU only).

* Library special case: torch SDPA in fp64 on the CPU, causal, with K and V
  repeated for GQA the way HF ``repeat_kv`` does, and an explicit
  block-diagonal mask for packed documents.
* Closed forms: a zero query gives the mean of the visible values; row 0 sees
  only key 0; a constant V gives a constant output; with a zero query the
  logsumexp is log of the number of visible keys.
* Invariant from the DeepSpeed-Ulysses blog (section "收敛性研究"): sequence
  parallelism leaves the result unchanged, for every P that divides the heads.
* Documents are isolated when position ids reset at each document start
  (ALST guide, section 2.2).
"""
import math

import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import random_inputs

F64 = torch.float64


def sdpa_reference(q, k, v, causal=True, mask=None):
    """torch SDPA on [sl, bs, H, hs] tensors, GQA by repeat_interleave."""
    hc, hkv = q.shape[2], k.shape[2]
    g = hc // hkv
    qq = q.to(F64).permute(1, 2, 0, 3)
    kk = k.to(F64).repeat_interleave(g, dim=2).permute(1, 2, 0, 3)
    vv = v.to(F64).repeat_interleave(g, dim=2).permute(1, 2, 0, 3)
    o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, is_causal=causal and mask is None)
    return o.permute(2, 0, 1, 3)


def block_causal_mask(lengths):
    """Block-diagonal lower-triangular mask built from document lengths."""
    blocks = [torch.tril(torch.ones(n, n, dtype=torch.bool)) for n in lengths]
    return torch.block_diag(*blocks)


@pytest.mark.parametrize("hc,hkv,causal", [(4, 4, True), (8, 2, True), (4, 1, True), (4, 2, False)])
def test_forward_matches_sdpa(hc, hkv, causal):
    x = random_inputs(48, 2, hc, hkv, 16, torch.float32, seed=11, with_grad=False)
    O, _ = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=causal)
    ref = sdpa_reference(x["q"], x["k"], x["v"], causal=causal)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)


def test_packed_documents_match_sdpa_block_mask():
    lengths = [5, 17, 9, 1, 16]
    offs = [0]
    for n in lengths:
        offs.append(offs[-1] + n)
    sl = offs[-1]
    x = random_inputs(sl, 1, 4, 2, 8, torch.float32, seed=12, with_grad=False)
    O, _ = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=True, doc_offsets=offs)
    ref = sdpa_reference(x["q"], x["k"], x["v"], mask=block_causal_mask(lengths))
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)


def test_bf16_inputs_widen_exactly():
    x = random_inputs(32, 1, 2, 2, 8, torch.bfloat16, seed=13, with_grad=False)
    O, _ = oracle.unsharded_forward(x["q"], x["k"], x["v"])
    ref = sdpa_reference(x["q"], x["k"], x["v"])
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)


def test_zero_query_gives_prefix_mean_and_log_count():
    sl, hs = 20, 6
    x = random_inputs(sl, 1, 2, 1, hs, torch.float32, seed=14, with_grad=False)
    q = torch.zeros_like(x["q"])
    O, L = oracle.unsharded_forward(q, x["k"], x["v"], causal=True)
    v = x["v"].to(F64)[:, 0, 0]
    prefix_mean = torch.cumsum(v, 0) / torch.arange(1, sl + 1, dtype=F64)[:, None]
    for h in range(2):
        assert torch.allclose(O[:, 0, h], prefix_mean, atol=1e-13)
        assert torch.allclose(L[0, h], torch.log(torch.arange(1, sl + 1, dtype=F64)), atol=1e-13)
    # non-causal: the mean of all values
    O2, _ = oracle.unsharded_forward(q, x["k"], x["v"], causal=False)
    assert torch.allclose(O2[:, 0, 0], v.mean(0).expand(sl, hs), atol=1e-13)


def test_first_row_sees_only_first_key():
    x = random_inputs(16, 1, 2, 2, 8, torch.float32, seed=15, with_grad=False)
    O, L = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=True)
    for h in range(2):
        assert torch.equal(O[0, 0, h], x["v"][0, 0, h].to(F64))
        s00 = (x["q"][0, 0, h].to(F64) @ x["k"][0, 0, h].to(F64)) / math.sqrt(8)
        assert abs(float(L[0, h, 0] - s00)) < 1e-13


def test_constant_values_give_constant_output():
    x = random_inputs(24, 1, 4, 2, 8, torch.float32, seed=16, with_grad=False)
    v = torch.full_like(x["v"], 0.75)
    O, _ = oracle.unsharded_forward(x["q"], x["k"], v, causal=True, doc_offsets=[0, 7, 24])
    assert torch.allclose(O, torch.full_like(O, 0.75), atol=1e-14)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_ulysses_equals_unsharded(P):
    hc, hkv, sl = 8, 2, 32   # P=4 and P=8 replicate the 2 kv heads
    x = random_inputs(sl, 2, hc, hkv, 8, torch.float32, seed=17, with_grad=False)
    offs = [0, 9, 20, 32]
    res = oracle.ulysses_forward(oracle.shard_sequence(x["q"], P), oracle.shard_sequence(x["k"], P),
                                 oracle.shard_sequence(x["v"], P), P, causal=True, doc_offsets=offs)
    O, L = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=True, doc_offsets=offs)
    assert torch.allclose(oracle.unshard_sequence(res["o"]), O, atol=1e-13, rtol=0)
    Hq = hc // P
    for r in range(P):
        assert torch.allclose(res["lse"][r], L[:, r * Hq:(r + 1) * Hq], atol=1e-13)


def test_documents_are_isolated():
    offs = [0, 10, 23, 40]
    x = random_inputs(40, 1, 4, 2, 8, torch.float32, seed=18, with_grad=False)
    O, _ = oracle.unsharded_forward(x["q"], x["k"], x["v"], causal=True, doc_offsets=offs)
    k2, v2 = x["k"].clone(), x["v"].clone()
    k2[10:23] += 3.0
    v2[10:23] -= 2.0
    O2, _ = oracle.unsharded_forward(x["q"], k2, v2, causal=True, doc_offsets=offs)
    assert torch.equal(O[:10], O2[:10])
    assert torch.equal(O[23:], O2[23:])
    assert not torch.allclose(O[10:23], O2[10:23])


def test_row_sampling_matches_whole_head():
    x = random_inputs(64, 1, 1, 1, 8, torch.float32, seed=19, with_grad=True)
    q, k, v, do = (x[n][:, 0, 0].to(F64) for n in ("q", "k", "v", "do"))
    s = 1 / math.sqrt(8)
    offs = [0, 30, 64]
    O, L = oracle.attention_head_forward(q, k, v, s, True, offs)
    dQ, dK, dV = oracle.attention_head_backward(q, k, v, do, s, True, offs)
    rows = torch.tensor([0, 5, 29, 30, 63])
    o_r, l_r, dq_r = oracle.attention_head_dq_rows(q, k, v, do, s, True, offs, rows)
    assert torch.allclose(o_r, O[rows], atol=1e-14)
    assert torch.allclose(l_r, L[rows], atol=1e-14)
    assert torch.allclose(dq_r, dQ[rows], atol=1e-13)
    cols = torch.tensor([0, 7, 31, 62, 63])
    dk_c, dv_c = oracle.attention_head_dkdv_cols(q, k, v, do, s, True, offs, cols, row_chunk=7)
    assert torch.allclose(dk_c, dK[cols], atol=1e-13)
    assert torch.allclose(dv_c, dV[cols], atol=1e-13)
