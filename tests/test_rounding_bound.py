"""The derived bound of the dK/dV parity checks, against a plain evaluation of its model (CPU only).

tests/_gpu.py holds dK and dV to max(2e-2, ulp(ref), 6 sigma + ulp(ref)),
with sigma from rounding_sigma: the standard deviation of the error that the
bf16 roundings of the backward's tensor-core operands (P, dS) and of D
(P in the forward's O = P V, and O itself) put into each column sum. This
test evaluates the same formulas in fp64 with exactly those roundings applied
(torch's round-to-nearest-even conversion to bf16) and checks that sigma
describes the errors that result:

* no error exceeds 6 sigma + ulp (the bound does not fail a correct result);
* the median of |error| / sigma lies between 0.2 and 1, where independent
  errors uniform in [-u, u] would put it near 0.67 (sigma is neither a
  vacuous over-estimate nor an under-estimate);
* a packed layer has elements whose error exceeds 2e-2 at |ref| < 4, and all
  of them are inside the derived bound (the reason the bound exists).
"""
import math

import torch

import oracle
from tests._gpu import LAMBDA, rounding_sigma, ulp
from workloads import random_inputs

F = torch.float64


def bf(t):
    return t.to(torch.bfloat16).to(F)


def emulated(x, causal, offs):
    """dK, dV and their exact values, with the bf16 operand roundings applied ([sl, bs, hkv, hs])."""
    q, k, v, do = (x[n].to(F) for n in ("q", "k", "v", "do"))
    sl, bs, hc, hs = q.shape
    hkv = k.shape[2]
    g = hc // hkv
    s = 1.0 / math.sqrt(hs)
    vis = oracle.visible_mask(torch.arange(sl), sl, causal, offs)
    out = {n: torch.zeros(sl, bs, hkv, hs, dtype=F) for n in ("dk", "dv", "dk_exact", "dv_exact")}
    for b in range(bs):
        for kv in range(hkv):
            K, V = k[:, b, kv], v[:, b, kv]
            for h in range(kv * g, (kv + 1) * g):
                Q, dO = q[:, b, h], do[:, b, h]
                Pm = torch.softmax((s * Q @ K.T).masked_fill(~vis, float("-inf")), dim=1)
                dP = dO @ V.T
                D = (dO * (Pm @ V)).sum(1, keepdim=True)
                D_fwd = (dO * bf(bf(Pm) @ V)).sum(1, keepdim=True)   # O from rounded P, then rounded
                out["dk_exact"][:, b, kv] += s * (Pm * (dP - D)).T @ Q
                out["dv_exact"][:, b, kv] += Pm.T @ dO
                out["dk"][:, b, kv] += s * bf(Pm * (dP - D_fwd)).T @ Q
                out["dv"][:, b, kv] += bf(Pm).T @ dO
    return out


def check(x, causal, offs):
    sig = rounding_sigma(x, causal, offs)
    em = emulated(x, causal, offs)
    over = 0
    for n in ("dk", "dv"):
        ref = em[n + "_exact"]
        err = (bf(em[n]) - ref).abs()
        lim = torch.maximum(torch.full_like(ref, 2e-2), ulp(ref, 7))
        lim = torch.maximum(lim, LAMBDA * sig[n] + ulp(ref, 7))
        assert bool((err <= lim).all()), (n, float((err / lim).max()))
        pre = (em[n] - ref).abs()            # before the output's own rounding
        med = float((pre / sig[n]).median())
        assert 0.2 < med < 1.0, (n, med)
        over += int(((err > 2e-2) & (ref.abs() < 4)).sum())
    return over


def test_sigma_describes_the_rounding_errors_of_a_plain_layer():
    x = random_inputs(512, 1, 8, 2, 128, torch.bfloat16, 71)
    check(x, True, None)


def test_derived_bound_covers_the_packed_layer_that_exceeds_2e_2():
    x = random_inputs(2048, 1, 8, 2, 128, torch.bfloat16, 12)
    over = check(x, True, [0, 57, 700, 1500, 2048])
    assert over >= 1
