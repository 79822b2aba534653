"""GPU parity at the workloads' full sizes, on sampled outputs.

Each test runs the whole layer through the C-ABI on the seeded workload input,
in the launch configuration that bench.py times. It then checks a seeded
sample of outputs that the oracle can compute one by one:

* O, LSE and dQ at sampled query rows. Each depends on its row alone: the
  oracle's own O_i gives D_i.
* dK and dV at sampled key rows. They need every query that sees the key, and
  the oracle sums over those queries in row chunks.

Tolerances as in the other parity tests: |x - ref| <= max(2e-2, one bf16 ulp
of the reference) per element, and mean-abs 2e-3. The stored-dS workloads
(32K, packed 64K) also repeat their backward and require identical bits.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._gpu import TOL, assert_close
from workloads import WORKLOADS, doc_offsets_for, make_global_inputs, split_shards

pytestmark = pytest.mark.gpu
F64 = torch.float64


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def run_workload(u, w, x, repeats=0, stores_ds=None):
    """The layer on the workload input as bench.py runs it (default dS budget).

    ``repeats``: that many more backwards on the same inputs, each compared
    bit for bit with the first on the GPU (the kernels have no atomics and a
    fixed order of every sum, so a difference is a race). ``stores_ds``:
    the dQ path the default budget must pick.
    """
    offs = doc_offsets_for(w)
    L = u.UlyssesLayer(w.sl, w.bs, w.hc, w.hkv, w.hs, w.P, w.causal, offs, w.torch_dtype)
    if stores_ds is not None:
        assert L.stores_ds == stores_ds
    cu = lambda t: [s.cuda() for s in split_shards(t, w.P)]  # noqa: E731
    o = L.new_seq_shards(w.hc)
    L.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
    out = {"o": torch.cat([t.cpu() for t in o]), "lse": [t.cpu() for t in L.lse]}
    if w.backward:
        do = cu(x["do"])
        dq, dk, dv = L.new_seq_shards(w.hc), L.new_seq_shards(w.hkv), L.new_seq_shards(w.hkv)
        L.backward(do, dq, dk, dv)
        for rep in range(repeats):
            dq2, dk2, dv2 = L.new_seq_shards(w.hc), L.new_seq_shards(w.hkv), L.new_seq_shards(w.hkv)
            L.backward(do, dq2, dk2, dv2)
            for name, a, b in (("dq", dq, dq2), ("dk", dk, dk2), ("dv", dv, dv2)):
                assert all(torch.equal(s, t) for s, t in zip(a, b)), (rep, name)
            del dq2, dk2, dv2
        out.update(dq=torch.cat([t.cpu() for t in dq]), dk=torch.cat([t.cpu() for t in dk]),
                   dv=torch.cat([t.cpu() for t in dv]))
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    del L
    torch.cuda.empty_cache()
    return out


def check_rows(w, x, got, heads, rows_per_head, seed):
    """O, LSE (and dQ) at sampled (head, row) pairs against the oracle."""
    rng = np.random.default_rng(seed)
    offs = doc_offsets_for(w)
    s = 1.0 / math.sqrt(w.hs)
    g = w.hc // w.hkv
    Hq = w.hc // w.P
    errs = {"o": [], "dq": []}
    refs = {"o": [], "dq": []}
    lse_err = 0.0
    for h in heads:
        rows = torch.tensor(np.sort(rng.choice(w.sl, rows_per_head, replace=False)))
        rows = torch.unique(torch.cat([rows, torch.tensor([0, w.sl - 1])]))
        kv = h // g
        q = x["q"][:, 0, h].to(F64)
        k = x["k"][:, 0, kv].to(F64)
        v = x["v"][:, 0, kv].to(F64)
        do = x["do"][:, 0, h].to(F64) if w.backward else torch.zeros_like(q)
        O, LSE, dQ = oracle.attention_head_dq_rows(q, k, v, do, s, w.causal, offs, rows)
        errs["o"].append(got["o"][rows, 0, h])
        refs["o"].append(O)
        r, j = h // Hq, h % Hq
        lse_err = max(lse_err, float((got["lse"][r][0, j, rows].to(F64) - LSE).abs().max()))
        if w.backward:
            errs["dq"].append(got["dq"][rows, 0, h])
            refs["dq"].append(dQ)
    assert_close("O rows", torch.cat(errs["o"]), torch.cat(refs["o"]), w.torch_dtype)
    assert lse_err <= 1e-3, f"LSE max-abs {lse_err}"
    if w.backward:
        assert_close("dQ rows", torch.cat(errs["dq"]), torch.cat(refs["dq"]), w.torch_dtype)


def check_cols(w, x, got, kv_heads, cols, row_chunk=2048, uniform=True):
    """dK and dV at sampled key rows of some kv heads (sums over the GQA group).

    ``uniform``: the keys are a uniform sample, so the mean-abs bound applies.
    """
    offs = doc_offsets_for(w)
    s = 1.0 / math.sqrt(w.hs)
    g = w.hc // w.hkv
    gk, gv, rk, rv = [], [], [], []
    for kv in kv_heads:
        dk = torch.zeros(len(cols), w.hs, dtype=F64)
        dv = torch.zeros(len(cols), w.hs, dtype=F64)
        k = x["k"][:, 0, kv].to(F64)
        v = x["v"][:, 0, kv].to(F64)
        for h in range(kv * g, (kv + 1) * g):
            a, b_ = oracle.attention_head_dkdv_cols(x["q"][:, 0, h].to(F64), k, v, x["do"][:, 0, h].to(F64), s,
                                                    w.causal, offs, cols, row_chunk=row_chunk)
            dk += a
            dv += b_
        gk.append(got["dk"][cols, 0, kv])
        gv.append(got["dv"][cols, 0, kv])
        rk.append(dk)
        rv.append(dv)
    assert_close("dK cols", torch.cat(gk), torch.cat(rk), w.torch_dtype, check_mean=uniform)
    assert_close("dV cols", torch.cat(gv), torch.cat(rv), w.torch_dtype, check_mean=uniform)


def test_llama8b_8k_forward(u):
    w = WORKLOADS["llama8b_8k"]
    x = make_global_inputs(w)
    got = run_workload(u, w, x)
    check_rows(w, x, got, heads=range(w.hc), rows_per_head=48, seed=81)


@pytest.mark.slow
def test_llama8b_32k_forward_backward(u):
    w = WORKLOADS["llama8b_32k"]
    x = make_global_inputs(w)
    got = run_workload(u, w, x, repeats=3, stores_ds=True)
    check_rows(w, x, got, heads=range(w.hc), rows_per_head=24, seed=82)
    # the first 32 keys of every kv head: seen by every query, the largest
    # sums (a biased sample: element-wise bound only)
    check_cols(w, x, got, kv_heads=range(w.hkv), cols=torch.arange(32), row_chunk=4096, uniform=False)
    rng = np.random.default_rng(83)
    tail = torch.tensor(np.sort(rng.choice(np.arange(w.sl - 1024, w.sl), 24, replace=False)))
    check_cols(w, x, got, kv_heads=range(w.hkv), cols=tail)          # tail keys of every kv head
    anywhere = torch.tensor(np.sort(rng.choice(w.sl, 16, replace=False)))
    check_cols(w, x, got, kv_heads=[5], cols=anywhere)                # keys anywhere, one kv head


@pytest.mark.slow
def test_packed_64k_forward_backward(u):
    w = WORKLOADS["packed_64k"]
    x = make_global_inputs(w)
    got = run_workload(u, w, x, repeats=3, stores_ds=True)
    check_rows(w, x, got, heads=range(0, w.hc, 3), rows_per_head=24, seed=84)
    offs = doc_offsets_for(w)
    rng = np.random.default_rng(85)
    # keys next to document boundaries (first keys of documents carry the
    # largest gradients: element-wise bound only), then keys at random places
    near = sorted({o + d for o in offs[1:-1] for d in (-1, 0, 1)})
    check_cols(w, x, got, kv_heads=[2], cols=torch.tensor(near[:18]), row_chunk=4096, uniform=False)
    check_cols(w, x, got, kv_heads=[6], cols=torch.tensor(np.sort(rng.choice(w.sl, 12, replace=False))),
               row_chunk=4096)


@pytest.mark.slow
def test_alst_128k_spot_check(u):
    w = WORKLOADS["alst_128k"]
    x = make_global_inputs(w)
    got = run_workload(u, w, x)
    # 1024 random query rows spread over the heads
    check_rows(w, x, got, heads=range(w.hc), rows_per_head=32, seed=86)
    rng = np.random.default_rng(87)
    tail = torch.tensor(np.sort(rng.choice(np.arange(w.sl - 512, w.sl), 16, replace=False)))
    check_cols(w, x, got, kv_heads=[0, 7], cols=tail)


@pytest.mark.slow
def test_alst_512k_spot_check(u):
    """The 512K-token layer (context for the pages' 500K-token ALST run): sampled rows and tail keys."""
    w = WORKLOADS["alst_512k"]
    x = make_global_inputs(w)
    got = run_workload(u, w, x)
    check_rows(w, x, got, heads=range(0, w.hc, 4), rows_per_head=16, seed=88)
    rng = np.random.default_rng(89)
    tail = torch.tensor(np.sort(rng.choice(np.arange(w.sl - 512, w.sl), 8, replace=False)))
    check_cols(w, x, got, kv_heads=[3], cols=tail)
