"""GPU parity of the whole layer (exchanges + attention fwd/bwd) against the oracle.

Each case runs the layer through the C-ABI, the way a user calls it, on both
paths:
* explicit: seq->head of Q, K and V, the attention forward, and head->seq of
  O; then seq->head of dO, the attention backward, and head->seq of dQ, dK and
  dV;
* fused: ulysses_layer_fwd and ulysses_layer_bwd, whose kernels read and write
  the sequence shards directly (where the shape allows it).
It compares every element with the oracle's fp64 result on the same seeded
inputs. The tolerances are max-abs 2e-2 and mean-abs 2e-3 for bf16, and 1e-4
for fp32. The logsumexp is compared per rank in its [bs, Hq, sl] layout.
"""
import pytest
import torch

import oracle
from tests._gpu import TOL, assert_close, cat_cpu, errors, replica_allowance, rounding_sigma
from workloads import WORKLOADS, make_global_inputs, random_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def run_layer(u, x, P, causal, offs, backward=True, fused=False):
    q, k, v = x["q"], x["k"], x["v"]
    sl, bs, hc, hs = q.shape
    hkv = k.shape[2]
    L = u.UlyssesLayer(sl, bs, hc, hkv, hs, P, causal, offs, q.dtype, fused=fused)
    qs, ks, vs = (split_shards(t, P) for t in (q, k, v))
    o = L.new_seq_shards(hc)
    L.forward([t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs], o)
    out = {"o": cat_cpu(o), "lse": [t.cpu() for t in L.lse]}
    if backward:
        dq, dk, dv = L.new_seq_shards(hc), L.new_seq_shards(hkv), L.new_seq_shards(hkv)
        L.backward([t.cuda() for t in split_shards(x["do"], P)], dq, dk, dv)
        out.update(dq=cat_cpu(dq), dk=cat_cpu(dk), dv=cat_cpu(dv))
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    return out


def oracle_layer(x, P, causal, offs, backward=True):
    """The oracle's layer; with the backward of a bf16 layer, also the rounding sigma of dK and dV."""
    qs, ks, vs = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v"))
    f = oracle.ulysses_forward(qs, ks, vs, P, causal=causal, doc_offsets=offs)
    res = {"o": oracle.unshard_sequence(f["o"]), "lse": f["lse"]}
    if backward:
        b = oracle.ulysses_backward(qs, ks, vs, oracle.shard_sequence(x["do"], P), P, causal=causal,
                                    doc_offsets=offs)
        res.update(dq=oracle.unshard_sequence(b["dq"]), dk=oracle.unshard_sequence(b["dk"]),
                   dv=oracle.unshard_sequence(b["dv"]), grad=b, P=P, hkv=x["k"].shape[2])
        if x["q"].dtype == torch.bfloat16:
            res["sigma"] = rounding_sigma(x, causal, offs)
    return res


def compare_all(got, want, dtype, backward=True):
    report = {}
    report["o"] = assert_close("O", got["o"], want["o"], dtype)
    for r, (a, b) in enumerate(zip(got["lse"], want["lse"])):
        mx, mean = errors(a, b)
        print(f"LSE rank {r}: max-abs {mx:.3g}, mean-abs {mean:.3g}")
        assert mx <= 1e-3, f"LSE rank {r}: max-abs {mx}"
    if backward:
        for n in ("dq", "dk", "dv"):
            extra = replica_allowance(want["grad"], n, want["P"], want["hkv"], dtype)
            sigma = want.get("sigma", {}).get(n)
            report[n] = assert_close(n, got[n], want[n], dtype, extra=extra, sigma=sigma)
    return report


def test_tiny_fp32_workload_forward(u):
    """The tiny fp32 workload: P=2, sl=256, 4 heads, hs=32, causal; 1e-4."""
    w = WORKLOADS["tiny"]
    x = make_global_inputs(w)
    got = run_layer(u, x, w.P, True, None, backward=False)
    want = oracle_layer(x, w.P, True, None, backward=False)
    compare_all(got, want, torch.float32, backward=False)


PARITY = [
    # sl, bs, hc, hkv, hs, P, dtype, causal, doc offsets, seed
    (256, 1, 4, 4, 32, 2, torch.float32, True, None, 1),           # fp32 backward
    (512, 1, 4, 2, 128, 2, torch.bfloat16, True, None, 2),         # several 128-tiles
    (1000, 1, 4, 2, 128, 2, torch.bfloat16, True, None, 3),        # ragged tail (1000 = 7*128 + 104)
    (1024, 1, 8, 2, 128, 4, torch.bfloat16, True, [0, 300, 301, 777, 1024], 4),   # packed, ragged docs
    (640, 2, 4, 4, 128, 2, torch.bfloat16, False, [0, 129, 640], 5),  # non-causal, batch 2
    (384, 1, 8, 2, 128, 8, torch.bfloat16, True, None, 6),         # replicated kv heads (P > hkv)
    (256, 1, 4, 4, 64, 1, torch.bfloat16, True, None, 7),          # P = 1, hs 64
    (96, 1, 2, 1, 32, 2, torch.float32, True, [0, 1, 2, 96], 8),   # single-token documents
    (2, 1, 2, 2, 128, 2, torch.bfloat16, True, None, 9),           # two tokens in all
    (2048, 1, 32, 8, 128, 8, torch.bfloat16, True, None, 11),      # Llama-8B heads, GQA group 4
    (2048, 1, 32, 8, 128, 8, torch.bfloat16, True, [0, 57, 700, 1500, 2048], 12),  # packed
    (1152, 1, 6, 2, 128, 2, torch.bfloat16, True, None, 13),       # group 3: a pair and a single
]


@pytest.mark.parametrize("sl,bs,hc,hkv,hs,P,dtype,causal,offs,seed", PARITY)
def test_layer_parity(u, sl, bs, hc, hkv, hs, P, dtype, causal, offs, seed):
    x = random_inputs(sl, bs, hc, hkv, hs, dtype, seed)
    got = run_layer(u, x, P, causal, offs)
    want = oracle_layer(x, P, causal, offs)
    compare_all(got, want, dtype)


def fused_ok(sl, hkv, hs, P, dtype):
    """The shapes ulysses_layer_fwd/_bwd accept (ulysses_fused_supported)."""
    return dtype == torch.bfloat16 and hs == 128 and P <= 8 and (sl // P) % 128 == 0 and hkv % P == 0


FUSED = [
    # sl, bs, hc, hkv, P, causal, doc offsets, seed
    (256, 1, 4, 2, 2, True, None, 21),             # one 128-row tile per shard
    (384, 1, 4, 4, 1, True, None, 22),             # P = 1, a half pair at the end
    (768, 2, 8, 4, 2, True, [0, 200, 768], 23),    # batch 2, a document across the shard boundary
    (1536, 1, 8, 4, 4, False, [0, 700, 1536], 24),  # non-causal, 3 tiles per shard
    (2048, 1, 32, 8, 8, True, None, 25),           # Llama-8B heads, 8 shards of 256
    (3072, 1, 32, 8, 8, True, [0, 57, 1100, 1101, 2900, 3072], 26),  # packed, shards of 384
    (640, 1, 10, 5, 5, True, None, 27),            # five shards, a half pair at the end
]


@pytest.mark.parametrize("sl,bs,hc,hkv,P,causal,offs,seed", FUSED)
def test_fused_layer_parity(u, sl, bs, hc, hkv, P, causal, offs, seed):
    """The fused entry points against the oracle, and bit for bit against the explicit path."""
    assert fused_ok(sl, hkv, 128, P, torch.bfloat16)
    x = random_inputs(sl, bs, hc, hkv, 128, torch.bfloat16, seed)
    got = run_layer(u, x, P, causal, offs, fused=True)
    want = oracle_layer(x, P, causal, offs)
    compare_all(got, want, torch.bfloat16)
    ref = run_layer(u, x, P, causal, offs, fused=False)
    for n in ("o", "dq", "dk", "dv"):
        assert torch.equal(got[n], ref[n]), n
    for a, b in zip(got["lse"], ref["lse"]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("sl,hc,hkv,hs,P,dtype", [
    (1000, 4, 2, 128, 2, torch.bfloat16),   # shards of 500 tokens: tiles would straddle two shards
    (1024, 8, 2, 128, 8, torch.bfloat16),   # replicated kv heads (shards of 128 tokens)
    (4096, 32, 16, 128, 16, torch.bfloat16),  # more shards than a launch holds maps for
    (256, 4, 4, 64, 2, torch.bfloat16),     # head size 64: the SIMT kernels
    (256, 4, 4, 128, 2, torch.float32),     # fp32
])
def test_fused_rejects_other_shapes(u, sl, hc, hkv, hs, P, dtype):
    assert not fused_ok(sl, hkv, hs, P, dtype)
    h = u.ulysses_create(sl, 1, hc, hkv, hs, P, True, None, dtype)
    assert not u.ulysses_fused_supported(h)
    n0 = u.ulysses_launch_count()
    n, Hq = sl // P, hc // P
    mk = lambda H: [torch.zeros((n, 1, H, hs), dtype=dtype, device="cuda") for _ in range(P)]  # noqa: E731
    lse = [torch.zeros((1, Hq, sl), dtype=torch.float32, device="cuda") for _ in range(P)]
    with pytest.raises(u.UlyssesError) as e:
        u.ulysses_layer_fwd(h, mk(hc), mk(hkv), mk(hkv), mk(hc), lse)
    assert e.value.status == u.ULYSSES_ERR_UNSUPPORTED
    assert u.ulysses_launch_count() == n0
    with pytest.raises(u.UlyssesError):
        u.UlyssesLayer(sl, 1, hc, hkv, hs, P, True, None, dtype, fused=True)
    h.destroy()


def test_empty_sequence_is_a_no_op(u):
    L = u.UlyssesLayer(0, 1, 4, 4, 128, 2, True, None, torch.bfloat16)
    o = L.new_seq_shards(4)
    e = [torch.empty((0, 1, 4, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ek = [torch.empty((0, 1, 4, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    L.forward(e, ek, ek, o)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK


def test_repeat_calls_are_deterministic(u):
    x = random_inputs(512, 1, 4, 2, 128, torch.bfloat16, 10)
    a = run_layer(u, x, 2, True, None)
    b = run_layer(u, x, 2, True, None)
    for n in ("o", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
