"""GPU parity of the two exchanges against the oracle: bit for bit.

HF blog "Ulysses Sequence Parallelism: Training with Million-Token Contexts",
algorithm steps 3 and 5. Transformers guide, section "Ulysses 序列并行的核心原理"
(the 2-GPU layout diagram).
"""
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_global_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _run_s2h(u, h, H, seq):
    heads = H // h.P if H % h.P == 0 else 1
    out = [torch.full((h.sl, h.bs, heads, h.hs), float("nan"), dtype=seq[0].dtype, device="cuda")
           for _ in range(h.P)]
    u.ulysses_seq_to_head(h, H, [s.cuda() for s in seq], out)
    return out


def _run_h2s(u, h, H, heads_in):
    n = h.sl // h.P
    out = [torch.full((n, h.bs, H, h.hs), float("nan"), dtype=heads_in[0].dtype, device="cuda")
           for _ in range(h.P)]
    u.ulysses_head_to_seq(h, H, [s.cuda() for s in heads_in], out)
    return out


CASES = [
    # sl, bs, hc, hkv, hs, P, dtype
    (256, 1, 4, 4, 32, 2, torch.float32),
    (64, 1, 8, 8, 64, 1, torch.bfloat16),
    (1000, 2, 8, 2, 128, 2, torch.bfloat16),
    (96, 3, 12, 4, 64, 4, torch.bfloat16),
    (4096, 1, 32, 8, 128, 8, torch.bfloat16),
    (384, 1, 32, 32, 128, 32, torch.bfloat16),
    (128, 2, 16, 16, 32, 16, torch.float32),
]


@pytest.mark.parametrize("sl,bs,hc,hkv,hs,P,dtype", CASES)
def test_exchanges_bit_exact(u, sl, bs, hc, hkv, hs, P, dtype):
    g = torch.Generator().manual_seed(sl + P)
    h = u.ulysses_create(sl, bs, hc, hkv, hs, P, True, None, dtype)
    for H in sorted({hc, hkv}):
        x = torch.randn((sl, bs, H, hs), generator=g).to(dtype)
        seq = oracle.shard_sequence(x, P)
        want = oracle.seq_to_head(seq, P)
        got = _run_s2h(u, h, H, seq)
        for r in range(P):
            assert torch.equal(_bits(got[r].cpu()), _bits(want[r])), (H, r)
        if H % P == 0:
            back = _run_h2s(u, h, H, want)
            want_back = oracle.head_to_seq(want, P, H)
            for r in range(P):
                assert torch.equal(_bits(back[r].cpu()), _bits(want_back[r]))
                assert torch.equal(_bits(back[r].cpu()), _bits(seq[r]))
    torch.cuda.synchronize()
    h.destroy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_replicated_kv_exchange_and_gradient_sum(u, dtype):
    sl, bs, hc, hkv, hs, P = 64, 2, 8, 2, 32, 8
    g = torch.Generator().manual_seed(5)
    h = u.ulysses_create(sl, bs, hc, hkv, hs, P, True, None, dtype)
    x = torch.randn((sl, bs, hkv, hs), generator=g).to(dtype)
    seq = oracle.shard_sequence(x, P)
    got = _run_s2h(u, h, hkv, seq)
    want = oracle.seq_to_head(seq, P)
    for r in range(P):
        assert torch.equal(_bits(got[r].cpu()), _bits(want[r]))
    grads = [torch.randn((sl, bs, 1, hs), generator=g).to(dtype) for _ in range(P)]
    summed = _run_h2s(u, h, hkv, grads)
    ref = oracle.head_to_seq([t.to(torch.float64) for t in grads], P, hkv, sum_replicas=True)
    mag = oracle.head_to_seq([t.to(torch.float64).abs() for t in grads], P, hkv, sum_replicas=True)
    for r in range(P):
        # an fp32 sum of the replicas (error <= reps * 2^-24 * sum|x|), rounded once to the
        # element type (half an ulp of the result)
        d = (summed[r].cpu().to(torch.float64) - ref[r]).abs()
        half_ulp = ref[r].abs() * (2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24)
        bound = half_ulp + (P // hkv) * 2.0 ** -24 * mag[r] + 1e-30
        assert torch.all(d <= bound), float((d / bound).max())
    h.destroy()


def test_empty_layer_is_a_no_op(u):
    h = u.ulysses_create(0, 1, 4, 4, 32, 2, True, None, torch.bfloat16)
    e = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    u.ulysses_seq_to_head(h, 4, [e, e], [e, e])
    u.ulysses_head_to_seq(h, 4, [e, e], [e, e])
    assert u.ulysses_get_status(h) == u.ULYSSES_OK
    h.destroy()


def test_misaligned_pointer_is_rejected_before_launch(u):
    h = u.ulysses_create(64, 1, 4, 4, 32, 2, True, None, torch.float32)
    buf = torch.zeros(64 * 4 * 32 + 4, device="cuda")
    src = [buf[1:1 + 32 * 4 * 32], buf[1:1 + 32 * 4 * 32]]   # 4-byte offset
    dst = [torch.zeros(64 * 2 * 32, device="cuda") for _ in range(2)]
    with pytest.raises(u.UlyssesError) as ei:
        u.ulysses_seq_to_head(h, 4, src, dst)
    assert ei.value.status == u.ULYSSES_ERR_ALIGNMENT
    h.destroy()


@pytest.mark.parametrize("name", ["llama8b_32k", "alst_128k"])
def test_fullsize_exchanges_bit_exact(u, name):
    w = WORKLOADS[name]
    x = make_global_inputs(w, with_grad=False)
    h = u.ulysses_create(w.sl, w.bs, w.hc, w.hkv, w.hs, w.P, True, None, w.torch_dtype)
    for key, H in (("q", w.hc), ("k", w.hkv)):
        seq = split_shards(x[key], w.P)
        got = _run_s2h(u, h, H, seq)
        want = oracle.seq_to_head(seq, w.P)
        for r in range(w.P):
            assert torch.equal(_bits(got[r].cpu()), _bits(want[r]))
        back = _run_h2s(u, h, H, [g.cpu() for g in got])
        for r in range(w.P):
            assert torch.equal(_bits(back[r].cpu()), _bits(seq[r]))
        del got, back
    h.destroy()


@pytest.mark.parametrize("sl,bs,hc,hkv,hs,P,dtype", [
    (1000, 2, 8, 2, 128, 2, torch.bfloat16),
    (4096, 1, 32, 8, 128, 8, torch.bfloat16),
    (96, 3, 12, 4, 64, 4, torch.float32),
    (64, 2, 8, 2, 32, 8, torch.bfloat16),      # replicated kv heads (P > hkv)
])
def test_qkv_exchanges_in_one_call(u, sl, bs, hc, hkv, hs, P, dtype):
    """ulysses_seq_to_head_qkv / ulysses_head_to_seq_qkv: each tensor as the single-tensor exchange, bit for bit."""
    g = torch.Generator().manual_seed(sl * 3 + P)
    h = u.ulysses_create(sl, bs, hc, hkv, hs, P, True, None, dtype)
    xs = {"q": torch.randn((sl, bs, hc, hs), generator=g).to(dtype),
          "k": torch.randn((sl, bs, hkv, hs), generator=g).to(dtype),
          "v": torch.randn((sl, bs, hkv, hs), generator=g).to(dtype)}
    seq = {k: oracle.shard_sequence(x, P) for k, x in xs.items()}
    Hk = hkv // P if hkv % P == 0 else 1
    heads = {"q": hc // P, "k": Hk, "v": Hk}
    out = {k: [torch.full((sl, bs, heads[k], hs), float("nan"), dtype=dtype, device="cuda") for _ in range(P)]
           for k in xs}
    u.ulysses_seq_to_head_qkv(h, *[[s.cuda() for s in seq[k]] for k in ("q", "k", "v")],
                              out["q"], out["k"], out["v"])
    for k in xs:
        want = oracle.seq_to_head(seq[k], P)
        for r in range(P):
            assert torch.equal(_bits(out[k][r].cpu()), _bits(want[r])), (k, r)
    # head->seq of three gradients (summed over replicas when P > hkv)
    grads = {k: [torch.randn((sl, bs, heads[k], hs), generator=g).to(dtype) for _ in range(P)] for k in xs}
    back = {k: [torch.full((sl // P, bs, xs[k].shape[2], hs), float("nan"), dtype=dtype, device="cuda")
                for _ in range(P)] for k in xs}
    u.ulysses_head_to_seq_qkv(h, *[[t.cuda() for t in grads[k]] for k in ("q", "k", "v")],
                              back["q"], back["k"], back["v"])
    for k, H in (("q", hc), ("k", hkv), ("v", hkv)):
        ref = _run_h2s(u, h, H, grads[k])        # the single-tensor exchange
        for r in range(P):
            assert torch.equal(_bits(back[k][r].cpu()), _bits(ref[r].cpu())), (k, r)
    n0 = u.ulysses_launch_count()
    u.ulysses_seq_to_head_qkv(h, *[[s.cuda() for s in seq[kk]] for kk in ("q", "k", "v")],
                              out["q"], out["k"], out["v"])
    assert u.ulysses_launch_count() - n0 == 1
    torch.cuda.synchronize()
    h.destroy()
