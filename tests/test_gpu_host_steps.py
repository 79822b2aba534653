"""Training steps from host memory (ulysses_host_begin / _step / _end).

Four steps with different inputs run back to back through HostSteps: the
inputs come from pinned host tensors and the outputs go to host tensors, with
the copies on the library's copy streams and the two device slots used
alternately. Each step's outputs must equal, bit for bit, what the fused
layer computes from the same inputs already on the device. Any missing order
between a slot's copies and its kernels would mix one step's data into
another's. The first step is also checked against the fp64 oracle.
"""
import pytest
import torch

import oracle
from tests._gpu import assert_close, rounding_sigma
from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


@pytest.mark.parametrize("sl,bs,hc,hkv,P,offs", [
    (1024, 1, 8, 4, 4, None),
    (1536, 2, 8, 2, 2, [0, 100, 900, 1536]),
])
def test_host_steps_match_the_device_path(u, sl, bs, hc, hkv, P, offs):
    L = u.UlyssesLayer(sl, bs, hc, hkv, 128, P, True, offs, torch.bfloat16)
    assert L.fused
    hs = u.HostSteps(L)
    steps = 4
    xs = [random_inputs(sl, bs, hc, hkv, 128, torch.bfloat16, 100 + i) for i in range(steps)]
    host_in = [{n: [t.pin_memory() for t in split_shards(x[n], P)] for n in ("q", "k", "v", "do")} for x in xs]

    def outs():
        mk = lambda H: [torch.full((sl // P, bs, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()  # noqa: E731
                        for _ in range(P)]
        return {"o": mk(hc), "dq": mk(hc), "dk": mk(hkv), "dv": mk(hkv)}

    host_out = [outs() for _ in range(steps)]
    stream = torch.cuda.current_stream()
    hs.begin(stream)
    for i in range(steps):
        hs.step(host_in[i], host_out[i], stream)
    hs.end(stream)
    stream.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK

    h2d, d2h = hs.host_bytes_per_step()
    assert h2d == d2h == (2 * hc + 2 * hkv) * sl * bs * 128 * 2

    R = u.UlyssesLayer(sl, bs, hc, hkv, 128, P, True, offs, torch.bfloat16)
    for i, x in enumerate(xs):
        cu = lambda t: [s.cuda() for s in split_shards(t, P)]  # noqa: E731
        o = R.new_seq_shards(hc)
        dq, dk, dv = R.new_seq_shards(hc), R.new_seq_shards(hkv), R.new_seq_shards(hkv)
        R.forward(cu(x["q"]), cu(x["k"]), cu(x["v"]), o)
        R.backward(cu(x["do"]), dq, dk, dv)
        torch.cuda.synchronize()
        for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            for r in range(P):
                assert torch.equal(host_out[i][name][r], ref[r].cpu()), (i, name, r)

    x = xs[0]
    qs, ks, vs, dos = (oracle.shard_sequence(x[n], P) for n in ("q", "k", "v", "do"))
    f = oracle.ulysses_forward(qs, ks, vs, P, causal=True, doc_offsets=offs)
    g = oracle.ulysses_backward(qs, ks, vs, dos, P, causal=True, doc_offsets=offs)
    sig = rounding_sigma(x, True, offs)
    for name, want in (("o", f["o"]), ("dq", g["dq"]), ("dk", g["dk"]), ("dv", g["dv"])):
        got = torch.cat(host_out[0][name])
        assert_close(name, got, oracle.unshard_sequence(want), torch.bfloat16, sigma=sig.get(name))


def test_host_step_rejects_bad_arguments(u):
    L = u.UlyssesLayer(1000, 1, 4, 2, 128, 2, True, None, torch.bfloat16)   # shards of 500: not fused
    assert not L.fused
    with pytest.raises(u.UlyssesError) as e:
        u.HostSteps(L)
    assert e.value.status == u.ULYSSES_ERR_UNSUPPORTED
    with pytest.raises(u.UlyssesError):
        u.ulysses_host_begin(L.h)
    F = u.UlyssesLayer(512, 1, 4, 2, 128, 2, True, None, torch.bfloat16)
    hs = u.HostSteps(F)
    lib = u._binding.lib
    n0 = u.ulysses_launch_count()
    assert lib.ulysses_host_step(F.h.ptr, 2, None, None, None, None, None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_host_step(F.h.ptr, 0, None, None, None, None, None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert u.ulysses_launch_count() == n0
    del hs
