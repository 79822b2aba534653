"""No kernel writes outside its output buffers, or into its inputs.

Every shard the layer reads or writes is a slice in the middle of a larger
allocation, with guard regions before and after it holding a sentinel bit
pattern. After a whole forward and backward (explicit and fused paths, ragged
lengths, a half pair of tiles at the end, packed documents), every guard must
still hold the sentinel, and every input must be unchanged. The TMA stores
clip tiles that run past the sequence; a wrong tensor-map extent or shard
offset would show up here as a changed guard.
"""
import pytest
import torch

from workloads import random_inputs, split_shards

pytestmark = pytest.mark.gpu

GUARD = 4096           # elements on each side (a multiple of 8: keeps 16-byte alignment)
SENTINEL = 0x7F3B      # a bf16 NaN bit pattern no kernel produces


@pytest.fixture(scope="module")
def u():
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


class Guarded:
    """A tensor of `shape` in the middle of a buffer with sentinel guards."""

    def __init__(self, shape, dtype, fill=None):
        n = 1
        for d in shape:
            n *= d
        self.n = n
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        self._bits(self.buf).fill_(SENTINEL if dtype == torch.bfloat16 else 0x7FBADBAD)
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    @staticmethod
    def _bits(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)

    def guards_intact(self):
        b = self._bits(self.buf)
        want = SENTINEL if self.buf.dtype == torch.bfloat16 else 0x7FBADBAD
        return bool((b[:GUARD] == want).all()) and bool((b[GUARD + self.n:] == want).all())


CASES = [
    # sl, bs, hc, hkv, P, causal, doc offsets, fused
    (1000, 1, 4, 2, 2, True, None, False),            # ragged tail (explicit path)
    (384, 2, 4, 4, 1, True, None, True),              # half pair of tiles at the end, batch 2
    (640, 1, 10, 5, 5, True, [0, 100, 640], True),    # five shards, packed, half pair
    (768, 1, 8, 2, 2, False, None, True),             # non-causal
    (384, 1, 8, 2, 8, True, None, False),             # replicated kv heads
]


@pytest.mark.parametrize("sl,bs,hc,hkv,P,causal,offs,fused", CASES)
def test_no_write_outside_the_buffers(u, sl, bs, hc, hkv, P, causal, offs, fused):
    dt = torch.bfloat16
    x = random_inputs(sl, bs, hc, hkv, 128, dt, 900 + sl)
    L = u.UlyssesLayer(sl, bs, hc, hkv, 128, P, causal, offs, dt, fused=fused)
    n = sl // P
    ins = {k: [Guarded(s.shape, dt, s.cuda()) for s in split_shards(x[k], P)] for k in ("q", "k", "v", "do")}
    copies = {k: [g.t.clone() for g in v] for k, v in ins.items()}
    outs = {k: [Guarded((n, bs, H, 128), dt) for _ in range(P)]
            for k, H in (("o", hc), ("dq", hc), ("dk", hkv), ("dv", hkv))}
    t = lambda gs: [g.t for g in gs]  # noqa: E731
    L.forward(t(ins["q"]), t(ins["k"]), t(ins["v"]), t(outs["o"]))
    L.backward(t(ins["do"]), t(outs["dq"]), t(outs["dk"]), t(outs["dv"]))
    torch.cuda.synchronize()
    assert u.ulysses_get_status(L.h) == u.ULYSSES_OK
    for k, gs in list(ins.items()) + list(outs.items()):
        for r, g in enumerate(gs):
            assert g.guards_intact(), f"{k}[{r}]: a guard region was written"
    for k, gs in ins.items():
        for r, g in enumerate(gs):
            assert torch.equal(g.t.view(torch.int16), copies[k][r].view(torch.int16)), f"input {k}[{r}] changed"
    for k, gs in outs.items():
        for r, g in enumerate(gs):
            assert not bool(torch.isnan(g.t).any()), f"{k}[{r}]: an output element was never written"


@pytest.mark.parametrize("stored_ds", [False, True])
def test_lse_and_workspace_stay_in_bounds(u, stored_ds):
    """The explicit calls with guarded LSE, head shards and workspace (with and without stored dS)."""
    sl, bs, hc, hkv, P = 1000, 1, 4, 2, 2
    dt = torch.bfloat16
    h = u.ulysses_create(sl, bs, hc, hkv, 128, P, True, [0, 333, 1000], dt)
    u.ulysses_set_ds_budget(h, 1 << 40 if stored_ds else 0)
    need, reserved = u.ulysses_ds_bytes(h)
    assert (0 < need <= reserved) == stored_ds
    x = random_inputs(sl, bs, hc, hkv, 128, dt, 77)
    Hq, Hk = hc // P, hkv // P
    heads = {k: [Guarded((sl, bs, H, 128), dt) for _ in range(P)]
             for k, H in (("q", Hq), ("k", Hk), ("v", Hk), ("o", Hq), ("do", Hq), ("dq", Hq), ("dk", Hk), ("dv", Hk))}
    lse = [Guarded((bs, Hq, sl), torch.float32) for _ in range(P)]
    nws = u.ulysses_workspace_size(h)
    ws = Guarded(((nws + 3) // 4,), torch.float32)
    t = lambda gs: [g.t for g in gs]  # noqa: E731
    for key, H in (("q", hc), ("k", hkv), ("v", hkv), ("do", hc)):
        u.ulysses_seq_to_head(h, H, [s.cuda() for s in split_shards(x[key], P)], t(heads[key]))
    u.ulysses_attn_fwd(h, t(heads["q"]), t(heads["k"]), t(heads["v"]), t(heads["o"]), t(lse))
    u.ulysses_attn_bwd(h, t(heads["q"]), t(heads["k"]), t(heads["v"]), t(heads["o"]), t(heads["do"]), t(lse),
                       t(heads["dq"]), t(heads["dk"]), t(heads["dv"]), ws.t)
    torch.cuda.synchronize()
    assert u.ulysses_get_status(h) == u.ULYSSES_OK
    for k, gs in heads.items():
        for r, g in enumerate(gs):
            assert g.guards_intact(), f"{k}[{r}]"
    for r, g in enumerate(lse):
        assert g.guards_intact(), f"lse[{r}]"
    assert ws.guards_intact(), "workspace"
    h.destroy()
