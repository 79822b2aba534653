"""UlyssesLayer: the layer's forward and backward on P virtual ranks of one GPU.

The steps follow the HF blog "Ulysses Sequence Parallelism: Training with
Million-Token Contexts" (algorithm steps 3 to 5) and their reverse for the
backward:

  forward:  Q, K, V seq->head  ->  attention forward  ->  O head->seq
  backward: dO seq->head  ->  attention backward  ->  dQ, dK, dV head->seq

Two ways to run them, both through the C-ABI of libulysses.so:

* fused (ulysses_layer_fwd / ulysses_layer_bwd): one call per pass. The
  attention kernels read the sequence shards and write the outputs back into
  sequence shards through their TMA tensor maps, so no exchange kernel runs
  and no head-shard copy exists. Used whenever ulysses_fused_supported allows.
* explicit: one call per step, with head-shard buffers in between. Used for
  every other shape, or when asked for with fused=False.

Both give bit-identical results. This class only owns the intermediate buffers
(torch device memory) and enqueues the calls on the current stream.

The backward's workspace can also hold dS (ulysses_set_ds_budget; by default
up to 64 GiB and a quarter of the device): the dK/dV kernel writes it and dQ
reads it back, instead of recomputing S and dP, for every sequence whose dS
fits the reserved area.

HostSteps runs whole training steps from host memory (ulysses_host_*): inputs
in, forward and backward, outputs out, with the copies overlapped with the
neighbouring steps' kernels.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import torch

from . import _binding as B


# Stored dS takes at most this much, and at most a quarter of the device.
DS_BUDGET_CAP = 64 << 30


def default_ds_budget(device="cuda") -> int:
    """The dS budget a layer gets unless told otherwise."""
    if not torch.cuda.is_available():
        return 0
    total = torch.cuda.get_device_properties(torch.device(device)).total_memory
    return min(DS_BUDGET_CAP, total // 4)


class UlyssesLayer:
    def __init__(self, sl: int, bs: int, hc: int, hkv: int, hs: int, P: int, causal: bool = True,
                 doc_offsets: Optional[Sequence[int]] = None, dtype=torch.bfloat16,
                 device: str = "cuda", fused: Optional[bool] = None, ds_budget: Optional[int] = None,
                 _handle=None):
        """fused: None picks the fused path when the shape allows it; True requires it.

        ds_budget: bytes of workspace the backward may keep dS in
        (ulysses_set_ds_budget); dQ then reads dS back instead of
        recomputing it, for every sequence whose dS fits. None: a layer of
        fixed length reserves what its own sequence needs, if that is within
        default_ds_budget(device), else nothing; a variable-length layer
        reserves up to default_ds_budget(device).
        """
        self.h = _handle or B.ulysses_create(sl, bs, hc, hkv, hs, P, causal, doc_offsets, dtype)
        if ds_budget is None:
            cap = default_ds_budget(device)
            need = B.ulysses_ds_bytes(self.h)[0]
            ds_budget = cap if _handle is not None else (need if need <= cap else 0)
        B.ulysses_set_ds_budget(self.h, int(ds_budget))
        self.cap_sl = getattr(self.h, "max_sl", sl)
        self.sl, self.bs, self.hc, self.hkv, self.hs, self.P = sl, bs, hc, hkv, hs, P
        self.dtype = dtype
        self.device = device
        self.Hq, self.Hk = self.h.Hq, self.h.Hk
        self._fused_pref = fused
        self._bufs = None
        self._saved = None
        self._pick_path()

    @classmethod
    def variable_length(cls, max_sl: int, bs: int, hc: int, hkv: int, hs: int, P: int, causal: bool = True,
                        max_docs: int = 1, dtype=torch.bfloat16, device: str = "cuda",
                        fused: Optional[bool] = None, ds_budget: Optional[int] = None) -> "UlyssesLayer":
        """A layer for batches of varying length (the pages' seq_length_is_variable=True).

        Starts empty; call set_seq before each batch of a new length or packing.
        Buffers are sized for max_sl once, so a new length allocates nothing.
        """
        h = B.ulysses_create_varlen(max_sl, bs, hc, hkv, hs, P, causal, max_docs, dtype)
        return cls(0, bs, hc, hkv, hs, P, causal, None, dtype, device, fused, ds_budget, _handle=h)

    def set_seq(self, sl: int, doc_offsets: Optional[Sequence[int]] = None, stream=None):
        """Switch to a sequence of sl tokens (packed at doc_offsets), in order on `stream`."""
        B.ulysses_set_seq(self.h, sl, doc_offsets, stream)
        self.sl = sl
        self._saved = None
        self._pick_path()

    @property
    def stores_ds(self) -> bool:
        """Whether the backward of the current sequence keeps dS (its blocks fit the reserved area)."""
        need, reserved = B.ulysses_ds_bytes(self.h)
        return 0 < need <= reserved

    def _pick_path(self):
        can = B.ulysses_fused_supported(self.h)
        if self._fused_pref and not can:
            raise B.UlyssesError(B.ULYSSES_ERR_UNSUPPORTED, "UlyssesLayer(fused=True)")
        self.fused = can if self._fused_pref is None else bool(self._fused_pref)

    # -- buffers -----------------------------------------------------------
    def _alloc(self, backward: bool):
        """Intermediate buffers, allocated once for the capacity; views of the current sl."""
        P, cap, bs, hs, dt, dev = self.P, self.cap_sl, self.bs, self.hs, self.dtype, self.device

        def heads(H):
            return [torch.empty(cap * bs * H * hs, dtype=dt, device=dev) for _ in range(P)]

        s = self._store = getattr(self, "_store", None) or {}
        if "lse" not in s:
            s["lse"] = [torch.empty(bs * self.Hq * cap, dtype=torch.float32, device=dev) for _ in range(P)]
        if not self.fused and "qh" not in s:
            s["qh"], s["kh"], s["vh"], s["oh"] = heads(self.Hq), heads(self.Hk), heads(self.Hk), heads(self.Hq)
        if backward and "ws" not in s:
            nbytes = B.ulysses_workspace_size(self.h)
            s["ws"] = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=dev)
        if backward and not self.fused and "doh" not in s:
            s["doh"], s["dqh"], s["dkh"], s["dvh"] = heads(self.Hq), heads(self.Hq), heads(self.Hk), heads(self.Hk)
        sl = self.sl
        shape = {"lse": (bs, self.Hq, sl), "qh": (sl, bs, self.Hq, hs), "oh": (sl, bs, self.Hq, hs),
                 "doh": (sl, bs, self.Hq, hs), "dqh": (sl, bs, self.Hq, hs), "kh": (sl, bs, self.Hk, hs),
                 "vh": (sl, bs, self.Hk, hs), "dkh": (sl, bs, self.Hk, hs), "dvh": (sl, bs, self.Hk, hs)}
        b = {n: [t[:math.prod(shape[n])].view(shape[n]) for t in v] for n, v in s.items() if n != "ws"}
        if "ws" in s:
            b["ws"] = s["ws"]
        self._bufs = b
        return b

    def new_seq_shards(self, H: int) -> List[torch.Tensor]:
        n = self.sl // self.P
        return [torch.empty((n, self.bs, H, self.hs), dtype=self.dtype, device=self.device)
                for _ in range(self.P)]

    # -- steps -------------------------------------------------------------
    def forward(self, q_seq, k_seq, v_seq, o_seq, stream=None):
        """Seq-sharded Q, K, V in, seq-sharded O out (all lists of P tensors).

        The fused path keeps references to q_seq, k_seq, v_seq and o_seq for
        the backward, as autograd keeps saved tensors: leave them unchanged
        until backward has been enqueued.
        """
        b = self._alloc(backward=False)
        if self.fused:
            B.ulysses_layer_fwd(self.h, q_seq, k_seq, v_seq, o_seq, b["lse"], stream)
            self._saved = (q_seq, k_seq, v_seq, o_seq)
            return o_seq
        B.ulysses_seq_to_head_qkv(self.h, q_seq, k_seq, v_seq, b["qh"], b["kh"], b["vh"], stream)
        B.ulysses_attn_fwd(self.h, b["qh"], b["kh"], b["vh"], b["oh"], b["lse"], stream)
        B.ulysses_head_to_seq(self.h, self.hc, b["oh"], o_seq, stream)
        return o_seq

    def backward(self, do_seq, dq_seq, dk_seq, dv_seq, stream=None):
        """Seq-sharded dO in, seq-sharded dQ, dK, dV out. Uses the last forward's state."""
        b = self._alloc(backward=True)
        if self.fused:
            if self._saved is None:
                raise RuntimeError("UlyssesLayer.backward before forward")
            q, k, v, o = self._saved
            B.ulysses_layer_bwd(self.h, q, k, v, o, do_seq, b["lse"], dq_seq, dk_seq, dv_seq, b["ws"], stream)
            return dq_seq, dk_seq, dv_seq
        B.ulysses_seq_to_head(self.h, self.hc, do_seq, b["doh"], stream)
        B.ulysses_attn_bwd(self.h, b["qh"], b["kh"], b["vh"], b["oh"], b["doh"], b["lse"],
                           b["dqh"], b["dkh"], b["dvh"], b["ws"], stream)
        B.ulysses_head_to_seq_qkv(self.h, b["dqh"], b["dkh"], b["dvh"], dq_seq, dk_seq, dv_seq, stream)
        return dq_seq, dk_seq, dv_seq

    @property
    def lse(self):
        return self._bufs["lse"]

    @property
    def head_buffers(self):
        return self._bufs


class HostSteps:
    """Training steps of a layer from host memory, copies overlapped with compute.

    Wraps ulysses_host_begin / ulysses_host_step / ulysses_host_end: the
    inputs (Q, K, V, dO sequence shards) come from host tensors and the
    outputs (O, dQ, dK, dV) go back to host tensors. Two slots of device
    buffers alternate, so one step's copies overlap its neighbours' kernels.
    Needs a shape that ulysses_fused_supported accepts.

        hs = HostSteps(layer)
        hs.begin()
        for batch, out in zip(batches, outs):   # dicts of lists of P CPU tensors
            hs.step(batch, out)
        hs.end()
        torch.cuda.current_stream().synchronize()   # outs are valid now
    """

    IN = ("q", "k", "v", "do")
    OUT = ("o", "dq", "dk", "dv")

    def __init__(self, layer: UlyssesLayer):
        if not layer.fused:
            raise B.UlyssesError(B.ULYSSES_ERR_UNSUPPORTED, "HostSteps needs the fused layer path")
        self.L = layer
        heads = {"q": layer.hc, "k": layer.hkv, "v": layer.hkv, "do": layer.hc,
                 "o": layer.hc, "dq": layer.hc, "dk": layer.hkv, "dv": layer.hkv}
        self.slots = [{n: layer.new_seq_shards(H) for n, H in heads.items()} for _ in range(2)]
        b = layer._alloc(backward=True)
        self.lse, self.ws = b["lse"], b["ws"]
        self.i = 0

    def host_bytes_per_step(self):
        """(host->device, device->host) bytes that one step copies."""
        per = lambda names: sum(t.numel() * t.element_size() for n in names for t in self.slots[0][n])  # noqa: E731
        return per(self.IN), per(self.OUT)

    def begin(self, stream=None):
        B.ulysses_host_begin(self.L.h, stream)

    def step(self, host_in, host_out, stream=None):
        s = self.slots[self.i % 2]
        dev = [s[n] for n in self.IN + self.OUT]
        B.ulysses_host_step(self.L.h, self.i % 2, [host_in[n] for n in self.IN], [host_out[n] for n in self.OUT],
                            dev, self.lse, self.ws, stream)
        self.i += 1

    def end(self, stream=None):
        B.ulysses_host_end(self.L.h, stream)
