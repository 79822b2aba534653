"""Seeded synthetic inputs for the Ulysses attention layer.

This module is shared by the tests, the benchmark and the oracle checks. It
holds shapes, seeds and random draws only. It holds none of the layer's
arithmetic: no exchange, no attention, no masking.

The workloads stand in for the long-sequence Llama-8B training runs that the
DeepSpeed Ulysses / ALST pages describe ("DeepSpeed Ulysses 序列并行与 Arctic
长序列训练（ALST）集成指南", section 1.1). Those runs used real models and real
datasets. Attention cost depends only on the shapes and on the mask structure,
so seeded N(0, 1) tensors of the same shapes replace them.

Recipe (the pages are silent on it):
  * ``g = torch.Generator('cpu').manual_seed(seed)``.
  * Draw ``torch.randn`` in fp32, in this order: Q ``[sl, bs, hc, hs]``,
    K ``[sl, bs, hkv, hs]``, V ``[sl, bs, hkv, hs]``, dO ``[sl, bs, hc, hs]``.
  * Cast to the workload dtype. The bf16 cast rounds to nearest even.
  * The global ``[sl, bs, H, hs]`` tensor is the concatenation of the P
    sequence shards. Rank i holds tokens ``[i*sl/P, (i+1)*sl/P)``.
  * Packed documents: ``numpy.random.default_rng(seed)``. Draw 16 lengths
    from ``integers(1024, 7169, 16)`` (uniform in [1024, 7168]). Repeat the
    draw until the sum is at most sl. Extend the last document so that it
    ends at sl: the padding joins the last document.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int          # virtual ranks (sequence-parallel degree)
    bs: int         # batch
    sl: int         # global sequence length
    hc: int         # query heads
    hkv: int        # key/value heads
    hs: int         # head size
    dtype: str      # "bf16" or "fp32"
    causal: bool
    seed: int
    backward: bool  # whether the workload runs the backward pass
    ndoc: int = 0   # 0: one document spanning the whole sequence
    doc_len_range: tuple = (1024, 7168)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "fp32": torch.float32}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return {"bf16": 2, "fp32": 4}[self.dtype]


WORKLOADS = {
    # P=2, tiny, fp32, forward only.
    "tiny": Workload("tiny", P=2, bs=1, sl=256, hc=4, hkv=4, hs=32, dtype="fp32",
                     causal=True, seed=0, backward=False),
    # Llama-8B-shaped layer (32 q heads, 8 kv heads, head size 128), forward only.
    "llama8b_8k": Workload("llama8b_8k", P=4, bs=1, sl=8192, hc=32, hkv=8, hs=128,
                           dtype="bf16", causal=True, seed=1, backward=False),
    # Llama-8B-shaped layer, forward + backward.
    "llama8b_32k": Workload("llama8b_32k", P=8, bs=1, sl=32768, hc=32, hkv=8, hs=128,
                            dtype="bf16", causal=True, seed=2, backward=True),
    # Long-sequence ALST-style layer, forward + backward.
    "alst_128k": Workload("alst_128k", P=8, bs=1, sl=131072, hc=32, hkv=8, hs=128,
                          dtype="bf16", causal=True, seed=3, backward=True),
    # Packed batch of 16 documents, per-document causal, forward + backward.
    "packed_64k": Workload("packed_64k", P=8, bs=1, sl=65536, hc=32, hkv=8, hs=128,
                           dtype="bf16", causal=True, seed=4, backward=True, ndoc=16),
    # Context for the pages' ALST figure (a 500K-token Llama-8B sequence trained
    # on one H100): the attention layer of a 512K-token sequence, forward +
    # backward, on one GPU.
    "alst_512k": Workload("alst_512k", P=8, bs=1, sl=524288, hc=32, hkv=8, hs=128,
                          dtype="bf16", causal=True, seed=5, backward=True),
}


def document_lengths(seed: int, ndoc: int, sl: int, lo: int = 1024, hi: int = 7168):
    """Seeded document lengths for a packed batch (see the module docstring)."""
    rng = np.random.default_rng(seed)
    for _ in range(10000):
        lens = rng.integers(lo, hi + 1, ndoc)
        if int(lens.sum()) <= sl:
            lens = lens.astype(np.int64)
            lens[-1] += sl - int(lens.sum())
            return [int(x) for x in lens]
    raise RuntimeError("no accepted draw of document lengths")


def doc_offsets_for(w: Workload) -> Optional[list]:
    """Document start offsets (cu_seqlens style, ndoc+1 entries), or None."""
    if w.ndoc == 0:
        return None
    lens = document_lengths(w.seed, w.ndoc, w.sl, *w.doc_len_range)
    offs = [0]
    for n in lens:
        offs.append(offs[-1] + n)
    return offs


def make_global_inputs(w: Workload, with_grad: Optional[bool] = None, sl: Optional[int] = None):
    """Seeded global tensors Q, K, V (and dO) on the CPU, in the workload dtype.

    ``sl`` overrides the sequence length (smaller parity cases of the same
    head shape). Returns a dict with keys q, k, v and, when the workload runs
    the backward pass, do.
    """
    if with_grad is None:
        with_grad = w.backward
    sl = w.sl if sl is None else sl
    g = torch.Generator("cpu").manual_seed(w.seed)
    out = {}
    out["q"] = torch.randn((sl, w.bs, w.hc, w.hs), generator=g, dtype=torch.float32)
    out["k"] = torch.randn((sl, w.bs, w.hkv, w.hs), generator=g, dtype=torch.float32)
    out["v"] = torch.randn((sl, w.bs, w.hkv, w.hs), generator=g, dtype=torch.float32)
    if with_grad:
        out["do"] = torch.randn((sl, w.bs, w.hc, w.hs), generator=g, dtype=torch.float32)
    return {k: v.to(w.torch_dtype) for k, v in out.items()}


def random_inputs(sl, bs, hc, hkv, hs, dtype, seed, with_grad=True):
    """Seeded N(0,1) tensors for an arbitrary shape (parity and edge cases)."""
    g = torch.Generator("cpu").manual_seed(seed)
    out = {
        "q": torch.randn((sl, bs, hc, hs), generator=g),
        "k": torch.randn((sl, bs, hkv, hs), generator=g),
        "v": torch.randn((sl, bs, hkv, hs), generator=g),
    }
    if with_grad:
        out["do"] = torch.randn((sl, bs, hc, hs), generator=g)
    return {k: v.to(dtype) for k, v in out.items()}


def random_doc_offsets(sl: int, ndoc: int, seed: int, multiple: int = 1):
    """Seeded strictly increasing document offsets [0, ..., sl] with ndoc documents.

    ``multiple`` forces every boundary onto a multiple of that many tokens.
    """
    if ndoc <= 1:
        return [0, sl]
    rng = np.random.default_rng(seed)
    units = sl // multiple
    cuts = np.sort(rng.choice(np.arange(1, units), size=ndoc - 1, replace=False)) * multiple
    return [0] + [int(c) for c in cuts] + [sl]


def split_shards(x: torch.Tensor, P: int):
    """The P sequence shards of a global [sl, ...] tensor (contiguous copies)."""
    n = x.shape[0] // P
    return [x[i * n:(i + 1) * n].contiguous() for i in range(P)]
