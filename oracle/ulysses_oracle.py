"""Plain, slow fp64 CPU oracle of the Ulysses sequence-parallel attention layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it. It shares no code with the CUDA
library and imports nothing from it.

What it computes comes from these pages:

* [HF] "Ulysses Sequence Parallelism: Training with Million-Token Contexts"
  (HF blog, Chinese translation). The numbered algorithm steps: sequence
  sharding, QKV projection, all-to-all, local attention, all-to-all, output
  projection. The note after them says that heads are independent.
* [TF] "Transformers 中的 DeepSpeed Ulysses 序列并行…技术指南", section
  "Ulysses 序列并行的核心原理". It has the 2-GPU layout diagram: before the
  exchange GPU0 holds tokens 0..N/2 with all H heads; after it GPU0 holds all
  N tokens and heads 0..H/2.
* [DS] "DeepSpeed Ulysses: 训练极长序列Transformer模型的系统优化", section
  "DeepSpeed-Ulysses的核心设计". The per-head attention equation is an image
  that did not survive extraction. Section "收敛性研究" says that sequence
  parallelism is a pure system optimisation that does not change the model's
  result.
* [ALST] "DeepSpeed Ulysses 序列并行与 Arctic 长序列训练（ALST）集成指南",
  section 2.1. Causality comes from ``position_ids`` plus ``is_causal``, with
  no 4D mask, and the position ids reset at each packed-document boundary
  (section 2.2). GQA needs the kv heads to be divisible by the sequence-parallel
  degree, or the degree divisible by the kv heads (with replication).

Readings taken where the pages are silent:

* Attention is ``softmax(Q K^T / sqrt(hs) + mask) V``, the SDPA / FlashAttention
  definition that the [HF] page names for the local step.
* Rank r holds the contiguous head block ``[r*H/P, (r+1)*H/P)`` ([TF] diagram).
* Query head h reads kv head ``h // (hc // hkv)``, the HF ``repeat_kv`` order.
  When P > hkv, rank r gets kv head ``r * hkv // P`` and the gradient of each
  kv head is the sum over its replicas.
* Mask: key j is visible from query i when ``doc(i) == doc(j)``, and, for
  causal attention, ``j <= i``. This is position-id reset semantics, i.e.
  block-diagonal causal attention for packed sequences.
* The logsumexp is the natural log of sum(exp) over the scaled, visible scores.
  Per rank it is stored as ``[bs, H/P, sl]``.
* dO arrives in the same sequence-sharded layout as O. dQ, dK and dV leave in
  the Q, K and V sequence-sharded layouts.

Every computation runs in torch float64 on the CPU. Inputs in bf16 or fp32 are
widened exactly.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import torch

F64 = torch.float64

__all__ = [
    "shard_sequence", "unshard_sequence", "heads_of_rank", "seq_to_head",
    "head_to_seq", "kv_head_of", "document_ids", "visible_mask",
    "attention_rows", "attention_head_forward", "attention_head_backward",
    "attention_head_dq_rows", "attention_head_dkdv_cols", "ulysses_forward",
    "ulysses_backward", "unsharded_forward", "unsharded_backward",
    "exchange_bytes",
]


# --------------------------------------------------------------------------
# Step 1: sequence sharding ([HF] step "sequence sharding")
# --------------------------------------------------------------------------
def shard_sequence(x: torch.Tensor, P: int) -> List[torch.Tensor]:
    """GPU i holds tokens [i*n/P, (i+1)*n/P) of x = [sl, bs, H, hs], all heads."""
    sl = x.shape[0]
    if sl % P != 0:
        raise ValueError("sequence length must be divisible by P")
    n = sl // P
    return [x[i * n:(i + 1) * n].clone() for i in range(P)]


def unshard_sequence(shards: Sequence[torch.Tensor]) -> torch.Tensor:
    """Concatenate sequence shards back into the global [sl, bs, H, hs] tensor."""
    return torch.cat(list(shards), dim=0)


# --------------------------------------------------------------------------
# Steps 3 and 5: the two all-to-all exchanges ([HF] steps 3 and 5; [TF] diagram)
# --------------------------------------------------------------------------
def heads_of_rank(r: int, H: int, P: int) -> List[int]:
    """Global heads that rank r holds after the seq->head exchange.

    H % P == 0: the contiguous block [r*H/P, (r+1)*H/P) ([TF] diagram).
    P % H == 0 (kv heads replicated, [ALST] 2.1): the single head r*H//P.
    """
    if H % P == 0:
        Hh = H // P
        return [r * Hh + j for j in range(Hh)]
    if P % H == 0:
        return [r * H // P]
    raise ValueError("heads must divide P or be divisible by P")


def seq_to_head(seq_shards: Sequence[torch.Tensor], P: int) -> List[torch.Tensor]:
    """seq->head all-to-all: P shards [sl/P, bs, H, hs] -> P shards [sl, bs, Hh, hs].

    Destination rank r, global token t = s*n + t' from source rank s, local
    head j (global head heads_of_rank(r)[j]):
        out[r][s*n + t', b, j, :] = seq_shards[s][t', b, heads_of_rank(r)[j], :]
    """
    n, bs, H, hs = seq_shards[0].shape
    sl = n * P
    out = []
    for r in range(P):
        hr = heads_of_rank(r, H, P)
        dst = torch.empty((sl, bs, len(hr), hs), dtype=seq_shards[0].dtype)
        for s in range(P):
            for j, h in enumerate(hr):
                dst[s * n:(s + 1) * n, :, j, :] = seq_shards[s][:, :, h, :]
        out.append(dst)
    return out


def head_to_seq(head_shards: Sequence[torch.Tensor], P: int, H: int,
                sum_replicas: bool = False) -> List[torch.Tensor]:
    """head->seq all-to-all, the inverse of seq_to_head.

        out[s][t', b, h, :] = head_shards[r][s*n + t', b, j, :]  for h = heads_of_rank(r)[j]

    With replicated heads (P > H) several ranks hold head h. For gradients
    (``sum_replicas=True``) their contributions add up. Otherwise every replica
    must be identical and the first one is taken.
    """
    sl, bs, _, hs = head_shards[0].shape
    n = sl // P
    dtype = head_shards[0].dtype
    out = [torch.zeros((n, bs, H, hs), dtype=dtype) for _ in range(P)]
    seen = set()
    for r in range(P):
        for j, h in enumerate(heads_of_rank(r, H, P)):
            for s in range(P):
                piece = head_shards[r][s * n:(s + 1) * n, :, j, :]
                if sum_replicas:
                    out[s][:, :, h, :] += piece
                elif h not in seen:
                    out[s][:, :, h, :] = piece
            seen.add(h)
    return out


def exchange_bytes(sl: int, bs: int, H: int, hs: int, elem_bytes: int) -> int:
    """Bytes one exchange moves in total: the whole [sl, bs, H, hs] tensor once.

    [DS] "显著的通信量减少": the Q, K, V exchange carries an aggregate message
    of 3Nh and the output exchange Nh. Each link carries M/P of an aggregate
    message of size M.
    """
    return sl * bs * H * hs * elem_bytes


# --------------------------------------------------------------------------
# Step 4: local attention per head ([HF] step 4; readings in the docstring)
# --------------------------------------------------------------------------
def kv_head_of(h: int, hc: int, hkv: int) -> int:
    """kv head read by query head h: h // (hc / hkv)."""
    return h // (hc // hkv)


def document_ids(sl: int, doc_offsets: Optional[Sequence[int]]) -> torch.Tensor:
    """Document index of every position. Position ids restart at each offset."""
    doc = torch.zeros(sl, dtype=torch.int64)
    if doc_offsets is not None:
        for d in range(len(doc_offsets) - 1):
            doc[doc_offsets[d]:doc_offsets[d + 1]] = d
    return doc


def visible_mask(rows: torch.Tensor, sl: int, causal: bool,
                 doc_offsets: Optional[Sequence[int]]) -> torch.Tensor:
    """Boolean [len(rows), sl]: key j is visible from query i."""
    doc = document_ids(sl, doc_offsets)
    j = torch.arange(sl)
    m = doc[rows][:, None] == doc[None, :]
    if causal:
        m &= j[None, :] <= rows[:, None]
    return m


def attention_rows(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                   causal: bool, doc_offsets, rows: torch.Tensor):
    """Attention of one head for the query rows ``rows``.

    q: [sl, hs], k and v: [sl, hs] (fp64). Returns O[rows] ([R, hs]) and
    LSE[rows] ([R]):
        S_ij = scale * q_i . k_j
        O_i = sum_j softmax_j(S_i + log M_i) v_j
        LSE_i = log sum_{j visible} exp(S_ij)
    The softmax subtracts the row maximum before exponentiating.
    """
    sl = k.shape[0]
    S = scale * (q[rows] @ k.T)
    M = visible_mask(rows, sl, causal, doc_offsets)
    S = S.masked_fill(~M, float("-inf"))
    m = S.max(dim=1).values
    E = torch.exp(S - m[:, None])
    l = E.sum(dim=1)
    O = (E @ v) / l[:, None]
    LSE = m + torch.log(l)
    return O, LSE


def attention_head_forward(q, k, v, scale, causal, doc_offsets):
    """Whole-head forward: O [sl, hs] and LSE [sl]."""
    return attention_rows(q, k, v, scale, causal, doc_offsets, torch.arange(q.shape[0]))


def attention_head_backward(q, k, v, dO, scale, causal, doc_offsets):
    """Gradients of one head for L with dL/dO = dO (whole head).

    With the forward's P_ij = M_ij exp(S_ij - LSE_i) and D_i = sum_d dO_id O_id:
        dV = P^T dO
        dP = dO V^T
        dS = P * (dP - D)
        dQ = scale * dS K
        dK = scale * dS^T Q
    Returns dQ, dK, dV ([sl, hs] each).
    """
    sl = q.shape[0]
    rows = torch.arange(sl)
    O, LSE = attention_rows(q, k, v, scale, causal, doc_offsets, rows)
    S = scale * (q @ k.T)
    M = visible_mask(rows, sl, causal, doc_offsets)
    Pm = torch.where(M, torch.exp(S - LSE[:, None]), torch.zeros((), dtype=F64))
    D = (dO * O).sum(dim=1)
    dV = Pm.T @ dO
    dP = dO @ v.T
    dS = Pm * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV


def attention_head_dq_rows(q, k, v, dO, scale, causal, doc_offsets, rows):
    """O, LSE and dQ of one head at the query rows ``rows`` only.

    Each of these depends on row i alone (D_i uses the oracle's own O_i), so a
    sample of rows is exact.
    """
    sl = q.shape[0]
    O, LSE = attention_rows(q, k, v, scale, causal, doc_offsets, rows)
    S = scale * (q[rows] @ k.T)
    M = visible_mask(rows, sl, causal, doc_offsets)
    Pm = torch.where(M, torch.exp(S - LSE[:, None]), torch.zeros((), dtype=F64))
    D = (dO[rows] * O).sum(dim=1)
    dP = dO[rows] @ v.T
    dS = Pm * (dP - D[:, None])
    dQ = scale * (dS @ k)
    return O, LSE, dQ


def attention_head_dkdv_cols(q, k, v, dO, scale, causal, doc_offsets, cols,
                             row_chunk: int = 1024):
    """dK and dV of one head at the key rows ``cols`` only.

    dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij q_i need LSE_i and
    D_i of every query i that sees key j. The sum over i runs over row chunks
    so that only a [row_chunk, sl] score block is in memory at a time. The
    terms and the sum are the ones of attention_head_backward.
    Returns dK[cols], dV[cols] ([C, hs] each).
    """
    sl, hs = q.shape
    C = cols.shape[0]
    dK = torch.zeros((C, hs), dtype=F64)
    dV = torch.zeros((C, hs), dtype=F64)
    i_lo = 0
    if causal:
        i_lo = int(cols.min())  # causal: no query before the earliest key sees it
    for a in range(i_lo, sl, row_chunk):
        rows = torch.arange(a, min(a + row_chunk, sl))
        O, LSE = attention_rows(q, k, v, scale, causal, doc_offsets, rows)
        D = (dO[rows] * O).sum(dim=1)
        S = scale * (q[rows] @ k[cols].T)
        M = visible_mask(rows, sl, causal, doc_offsets)[:, cols]
        Pm = torch.where(M, torch.exp(S - LSE[:, None]), torch.zeros((), dtype=F64))
        dP = dO[rows] @ v[cols].T
        dS = Pm * (dP - D[:, None])
        dV += Pm.T @ dO[rows]
        dK += scale * (dS.T @ q[rows])
    return dK, dV


# --------------------------------------------------------------------------
# The layer: exchange, per-rank attention, inverse exchange
# --------------------------------------------------------------------------
def _local_kv_index(r: int, j: int, hc: int, hkv: int, P: int) -> int:
    """Local kv index (on rank r) read by the rank's local query head j."""
    h = heads_of_rank(r, hc, P)[j]
    kv = kv_head_of(h, hc, hkv)
    return heads_of_rank(r, hkv, P).index(kv)


def ulysses_forward(q_shards, k_shards, v_shards, P: int, causal: bool = True,
                    doc_offsets=None, scale: Optional[float] = None):
    """The layer forward on P sequence shards.

    Returns a dict: ``o`` (P sequence shards of O, fp64), ``lse`` (per rank
    [bs, Hq, sl]), and the head-sharded intermediates ``qh``, ``kh``, ``vh``
    and ``oh``.
    """
    q_shards = [x.to(F64) for x in q_shards]
    k_shards = [x.to(F64) for x in k_shards]
    v_shards = [x.to(F64) for x in v_shards]
    n, bs, hc, hs = q_shards[0].shape
    hkv = k_shards[0].shape[2]
    sl = n * P
    if scale is None:
        scale = 1.0 / math.sqrt(hs)
    qh = seq_to_head(q_shards, P)
    kh = seq_to_head(k_shards, P)
    vh = seq_to_head(v_shards, P)
    Hq = qh[0].shape[2]
    oh, lse = [], []
    for r in range(P):
        o_r = torch.empty((sl, bs, Hq, hs), dtype=F64)
        lse_r = torch.empty((bs, Hq, sl), dtype=F64)
        for b in range(bs):
            for j in range(Hq):
                jk = _local_kv_index(r, j, hc, hkv, P)
                O, L = attention_head_forward(qh[r][:, b, j], kh[r][:, b, jk], vh[r][:, b, jk],
                                              scale, causal, doc_offsets)
                o_r[:, b, j] = O
                lse_r[b, j] = L
        oh.append(o_r)
        lse.append(lse_r)
    o = head_to_seq(oh, P, hc)
    return {"o": o, "lse": lse, "qh": qh, "kh": kh, "vh": vh, "oh": oh}


def ulysses_backward(q_shards, k_shards, v_shards, do_shards, P: int, causal: bool = True,
                     doc_offsets=None, scale: Optional[float] = None):
    """The layer backward: dO seq->head, per-head gradients, dQ/dK/dV head->seq.

    dK and dV of a kv head sum over the query heads of its group and, when kv
    heads are replicated, over the replicas. Returns a dict with ``dq``,
    ``dk``, ``dv`` (sequence shards, fp64) and the head-sharded
    ``dqh``, ``dkh``, ``dvh``.
    """
    q_shards = [x.to(F64) for x in q_shards]
    k_shards = [x.to(F64) for x in k_shards]
    v_shards = [x.to(F64) for x in v_shards]
    do_shards = [x.to(F64) for x in do_shards]
    n, bs, hc, hs = q_shards[0].shape
    hkv = k_shards[0].shape[2]
    sl = n * P
    if scale is None:
        scale = 1.0 / math.sqrt(hs)
    qh = seq_to_head(q_shards, P)
    kh = seq_to_head(k_shards, P)
    vh = seq_to_head(v_shards, P)
    doh = seq_to_head(do_shards, P)
    Hq, Hk = qh[0].shape[2], kh[0].shape[2]
    dqh, dkh, dvh = [], [], []
    for r in range(P):
        dq_r = torch.zeros((sl, bs, Hq, hs), dtype=F64)
        dk_r = torch.zeros((sl, bs, Hk, hs), dtype=F64)
        dv_r = torch.zeros((sl, bs, Hk, hs), dtype=F64)
        for b in range(bs):
            for j in range(Hq):
                jk = _local_kv_index(r, j, hc, hkv, P)
                dQ, dK, dV = attention_head_backward(qh[r][:, b, j], kh[r][:, b, jk],
                                                     vh[r][:, b, jk], doh[r][:, b, j],
                                                     scale, causal, doc_offsets)
                dq_r[:, b, j] = dQ
                dk_r[:, b, jk] += dK
                dv_r[:, b, jk] += dV
        dqh.append(dq_r)
        dkh.append(dk_r)
        dvh.append(dv_r)
    dq = head_to_seq(dqh, P, hc)
    dk = head_to_seq(dkh, P, hkv, sum_replicas=True)
    dv = head_to_seq(dvh, P, hkv, sum_replicas=True)
    return {"dq": dq, "dk": dk, "dv": dv, "dqh": dqh, "dkh": dkh, "dvh": dvh}


# --------------------------------------------------------------------------
# Unsharded single-device attention ([DS] "收敛性研究": SP leaves the result unchanged)
# --------------------------------------------------------------------------
def unsharded_forward(q, k, v, causal=True, doc_offsets=None, scale=None):
    """Single-device attention on the global [sl, bs, hc, hs] tensors (fp64).

    Returns O [sl, bs, hc, hs] and LSE [bs, hc, sl].
    """
    q, k, v = q.to(F64), k.to(F64), v.to(F64)
    sl, bs, hc, hs = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(hs)
    O = torch.empty((sl, bs, hc, hs), dtype=F64)
    L = torch.empty((bs, hc, sl), dtype=F64)
    for b in range(bs):
        for h in range(hc):
            kv = kv_head_of(h, hc, hkv)
            O[:, b, h], L[b, h] = attention_head_forward(q[:, b, h], k[:, b, kv], v[:, b, kv],
                                                         scale, causal, doc_offsets)
    return O, L


def unsharded_backward(q, k, v, dO, causal=True, doc_offsets=None, scale=None):
    """Single-device gradients dQ, dK, dV on the global tensors (fp64)."""
    q, k, v, dO = q.to(F64), k.to(F64), v.to(F64), dO.to(F64)
    sl, bs, hc, hs = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(hs)
    dq = torch.zeros((sl, bs, hc, hs), dtype=F64)
    dk = torch.zeros((sl, bs, hkv, hs), dtype=F64)
    dv = torch.zeros((sl, bs, hkv, hs), dtype=F64)
    for b in range(bs):
        for h in range(hc):
            kv = kv_head_of(h, hc, hkv)
            dQ, dK, dV = attention_head_backward(q[:, b, h], k[:, b, kv], v[:, b, kv], dO[:, b, h],
                                                 scale, causal, doc_offsets)
            dq[:, b, h] = dQ
            dk[:, b, kv] += dK
            dv[:, b, kv] += dV
    return dq, dk, dv
