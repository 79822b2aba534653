"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in the oracle (monkeypatched for the duration of
the test) and checks that at least one pin then fails. The mistakes are the
kind a restatement of the pages could make: a wrong GQA head map, a flipped
causal direction, a dropped softmax scale, strided instead of contiguous head
blocks, a document boundary off by one, a dropped term or a transposed operand
in the backward.
"""
import pytest
import torch

import oracle
import oracle.ulysses_oracle as uo
from tests import test_oracle_attention as fwd_pins
from tests import test_oracle_backward as bwd_pins
from tests import test_oracle_exchange as xch_pins

F64 = torch.float64


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _all_pins():
    """Every pin, as (callable, args)."""
    return [
        (xch_pins.test_layout_matches_2gpu_diagram, ()),
        (xch_pins.test_replicated_kv_heads, ()),
        (fwd_pins.test_forward_matches_sdpa, (8, 2, True)),
        (fwd_pins.test_forward_matches_sdpa, (4, 4, True)),
        (fwd_pins.test_packed_documents_match_sdpa_block_mask, ()),
        (fwd_pins.test_zero_query_gives_prefix_mean_and_log_count, ()),
        (fwd_pins.test_first_row_sees_only_first_key, ()),
        (bwd_pins.test_backward_matches_sdpa_autograd, (8, 2)),
        (bwd_pins.test_key_gradient_sums_to_zero_per_head, ()),
        (bwd_pins.test_zero_query_value_gradient_closed_form, ()),
        (bwd_pins.test_constant_values_zero_query_key_gradients, ()),
    ]


def _backward_mutant(drop_d=False, transpose_dk=False, sign=1.0):
    def mutant(q, k, v, dO, scale, causal, doc_offsets):
        sl = q.shape[0]
        rows = torch.arange(sl)
        O, LSE = uo.attention_rows(q, k, v, scale, causal, doc_offsets, rows)
        S = scale * (q @ k.T)
        M = uo.visible_mask(rows, sl, causal, doc_offsets)
        Pm = torch.where(M, torch.exp(S - LSE[:, None]), torch.zeros((), dtype=F64))
        D = (dO * O).sum(dim=1)
        if drop_d:
            D = torch.zeros_like(D)
        dV = Pm.T @ dO
        dS = Pm * (dO @ v.T - sign * D[:, None])
        dQ = scale * (dS @ k)
        dK = scale * ((dS @ q) if transpose_dk else (dS.T @ q))
        return dQ, dK, dV
    return mutant


_orig_kv = uo.kv_head_of
_orig_mask = uo.visible_mask
_orig_rows = uo.attention_rows
_orig_heads = uo.heads_of_rank
_orig_docs = uo.document_ids


def _flipped_mask(rows, sl, causal, offs):
    m = _orig_mask(rows, sl, False, offs)
    if causal:
        m &= torch.arange(sl)[None, :] >= rows[:, None]
    return m


def _strided_heads(r, H, P):
    if H % P == 0:
        return [r + P * j for j in range(H // P)]
    return _orig_heads(r, H, P)


def _docs_off_by_one(sl, offs):
    doc = torch.zeros(sl, dtype=torch.int64)
    if offs is not None:
        for d in range(len(offs) - 1):
            doc[offs[d] + 1:offs[d + 1] + 1] = d
    return doc[:sl]


MUTANTS = {
    "gqa_modulo_map": ("kv_head_of", lambda h, hc, hkv: h % hkv),
    "causal_flipped": ("visible_mask", _flipped_mask),
    "scale_dropped": ("attention_rows", lambda q, k, v, s, c, o, r: _orig_rows(q, k, v, 1.0, c, o, r)),
    "strided_head_blocks": ("heads_of_rank", _strided_heads),
    "doc_boundary_off_by_one": ("document_ids", _docs_off_by_one),
    "bwd_drops_D": ("attention_head_backward", _backward_mutant(drop_d=True)),
    "bwd_transposed_dk": ("attention_head_backward", _backward_mutant(transpose_dk=True)),
    "bwd_sign_of_D": ("attention_head_backward", _backward_mutant(sign=-1.0)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(uo, attr, fn)
    monkeypatch.setattr(oracle, attr, fn, raising=False)
    caught = [p.__name__ for p, a in _all_pins() if _fails(p, *a)]
    assert caught, f"no pin catches the mistake {name}"
