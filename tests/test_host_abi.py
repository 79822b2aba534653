"""Host-side checks of the C-ABI library (no GPU needed).

* libulysses.so loads and exports every function that include/ulysses.h declares.
* ulysses_create applies the pages' divisibility rules before it touches the
  device. The rules come from the ALST guide, section 2.1 items (5) and (6),
  and from the HF blog section "比较 Ulysses 和 Ring Attention": sl and the
  heads divisible by the SP degree, num_heads >= sp_size, and kv heads that
  divide or are divided by the degree.
* Malformed document offsets, bad dtypes and NULL pointers are rejected.
"""
import ctypes
import json
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ulysses.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def u():
    import __graft_entry__
    __graft_entry__.build()
    import ulysses_sequence_attention_gb300 as pkg
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+(ulysses_[a-z0-9_]+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("ulysses_create", "ulysses_destroy", "ulysses_seq_to_head", "ulysses_head_to_seq",
                 "ulysses_attn_fwd", "ulysses_attn_bwd", "ulysses_workspace_size",
                 "ulysses_get_status", "ulysses_strerror"):
        assert need in names


def test_library_exports_every_declared_symbol(u):
    lib = ctypes.CDLL(u.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", u.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(ulysses_\w+)", out))
    assert set(declared_functions()) <= exported


def _status(u, **kw):
    args = dict(sl=1024, bs=1, hc=32, hkv=32, hs=128, P=1, causal=True, doc_offsets=None, dtype="bf16")
    args.update(kw)
    try:
        h = u.ulysses_create(**args)
        h.destroy()
        return u.ULYSSES_OK
    except u.UlyssesError as e:
        return e.status


def test_divisibility_rules_from_the_pages(u):
    g = json.load(open(os.path.join(GOLDEN, "divisibility_rules.json")))
    for case in g["accept"]:
        st = _status(u, sl=case["sl"], hc=case["hc"], hkv=case["hkv"], P=case["P"])
        # no GPU here: a valid shape gets as far as the device allocation
        assert st in (u.ULYSSES_OK, u.ULYSSES_ERR_CUDA), case
    for case in g["reject"]:
        st = _status(u, sl=case["sl"], hc=case["hc"], hkv=case["hkv"], P=case["P"])
        assert st == u.ULYSSES_ERR_DIVISIBILITY, case


@pytest.mark.parametrize("kw,expect", [
    (dict(hs=96), "UNSUPPORTED"),
    (dict(hs=256), "UNSUPPORTED"),
    (dict(P=256, hc=256, hkv=256, sl=1024), "UNSUPPORTED"),
    (dict(dtype=7), "INVALID_ARG"),
    (dict(sl=-8), "INVALID_ARG"),
    (dict(hc=0), "INVALID_ARG"),
    (dict(hc=32, hkv=5), "DIVISIBILITY"),
    (dict(doc_offsets=[0, 10, 10, 1024]), "INVALID_ARG"),
    (dict(doc_offsets=[0, 500, 1023]), "INVALID_ARG"),
    (dict(doc_offsets=[1, 500, 1024]), "INVALID_ARG"),
    (dict(doc_offsets=[0]), "INVALID_ARG"),
])
def test_rejections(u, kw, expect):
    assert _status(u, **kw) == getattr(u, "ULYSSES_ERR_" + expect)


def test_create_rejects_null_out_and_strerror_is_total(u):
    lib = u._binding.lib
    assert lib.ulysses_create(None, 64, 1, 4, 4, 32, 1, 1, None, 0, 0) == u.ULYSSES_ERR_INVALID_ARG
    for st in range(-8, 2):
        assert isinstance(u.ulysses_strerror(st), str)
    assert u.ulysses_strerror(u.ULYSSES_ERR_TIMEOUT) == "device-side wait timed out"


def test_null_handle_calls_are_rejected(u):
    lib = u._binding.lib
    n = ctypes.c_size_t()
    assert lib.ulysses_workspace_size(None, ctypes.byref(n)) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_seq_to_head(None, 4, None, None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_attn_fwd(None, None, None, None, None, None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_get_status(None) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_timing_enable(None, 1) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_timing_read(None, 0, None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_set_ds_budget(None, 1 << 30) == u.ULYSSES_ERR_INVALID_ARG
    assert lib.ulysses_ds_bytes(None, ctypes.byref(n), None) == u.ULYSSES_ERR_INVALID_ARG
    lib.ulysses_destroy(None)


def test_kernel_ids_match_the_header(u):
    text = open(HEADER).read()
    for i, name in enumerate(u.KERNEL_NAMES):
        assert re.search(rf"ULYSSES_KERNEL_{name.upper()}\s*=\s*{i},", text), name
    assert re.search(rf"ULYSSES_KERNEL_COUNT\s*=\s*{u.ULYSSES_KERNEL_COUNT}\b", text)


def declared_prototypes():
    """name -> number of parameters, from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"(ulysses_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, re.S):
        params = m.group(2).strip()
        protos[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_argument_counts_match_the_header(u):
    protos = declared_prototypes()
    assert set(protos) == set(declared_functions())
    for name, n in protos.items():
        fn = getattr(u._binding.lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def _varlen_status(u, **kw):
    args = dict(max_sl=4096, bs=1, hc=32, hkv=8, hs=128, P=8, causal=True, max_docs=4, dtype="bf16")
    args.update(kw)
    try:
        u.ulysses_create_varlen(**args).destroy()
        return u.ULYSSES_OK
    except u.UlyssesError as e:
        return e.status


@pytest.mark.parametrize("kw,expect", [
    (dict(max_docs=0), "INVALID_ARG"),
    (dict(max_sl=-1), "INVALID_ARG"),
    (dict(hc=30), "DIVISIBILITY"),          # heads not divisible by the degree
    (dict(hkv=3, hc=30, P=2), "DIVISIBILITY"),  # kv heads neither divide nor are divided by P
    (dict(hs=80), "UNSUPPORTED"),
    (dict(max_sl=(1 << 30) + 8), "UNSUPPORTED"),
])
def test_varlen_create_rejections(u, kw, expect):
    """The varying-length handle applies the same head rules as the fixed one, before any device call."""
    assert _varlen_status(u, **kw) == getattr(u, "ULYSSES_ERR_" + expect)


def test_varlen_capacity_need_not_divide_by_the_degree(u):
    # sl % P is a rule on each sequence (checked by ulysses_set_seq), not on the capacity
    st = _varlen_status(u, max_sl=4100)
    assert st in (u.ULYSSES_OK, u.ULYSSES_ERR_CUDA)   # no GPU here: it gets as far as the allocation


def test_set_seq_rejects_a_null_handle(u):
    assert u._binding.lib.ulysses_set_seq(None, 128, None, 0, None) == u.ULYSSES_ERR_INVALID_ARG
    assert u._binding.lib.ulysses_host_begin(None, None) == u.ULYSSES_ERR_INVALID_ARG
    assert u._binding.lib.ulysses_host_end(None, None) == u.ULYSSES_ERR_INVALID_ARG
