"""ctypes binding of libulysses.so: the C-ABI calls under the same names.

Marshalling only: torch tensors become device pointers, the current torch
stream becomes a cudaStream_t, and a non-zero status becomes an exception.
The binding checks each tensor's device, dtype, contiguity and element count
against the handle's shape before it passes the pointer on, so that a wrong
buffer fails on the host instead of on the GPU. All compute runs in the
library's CUDA kernels. There is no fallback: importing this module fails when
the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libulysses.so")

ULYSSES_OK = 0
ULYSSES_ERR_INVALID_ARG = -1
ULYSSES_ERR_DIVISIBILITY = -2
ULYSSES_ERR_ALIGNMENT = -3
ULYSSES_ERR_UNSUPPORTED = -4
ULYSSES_ERR_CUDA = -5
ULYSSES_ERR_TIMEOUT = -6
ULYSSES_ERR_TOO_LARGE = -7
ULYSSES_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
ULYSSES_BF16 = 0
ULYSSES_FP32 = 1
ULYSSES_MAX_P = 128
ULYSSES_KERNEL_SEQ_TO_HEAD = 0
ULYSSES_KERNEL_HEAD_TO_SEQ = 1
ULYSSES_KERNEL_ATTN_FWD = 2
ULYSSES_KERNEL_BWD_PREP = 3
ULYSSES_KERNEL_BWD_DKDV = 4
ULYSSES_KERNEL_BWD_DQ = 5
ULYSSES_KERNEL_COUNT = 6
KERNEL_NAMES = ("seq_to_head", "head_to_seq", "attn_fwd", "bwd_prep", "bwd_dkdv", "bwd_dq")

_DTYPES = {"bf16": ULYSSES_BF16, "fp32": ULYSSES_FP32,
           torch.bfloat16: ULYSSES_BF16, torch.float32: ULYSSES_FP32}
_TORCH = {ULYSSES_BF16: torch.bfloat16, ULYSSES_FP32: torch.float32}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "ulysses_sequence_attention_gb300.build.build()")

lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_pp = ctypes.POINTER(ctypes.c_void_p)
lib.ulysses_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int]
lib.ulysses_create.restype = ctypes.c_int
lib.ulysses_create_varlen.argtypes = [ctypes.POINTER(_vp), ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int]
lib.ulysses_create_varlen.restype = ctypes.c_int
lib.ulysses_set_seq.argtypes = [_vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, _vp]
lib.ulysses_set_seq.restype = ctypes.c_int
lib.ulysses_destroy.argtypes = [_vp]
lib.ulysses_destroy.restype = None
lib.ulysses_strerror.argtypes = [ctypes.c_int]
lib.ulysses_strerror.restype = ctypes.c_char_p
lib.ulysses_workspace_size.argtypes = [_vp, ctypes.POINTER(ctypes.c_size_t)]
lib.ulysses_workspace_size.restype = ctypes.c_int
lib.ulysses_set_ds_budget.argtypes = [_vp, ctypes.c_size_t]
lib.ulysses_set_ds_budget.restype = ctypes.c_int
lib.ulysses_ds_bytes.argtypes = [_vp, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
lib.ulysses_ds_bytes.restype = ctypes.c_int
lib.ulysses_seq_to_head.argtypes = [_vp, ctypes.c_int, _pp, _pp, _vp]
lib.ulysses_seq_to_head.restype = ctypes.c_int
lib.ulysses_head_to_seq.argtypes = [_vp, ctypes.c_int, _pp, _pp, _vp]
lib.ulysses_head_to_seq.restype = ctypes.c_int
lib.ulysses_seq_to_head_qkv.argtypes = [_vp] + [_pp] * 6 + [_vp]
lib.ulysses_seq_to_head_qkv.restype = ctypes.c_int
lib.ulysses_head_to_seq_qkv.argtypes = [_vp] + [_pp] * 6 + [_vp]
lib.ulysses_head_to_seq_qkv.restype = ctypes.c_int
lib.ulysses_attn_fwd.argtypes = [_vp, _pp, _pp, _pp, _pp, _pp, _vp]
lib.ulysses_attn_fwd.restype = ctypes.c_int
lib.ulysses_attn_bwd.argtypes = [_vp] + [_pp] * 9 + [_vp, _vp]
lib.ulysses_attn_bwd.restype = ctypes.c_int
lib.ulysses_layer_fwd.argtypes = [_vp, _pp, _pp, _pp, _pp, _pp, _vp]
lib.ulysses_layer_fwd.restype = ctypes.c_int
lib.ulysses_layer_bwd.argtypes = [_vp] + [_pp] * 9 + [_vp, _vp]
lib.ulysses_layer_bwd.restype = ctypes.c_int
lib.ulysses_fused_supported.argtypes = [_vp]
lib.ulysses_fused_supported.restype = ctypes.c_int
lib.ulysses_host_begin.argtypes = [_vp, _vp]
lib.ulysses_host_begin.restype = ctypes.c_int
lib.ulysses_host_end.argtypes = [_vp, _vp]
lib.ulysses_host_end.restype = ctypes.c_int
lib.ulysses_host_step.argtypes = [_vp, ctypes.c_int, _pp, _pp, _pp, _pp, _vp, _vp]
lib.ulysses_host_step.restype = ctypes.c_int
lib.ulysses_get_status.argtypes = [_vp]
lib.ulysses_get_status.restype = ctypes.c_int
lib.ulysses_attn_bwd_noalloc.argtypes = [_vp] + [_pp] * 9 + [_vp]
lib.ulysses_attn_bwd_noalloc.restype = ctypes.c_int
lib.ulysses_set_wait_limit.argtypes = [_vp, ctypes.c_int64]
lib.ulysses_set_wait_limit.restype = ctypes.c_int
lib.ulysses_inject_fault.argtypes = [_vp, ctypes.c_int]
lib.ulysses_inject_fault.restype = ctypes.c_int
lib.ulysses_launch_count.argtypes = []
lib.ulysses_launch_count.restype = ctypes.c_uint64
lib.ulysses_timing_enable.argtypes = [_vp, ctypes.c_int]
lib.ulysses_timing_enable.restype = ctypes.c_int
lib.ulysses_timing_read.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_int64)]
lib.ulysses_timing_read.restype = ctypes.c_int


class UlyssesError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {ulysses_strerror(status)} ({status})")


def ulysses_strerror(status: int) -> str:
    return lib.ulysses_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != ULYSSES_OK:
        raise UlyssesError(status, what)


class UlyssesHandle:
    """Owns one ulysses_t. Shape fields mirror the ulysses_create arguments."""

    def __init__(self, ptr, sl, bs, hc, hkv, hs, P, causal, doc_offsets, dtype):
        self._ptr = ptr
        self.sl, self.bs, self.hc, self.hkv, self.hs, self.P = sl, bs, hc, hkv, hs, P
        self.causal = causal
        self.doc_offsets = doc_offsets
        self.dtype = dtype
        self.Hq = hc // P
        self.Hk = hkv // P if hkv % P == 0 else 1

    @property
    def ptr(self):
        return self._ptr

    @property
    def torch_dtype(self):
        return _TORCH[self.dtype]

    def destroy(self):
        if self._ptr:
            lib.ulysses_destroy(self._ptr)
            self._ptr = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def ulysses_create(sl: int, bs: int, hc: int, hkv: int, hs: int, P: int, causal: bool = True,
                   doc_offsets: Optional[Sequence[int]] = None, dtype="bf16") -> UlyssesHandle:
    dt = _DTYPES.get(dtype, dtype)
    out = _vp()
    if doc_offsets is not None:
        offs = (ctypes.c_int32 * len(doc_offsets))(*[int(x) for x in doc_offsets])
        nd = len(doc_offsets) - 1
    else:
        offs, nd = None, 0
    st = lib.ulysses_create(ctypes.byref(out), int(sl), int(bs), int(hc), int(hkv), int(hs), int(P),
                            int(bool(causal)), offs, nd, int(dt))
    _check(st, "ulysses_create")
    return UlyssesHandle(out.value, sl, bs, hc, hkv, hs, P, bool(causal),
                         None if doc_offsets is None else list(doc_offsets), dt)


def ulysses_create_varlen(max_sl: int, bs: int, hc: int, hkv: int, hs: int, P: int, causal: bool = True,
                          max_docs: int = 1, dtype="bf16") -> UlyssesHandle:
    """A handle for sequences of varying length up to max_sl; empty until ulysses_set_seq."""
    dt = _DTYPES.get(dtype, dtype)
    out = _vp()
    st = lib.ulysses_create_varlen(ctypes.byref(out), int(max_sl), int(bs), int(hc), int(hkv), int(hs), int(P),
                                   int(bool(causal)), int(max_docs), int(dt))
    _check(st, "ulysses_create_varlen")
    h = UlyssesHandle(out.value, 0, bs, hc, hkv, hs, P, bool(causal), None, dt)
    h.max_sl, h.max_docs = int(max_sl), int(max_docs)
    return h


def ulysses_set_seq(h: UlyssesHandle, sl: int, doc_offsets: Optional[Sequence[int]] = None, stream=None):
    """Switch h to a new sequence (length and document offsets), in order on `stream`."""
    if doc_offsets is not None:
        offs = (ctypes.c_int32 * len(doc_offsets))(*[int(x) for x in doc_offsets])
        nd = len(doc_offsets) - 1
    else:
        offs, nd = None, 0
    _check(lib.ulysses_set_seq(h.ptr, int(sl), offs, nd, _stream(stream)), "ulysses_set_seq")
    h.sl = int(sl)
    h.doc_offsets = None if doc_offsets is None else list(doc_offsets)


def ulysses_destroy(h: UlyssesHandle):
    h.destroy()


def ulysses_workspace_size(h: UlyssesHandle) -> int:
    n = ctypes.c_size_t()
    _check(lib.ulysses_workspace_size(h.ptr, ctypes.byref(n)), "ulysses_workspace_size")
    return int(n.value)


def ulysses_set_ds_budget(h: UlyssesHandle, nbytes: int):
    _check(lib.ulysses_set_ds_budget(h.ptr, int(nbytes)), "ulysses_set_ds_budget")


def ulysses_ds_bytes(h: UlyssesHandle):
    """(needed, reserved): the stored-dS area the current sequence uses, and the one reserved."""
    n, r = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.ulysses_ds_bytes(h.ptr, ctypes.byref(n), ctypes.byref(r)), "ulysses_ds_bytes")
    return int(n.value), int(r.value)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptrs(h: UlyssesHandle, tensors, numel: int, dtype: torch.dtype, name: str):
    if len(tensors) != h.P:
        raise ValueError(f"{name}: expected {h.P} rank buffers, got {len(tensors)}")
    out = (_vp * h.P)()
    for r, t in enumerate(tensors):
        if isinstance(t, int):
            out[r] = t
            continue
        if t.dtype != dtype:
            raise TypeError(f"{name}[{r}]: dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{r}] must be contiguous")
        if t.numel() != numel:
            raise ValueError(f"{name}[{r}]: {t.numel()} elements, expected {numel}")
        if t.device.type != "cuda":
            raise ValueError(f"{name}[{r}] must be a CUDA tensor")
        out[r] = t.data_ptr()
    return ctypes.cast(out, _pp)


def _heads_per_rank(h: UlyssesHandle, nheads: int) -> int:
    return nheads // h.P if nheads % h.P == 0 else 1


def ulysses_seq_to_head(h: UlyssesHandle, nheads: int, seq_shards, head_shards, stream=None):
    dt = h.torch_dtype
    n = h.sl // h.P
    src = _ptrs(h, seq_shards, n * h.bs * nheads * h.hs, dt, "seq_shards")
    dst = _ptrs(h, head_shards, h.sl * h.bs * _heads_per_rank(h, nheads) * h.hs, dt, "head_shards")
    _check(lib.ulysses_seq_to_head(h.ptr, int(nheads), src, dst, _stream(stream)), "ulysses_seq_to_head")


def ulysses_head_to_seq(h: UlyssesHandle, nheads: int, head_shards, seq_shards, stream=None):
    dt = h.torch_dtype
    n = h.sl // h.P
    src = _ptrs(h, head_shards, h.sl * h.bs * _heads_per_rank(h, nheads) * h.hs, dt, "head_shards")
    dst = _ptrs(h, seq_shards, n * h.bs * nheads * h.hs, dt, "seq_shards")
    _check(lib.ulysses_head_to_seq(h.ptr, int(nheads), src, dst, _stream(stream)), "ulysses_head_to_seq")


def ulysses_seq_to_head_qkv(h: UlyssesHandle, q_seq, k_seq, v_seq, q_head, k_head, v_head, stream=None):
    """seq->head of Q, K and V in one launch."""
    dt = h.torch_dtype
    n = h.sl // h.P
    sq, sk = n * h.bs * h.hc * h.hs, n * h.bs * h.hkv * h.hs
    hq, hk = h.sl * h.bs * h.Hq * h.hs, h.sl * h.bs * h.Hk * h.hs
    args = [_ptrs(h, q_seq, sq, dt, "q_seq"), _ptrs(h, k_seq, sk, dt, "k_seq"), _ptrs(h, v_seq, sk, dt, "v_seq"),
            _ptrs(h, q_head, hq, dt, "q_head"), _ptrs(h, k_head, hk, dt, "k_head"), _ptrs(h, v_head, hk, dt, "v_head")]
    _check(lib.ulysses_seq_to_head_qkv(h.ptr, *args, _stream(stream)), "ulysses_seq_to_head_qkv")


def ulysses_head_to_seq_qkv(h: UlyssesHandle, q_head, k_head, v_head, q_seq, k_seq, v_seq, stream=None):
    """head->seq of dQ, dK and dV in one launch (three when kv heads are replicated)."""
    dt = h.torch_dtype
    n = h.sl // h.P
    sq, sk = n * h.bs * h.hc * h.hs, n * h.bs * h.hkv * h.hs
    hq, hk = h.sl * h.bs * h.Hq * h.hs, h.sl * h.bs * h.Hk * h.hs
    args = [_ptrs(h, q_head, hq, dt, "q_head"), _ptrs(h, k_head, hk, dt, "k_head"), _ptrs(h, v_head, hk, dt, "v_head"),
            _ptrs(h, q_seq, sq, dt, "q_seq"), _ptrs(h, k_seq, sk, dt, "k_seq"), _ptrs(h, v_seq, sk, dt, "v_seq")]
    _check(lib.ulysses_head_to_seq_qkv(h.ptr, *args, _stream(stream)), "ulysses_head_to_seq_qkv")


def ulysses_attn_fwd(h: UlyssesHandle, q, k, v, o, lse, stream=None):
    dt = h.torch_dtype
    nq = h.sl * h.bs * h.Hq * h.hs
    nk = h.sl * h.bs * h.Hk * h.hs
    args = [_ptrs(h, q, nq, dt, "q"), _ptrs(h, k, nk, dt, "k"), _ptrs(h, v, nk, dt, "v"),
            _ptrs(h, o, nq, dt, "o"), _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse")]
    _check(lib.ulysses_attn_fwd(h.ptr, *args, _stream(stream)), "ulysses_attn_fwd")


def ulysses_attn_bwd(h: UlyssesHandle, q, k, v, o, do, lse, dq, dk, dv, workspace, stream=None):
    dt = h.torch_dtype
    nq = h.sl * h.bs * h.Hq * h.hs
    nk = h.sl * h.bs * h.Hk * h.hs
    ws = _workspace_ptr(h, workspace)
    args = [_ptrs(h, q, nq, dt, "q"), _ptrs(h, k, nk, dt, "k"), _ptrs(h, v, nk, dt, "v"),
            _ptrs(h, o, nq, dt, "o"), _ptrs(h, do, nq, dt, "do"),
            _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse"),
            _ptrs(h, dq, nq, dt, "dq"), _ptrs(h, dk, nk, dt, "dk"), _ptrs(h, dv, nk, dt, "dv")]
    _check(lib.ulysses_attn_bwd(h.ptr, *args, ws, _stream(stream)), "ulysses_attn_bwd")


def _workspace_ptr(h: UlyssesHandle, workspace) -> int:
    if isinstance(workspace, torch.Tensor):
        need = ulysses_workspace_size(h)
        if workspace.device.type != "cuda" or workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace must be a CUDA buffer of at least {need} bytes")
        return workspace.data_ptr()
    return int(workspace)


def ulysses_fused_supported(h: UlyssesHandle) -> bool:
    """True when ulysses_layer_fwd / ulysses_layer_bwd accept this handle."""
    st = int(lib.ulysses_fused_supported(h.ptr))
    if st not in (ULYSSES_OK, ULYSSES_ERR_UNSUPPORTED):
        _check(st, "ulysses_fused_supported")
    return st == ULYSSES_OK


def ulysses_layer_fwd(h: UlyssesHandle, q, k, v, o, lse, stream=None):
    """Forward on sequence shards; both exchanges fused into the attention kernel."""
    dt = h.torch_dtype
    n = h.sl // h.P
    nq = n * h.bs * h.hc * h.hs
    nk = n * h.bs * h.hkv * h.hs
    args = [_ptrs(h, q, nq, dt, "q"), _ptrs(h, k, nk, dt, "k"), _ptrs(h, v, nk, dt, "v"),
            _ptrs(h, o, nq, dt, "o"), _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse")]
    _check(lib.ulysses_layer_fwd(h.ptr, *args, _stream(stream)), "ulysses_layer_fwd")


def ulysses_layer_bwd(h: UlyssesHandle, q, k, v, o, do, lse, dq, dk, dv, workspace, stream=None):
    """Backward on sequence shards; both exchanges fused into the attention kernels."""
    dt = h.torch_dtype
    n = h.sl // h.P
    nq = n * h.bs * h.hc * h.hs
    nk = n * h.bs * h.hkv * h.hs
    ws = _workspace_ptr(h, workspace)
    args = [_ptrs(h, q, nq, dt, "q"), _ptrs(h, k, nk, dt, "k"), _ptrs(h, v, nk, dt, "v"),
            _ptrs(h, o, nq, dt, "o"), _ptrs(h, do, nq, dt, "do"),
            _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse"),
            _ptrs(h, dq, nq, dt, "dq"), _ptrs(h, dk, nk, dt, "dk"), _ptrs(h, dv, nk, dt, "dv")]
    _check(lib.ulysses_layer_bwd(h.ptr, *args, ws, _stream(stream)), "ulysses_layer_bwd")


def _host_ptrs(groups, numels, dtype, name):
    """HOST pointers of the tensors of each group, in order (CPU tensors, contiguous)."""
    flat = []
    for g, (tensors, numel) in enumerate(zip(groups, numels)):
        for r, t in enumerate(tensors):
            if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != dtype or t.numel() != numel:
                raise ValueError(f"{name}[{g}][{r}]: expected a contiguous CPU {dtype} tensor of {numel} elements")
            flat.append(t.data_ptr())
    arr = (_vp * len(flat))(*flat)
    return ctypes.cast(arr, _pp)


def ulysses_host_begin(h: UlyssesHandle, stream=None):
    """The handle's copy streams wait for the work already enqueued on `stream`."""
    _check(lib.ulysses_host_begin(h.ptr, _stream(stream)), "ulysses_host_begin")


def ulysses_host_end(h: UlyssesHandle, stream=None):
    """`stream` waits for every copy of the host steps enqueued so far."""
    _check(lib.ulysses_host_end(h.ptr, _stream(stream)), "ulysses_host_end")


def ulysses_host_step(h: UlyssesHandle, slot: int, host_in, host_out, dev, lse, workspace, stream=None):
    """One fwd+bwd step from host shards to host shards (see the C header).

    host_in: [q, k, v, do] and host_out: [o, dq, dk, dv], each a list of P CPU
    tensors (pinned for overlap). dev: [q, k, v, do, o, dq, dk, dv], each a
    list of P device tensors: the slot's buffers.
    """
    dt = h.torch_dtype
    n = h.sl // h.P
    nq = n * h.bs * h.hc * h.hs
    nk = n * h.bs * h.hkv * h.hs
    sizes_in = [nq, nk, nk, nq]
    sizes_out = [nq, nq, nk, nk]
    hin = _host_ptrs(host_in, sizes_in, dt, "host_in")
    hout = _host_ptrs(host_out, sizes_out, dt, "host_out")
    flat = []
    for g, (tensors, numel) in enumerate(zip(dev, sizes_in + sizes_out)):
        p = _ptrs(h, tensors, numel, dt, f"dev[{g}]")
        flat.extend(p[r] for r in range(h.P))
    darr = (_vp * len(flat))(*flat)
    _check(lib.ulysses_host_step(h.ptr, int(slot), hin, hout, ctypes.cast(darr, _pp),
                                 _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse"),
                                 _workspace_ptr(h, workspace), _stream(stream)), "ulysses_host_step")


def ulysses_get_status(h: UlyssesHandle) -> int:
    return int(lib.ulysses_get_status(h.ptr))


def ulysses_launch_count() -> int:
    return int(lib.ulysses_launch_count())


def ulysses_attn_bwd_noalloc(h: UlyssesHandle, q, k, v, o, do, lse, dq, dk, dv, stream=None):
    """ulysses_attn_bwd on the library's built-in scratch: no workspace argument.

    For callers that may not allocate device memory. See the C header for the
    size limit and for the sharing rules of the built-in scratch.
    """
    dt = h.torch_dtype
    nq = h.sl * h.bs * h.Hq * h.hs
    nk = h.sl * h.bs * h.Hk * h.hs
    args = [_ptrs(h, q, nq, dt, "q"), _ptrs(h, k, nk, dt, "k"), _ptrs(h, v, nk, dt, "v"),
            _ptrs(h, o, nq, dt, "o"), _ptrs(h, do, nq, dt, "do"),
            _ptrs(h, lse, h.bs * h.Hq * h.sl, torch.float32, "lse"),
            _ptrs(h, dq, nq, dt, "dq"), _ptrs(h, dk, nk, dt, "dk"), _ptrs(h, dv, nk, dt, "dv")]
    _check(lib.ulysses_attn_bwd_noalloc(h.ptr, *args, _stream(stream)), "ulysses_attn_bwd_noalloc")


def ulysses_set_wait_limit(h: UlyssesHandle, cycles: int):
    _check(lib.ulysses_set_wait_limit(h.ptr, int(cycles)), "ulysses_set_wait_limit")


def ulysses_inject_fault(h: UlyssesHandle, kind: int):
    _check(lib.ulysses_inject_fault(h.ptr, int(kind)), "ulysses_inject_fault")


def ulysses_timing_enable(h: UlyssesHandle, enable: bool = True):
    """Start (clearing the totals) or stop per-kernel device timing of h."""
    _check(lib.ulysses_timing_enable(h.ptr, 1 if enable else 0), "ulysses_timing_enable")


def ulysses_timing_read(h: UlyssesHandle, kernel: int):
    """(total device ms, launches) of one kernel since timing was enabled; waits for them."""
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(lib.ulysses_timing_read(h.ptr, int(kernel), ctypes.byref(ms), ctypes.byref(n)), "ulysses_timing_read")
    return float(ms.value), int(n.value)
