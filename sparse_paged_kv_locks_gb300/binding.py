"""Thin Python binding of liblocks.so (include/locks.h).

Argument marshalling only: every function checks tensor placement, dtype,
shape and contiguity, passes raw pointers and sizes to the C ABI of the same
name, and raises LocksError on a non-zero status.  All compute runs in the
CUDA library; there is no fallback.  Kernels are launched on the current
torch CUDA stream unless `stream` is given.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

PAGE = 16
HEAD_DIM = 128
RANK = 8
RECORD_BYTES = 832

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib",
                        "liblocks.so")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(
    __file__))), "include", "locks.h")

DEV_BAD_PAGE_ID = 0x1
DEV_BAD_INDEX = 0x2
DEV_BAD_SEQ_LEN = 0x4
DEV_BAD_PAIR = 0x8
DEV_TIMEOUT = 0x10

BUILD_VSCALE_PER_PAGE = 0x1   # one basis scale per page (see locks.h)


class LocksError(RuntimeError):
    pass


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "locks_status_string": (ctypes.c_char_p, [_I]),
    "locks_last_cuda_error": (_I, []),
    "locks_kernel_launches": (_I64, []),
    "locks_summary_record_bytes": (_SZ, []),
    "locks_workspace_size": (_I, [_I, _I, _I, _I, _I,
                                  ctypes.POINTER(_SZ)]),
    "locks_build_summaries": (_I, [_P, _I64, _I, _P, _I, _I, _P, _P, _I, _P,
                                   _P, _P, _P, _P]),
    "locks_pack_summaries": (_I, [_P, _P, _P, _I, _P, _P]),
    "locks_pack_summaries_ex": (_I, [_P, _P, _P, _I, _P, _I, _P]),
    "locks_build_summaries_ex": (_I, [_P, _I64, _I, _P, _I, _I, _P, _P, _I,
                                      _P, _P, _P, _I, _P, _P]),
    "locks_append_kv_ex": (_I, [_P, _P, _P, _P, _I64, _I, _P, _I, _I, _P, _P,
                                _P, _I, _P, _P]),
    "locks_score_select": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                _P]),
    "locks_score_pages": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "locks_select_pages": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                _P]),
    "locks_select_pages_merge": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                      _SZ, _P]),
    "locks_variant_record_bytes": (_SZ, [_I, _I]),
    "locks_build_variant": (_I, [_P, _I64, _I, _P, _I, _I, _P, _P, _I, _I, _I,
                                 _P, _P, _P, _P]),
    "locks_score_variant": (_I, [_P, _P, _I, _I, _P, _I, _I, _I, _I, _P, _P,
                                 _P]),
    "locks_exact_page_scores": (_I, [_P, _P, _I64, _P, _P, _I, _I, _I, _I,
                                     _P, _P, _P]),
    "locks_sparse_decode": (_I, [_P, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _I,
                                 _I, _P, _P, _P, _SZ, _P]),
    "locks_append_kv": (_I, [_P, _P, _P, _P, _I64, _I, _P, _I, _I, _P, _P, _P,
                             _P, _P]),
    "locks_decoder_create": (_I, [_P, _P, _I64, _P, _P, _P, _I, _I, _I, _I,
                                  _I, _P, _P, _P, _SZ, ctypes.POINTER(_P)]),
    "locks_decoder_step_host": (_I, [_P, _P, _P, _P,
                                     ctypes.POINTER(ctypes.c_int32), _P]),
    "locks_decoder_last_cuda_error": (_I, [_P]),
    "locks_decoder_destroy": (None, [_P]),
    "locks_clear_status": (_I, [_P, _P]),
    "locks_read_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
}


def lib():
    """Load liblocks.so once; fail loudly when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LocksError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m sparse_paged_kv_locks_gb300.build` (or "
                "__graft_entry__.build()); there is no fallback path")
        import torch.cuda  # noqa: F401  (loads the CUDA runtime first)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions():
    """Names of the functions include/locks.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(locks_[a-z_]+)\s*\(", text)))


def _check(name: str, status: int):
    if status != 0:
        L = lib()
        msg = L.locks_status_string(status).decode()
        raise LocksError(f"{name}: {msg} (status {status}, cuda error "
                         f"{L.locks_last_cuda_error()})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, name, dtype, ndim=None, device="cuda"):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device == "cuda" and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------------------
# sizes and allocation helpers (allocation happens here, in torch, never in
# the library)
# ---------------------------------------------------------------------------
def locks_summary_record_bytes() -> int:
    return int(lib().locks_summary_record_bytes())


def locks_kernel_launches() -> int:
    """Kernels this process has launched through the library so far."""
    return int(lib().locks_kernel_launches())


def locks_workspace_size(batch, h_q, h_kv, max_pages, k) -> int:
    out = _SZ(0)
    _check("locks_workspace_size",
           lib().locks_workspace_size(batch, h_q, h_kv, max_pages, k,
                                      ctypes.byref(out)))
    return int(out.value)


def new_workspace(batch, h_q, h_kv, max_pages, k, device="cuda"):
    n = locks_workspace_size(batch, h_q, h_kv, max_pages, k)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def new_summary_store(batch, h_kv, max_pages, device="cuda"):
    return torch.zeros(batch, h_kv, max_pages, RECORD_BYTES,
                       dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# the C ABI, one function each
# ---------------------------------------------------------------------------
UNQUANTISED_FLOATS = 1296


def locks_build_summaries(k_cache, page_table, seq_ids, page_ids, summaries,
                          tau_out=None, unquantised_out=None, status=None,
                          stream=None, flags=0):
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_ids, "seq_ids", torch.int32, 1)
    _req(page_ids, "page_ids", torch.int32, 1)
    _req(summaries, "summaries", torch.uint8, 4)
    P, h_kv = k_cache.shape[:2]
    batch, max_pages = page_table.shape
    if tuple(k_cache.shape[2:]) != (PAGE, HEAD_DIM):
        raise ValueError("k_cache must be [P][h_kv][16][128]")
    if tuple(summaries.shape) != (batch, h_kv, max_pages, RECORD_BYTES):
        raise ValueError("summaries must be [batch][h_kv][max_pages][832]")
    n = seq_ids.numel()
    if page_ids.numel() != n:
        raise ValueError("seq_ids and page_ids differ in length")
    if tau_out is not None:
        _req(tau_out, "tau_out", torch.float32)
        if tau_out.numel() < n * h_kv:
            raise ValueError("tau_out must hold n_pairs*h_kv floats")
    if unquantised_out is not None:
        _req(unquantised_out, "unquantised_out", torch.float32)
        if unquantised_out.numel() < n * h_kv * UNQUANTISED_FLOATS:
            raise ValueError("unquantised_out must hold n_pairs*h_kv*1296 "
                             "floats")
    if status is not None:
        _req(status, "status", torch.int32)
    _check("locks_build_summaries_ex", lib().locks_build_summaries_ex(
        _ptr(k_cache), P, h_kv, _ptr(page_table), batch, max_pages,
        _ptr(seq_ids), _ptr(page_ids), n, _ptr(summaries), _ptr(tau_out),
        _ptr(unquantised_out), flags, _ptr(status), _stream(stream)))


def locks_pack_summaries(mu, basis, coeffs, records, stream=None, flags=0):
    _req(mu, "mu", torch.float32, 2)
    _req(basis, "basis", torch.float32, 3)
    _req(coeffs, "coeffs", torch.float32, 3)
    _req(records, "records", torch.uint8)
    n = mu.shape[0]
    if tuple(basis.shape) != (n, HEAD_DIM, RANK) or \
            tuple(coeffs.shape) != (n, PAGE, RANK) or mu.shape[1] != HEAD_DIM:
        raise ValueError("mu [n][128], basis [n][128][8], coeffs [n][16][8]")
    if records.numel() < n * RECORD_BYTES:
        raise ValueError("records must hold n*832 bytes")
    _check("locks_pack_summaries_ex", lib().locks_pack_summaries_ex(
        _ptr(mu), _ptr(basis), _ptr(coeffs), n, _ptr(records), flags,
        _stream(stream)))


def locks_score_select(q, summaries, seq_lens, k, idx_out, workspace,
                       stream=None):
    _req(q, "q", torch.bfloat16, 3)
    _req(summaries, "summaries", torch.uint8, 4)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(idx_out, "idx_out", torch.int32, 3)
    _req(workspace, "workspace", torch.uint8, 1)
    batch, h_q, d = q.shape
    _, h_kv, max_pages, rb = summaries.shape
    if d != HEAD_DIM or rb != RECORD_BYTES or summaries.shape[0] != batch:
        raise ValueError("q [batch][h_q][128], summaries [batch][h_kv][P][832]")
    if tuple(idx_out.shape) != (batch, h_kv, k) or seq_lens.numel() != batch:
        raise ValueError("idx_out must be [batch][h_kv][k]")
    _check("locks_score_select", lib().locks_score_select(
        _ptr(q), _ptr(summaries), _ptr(seq_lens), batch, h_q, h_kv,
        max_pages, k, _ptr(idx_out), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def locks_score_pages(q, summaries, seq_lens, scores_out, status=None,
                      stream=None):
    _req(q, "q", torch.bfloat16, 3)
    _req(summaries, "summaries", torch.uint8, 4)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(scores_out, "scores_out", torch.float32, 4)
    batch, h_q, d = q.shape
    _, h_kv, max_pages, rb = summaries.shape
    if d != HEAD_DIM or rb != RECORD_BYTES or summaries.shape[0] != batch:
        raise ValueError("q [batch][h_q][128], summaries [batch][h_kv][P][832]")
    if tuple(scores_out.shape) != (batch, h_kv, h_q // h_kv, max_pages):
        raise ValueError("scores_out must be [batch][h_kv][G][max_pages]")
    if status is not None:
        _req(status, "status", torch.int32)
    _check("locks_score_pages", lib().locks_score_pages(
        _ptr(q), _ptr(summaries), _ptr(seq_lens), batch, h_q, h_kv,
        max_pages, _ptr(scores_out), _ptr(status), _stream(stream)))


def locks_exact_page_scores(q, k_cache, page_table, seq_lens, scores_out,
                            status=None, stream=None):
    """Exact page LSE of every full page (the exact-mass selector's scores),
    same layout as locks_score_pages."""
    _req(q, "q", torch.bfloat16, 3)
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(scores_out, "scores_out", torch.float32, 4)
    batch, h_q, _ = q.shape
    P, h_kv = k_cache.shape[:2]
    max_pages = page_table.shape[1]
    if tuple(scores_out.shape) != (batch, h_kv, h_q // h_kv, max_pages):
        raise ValueError("scores_out must be [batch][h_kv][G][max_pages]")
    _check("locks_exact_page_scores", lib().locks_exact_page_scores(
        _ptr(q), _ptr(k_cache), P, _ptr(page_table), _ptr(seq_lens), batch,
        h_q, h_kv, max_pages, _ptr(scores_out), _ptr(status),
        _stream(stream)))


def locks_variant_record_bytes(rank, vbits) -> int:
    return int(lib().locks_variant_record_bytes(rank, vbits))


def new_variant_store(batch, h_kv, max_pages, rank, vbits, device="cuda"):
    """Zeroed variant-record store [batch][h_kv][max_pages][stride] uint8."""
    stride = locks_variant_record_bytes(rank, vbits)
    if stride == 0:
        raise ValueError(f"unsupported variant rank={rank} vbits={vbits}")
    return torch.zeros(batch, h_kv, max_pages, stride, dtype=torch.uint8,
                       device=device)


def locks_build_variant(k_cache, page_table, seq_ids, page_ids, records,
                        rank, vbits, tau_out=None, status=None, stream=None):
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_ids, "seq_ids", torch.int32, 1)
    _req(page_ids, "page_ids", torch.int32, 1)
    _req(records, "records", torch.uint8, 4)
    P, h_kv = k_cache.shape[:2]
    batch, max_pages = page_table.shape
    if records.shape[3] != locks_variant_record_bytes(rank, vbits):
        raise ValueError("records stride does not match the variant")
    _check("locks_build_variant", lib().locks_build_variant(
        _ptr(k_cache), P, h_kv, _ptr(page_table), batch, max_pages,
        _ptr(seq_ids), _ptr(page_ids), seq_ids.numel(), rank, vbits,
        _ptr(records), _ptr(tau_out), _ptr(status), _stream(stream)))


def locks_score_variant(q, records, rank, vbits, seq_lens, scores_out,
                        status=None, stream=None):
    _req(q, "q", torch.bfloat16, 3)
    _req(records, "records", torch.uint8, 4)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(scores_out, "scores_out", torch.float32, 4)
    batch, h_q, _ = q.shape
    _, h_kv, max_pages, stride = records.shape
    if stride != locks_variant_record_bytes(rank, vbits):
        raise ValueError("records stride does not match the variant")
    _check("locks_score_variant", lib().locks_score_variant(
        _ptr(q), _ptr(records), rank, vbits, _ptr(seq_lens), batch, h_q,
        h_kv, max_pages, _ptr(scores_out), _ptr(status), _stream(stream)))


def locks_select_pages(scores, seq_lens, h_q, k, idx_out, workspace,
                       stream=None):
    _req(scores, "scores", torch.float32, 4)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(idx_out, "idx_out", torch.int32, 3)
    _req(workspace, "workspace", torch.uint8, 1)
    batch, h_kv, G, max_pages = scores.shape
    if G * h_kv != h_q:
        raise ValueError("scores must be [batch][h_kv][h_q/h_kv][max_pages]")
    if tuple(idx_out.shape) != (batch, h_kv, k) or seq_lens.numel() != batch:
        raise ValueError("idx_out must be [batch][h_kv][k]")
    _check("locks_select_pages", lib().locks_select_pages(
        _ptr(scores), _ptr(seq_lens), batch, h_q, h_kv, max_pages, k,
        _ptr(idx_out), _ptr(workspace), workspace.numel(), _stream(stream)))


MERGE_SHARE_AVERAGE, MERGE_GROUP_MAX, MERGE_GROUP_MASS = 0, 1, 2
MERGE_RULES = {"share_average": MERGE_SHARE_AVERAGE,
               "group_max": MERGE_GROUP_MAX, "group_mass": MERGE_GROUP_MASS}


def locks_select_pages_merge(scores, seq_lens, h_q, k, rule, idx_out,
                             workspace, stream=None):
    """locks_select_pages with another GQA merge rule (name or code)."""
    rule = MERGE_RULES.get(rule, rule)
    _req(scores, "scores", torch.float32, 4)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(idx_out, "idx_out", torch.int32, 3)
    _req(workspace, "workspace", torch.uint8, 1)
    batch, h_kv, G, max_pages = scores.shape
    if G * h_kv != h_q:
        raise ValueError("scores must be [batch][h_kv][h_q/h_kv][max_pages]")
    if tuple(idx_out.shape) != (batch, h_kv, k) or seq_lens.numel() != batch:
        raise ValueError("idx_out must be [batch][h_kv][k]")
    _check("locks_select_pages_merge", lib().locks_select_pages_merge(
        _ptr(scores), _ptr(seq_lens), batch, h_q, h_kv, max_pages, k,
        int(rule), _ptr(idx_out), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def locks_sparse_decode(q, k_cache, v_cache, page_table, seq_lens, idx, k,
                        o_out, lse_out, workspace, stream=None):
    _req(q, "q", torch.bfloat16, 3)
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(v_cache, "v_cache", torch.bfloat16, 4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(o_out, "o_out", torch.bfloat16, 3)
    _req(lse_out, "lse_out", torch.float32, 2)
    _req(workspace, "workspace", torch.uint8, 1)
    batch, h_q, _ = q.shape
    P, h_kv = k_cache.shape[:2]
    max_pages = page_table.shape[1]
    if v_cache.shape != k_cache.shape or tuple(o_out.shape) != tuple(q.shape):
        raise ValueError("v_cache like k_cache, o_out like q")
    if idx is not None:
        _req(idx, "idx", torch.int32, 3)
        if tuple(idx.shape) != (batch, h_kv, k):
            raise ValueError("idx must be [batch][h_kv][k]")
    _check("locks_sparse_decode", lib().locks_sparse_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), P, _ptr(page_table),
        _ptr(seq_lens), _ptr(idx), k, batch, h_q, h_kv, max_pages,
        _ptr(o_out), _ptr(lse_out), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def locks_append_kv(k_new, v_new, k_cache, v_cache, page_table, seq_lens,
                    summaries, tau_out=None, status=None, stream=None,
                    flags=0):
    _req(k_new, "k_new", torch.bfloat16, 3)
    _req(v_new, "v_new", torch.bfloat16, 3)
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(v_cache, "v_cache", torch.bfloat16, 4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(summaries, "summaries", torch.uint8, 4)
    P, h_kv = k_cache.shape[:2]
    batch, max_pages = page_table.shape
    if tuple(k_new.shape) != (batch, h_kv, HEAD_DIM):
        raise ValueError("k_new must be [batch][h_kv][128]")
    if tau_out is not None:
        _req(tau_out, "tau_out", torch.float32)
    if status is not None:
        _req(status, "status", torch.int32)
    _check("locks_append_kv_ex", lib().locks_append_kv_ex(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), P, h_kv,
        _ptr(page_table), batch, max_pages, _ptr(seq_lens), _ptr(summaries),
        _ptr(tau_out), flags, _ptr(status), _stream(stream)))


def locks_clear_status(status_word, stream=None):
    _check("locks_clear_status",
           lib().locks_clear_status(_ptr(status_word), _stream(stream)))


def locks_read_status(status_word, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("locks_read_status", lib().locks_read_status(
        _ptr(status_word), ctypes.byref(out), _stream(stream)))
    return int(out.value)


# ---------------------------------------------------------------------------
# a decode step for one layer: score + select + sparse attention
# ---------------------------------------------------------------------------
class LocksDecoder:
    """Owns the per-step buffers of one layer's decode step.

    With graph=True, `step` captures the device-resident step (score +
    select + sparse attention, five kernels) once into a CUDA graph and
    replays it, and `step_host` runs the C ABI decoder object
    (locks_decoder_step_host): the query copy in, the kernels and the
    copies of (o, lse) out replay as one CUDA graph per step.  With
    graph=False both run the kernels eagerly.  `seq_lens`, when given, is
    the device length buffer the step reads (it is bound, so appends that
    update it in place take effect); otherwise the decoder keeps its own
    and copies the lengths passed to each step into it.  The library
    allocates no device memory and the eager step never synchronises.

    With append=True every `step` first appends one token per sequence
    (k_new, v_new [batch][h_kv][128]) at the current length and builds the
    summary of a page that this fills (locks_append_kv, the notes' §2
    Fig. 1 build step), then decodes with the lengths it has grown; with
    graph=True the append, with its page build, is part of the one graph."""

    def __init__(self, k_cache, v_cache, page_table, summaries, h_q, k,
                 graph=False, seq_lens=None, append=False):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.page_table, self.summaries = page_table, summaries
        self.batch, self.h_kv, self.max_pages = summaries.shape[:3]
        self.h_q, self.k = h_q, k
        dev = k_cache.device
        self.workspace = new_workspace(self.batch, h_q, self.h_kv,
                                       self.max_pages, k, dev)
        self.idx = torch.empty(self.batch, self.h_kv, k, dtype=torch.int32,
                               device=dev)
        self.o = torch.empty(self.batch, h_q, HEAD_DIM, dtype=torch.bfloat16,
                             device=dev)
        self.lse = torch.empty(self.batch, h_q, dtype=torch.float32,
                               device=dev)
        self.q_dev = torch.empty(self.batch, h_q, HEAD_DIM,
                                 dtype=torch.bfloat16, device=dev)
        if seq_lens is None:
            self.seq_lens_dev = torch.empty(self.batch, dtype=torch.int32,
                                            device=dev)
        else:
            _req(seq_lens, "seq_lens", torch.int32, 1)
            if seq_lens.numel() != self.batch:
                raise ValueError("seq_lens must have one entry per sequence")
            self.seq_lens_dev = seq_lens
        self.append = append
        if append:
            self.k_new = torch.empty(self.batch, self.h_kv, HEAD_DIM,
                                     dtype=torch.bfloat16, device=dev)
            self.v_new = torch.empty_like(self.k_new)
        self.use_graph = graph
        self._graph = None
        self._native = None
        self._out = None
        self._stream_arg = None
        self._st = ctypes.c_int32(0)
        self._st_ref = ctypes.byref(self._st)
        self._step_fn = lib().locks_decoder_step_host

    def _eager(self, q, seq_lens, stream=None, k_new=None, v_new=None):
        if self.append:
            locks_append_kv(k_new, v_new, self.k_cache, self.v_cache,
                            self.page_table, seq_lens, self.summaries,
                            status=self.workspace[:4].view(torch.int32),
                            stream=stream)
        locks_score_select(q, self.summaries, seq_lens, self.k, self.idx,
                           self.workspace, stream)
        locks_sparse_decode(q, self.k_cache, self.v_cache, self.page_table,
                            seq_lens, self.idx, self.k, self.o, self.lse,
                            self.workspace, stream)

    def _capture(self):
        cur = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):   # one-time setup outside the capture
            self._eager(self.q_dev, self.seq_lens_dev, None, self.k_new_b,
                        self.v_new_b)
            if self.append:
                # the warm-up appended this step's token; the replay that
                # follows writes it (and any page build) again at the same
                # position, so the lengths go back by one
                self.seq_lens_dev.sub_(1)
        cur.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._eager(self.q_dev, self.seq_lens_dev, None, self.k_new_b,
                        self.v_new_b)
        self._graph = g

    @property
    def k_new_b(self):
        return self.k_new if self.append else None

    @property
    def v_new_b(self):
        return self.v_new if self.append else None

    def _bind_lens(self, seq_lens, stream=None):
        if seq_lens is not None and seq_lens is not self.seq_lens_dev:
            _req(seq_lens, "seq_lens", torch.int32, 1)
            s = torch.cuda.current_stream() if stream is None else stream
            with torch.cuda.stream(s):
                self.seq_lens_dev.copy_(seq_lens, non_blocking=True)

    def step(self, q, seq_lens=None, stream=None, k_new=None, v_new=None):
        """Device-resident query -> (o, lse) on the device (append mode:
        after appending k_new, v_new)."""
        if self.append:
            if k_new is None or v_new is None:
                raise ValueError("an appending decoder needs k_new and v_new")
            _req(k_new, "k_new", torch.bfloat16, 3)
            _req(v_new, "v_new", torch.bfloat16, 3)
            if tuple(k_new.shape) != tuple(self.k_new.shape) or \
                    tuple(v_new.shape) != tuple(self.k_new.shape):
                raise ValueError("k_new, v_new must be [batch][h_kv][128]")
        if not self.use_graph:
            self._eager(q, self.seq_lens_dev if seq_lens is None else seq_lens,
                        stream, k_new, v_new)
            return self.o, self.lse
        if stream is not None:
            raise ValueError("graph replay runs on the current stream")
        if q is not self.q_dev:
            self.q_dev.copy_(q, non_blocking=True)
        if self.append:
            if k_new is not self.k_new:
                self.k_new.copy_(k_new, non_blocking=True)
            if v_new is not self.v_new:
                self.v_new.copy_(v_new, non_blocking=True)
        self._bind_lens(seq_lens)
        if self._graph is None:
            self._capture()
        self._graph.replay()
        return self.o, self.lse

    def handle(self):
        """The C ABI decoder object (a locks_decoder_t *, as a ctypes
        pointer) bound to this decoder's device buffers, for callers that
        drive locks_decoder_step_host directly; owned by this object."""
        return self._native_decoder()

    def _native_decoder(self):
        if self._native is None:
            h = ctypes.c_void_p(None)
            L = lib()
            _check("locks_decoder_create", L.locks_decoder_create(
                _ptr(self.k_cache), _ptr(self.v_cache), self.k_cache.shape[0],
                _ptr(self.page_table), _ptr(self.summaries),
                _ptr(self.seq_lens_dev), self.batch, self.h_q, self.h_kv,
                self.max_pages, self.k, _ptr(self.q_dev), _ptr(self.idx),
                _ptr(self.workspace), self.workspace.numel(),
                ctypes.byref(h)))
            self._native = h
        return self._native

    def step_host(self, q_host, seq_lens, o_host, lse_host, stream=None):
        """Pinned host query in, pinned host (o, lse) out (synchronises).
        Returns (o_host, lse_host, device status word).

        With graph=True the output buffers are checked once per distinct
        pair and the query with a few attribute reads per call, so that the
        per-step host cost stays small (the C call checks that every buffer
        is page-locked)."""
        if not self.use_graph:
            self._check_host(q_host, o_host, lse_host)
            s = torch.cuda.current_stream() if stream is None else stream
            with torch.cuda.stream(s):
                self.q_dev.copy_(q_host, non_blocking=True)
                self._bind_lens(seq_lens, s)
                self._eager(self.q_dev, self.seq_lens_dev, s)
                o_host.copy_(self.o, non_blocking=True)
                lse_host.copy_(self.lse, non_blocking=True)
            s.synchronize()
            return o_host, lse_host, self.status()
        out = self._out
        if out is None or out[0] is not o_host or out[1] is not lse_host:
            self._check_host(q_host, o_host, lse_host)
            out = self._out = (o_host, lse_host,
                               ctypes.c_void_p(o_host.data_ptr()),
                               ctypes.c_void_p(lse_host.data_ptr()))
        elif (q_host.dtype is not torch.bfloat16 or q_host.is_cuda or
              q_host.shape != self.q_dev.shape or
              not q_host.is_contiguous()):
            raise ValueError("q_host must be a contiguous bf16 host tensor "
                             "[batch][h_q][128]")
        if seq_lens is not None and seq_lens is not self.seq_lens_dev:
            self._bind_lens(seq_lens, stream)
        st = self._st
        sc = self._stream_arg
        if sc is None or sc[0] is not stream:
            sc = self._stream_arg = (stream, _stream(stream)) \
                if stream is not None else (None, None)
        rc = self._step_fn(self._native_decoder(),
                           ctypes.c_void_p(q_host.data_ptr()), out[2], out[3],
                           self._st_ref,
                           sc[1] if stream is not None else _stream(None))
        if rc != 0:
            L = lib()
            raise LocksError(
                f"locks_decoder_step_host: "
                f"{L.locks_status_string(rc).decode()} (status {rc}, cuda "
                f"error {L.locks_decoder_last_cuda_error(self._native)})")
        return o_host, lse_host, int(st.value)

    def _check_host(self, q_host, o_host, lse_host):
        for t, name, dt in ((q_host, "q_host", torch.bfloat16),
                            (o_host, "o_host", torch.bfloat16),
                            (lse_host, "lse_host", torch.float32)):
            _req(t, name, dt, device="host")
            if t.is_cuda:
                raise ValueError(f"{name} must be a (pinned) host tensor")
        if tuple(q_host.shape) != (self.batch, self.h_q, HEAD_DIM) or \
                tuple(o_host.shape) != tuple(q_host.shape) or \
                tuple(lse_host.shape) != (self.batch, self.h_q):
            raise ValueError("host buffers must be [batch][h_q][128] and "
                             "[batch][h_q]")

    def close(self):
        if self._native is not None:
            lib().locks_decoder_destroy(self._native)
            self._native = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def status(self) -> int:
        return locks_read_status(self.workspace)
