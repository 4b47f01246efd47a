"""locks_score_select_static: the allocation-free score-and-select.

It serves callers that may not allocate device memory while decoding (for
example an engine whose memory plan is frozen after start-up, or a plugin
that only receives its input and output buffers), using a scratch array
built into the library.  Its selection must equal the selection of the
workspace entry point, on two calls in a row (the second call reuses the
scratch the first one left behind).  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_paged_kv_locks_gb300 import binding as B
from sparse_paged_kv_locks_gb300 import workload as W

pytestmark = pytest.mark.gpu


def _static_fn():
    fn = B.lib().locks_score_select_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + \
        [ctypes.c_void_p] * 3
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    spec = W.custom_spec(batch=3, h_q=8, h_kv=2, ctx=16 * 90 + 7, k=12,
                         steps=2, needles=1, seed=21)
    wl = W.generate(spec, "cpu")
    kc, pt = wl.k_cache.to(dev), wl.page_table.to(dev)
    lens = torch.tensor([16 * 90 + 7, 16 * 41, 16 * 77 + 2],
                        dtype=torch.int32, device=dev)
    batch, max_pages = wl.page_table.shape
    L = lens.cpu().tolist()
    seq = torch.tensor([b for b in range(batch) for _ in range(L[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch) for p in range(L[b] // 16)],
                       dtype=torch.int32, device=dev)
    store = B.new_summary_store(batch, spec.h_kv, max_pages, dev)
    B.locks_build_summaries(kc, pt, seq, pgs, store)
    fn = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for step in range(2):
        q = wl.queries[step].to(dev)
        ws = B.new_workspace(batch, spec.h_q, spec.h_kv, max_pages, spec.k,
                             dev)
        ref = torch.full((batch, spec.h_kv, spec.k), -7, dtype=torch.int32,
                         device=dev)
        B.locks_score_select(q, store, lens, spec.k, ref, ws)
        got = torch.full_like(ref, -7)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        rc = fn(_ptr(q), _ptr(store), _ptr(lens), batch, spec.h_q, spec.h_kv,
                max_pages, spec.k, _ptr(got), _ptr(status), stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and B.locks_read_status(ws) == 0
        assert torch.equal(got, ref), (step, got, ref)


def test_static_scratch_rejects_oversize_requests():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _static_fn()
    fake = ctypes.c_void_p(256)   # never dereferenced: rejected first
    # 64 x 8 heads x 4 x 8192 pages of scores is 64 MiB > 16 MiB
    rc = fn(fake, fake, fake, 64, 32, 8, 8192, 128, fake, None, None)
    assert rc == 2
    assert B.lib().locks_status_string(rc) == b"unsupported size"
