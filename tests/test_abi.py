"""The C ABI library loads, exports every declared symbol and validates
arguments on the host (no GPU needed: nothing here launches a kernel)."""
import ctypes
import os

import pytest

from sparse_paged_kv_locks_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(B.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return B.lib()


def test_exports_every_declared_function(L):
    names = B.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n


def test_record_and_status_strings(L):
    assert B.locks_summary_record_bytes() == 832
    # rejected calls launch nothing
    n0 = B.locks_kernel_launches()
    assert n0 >= 0
    assert L.locks_score_select(None, None, None, 1, 8, 2, 16, 4, None, None,
                                0, None) == 1
    assert B.locks_kernel_launches() == n0
    assert L.locks_status_string(0) == b"ok"
    assert L.locks_status_string(3) == b"workspace too small"
    assert L.locks_last_cuda_error() == 0


def test_workspace_size_rules(L):
    # 256-byte header + max(score region, split-K region)
    a = B.locks_workspace_size(32, 32, 8, 8192, 128)
    assert a == 256 + 32 * 8 * 4 * 8192 * 4 + 32 * 8 * 8192 * 4
    b = B.locks_workspace_size(1, 8, 2, 256, 16)
    assert b >= 256 + 2 * 4 * 256 * 4
    out = ctypes.c_size_t(0)
    assert L.locks_workspace_size(1, 7, 2, 10, 4, ctypes.byref(out)) == 1
    assert L.locks_workspace_size(1, 34, 2, 10, 4, ctypes.byref(out)) == 2
    assert L.locks_workspace_size(1, 8, 2, 0, 4, ctypes.byref(out)) == 1


def test_host_validation_before_launch(L):
    s = None
    # score_select: k < 2, bad heads, null pointers, small workspace
    assert L.locks_score_select(None, None, None, 1, 8, 2, 16, 1, None, None,
                                0, s) == 1
    assert L.locks_score_select(None, None, None, 1, 7, 2, 16, 4, None, None,
                                0, s) == 1
    assert L.locks_score_select(None, None, None, 1, 8, 2, 16, 4, None, None,
                                0, s) == 1
    fake = ctypes.c_void_p(16)   # never dereferenced: rejected first
    assert L.locks_score_select(fake, fake, fake, 1, 8, 2, 16, 4, fake, fake,
                                8, s) == 3
    assert L.locks_score_select(fake, fake, fake, 1, 64, 2, 16, 4, fake, fake,
                                1 << 30, s) == 2
    # sparse_decode
    assert L.locks_sparse_decode(fake, fake, fake, 0, fake, fake, fake, 4, 1,
                                 8, 2, 16, fake, fake, fake, 1 << 20, s) == 1
    assert L.locks_sparse_decode(fake, fake, fake, 10, fake, fake, fake, 4, 1,
                                 8, 2, 16, fake, fake, fake, 16, s) == 3
    # build / append / pack / status
    assert L.locks_build_summaries(None, 10, 2, None, 1, 16, None, None, 3,
                                   None, None, None, None, s) == 1
    assert L.locks_build_summaries(None, 10, 2, None, 1, 16, None, None, 0,
                                   None, None, None, None, s) == 0
    assert L.locks_append_kv(fake, fake, fake, fake, 10, 33, fake, 1, 16,
                             fake, fake, None, None, s) == 2
    assert L.locks_pack_summaries(None, None, None, -1, None, s) == 1
    # variant scoring: unsupported (rank, bits), records not 16-byte aligned
    assert L.locks_score_variant(fake, fake, 7, 4, fake, 1, 8, 2, 16, fake,
                                 None, s) == 1
    assert L.locks_score_variant(fake, ctypes.c_void_p(24), 8, 4, fake, 1, 8,
                                 2, 16, fake, None, s) == 1
    assert L.locks_clear_status(None, s) == 1
    assert L.locks_read_status(None, None, s) == 1
    # decoder object: argument and workspace checks before any CUDA call
    out = ctypes.c_void_p(123)
    args = [fake, fake, 10, fake, fake, fake, 2, 8, 2, 16, 4, fake, fake,
            fake]
    assert L.locks_decoder_create(*args, 1 << 30, None) == 1
    assert L.locks_decoder_create(*args, 64, ctypes.byref(out)) == 3
    assert out.value is None
    bad = list(args)
    bad[10] = 1                      # k < 2
    assert L.locks_decoder_create(*bad, 1 << 30, ctypes.byref(out)) == 1
    bad = list(args)
    bad[7] = 7                       # h_q not a multiple of h_kv
    assert L.locks_decoder_create(*bad, 1 << 30, ctypes.byref(out)) == 1
    assert L.locks_decoder_step_host(None, fake, fake, fake, None, s) == 1
    assert L.locks_decoder_last_cuda_error(None) == 0
    L.locks_decoder_destroy(None)
    # batch limits (per-sequence tables on chip): refused above them, the
    # argument checks go on below them (here: the workspace is too small)
    assert L.locks_score_select(fake, fake, fake, 1595, 8, 2, 16, 4, fake,
                                fake, 64, s) == 2
    assert L.locks_score_select(fake, fake, fake, 1594, 8, 2, 16, 4, fake,
                                fake, 64, s) == 3
    assert L.locks_sparse_decode(fake, fake, fake, 10, fake, fake, fake, 4,
                                 41713, 8, 2, 16, fake, fake, fake, 64, s) == 2
    assert L.locks_sparse_decode(fake, fake, fake, 10, fake, fake, fake, 4,
                                 41712, 8, 2, 16, fake, fake, fake, 64, s) == 3
    # empty batches launch nothing and succeed
    assert L.locks_score_select(None, None, None, 0, 8, 2, 16, 4, None, None,
                                0, s) == 0


def test_binding_refuses_cpu_tensors(L):
    import torch
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        B.locks_score_select(q, torch.zeros(1, 2, 16, 832, dtype=torch.uint8),
                             torch.zeros(1, dtype=torch.int32), 4,
                             torch.zeros(1, 2, 4, dtype=torch.int32),
                             torch.zeros(10, dtype=torch.uint8))
