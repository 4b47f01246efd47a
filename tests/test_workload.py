"""The seeded generator draws what the workloads state (CPU only)."""
import numpy as np
import torch

from sparse_paged_kv_locks_gb300 import workload as W


def test_tiny_workload_shapes_and_needles():
    spec = W.SPECS["tiny_4k"]
    wl = W.generate(spec, "cpu")
    assert wl.k_cache.shape == (256, 2, 16, 128)
    assert wl.k_cache.dtype == torch.bfloat16
    assert wl.page_table.shape == (1, 256)
    assert (wl.page_table[0] == torch.arange(256, dtype=torch.int32)).all()
    assert wl.queries.shape == (8, 1, 8, 128)
    # every query head of a group is at cosine 0.6 with its needle direction
    q = wl.queries.float()
    for h in range(2):
        nd = wl.needle_dirs[0, h, 0]
        for g in range(4):
            c = (q[:, 0, h * 4 + g] @ nd) / q[:, 0, h * 4 + g].norm(dim=-1)
            assert torch.allclose(c, torch.full_like(c, 0.6), atol=1e-2)
        # the needle key points along the needle direction
        p = int(wl.needle_pages[0, h, 0])
        keys = wl.k_cache[int(wl.page_table[0, p]), h].float()
        cos = (keys @ nd) / keys.norm(dim=-1)
        assert cos.max() > 0.99
    # same seed, same draw
    wl2 = W.generate(spec, "cpu")
    assert torch.equal(wl.k_cache, wl2.k_cache)


def test_planted_spectrum():
    g = torch.Generator().manual_seed(0)
    rho = torch.full((4,), 0.6)
    keys = W.page_keys(g, 4, rho, "cpu").double()
    D = keys - keys.mean(dim=1, keepdim=True)
    sv = torch.linalg.svdvals(D)
    # leading squared singular values are s_m^2 = (4*0.6^m)^2 plus the noise
    # energy per direction (16x128 noise at 0.05: squared values 0.18..0.6)
    for m in range(3):
        excess = sv[:, m] ** 2 - (4 * 0.6 ** m) ** 2
        assert float(excess.min()) > -0.5 and float(excess.max()) < 1.0


def test_ragged_lengths_and_table():
    spec = W.SPECS["ragged_64"]
    lens = W.seq_lengths(spec)
    assert len(lens) == 64 and all(4096 <= L <= 131072 for L in lens)
    assert all(L % 16 for L in lens)


def test_append_workload_small():
    spec = W.custom_spec(batch=2, h_q=4, h_kv=2, ctx=64, k=4, steps=20,
                         needles=0, append_steps=20)
    wl = W.generate(spec, "cpu")
    assert wl.k_append.shape == (20, 2, 2, 128)
    # appended positions are empty in the cache until appended
    for b in range(2):
        for s in range(20):
            pos = 64 + s
            pid = int(wl.page_table[b, pos // 16])
            assert (wl.k_cache[pid, :, pos % 16] == 0).all()
        assert wl.k_append[:, b].abs().sum() > 0
