"""Parity at the 128K-context bench workload (batch 32, 32q/8kv, k=128), in
the launch configuration bench.py times, on sampled outputs.

The full-batch GPU build is checked first: for sampled (sequence, KV head)
pairs its records are compared with the oracle's build of the same keys
(tests/build_parity.py).  Then the oracle's own records of those pairs
replace the GPU-built ones in the full store, and the full-batch kernels
run.  Scores and selections of
the sampled pairs must match the oracle's exactly as on small cases; the
attention outputs of the sampled pairs are checked with the oracle's
selection fed to the full-batch decode.
"""
import numpy as np
import pytest
import torch

from build_parity import check_full_size_build
from oracle import locks_oracle as O
from sparse_paged_kv_locks_gb300 import binding as B
from sparse_paged_kv_locks_gb300 import workload as W

pytestmark = pytest.mark.gpu


def test_full_size_sampled_parity():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    spec = W.SPECS["llama8b_128k"]
    wl = W.generate(spec, dev, steps=2)
    lens = [int(x) for x in wl.seq_lens]
    batch, max_pages = wl.page_table.shape
    h_kv, G, k = spec.h_kv, spec.group, spec.k
    seq = torch.tensor([b for b in range(batch) for _ in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch) for p in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    store = B.new_summary_store(batch, h_kv, max_pages, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store,
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    samples = [(0, 0), (13, 5), (31, 7)]
    stats = check_full_size_build(B, wl, store, samples, dev, "llama8b_128k")
    for st in stats.values():
        assert st["sub_ok"] > 0.8 and st["full"] > 0.5, st
    q = wl.queries[1]
    qn = q.float().cpu().numpy()
    orc = {}
    for b, h in samples:
        nf = lens[b] // 16
        phys = wl.page_table[b, :nf].long()
        keys = wl.k_cache[phys, h].float().cpu().numpy()       # [nf][16][128]
        q8, _ = O.build_page(keys)
        rec = O.encode_records(q8)                              # [nf][832]
        store[b, h, :nf] = torch.from_numpy(rec).to(dev)
        mu, V, C = O.dequantize(q8)
        s_hat = O.score_from_summaries(qn[b, h * G:(h + 1) * G], mu, V, C)
        orc[(b, h)] = (s_hat, O.select_one(s_hat, lens[b], k))
    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages, k, dev)
    idx = torch.empty(batch, h_kv, k, dtype=torch.int32, device=dev)
    B.locks_score_select(q, store, wl.seq_lens, k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    n = batch * h_kv * G * max_pages
    s_gpu = ws[256:256 + 4 * n].view(torch.float32).view(
        batch, h_kv, G, max_pages)
    ig = idx.cpu().numpy()
    for (b, h), (s_hat, sel) in orc.items():
        nf = lens[b] // 16
        d = np.abs(s_gpu[b, h, :, :nf].cpu().numpy() - s_hat).max()
        assert d <= 1e-3, (b, h, d)
        got = sorted(int(x) for x in ig[b, h] if x >= 0)
        if got != sel:
            lm = np.log(O.share_average(s_hat, nf))
            cand = np.arange(1, nf - 1)
            order = cand[np.lexsort((cand, -lm[cand]))]
            edge = lm[order[k - 3]]
            for p in set(got) ^ set(sel):
                assert abs(lm[p] - edge) <= 1e-3, (b, h, p)
    # attention in the bench configuration with the oracle's selections
    for (b, h), (_, sel) in orc.items():
        idx[b, h] = torch.tensor(sel + [-1] * (k - len(sel)), dtype=torch.int32)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=dev)
    B.locks_sparse_decode(q, wl.k_cache, wl.v_cache, wl.page_table,
                          wl.seq_lens, idx, k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    for (b, h), (_, sel) in orc.items():
        phys = wl.page_table[b, sel].long()
        K = wl.k_cache[phys, h].float().cpu().numpy().reshape(-1, 128)
        V = wl.v_cache[phys, h].float().cpu().numpy().reshape(-1, 128)
        o_ref, lse_ref = O.attend(qn[b, h * G:(h + 1) * G], K, V)
        og = o[b, h * G:(h + 1) * G].float().cpu().numpy()
        assert np.abs(og - o_ref).max() <= 2e-2 * np.abs(o_ref).max()
        assert np.abs(lse[b, h * G:(h + 1) * G].cpu().numpy() - lse_ref).max() \
            <= 1e-3
