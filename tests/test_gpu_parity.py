"""GPU parity: every step of the CUDA path against the float64 oracle.

Tolerances of the LOCKS decode path against the float64 oracle:
  * quantised bytes: bit-exact where both sides quantise the same fp32
    values (the pack entry point, the centroid); after the eigensolver,
    codes may differ by one step only inside the window that the measured
    fp32 eigensolver error carries through the scale (tests/build_parity.py),
    up to eigenvector sign
  * reconstructions C V^T (fp32, before quantisation): relative Frobenius
    error <= 1e-3, up to sign, on pages whose kept spectrum is separated
  * page scores from the same records: absolute error <= 1e-3
  * selections: identical except pages whose oracle log share-average lies
    within 1e-3 of the k-th boundary's
  * attention: max |o - o_ref| <= 2e-2 * max |o_ref|; |lse - lse_ref| <= 1e-3
Inputs flow only oracle -> GPU (records, indices), never the other way.
"""
import math

import numpy as np
import pytest
import torch

from build_parity import check_build
from oracle import locks_oracle as O
from sparse_paged_kv_locks_gb300 import binding as B
from sparse_paged_kv_locks_gb300 import workload as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
S_TOL = 1e-3
O_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def full_pairs(lens):
    seq, pg = [], []
    for b, L in enumerate(lens):
        for p in range(int(L) // 16):
            seq.append(b)
            pg.append(p)
    return np.array(seq, np.int32), np.array(pg, np.int32)


def i32(x):
    return torch.as_tensor(np.asarray(x), dtype=torch.int32, device=DEV)


def gpu_build(wl_dev, lens, want_unq=False, flags=0):
    seq, pg = full_pairs(lens)
    batch, max_pages = wl_dev.page_table.shape
    h_kv = wl_dev.k_cache.shape[1]
    store = B.new_summary_store(batch, h_kv, max_pages, DEV)
    tau = torch.zeros(len(seq) * h_kv, dtype=torch.float32, device=DEV)
    unq = torch.zeros(len(seq) * h_kv * B.UNQUANTISED_FLOATS,
                      dtype=torch.float32, device=DEV) if want_unq else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_build_summaries(wl_dev.k_cache, wl_dev.page_table, i32(seq),
                            i32(pg), store, tau, unq, status, flags=flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return store, tau, unq, seq, pg


class Dev:
    """A workload moved to the GPU."""

    def __init__(self, wl):
        self.k_cache = wl.k_cache.to(DEV)
        self.v_cache = wl.v_cache.to(DEV)
        self.page_table = wl.page_table.to(DEV)
        self.seq_lens = wl.seq_lens.to(DEV)
        self.queries = wl.queries.to(DEV)


def host(wl):
    return (wl.k_cache.float().numpy(), wl.v_cache.float().numpy(),
            wl.page_table.numpy(), [int(x) for x in wl.seq_lens])


def s_hat_from_ws(ws, batch, h_kv, G, max_pages):
    n = batch * h_kv * G * max_pages
    return ws[256:256 + 4 * n].view(torch.float32).view(
        batch, h_kv, G, max_pages).cpu().numpy()


def log_share_average(s_hat_bh, L):
    nf = L // 16
    return np.log(O.share_average(s_hat_bh, nf))


def selection_agrees(idx_gpu, idx_orc, s_hat_bh, L, k, window):
    """Sets equal except pages whose oracle log share-average lies within
    `window` of the (k-2)-th candidate's."""
    a = set(int(x) for x in idx_gpu if x >= 0)
    b = set(int(x) for x in idx_orc if x >= 0)
    if a == b:
        return True, 0
    n = -(-L // 16)
    lm = log_share_average(s_hat_bh, L)
    cand = np.arange(1, n - 1)
    order = cand[np.lexsort((cand, -lm[cand]))]
    boundary = lm[order[k - 3]]
    for p in a ^ b:
        if p in (0, n - 1) or abs(lm[p] - boundary) > window:
            return False, len(a ^ b)
    return True, len(a ^ b)


# ---------------------------------------------------------------------------
# quantiser and record layout: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("vscale", ["column", "page"])
def test_pack_is_bit_exact(vscale):
    rng = np.random.default_rng(0)
    n = 300
    mu = rng.normal(0, 0.5, (n, 128)).astype(np.float32)
    V = np.linalg.qr(rng.normal(size=(n, 128, 8)))[0].astype(np.float32)
    C = (rng.normal(size=(n, 16, 8)) * 3).astype(np.float32)
    # edge cases: zero column / row / centroid, tiny values, saturation,
    # exact half-way codes (scale 0.0625 with values k.5 * scale)
    V[0, :, 3] = 0.0
    C[1, 5, :] = 0.0
    mu[2, :] = 0.0
    V[3] *= 1e-30
    C[4] *= 1e9
    V[5, :, 0] = 0.0
    V[5, 0, 0] = 7 * 0.0625
    V[5, 1:8, 0] = np.array([3.5, 2.5, -2.5, -3.5, 0.5, -0.5, 1.5]) * 0.0625
    q = O.quantize_summary(mu, V, C, vscale)
    expect = O.encode_records(q)
    rec = torch.zeros(n * 832, dtype=torch.uint8, device=DEV)
    B.locks_pack_summaries(torch.from_numpy(mu).to(DEV),
                           torch.from_numpy(V).to(DEV),
                           torch.from_numpy(C).to(DEV), rec,
                           flags=B.BUILD_VSCALE_PER_PAGE if vscale == "page"
                           else 0)
    got = rec.view(n, 832).cpu().numpy()
    bad = np.nonzero((got != expect).any(axis=1))[0]
    assert bad.size == 0, f"records differ: {bad[:10]}"


# ---------------------------------------------------------------------------
# build (Algorithm 1)
# ---------------------------------------------------------------------------
def _degenerate_workload():
    spec = W.custom_spec(batch=2, h_q=4, h_kv=2, ctx=16 * 24, k=6, needles=0,
                         seed=5)
    wl = W.generate(spec, "cpu")
    kc = wl.k_cache
    pt = wl.page_table
    # page 3 of seq 0: 16 identical keys (D = 0); page 4: exact rank 2 with
    # small integers, so bf16 holds it exactly and the centring is exact
    p3 = int(pt[0, 3])
    kc[p3] = kc[p3, :, :1].clone().expand(-1, 16, -1)
    p4 = int(pt[0, 4])
    g = torch.Generator().manual_seed(3)
    base = torch.randint(-4, 5, (2, 1, 128), generator=g).float()
    dirs = torch.randint(-1, 2, (2, 2, 128), generator=g).float()
    coef = torch.randint(-3, 4, (2, 16, 2), generator=g).float()
    kc[p4] = (base + coef @ dirs).to(torch.bfloat16)
    return wl


def _ragged_decay_workload():
    """Small pages with the ragged workload's spectra: per-page decay
    rho ~ U(0.4, 0.8), so the kept spectrum reaches the noise floor and
    near-degenerate tails occur."""
    spec = W.custom_spec(batch=3, h_q=8, h_kv=2, ctx=16 * 300 + 5, k=8,
                         steps=4, needles=1, seed=41, decay_range=(0.4, 0.8),
                         ragged_min=16 * 120)
    return W.generate(spec, "cpu")


@pytest.mark.parametrize("which", ["tiny_4k", "degenerate", "ragged_decay"])
def test_build_matches_oracle(which):
    wl = {"tiny_4k": lambda: W.generate(W.SPECS["tiny_4k"], "cpu"),
          "degenerate": _degenerate_workload,
          "ragged_decay": _ragged_decay_workload}[which]()
    d = Dev(wl)
    kc, vc, pt, lens = host(wl)
    store, tau, unq, seq, pg = gpu_build(d, lens, want_unq=True)
    h_kv = kc.shape[1]
    n = len(seq) * h_kv
    keys = kc[pt[seq, pg]].reshape(n, 16, 128)
    got = store.cpu().numpy()[seq, :, pg].reshape(n, 832)
    stats = check_build(got, unq.view(n, -1).cpu().numpy(),
                        tau.cpu().numpy(), keys, which)
    if which != "degenerate":
        assert stats["sub_ok"] > 0.8 and stats["full"] > 0.5, stats
    else:
        assert stats["sub_ok"] > 0


def test_build_per_page_basis_scale():
    """LOCKS_BUILD_VSCALE_PER_PAGE: the records are the oracle's per-page
    quantiser applied to the build's own fp32 values (bit for bit), and the
    eigensolve, coefficients and centroid are those of the default build."""
    wl = W.generate(W.SPECS["tiny_4k"], "cpu")
    d = Dev(wl)
    _, _, _, lens = host(wl)
    col, _, unq_c, seq, pg = gpu_build(d, lens, want_unq=True)
    page, _, unq_p, _, _ = gpu_build(d, lens, want_unq=True,
                                     flags=B.BUILD_VSCALE_PER_PAGE)
    assert torch.equal(unq_c, unq_p)
    h_kv = d.k_cache.shape[1]
    u = unq_p.view(len(seq), h_kv, -1).cpu().numpy()
    q = O.quantize_summary(u[..., 16:144], u[..., 144:1168].reshape(
        len(seq), h_kv, 128, 8), u[..., 1168:].reshape(len(seq), h_kv, 16, 8),
        vscale="page")
    got = page.cpu().numpy()[seq, :, pg]
    assert np.array_equal(got, O.encode_records(q))
    gq = O.decode_records(got)
    assert (gq["sV"] == gq["sV"][..., :1]).all()
    cq = O.decode_records(col.cpu().numpy()[seq, :, pg])
    assert (cq["C8"] == gq["C8"]).all() and (cq["mu8"] == gq["mu8"]).all()
    assert (gq["sV"][..., 0] == cq["sV"].max(axis=-1)).all()


# ---------------------------------------------------------------------------
# score (Eq.(4)) from identical records
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("vscale", ["column", "page"])
@pytest.mark.parametrize("G,h_kv", [(4, 2), (1, 4), (8, 1), (16, 1), (5, 2)])
def test_score_matches_oracle_on_same_records(G, h_kv, vscale):
    spec = W.custom_spec(batch=3, h_q=G * h_kv, h_kv=h_kv, ctx=16 * 70 + 9,
                         k=10, needles=0, seed=20 + G)
    wl = W.generate(spec, "cpu")
    kc, vc, pt, lens = host(wl)
    lens = [16 * 70 + 9, 16 * 3, 16 * 45 + 1]
    batch, max_pages = pt.shape
    seq, pg = full_pairs(lens)
    store, _ = O.build_summaries(kc, pt, seq, pg, batch, max_pages,
                                 vscale=vscale)
    q = wl.queries[0].float().numpy()
    s_orc = O.score_store(q, store, lens)
    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages, spec.k, DEV)
    idx = torch.zeros(batch, h_kv, spec.k, dtype=torch.int32, device=DEV)
    B.locks_score_select(wl.queries[0].to(DEV), torch.from_numpy(store).to(DEV),
                         i32(lens), spec.k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    s_gpu = s_hat_from_ws(ws, batch, h_kv, G, max_pages)
    for b in range(batch):
        nf = lens[b] // 16
        d = np.abs(s_gpu[b, :, :, :nf] - s_orc[b, :, :, :nf])
        assert d.max(initial=0) <= S_TOL, (b, float(d.max()))
    idx_o = O.select_store(s_orc, lens, spec.k)
    ig = idx.cpu().numpy()
    for b in range(batch):
        for h in range(h_kv):
            ok, _ = selection_agrees(ig[b, h], idx_o[b, h], s_orc[b, h],
                                     lens[b], spec.k, 1e-3)
            assert ok, (b, h, ig[b, h], idx_o[b, h])


@pytest.mark.parametrize("G,h_kv", [(4, 2), (16, 1)])
def test_score_extreme_query_magnitude(G, h_kv):
    """Queries far beyond the fp16 range (|q| up to ~6e4): the kernels carry
    fp16 tensor-core operands, so each (sequence, KV head) prescales its
    query by a power of two.  Scores must stay finite and keep fp32-level
    relative accuracy (1e-4 of the largest score; the absolute 1e-3 bound
    of the specification does not apply to scores of this size)."""
    spec = W.custom_spec(batch=2, h_q=G * h_kv, h_kv=h_kv, ctx=16 * 24,
                         k=6, needles=0, seed=60 + G)
    wl = W.generate(spec, "cpu")
    kc, vc, pt, _ = host(wl)
    lens = [16 * 24, 16 * 9 + 3]
    batch, max_pages = pt.shape
    seq, pg = full_pairs(lens)
    store, _ = O.build_summaries(kc, pt, seq, pg, batch, max_pages)
    qb = (wl.queries[0].float() * 16384.0).to(torch.bfloat16)
    s_orc = O.score_store(qb.float().numpy(), store, lens)
    sc = torch.zeros(batch, h_kv, G, max_pages, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_score_pages(qb.to(DEV), torch.from_numpy(store).to(DEV),
                        i32(lens), sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    s = sc.cpu().numpy()
    for b in range(batch):
        nf = lens[b] // 16
        got, ref = s[b, :, :, :nf], s_orc[b, :, :, :nf]
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


@pytest.mark.parametrize("G,h_kv", [(4, 2), (1, 3), (8, 1), (16, 1)])
def test_exact_page_scores_match_oracle(G, h_kv):
    """Exact page LSE (what Eq.(4) estimates) of every full page, and the
    exact-mass selection obtained by feeding it to the selection kernel."""
    spec = W.custom_spec(batch=3, h_q=G * h_kv, h_kv=h_kv, ctx=16 * 70 + 9,
                         k=10, needles=0, seed=80 + G)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    kc, _, pt, _ = host(wl)
    lens = [16 * 70 + 9, 16 * 3, 0]
    batch, max_pages = pt.shape
    q = wl.queries[0]
    ex_o = O.exact_store(q.float().numpy(), kc, pt, lens, h_kv)
    sc = torch.full((batch, h_kv, G, max_pages), 7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_exact_page_scores(q.to(DEV), d.k_cache, d.page_table, i32(lens),
                              sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    s = sc.cpu().numpy()
    for b in range(batch):
        nf = lens[b] // 16
        assert np.abs(s[b, :, :, :nf] - ex_o[b, :, :, :nf]).max(initial=0) \
            <= S_TOL
        assert (s[b, :, :, nf:] == 7.0).all()
    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages, spec.k, DEV)
    idx = torch.zeros(batch, h_kv, spec.k, dtype=torch.int32, device=DEV)
    B.locks_select_pages(sc, i32(lens), spec.h_q, spec.k, idx, ws)
    torch.cuda.synchronize()
    ig = idx.cpu().numpy()
    io = O.select_store(ex_o, lens, spec.k)
    for b in range(batch):
        for h in range(h_kv):
            ok, _ = selection_agrees(ig[b, h], io[b, h], ex_o[b, h], lens[b],
                                     spec.k, 1e-3)
            assert ok, (b, h)


# ---------------------------------------------------------------------------
# rank / precision variants (notes §6 ablation)
# ---------------------------------------------------------------------------
def test_variant_r8_int4_build_equals_shipped_build():
    """On the GPU, the (r = 8, 4-bit) variant record is the shipped record
    byte for byte (one eigensolver, one quantiser, one layout rule)."""
    wl = W.generate(W.SPECS["tiny_4k"], "cpu")
    d = Dev(wl)
    _, _, pt, lens = host(wl)
    store, _, _, seq, pg = gpu_build(d, lens)
    batch, max_pages = pt.shape
    h_kv = d.k_cache.shape[1]
    var = B.new_variant_store(batch, h_kv, max_pages, 8, 4, DEV)
    assert var.shape[-1] == store.shape[-1] == 832
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_build_variant(d.k_cache, d.page_table, i32(seq), i32(pg), var, 8,
                          4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(var[seq, :, pg], store[seq, :, pg])


@pytest.mark.parametrize("rank,vbits", [(r, b) for r in O.VARIANT_RANKS
                                        for b in O.VARIANT_BITS])
def test_variant_build_and_score_match_oracle(rank, vbits):
    wl = W.generate(W.SPECS["tiny_4k"], "cpu", steps=1)
    d = Dev(wl)
    kc, _, pt, lens = host(wl)
    lens = [lens[0] - 5]                       # partial last page
    seq, pg = full_pairs(lens)
    batch, max_pages = pt.shape
    h_kv, G = kc.shape[1], W.SPECS["tiny_4k"].group
    var = B.new_variant_store(batch, h_kv, max_pages, rank, vbits, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_build_variant(d.k_cache, d.page_table, i32(seq), i32(pg), var,
                          rank, vbits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    keys = kc[pt[seq, pg]]                                 # [n][h_kv][16][128]
    qo, s = O.build_page_variant(keys, rank, vbits)
    got = O.decode_variant(var.cpu().numpy()[seq, :, pg], rank, vbits)
    # centroid bytes exact; basis codes equal up to eigenvector sign and a
    # one-step rounding difference on well separated components
    assert (got["mu8"] == qo["mu8"]).all() and (got["smu"] == qo["smu"]).all()
    _, Vg, _ = O.dequantize(got)
    sgn = np.sign(np.einsum("nhdk,nhdk->nhk", Vg, s["V"]))
    sgn[sgn == 0] = 1
    lam = s["lam"]
    gap = np.minimum(np.concatenate([np.full(lam[..., :1].shape, np.inf),
                                     lam[..., :rank - 1]], -1) - lam[..., :rank],
                     lam[..., :rank] - lam[..., 1:rank + 1]) / lam[..., :1]
    ok = gap > 1e-3
    dv = np.abs(got["Vq"].astype(int) * sgn[..., None, :].astype(int) -
                qo["Vq"].astype(int))
    m = ok[..., None, :] & np.ones_like(dv, bool)
    assert dv[m].max(initial=0) <= 1 and (dv[m] > 0).mean() < 0.02
    # scores from the oracle's own records (encoded as variant records)
    recs = torch.zeros_like(var)
    recs[seq, :, pg] = torch.from_numpy(O.encode_variant(qo, rank, vbits)).to(
        DEV)
    q = wl.queries[0]
    sc = torch.full((batch, h_kv, G, max_pages), 5.0, device=DEV)
    B.locks_score_variant(q.to(DEV), recs, rank, vbits, i32(lens), sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    mu, V, C = O.dequantize(qo)                            # [n][h_kv] ...
    qn = q.float().numpy()
    nf = lens[0] // 16
    s_gpu = sc.cpu().numpy()
    for h in range(h_kv):
        ref = O.score_from_summaries(qn[0, h * G:(h + 1) * G], mu[:, h],
                                     V[:, h], C[:, h])
        assert np.abs(s_gpu[0, h, :, :nf] - ref).max() <= S_TOL
        assert (s_gpu[0, h, :, nf:] == 5.0).all()


# every (rank, head form) of the variant scorer: G <= 4 with ranks 4 and 8
# pairs pages in the coefficient product, G <= 8 keeps heads in its rows,
# G > 8 runs it per half of the heads; strides above 832 bytes take 4-page
# tiles
VARIANT_GROUP_CASES = [
    (1, 3, 4, 2), (4, 2, 4, 4), (3, 2, 8, 4), (2, 1, 8, 8), (4, 2, 8, 2),
    (8, 1, 4, 8), (6, 1, 4, 2), (8, 1, 8, 4), (5, 2, 8, 2), (4, 1, 12, 4),
    (8, 1, 12, 8), (8, 1, 15, 8), (4, 2, 15, 4), (2, 2, 15, 2),
    (16, 1, 12, 2), (12, 1, 4, 4), (9, 1, 8, 8), (16, 1, 15, 4)]


@pytest.mark.parametrize("G,h_kv,rank,vbits", VARIANT_GROUP_CASES)
def test_variant_score_group_sizes(G, h_kv, rank, vbits):
    """Variant scores from the oracle's own variant records at several
    group sizes, over enough pages for several CTAs and a ragged tail."""
    spec = W.custom_spec(batch=2, h_q=G * h_kv, h_kv=h_kv, ctx=16 * 150 + 7,
                         k=8, needles=0, seed=60 + G)
    wl = W.generate(spec, "cpu", steps=1)
    kc, _, pt, _ = host(wl)
    lens = [16 * 150 + 7, 16 * 70]
    batch, max_pages = pt.shape
    seq, pg = full_pairs(lens)
    keys = kc[pt[seq, pg]]                                 # [n][h_kv][16][128]
    qo, _ = O.build_page_variant(keys, rank, vbits)
    recs = B.new_variant_store(batch, h_kv, max_pages, rank, vbits, DEV)
    recs[seq, :, pg] = torch.from_numpy(O.encode_variant(qo, rank, vbits)).to(
        DEV)
    q = wl.queries[0]
    sc = torch.full((batch, h_kv, G, max_pages), 5.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_score_variant(q.to(DEV), recs, rank, vbits, i32(lens), sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    mu, V, C = O.dequantize(qo)
    qn = q.float().numpy()
    s_gpu = sc.cpu().numpy()
    seq, pg = np.asarray(seq), np.asarray(pg)
    for b in range(batch):
        nf = lens[b] // 16
        sel = seq == b
        for h in range(h_kv):
            ref = O.score_from_summaries(qn[b, h * G:(h + 1) * G],
                                         mu[sel, h], V[sel, h], C[sel, h])
            assert np.abs(s_gpu[b, h, :, pg[sel]].T - ref).max() <= S_TOL
            assert (s_gpu[b, h, :, nf:] == 5.0).all()


@pytest.mark.parametrize("G,rank,vbits", [(4, 8, 4), (8, 15, 8), (4, 4, 2)])
def test_variant_score_many_tiles_per_warp(G, rank, vbits):
    """More tiles than warps in the grid: every warp streams several tiles
    across (sequence, KV head) boundaries through its double-buffered ring;
    scores against the oracle's own records on sampled pages of every unit
    and on every page of the last one."""
    h_kv, n_pages = 8, 2600
    lens = [16 * n_pages - 3, 16 * (n_pages // 2) + 8]
    spec = W.custom_spec(batch=2, h_q=G * h_kv, h_kv=h_kv,
                         ctx=16 * n_pages, k=8, needles=0, seed=90 + rank)
    wl = W.generate(spec, "cpu", steps=1)
    kc, _, pt, _ = host(wl)
    batch, max_pages = pt.shape
    seq, pg = full_pairs(lens)
    seq, pg = np.asarray(seq), np.asarray(pg)
    keys = kc[pt[seq, pg]]
    qo, _ = O.build_page_variant(keys, rank, vbits)
    recs = B.new_variant_store(batch, h_kv, max_pages, rank, vbits, DEV)
    recs[torch.as_tensor(seq), :, torch.as_tensor(pg)] = torch.from_numpy(
        O.encode_variant(qo, rank, vbits)).to(DEV)
    q = wl.queries[0]
    sc = torch.full((batch, h_kv, G, max_pages), 5.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_score_variant(q.to(DEV), recs, rank, vbits, i32(lens), sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    mu, V, C = O.dequantize(qo)
    qn = q.float().numpy()
    s_gpu = sc.cpu().numpy()
    rng = np.random.default_rng(rank)
    for b in range(batch):
        nf = lens[b] // 16
        rows = np.flatnonzero(seq == b)
        for h in range(h_kv):
            pick = rows if (b, h) == (batch - 1, h_kv - 1) else \
                np.sort(rng.choice(rows, 64, replace=False))
            ref = O.score_from_summaries(qn[b, h * G:(h + 1) * G],
                                         mu[pick, h], V[pick, h], C[pick, h])
            assert np.abs(s_gpu[b, h, :, pg[pick]].T - ref).max() <= S_TOL
            assert (s_gpu[b, h, :, nf:] == 5.0).all()


# ---------------------------------------------------------------------------
# select (Eq.(5) + sink/recent) from identical scores
# ---------------------------------------------------------------------------
def test_select_matches_oracle_on_same_scores():
    rng = np.random.default_rng(7)
    batch, h_kv, G, max_pages, k = 7, 3, 4, 300, 12
    lens = [0, 5, 16, 16 * 12, 16 * 12 + 3, 16 * 300, 16 * 257 + 15]
    scores = rng.normal(0, 3, (batch, h_kv, G, max_pages)).astype(np.float32)
    scores[5, 1, :, :] = 1.0                      # all equal: lowest index
    ws = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    B.locks_select_pages(torch.from_numpy(scores).to(DEV), i32(lens),
                         G * h_kv, k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    io = O.select_store(scores.astype(np.float64), lens, k)
    for b in range(batch):
        for h in range(h_kv):
            ok, nd = selection_agrees(ig[b, h], io[b, h],
                                      scores[b, h].astype(np.float64),
                                      lens[b], k, 1e-4)
            assert ok, (b, h, ig[b, h], io[b, h])
    assert (ig[0] == -1).all()
    assert (ig[1, :, 0] == 0).all() and (ig[1, :, 1:] == -1).all()
    assert list(ig[3, 0]) == list(range(12))        # 12 pages = k: all
    assert list(ig[5, 1]) == list(range(11)) + [299]
    for b in range(batch):
        for h in range(h_kv):
            v = [x for x in ig[b, h] if x >= 0]
            assert v == sorted(v) and len(set(v)) == len(v)


@pytest.mark.parametrize("G,h_kv,batch,max_pages,k",
                         [(4, 2, 1, 40, 8), (8, 4, 3, 700, 12),
                          (4, 8, 8, 2048, 64), (1, 1, 2, 300, 6),
                          (5, 2, 5, 129, 10), (4, 8, 4, 8192, 128),
                          (8, 8, 19, 64, 2), (4, 2, 3, 90, 200)])
def test_fused_score_select_matches_two_kernels(G, h_kv, batch, max_pages, k):
    """Short page lists on at most one unit per SM take the single-launch
    score and select (one thread-block cluster per (sequence, KV head)):
    locks_score_select then writes the scores locks_score_pages writes,
    bit for bit, and selects what the oracle selects from them (identical
    sets except pages within 1e-3 of the boundary in log share-average);
    the two-kernel path (locks_score_pages + locks_select_pages) on the
    same records agrees with it the same way.  Shapes: clusters of 8, 4, 2
    and 1 CTAs, both scoring forms (G <= 4, G <= 8), 8,192 pages, empty and
    one-page sequences, k = 2 and k above every sequence's pages."""
    spec = W.custom_spec(batch=batch, h_q=G * h_kv, h_kv=h_kv,
                         ctx=16 * max_pages, k=max(k, 2), needles=1,
                         seed=300 + G + batch)
    wl = W.generate(spec, "cpu")
    kc, _, pt, _ = host(wl)
    rng = np.random.default_rng(G * 7 + batch)
    lens = [int(x) for x in rng.integers(0, 16 * max_pages + 1, batch)]
    lens[0] = 16 * max_pages
    if batch > 2:
        lens[1], lens[2] = 0, 16 + 3
    seq, pg = full_pairs(lens)
    store, _ = O.build_summaries(kc, pt, seq, pg, batch, max_pages)
    q = wl.queries[0].to(DEV)
    st = torch.from_numpy(store).to(DEV)
    sl = i32(lens)
    ws_f = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    ws_t = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    idx_f = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    idx_t = torch.zeros_like(idx_f)
    B.locks_score_select(q, st, sl, k, idx_f, ws_f)
    n = batch * h_kv * G * max_pages
    sc_t = ws_t[256:256 + 4 * n].view(torch.float32).view(
        batch, h_kv, G, max_pages)
    B.locks_score_pages(q, st, sl, sc_t, ws_t[:4].view(torch.int32))
    B.locks_select_pages(sc_t, sl, G * h_kv, k, idx_t, ws_t)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws_f) == 0 and B.locks_read_status(ws_t) == 0
    sc_f = ws_f[256:256 + 4 * n].view(torch.float32).view(sc_t.shape)
    s_orc = O.score_store(wl.queries[0].float().numpy(), store, lens)
    idx_o = O.select_store(s_orc, lens, k)
    i_f, i_t = idx_f.cpu().numpy(), idx_t.cpu().numpy()
    for b in range(batch):
        nf = lens[b] // 16
        assert torch.equal(sc_f[b, :, :, :nf], sc_t[b, :, :, :nf]), b
        for h in range(h_kv):
            for ig in (i_f, i_t):
                ok, _ = selection_agrees(ig[b, h], idx_o[b, h], s_orc[b, h],
                                         lens[b], k, 1e-3)
                assert ok, (b, h, ig[b, h], idx_o[b, h])
            v = [x for x in i_f[b, h] if x >= 0]
            assert v == sorted(v) and len(set(v)) == len(v)
            if set(i_f[b, h]) != set(i_t[b, h]):
                ok, _ = selection_agrees(i_f[b, h], i_t[b, h], s_orc[b, h],
                                         lens[b], k, 1e-3)
                assert ok, (b, h)


@pytest.mark.parametrize("G", [1, 4, 16])
def test_select_normaliser_fallback(G):
    """Scores for which the normaliser's common reference (each head's
    page-0 score) does not serve: page 0 at -inf, page 0 far below every
    other page, one page far above page 0 (the sum against the reference
    overflows).  The selection must still be the oracle's (Eq.(5) with the
    normaliser over all full pages)."""
    rng = np.random.default_rng(11 + G)
    batch, h_kv, max_pages, k = 3, 2, 400, 20
    lens = [16 * 400, 16 * 333 + 7, 16 * 400]
    scores = rng.normal(0, 2, (batch, h_kv, G, max_pages)).astype(np.float32)
    scores[0, 0, :, 0] = -np.inf
    scores[0, 1, :, 0] = -200.0
    scores[1, :, :, 0] = -120.0
    scores[2, 1, 0, 5] = 90.0
    ws = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    B.locks_select_pages(torch.from_numpy(scores).to(DEV), i32(lens),
                         G * h_kv, k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    io = O.select_store(scores.astype(np.float64), lens, k)
    for b in range(batch):
        for h in range(h_kv):
            ok, _ = selection_agrees(ig[b, h], io[b, h],
                                     scores[b, h].astype(np.float64),
                                     lens[b], k, 1e-4)
            assert ok, (b, h, ig[b, h], io[b, h])
    assert 5 in ig[2, 1]


# Few units of at least 4,096 pages take the selection's cluster form (4 or
# 2 CTAs per unit, the passes split by page range, the normaliser's sums
# merged across the cluster, CTA 0 selecting): every head-count width, the
# three merge rules, the normaliser's fallback form, k = 2, ragged and empty
# lists, page counts that split unevenly; one case below the floor.
SELECT_CLUSTER_CASES = [
    (1, 2, 3, 4100, 40, "share_average", False),
    (2, 4, 4, 4096, 16, "group_max", False),
    (4, 8, 9, 8192, 128, "share_average", False),
    (2, 8, 5, 4500, 50, "group_mass", False),
    (8, 4, 3, 4097, 128, "group_mass", False),
    (16, 1, 5, 5030, 20, "share_average", False),
    (4, 2, 3, 4777, 30, "share_average", True),
    (8, 1, 3, 4900, 25, "group_max", True),
    (3, 2, 2, 4099, 2, "share_average", False),
    (4, 8, 8, 2048, 64, "share_average", False),
]


@pytest.mark.parametrize("G,h_kv,batch,max_pages,k,rule,extreme",
                         SELECT_CLUSTER_CASES)
def test_select_cluster_forms(G, h_kv, batch, max_pages, k, rule, extreme):
    rng = np.random.default_rng(500 + G * 11 + max_pages)
    lens = [int(x) for x in rng.integers(16 * k, 16 * max_pages + 1, batch)]
    lens[0] = 16 * max_pages
    if batch > 2:
        lens[1] = 16 * (max_pages - 3) + 5       # partial last page
        lens[2] = 16 * (k - 1)                   # fewer pages than k
    if batch > 4:
        lens[4] = 0
    scores = (rng.normal(0, 3, (batch, h_kv, G, max_pages)) +
              rng.normal(0, 4, (batch, h_kv, 1, max_pages))).astype(np.float32)
    if extreme:  # the normaliser's common reference does not serve
        scores[0, 0, :, 0] = -np.inf
        scores[0, h_kv - 1, :, 0] = -200.0
        scores[1, 0, 0, 7] = 95.0
        scores[1, :, :, max_pages - 40] = 60.0
    sd = torch.from_numpy(scores).to(DEV)
    ws = B.new_workspace(batch, h_kv * G, h_kv, max_pages, k, DEV)
    idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    B.locks_select_pages_merge(sd, i32(lens), h_kv * G, k, rule, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    s64 = scores.astype(np.float64)
    for b in range(batch):
        n = -(-lens[b] // 16)
        for h in range(h_kv):
            row = [int(x) for x in ig[b, h]]
            valid = [x for x in row if x >= 0]
            assert valid == sorted(valid) and len(set(valid)) == len(valid)
            want = set(O.select_one_rule(s64[b, h], lens[b], k, rule))
            got = set(valid)
            if n <= k:
                assert row == list(range(n)) + [-1] * (k - n), (b, h)
                continue
            if got == want:
                continue
            nf = lens[b] // 16
            lk = O.merge_key(s64[b, h], nf, rule)
            lk = lk if rule == "group_mass" else np.log(lk)
            cand = np.arange(1, n - 1)
            order = cand[np.lexsort((cand, -lk[cand]))]
            edge = lk[order[k - 3]]
            for p in got ^ want:
                assert p not in (0, n - 1) and abs(lk[p] - edge) <= 1e-4, \
                    (rule, b, h, p)
    if extreme:
        assert 7 in ig[1, 0] or rule == "group_max"


# ---------------------------------------------------------------------------
# sparse attention over the oracle's selection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("G,h_kv,k", [(4, 2, 8), (8, 1, 5), (16, 1, 16),
                                      (1, 3, 4), (3, 2, 64)])
def test_sparse_decode_matches_oracle(G, h_kv, k):
    spec = W.custom_spec(batch=4, h_q=G * h_kv, h_kv=h_kv, ctx=16 * 40,
                         k=k, needles=0, seed=40 + G + k)
    wl = W.generate(spec, "cpu")
    kc, vc, pt, _ = host(wl)
    lens = [16 * 40, 16 * 33 + 7, 0, 9]
    batch, max_pages = pt.shape
    rng = np.random.default_rng(G + k)
    s_hat = rng.normal(0, 2, (batch, h_kv, G, max_pages))
    idx_o = O.select_store(s_hat, lens, k)
    q = wl.queries[0].float().numpy()
    o_ref, lse_ref = O.sparse_decode(q, kc, vc, pt, lens, idx_o)
    d = Dev(wl)
    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages,
                         max(k, max_pages), DEV)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=DEV)
    for mode in ("sparse", "dense"):
        if mode == "sparse":
            B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache,
                                  d.page_table, i32(lens), i32(idx_o), k, o,
                                  lse, ws)
            ro, rl = o_ref, lse_ref
        else:
            B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache,
                                  d.page_table, i32(lens), None, 0, o, lse,
                                  ws)
            ro, rl = O.dense_decode(q, kc, vc, pt, lens)
        torch.cuda.synchronize()
        assert B.locks_read_status(ws) == 0
        og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
        for b in range(batch):
            if lens[b] == 0:
                assert (og[b] == 0).all() and np.isneginf(lg[b]).all()
                continue
            assert np.abs(og[b] - ro[b]).max() <= O_TOL * np.abs(ro[b]).max()
            assert np.abs(lg[b] - rl[b]).max() <= LSE_TOL


# at least one (sequence, KV head) unit per SM: sparse decode takes its unit
# form (a CTA per unit, four warps on a quarter of the list each, merged in
# shared memory); k not a multiple of 4, k = 3 (an empty quarter), lists
# with -1 padding, partial pages and empty sequences, G = 16
# (fewer units than SMs: clusters of 4 or 8 CTAs per unit, the partials
# merged across the cluster; too few positions per warp: the split form
# and its merge)
@pytest.mark.parametrize("G,k,batch", [(4, 7, 40), (8, 3, 40), (16, 10, 40),
                                       (1, 64, 40), (4, 64, 3), (8, 128, 16),
                                       (16, 128, 5), (2, 256, 2), (4, 32, 3),
                                       (4, 40, 16), (2, 16, 3)])
def test_decode_unit_form_matches_oracle(G, k, batch):
    h_kv, n_pages = 4, max(24, k + 8)
    spec = W.custom_spec(batch=batch, h_q=G * h_kv, h_kv=h_kv,
                         ctx=16 * n_pages, k=k, needles=0, seed=140 + G + k)
    wl = W.generate(spec, "cpu")
    kc, vc, pt, _ = host(wl)
    rng = np.random.default_rng(G * 3 + k)
    lens = [int(x) for x in rng.integers(1, 16 * n_pages + 1, batch)]
    lens[0] = 16 * n_pages
    if batch > 1:
        lens[1] = 0
    if batch > 3:
        lens[2], lens[3] = 5, 16 * 2 + 9
    max_pages = pt.shape[1]
    s_hat = rng.normal(0, 2, (batch, h_kv, G, max_pages))
    idx_o = O.select_store(s_hat, lens, k)
    q = wl.queries[0].float().numpy()
    o_ref, lse_ref = O.sparse_decode(q, kc, vc, pt, lens, idx_o)
    d = Dev(wl)
    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages, k, DEV)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=DEV)
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, d.page_table,
                          i32(lens), i32(idx_o), k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(batch):
        if lens[b] == 0:
            assert (og[b] == 0).all() and np.isneginf(lg[b]).all()
            continue
        assert np.abs(og[b] - o_ref[b]).max() <= O_TOL * np.abs(o_ref[b]).max()
        assert np.abs(lg[b] - lse_ref[b]).max() <= LSE_TOL


@pytest.mark.parametrize("batch,h_kv,k", [(40, 4, 6), (4, 2, 16)])
def test_native_decoder_unit_form_status(batch, h_kv, k):
    """The host-buffer decoder with the decode's unit form (160 units: a CTA
    per unit; 8 units of 16 list positions: clusters of 4 CTAs), whose
    status word reaches the host through its own copy kernel: o and lse
    equal the eager step's bytes, and a page table entry outside the cache
    comes back in the step's status."""
    spec = W.custom_spec(batch=batch, h_q=4 * h_kv, h_kv=h_kv,
                         ctx=16 * 20 + 3, k=k, needles=0, seed=151 + batch)
    wl = W.generate(spec, "cpu", steps=3)
    d = Dev(wl)
    lens = [16 * 20 + 3] * batch
    empty, bad = (5, 7) if batch > 7 else (batch - 1, 1)
    lens[empty] = 0
    lens_dev = i32(lens)
    store, _, _, _, _ = gpu_build(d, lens)
    pt = d.page_table.clone()
    native = B.LocksDecoder(d.k_cache, d.v_cache, pt, store, spec.h_q,
                            spec.k, graph=True, seq_lens=lens_dev)
    eager = B.LocksDecoder(d.k_cache, d.v_cache, pt, store, spec.h_q, spec.k)
    shape = (batch, spec.h_q, 128)
    qh = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    oh = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(batch, spec.h_q).pin_memory()
    for step in range(3):
        if step == 1:        # the recent page of sequence `bad`: always selected
            pt[bad, 20] = d.k_cache.shape[0] + 11
        if step == 2:
            pt[bad, 20] = int(d.page_table[bad, 20])
            B.locks_clear_status(native.workspace)
            B.locks_clear_status(eager.workspace)
        qh.copy_(wl.queries[step])
        oe, le = eager.step(qh.to(DEV), lens_dev)
        torch.cuda.synchronize()
        _, _, st = native.step_host(qh, lens_dev, oh, lh)
        assert st == (B.DEV_BAD_PAGE_ID if step == 1 else 0), (step, st)
        assert st == eager.status()
        assert torch.equal(oe.cpu(), oh) and torch.equal(le.cpu(), lh)
        assert (oh[empty] == 0).all() and torch.isinf(lh[empty]).all()
    native.close()


def test_step_at_the_largest_batch():
    """The step at the scoring and selection calls' batch limit (1594
    sequences, whose per-sequence tables fill the on-chip space beside the
    summary ring): scores from the oracle's records against the oracle on
    every page, selections within the 1e-3 window, outputs of the decode's
    unit form (1594 units) against the oracle's attention over the GPU's
    selection."""
    batch, G, k = 1594, 4, 3
    spec = W.custom_spec(batch=batch, h_q=G, h_kv=1, ctx=16 * 5 + 7, k=k,
                         needles=0, seed=1594)
    wl = W.generate(spec, "cpu", steps=1)
    kc, vc, pt, _ = host(wl)
    rng = np.random.default_rng(1594)
    lens = [int(x) for x in rng.integers(16 * 4, 16 * 5 + 8, batch)]
    max_pages = pt.shape[1]
    seq, pg = full_pairs(lens)
    store, _ = O.build_summaries(kc, pt, seq, pg, batch, max_pages)
    q = wl.queries[0]
    st = torch.from_numpy(store).to(DEV)
    ws = B.new_workspace(batch, G, 1, max_pages, k, DEV)
    idx = torch.zeros(batch, 1, k, dtype=torch.int32, device=DEV)
    B.locks_score_select(q.to(DEV), st, i32(lens), k, idx, ws)
    n = batch * G * max_pages
    sc = ws[256:256 + 4 * n].view(torch.float32).view(batch, 1, G,
                                                      max_pages).clone()
    d = Dev(wl)
    o = torch.empty(batch, G, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, G, dtype=torch.float32, device=DEV)
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, d.page_table,
                          i32(lens), idx, k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    s_orc = O.score_store(q.float().numpy(), store, lens)
    s_gpu = sc.cpu().numpy()
    full = ~np.isnan(s_orc)
    assert np.abs(s_gpu[full] - s_orc[full]).max() <= S_TOL
    ig = idx.cpu().numpy()
    io = O.select_store(s_orc, lens, k)
    for b in range(batch):
        ok, _ = selection_agrees(ig[b, 0], io[b, 0], s_orc[b, 0], lens[b], k,
                                 1e-3)
        assert ok, (b, ig[b, 0], io[b, 0])
    o_ref, lse_ref = O.sparse_decode(q.float().numpy(), kc, vc, pt, lens, ig)
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    scale = np.abs(o_ref).max(axis=(1, 2))
    assert (np.abs(og - o_ref).max(axis=(1, 2)) <= O_TOL * scale).all()
    assert np.abs(lg - lse_ref).max() <= LSE_TOL


@pytest.mark.parametrize("G,mode", [(4, "sparse"), (4, "dense"),
                                    (16, "sparse"), (2, "dense")])
def test_decode_many_short_units(G, mode):
    """Thousands of short page lists, so that runs of consecutive list
    entries hold several whole (sequence, KV head) lists as well as pieces
    of lists shared with the neighbouring runs; empty sequences, partial
    pages and -1 padding give skipped entries at every place in a run."""
    rng = np.random.default_rng(90 + G)
    batch, h_kv, max_pages, k = 2048, 1, 4, 2
    h_q = G * h_kv
    lens = rng.integers(0, 16 * max_pages + 1, batch)
    lens[::97] = 0
    lens[1::89] = 1
    num_phys = batch * max_pages
    pt = rng.permutation(num_phys).reshape(batch, max_pages).astype(np.int32)
    gen = torch.Generator().manual_seed(int(G))
    kc = torch.randn(num_phys, h_kv, 16, 128, generator=gen).to(torch.bfloat16)
    vc = torch.randn(num_phys, h_kv, 16, 128, generator=gen).to(torch.bfloat16)
    q = torch.randn(batch, h_q, 128, generator=gen).to(torch.bfloat16)
    idx = np.full((batch, h_kv, k), -1, np.int32)
    for b in range(batch):
        n = -(-int(lens[b]) // 16)
        m = min(k, n)
        if m:
            idx[b, :, :m] = np.sort(rng.choice(n, m, replace=False))
    o_ref, lse_ref = O.sparse_decode(q.float().numpy(), kc.float().numpy(),
                                     vc.float().numpy(), pt, lens,
                                     None if mode == "dense" else idx)
    ws = B.new_workspace(batch, h_q, h_kv, max_pages, max(k, max_pages), DEV)
    o = torch.empty(batch, h_q, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, h_q, dtype=torch.float32, device=DEV)
    B.locks_sparse_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), i32(pt),
                          i32(lens), None if mode == "dense" else i32(idx),
                          k if mode == "sparse" else 0, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    empty = lens == 0
    assert (og[empty] == 0).all() and np.isneginf(lg[empty]).all()
    scale = np.abs(o_ref[~empty]).max(axis=(1, 2))
    err = np.abs(og[~empty] - o_ref[~empty]).max(axis=(1, 2))
    assert (err <= O_TOL * scale).all(), float((err / scale).max())
    assert np.abs(lg[~empty] - lse_ref[~empty]).max() <= LSE_TOL


# ---------------------------------------------------------------------------
# the whole step on the 4K-context workload, 8 decode steps
# ---------------------------------------------------------------------------
SEL_WIN = 1e-3


@pytest.mark.parametrize("which", ["tiny_4k", "ragged_decay"])
def test_end_to_end_workload(which):
    """The whole product path (GPU build, then every decode step through the
    decoder object: score, select, sparse attention) against the oracle's
    own build, selection and attention on the same inputs.  Selections must
    be identical except pages whose oracle log share-average lies within
    1e-3 of the boundary candidate's; o and lse are compared for every
    (step, query head): directly where the sets agree, and where they differ
    within the window, by running the GPU decode on the oracle's selection."""
    if which == "tiny_4k":
        spec = W.SPECS["tiny_4k"]
        wl = W.generate(spec, "cpu")
    else:
        wl = _ragged_decay_workload()
        spec = wl.spec
    d = Dev(wl)
    kc, vc, pt, lens = host(wl)
    batch, max_pages = pt.shape
    G = spec.group
    store, _, _, seq, pg = gpu_build(d, lens)
    ostore, _ = O.build_summaries(kc, pt, seq, pg, batch, max_pages)
    dec = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store, spec.h_q,
                         spec.k)
    steps = min(spec.steps, 8)
    n_diff = 0
    for step in range(steps):
        o, lse = dec.step(d.queries[step], d.seq_lens)
        torch.cuda.synchronize()
        assert dec.status() == 0
        q = wl.queries[step].float().numpy()
        s_orc = O.score_store(q, ostore, lens)
        idx_o = O.select_store(s_orc, lens, spec.k)
        ig = dec.idx.cpu().numpy()
        og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
        o_ref, lse_ref = O.sparse_decode(q, kc, vc, pt, lens, idx_o)
        differs = np.zeros((batch, spec.h_kv), bool)
        for b in range(batch):
            for h in range(spec.h_kv):
                ok, nd = selection_agrees(ig[b, h], idx_o[b, h], s_orc[b, h],
                                          lens[b], spec.k, SEL_WIN)
                assert ok, (step, b, h)
                differs[b, h] = nd > 0
        if differs.any():
            n_diff += int(differs.sum())
            o2 = torch.empty_like(o)
            l2 = torch.empty_like(lse)
            B.locks_sparse_decode(d.queries[step], d.k_cache, d.v_cache,
                                  d.page_table, d.seq_lens, i32(idx_o),
                                  spec.k, o2, l2, dec.workspace)
            torch.cuda.synchronize()
            assert dec.status() == 0
            o2, l2 = o2.float().cpu().numpy(), l2.cpu().numpy()
            for b, h in zip(*np.nonzero(differs)):
                sl = slice(h * G, (h + 1) * G)
                og[b, sl], lg[b, sl] = o2[b, sl], l2[b, sl]
        for b in range(batch):
            for h in range(spec.h_kv):
                sl = slice(h * G, (h + 1) * G)
                assert np.abs(og[b, sl] - o_ref[b, sl]).max() <= \
                    O_TOL * np.abs(o_ref[b, sl]).max(), (step, b, h)
                assert np.abs(lg[b, sl] - lse_ref[b, sl]).max() <= LSE_TOL
    # the differing sets are rare: the boundary window is narrow
    assert n_diff <= max(1, steps * batch * spec.h_kv // 10)


@pytest.mark.parametrize("name", ["tiny_4k", "ragged"])
def test_decoder_graph_replay_matches_eager(name):
    """The decode step captured once into a CUDA graph (five kernels with
    programmatic dependencies) and replayed with new queries gives the
    eager step's bytes: indices, o and lse identical."""
    if name == "tiny_4k":
        spec = W.SPECS["tiny_4k"]
    else:
        spec = W.custom_spec(batch=6, h_q=16, h_kv=4, ctx=16 * 90, k=12,
                             needles=1, seed=77, ragged_min=16 * 3)
    wl = W.generate(spec, "cpu", steps=4)
    d = Dev(wl)
    _, _, _, lens = host(wl)
    store, _, _, _, _ = gpu_build(d, lens)
    eager = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store,
                           spec.h_q, spec.k)
    graph = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store,
                           spec.h_q, spec.k, graph=True)
    for step in range(4):
        oe, le = eager.step(d.queries[step], d.seq_lens)
        oe, le, ie = oe.clone(), le.clone(), eager.idx.clone()
        og, lg = graph.step(d.queries[step], d.seq_lens)
        torch.cuda.synchronize()
        assert eager.status() == 0 and graph.status() == 0
        assert torch.equal(ie, graph.idx)
        assert torch.equal(oe, og) and torch.equal(le, lg)
    assert graph._graph is not None


def test_decoder_append_graph_matches_eager():
    """The decode step with its append (the new token written at the
    current length and, when that fills a page, the page's summary built)
    captured into one CUDA graph gives the eager step's bytes: o, lse and
    indices every step, and the same caches, summary store and lengths
    after 20 steps that fill a page of every sequence."""
    spec = W.custom_spec(batch=3, h_q=16, h_kv=4, ctx=16 * 40 + 9, k=8,
                         steps=20, needles=1, seed=23, append_steps=20,
                         ragged_min=16 * 30)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    batch, max_pages = wl.page_table.shape
    lens0 = [int(x) for x in wl.seq_lens]
    seq, pg = full_pairs(lens0)
    store = B.new_summary_store(batch, spec.h_kv, max_pages, DEV)
    B.locks_build_summaries(d.k_cache, d.page_table, i32(seq), i32(pg), store)
    kc2, vc2, st2 = d.k_cache.clone(), d.v_cache.clone(), store.clone()
    lens_e, lens_g = d.seq_lens.clone(), d.seq_lens.clone()
    eager = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store,
                           spec.h_q, spec.k, seq_lens=lens_e, append=True)
    graph = B.LocksDecoder(kc2, vc2, d.page_table, st2, spec.h_q, spec.k,
                           graph=True, seq_lens=lens_g, append=True)
    ka, va = wl.k_append.to(DEV), wl.v_append.to(DEV)
    for s in range(spec.append_steps):
        q = d.queries[s]
        oe, le = eager.step(q, k_new=ka[s], v_new=va[s])
        oe, le, ie = oe.clone(), le.clone(), eager.idx.clone()
        og, lg = graph.step(q, k_new=ka[s], v_new=va[s])
        torch.cuda.synchronize()
        assert eager.status() == 0 and graph.status() == 0, s
        assert torch.equal(ie, graph.idx), s
        assert torch.equal(oe, og) and torch.equal(le, lg), s
    assert graph._graph is not None
    assert lens_g.cpu().tolist() == [L + spec.append_steps for L in lens0]
    assert torch.equal(lens_e, lens_g)
    assert torch.equal(d.k_cache, kc2) and torch.equal(d.v_cache, vc2)
    assert torch.equal(store, st2)
    # every sequence filled at least one page during the appends
    assert all((L + spec.append_steps) // 16 > L // 16 for L in lens0)


def test_native_host_decoder_matches_eager():
    """locks_decoder_step_host (query copy in, five kernels, copies of o,
    lse and the status word out, replayed as one CUDA graph) returns the
    eager step's bytes, with the host buffers changed between steps (the
    graph's copy nodes retargeted) and the bound lengths grown in place by
    appends between steps."""
    spec = W.custom_spec(batch=5, h_q=16, h_kv=4, ctx=16 * 70 + 5, k=10,
                         needles=1, seed=83, ragged_min=16 * 2 + 1,
                         append_steps=12)
    wl = W.generate(spec, "cpu", steps=6)
    d = Dev(wl)
    _, _, _, lens = host(wl)
    store, _, _, _, _ = gpu_build(d, lens)
    lens_dev = d.seq_lens.clone()
    eager = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store,
                           spec.h_q, spec.k)
    native = B.LocksDecoder(d.k_cache, d.v_cache, d.page_table, store,
                            spec.h_q, spec.k, graph=True, seq_lens=lens_dev)
    shape = (spec.batch, spec.h_q, 128)
    q_bufs = [torch.empty(shape, dtype=torch.bfloat16).pin_memory()
              for _ in range(2)]
    o_bufs = [torch.empty(shape, dtype=torch.bfloat16).pin_memory()
              for _ in range(2)]
    lse_buf = torch.empty(spec.batch, spec.h_q).pin_memory()
    for step in range(6):
        if step in (2, 4):   # one token per sequence, lengths grow on device
            for a in range(step // 2 * 3):
                B.locks_append_kv(wl.k_append[a % 12].to(DEV),
                                  wl.v_append[a % 12].to(DEV), d.k_cache,
                                  d.v_cache, d.page_table, lens_dev, store)
        qh = q_bufs[step % 2]
        qh.copy_(wl.queries[step])
        oe, le = eager.step(qh.to(DEV), lens_dev.clone())
        torch.cuda.synchronize()
        oh, lh, st = native.step_host(qh, lens_dev, o_bufs[step % 3 % 2],
                                      lse_buf)
        assert st == 0 and eager.status() == 0
        assert torch.equal(eager.idx, native.idx)
        assert torch.equal(oe.cpu(), oh) and torch.equal(le.cpu(), lh)
    assert native._native is not None
    pageable = torch.empty(shape, dtype=torch.bfloat16)
    with pytest.raises(B.LocksError):
        native.step_host(pageable, lens_dev, o_bufs[0], lse_buf)
    native.close()


# ---------------------------------------------------------------------------
# append + incremental build
# ---------------------------------------------------------------------------
def test_append_per_page_scale_matches_build():
    """Pages filled by appends with LOCKS_BUILD_VSCALE_PER_PAGE carry the
    record a per-page build of the final cache gives, byte for byte."""
    spec = W.custom_spec(batch=2, h_q=8, h_kv=2, ctx=16 * 5 + 9, k=4,
                         steps=20, needles=0, seed=19, append_steps=20)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    batch, max_pages = wl.page_table.shape
    flags = B.BUILD_VSCALE_PER_PAGE
    lens0 = [int(x) for x in wl.seq_lens]
    seq, pg = full_pairs(lens0)
    store = B.new_summary_store(batch, spec.h_kv, max_pages, DEV)
    B.locks_build_summaries(d.k_cache, d.page_table, i32(seq), i32(pg), store,
                            flags=flags)
    seq_lens = d.seq_lens.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in range(spec.append_steps):
        B.locks_append_kv(wl.k_append[s].to(DEV), wl.v_append[s].to(DEV),
                          d.k_cache, d.v_cache, d.page_table, seq_lens, store,
                          status=status, flags=flags)
    lens1 = [L + spec.append_steps for L in lens0]
    seq1, pg1 = full_pairs(lens1)
    fresh = B.new_summary_store(batch, spec.h_kv, max_pages, DEV)
    B.locks_build_summaries(d.k_cache, d.page_table, i32(seq1), i32(pg1),
                            fresh, flags=flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b, p in zip(seq1, pg1):
        assert torch.equal(store[b, :, p], fresh[b, :, p]), (b, p)
    rec = O.decode_records(fresh.cpu().numpy()[seq1, :, pg1])
    assert (rec["sV"] == rec["sV"][..., :1]).all()


def test_append_builds_filled_pages():
    spec = W.custom_spec(batch=3, h_q=8, h_kv=2, ctx=16 * 6 + 13, k=4,
                         steps=20, needles=0, seed=9, append_steps=20)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    batch, max_pages = wl.page_table.shape
    store = B.new_summary_store(batch, spec.h_kv, max_pages, DEV)
    lens0 = [int(x) for x in wl.seq_lens]
    seq, pg = full_pairs(lens0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_build_summaries(d.k_cache, d.page_table, i32(seq), i32(pg), store,
                            status=status)
    seq_lens = d.seq_lens.clone()
    for s in range(spec.append_steps):
        B.locks_append_kv(wl.k_append[s].to(DEV), wl.v_append[s].to(DEV),
                          d.k_cache, d.v_cache, d.page_table, seq_lens, store,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert seq_lens.cpu().tolist() == [L + 20 for L in lens0]
    # the host applies the same appends to its own copy of the cache
    pt = wl.page_table.numpy()
    kc = wl.k_cache.float().numpy().copy()
    for s in range(spec.append_steps):
        for b in range(batch):
            pos = lens0[b] + s
            kc[pt[b, pos // 16], :, pos % 16] = wl.k_append[s, b].float().numpy()
    assert np.array_equal(d.k_cache.float().cpu().numpy(), kc)
    # every page the appends filled holds, byte for byte, the record a
    # fresh build of the final cache writes, and that build (with its fp32
    # values before quantisation) matches the oracle's build
    lens1 = [L + 20 for L in lens0]
    seq1, pg1 = full_pairs(lens1)
    filled = [(b, p) for b, p in zip(seq1, pg1) if p >= lens0[b] // 16]
    assert len(filled) >= batch
    fs = np.array([b for b, _ in filled], np.int32)
    fp = np.array([p for _, p in filled], np.int32)
    fresh = B.new_summary_store(batch, spec.h_kv, max_pages, DEV)
    n = len(filled) * spec.h_kv
    unq = torch.zeros(n * B.UNQUANTISED_FLOATS, dtype=torch.float32,
                      device=DEV)
    tau = torch.zeros(n, dtype=torch.float32, device=DEV)
    B.locks_build_summaries(d.k_cache, d.page_table, i32(fs), i32(fp), fresh,
                            tau, unq, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b, p in filled:
        assert torch.equal(store[b, :, p], fresh[b, :, p]), (b, p)
    check_build(fresh.cpu().numpy()[fs, :, fp].reshape(n, 832),
                unq.view(n, -1).cpu().numpy(), tau.cpu().numpy(),
                kc[pt[fs, fp]].reshape(n, 16, 128), "append")
    # appended tokens are in the cache
    for s in (0, 7, 19):
        for b in range(batch):
            pos = lens0[b] + s
            got_k = d.k_cache[int(pt[b, pos // 16]), :, pos % 16].cpu()
            assert torch.equal(got_k, wl.k_append[s, b])


# ---------------------------------------------------------------------------
# device-detected data errors set status bits, never trap
# ---------------------------------------------------------------------------
def test_device_status_flags():
    spec = W.custom_spec(batch=2, h_q=4, h_kv=1, ctx=16 * 10, k=4, needles=0,
                         seed=3)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    batch, max_pages = wl.page_table.shape
    P = d.k_cache.shape[0]
    bad_pt = d.page_table.clone()
    bad_pt[0, 2] = P + 5
    store = B.new_summary_store(batch, 1, max_pages, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.locks_build_summaries(d.k_cache, bad_pt, i32([0, 0, 1]), i32([1, 2, 99]),
                            store, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == B.DEV_BAD_PAGE_ID | B.DEV_BAD_PAIR
    ws = B.new_workspace(batch, 4, 1, max_pages, max_pages, DEV)
    o = torch.empty(batch, 4, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, 4, dtype=torch.float32, device=DEV)
    idx = i32([[[0, 3, 50, -1]], [[0, 1, 2, 9]]])
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, bad_pt,
                          d.seq_lens, idx, 4, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == B.DEV_BAD_INDEX
    B.locks_clear_status(ws)
    long = i32([16 * max_pages + 1, 16])
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, d.page_table,
                          long, idx, 4, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) & B.DEV_BAD_SEQ_LEN
    B.locks_clear_status(ws)
    idx2 = i32([[[0, 2, 5, 9]], [[0, 1, 2, 9]]])
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, bad_pt,
                          d.seq_lens, idx2, 4, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == B.DEV_BAD_PAGE_ID


@pytest.mark.parametrize("batch,k", [(2, 16), (160, 4)])
def test_device_status_flags_unit_form(batch, k):
    """The same data errors through the decode's unit form (2 units of 16
    list positions: clusters of 4 CTAs; 160 units: a CTA per unit): a
    selected page outside the sequence, a length above the page table, a
    page table entry outside the cache; the step still finishes."""
    spec = W.custom_spec(batch=batch, h_q=4, h_kv=1, ctx=16 * 20, k=k,
                         needles=0, seed=5)
    wl = W.generate(spec, "cpu")
    d = Dev(wl)
    max_pages = wl.page_table.shape[1]
    P = d.k_cache.shape[0]
    ws = B.new_workspace(batch, 4, 1, max_pages, max_pages, DEV)
    o = torch.empty(batch, 4, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(batch, 4, dtype=torch.float32, device=DEV)
    good = np.tile(np.arange(k, dtype=np.int32), (batch, 1, 1))
    idx = good.copy()
    idx[0, 0, 1] = 50                          # beyond the 20 pages
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, d.page_table,
                          d.seq_lens, i32(idx), k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == B.DEV_BAD_INDEX
    B.locks_clear_status(ws)
    long = d.seq_lens.clone()
    long[batch - 1] = 16 * max_pages + 1
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, d.page_table,
                          long, i32(good), k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) & B.DEV_BAD_SEQ_LEN
    B.locks_clear_status(ws)
    bad_pt = d.page_table.clone()
    bad_pt[batch - 1, 2] = P + 5
    B.locks_sparse_decode(d.queries[0], d.k_cache, d.v_cache, bad_pt,
                          d.seq_lens, i32(good), k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == B.DEV_BAD_PAGE_ID
    assert torch.isfinite(lse).all()


def test_native_decoder_status_wide_group_and_empty_sequence():
    """The host-buffer decoder with a group of 16 query heads: an empty
    sequence gives o = 0 and lse = -inf, a page table entry outside the
    cache comes back as LOCKS_DEV_BAD_PAGE_ID in the step's status (sticky
    until cleared), and o / lse equal the eager step's bytes throughout."""
    spec = W.custom_spec(batch=3, h_q=16, h_kv=1, ctx=16 * 40 + 3, k=8,
                         needles=0, seed=47)
    wl = W.generate(spec, "cpu", steps=3)
    d = Dev(wl)
    batch, max_pages = wl.page_table.shape
    lens = [16 * 40 + 3, 0, 16 * 7]
    lens_dev = i32(lens)
    store, _, _, _, _ = gpu_build(d, lens)
    pt = d.page_table.clone()
    good = int(pt[2, 3])
    pt[2, 3] = d.k_cache.shape[0] + 7          # outside the cache
    native = B.LocksDecoder(d.k_cache, d.v_cache, pt, store, spec.h_q,
                            spec.k, graph=True, seq_lens=lens_dev)
    eager = B.LocksDecoder(d.k_cache, d.v_cache, pt, store, spec.h_q, spec.k)
    shape = (batch, spec.h_q, 128)
    qh = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    oh = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(batch, spec.h_q).pin_memory()
    for step in range(3):
        if step == 2:                           # repair the table, clear
            pt[2, 3] = good
            B.locks_clear_status(native.workspace)
            B.locks_clear_status(eager.workspace)
        qh.copy_(wl.queries[step])
        oe, le = eager.step(qh.to(DEV), lens_dev)
        torch.cuda.synchronize()
        _, _, st = native.step_host(qh, lens_dev, oh, lh)
        assert st == (0 if step == 2 else B.DEV_BAD_PAGE_ID), (step, st)
        assert st == eager.status()
        assert torch.equal(oe.cpu(), oh) and torch.equal(le.cpu(), lh)
        assert (oh[1] == 0).all() and torch.isinf(lh[1]).all()
        assert (lh[1] < 0).all()
    native.close()


@pytest.mark.parametrize("rule", ["share_average", "group_max",
                                  "group_mass", "per_head"])
@pytest.mark.parametrize("G", [4, 8])
def test_merge_rules_match_oracle(rule, G):
    """GQA merge rules of the selection on identical scores; per-head
    selection is the selection kernel with every query head as its own
    group."""
    rng = np.random.default_rng(100 + G)
    batch, h_kv, max_pages, k = 5, 2, 400, 14
    lens = [16 * 400, 16 * 123 + 7, 16 * 9, 16 * 250, 16 * 16]
    scores = (rng.normal(0, 3, (batch, h_kv, G, max_pages)) +
              rng.normal(0, 4, (batch, h_kv, 1, max_pages))).astype(np.float32)
    sd = torch.from_numpy(scores).to(DEV)
    if rule == "per_head":
        hq = h_kv * G
        ws = B.new_workspace(batch, hq, hq, max_pages, k, DEV)
        idx = torch.zeros(batch, hq, k, dtype=torch.int32, device=DEV)
        B.locks_select_pages(sd.view(batch, hq, 1, max_pages), i32(lens), hq,
                             k, idx, ws)
        s_rows = scores.reshape(batch, hq, 1, max_pages).astype(np.float64)
        orc = lambda b, h: O.select_one(s_rows[b, h], lens[b], k)   # noqa
        key = lambda b, h, nf: np.log(O.share_average(s_rows[b, h], nf))  # noqa
        n_rows = hq
    else:
        ws = B.new_workspace(batch, h_kv * G, h_kv, max_pages, k, DEV)
        idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
        B.locks_select_pages_merge(sd, i32(lens), h_kv * G, k, rule, idx, ws)
        s64 = scores.astype(np.float64)
        orc = lambda b, h: O.select_one_rule(s64[b, h], lens[b], k, rule)  # noqa
        key = lambda b, h, nf: (O.merge_key(s64[b, h], nf, rule)   # noqa
                                if rule == "group_mass" else
                                np.log(O.merge_key(s64[b, h], nf, rule)))
        n_rows = h_kv
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    for b in range(batch):
        n = -(-lens[b] // 16)
        for h in range(n_rows):
            got = set(int(x) for x in ig[b, h] if x >= 0)
            want = set(orc(b, h))
            if got == want:
                continue
            lk = key(b, h, lens[b] // 16)
            cand = np.arange(1, n - 1)
            order = cand[np.lexsort((cand, -lk[cand]))]
            edge = lk[order[k - 3]]
            for p in got ^ want:
                assert p not in (0, n - 1) and abs(lk[p] - edge) <= 1e-4, \
                    (rule, b, h, p)


@pytest.mark.parametrize("G", [1, 8, 16])
def test_select_more_units_than_sms(G):
    """160 (sequence, KV head) units, more than a GB300 has SMs: the launch
    takes the form compiled for two CTAs per SM (G <= 8) or the one-CTA-per-
    SM form in two waves (G = 16); every unit must still match the oracle's
    selection on the same scores."""
    rng = np.random.default_rng(300 + G)
    batch, h_kv, max_pages, k = 40, 4, 64, 12
    lens = [int(x) for x in rng.integers(0, 16 * max_pages + 1, batch)]
    lens[0], lens[1] = 16 * max_pages, 16 * k
    scores = rng.normal(0, 3, (batch, h_kv, G, max_pages)).astype(np.float32)
    ws = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    B.locks_select_pages(torch.from_numpy(scores).to(DEV), i32(lens),
                         G * h_kv, k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    io = O.select_store(scores.astype(np.float64), lens, k)
    for b in range(batch):
        for h in range(h_kv):
            ok, _ = selection_agrees(ig[b, h], io[b, h],
                                     scores[b, h].astype(np.float64),
                                     lens[b], k, 1e-4)
            assert ok, (b, h, ig[b, h], io[b, h])


@pytest.mark.parametrize("G,max_pages", [(8, 300), (16, 97), (4, 33001),
                                         (2, 33004)])
def test_select_group_sizes_and_long_tables(G, max_pages):
    """Selection with other group sizes and with page tables too long for
    the on-chip key buffer (keys then live in the workspace)."""
    rng = np.random.default_rng(G * 1000 + max_pages)
    batch, h_kv, k = 2, 2, 20
    lens = [16 * max_pages - 3, 16 * (max_pages // 3)]
    scores = rng.normal(0, 3, (batch, h_kv, G, max_pages)).astype(np.float32)
    ws = B.new_workspace(batch, G * h_kv, h_kv, max_pages, k, DEV)
    idx = torch.zeros(batch, h_kv, k, dtype=torch.int32, device=DEV)
    B.locks_select_pages(torch.from_numpy(scores).to(DEV), i32(lens),
                         G * h_kv, k, idx, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    ig = idx.cpu().numpy()
    io = O.select_store(scores.astype(np.float64), lens, k)
    for b in range(batch):
        for h in range(h_kv):
            ok, _ = selection_agrees(ig[b, h], io[b, h],
                                     scores[b, h].astype(np.float64),
                                     lens[b], k, 1e-4)
            assert ok, (b, h, ig[b, h], io[b, h])
