"""Pins of the float64 oracle against what the LOCKS pages and mathematics fix.

None of these checks retypes an oracle formula: each compares the oracle with
a closed form, an independent library routine (the Gram eigensolver of
Eq.(3) against the oracle's SVD of the centred keys), brute force on tiny
inputs, an identity of the pages, or a hand-derived byte fixture.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import locks_oracle as O


def _rng(seed=0):
    return np.random.default_rng(seed)


def _pages(rng, n, B=16, d=128, rank=8, noise=0.05):
    mu = rng.normal(0, 0.5, (n, 1, d))
    W = np.linalg.qr(rng.normal(size=(n, d, rank)))[0]
    A = rng.normal(size=(n, B, rank))
    A = np.linalg.qr(A - A.mean(axis=1, keepdims=True))[0]
    s = 4.0 * 0.6 ** np.arange(rank)
    return mu + (A * s) @ np.swapaxes(W, 1, 2) + rng.normal(0, noise, (n, B, d))


# --------------------------------------------------------------------------
# §5.1 toy example (closed form derived by hand from the printed deltas)
# --------------------------------------------------------------------------
def test_toy_example_closed_form(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "toy_example_5_1.json")))
    deltas = np.array(g["deltas"])
    offset = np.array([0.3, -0.2, 0.5, 1.0])          # any centroid
    keys = deltas + offset
    s = O.page_summary(keys, r=g["r"])
    tr, det = 3.64, 3.62 * 0.02 - 0.18 ** 2
    lam1 = (tr + math.sqrt(tr * tr - 4 * det)) / 2
    lam2 = (tr - math.sqrt(tr * tr - 4 * det)) / 2
    assert s["mu"] == pytest.approx(offset, abs=1e-14)
    assert s["lam"][0] == pytest.approx(lam1, rel=1e-12)
    assert s["lam"][1] == pytest.approx(lam2, rel=1e-10)
    assert np.abs(s["lam"][2:]).max() < 1e-12
    assert lam1 == pytest.approx(3.628978, abs=1e-6)
    assert lam2 == pytest.approx(0.011022, abs=1e-6)
    assert s["tau"] == pytest.approx(lam2, rel=1e-10)   # tau_{j,1} = sigma_2^2
    v = np.array([0.18, lam1 - 3.62, 0.0, 0.0])
    v /= np.linalg.norm(v)
    assert abs(s["V"][:, 0] @ v) == pytest.approx(1.0, abs=1e-12)
    # c_i = V^T delta_i
    assert s["C"][:, 0] == pytest.approx(deltas @ s["V"][:, 0], abs=1e-12)
    # query along the dropped axis: the rank-1 logits cannot tell delta_1
    # from delta_2 (nor delta_3 from delta_4), the exact logits can
    q = np.array(g["query"])
    exact = keys @ q / 2.0
    recon = (q @ s["mu"] + (s["V"].T @ q) @ s["C"].T) / 2.0
    assert abs(exact[1] - exact[0]) == pytest.approx(0.05, abs=1e-12)
    assert abs(recon[1] - recon[0]) < 0.1 * abs(exact[1] - exact[0])
    # Eq.(7): |s_hat - s| <= ||q_perp|| sqrt(tau) / sqrt(d)
    s_hat = O.logsumexp(recon)
    s_ex = O.logsumexp(exact)
    bound = O.eq7_bound(q, s["V"], s["tau"])
    assert abs(s_hat - s_ex) <= bound + 1e-12


# --------------------------------------------------------------------------
# Eq.(3) as printed (eigenpairs of the Gram matrix D D^T, a different library
# routine from the oracle's SVD) and basis properties
# --------------------------------------------------------------------------
def test_summary_matches_gram_eigensolver():
    rng = _rng(1)
    keys = _pages(rng, 24)
    s = O.page_summary(keys, r=8)
    for j in range(keys.shape[0]):
        D = keys[j] - keys[j].mean(axis=0)
        lam, U = np.linalg.eigh(D @ D.T)
        lam, U = lam[::-1], U[:, ::-1]
        # the eigenvalues (the zero one only to rounding of the squared scale)
        assert s["lam"][j] == pytest.approx(np.maximum(lam, 0), rel=1e-9,
                                            abs=1e-13 * lam[0])
        for k in range(8):
            gap = min(lam[k - 1] - lam[k] if k else np.inf, lam[k] - lam[k + 1])
            if gap < 1e-6 * lam[0]:
                continue
            # V = D^T U_r Sigma_r^{-1}, column by column, up to sign
            v = D.T @ U[:, k] / math.sqrt(lam[k])
            assert abs(s["V"][j][:, k] @ v) == pytest.approx(1, abs=1e-9)
            # the sign rule: u_k's largest-magnitude entry is positive
            u = s["C"][j][:, k] / math.sqrt(s["lam"][j][k])
            assert u[np.argmax(np.abs(u))] > 0
        # C = U_r Sigma_r equals D V (c_i = V^T delta_i)
        assert s["C"][j] == pytest.approx(D @ s["V"][j], abs=1e-10)


def test_basis_orthonormal():
    s = O.page_summary(_pages(_rng(2), 16), r=8)
    VtV = np.swapaxes(s["V"], 1, 2) @ s["V"]
    assert np.abs(VtV - np.eye(8)).max() < 1e-10


def test_exact_when_rank_reached():
    """r = 15 = rank of 16 centred keys: reconstructed logits equal the exact
    logits, so s_hat equals the exact page LSE."""
    rng = _rng(3)
    keys = _pages(rng, 12)
    s = O.page_summary(keys, r=15)
    q = rng.normal(size=(4, 128))
    s_hat = O.score_from_summaries(q, s["mu"], s["V"], s["C"])
    s_ex = O.exact_page_lse(q, keys)
    assert np.abs(s_hat - s_ex).max() < 1e-10
    # a planted rank-3 page is exact already at r = 3
    W = np.linalg.qr(rng.normal(size=(128, 3)))[0]
    A = rng.normal(size=(16, 3))
    page = (A - A.mean(0)) @ W.T + rng.normal(size=128)
    s3 = O.page_summary(page[None], r=3)
    assert s3["tau"][0] < 1e-13 * s3["lam"][0, 0]
    assert np.abs(O.score_from_summaries(q, s3["mu"], s3["V"], s3["C"])
                  - O.exact_page_lse(q, page[None])).max() < 1e-10


@pytest.mark.parametrize("r", [1, 2, 4, 8, 12, 15])
def test_eckart_young_tail(r):
    """Retained reconstruction error equals the spectral tail tau_{j,r}."""
    rng = _rng(4 + r)
    keys = _pages(rng, 10)
    s = O.page_summary(keys, r=r)
    for j in range(keys.shape[0]):
        D = keys[j] - keys[j].mean(axis=0)
        err = ((D - s["C"][j] @ s["V"][j].T) ** 2).sum()
        assert err == pytest.approx(s["tau"][j], rel=1e-8, abs=1e-12)
        # and no other orthonormal rank-r basis does better
        Q = np.linalg.qr(rng.normal(size=(128, r)))[0]
        assert ((D - D @ Q @ Q.T) ** 2).sum() >= err - 1e-9


# --------------------------------------------------------------------------
# Eq.(1) identity and Eq.(7) bound
# --------------------------------------------------------------------------
def test_output_error_identity():
    rng = _rng(5)
    for trial in range(20):
        T = 48
        K = rng.normal(size=(T, 128)) * 1.5
        V = rng.normal(size=(T, 128))
        q = rng.normal(size=128)
        keep = rng.random(T) < 0.4
        keep[0] = True
        keep[-1] = False
        o, o_S, eps, vS, vC = O.identity_terms(q, K, V, keep)
        assert np.abs((o - o_S) - eps * (vC - vS)).max() < 1e-12


def test_eq7_bound_unquantised():
    rng = _rng(6)
    keys = _pages(rng, 32)
    s = O.page_summary(keys, r=8)
    q = rng.normal(size=(8, 128)) * 1.3
    s_hat = O.score_from_summaries(q, s["mu"], s["V"], s["C"])
    s_ex = O.exact_page_lse(q, keys)
    for g in range(q.shape[0]):
        for j in range(keys.shape[0]):
            b = O.eq7_bound(q[g], s["V"][j], s["tau"][j])
            assert abs(s_hat[g, j] - s_ex[g, j]) <= b + 1e-12


@pytest.mark.parametrize("r,G,k", [(1, 4, 5), (2, 1, 4), (4, 4, 8),
                                   (8, 3, 6)])
def test_theorem1_coverage_and_output_bounds(r, G, k):
    """§5 Theorem 1 on unquantised summaries, by brute force: with eta the
    largest page-score error (Eq.(6)), the share-average selection from the
    summaries keeps at least exp(-4 eta) of the exact-mass selection's group
    coverage (Eq.(8)) and never more than it (the exact-mass selection
    maximises group coverage); the group-average output error, measured by
    attending over all tokens and over the selected pages, stays within
    2R(1 - gamma_bar(S_hat)) (Eq.(1) per head) and so within
    2R(1 - e^{-4 eta} gamma_bar*) (Eq.(9), reading in eq9_bound)."""
    rng = _rng(40 + r + G + k)
    n = 12
    for _ in range(6):
        keys = _pages(rng, n)
        vals = rng.normal(size=(n, 16, 128))
        s = O.page_summary(keys, r=r)
        q = rng.normal(size=(G, 128)) * rng.uniform(0.5, 3.0)
        s_hat = O.score_from_summaries(q, s["mu"], s["V"], s["C"])
        s_ex = O.exact_page_lse(q, keys)
        t = O.theorem1_terms(s_hat, s_ex, 16 * n, k)
        assert t["eta"] > 0
        assert t["gamma_hat"] >= t["eq8"] - 1e-12
        assert t["gamma_star"] >= t["gamma_hat"] - 1e-12
        R = np.linalg.norm(vals.reshape(-1, 128), axis=1).max()
        o_full, _ = O.attend(q, keys.reshape(-1, 128), vals.reshape(-1, 128))
        sel = t["S_hat"]
        o_sel, _ = O.attend(q, keys[sel].reshape(-1, 128),
                            vals[sel].reshape(-1, 128))
        err = np.linalg.norm(o_sel - o_full, axis=1).mean()
        assert err <= 2 * R * (1 - t["gamma_hat"]) + 1e-12
        assert err <= O.eq9_bound(R, t["eta"], t["gamma_star"]) + 1e-12
    # at r = rank the summaries are exact: eta = 0 and the two selections
    # coincide
    keys = _pages(rng, n)
    s = O.page_summary(keys, r=15)
    q = rng.normal(size=(G, 128))
    t = O.theorem1_terms(O.score_from_summaries(q, s["mu"], s["V"], s["C"]),
                         O.exact_page_lse(q, keys), 16 * n, k)
    assert t["eta"] < 1e-9 and t["S_hat"] == t["S_star"]


def test_exact_store_brute_force():
    """Exact page LSE over the page table, by a direct double loop."""
    rng = _rng(51)
    h_kv, G = 2, 2
    kc = rng.normal(size=(7, h_kv, 16, 128))
    pt = np.array([[3, 0, 5, -1], [6, 1, 2, 4]])
    lens = [16 * 3 + 5, 16 * 4]
    q = rng.normal(size=(2, h_kv * G, 128))
    ex = O.exact_store(q, kc, pt, lens, h_kv)
    for b in range(2):
        for h in range(h_kv):
            for g in range(G):
                for j in range(4):
                    if j < lens[b] // 16:
                        z = [float(q[b, h * G + g] @ kc[pt[b, j], h, i])
                             / math.sqrt(128) for i in range(16)]
                        ref = math.log(sum(math.exp(x) for x in z))
                        assert abs(ex[b, h, g, j] - ref) < 1e-9
                    else:
                        assert np.isnan(ex[b, h, g, j])


def _brute_rule_select(s, L, k, rule):
    """Top-(k-2) subset by brute force with the rule's per-page value
    computed by plain loops (ties: lexicographically smallest pages)."""
    n, nf, G = -(-L // 16), L // 16, len(s)
    if n <= k:
        return list(range(n))
    z = [sum(math.exp(s[g][jj]) for jj in range(nf)) for g in range(G)]
    val = []
    for j in range(nf):
        fr = [math.exp(s[g][j]) / z[g] for g in range(G)]
        if rule == "share_average":
            val.append(sum(fr) / G)
        elif rule == "group_max":
            val.append(max(fr))
        else:
            val.append(math.log(sum(math.exp(s[g][j]) for g in range(G))))
    best, best_key = None, None
    for sub in itertools.combinations(range(1, n - 1), k - 2):
        vals = sorted((val[j] for j in sub), reverse=True)
        key = (tuple(vals), tuple(-j for j in sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return sorted([0, n - 1] + list(best))


@pytest.mark.parametrize("rule", O.MERGE_RULES)
def test_merge_rules_match_brute_force(rule):
    rng = _rng(61)
    for trial in range(20):
        G = int(rng.integers(1, 5))
        n = int(rng.integers(3, 10))
        L = 16 * n - int(rng.integers(0, 2)) * int(rng.integers(1, 15))
        k = int(rng.integers(2, n + 1))
        s = rng.normal(0, 2, (G, n))
        assert O.select_one_rule(s, L, k, rule) == \
            _brute_rule_select(s.tolist(), L, k, rule), (trial, rule)


def test_share_average_maximises_group_coverage():
    """The notes' Corollary 3 (§4.2 design discussion): among selections
    shared by the group, ranking by the share-average of the exact masses
    maximises the group-average coverage; per-head selection bounds every
    head's coverage from above; with G = 1 the rules coincide."""
    rng = _rng(62)
    for trial in range(40):
        G = int(rng.integers(2, 6))
        n = int(rng.integers(6, 30))
        k = int(rng.integers(3, n))
        s = rng.normal(0, 2.5, (G, n)) + rng.normal(0, 1, (1, n))
        cov = {r: O.head_coverage(s, O.select_one_rule(s, 16 * n, k, r), n)
               for r in O.MERGE_RULES}
        for r in O.MERGE_RULES:
            assert cov["share_average"].mean() >= cov[r].mean() - 1e-12
        for g in range(G):
            own = O.head_coverage(s[g:g + 1],
                                  O.select_one(s[g:g + 1], 16 * n, k), n)[0]
            for r in O.MERGE_RULES:
                assert own >= cov[r][g] - 1e-12
    s1 = rng.normal(size=(1, 25))
    sels = {tuple(O.select_one_rule(s1, 16 * 25, 7, r)) for r in O.MERGE_RULES}
    assert len(sels) == 1


def test_variant_record_bytes_by_hand():
    """Variant record codec against bytes worked out by hand from the
    layout rule (include/locks.h, variant records): rank 4 with a 2-bit
    basis puts the codes of dims 0, 8, 16, 24 of component 0 into byte 0
    (two bits each: e = 0, h = 0/1, k-steps 0/1), dim 1 (e = 1) into byte 2,
    component 1's slot 32 bytes further on; coefficients go by scorer lane,
    centroid codes in the shipped order, scales in the 64-byte block."""
    r, vb = 4, 2
    off = O.variant_layout(r, vb)
    assert (off["C"], off["MU"], off["S"], off["SMU"], off["payload"],
            off["stride"]) == (128, 192, 320, 332, 362, 384)
    Vq = np.zeros((128, r), np.int8)
    Vq[0] = [1, -1, 0, 1]      # 0b01, 0b11, 0b00, 0b01
    Vq[8, 0] = -1              # 0b11 at bits 2-3 of byte 0
    Vq[16, 0] = 1              # 0b01 at bits 4-5
    Vq[1, 0] = -2              # 0b10 at bits 0-1 of byte 2
    Vq[64, 0] = 1              # k-step 4: second word of the slot, byte 4
    Vq[2, 0] = -1              # t = 1: the next slot, byte 8
    q = dict(Vq=Vq, C8=np.arange(-32, 32, dtype=np.int8).reshape(16, r),
             mu8=np.full(128, -3, np.int8),
             sV=np.array([1, 2, 0.5, 0.25], np.float16),
             sC=np.arange(16, dtype=np.float16) / 8,
             smu=np.float16(3.0))
    rec = O.encode_variant(q, r, vb)
    assert rec[0] == 0b00011101 and rec[2] == 0b10 and rec[4] == 1
    assert rec[8] == 0b11 and rec[32] == 0b11 and rec[64] == 0
    assert rec[96] == 1
    # C[0][0..2], C[8][0], C[1][0] (excess-128)
    assert (rec[128], rec[129], rec[132], rec[130], rec[136]) == (
        96, 97, 98, 128, 100)
    assert (rec[192:320] == 125).all()                        # mu = -3
    f16 = lambda x: np.float16(x).tobytes()
    assert rec[320:322].tobytes() == f16(1)                   # sV[0]
    assert rec[336:338].tobytes() == f16(0.5)                 # sV[2]
    assert rec[324:326].tobytes() == f16(0)                   # sC[0]
    assert rec[328:330].tobytes() == f16(1)                   # sC[8]
    assert rec[340:342].tobytes() == f16(0.25)                # sC[2]
    assert rec[332:334].tobytes() == f16(3)                   # smu
    d = O.decode_variant(rec, r, vb)
    for key in ("Vq", "C8", "mu8"):
        assert (d[key] == q[key]).all()
    assert (d["sC"] == q["sC"]).all() and d["smu"] == q["smu"]

    # rank 15, 8-bit basis: one byte per code (excess-128), 32 bytes of
    # coefficients per lane row g, sV[8..14] in the groups' last bytes
    r, vb = 15, 8
    off = O.variant_layout(r, vb)
    assert (off["C"], off["MU"], off["S"], off["SMU"], off["stride"]) == (
        1920, 2176, 2304, 2366, 2368)
    Vq = np.zeros((128, r), np.int8)
    Vq[0, 0], Vq[1, 0], Vq[8, 0], Vq[16, 0], Vq[2, 0] = 5, 6, 7, 8, 9
    Vq[0, 14] = -127
    C8 = np.zeros((16, r), np.int8)
    C8[0, 14], C8[9, 9] = 11, -12
    q = dict(Vq=Vq, C8=C8, mu8=np.zeros(128, np.int8),
             sV=np.arange(1, 16, dtype=np.float16),
             sC=np.ones(16, np.float16), smu=np.float16(0.5))
    rec = O.encode_variant(q, r, vb)
    assert (rec[0], rec[1], rec[2], rec[4], rec[32], rec[1792]) == (
        133, 134, 135, 136, 137, 1)
    assert rec[1920 + 26] == 139 and rec[1920 + 39] == 116
    assert rec[1920 + 27] == 128                   # component 15: padding
    assert rec[2364:2366].tobytes() == f16(15)     # sV[14]
    assert rec[2318:2320].tobytes() == f16(10)     # sV[9]
    assert rec[2366:2368].tobytes() == f16(0.5)    # smu
    d = O.decode_variant(rec, r, vb)
    assert (d["Vq"] == Vq).all() and (d["C8"] == C8).all()
    assert (d["sV"] == q["sV"]).all()

    # rank 12, 4-bit basis: components 4..7 of a coefficient row share one
    # word per lane for both tokens g and g + 8
    r, vb = 12, 4
    off = O.variant_layout(r, vb)
    assert (off["C"], off["MU"], off["S"], off["SMU"], off["stride"]) == (
        768, 960, 1088, 1150, 1152)
    Vq = np.zeros((128, r), np.int8)
    Vq[0, 0], Vq[8, 0], Vq[16, 0], Vq[1, 0] = 3, -2, -7, 1
    C8 = np.zeros((16, r), np.int8)
    C8[8, 6], C8[3, 9] = 21, -22
    q = dict(Vq=Vq, C8=C8, mu8=np.zeros(128, np.int8),
             sV=np.ones(r, np.float16), sC=np.ones(16, np.float16),
             smu=np.float16(1))
    rec = O.encode_variant(q, r, vb)
    # byte 0: dim 0 low nibble, dim 8 (h = 1) high nibble; byte 1: dim 16
    assert rec[0] == 0x3 | (0xE << 4) and rec[1] == 0x9 and rec[2] == 1
    assert rec[768 + 22] == 149 and rec[768 + 75] == 106
    d = O.decode_variant(rec, r, vb)
    assert (d["Vq"] == Vq).all() and (d["C8"] == C8).all()


def test_variant_r8_int4_is_the_shipped_summary():
    """Rank 8 with a 4-bit basis quantises exactly as the shipped record
    (same codes and scales, same page scores); finer basis bits reconstruct
    the unquantised basis more closely."""
    rng = _rng(71)
    keys = _pages(rng, 20).astype(np.float32)
    q8, _ = O.build_page(keys)
    qv, _ = O.build_page_variant(keys, 8, 4)
    for a, b in (("V4", "Vq"), ("C8", "C8"), ("mu8", "mu8")):
        assert (q8[a] == qv[b]).all()
    for a in ("sV", "sC", "smu"):
        assert (np.asarray(q8[a]).view(np.uint16) ==
                np.asarray(qv[a]).view(np.uint16)).all()
    # the (8, 4) variant record is the shipped record, byte for byte
    assert np.array_equal(O.encode_variant(qv, 8, 4), O.encode_records(q8))
    qh = rng.normal(size=(4, 128))
    rec = O.decode_variant(O.encode_variant(qv, 8, 4), 8, 4)
    assert np.array_equal(O.score_from_summaries(qh, *O.dequantize(q8)),
                          O.score_from_summaries(qh, *O.dequantize(rec)))
    err = {}
    for vb in O.VARIANT_BITS:
        q, s = O.build_page_variant(keys, 8, vb)
        _, V, _ = O.dequantize(q)
        err[vb] = np.abs(V - s["V"]).mean()
    assert err[8] < err[4] < err[2]


def test_carrier_retention_counts():
    idx = np.array([[[0, 3, 9, -1]], [[0, 1, 2, 7]]])
    car = np.array([[[3, 5]], [[7, -1]]])
    assert O.carrier_retention(idx, car) == pytest.approx(2 / 3)


# --------------------------------------------------------------------------
# Selection: brute force, ties, degenerate cases (Eq.(5) and sink/recent)
# --------------------------------------------------------------------------
def _brute_select(s_hat, L, k):
    n = -(-L // 16)
    if n <= k:
        return list(range(n))
    nf = L // 16
    G = len(s_hat)
    m = []
    for j in range(nf):
        acc = 0.0
        for g in range(G):
            z = sum(math.exp(s_hat[g][jj]) for jj in range(nf))
            acc += math.exp(s_hat[g][j]) / z
        m.append(acc / G)
    best, best_key = None, None
    for sub in itertools.combinations(range(1, n - 1), k - 2):
        key = (sum(m[j] for j in sub), tuple(-j for j in sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return sorted([0, n - 1] + list(best))


@pytest.mark.parametrize("G", [1, 3])
def test_select_matches_brute_force(G):
    rng = _rng(7 + G)
    for trial in range(40):
        n = int(rng.integers(3, 13))
        L = 16 * n - int(rng.integers(0, 16))
        k = int(rng.integers(2, n + 1))
        s_hat = rng.normal(0, 2.0, (G, n))
        assert O.select_one(s_hat, L, k) == _brute_select(s_hat, L, k)


def test_select_ties_and_degenerate():
    s = np.zeros((2, 10))
    assert O.select_one(s, 160, 5) == [0, 1, 2, 3, 9]   # equal mass: low index
    assert O.select_one(s, 0, 4) == []
    assert O.select_one(s, 5, 4) == [0]                 # one partial page
    assert O.select_one(s, 17, 4) == [0, 1]
    assert O.select_one(s, 160, 10) == list(range(10))
    assert O.select_one(s, 160, 2) == [0, 9]


def test_group_of_one_ranks_by_score():
    rng = _rng(9)
    s_hat = rng.normal(size=(1, 40))
    sel = O.select_one(s_hat, 640, 10)
    mid = [j for j in sel if j not in (0, 39)]
    order = sorted(range(1, 39), key=lambda j: (-s_hat[0, j], j))
    assert sorted(order[:8]) == mid


def test_mass_fractions_sum_to_one():
    rng = _rng(10)
    s_hat = rng.normal(0, 3, (4, 50))
    assert O.mass_fractions(s_hat, 50).sum(axis=1) == pytest.approx(1, abs=1e-12)
    assert O.share_average(s_hat, 50).sum() == pytest.approx(1, abs=1e-12)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
def test_attend_brute_force():
    rng = _rng(11)
    q = rng.normal(size=(2, 8))
    K = rng.normal(size=(5, 8))
    V = rng.normal(size=(5, 8))
    o, lse = O.attend(q, K, V)
    for g in range(2):
        logits = [sum(q[g][i] * K[t][i] for i in range(8)) / math.sqrt(8)
                  for t in range(5)]
        z = sum(math.exp(x) for x in logits)
        assert lse[g] == pytest.approx(math.log(z), abs=1e-12)
        for i in range(8):
            ref = sum(math.exp(logits[t]) / z * V[t][i] for t in range(5))
            assert o[g][i] == pytest.approx(ref, abs=1e-12)


def test_all_pages_selected_equals_dense():
    rng = _rng(12)
    P, h_kv, G = 10, 2, 2
    kc = rng.normal(size=(P, h_kv, 16, 128))
    vc = rng.normal(size=(P, h_kv, 16, 128))
    pt = np.array([[3, 7, 1, 0, -1], [2, 9, 8, 5, 4]])
    lens = np.array([55, 80])
    q = rng.normal(size=(2, h_kv * G, 128))
    s_hat = rng.normal(size=(2, h_kv, G, 5))
    idx = O.select_store(s_hat, lens, 8)
    o1, l1 = O.sparse_decode(q, kc, vc, pt, lens, idx)
    o2, l2 = O.dense_decode(q, kc, vc, pt, lens)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12


# --------------------------------------------------------------------------
# Paged gather (notes §2 and Algorithm 2: attention over the selected pages'
# tokens, found through the page table) and the full-page score cut (a
# summary exists only for a page that has filled, notes §2 Fig. 1)
# --------------------------------------------------------------------------
def _paged_case(seed=71):
    rng = _rng(seed)
    P, h_kv, G, max_pages = 11, 2, 3, 5
    kc = rng.normal(size=(P, h_kv, 16, 128))
    vc = rng.normal(size=(P, h_kv, 16, 128))
    # non-identity tables: no logical page maps to its own index
    pt = np.array([[7, 2, 9, 4, 0],
                   [3, 10, 6, 8, 1],
                   [5, 1, 0, -1, -1],
                   [8, 6, 7, 9, 2]], np.int32)
    lens = np.array([16 * 3 + 5, 16 * 5, 0, 1])
    q = rng.normal(size=(4, h_kv * G, 128))
    # selections: out of order, -1 padded, the partial page included or not
    idx = np.array([[[3, 0, 1, -1], [0, 2, 3, -1]],
                    [[4, 0, 2, 1], [0, 4, -1, -1]],
                    [[-1, -1, -1, -1], [-1, -1, -1, -1]],
                    [[0, -1, -1, -1], [-1, 0, -1, -1]]], np.int32)
    return kc, vc, pt, lens, q, idx, h_kv, G


def _token_loop_attention(q, kc, vc, pt, L, pages, h, G):
    """Attention by a loop over the sequence's token positions: token t lives
    in logical page t // 16, slot t % 16, physical page pt[t // 16]; it is
    attended when its logical page is selected."""
    sel = {int(p) for p in pages if p >= 0}
    toks = [t for t in range(int(L)) if t // 16 in sel]
    o = np.zeros((G, 128))
    lse = np.full(G, -np.inf)
    for g in range(G):
        if not toks:
            continue
        z = [float(np.dot(q[h * G + g], kc[pt[t // 16], h, t % 16]))
             / math.sqrt(128) for t in toks]
        m = max(z)
        w = [math.exp(x - m) for x in z]
        tot = sum(w)
        lse[g] = m + math.log(tot)
        for wi, t in zip(w, toks):
            o[g] += (wi / tot) * vc[pt[t // 16], h, t % 16]
    return o, lse


def test_paged_gather_by_token_loop():
    kc, vc, pt, lens, q, idx, h_kv, G = _paged_case()
    o, lse = O.sparse_decode(q, kc, vc, pt, lens, idx)
    od, ld = O.dense_decode(q, kc, vc, pt, lens)
    for b in range(len(lens)):
        n = -(-int(lens[b]) // 16)
        for h in range(h_kv):
            ro, rl = _token_loop_attention(q[b], kc, vc, pt[b], lens[b],
                                           idx[b, h], h, G)
            sl = slice(h * G, (h + 1) * G)
            assert np.abs(o[b, sl] - ro).max() < 1e-12, (b, h)
            assert np.array_equal(np.isinf(lse[b, sl]), np.isinf(rl))
            fin = np.isfinite(rl)
            assert np.abs(lse[b, sl][fin] - rl[fin]).max(initial=0) < 1e-12
            ro, rl = _token_loop_attention(q[b], kc, vc, pt[b], lens[b],
                                           range(n), h, G)
            assert np.abs(od[b, sl] - ro).max() < 1e-12, (b, h)
    # the empty sequence attends nothing: o = 0, lse = -inf
    assert (o[2] == 0).all() and np.isneginf(lse[2]).all()
    # a one-token sequence attends that token alone: o_g = v_0
    assert np.abs(o[3, :G] - vc[pt[3, 0], 0, 0]).max() < 1e-12


def _reconstructed_page_lse(q, rec):
    """LSE over one page's tokens of q . k_hat_i / sqrt(d), with the keys
    reconstructed from the record first: k_hat_i = mu_hat + V_hat c_hat_i."""
    mu, V, C = O.dequantize(O.decode_records(rec))
    z = [float(np.dot(q, mu + V @ C[i])) / math.sqrt(128) for i in range(16)]
    m = max(z)
    return m + math.log(sum(math.exp(x - m) for x in z))


def test_score_store_cut_and_head_groups():
    rng = _rng(72)
    P, h_kv, G, max_pages = 9, 2, 3, 4
    keys = np.stack([_pages(rng, h_kv) for _ in range(P)]).astype(np.float32)
    pt = np.array([[4, 1, 7, 2], [8, 3, 0, 6], [5, 0, 1, 2]], np.int32)
    lens = np.array([16 * 3 + 7, 16 * 4, 15])
    seq_ids = [0, 0, 0, 0, 1, 1, 1, 1]
    page_ids = [0, 1, 2, 3, 0, 1, 2, 3]
    # records for every slot, the partial pages' too, so that a store read
    # past the full pages would find a well-formed record
    store, _ = O.build_summaries(keys, pt, seq_ids, page_ids, 3, max_pages)
    store[2, :, 0] = store[0, :, 1]
    q = rng.normal(size=(3, h_kv * G, 128))
    s = O.score_store(q, store, lens)
    assert s.shape == (3, h_kv, G, max_pages)
    for b in range(3):
        nf = int(lens[b]) // 16
        for h in range(h_kv):
            for g in range(G):
                for j in range(max_pages):
                    if j >= nf:
                        assert np.isnan(s[b, h, g, j]), (b, h, g, j)
                        continue
                    ref = _reconstructed_page_lse(q[b, h * G + g],
                                                  store[b, h, j])
                    assert abs(s[b, h, g, j] - ref) < 1e-9, (b, h, g, j)


def test_planted_gather_and_cut_mistakes_are_caught(monkeypatch):
    orig_gather = O.gather_tokens

    def gather_variant(ignore_table=False, extra=0, keep_pad=False):
        def f(k_cache, v_cache, page_table, b, h, pages, seq_len):
            Ks, Vs = [], []
            for p in pages:
                if p < 0 and not keep_pad:
                    continue
                ntok = min(16, int(seq_len) - 16 * int(p) + extra)
                if ntok <= 0:
                    continue
                phys = int(p) if ignore_table else int(page_table[b][p])
                Ks.append(np.asarray(k_cache[phys, h, :ntok], np.float64))
                Vs.append(np.asarray(v_cache[phys, h, :ntok], np.float64))
            if not Ks:
                return np.zeros((0, 128)), np.zeros((0, 128))
            return np.concatenate(Ks), np.concatenate(Vs)
        return f

    for plant in (dict(ignore_table=True), dict(extra=1), dict(extra=-1),
                  dict(keep_pad=True)):
        monkeypatch.setattr(O, "gather_tokens", gather_variant(**plant))
        with pytest.raises(AssertionError):
            test_paged_gather_by_token_loop()
    monkeypatch.setattr(O, "gather_tokens", orig_gather)
    test_paged_gather_by_token_loop()

    def score_store_variant(ceil_cut=False, interleave=False):
        def f(q, store, seq_lens):
            q = np.asarray(q, np.float64)
            batch, h_kv, max_pages, _ = store.shape
            G = q.shape[1] // h_kv
            out = np.full((batch, h_kv, G, max_pages), np.nan)
            for b in range(batch):
                L = int(seq_lens[b])
                nf = -(-L // 16) if ceil_cut else L // 16
                for h in range(h_kv):
                    if nf == 0:
                        continue
                    mu, V, C = O.dequantize(O.decode_records(store[b, h, :nf]))
                    heads = [g * h_kv + h for g in range(G)] if interleave \
                        else list(range(h * G, (h + 1) * G))
                    out[b, h, :, :nf] = O.score_from_summaries(
                        q[b, heads], mu, V, C)
            return out
        return f

    for plant in (dict(ceil_cut=True), dict(interleave=True)):
        monkeypatch.setattr(O, "score_store", score_store_variant(**plant))
        with pytest.raises(AssertionError):
            test_score_store_cut_and_head_groups()


# --------------------------------------------------------------------------
# Quantiser invariants and the byte layout fixture
# --------------------------------------------------------------------------
def test_quantiser_invariants():
    rng = _rng(13)
    V = rng.normal(size=(20, 128, 8)).astype(np.float32)
    V[3, :, 5] = 0.0
    q = O.quantize_summary(np.ones((20, 128), np.float32), V,
                           np.ones((20, 16, 8), np.float32))
    s = q["sV"].astype(np.float32)
    assert q["V4"].min() >= -7 and q["V4"].max() <= 7
    assert (q["sV"][3, 5] == 0) and (q["V4"][3, :, 5] == 0).all()
    amax = np.abs(V).argmax(axis=1)
    for j in range(20):
        for k in range(8):
            if s[j, k] == 0:
                continue
            assert abs(q["V4"][j, amax[j, k], k]) == 7
            err = np.abs(V[j, :, k] - s[j, k] * q["V4"][j, :, k])
            assert err.max() <= 0.5 * s[j, k] * (1 + 1e-3) + 1e-3 * s[j, k]
    assert (q["mu8"] == 127).all() and (q["C8"] == 127).all()
    # overflowing scale saturates at the largest finite fp16
    big = O._scale(np.array([1e9], np.float32), 127)
    assert big[0] == np.float16(65504)


def test_per_page_basis_scale():
    """The per-page reading of the basis scale: one fp16 scale for the page,
    fp16(max over every column of |V| / 7), stored once per column."""
    # hand example: column k holds one non-zero entry; page scale
    # fp16(14 / 7) = 2, codes rint(V / 2), halves to even
    V = np.zeros((1, 128, 8), np.float32)
    for k, (d, v) in enumerate([(0, 14.0), (1, 3.5), (2, -7.0), (3, 5.0),
                                (4, 1.0), (5, 3.0), (6, -2.9), (7, 0.0)]):
        V[0, d, k] = v
    mu = np.ones((1, 128), np.float32)
    C = np.ones((1, 16, 8), np.float32)
    q = O.quantize_summary(mu, V, C, vscale="page")
    assert (q["sV"] == np.float16(2.0)).all()
    assert [int(q["V4"][0, k, k]) for k in range(8)] == [7, 2, -4, 2, 0, 2,
                                                         -1, 0]
    col = O.quantize_summary(mu, V, C)
    assert col["sV"][0].tolist() == [2.0, 0.5, 1.0, np.float16(5 / 7),
                                     np.float16(1 / 7), np.float16(3 / 7),
                                     np.float16(np.float32(2.9) / 7), 0.0]
    # random pages: the page scale is the largest column scale (fp16
    # rounding is monotone), the page's largest entry codes to +-7, and
    # every entry is within half a step
    rng = _rng(31)
    V = (rng.normal(size=(30, 128, 8)) * rng.uniform(0.01, 3, (30, 1, 8))
         ).astype(np.float32)
    qp = O.quantize_summary(np.ones((30, 128), np.float32), V,
                            np.ones((30, 16, 8), np.float32), vscale="page")
    qc = O.quantize_summary(np.ones((30, 128), np.float32), V,
                            np.ones((30, 16, 8), np.float32))
    assert (qp["sV"] == qc["sV"].max(axis=-1, keepdims=True)).all()
    s = qp["sV"][:, :1].astype(np.float32)[..., None]
    assert qp["V4"].min() >= -7 and qp["V4"].max() <= 7
    flat = np.abs(V).reshape(30, -1).argmax(axis=1)
    assert (np.abs(qp["V4"].reshape(30, -1)[np.arange(30), flat]) == 7).all()
    assert (np.abs(V - s * qp["V4"]) <= 0.5 * s * (1 + 1e-3)).all()
    # coefficients and centroid do not depend on the basis reading
    assert (qp["C8"] == qc["C8"]).all() and (qp["mu8"] == qc["mu8"]).all()
    with pytest.raises(ValueError):
        O.quantize_summary(mu, V[:1], C, vscale="row")


def test_centroid_fp32_sequential():
    rng = _rng(14)
    k = (rng.integers(-64, 64, (5, 16, 128)) / 8.0).astype(np.float32)
    assert O.centroid_f32(k) == pytest.approx(k.mean(axis=1), abs=0)
    # sequential order is what is stated: one value that rounds away
    x = np.zeros((1, 16, 1), np.float32)
    x[0, 0, 0] = 1.0
    x[0, 1:, 0] = 2.0 ** -25
    seq = np.float32(1.0)
    for t in range(1, 16):
        seq = np.float32(seq + np.float32(2.0 ** -25))
    assert O.centroid_f32(x)[0, 0] == np.float32(seq / 16)


def test_record_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "record_fixture.json")))
    e = g["entries"]
    q = dict(V4=np.zeros((128, 8), np.int8), C8=np.zeros((16, 8), np.int8),
             mu8=np.zeros(128, np.int8), sV=np.zeros(8, np.float16),
             sC=np.zeros(16, np.float16), smu=np.float16(e["smu"]))
    for d, k, v in e["V4"]:
        q["V4"][d, k] = v
    for i, k, v in e["C8"]:
        q["C8"][i, k] = v
    for d, v in e["mu8"]:
        q["mu8"][d] = v
    for k, v in e["sV"]:
        q["sV"][k] = v
    for i, v in e["sC"]:
        q["sC"][i] = v
    q["smu"] = np.array(q["smu"], np.float16)
    rec = O.encode_records(q)
    expect = np.zeros(O.RECORD_BYTES, np.uint8)
    for lo, hi, val in g["defaults"]:
        expect[lo:hi] = val
    for off, val in g["expected_bytes"]:
        expect[off] = val
    assert (rec == expect).all(), np.nonzero(rec != expect)
    back = O.decode_records(rec)
    for key in q:
        assert (np.asarray(back[key]) == np.asarray(q[key])).all(), key


def test_record_byte_accounting():
    """768 B logical payload per page-head at r=8, B=16, d=128, i.e. 9.4% of
    the page's 8 KB of bf16 K/V; with the fp16 scales about one tenth."""
    payload = 128 * 8 // 2 + 16 * 8 + 128
    assert payload == 768
    assert round(100 * payload / (2 * 16 * 128 * 2), 1) == 9.4
    assert O.PAYLOAD_BYTES == payload + 2 * (8 + 16 + 1)
    assert abs(O.PAYLOAD_BYTES / 8192 - 0.1) < 0.001
    assert O.RECORD_BYTES % 16 == 0 and O.RECORD_BYTES >= O.PAYLOAD_BYTES


def test_quantised_score_close_to_exact():
    """End to end on the synthetic key model: quantised r=8 scores track the
    exact page LSE (the page's claim that the summary ranks like exact LSE)."""
    rng = _rng(15)
    keys = _pages(rng, 64)
    kb = keys.astype(np.float32)
    q8, s = O.build_page(kb)
    mu, V, C = O.dequantize(O.decode_records(O.encode_records(q8)))
    qv = rng.normal(size=(4, 128))
    err = np.abs(O.score_from_summaries(qv, mu, V, C)
                 - O.exact_page_lse(qv, kb.astype(np.float64)))
    assert err.max() < 0.1


# --------------------------------------------------------------------------
# Planted mistakes in the oracle are caught by the pins above
# --------------------------------------------------------------------------
def test_planted_mistakes_are_caught(monkeypatch):
    orig = O.score_from_summaries

    def no_centroid(q, mu, V, C):                    # dropped q.mu term
        return orig(q, 0 * mu, V, C)
    monkeypatch.setattr(O, "score_from_summaries", no_centroid)
    with pytest.raises(AssertionError):
        test_exact_when_rank_reached()
    monkeypatch.setattr(O, "score_from_summaries", orig)

    def select_variant(s_hat, L, k, merge, tie_high):
        n = -(-L // 16)
        if n <= k:
            return list(range(n))
        nf = L // 16
        s = np.asarray(s_hat, np.float64)
        m = merge(s, nf)
        cand = np.arange(1, n - 1)
        tie = -cand if tie_high else cand
        top = cand[np.lexsort((tie, -m[cand]))[:k - 2]]
        return sorted([0, n - 1] + top.tolist())

    # ties to the higher index instead of the lower one
    monkeypatch.setattr(O, "select_one", lambda s, L, k: select_variant(
        s, L, k, O.share_average, True))
    with pytest.raises(AssertionError):
        test_select_ties_and_degenerate()
    # averaging raw scores over the group instead of mass fractions (Eq.(5))
    monkeypatch.setattr(O, "select_one", lambda s, L, k: select_variant(
        s, L, k, lambda x, nf: x[:, :nf].mean(axis=0), False))
    with pytest.raises(AssertionError):
        test_select_matches_brute_force(3)
