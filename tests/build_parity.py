"""Checks of GPU-built summary records against the float64 oracle's build.

Shared by the GPU parity tests (small workloads, the 128K bench workload and
the ragged workload).  The oracle's eigenvectors come from a float64 SVD and
the kernel's from an fp32 Jacobi eigensolve, so bytes after the eigensolve
cannot be compared bit for bit; what is compared, and the measured bounds
the tolerances come from (GB300, tiny_4k, llama8b_32k, two 128K sequences
and two ragged_64 sequences with per-page decay U(0.4, 0.8): 207K page-heads):

  * eigenvalues within 1e-5 * max(1, lambda_1); tau within 1e-4
  * centroid codes and scale: bit-exact (the same fp32 rule on both sides)
  * reconstructions C V^T (fp32, before quantisation): relative Frobenius
    error <= 1e-3 on page-heads whose 8th and 9th eigenvalues are separated
    by more than 1e-3 * lambda_1 (measured <= 6.8e-6)
  * basis values, unit columns, on components separated from both
    neighbours by more than 1e-3 * lambda_1, up to sign:
    |V_gpu - V| <= ETA_V (measured <= 1.6e-5)
  * components the oracle zeroes (eigenvalue <= 1e-6 lambda_1) are zero
  * coefficient values on page-heads whose eight components are each
    separated or zeroed: |C_gpu - C| <= ETA_C * sigma_1 (measured <= 4.8e-6 sigma_1)
  * scales (fp16 of absmax / qmax): equal, or one fp16 step apart where the
    oracle's unrounded absmax / qmax lies within the value tolerance of the
    midpoint between the two fp16 values
  * codes: differ by at most one, and only where the oracle's x / s lies
    closer to a rounding boundary (.5) than the value tolerance carried
    through the scale, ETA / s, plus |x / s| * 2^-10 where the two scales
    are one fp16 step apart (measured: every differing code inside it)
"""
import numpy as np

from oracle import locks_oracle as O

ETA_V = 5e-5
ETA_C = 1e-5
GAP = 1e-3
UNQ_FLOATS = 1296       # lam[16], mu[128], V[128][8], C[16][8]


def _split_unq(unq):
    u = np.asarray(unq, np.float64)
    lead = u.shape[:-1]
    return (u[..., :16], u[..., 16:144],
            u[..., 144:1168].reshape(lead + (128, 8)),
            u[..., 1168:].reshape(lead + (16, 8)))


def _f16_step(s16):
    """Distance from each fp16 value to the next one up, as float64."""
    s16 = np.asarray(s16, np.float16)
    up = np.nextafter(s16, np.float16(np.inf))
    return up.astype(np.float64) - s16.astype(np.float64)


def _scale_check(s_g, s_o, absmax_o, qmax, eta, mask, tag):
    """Scales equal, or one fp16 step apart at a rounding midpoint (checked
    where `mask` holds; elsewhere reported as equal)."""
    eq = (s_g.view(np.uint16) == s_o.view(np.uint16)) | ~mask
    if eq.all():
        return eq
    bad = ~eq
    lo = np.minimum(s_g.astype(np.float64), s_o.astype(np.float64))
    hi = np.maximum(s_g.astype(np.float64), s_o.astype(np.float64))
    step = _f16_step(np.minimum(s_g, s_o))
    assert np.all(np.abs((hi - lo) - step)[bad] == 0), \
        (tag, "scales more than one fp16 step apart")
    mid = (lo + hi) / 2
    ratio = np.asarray(absmax_o, np.float64) / qmax
    assert np.all(np.abs(ratio - mid)[bad] <= eta[bad] / qmax + 1e-12), \
        (tag, "scales differ away from an fp16 rounding midpoint")
    return eq


def _code_check(code_g, code_o, x_o, s_o, s_eq, eta, mask, tag):
    """|code difference| <= 1, and only inside the propagated window."""
    d = np.abs(code_g.astype(np.int64) - code_o.astype(np.int64))
    d = np.where(mask, d, 0)
    assert d.max(initial=0) <= 1, (tag, "codes more than one step apart")
    s = s_o.astype(np.float64)
    safe = np.where(s == 0, 1.0, s)
    xs = np.asarray(x_o, np.float32).astype(np.float64) / safe
    frac = np.abs(np.abs(xs - np.floor(xs)) - 0.5)
    win = eta / safe + np.where(s_eq, 0.0, np.abs(xs) * 2.0 ** -10) + 1e-6
    outside = (d > 0) & (frac > win)
    assert not outside.any(), (tag, "a code differs away from a boundary",
                               int(outside.sum()))
    return d


def check_build(records, unq, tau, keys, tag="build"):
    """records uint8 [n][832] built by the GPU, its unquantised dump
    [n][1296] and tau [n], for page-heads whose keys are [n][16][128]
    (float32 holding bf16 values).  Returns a dict of measured deviations."""
    n = len(records)
    q8, s = O.build_page(keys)
    gq = O.decode_records(records)
    lam_g, mu_g, V_g, C_g = _split_unq(unq)
    lam = s["lam"]
    lam1 = lam[:, 0]
    scale1 = np.maximum(1.0, lam1.max())
    # eigenvalues, tau, centroid
    assert np.abs(lam_g - lam).max() <= 1e-5 * scale1, tag
    assert np.abs(np.asarray(tau, np.float64) - s["tau"]).max() <= \
        1e-4 * scale1, tag
    assert np.abs(mu_g - s["mu"]).max() < 1e-6, tag
    assert (gq["mu8"] == q8["mu8"]).all(), tag
    assert (gq["smu"].view(np.uint16) == q8["smu"].view(np.uint16)).all(), tag
    # reconstructions on page-heads with a separated rank-8 subspace
    R_g = C_g @ np.swapaxes(V_g, -1, -2)
    R_o = s["C"] @ np.swapaxes(s["V"], -1, -2)
    nrm = np.linalg.norm(R_o, axis=(-2, -1))
    zero = nrm < 1e-12
    assert (np.linalg.norm(R_g, axis=(-2, -1))[zero] < 1e-6).all(), tag
    gap8 = (lam[:, 7] - lam[:, 8]) / np.maximum(lam1, 1e-30)
    err = np.linalg.norm(R_g - R_o, axis=(-2, -1)) / np.maximum(nrm, 1e-30)
    sub_ok = (gap8 > GAP) & ~zero
    assert err[sub_ok].max(initial=0) <= 1e-3, (tag, float(err[sub_ok].max()))
    # per-component separation
    keep = lam[:, :8] > O.ZERO_TOL * lam1[:, None]
    above = np.concatenate([np.full((n, 1), np.inf), lam[:, :7]], -1)
    rel_gap = np.minimum(above - lam[:, :8], lam[:, :8] - lam[:, 1:9]) / \
        np.maximum(lam1, 1e-30)[:, None]
    comp_ok = (rel_gap > GAP) & keep                         # [n][8]
    # page-heads whose every component is either separated or zeroed
    full = (comp_ok | ~keep).all(axis=-1) & ~zero             # [n]
    # components the oracle zeroes (rank-deficient pages) are zero here too
    zc = ~keep
    assert np.abs(V_g * zc[:, None, :]).max(initial=0) < 1e-6, tag
    assert np.abs(C_g * zc[:, None, :]).max(initial=0) < 1e-6, tag
    # the kept basis columns are orthonormal
    VtV = np.swapaxes(V_g, -1, -2) @ V_g
    kept_all = keep.all(axis=-1)
    assert np.abs(VtV[kept_all] - np.eye(8)).max(initial=0) < 1e-4, tag
    # values up to eigenvector sign
    sgn = np.sign(np.einsum("ndk,ndk->nk", V_g, s["V"]))
    sgn[sgn == 0] = 1
    Vs = V_g * sgn[:, None, :]
    Cs = C_g * sgn[:, None, :]
    dV = np.abs(Vs - s["V"])
    mV = np.broadcast_to(comp_ok[:, None, :], dV.shape)
    assert dV[mV].max(initial=0) <= ETA_V, (tag, float(dV[mV].max()))
    sig1 = np.sqrt(np.maximum(lam1, 0))
    dC = np.abs(Cs - s["C"]) / np.maximum(sig1, 1e-30)[:, None, None]
    assert dC[full].max(initial=0) <= ETA_C, (tag, float(dC[full].max()))
    # basis scales and codes
    V32 = s["V"].astype(np.float32)
    etaV = np.full(comp_ok.shape, ETA_V)
    sv_eq = _scale_check(gq["sV"], q8["sV"], np.abs(V32).max(axis=-2), 7,
                         etaV, comp_ok, tag + " sV")
    dv = _code_check(gq["V4"] * sgn[:, None, :].astype(np.int8), q8["V4"],
                     V32, np.broadcast_to(q8["sV"][:, None, :], V32.shape),
                     np.broadcast_to(sv_eq[:, None, :], V32.shape), ETA_V,
                     mV, tag + " V4")
    # coefficient scales and codes (page-heads with every component separated)
    C32 = s["C"].astype(np.float32)
    etaC = np.broadcast_to((ETA_C * sig1)[:, None], (n, 16))
    sc_eq_all = _scale_check(gq["sC"], q8["sC"], np.abs(C32).max(axis=-1),
                             127, etaC,
                             np.broadcast_to(full[:, None], (n, 16)),
                             tag + " sC")
    mC = np.broadcast_to(full[:, None, None], C32.shape)
    dc = _code_check(gq["C8"] * sgn[:, None, :].astype(np.int8), q8["C8"],
                     C32, np.broadcast_to(q8["sC"][:, :, None], C32.shape),
                     np.broadcast_to(sc_eq_all[:, :, None], C32.shape),
                     (ETA_C * sig1)[:, None, None], mC, tag + " C8")
    return dict(
        n=n, sub_ok=float(sub_ok.mean()), comp_ok=float(comp_ok.mean()),
        full=float(full.mean()), recon=float(err[sub_ok].max(initial=0)),
        dV=float(dV[mV].max(initial=0)), dC=float(dC[full].max(initial=0)),
        v_codes_differ=float((dv > 0)[mV].mean()),
        c_codes_differ=float((dc > 0)[mC].mean()) if full.any() else 0.0)


def check_full_size_build(binding, wl, store, samples, dev, tag):
    """GPU-build parity at full size on sampled (sequence, KV head) pairs.

    `store` holds the full-batch build of every full page.  The sampled
    sequences' pages are built again with the fp32 dump enabled (the same
    kernel on a subset of the pairs); their records must equal the
    full-batch records byte for byte, and they are checked against the
    oracle's build of the same keys with check_build."""
    import torch
    lens = [int(x) for x in wl.seq_lens]
    seqs = sorted({b for b, _ in samples})
    sid = np.array([b for b in seqs for _ in range(lens[b] // 16)], np.int32)
    pid = np.array([p for b in seqs for p in range(lens[b] // 16)], np.int32)
    h_kv = store.shape[1]
    n = len(sid) * h_kv
    again = torch.zeros_like(store)
    unq = torch.zeros(n * UNQ_FLOATS, dtype=torch.float32, device=dev)
    tau = torch.zeros(n, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t_sid = torch.as_tensor(sid, device=dev)
    t_pid = torch.as_tensor(pid, device=dev)
    binding.locks_build_summaries(wl.k_cache, wl.page_table, t_sid, t_pid,
                                  again, tau, unq, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in seqs:
        nf = lens[b] // 16
        assert torch.equal(again[b, :, :nf], store[b, :, :nf]), (tag, b)
    unq = unq.view(len(sid), h_kv, UNQ_FLOATS)
    tau = tau.view(len(sid), h_kv)
    out = {}
    for b, h in samples:
        rows = torch.as_tensor(np.nonzero(sid == b)[0], device=dev)
        nf = lens[b] // 16
        phys = wl.page_table[b, :nf].long()
        keys = wl.k_cache[phys, h].float().cpu().numpy()
        out[(b, h)] = check_build(
            store[b, h, :nf].cpu().numpy(),
            unq[rows, h].cpu().numpy(), tau[rows, h].cpu().numpy(), keys,
            f"{tag} seq {b} head {h}")
    return out
