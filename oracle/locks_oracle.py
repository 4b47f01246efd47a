"""LOCKS oracle: a plain, slow float64 CPU statement of the LOCKS decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: only the tests, `__graft_entry__.smoke()` and `bench.py`'s CPU
baseline / reference arm use it.  It shares no code with the CUDA library and
never imports it.

Sources (cited by page title and section, equation or algorithm):
  [notes]  "LOCKS 阅读笔记：为什么 KV Cache 摘要要按「页」而不是按「序列」或
           「全局」来建" (Zhongzhu Zhou, zhongzhuzhou.org, 2026-07-29):
           §3.1 Eq.(1); §4.1 Eq.(2), Eq.(3) and the "存储" (storage)
           paragraph; §4.2 Eq.(4), Eq.(5) and the sink/recent rule;
           §4.3 Algorithm 1; §4.4 Algorithm 2; §5 Eq.(6)-(7); §5.1 toy example.
  [gist]   "Resumo Técnico: LOCKS – Sumários de Chaves Compactos por Página
           para Decodificação Eficiente de Contexto Longo" (gist.science), §2.

Readings taken where the pages are silent:
  * quantiser: symmetric, fp16 scales (basis: one per column; coefficients:
    one per row; centroid: one per page), scale = fp16_rn(fp32(absmax)/qmax),
    code = clamp(rint_fp32(fp32(x)/fp32(scale)), -qmax, qmax), qmax = 7 for
    int4 and 127 for int8; a zero scale gives zero codes; a scale that
    overflows fp16 saturates to 65504.  The quantiser decides integers, so it
    runs in the kernel's precision (fp32), on fp32 copies of the float64
    basis/coefficients.
  * the centroid that is quantised is the fp32 mean with the 16 tokens summed
    in order 0..15, then scaled by 1/16 (the kernel's precision); centring for
    the eigenproblem uses the exact float64 mean of Eq.(2).
  * eigenpairs in descending order; each kept eigenvector u_k is signed so its
    entry of largest magnitude is positive (lowest index on exact ties);
    components with eigenvalue <= 1e-6 * lambda_1 (or lambda_1 == 0) are zeroed.
  * page mass fractions are normalised over all summarised (full) pages of the
    sequence, sink included; sink = logical page 0, recent = the page holding
    the last token; ties in the share-average go to the lower page index.

Pins (tests/test_oracle_pins.py): the §5.1 toy example in closed form, a
cross-check against the Gram-matrix eigensolver of Eq.(3), orthonormal
bases, exactness at r = rank, the Eckart-Young tail, Eq.(1) identity, Eq.(7) bound, brute-force top-k, k >= pages giving dense
attention, attention and page scores by token-position loops through the page
table, and hand-written record fixtures.  Parity unpinned by the pages:
the quantiser's scale dtype/granularity, rounding and sign rule are readings
(pinned only by their own invariants and by hand-written byte fixtures).
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 16
HEAD_DIM = 128
RANK = 8
RECORD_BYTES = 832          # 818 B payload + 14 B zero padding
OFF_V4, OFF_C8, OFF_MU8 = 0, 512, 640
OFF_SV = 768                # start of the 64-byte scale block
PAYLOAD_BYTES = 818
ZERO_TOL = 1e-6


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def logsumexp(x, axis=-1):
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=axis, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        out = np.log(np.sum(np.exp(x - m), axis=axis, keepdims=True)) + m
    return np.squeeze(out, axis=axis)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Build: notes §4.1 Eq.(2)-(3), §4.3 Algorithm 1
# ----------------------------------------------------------------------------
def page_summary(keys: np.ndarray, r: int = RANK):
    """Unquantised rank-r page summary of §4.1 for keys [..., B, d].

    Eq.(2) centres the page on its mean; Eq.(3) takes the eigenpairs of the
    token-space Gram matrix D D^T.  Those are the singular triplets of the
    centred keys themselves: with D = U diag(sigma) W^T, the eigenvectors of
    D D^T are the columns of U with eigenvalues sigma^2, the basis
    V = D^T U_r Sigma_r^{-1} is W_r, and the coefficients c_i = V^T delta_i
    are the rows of U_r Sigma_r.  This statement takes that route (one SVD
    of D), so it does not repeat the Gram/eigensolver steps the kernels take.

    Returns dict with
      mu   [..., d]     page centroid (Eq.(2))
      D    [..., B, d]  centred deviations delta_i = k_i - mu
      lam  [..., B]     sigma_k^2: eigenvalues of D D^T, descending
      U    [..., B, B]  left singular vectors (columns), sign-canonicalised
      V    [..., d, r]  orthonormal basis of the top-r directions
      C    [..., B, r]  coefficients, c_i = V^T delta_i
      tau  [...]        spectral tail sum_{k>r} sigma_k^2 (Eckart-Young)
    """
    K = np.asarray(keys, dtype=np.float64)
    mu = K.mean(axis=-2)                                  # Eq.(2)
    D = K - mu[..., None, :]                              # delta_i rows
    U, sigma, Wt = np.linalg.svd(D, full_matrices=False)  # descending sigma
    # sign: each u_k's entry of largest magnitude positive (lowest index on
    # exact ties); w_k flips with it so that D = U diag(sigma) W^T still holds
    piv = np.argmax(np.abs(U), axis=-2)                   # [..., B]
    pv = np.take_along_axis(U, piv[..., None, :], axis=-2)[..., 0, :]
    flip = np.where(pv < 0, -1.0, 1.0)
    U = U * flip[..., None, :]
    Wt = Wt * flip[..., :, None]
    lam = sigma * sigma
    lam1 = lam[..., :1]
    keep = (lam[..., :r] > ZERO_TOL * lam1) & (lam1 > 0)  # [..., r]
    V = np.where(keep[..., None, :],
                 np.ascontiguousarray(np.swapaxes(Wt[..., :r, :], -1, -2)), 0.0)
    C = np.where(keep[..., None, :], U[..., :r] * sigma[..., None, :r], 0.0)
    tau = lam[..., r:].sum(axis=-1)
    return dict(mu=mu, D=D, lam=lam, U=U, V=V, C=C, tau=tau)


def centroid_f32(keys_f32: np.ndarray) -> np.ndarray:
    """fp32 mean with tokens summed in order 0..15 then scaled by 1/16."""
    k = np.asarray(keys_f32, dtype=np.float32)
    acc = np.zeros(k.shape[:-2] + k.shape[-1:], dtype=np.float32)
    for t in range(k.shape[-2]):
        acc = (acc + k[..., t, :]).astype(np.float32)
    return (acc * np.float32(1.0 / k.shape[-2])).astype(np.float32)


def _scale(absmax_f32: np.ndarray, qmax: int) -> np.ndarray:
    s = (np.asarray(absmax_f32, np.float32) / np.float32(qmax)).astype(
        np.float32)
    with np.errstate(over="ignore"):
        s16 = s.astype(np.float16)
    return np.where(np.isinf(s16), np.float16(65504.0), s16).astype(np.float16)


def _codes(x_f32: np.ndarray, s16: np.ndarray, qmax: int) -> np.ndarray:
    s = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (np.asarray(x_f32, np.float32) / s).astype(np.float32)
    c = np.rint(y)
    c = np.where(s == 0, 0.0, c)
    return np.clip(c, -qmax, qmax).astype(np.int8)


VSCALE_MODES = ("column", "page")


def quantize_summary(mu32, V32, C32, vscale="column"):
    """Storage paragraph of §4.1 / Algorithm 1: int4 basis with a per-column
    scale, int8 coefficients with a per-row scale, int8 centroid.

    vscale="page" is the other reading of the basis scale (one fp16 scale
    for the whole page's basis, the absolute maximum over every column; the
    record still stores it once per column, eight equal values)."""
    if vscale not in VSCALE_MODES:
        raise ValueError(f"vscale must be one of {VSCALE_MODES}")
    mu32 = np.asarray(mu32, np.float32)
    V32 = np.asarray(V32, np.float32)
    C32 = np.asarray(C32, np.float32)
    smu = _scale(np.abs(mu32).max(axis=-1), 127)
    mu8 = _codes(mu32, smu[..., None], 127)
    absV = np.abs(V32).max(axis=-2)                                # [..., r]
    if vscale == "page":
        absV = np.broadcast_to(absV.max(axis=-1, keepdims=True), absV.shape)
    sV = _scale(absV, 7)
    V4 = _codes(V32, sV[..., None, :], 7)
    sC = _scale(np.abs(C32).max(axis=-1), 127)
    C8 = _codes(C32, sC[..., :, None], 127)
    return dict(V4=V4, C8=C8, mu8=mu8, sV=sV, sC=sC, smu=smu)


def dequantize(q):
    """(mu_hat [..., d], V_hat [..., d, r], C_hat [..., B, r]) in float64."""
    mu = q["smu"].astype(np.float64)[..., None] * q["mu8"].astype(np.float64)
    Vc = q["V4"] if "V4" in q else q["Vq"]
    V = q["sV"].astype(np.float64)[..., None, :] * Vc.astype(np.float64)
    C = q["sC"].astype(np.float64)[..., :, None] * q["C8"].astype(np.float64)
    return mu, V, C


def build_page(keys_bf16_as_f32: np.ndarray, vscale="column"):
    """Algorithm 1 for full pages, keys [..., 16, 128] holding bf16 values.

    Returns (quantised summary dict, unquantised summary dict)."""
    s = page_summary(keys_bf16_as_f32, RANK)
    q = quantize_summary(centroid_f32(keys_bf16_as_f32),
                         s["V"].astype(np.float32), s["C"].astype(np.float32),
                         vscale)
    return q, s


# ----------------------------------------------------------------------------
# Rank / precision variants (notes §6 ablation: "秩与量化精度" -- int8, int4
# and int2 bases at several ranks).  Same quantiser readings as the shipped
# int4 basis, with qmax = 2^(bits-1) - 1 for the basis codes (1 for int2, 7
# for int4, 127 for int8); coefficients and centroid stay int8.
# ----------------------------------------------------------------------------
VARIANT_RANKS = (4, 8, 12, 15)
VARIANT_BITS = (2, 4, 8)


def quantize_variant(mu32, V32, C32, vbits):
    q = quantize_summary(mu32, np.zeros(np.shape(V32)[:-2] + (1, 1),
                                        np.float32), C32)
    qv = (1 << (vbits - 1)) - 1
    V32 = np.asarray(V32, np.float32)
    sV = _scale(np.abs(V32).max(axis=-2), qv)
    return dict(Vq=_codes(V32, sV[..., None, :], qv), C8=q["C8"],
                mu8=q["mu8"], sV=sV, sC=q["sC"], smu=q["smu"], vbits=vbits)


def build_page_variant(keys_bf16_as_f32, r, vbits):
    """Algorithm 1 at rank r with a `vbits`-bit basis (full pages)."""
    s = page_summary(keys_bf16_as_f32, r)
    return quantize_variant(centroid_f32(keys_bf16_as_f32),
                            s["V"].astype(np.float32),
                            s["C"].astype(np.float32), vbits), s


def variant_layout(r, vbits):
    """Byte offsets of a variant record (include/locks.h, variant records):
    basis codes in per-(component, lane) slots; coefficient codes in the
    order of the scorer's lanes (16 r bytes for r <= 8, 192 for r = 12,
    256 for r = 15); the centroid codes; the 64-byte fp16 scale block.
    `payload` counts the quantised summary's own bytes (codes and scales),
    `stride` the record with its layout padding."""
    off = {"V": 0}
    off["C"] = 16 * r * vbits
    off["MU"] = off["C"] + (16 * r if r <= 8 else 192 if r == 12 else 256)
    off["S"] = off["MU"] + HEAD_DIM
    off["SMU"] = off["S"] + (12 if r <= 8 else 62)
    off["stride"] = off["S"] + 64
    off["payload"] = 16 * r * vbits + 16 * r + HEAD_DIM + 2 * r + 2 * PAGE + 2
    return off


def _variant_v_bits(r, vbits):
    """First bit (within the record) of the basis code V[d][k], [128][r]:
    slot 4k + t holds the 32 codes of dims 16s + 2t + e + 8h (t = (d%8)/2,
    e = d%2, h = (d%16)/8, s = d/16) in 4*vbits bytes; inside the slot, a
    4-bit code sits in word s/2 at bit 16e + 8(s%2) + 4h, a 2-bit code in
    word s/4 at bit 16e + 2(2(s%4) + h), an 8-bit code in byte 4s + 2h + e."""
    d = np.arange(HEAD_DIM)[:, None]
    k = np.arange(r)[None, :]
    t, e, h, s = (d % 8) // 2, d % 2, (d % 16) // 8, d // 16
    base = 32 * vbits * (4 * k + t)
    if vbits == 4:
        inner = 32 * (s // 2) + 16 * e + 8 * (s % 2) + 4 * h
    elif vbits == 2:
        inner = 32 * (s // 4) + 16 * e + 2 * (2 * (s % 4) + h)
    else:
        inner = 8 * (4 * s + 2 * h + e)
    return base + inner


def _variant_c_offsets(r):
    """Byte (within the coefficient region) of C[i][k], [16][r]: the word of
    lane (g = i%8, t) of the scorer.  r <= 8: 4(g r/2 + k/2) + 2(i/8) + k%2;
    r = 15: 32g + 8t + 4(i/8) + 2(k/8) + k%2 with t = (k%8)/2; r = 12: the
    same with 24 bytes per g, except components 4..7, at
    24g + 16 + 4(t-2) + 2(i/8) + k%2."""
    i = np.arange(PAGE)[:, None]
    k = np.arange(r)[None, :]
    g, hi, t = i % 8, i // 8, (k % 8) // 2
    if r <= 8:
        return 4 * (g * (r // 2) + k // 2) + 2 * hi + k % 2
    per = 24 if r == 12 else 32
    main = per * g + 8 * t + 4 * hi + 2 * (k // 8) + k % 2
    if r == 12:
        main = np.where(t >= 2, 24 * g + 16 + 4 * (t - 2) + 2 * hi + k % 2,
                        main)
    return main


def _variant_scale_offsets(r):
    """Bytes (within the scale block) of sV[k] and sC[i]: group t (16 bytes)
    holds sV[2t], sV[2t+1], sC[2t], sC[2t+1], sC[8+2t], sC[9+2t], and for
    r > 8 sV[8+2t], sV[9+2t] in its last four bytes."""
    k = np.arange(r)
    sv = np.where(k < 8, 16 * (k // 2) + 2 * (k % 2),
                  16 * ((k - 8) // 2) + 12 + 2 * (k % 2))
    i = np.arange(PAGE)
    sc = 16 * ((i % 8) // 2) + 4 + 2 * (i % 2) + 4 * (i // 8)
    return sv, sc


def encode_variant(q, r, vbits):
    off = variant_layout(r, vbits)
    Vq = np.asarray(q["Vq"], np.int64)
    lead = Vq.shape[:-2]
    n = int(np.prod(lead)) if lead else 1
    out = np.zeros((n, off["stride"]), np.uint8)
    # basis codes: two's complement (2, 4 bits) or excess-128 (8 bits)
    codes = Vq.reshape(n, HEAD_DIM * r)
    codes = codes + 128 if vbits == 8 else codes & ((1 << vbits) - 1)
    bits = _variant_v_bits(r, vbits).reshape(-1)
    n_words = 4 * r * vbits
    words = np.zeros((n, n_words), np.uint64)
    for j in range(bits.size):       # codes never overlap inside a word
        words[:, bits[j] // 32] |= (codes[:, j].astype(np.uint64)
                                    << np.uint64(bits[j] % 32))
    out[:, :off["C"]] = np.ascontiguousarray(words.astype("<u4")).view(
        np.uint8).reshape(n, -1)
    # coefficient and centroid codes, excess-128 (padding = code 0)
    out[:, off["C"]:off["MU"]] = 128
    c8 = (np.asarray(q["C8"], np.int16).reshape(n, PAGE * r) + 128)
    out[:, off["C"] + _variant_c_offsets(r).reshape(-1)] = c8.astype(np.uint8)
    mu8 = np.asarray(q["mu8"], np.int16).reshape(n, HEAD_DIM) + 128
    out[:, off["MU"] + MU8_OFF - OFF_MU8] = mu8.astype(np.uint8)
    sv_off, sc_off = _variant_scale_offsets(r)
    for offs, key, cnt in ((off["S"] + sv_off, "sV", r),
                           (off["S"] + sc_off, "sC", PAGE),
                           (np.array([off["SMU"]]), "smu", 1)):
        f16 = np.ascontiguousarray(np.asarray(q[key], np.float16).reshape(
            n, cnt).astype("<f2")).view(np.uint8).reshape(n, cnt, 2)
        out[:, offs] = f16[..., 0]
        out[:, offs + 1] = f16[..., 1]
    return out.reshape(lead + (off["stride"],))


def decode_variant(rec, r, vbits):
    off = variant_layout(r, vbits)
    rec = np.ascontiguousarray(np.asarray(rec, np.uint8))
    lead = rec.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    x = rec.reshape(n, off["stride"])
    words = x[:, :off["C"]].copy().view("<u4").astype(np.int64)
    bits = _variant_v_bits(r, vbits)
    raw = (words[:, bits // 32] >> (bits % 32)) & ((1 << vbits) - 1)
    if vbits == 8:
        codes = raw - 128
    else:
        codes = np.where(raw >= (1 << (vbits - 1)), raw - (1 << vbits), raw)
    C8 = x[:, off["C"] + _variant_c_offsets(r)].astype(np.int16) - 128
    mu8 = x[:, off["MU"] + MU8_OFF - OFF_MU8].astype(np.int16) - 128
    sv_off, sc_off = _variant_scale_offsets(r)

    def halves(offs):
        lo = x[:, offs].astype(np.uint16)
        hi = x[:, offs + 1].astype(np.uint16)
        return (lo | (hi << 8)).view(np.float16)
    c = np.ascontiguousarray
    return dict(
        Vq=c(codes.astype(np.int8).reshape(lead + (HEAD_DIM, r))),
        C8=c(C8.astype(np.int8).reshape(lead + (PAGE, r))),
        mu8=c(mu8.astype(np.int8).reshape(lead + (HEAD_DIM,))),
        sV=c(halves(off["S"] + sv_off).reshape(lead + (r,))),
        sC=c(halves(off["S"] + sc_off).reshape(lead + (PAGE,))),
        smu=c(halves(np.array([off["SMU"]]))[:, 0].reshape(lead)),
        vbits=vbits)


# ----------------------------------------------------------------------------
# Record layout (include/locks.h documents the same bytes)
# ----------------------------------------------------------------------------
def _v4_positions():
    d = np.arange(HEAD_DIM)[:, None]
    n = np.arange(RANK)[None, :]
    c = (d % 8) // 2
    e = d % 2
    hi8 = (d % 16) // 8
    s = d // 16
    w, sp = s // 2, s % 2
    word = (4 * n + c) * 4 + w                 # u32 word index 0..127
    shift = 16 * e + 8 * sp + 4 * hi8
    return np.broadcast_to(word, (HEAD_DIM, RANK)), \
        np.broadcast_to(shift, (HEAD_DIM, RANK))


def _c8_offsets():
    i = np.arange(PAGE)[:, None]
    k = np.arange(RANK)[None, :]
    return OFF_C8 + 4 * (4 * (i % 8) + k // 2) + 2 * (i // 8) + k % 2


def _scale_offsets():
    """Byte offsets of the fp16 scales: the 64-byte scale block holds, for
    t = 0..3, 16 bytes at 768 + 16t: sV[2t], sV[2t+1], sC[2t], sC[2t+1],
    sC[8+2t], sC[9+2t], then sMU (t = 0 only) and zero padding."""
    sv = np.array([OFF_SV + 16 * (n // 2) + 2 * (n % 2) for n in range(RANK)])
    sc = np.array([OFF_SV + 16 * ((i % 8) // 2) + 4 + 2 * (i % 2) + 4 * (i // 8)
                   for i in range(PAGE)])
    return sv, sc, OFF_SV + 12


def _mu8_offsets():
    d = np.arange(HEAD_DIM)
    o = d % 16
    c = (o % 8) // 2
    j = (o % 2) + 2 * (o // 8)
    return OFF_MU8 + 32 * c + 4 * (d // 16) + j


SV_OFF, SC_OFF, SMU_OFF = _scale_offsets()
V4_WORD, V4_SHIFT = _v4_positions()
V4_WORD_COLS = np.argsort(V4_WORD.reshape(-1), kind="stable").reshape(128, 8)
C8_OFF = _c8_offsets()
MU8_OFF = _mu8_offsets()


def encode_records(q) -> np.ndarray:
    """Quantised summaries [...] -> uint8 records [..., 832]."""
    lead = q["mu8"].shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    V4 = q["V4"].reshape(n, HEAD_DIM, RANK).astype(np.int64) & 0xF
    flat_s = V4_SHIFT.reshape(-1).astype(np.uint64)
    vals = V4.reshape(n, -1).astype(np.uint64) << flat_s[None, :]
    # each u32 word gathers exactly 8 non-overlapping nibbles
    words = vals[:, V4_WORD_COLS].sum(axis=-1)            # [n][128]
    rec = np.zeros((n, RECORD_BYTES), dtype=np.uint8)
    rec[:, OFF_V4:OFF_V4 + 512] = np.ascontiguousarray(
        words.astype("<u4")).view(np.uint8).reshape(n, 512)
    # int8 codes of C and mu are stored excess-128 (byte = code + 128)
    C8 = (q["C8"].reshape(n, PAGE, RANK).astype(np.int16) + 128).astype(
        np.uint8)
    rec[:, C8_OFF.reshape(-1)] = C8.reshape(n, -1)
    mu8 = (q["mu8"].reshape(n, HEAD_DIM).astype(np.int16) + 128).astype(
        np.uint8)
    rec[:, MU8_OFF] = mu8
    for offs, key, cnt in ((SV_OFF, "sV", RANK), (SC_OFF, "sC", PAGE),
                           (np.array([SMU_OFF]), "smu", 1)):
        f16 = np.ascontiguousarray(q[key].reshape(n, cnt).astype("<f2"))
        b = f16.view(np.uint8).reshape(n, cnt, 2)
        rec[:, offs] = b[..., 0]
        rec[:, offs + 1] = b[..., 1]
    return rec.reshape(lead + (RECORD_BYTES,))


def decode_records(rec: np.ndarray):
    """uint8 records [..., 832] -> quantised summary dict."""
    rec = np.asarray(rec, dtype=np.uint8)
    lead = rec.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    r = rec.reshape(n, RECORD_BYTES)
    words = r[:, :512].copy().view("<u4").astype(np.int64)     # [n][128]
    nib = (words[:, V4_WORD] >> V4_SHIFT) & 0xF                 # [n][128][8]
    V4 = np.where(nib >= 8, nib - 16, nib).astype(np.int8)
    C8 = (r[:, C8_OFF.reshape(-1)].astype(np.int16) - 128).astype(
        np.int8).reshape(n, PAGE, RANK)
    mu8 = (r[:, MU8_OFF].astype(np.int16) - 128).astype(np.int8).reshape(
        n, HEAD_DIM)
    def halves(offs):
        lo = r[:, offs].astype(np.uint16)
        hi = r[:, offs + 1].astype(np.uint16)
        return (lo | (hi << 8)).view(np.float16)
    sV = halves(SV_OFF)
    sC = halves(SC_OFF)
    smu = halves(np.array([SMU_OFF]))[:, 0]
    return dict(V4=V4.reshape(lead + (HEAD_DIM, RANK)),
                C8=C8.reshape(lead + (PAGE, RANK)),
                mu8=mu8.reshape(lead + (HEAD_DIM,)),
                sV=sV.reshape(lead + (RANK,)).astype(np.float16),
                sC=sC.reshape(lead + (PAGE,)).astype(np.float16),
                smu=smu.reshape(lead).astype(np.float16))


def build_summaries(k_cache, page_table, seq_ids, page_ids, batch, max_pages,
                    store=None, vscale="column"):
    """Algorithm 1 over listed (sequence, logical page) pairs, every KV head.

    k_cache [P][h_kv][16][128] (float32 holding bf16 values), page_table
    [batch][max_pages].  Writes records into store [batch][h_kv][max_pages]
    [832] (zero-initialised if None); returns (store, tau [n][h_kv])."""
    k_cache = np.asarray(k_cache, dtype=np.float32)
    h_kv = k_cache.shape[1]
    if store is None:
        store = np.zeros((batch, h_kv, max_pages, RECORD_BYTES), np.uint8)
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    page_ids = np.asarray(page_ids, dtype=np.int64)
    phys = np.asarray(page_table)[seq_ids, page_ids].astype(np.int64)
    keys = k_cache[phys]                                 # [n][h_kv][16][128]
    q, s = build_page(keys, vscale)
    rec = encode_records(q)                              # [n][h_kv][832]
    for h in range(h_kv):
        store[seq_ids, h, page_ids] = rec[:, h]
    return store, s["tau"]


# ----------------------------------------------------------------------------
# Score: notes §4.2 Eq.(4), Algorithm 2
# ----------------------------------------------------------------------------
def score_from_summaries(q, mu_hat, V_hat, C_hat):
    """Eq.(4) for query heads q [G][d] against pages [n] of one KV head:
    s_hat[g][j] = log sum_i exp((q.mu_j + (V_j^T q).c_i) / sqrt(d))."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    qmu = np.einsum("gd,nd->gn", q, mu_hat)
    proj = np.einsum("gd,ndr->gnr", q, V_hat)                # V_j^T q
    logits = (qmu[..., None] + np.einsum("gnr,nir->gni", proj, C_hat)) \
        / math.sqrt(d)
    return logsumexp(logits, axis=-1)


def score_store(q, store, seq_lens):
    """s_hat [batch][h_kv][G][max_pages] (NaN where a page has no summary),
    q [batch][h_q][128] holding bf16 values, store as build_summaries."""
    q = np.asarray(q, dtype=np.float64)
    batch, h_kv, max_pages, _ = store.shape
    G = q.shape[1] // h_kv
    out = np.full((batch, h_kv, G, max_pages), np.nan)
    for b in range(batch):
        nf = int(seq_lens[b]) // PAGE
        if nf == 0:
            continue
        for h in range(h_kv):
            mu, V, C = dequantize(decode_records(store[b, h, :nf]))
            out[b, h, :, :nf] = score_from_summaries(
                q[b, h * G:(h + 1) * G], mu, V, C)
    return out


def exact_page_lse(q, keys):
    """s_j(q) = log sum_{i in P_j} exp(q.k_i / sqrt(d)) (the target of Eq.(4)),
    q [G][d], keys [n][B][d] -> [G][n]."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    return logsumexp(np.einsum("gd,nid->gni", q, keys)
                     / math.sqrt(q.shape[-1]), axis=-1)


# ----------------------------------------------------------------------------
# Select: notes §4.2 Eq.(5) and sink/recent rule, Algorithm 2
# ----------------------------------------------------------------------------
def mass_fractions(s_hat_g, n_full):
    """m_hat_g(j) = exp(s_hat_j(q_g)) / sum_{j'} exp(s_hat_j'(q_g)) over the
    n_full summarised pages; s_hat_g [G][>= n_full] -> [G][n_full]."""
    s = np.asarray(s_hat_g, np.float64)[:, :n_full]
    Z = logsumexp(s, axis=1)
    return np.exp(s - Z[:, None])


def select_one(s_hat_g, seq_len, k):
    """Selected logical pages (ascending) for one (sequence, KV head):
    the sink page 0, the recent page n-1 and the top-(k-2) remaining pages by
    the share-average m_bar_j = (1/G) sum_g m_hat_g(j) (Eq.(5))."""
    n = -(-int(seq_len) // PAGE)
    if n == 0:
        return []
    if n <= k:
        return list(range(n))
    nf = int(seq_len) // PAGE
    m_bar = mass_fractions(s_hat_g, nf).mean(axis=0)
    cand = np.arange(1, n - 1)
    order = np.lexsort((cand, -m_bar[cand]))       # mass desc, index asc
    top = cand[order[:k - 2]]
    return sorted([0, n - 1] + top.tolist())


# GQA merge rules of the notes' §4.2 design discussion and §6 ablation:
# share-average (the shipped rule, Eq.(5)), group-max (pages any head of the
# group gives a large mass fraction: the largest of the heads' fractions)
# and group-mass (the group's pooled page mass: the sum over heads of
# exp(s_hat), without per-head normalisation).  Per-head selection (each
# query head its own set) is select_one on that head alone.
MERGE_RULES = ("share_average", "group_max", "group_mass")


def merge_key(s_hat_g, n_full, rule):
    """Per-page ranking value of a merge rule, [n_full] (monotone in the
    rule's pooled quantity)."""
    s = np.asarray(s_hat_g, np.float64)[:, :n_full]
    if rule == "share_average":
        return mass_fractions(s, n_full).mean(axis=0)
    if rule == "group_max":
        return mass_fractions(s, n_full).max(axis=0)
    if rule == "group_mass":
        return logsumexp(s, axis=0)
    raise ValueError(rule)


def select_one_rule(s_hat_g, seq_len, k, rule):
    """select_one with the candidates ranked by a merge rule's key (ties to
    the lower page)."""
    n = -(-int(seq_len) // PAGE)
    if n == 0:
        return []
    if n <= k:
        return list(range(n))
    nf = int(seq_len) // PAGE
    key = merge_key(s_hat_g, nf, rule)
    cand = np.arange(1, n - 1)
    order = np.lexsort((cand, -key[cand]))
    return sorted([0, n - 1] + cand[order[:k - 2]].tolist())


def head_coverage(s_exact_g, pages, n_full):
    """gamma_g(S) = sum_{j in S} m_g(j) for every head g of the group: the
    exact attention mass over full pages that S keeps, [G]."""
    m = mass_fractions(s_exact_g, n_full)
    sel = [j for j in pages if j < n_full]
    return m[:, sel].sum(axis=1)


def select_store(s_hat, seq_lens, k):
    """idx [batch][h_kv][k] int32, ascending, -1 padded."""
    batch, h_kv = s_hat.shape[:2]
    idx = np.full((batch, h_kv, k), -1, dtype=np.int32)
    for b in range(batch):
        for h in range(h_kv):
            sel = select_one(s_hat[b, h], seq_lens[b], k)
            idx[b, h, :len(sel)] = sel
    return idx


def share_average(s_hat_g, n_full):
    return mass_fractions(s_hat_g, n_full).mean(axis=0)


def exact_store(q, k_cache, page_table, seq_lens, h_kv):
    """Exact page LSE s_j(q_g) of every full page (the quantity Eq.(4)
    estimates; ranking by it is the exact-mass selector the notes compare
    against in §6 Fig. 1(b) and Fig. 2): [batch][h_kv][G][max_pages], NaN
    where a page is not full.  q [batch][h_q][d]; caches as the C ABI."""
    q = np.asarray(q, np.float64)
    batch, max_pages = page_table.shape
    G = q.shape[1] // h_kv
    out = np.full((batch, h_kv, G, max_pages), np.nan)
    for b in range(batch):
        nf = int(seq_lens[b]) // PAGE
        if nf == 0:
            continue
        phys = np.asarray(page_table[b, :nf], np.int64)
        for h in range(h_kv):
            keys = np.asarray(k_cache[phys, h], np.float64)
            out[b, h, :, :nf] = exact_page_lse(q[b, h * G:(h + 1) * G], keys)
    return out


# ----------------------------------------------------------------------------
# Theorem 1 (notes §5): coverage retention and the output-error bound
# ----------------------------------------------------------------------------
def group_coverage(s_exact_g, pages, n_full):
    """gamma_bar(S) = (1/G) sum_g sum_{j in S} m_g(j): the group-average
    attention mass that the page set S keeps, m_g the exact mass fractions
    over the n_full full pages (§5 Theorem 1 (ii))."""
    m = mass_fractions(s_exact_g, n_full).mean(axis=0)
    return float(sum(m[j] for j in pages if j < n_full))


def theorem1_terms(s_hat_g, s_exact_g, seq_len, k):
    """For one (sequence, KV head) of full pages: eta of Eq.(6), the
    coverage of the share-average selection from the summaries (S_hat) and
    of the exact-mass selection (S_star), and the Eq.(8) guarantee
    exp(-4 eta) * gamma_bar(S_star)."""
    nf = int(seq_len) // PAGE
    eta = float(np.abs(np.asarray(s_hat_g)[:, :nf] -
                       np.asarray(s_exact_g)[:, :nf]).max())
    s_hat_sel = select_one(s_hat_g, seq_len, k)
    s_star = select_one(s_exact_g, seq_len, k)
    g_hat = group_coverage(s_exact_g, s_hat_sel, nf)
    g_star = group_coverage(s_exact_g, s_star, nf)
    return {"eta": eta, "S_hat": s_hat_sel, "S_star": s_star,
            "gamma_hat": g_hat, "gamma_star": g_star,
            "eq8": math.exp(-4.0 * eta) * g_star}


def eq9_bound(R, eta, gamma_star):
    """Output-error bound of §5 Theorem 1 (iii).  The printed form
    2R(1 - e^{-4 eta}) gamma_bar* vanishes at eta = 0, where the exact
    selection itself still drops mass; the bound that Eq.(1) and Eq.(8)
    give, and the reading taken here, is 2R(1 - e^{-4 eta} gamma_bar*)."""
    return 2.0 * R * (1.0 - math.exp(-4.0 * eta) * gamma_star)


def carrier_retention(idx, carriers):
    """Fraction of carrier (needle) pages present in the selections:
    idx [batch][h_kv][k], carriers [batch][h_kv][c] logical pages (<0
    ignored) — the key-page retention the notes measure in §6 Fig. 1(b)."""
    idx = np.asarray(idx)
    carriers = np.asarray(carriers)
    hit = tot = 0
    for b in range(carriers.shape[0]):
        for h in range(carriers.shape[1]):
            sel = set(int(x) for x in idx[b, h] if x >= 0)
            for p in carriers[b, h]:
                if p < 0:
                    continue
                tot += 1
                hit += int(p) in sel
    return hit / tot if tot else float("nan")


# ----------------------------------------------------------------------------
# Attention over selected pages: notes §2, Algorithm 2
# ----------------------------------------------------------------------------
def attend(q, K, V):
    """Softmax attention of query heads q [G][d] over tokens K, V [T][d].
    Returns (o [G][d], lse [G]) with natural-log LSE of the logits."""
    q = np.asarray(q, np.float64)
    if K.shape[0] == 0:
        return np.zeros_like(q), np.full(q.shape[0], -np.inf)
    logits = q @ np.asarray(K, np.float64).T / math.sqrt(q.shape[-1])
    lse = logsumexp(logits, axis=1)
    p = np.exp(logits - lse[:, None])
    return p @ np.asarray(V, np.float64), lse


def gather_tokens(k_cache, v_cache, page_table, b, h, pages, seq_len):
    Ks, Vs = [], []
    for p in pages:
        if p < 0:
            continue
        ntok = min(PAGE, int(seq_len) - PAGE * int(p))
        if ntok <= 0:
            continue
        phys = int(page_table[b][p])
        Ks.append(np.asarray(k_cache[phys, h, :ntok], np.float64))
        Vs.append(np.asarray(v_cache[phys, h, :ntok], np.float64))
    if not Ks:
        d = k_cache.shape[-1]
        return np.zeros((0, d)), np.zeros((0, d))
    return np.concatenate(Ks), np.concatenate(Vs)


def sparse_decode(q, k_cache, v_cache, page_table, seq_lens, idx):
    """o [batch][h_q][d], lse [batch][h_q] over the selected pages' tokens;
    idx None means every page (dense decode)."""
    q = np.asarray(q, np.float64)
    batch, h_q, d = q.shape
    h_kv = k_cache.shape[1]
    G = h_q // h_kv
    o = np.zeros((batch, h_q, d))
    lse = np.full((batch, h_q), -np.inf)
    for b in range(batch):
        n = -(-int(seq_lens[b]) // PAGE)
        for h in range(h_kv):
            pages = range(n) if idx is None else idx[b][h]
            K, V = gather_tokens(k_cache, v_cache, page_table, b, h, pages,
                                 seq_lens[b])
            ob, lb = attend(q[b, h * G:(h + 1) * G], K, V)
            o[b, h * G:(h + 1) * G] = ob
            lse[b, h * G:(h + 1) * G] = lb
    return o, lse


def dense_decode(q, k_cache, v_cache, page_table, seq_lens):
    return sparse_decode(q, k_cache, v_cache, page_table, seq_lens, None)


# ----------------------------------------------------------------------------
# Output-error identity and retention bound: notes §3.1 Eq.(1), §5 Eq.(6)-(7)
# ----------------------------------------------------------------------------
def identity_terms(q, K, V, keep_mask):
    """For one query q [d] and tokens K, V [T][d], a keep mask over tokens:
    returns (o, o_S, eps, vbar_S, vbar_Sc): o over every token, o_S over the
    kept tokens only, eps = 1 - gamma_S(q) the attention mass outside S, and
    the attention-weighted means of the kept / dropped values.  (o_S and
    vbar_S coincide by definition; both are returned so a check of Eq.(1)
    reads term by term.)"""
    q = np.asarray(q, np.float64)
    logits = np.asarray(K, np.float64) @ q / math.sqrt(q.shape[-1])
    p = np.exp(logits - logsumexp(logits))
    V = np.asarray(V, np.float64)
    o = p @ V
    pS, pC = p[keep_mask], p[~keep_mask]
    gamma = pS.sum()
    lS = logits[keep_mask]
    wS = np.exp(lS - logsumexp(lS))
    o_S = wS @ V[keep_mask]                 # attention restricted to S
    vS = pS @ V[keep_mask] / gamma
    vC = pC @ V[~keep_mask] / pC.sum()
    return o, o_S, 1.0 - gamma, vS, vC


def eq7_bound(q, V, tau):
    """||q_perp|| sqrt(tau) / sqrt(d), q_perp = q minus its projection on the
    span of the orthonormal basis V [d][r] (Eq.(7), one query, one page)."""
    q = np.asarray(q, np.float64)
    qp = q - V @ (V.T @ q)
    return np.linalg.norm(qp) * math.sqrt(max(tau, 0.0)) / math.sqrt(q.size)
