"""Seeded synthetic decode workloads for the LOCKS sparse paged decode path.

This module only draws inputs: paged bf16 K/V caches, page tables, sequence
lengths and per-step queries with the shapes and structure of the five
workloads below.  It holds none of the method's arithmetic (no summary build,
no scoring, no selection, no attention), so both the CUDA path and the
float64 oracle may consume what it produces.

Key model, per (page, KV head), following the structure the LOCKS reading
notes (zhongzhuzhou.org, 2026-07-29) describe in §1 and §4.1 (a page of B=16
post-RoPE keys whose centred deviations are concentrated in a few directions):

    k_i = mu_j + (A diag(s) W^T)_i + n_i

  * mu_j ~ N(0, 0.5^2 I_128)                  page centroid
  * W    128x8, random orthonormal columns     page-local directions
  * A    16x8, orthonormal columns, each orthogonal to the all-ones vector,
         so the planted component is already centred and its singular values
         are exactly s
  * s_m  = 4 * rho^m, m = 0..7 (rho = 0.6, or per page U(0.4, 0.8))
  * n_i  ~ N(0, 0.05^2 I_128)                 isotropic noise

Values are N(0, 1).  Queries are N(0, I) except for the planted needles: a
needle is one token of one page whose key is replaced by ||k|| * n_hat, and
every step the query of each head of that KV head's group is rebuilt as
q = ||z|| (0.6 n_hat + 0.8 u) with u a unit vector orthogonal to n_hat, so
cos(q, k_needle) = 0.6 exactly.

Layouts (shared with the C ABI, see include/locks.h):
  k_cache, v_cache  bf16 [num_phys_pages][h_kv][16][128]
  page_table        int32 [batch][max_pages]   (-1 past a sequence's pages)
  seq_lens          int32 [batch]
  queries           bf16 [steps][batch][h_q][128]
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

PAGE = 16      # tokens per page (B)
HEAD_DIM = 128  # d
RANK = 8       # planted directions per page (the summary rank r)


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and structure of one synthetic decode workload."""
    name: str
    batch: int
    h_q: int
    h_kv: int
    ctx: int                    # prompt length in tokens (max for ragged)
    k: int                      # page budget per (sequence, KV head)
    steps: int                  # decode steps
    needles: int                # needle pages per (sequence, KV head)
    seed: int
    contiguous: bool = False    # contiguous page table instead of a shuffle
    decay: float = 0.6          # spectral decay rho of the planted component
    decay_range: Optional[tuple] = None   # per-page rho ~ U(lo, hi) if set
    ragged_min: Optional[int] = None      # lengths ~ U{ragged_min..ctx}
    append_steps: int = 0       # tokens appended (one per decode step)
    k_sweep: tuple = ()

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv


# The five workloads the LOCKS decode path is specified and measured on.
SPECS = {
    # single-layer decode, 8q/2kv, 4K context, budget 16 pages, 8 steps
    "tiny_4k": WorkloadSpec("tiny_4k", batch=1, h_q=8, h_kv=2, ctx=4096,
                            k=16, steps=8, needles=1, seed=0,
                            contiguous=True),
    # Llama-3.1-8B-shaped layer: 32q/8kv, batch 8 at 32K, k=64, 64 steps
    "llama8b_32k": WorkloadSpec("llama8b_32k", batch=8, h_q=32, h_kv=8,
                                ctx=32768, k=64, steps=64, needles=4,
                                seed=1),
    # long-context bandwidth case: batch 32 at 128K, k=128, 32 steps
    "llama8b_128k": WorkloadSpec("llama8b_128k", batch=32, h_q=32, h_kv=8,
                                 ctx=131072, k=128, steps=32, needles=1,
                                 seed=2),
    # ragged serving batch: 64 sequences, 4K..128K, budget sweep
    "ragged_64": WorkloadSpec("ragged_64", batch=64, h_q=32, h_kv=8,
                              ctx=131072, k=64, steps=16, needles=1, seed=3,
                              decay_range=(0.4, 0.8), ragged_min=4096,
                              k_sweep=(16, 32, 64, 128, 256)),
    # Llama-3.1-70B-shaped layer, build + 256 decode steps with appends
    "llama70b_128k_append": WorkloadSpec("llama70b_128k_append", batch=8,
                                         h_q=64, h_kv=8, ctx=131072, k=128,
                                         steps=256, needles=1, seed=4,
                                         append_steps=256),
}


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    k_cache: torch.Tensor       # bf16 [P][h_kv][16][128]
    v_cache: torch.Tensor       # bf16 [P][h_kv][16][128]
    page_table: torch.Tensor    # int32 [batch][max_pages]
    seq_lens: torch.Tensor      # int32 [batch] (prompt lengths)
    queries: torch.Tensor       # bf16 [steps][batch][h_q][128]
    needle_pages: torch.Tensor  # int64 [batch][h_kv][needles] logical page ids
    needle_dirs: torch.Tensor   # float32 [batch][h_kv][needles][128]
    # appended tokens (one per step), bf16 [append_steps][batch][h_kv][128]
    k_append: Optional[torch.Tensor] = None
    v_append: Optional[torch.Tensor] = None

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    @property
    def num_phys_pages(self) -> int:
        return self.k_cache.shape[0]


def _seed_for(base: int, *parts: int) -> int:
    """Deterministic sub-stream seed (SplitMix64 over the parts)."""
    x = (base * 0x9E3779B97F4A7C15 + 0x632BE59BD9B4E019) & (2**64 - 1)
    for p in parts:
        x = (x ^ ((p + 0x9E3779B97F4A7C15) & (2**64 - 1))) & (2**64 - 1)
        x = (x * 0xBF58476D1CE4E5B9) & (2**64 - 1)
        x ^= x >> 31
        x = (x * 0x94D049BB133111EB) & (2**64 - 1)
        x ^= x >> 29
    return x & (2**63 - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed_for(*parts))
    return g


def _orthonormal_columns(x: torch.Tensor) -> torch.Tensor:
    """Batched modified Gram-Schmidt (two passes) over the last dim's columns."""
    cols = []
    for j in range(x.shape[-1]):
        v = x[..., j]
        for _ in range(2):
            for c in cols:
                v = v - (v * c).sum(-1, keepdim=True) * c
        v = v / v.norm(dim=-1, keepdim=True)
        cols.append(v)
    return torch.stack(cols, dim=-1)


def page_keys(gen: torch.Generator, n: int, rho: torch.Tensor,
              device) -> torch.Tensor:
    """n page-heads of 16 keys each, float32 [n][16][128] (see module doc)."""
    mu = torch.randn(n, 1, HEAD_DIM, generator=gen, device=device) * 0.5
    w = _orthonormal_columns(
        torch.randn(n, HEAD_DIM, RANK, generator=gen, device=device))
    a = torch.randn(n, PAGE, RANK, generator=gen, device=device)
    a = _orthonormal_columns(a - a.mean(dim=1, keepdim=True))
    m = torch.arange(RANK, device=device, dtype=torch.float32)
    s = 4.0 * rho.reshape(n, 1) ** m.reshape(1, RANK)        # [n][8]
    noise = torch.randn(n, PAGE, HEAD_DIM, generator=gen, device=device) * 0.05
    return mu + torch.bmm(a * s[:, None, :], w.transpose(1, 2)) + noise


def _rho(spec: WorkloadSpec, gen, n, device) -> torch.Tensor:
    if spec.decay_range is None:
        return torch.full((n,), spec.decay, device=device)
    lo, hi = spec.decay_range
    return lo + (hi - lo) * torch.rand(n, generator=gen, device=device)


def seq_lengths(spec: WorkloadSpec) -> list:
    """Prompt lengths in tokens.  Ragged lengths avoid multiples of 16."""
    if spec.ragged_min is None:
        return [spec.ctx] * spec.batch
    g = _gen("cpu", spec.seed, 101)
    lens = torch.randint(spec.ragged_min, spec.ctx + 1, (spec.batch,),
                         generator=g).tolist()
    return [L if L % PAGE else L - 1 for L in lens]


def _layout(spec: WorkloadSpec):
    """Prompt lengths, pages per sequence (appended tokens included)."""
    lens = seq_lengths(spec)
    n_pages = [math.ceil((L + spec.append_steps) / PAGE) for L in lens]
    return lens, n_pages


def _needles(spec: WorkloadSpec, b: int, full_prompt: int):
    """Needle pages [h_kv][needles], unit directions [h_kv][needles][128]
    and token slots [h_kv][needles] of sequence b (CPU sub-stream)."""
    gn = _gen("cpu", spec.seed, 2000 + b)
    nn = spec.needles
    pages = torch.zeros(spec.h_kv, nn, dtype=torch.int64)
    dirs = torch.zeros(spec.h_kv, nn, HEAD_DIM)
    for h in range(spec.h_kv):
        lo, hi = 1, max(1, full_prompt - 2)
        cand = torch.randperm(hi - lo + 1, generator=gn)[:nn] + lo
        pages[h, :len(cand)] = cand
        d = torch.randn(nn, HEAD_DIM, generator=gn)
        dirs[h] = d / d.norm(dim=-1, keepdim=True)
    toks = torch.randint(0, PAGE, (spec.h_kv, nn), generator=gn)
    return pages, dirs, toks


def sequence_chunks(spec: WorkloadSpec, b: int, device, chunk_pages=2048):
    """Yield (p0, p1, keys, values) for logical pages [p0, p1) of sequence b,
    float32 [p1-p0][h_kv][16][128], needles planted."""
    lens, n_pages = _layout(spec)
    n = n_pages[b]
    pages, dirs, toks = _needles(spec, b, lens[b] // PAGE)
    gk = _gen(device, spec.seed, 1000 + b)
    for p0 in range(0, n, chunk_pages):
        p1 = min(n, p0 + chunk_pages)
        cnt = (p1 - p0) * spec.h_kv
        keys = page_keys(gk, cnt, _rho(spec, gk, cnt, device), device)
        keys = keys.view(p1 - p0, spec.h_kv, PAGE, HEAD_DIM)
        for h in range(spec.h_kv):
            for t in range(spec.needles):
                pg = int(pages[h, t])
                if p0 <= pg < p1:
                    row = keys[pg - p0, h, int(toks[h, t])]
                    keys[pg - p0, h, int(toks[h, t])] = row.norm() * \
                        dirs[h, t].to(device)
        vals = torch.randn(p1 - p0, spec.h_kv, PAGE, HEAD_DIM, generator=gk,
                           device=device)
        yield p0, p1, keys, vals


def _queries(spec: WorkloadSpec, device, n_steps, needle_dirs):
    """[steps][batch][h_q][128] N(0, I), re-aimed at the needles."""
    gq = _gen(device, spec.seed, 3000)
    q = torch.randn(n_steps, spec.batch, spec.h_q, HEAD_DIM, generator=gq,
                    device=device)
    nn = spec.needles
    if nn:
        G = spec.group
        dirs = needle_dirs.to(device)
        for h in range(spec.h_kv):
            for g in range(G):
                nd = dirs[:, h, g % nn]                       # [batch][128]
                z = q[:, :, h * G + g]                        # [steps][batch][128]
                zn = z.norm(dim=-1, keepdim=True)
                u = z - (z * nd).sum(-1, keepdim=True) * nd
                u = u / u.norm(dim=-1, keepdim=True)
                q[:, :, h * G + g] = zn * (0.6 * nd + 0.8 * u)
    return q.to(torch.bfloat16)


def generate(spec: WorkloadSpec, device="cpu",
             seqs: Optional[Sequence[int]] = None,
             chunk_pages: int = 2048,
             steps: Optional[int] = None) -> Workload:
    """Draw the whole workload on `device`.

    Every sequence draws from its own seeded sub-stream, so a sequence's
    contents do not depend on which others are generated (on one device
    type).  `seqs` restricts generation to a subset (the others keep a zero
    cache); `steps` overrides the number of query steps drawn.
    """
    device = torch.device(device)
    lens, n_pages = _layout(spec)
    max_pages = max(n_pages)
    total = sum(n_pages)
    pg = _gen("cpu", spec.seed, 7)
    phys = torch.arange(total) if spec.contiguous else torch.randperm(
        total, generator=pg)
    page_table = torch.full((spec.batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(n_pages):
        page_table[b, :n] = phys[off:off + n].to(torch.int32)
        off += n
    shape = (total, spec.h_kv, PAGE, HEAD_DIM)
    k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    v_cache = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    nn = spec.needles
    needle_pages = torch.zeros(spec.batch, spec.h_kv, nn, dtype=torch.int64)
    needle_dirs = torch.zeros(spec.batch, spec.h_kv, nn, HEAD_DIM)
    k_app = v_app = None
    if spec.append_steps:
        k_app = torch.zeros(spec.append_steps, spec.batch, spec.h_kv,
                            HEAD_DIM, dtype=torch.bfloat16, device=device)
        v_app = torch.zeros_like(k_app)
    pt_dev = page_table.to(device)
    for b in (range(spec.batch) if seqs is None else seqs):
        needle_pages[b], needle_dirs[b], _ = _needles(spec, b,
                                                      lens[b] // PAGE)
        for p0, p1, keys, vals in sequence_chunks(spec, b, device,
                                                  chunk_pages):
            ids = pt_dev[b, p0:p1].long()
            k_cache.index_copy_(0, ids, keys.to(torch.bfloat16))
            v_cache.index_copy_(0, ids, vals.to(torch.bfloat16))
        # appended tokens (positions lens[b] ..) leave the cache for the
        # per-step append stream
        for s in range(spec.append_steps):
            pos = lens[b] + s
            pid = int(page_table[b, pos // PAGE])
            k_app[s, b] = k_cache[pid, :, pos % PAGE]
            v_app[s, b] = v_cache[pid, :, pos % PAGE]
            k_cache[pid, :, pos % PAGE] = 0
            v_cache[pid, :, pos % PAGE] = 0
    n_steps = spec.steps if steps is None else steps
    q = _queries(spec, device, n_steps, needle_dirs)
    return Workload(spec=spec, k_cache=k_cache, v_cache=v_cache,
                    page_table=page_table.to(device),
                    seq_lens=torch.tensor(lens, dtype=torch.int32,
                                          device=device),
                    queries=q, needle_pages=needle_pages,
                    needle_dirs=needle_dirs, k_append=k_app, v_append=v_app)


def generate_sequence(spec: WorkloadSpec, b: int, device="cpu",
                      steps: Optional[int] = None):
    """One sequence in logical page order (no page table): dict with keys and
    values bf16 [n_pages][h_kv][16][128], its prompt length and its queries
    bf16 [steps][h_q][128]."""
    lens, n_pages = _layout(spec)
    ks, vs = [], []
    for _, _, keys, vals in sequence_chunks(spec, b, device):
        ks.append(keys.to(torch.bfloat16))
        vs.append(vals.to(torch.bfloat16))
    needle_dirs = torch.zeros(spec.batch, spec.h_kv, spec.needles, HEAD_DIM)
    needle_dirs[b] = _needles(spec, b, lens[b] // PAGE)[1]
    n_steps = spec.steps if steps is None else steps
    q = _queries(spec, device, n_steps, needle_dirs)[:, b]
    return dict(keys=torch.cat(ks), values=torch.cat(vs), seq_len=lens[b],
                queries=q)


def custom_spec(**kw) -> WorkloadSpec:
    """A workload with explicit shape (used for small parity cases)."""
    base = dict(name="custom", batch=1, h_q=4, h_kv=1, ctx=256, k=4,
                steps=1, needles=0, seed=0)
    base.update(kw)
    return WorkloadSpec(**base)
