"""Seeded synthetic inputs for paged GQA decode attention.

This module is shared by the tests, the benchmark and the oracle checks.  It
only draws random numbers and lays them out (page pool, block table, sequence
lengths); it holds none of the attention arithmetic, and it imports neither the
oracle nor the CUDA library.

Workloads (the serving shapes of the decode-attention kernels on the pages:
FlashQuant wiki "CUDA Kernels", paged_decode.cu; OASR "Kernel Layer", "Fused
attention", paged streaming mode):

  tiny        B=1,   Hq=8,  Hkv=2, D=64,  P=16, L=256, 64-page pool, scale 1/8
  batch       B=8,   Hq=32, Hkv=8, D=128, P=16, L ~ U{1024..4096}
  ragged      B=64,  Hq=32, Hkv=8, D=128, P=16, L = round(2048 exp(N(0,1))) clipped
              to [17, 32768]; every fourth length forced off a page boundary;
              each K row (token, kv head) multiplied by U(0.5, 4)
  long        B=4,   Hq=64, Hkv=8, D=128, P=16, L=131072, pool 32768 pages
  bigpage     B=256, Hq=32, Hkv=8, D=128, P=64, L=2048,   pool 8192 pages
  bigpage_g16 B=256, Hq=32, Hkv=2, D=256, P=64, L=2048,   pool 8192 pages, scale 1/16

q, K and V are N(0, 1) drawn in float32 and rounded to bf16 (round to nearest
even).  Physical page ids are a seeded permutation of the pool; the pages of
all sequences are disjoint.  Unused block-table entries hold -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(B=1, Hq=8, Hkv=2, D=64, P=16, lens=("fixed", 256), pool=64, seed=0),
    "batch": dict(B=8, Hq=32, Hkv=8, D=128, P=16, lens=("uniform", 1024, 4096), pool=None, seed=1),
    "ragged": dict(B=64, Hq=32, Hkv=8, D=128, P=16, lens=("lognormal", 2048, 1.0, 17, 32768),
                   pool=None, seed=2, k_row_scale=(0.5, 4.0)),
    "long": dict(B=4, Hq=64, Hkv=8, D=128, P=16, lens=("fixed", 131072), pool=32768, seed=3),
    "bigpage": dict(B=256, Hq=32, Hkv=8, D=128, P=64, lens=("fixed", 2048), pool=8192, seed=4),
    "bigpage_g16": dict(B=256, Hq=32, Hkv=2, D=256, P=64, lens=("fixed", 2048), pool=8192, seed=5),
}

# The order in which the workloads are listed in the problem statement.
CONFIG_ORDER = ["tiny", "batch", "ragged", "long", "bigpage", "bigpage_g16"]


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def draw_seq_lens(spec, B: int, P: int, seed: int) -> np.ndarray:
    """Sequence lengths for one workload (numpy PCG64, seeded)."""
    rng = np.random.default_rng(seed)
    kind = spec[0]
    if kind == "fixed":
        lens = np.full(B, spec[1], dtype=np.int64)
    elif kind == "uniform":
        lens = rng.integers(spec[1], spec[2], size=B, endpoint=True)
    elif kind == "lognormal":
        median, sigma, lo, hi = spec[1:]
        lens = np.rint(median * np.exp(sigma * rng.standard_normal(B))).astype(np.int64)
        lens = np.clip(lens, lo, hi)
        # Partial last pages by construction: every fourth sequence ends mid-page.
        for i in range(0, B, 4):
            if lens[i] % P == 0:
                lens[i] = lens[i] + 1 if lens[i] < hi else lens[i] - 1
    elif kind == "list":
        lens = np.asarray(spec[1], dtype=np.int64)
    else:
        raise ValueError("unknown length spec %r" % (spec,))
    return lens.astype(np.int32)


@dataclass
class Case:
    """One batch of decode-attention inputs plus its shape metadata."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    num_pages: int
    max_pages: int
    scale: float
    q: torch.Tensor            # [B, Hq, D] bf16
    k_cache: torch.Tensor      # [num_pages, P, Hkv, D] bf16
    v_cache: torch.Tensor      # [num_pages, P, Hkv, D] bf16
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    meta: dict = field(default_factory=dict)
    qo_indptr: torch.Tensor = None  # [B+1] int32 for multi-token cases (q is then [total_q, Hq, D])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def to(self, device) -> "Case":
        c = Case(**{**self.__dict__})
        for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens", "qo_indptr"):
            if getattr(self, name) is not None:
                setattr(c, name, getattr(self, name).to(device))
        return c

    def host_bits(self):
        """(q, k, v) as numpy uint16 bf16 bit patterns, plus table and lengths."""
        return (bf16_bits(self.q), bf16_bits(self.k_cache), bf16_bits(self.v_cache),
                self.block_table.cpu().numpy(), self.seq_lens.cpu().numpy())


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a bf16 tensor as numpy uint16 (numpy has no bfloat16)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _randn_bf16(shape, gen: torch.Generator, device, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """N(0,1) in float32, rounded to bf16, drawn in chunks to bound scratch memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_case(name_or_spec, device="cpu", seed=None, poison=False, seq_lens=None, scale=None,
              pool=None, name=None) -> Case:
    """Build one seeded workload.

    name_or_spec: a key of CONFIGS or a dict with the same fields.
    poison:  fill every K/V row that no used token references with NaN, and
             put -1 / 2**30 in the block-table entries past each sequence's
             used pages (they must be ignored).
    seq_lens: optional explicit lengths (overrides the spec's length rule).
    """
    if isinstance(name_or_spec, str):
        spec = dict(CONFIGS[name_or_spec])
        name = name or name_or_spec
    else:
        spec = dict(name_or_spec)
        name = name or spec.get("name", "custom")
    B, Hq, Hkv, D, P = spec["B"], spec["Hq"], spec["Hkv"], spec["D"], spec["P"]
    seed = spec.get("seed", 0) if seed is None else seed
    if seq_lens is None:
        lens = draw_seq_lens(spec["lens"], B, P, seed)
    else:
        lens = np.asarray(seq_lens, dtype=np.int32)
        assert lens.shape == (B,)
    n_pages = (lens.astype(np.int64) + P - 1) // P
    used = int(n_pages.sum())
    pool = pool if pool is not None else spec.get("pool")
    num_pages = max(int(pool) if pool else used, used, 1)
    max_pages = max(int(spec.get("max_pages", 0)), int(n_pages.max()) if B else 0, 1)

    rng = np.random.default_rng(seed + 1000003)
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, : n_pages[b]] = perm[off: off + n_pages[b]]
        off += n_pages[b]
    if poison:
        for b in range(B):
            tail = table[b, n_pages[b]:]
            tail[0::2] = -1
            tail[1::2] = 1 << 30

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn_bf16((B, Hq, D), gen, device)
    k = _randn_bf16((num_pages, P, Hkv, D), gen, device)
    v = _randn_bf16((num_pages, P, Hkv, D), gen, device)
    krs = spec.get("k_row_scale")
    if krs is not None:
        lo, hi = krs
        kf = k.view(num_pages * P * Hkv, D)
        for s in range(0, kf.shape[0], 1 << 20):
            e = min(kf.shape[0], s + (1 << 20))
            u = torch.rand(e - s, 1, generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo
            kf[s:e] = (kf[s:e].float() * u).to(torch.bfloat16)
    if poison:
        mask = torch.ones(num_pages, P, dtype=torch.bool)
        for b in range(B):
            L = int(lens[b])
            for j in range(int(n_pages[b])):
                pg = int(table[b, j])
                valid = min(P, L - j * P)
                mask[pg, :valid] = False
        mask = mask.to(device)
        k[mask] = float("nan")
        v[mask] = float("nan")

    # The C interface takes scale as a float32; keep the rounded value so that every
    # consumer (oracle, kernels, brute force) sees the same number.
    sc = float(np.float32(scale if scale is not None else spec.get("scale", default_scale(D))))
    meta = dict(spec=spec, seed=seed, poison=poison, used_pages=used)
    return Case(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, num_pages=num_pages,
                max_pages=max_pages, scale=sc, q=q, k_cache=k, v_cache=v,
                block_table=torch.from_numpy(table).to(device),
                seq_lens=torch.from_numpy(lens.astype(np.int32)).to(device), meta=meta)


def used_slot_mask(case: Case) -> np.ndarray:
    """bool [num_pages, P]: the (page, slot) pairs some sequence's valid key occupies."""
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    table = case.block_table.cpu().numpy()
    mask = np.zeros((case.num_pages, case.P), dtype=bool)
    for b in range(case.B):
        for j in range(int((lens[b] + case.P - 1) // case.P)):
            mask[int(table[b, j]), : min(case.P, int(lens[b]) - j * case.P)] = True
    return mask


def algorithmic_bytes(case: Case, cache: str = "bf16") -> dict:
    """Bytes the computation must move at minimum, per call.

    K and V of the valid tokens only, plus q, out (bf16), lse (f32), the used
    block-table entries and the sequence lengths.  The padded tail of each last
    page is reported separately as ``tail_bytes`` (touched, not required).
    cache="fp8": one byte per K/V element plus one f32 scale per (token, kv head)
    for each of K and V.
    """
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    n_pages = (lens + case.P - 1) // case.P
    row = case.D * 2 if cache == "bf16" else case.D + 4  # bytes per (token, kv head) of K (or V)
    kv = 2 * int(lens.sum()) * case.Hkv * row
    q_rows = case.B if case.qo_indptr is None else int(case.q.shape[0])  # several rows per sequence
    qo = 2 * q_rows * case.Hq * case.D * 2
    lse = q_rows * case.Hq * 4
    table = int(n_pages.sum()) * 4
    total = kv + qo + lse + table + 4 * case.B + (0 if case.qo_indptr is None else 4 * (case.B + 1))
    tail = 2 * int((n_pages * case.P - lens).sum()) * case.Hkv * row
    return dict(total=total, kv=kv, q_out=qo, lse=lse, table=table, tail_bytes=tail,
                flops=4 * int(lens.sum()) * case.Hq * case.D)


def make_prefill_case(name_or_spec, q_lens, kv_lens=None, device="cpu", seed=None, poison=False, scale=None) -> Case:
    """A multi-token case: request b has q_lens[b] query rows (packed into q [total_q, Hq, D],
    qo_indptr [B+1]) over kv_lens[b] cached keys (default: the spec's length rule; the new
    tokens are counted in kv_lens).  Pool, table and K/V as in make_case."""
    c = make_case(name_or_spec, device=device, seed=seed, poison=poison, seq_lens=kv_lens, scale=scale)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    assert q_lens.shape == (c.B,) and (q_lens >= 0).all()
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    gen = torch.Generator(device=device)
    gen.manual_seed(c.meta["seed"] + 7919)
    c.q = _randn_bf16((int(qo[-1]), c.Hq, c.D), gen, device)
    c.qo_indptr = torch.from_numpy(qo).to(device)
    c.meta["q_lens"] = q_lens.tolist()
    return c