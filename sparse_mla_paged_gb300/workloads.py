"""Seeded synthetic inputs for the selected-index NoPE MLA paged decode.

This module only draws inputs. It holds none of the decode's arithmetic, and both the
CUDA path and the CPU oracle consume what it produces. The five named workloads follow
the shapes, sizes and value distributions of the decode the pages describe (one latent
KV head of 512 FP8-E4M3 bytes per token, BF16 absorbed queries, i32 selection rows with
-1 holes); every tensor is drawn from ``torch.Generator`` streams seeded per workload.

FP8 encoding of generated cache values is: divide by the cache scale, clamp to +-448,
cast to ``torch.float8_e4m3fn`` (round to nearest even). This matches the cache writer's
``RMSNorm(x) * (1/kv_scale)`` step as a quantiser with saturation; the decode only ever
reads the resulting bytes back.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

LATENT = 512
BASE_SEED = 20261202


@dataclass
class Workload:
    name: str
    q: torch.Tensor                 # bf16 [R, H, 512]
    k_cache: torch.Tensor           # uint8 [num_pages, cache_stride_bytes]
    v_cache: Optional[torch.Tensor]  # None: V is the same buffer as K
    block_tables: torch.Tensor      # int32 [table_rows, max_blocks_per_seq]
    seq_lens: torch.Tensor          # int32 [R], per decode row
    sel_indices: torch.Tensor       # int32 [R, W]
    num_seqs: int
    rows_per_seq: int
    num_q_heads: int
    block_size: int
    cache_stride_bytes: int
    max_blocks_per_seq: int         # block-table row stride (0 = one shared row)
    k_scale: float
    v_scale: float
    sm_scale: float
    base_lens: Optional[torch.Tensor] = None  # int32 [num_seqs] for k-row verify passes
    meta: dict = field(default_factory=dict)
    _host: Optional[dict] = None

    @property
    def rows(self) -> int:
        return self.num_seqs * self.rows_per_seq

    @property
    def sel_width(self) -> int:
        return int(self.sel_indices.shape[1])

    def host(self) -> dict:
        """numpy copies (q as uint16 BF16 bits, caches as uint8 codes), cached."""
        if self._host is None:
            h = {
                "q_bits": self.q.detach().view(torch.int16).cpu().numpy().view(np.uint16),
                "k_cache": self.k_cache.detach().cpu().numpy(),
                "v_cache": None if self.v_cache is None else self.v_cache.detach().cpu().numpy(),
                "block_tables": self.block_tables.detach().cpu().numpy(),
                "seq_lens": self.seq_lens.detach().cpu().numpy(),
                "sel_indices": self.sel_indices.detach().cpu().numpy(),
            }
            self._host = h
        return self._host

    def subset(self, seqs) -> tuple["Workload", list]:
        """The sequences `seqs` (all their rows) with only their pages, on the CPU.

        The bytes of every page they reference are copied unchanged; pages are renumbered
        in table order. Returns (workload, row indices of the original)."""
        seqs = list(seqs)
        rps = self.rows_per_seq
        rows = [s * rps + i for s in seqs for i in range(rps)]
        shared = self.max_blocks_per_seq == 0
        tables = self.block_tables[[0] if shared else seqs].to(torch.int64)
        cache = self.k_cache.reshape(self.k_cache.shape[0], -1)
        pages = tables.reshape(-1)
        valid = pages >= 0
        src = torch.where(valid, pages, torch.zeros_like(pages)).to(cache.device)
        kc = cache[src].cpu()
        vc = None if self.v_cache is None else self.v_cache.reshape(cache.shape[0], -1)[src].cpu()
        bt = torch.arange(pages.numel(), dtype=torch.int32).reshape(tables.shape)
        bt[~valid.cpu().reshape(tables.shape)] = -1
        sub = Workload(self.name + f" [sequences {seqs}]", self.q[rows].cpu(), kc, vc, bt,
                       self.seq_lens[rows].cpu(), self.sel_indices[rows].cpu(), len(seqs), rps,
                       self.num_q_heads, self.block_size, self.cache_stride_bytes,
                       0 if shared else int(self.block_tables.shape[1]), self.k_scale, self.v_scale,
                       self.sm_scale, None if self.base_lens is None else self.base_lens[seqs].cpu(),
                       dict(self.meta))
        return sub, rows

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return Workload(self.name, mv(self.q), mv(self.k_cache), mv(self.v_cache),
                        mv(self.block_tables), mv(self.seq_lens), mv(self.sel_indices),
                        self.num_seqs, self.rows_per_seq, self.num_q_heads, self.block_size,
                        self.cache_stride_bytes, self.max_blocks_per_seq, self.k_scale,
                        self.v_scale, self.sm_scale, mv(self.base_lens), dict(self.meta))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    return (x / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def _cache(num_pages: int, stride: int, dist: str, scale: float, device, g) -> torch.Tensor:
    """FP8 cache bytes [num_pages, stride]. Drawn in chunks so that large pools do not
    need a float copy of the whole pool."""
    out = torch.empty((num_pages, stride), dtype=torch.uint8, device=device)
    chunk = max(1, (64 << 20) // max(stride, 1))
    for p0 in range(0, num_pages, chunk):
        p1 = min(num_pages, p0 + chunk)
        n = (p1 - p0) * stride
        if dist == "normal":
            x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        elif dist == "t3":
            # Student-t with 3 degrees of freedom: N / sqrt(chi^2_3 / 3).
            z = torch.randn(n, generator=g, device=device, dtype=torch.float32)
            c = torch.randn((3, n), generator=g, device=device, dtype=torch.float32)
            x = z / torch.sqrt((c * c).sum(0) / 3.0)
        else:
            raise ValueError(dist)
        out[p0:p1].view(-1).copy_(_quantize_e4m3(x, scale))
    return out


def _q(rows: int, heads: int, sigma: float, device, g) -> torch.Tensor:
    return (sigma * torch.randn((rows, heads, LATENT), generator=g, device=device)).to(torch.bfloat16)


def _perm(n: int, device, g) -> torch.Tensor:
    return torch.randperm(n, generator=g, device=device)


def _distinct(lo: int, hi: int, k: int, device, g) -> torch.Tensor:
    """k distinct integers from [lo, hi), in random order."""
    assert 0 <= k <= hi - lo
    return _perm(hi - lo, device, g)[:k] + lo


def _shuffle(x: torch.Tensor, device, g) -> torch.Tensor:
    return x[_perm(x.numel(), device, g)]


# ------------------------------------------------------------------------------------
# The five named workloads.
# ------------------------------------------------------------------------------------

def tiny(device="cpu", seed: Optional[int] = None) -> Workload:
    """1 sequence, 4 query heads, seq_len 256, block_size 64 with identity pages,
    sel_width 64: 55 distinct ids from [0,256), 3 duplicates of them and 6 holes,
    shuffled; sm_scale = 1/sqrt(256)."""
    g = _gen(device, BASE_SEED + 0 if seed is None else seed)
    H, L, bs, W = 4, 256, 64, 64
    q = _q(1, H, 1.0, device, g)
    cache = _cache(L // bs, bs * LATENT, "normal", 0.05, device, g)
    bt = torch.arange(L // bs, dtype=torch.int32, device=device).reshape(1, -1)
    distinct = _distinct(0, L, 55, device, g)
    dups = distinct[:3].clone()
    holes = torch.full((6,), -1, dtype=torch.int64, device=device)
    sel = _shuffle(torch.cat([distinct, dups, holes]), device, g).to(torch.int32).reshape(1, W)
    return Workload("tiny: 1 seq x 4 heads, seq_len 256, sel_width 64", q, cache, None, bt,
                    torch.full((1,), L, dtype=torch.int32, device=device), sel,
                    1, 1, H, bs, bs * LATENT, L // bs, 0.05, 0.05, 1.0 / 16.0)


def decode_batch(device="cpu", seed: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    """8 sequences x 64 heads, seq_len 4096, block_size 64 over a randomly permuted
    512-page pool, sel_width 2048 = 2007 distinct ids + 41 holes (2%). num_seqs draws a
    smaller (or larger) batch of the same kind."""
    g = _gen(device, BASE_SEED + 1 if seed is None else seed)
    S, H, L, bs, W = num_seqs or 8, 64, 4096, 64, 2048
    q = _q(S, H, 1.0, device, g)
    pages_per_seq = L // bs
    cache = _cache(S * pages_per_seq, bs * LATENT, "normal", 0.05, device, g)
    bt = _perm(S * pages_per_seq, device, g).to(torch.int32).reshape(S, pages_per_seq)
    rows = []
    for _ in range(S):
        ids = _distinct(0, L, W - 41, device, g)
        holes = torch.full((41,), -1, dtype=torch.int64, device=device)
        rows.append(_shuffle(torch.cat([ids, holes]), device, g))
    sel = torch.stack(rows).to(torch.int32)
    return Workload(f"decode batch: {S} seqs x 64 heads, seq_len 4096, sel_width 2048", q, cache,
                    None, bt, torch.full((S,), L, dtype=torch.int32, device=device), sel,
                    S, 1, H, bs, bs * LATENT, pages_per_seq, 0.05, 0.05, 1.0 / math.sqrt(512))


def ragged(device="cpu", seed: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    """64 sequences x 64 heads, seq_len uniform in [8192, 32768], block_size 64, pages
    scattered over a 2M-token pool; sel_width 2048 = 1536 distinct ids from
    [0, L-512) + 512 distinct from the last 512 positions; rows shorter than 2048
    tokens would take every position and pad with holes. num_seqs draws a smaller batch
    of the same kind."""
    g = _gen(device, BASE_SEED + 2 if seed is None else seed)
    S, H, bs, W, pool_pages = num_seqs or 64, 64, 64, 2048, (2 << 20) // 64
    lens = torch.randint(8192, 32768 + 1, (S,), generator=g, device=device)
    q = _q(S, H, 1.0, device, g)
    cache = _cache(pool_pages, bs * LATENT, "normal", 0.05, device, g)
    need = (lens + bs - 1) // bs
    mbps = int(need.max().item())
    perm = _perm(pool_pages, device, g)
    bt = torch.zeros((S, mbps), dtype=torch.int32, device=device)
    off = 0
    rows = []
    for s in range(S):
        n = int(need[s].item())
        bt[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
        L = int(lens[s].item())
        if L < W:
            ids = torch.cat([_distinct(0, L, L, device, g),
                             torch.full((W - L,), -1, dtype=torch.int64, device=device)])
        else:
            ids = torch.cat([_distinct(0, L - 512, 1536, device, g),
                             _distinct(L - 512, L, 512, device, g)])
        rows.append(_shuffle(ids, device, g))
    sel = torch.stack(rows).to(torch.int32)
    return Workload(f"ragged long-context: {S} seqs x 64 heads, seq_len U[8192,32768], sel_width 2048",
                    q, cache, None, bt, lens.to(torch.int32), sel, S, 1, H, bs, bs * LATENT, mbps,
                    0.05, 0.05, 1.0 / math.sqrt(512))


def pooled_128k(device="cpu", seed: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    """128 sequences x 128 heads, seq_len 131072, block_size 64 (2048 pages each over a
    262144-page pool), index_kpool 4: 512 random distinct pools of 4 consecutive tokens
    (sel_width 2048); q ~ N(0, 2^2); cache from Student-t(3) before quantisation.
    num_seqs draws a smaller batch of the same kind (with its own pool)."""
    g = _gen(device, BASE_SEED + 3 if seed is None else seed)
    S, H, L, bs, kpool, npools = num_seqs or 128, 128, 131072, 64, 4, 512
    q = _q(S, H, 2.0, device, g)
    pps = L // bs
    cache = _cache(S * pps, bs * LATENT, "t3", 0.05, device, g)
    bt = _perm(S * pps, device, g).to(torch.int32).reshape(S, pps)
    rows = []
    for _ in range(S):
        pools = _distinct(0, L // kpool, npools, device, g)
        rows.append((pools[:, None] * kpool + torch.arange(kpool, device=device)[None, :]).reshape(-1))
    sel = torch.stack(rows).to(torch.int32)
    return Workload(f"pooled selection at 128K: {S} seqs x 128 heads, 512 pools of 4", q, cache,
                    None, bt, torch.full((S,), L, dtype=torch.int32, device=device), sel,
                    S, 1, H, bs, bs * LATENT, pps, 0.05, 0.05, 1.0 / math.sqrt(512),
                    meta={"index_kpool": kpool})


def verify_k4(device="cpu", seed: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    """32 sequences x k=4 consecutive verify rows (128 rows), 64 heads, base seq_len
    16384; row r sees positions < 16384 + r + 1; per row 2048 ids = 1536 shared by the
    sequence's rows + 512 row-specific; block_size 64 over a permuted pool. num_seqs
    draws a smaller batch of the same kind."""
    g = _gen(device, BASE_SEED + 4 if seed is None else seed)
    S, k, H, base, bs, W, shared = num_seqs or 32, 4, 64, 16384, 64, 2048, 1536
    q = _q(S * k, H, 1.0, device, g)
    pps = (base + k + bs - 1) // bs
    cache = _cache(S * pps, bs * LATENT, "normal", 0.05, device, g)
    bt = _perm(S * pps, device, g).to(torch.int32).reshape(S, pps)
    base_lens = torch.full((S,), base, dtype=torch.int32, device=device)
    lens = (base_lens[:, None].to(torch.int64) + torch.arange(k, device=device)[None, :] + 1)
    rows = []
    for s in range(S):
        common = _distinct(0, base, shared, device, g)
        taken = torch.zeros(base + k, dtype=torch.bool, device=device)
        taken[common] = True
        for r in range(k):
            L = int(lens[s, r].item())
            free = torch.nonzero(~taken[:L]).reshape(-1)
            own = free[_perm(free.numel(), device, g)[:W - shared]]
            rows.append(_shuffle(torch.cat([common, own]), device, g))
    sel = torch.stack(rows).to(torch.int32)
    return Workload(f"multi-row verify: {S} seqs x k=4 rows x 64 heads, base seq_len 16384", q, cache,
                    None, bt, lens.reshape(-1).to(torch.int32), sel, S, k, H, bs, bs * LATENT, pps,
                    0.05, 0.05, 1.0 / math.sqrt(512), base_lens=base_lens)


CONFIGS = [tiny, decode_batch, ragged, pooled_128k, verify_k4]


def pool_scores(rows: int = 128, n_pools: int = 32768, kpool: int = 4, q_pos=None, device="cpu",
                seed: Optional[int] = None) -> tuple[torch.Tensor, torch.Tensor]:
    """Selector input of the pooled 128K decode: float32 pooled indexer scores [rows,
    n_pools] ~ N(0, 1) (the indexer's weights are not on the pages, so its scores are
    drawn) and each row's position q_pos (int32 [rows]; default: the last position,
    n_pools*kpool - 1, so every pool is eligible). A list or tensor q_pos is taken as given."""
    g = _gen(device, BASE_SEED + 7 if seed is None else seed)
    scores = torch.randn((rows, n_pools), generator=g, device=device, dtype=torch.float32)
    if q_pos is None:
        q = torch.full((rows,), n_pools * kpool - 1, dtype=torch.int32, device=device)
    else:
        q = torch.as_tensor(q_pos, dtype=torch.int32).to(device)
    return scores, q


def config(index: int, device="cpu", seed: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    if num_seqs is None:
        return CONFIGS[index](device=device, seed=seed)
    if index == 0:
        raise ValueError("the tiny workload has one sequence")
    return CONFIGS[index](device=device, seed=seed, num_seqs=num_seqs)


# ------------------------------------------------------------------------------------
# Small random cases for tests.
# ------------------------------------------------------------------------------------

def random_case(*, num_seqs=1, rows_per_seq=1, heads=4, seq_len=256, block_size=64,
                sel_width=64, hole_frac=0.1, dup_frac=0.05, out_of_range_frac=0.0,
                seq_lens=None, extra_pages=3, stride_pad=0, split_kv=False,
                shared_table=False, q_sigma=1.0, cache_dist="normal", k_scale=0.05,
                v_scale=0.05, sm_scale=None, device="cpu", seed=12345) -> Workload:
    """A small paged case with scattered pages, holes, duplicates and (optionally)
    out-of-range ids, per-row lengths, padded page stride and a separate V cache."""
    g = _gen(device, seed)
    R = num_seqs * rows_per_seq
    if seq_lens is None:
        seq_lens = [seq_len] * R
    lens = torch.tensor(seq_lens, dtype=torch.int32, device=device).reshape(R)
    max_len = int(lens.max().item()) if R else 0
    mbps = max(1, (max_len + block_size - 1) // block_size)
    table_rows = 1 if shared_table else num_seqs
    num_pages = table_rows * mbps + extra_pages
    stride = block_size * LATENT + stride_pad
    q = _q(R, heads, q_sigma, device, g)
    kc = _cache(num_pages, stride, cache_dist, k_scale, device, g)
    vc = _cache(num_pages, stride, cache_dist, v_scale, device, g) if split_kv else None
    bt = _perm(num_pages, device, g)[: table_rows * mbps].to(torch.int32).reshape(table_rows, mbps)
    rows = []
    for r in range(R):
        L = int(lens[r].item())
        n_hole = int(round(hole_frac * sel_width))
        n_dup = int(round(dup_frac * sel_width))
        n_oor = int(round(out_of_range_frac * sel_width))
        n_valid = max(0, sel_width - n_hole - n_dup - n_oor)
        n_valid = min(n_valid, L)
        valid = _distinct(0, L, n_valid, device, g) if n_valid else torch.zeros(0, dtype=torch.int64, device=device)
        dups = valid[torch.randint(0, max(1, valid.numel()), (n_dup,), generator=g, device=device)] \
            if valid.numel() else torch.full((n_dup,), -1, dtype=torch.int64, device=device)
        oor = L + torch.randint(0, 1000, (n_oor,), generator=g, device=device)
        pad = sel_width - valid.numel() - dups.numel() - oor.numel()
        holes = torch.full((pad,), -1, dtype=torch.int64, device=device)
        rows.append(_shuffle(torch.cat([valid, dups, oor, holes]), device, g))
    sel = torch.stack(rows).to(torch.int32) if R else torch.zeros((0, sel_width), dtype=torch.int32)
    return Workload(f"random case seed {seed}", q, kc, vc, bt, lens, sel, num_seqs, rows_per_seq,
                    heads, block_size, stride, 0 if shared_table else mbps, k_scale, v_scale,
                    (1.0 / math.sqrt(LATENT)) if sm_scale is None else sm_scale)


def flat_tail(*, heads=64, width=2048, tail_value=20.0, dominant_at=("first", "middle", "last"),
              gap_lo=4.0, gap_hi=24.0, device="cpu", seed=31337) -> Workload:
    """One sequence per entry of `dominant_at`, each selecting `width` tokens: one dominant
    token (the lowest, a middle or the highest selected id) and width - 1 tokens whose
    cache rows are byte-identical (a flat tail of equal scores). The scores are set by
    dimension 0 alone: q[h, 0] = gap_h, with gap_h swept from gap_lo to gap_hi over the
    heads, the dominant row holds 448 there and the tail rows 0; with k_scale = 1/448 and
    sm_scale = ln 2 the dominant score sits gap_h log2 units above the tail. The tail rows
    hold `tail_value` (an E4M3 code) in every other dimension; the dominant row holds, in a
    block of 7 dimensions per head, the code that nearly cancels that head's tail, so the
    reference output there is close to zero and the absolute tolerance term decides."""
    g = _gen(device, seed)
    S, bs = len(dominant_at), 64
    pages = (width + bs - 1) // bs
    gaps = torch.linspace(gap_lo, gap_hi, heads, device=device, dtype=torch.float64)
    q = torch.zeros((S, heads, LATENT), dtype=torch.float32, device=device)
    q[:, :, 0] = gaps.to(torch.float32)
    q = q.to(torch.bfloat16)
    gq = q[0, :, 0].to(torch.float64)                      # the BF16 gaps actually used
    tail = torch.full((LATENT,), tail_value, dtype=torch.float32, device=device)
    tail[0] = 0.0
    dom = torch.zeros((LATENT,), dtype=torch.float32, device=device)
    dom[0] = 448.0
    for h in range(min(heads, (LATENT - 1) // 7)):
        share = (width - 1) * torch.exp2(-gq[h])         # tail weight over the dominant's
        dom[1 + 7 * h:8 + 7 * h] = float(-tail_value * share.clamp(max=448.0 / max(tail_value, 1e-30)))
    tail_b = tail.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    dom_b = dom.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    num_pages = S * pages
    cache = tail_b.repeat(num_pages * bs).reshape(num_pages, bs * LATENT).clone()
    bt = _perm(num_pages, device, g).to(torch.int32).reshape(S, pages)
    rows = []
    for s, where in enumerate(dominant_at):
        d = {"first": 0, "middle": width // 2 - 7, "last": width - 1}[where]
        page = int(bt[s, d // bs].item())
        cache[page, (d % bs) * LATENT:(d % bs + 1) * LATENT] = dom_b
        rows.append(_shuffle(torch.arange(width, device=device), device, g))
    sel = torch.stack(rows).to(torch.int32)
    return Workload(f"flat tail: {S} seqs x {heads} heads, width {width}, gaps {gap_lo}..{gap_hi}", q, cache,
                    None, bt, torch.full((S,), width, dtype=torch.int32, device=device), sel, S, 1, heads, bs,
                    bs * LATENT, pages, 1.0 / 448.0, 0.05, math.log(2.0))


def absorb_weights(heads: int = 64, nope: int = 256, vd: int = 256, kvl: int = LATENT, q_lora_rank: int = 2048,
                   hidden: int = 6144, device="cpu", seed: Optional[int] = None):
    """Synthetic BF16 weights for the load-time absorb transforms (the checkpoint's are not
    on the pages): q_b [heads*nope, q_lora_rank], kv_b [heads*(nope+vd), kvl] and o_proj
    [hidden, heads*vd], each N(0, 1/fan_in). Defaults: 64 heads, nope = vd = 256
    (qk_head_dim 256 and nope + v_head_dim 512 as the pages state), kvl 512, q_lora_rank
    2048, hidden 6144."""
    g = _gen(device, BASE_SEED + 11 if seed is None else seed)

    def w(rows, cols):
        return (torch.randn((rows, cols), generator=g, device=device) / math.sqrt(cols)).to(torch.bfloat16)
    return w(heads * nope, q_lora_rank), w(heads * (nope + vd), kvl), w(hidden, heads * vd)
