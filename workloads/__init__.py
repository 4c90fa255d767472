"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays out buffers.  It holds none of the
attention arithmetic, no slot formula and no cache-write logic: both the CUDA path and
the oracle receive the same tensors from here and do all of the method's work themselves.

Shapes follow the pages' workload: 24 query heads over 4 KV heads, head size 256, BF16,
pages of 832 (or 784) tokens, contexts of 4K..32K tokens, q=4096 prefill chunks
(page832 post §4, §6; measurement post §3).  Values are N(0, 1) rounded to BF16; an
optional fraction of K rows is scaled by 8 so that the softmax is peaked.  Pages that no
sequence maps, and the slots of a mapped page beyond the sequence's last token, hold BF16
NaN, so a kernel that reads outside the valid range cannot go unnoticed.

Random numbers come from ``torch.Generator`` seeded per workload; the same seed on the
same device gives the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HQ, HKV, HEAD_DIM = 24, 4, 256
BF16_NAN_BITS = -1  # 0xFFFF as int16: a quiet NaN with the sign bit set


@dataclass
class PagedCase:
    """One synthetic problem.  All tensors live on ``device``."""
    q: torch.Tensor                 # bf16 [S, Hq, D] (decode) or [q_len, Hq, D] (prefill)
    k_cache: torch.Tensor           # bf16 [num_pages, BS, Hkv, D]
    v_cache: torch.Tensor           # bf16 [num_pages, BS, Hkv, D]
    block_table: torch.Tensor       # int32 [S, max_blocks]; -1 past each sequence's pages
    seq_lens: torch.Tensor          # int32 [S]: keys per sequence, new tokens included
    block_size: int
    scale: float
    new_k: torch.Tensor | None = None      # bf16 [T, Hkv, D]: tokens still to be written
    new_v: torch.Tensor | None = None
    positions: torch.Tensor | None = None  # int32 [T]: absolute position of each new token
    seq_idx: torch.Tensor | None = None    # int32 [T]: sequence of each new token
    q_start: int = 0                       # prefill: absolute position of query row 0
    meta: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])


def _randn_bf16(shape, gen, device, chunk_rows=1 << 22):
    """N(0,1) in fp32, rounded to BF16, generated in slabs to bound temporary memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = chunk_rows
    for s in range(0, n, step):
        e = min(n, s + step)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
    return out


def _peak_rows(k_cache, frac, factor, gen):
    """Scale a Bernoulli(frac) subset of (slot, kv_head) rows of K by ``factor``
    (before nothing else: x8 is exact in BF16, so scaling after rounding is the same)."""
    if frac <= 0:
        return
    npg = k_cache.shape[0]
    for p0 in range(0, npg, 16):
        p1 = min(npg, p0 + 16)
        sel = torch.rand(k_cache[p0:p1].shape[:3], generator=gen, device=k_cache.device) < frac
        blk = k_cache[p0:p1]
        blk[sel] = blk[sel] * factor


def _poison(cache, block_table, seq_lens, block_size, num_pages):
    """NaN into pages no sequence maps and into slots past each sequence's end."""
    bits = cache.view(torch.int16)
    used = torch.zeros(num_pages, dtype=torch.bool)
    bt = block_table.cpu()
    sl = seq_lens.cpu()
    for s in range(bt.shape[0]):
        npg = -(-int(sl[s]) // block_size)
        if npg == 0:
            continue
        pages = bt[s, :npg]
        used[pages.long()] = True
        tail = int(sl[s]) - (npg - 1) * block_size
        if tail < block_size:
            bits[int(pages[-1]), tail:] = BF16_NAN_BITS
    unused = torch.nonzero(~used).flatten().to(cache.device)
    if unused.numel():
        bits.index_fill_(0, unused, BF16_NAN_BITS)


def paged_case(seed, seq_lens, block_size, num_pages, *, q_rows=None, q_start=0,
               new_tokens=0, peaked_frac=0.0, peaked_factor=8.0, hq=HQ, hkv=HKV,
               head_dim=HEAD_DIM, poison=True, device="cpu", max_blocks=None):
    """Build one problem.

    seq_lens   -- keys per sequence (each count includes that sequence's new tokens).
    q_rows     -- None for decode (one query row per sequence); an int for a prefill
                  chunk of that many rows of sequence 0 at positions q_start.. ; a list
                  (one count per sequence) for a mixed batch of chunks, each the last
                  q_rows[s] keys of sequence s, stacked row-wise in q (meta["cu_seqlens_q"]).
    new_tokens -- decode: 1 means each sequence's last token (position seq_len-1) is
                  supplied as new_k/new_v and its slot starts out as NaN.  For a prefill
                  chunk the q_rows chunk tokens are always supplied this way.
    The block tables take pages without replacement from one seeded permutation of the
    pool, so every sequence's pages are scattered at random over the pool.
    """
    gen = torch.Generator(device=device).manual_seed(int(seed))
    seq_lens = [int(x) for x in seq_lens]
    S = len(seq_lens)
    pages_needed = [-(-L // block_size) for L in seq_lens]
    if sum(pages_needed) > num_pages:
        raise ValueError(f"pool of {num_pages} pages too small for {sum(pages_needed)}")
    mb = max(pages_needed) if max_blocks is None else int(max_blocks)
    perm = torch.randperm(num_pages, generator=gen, device=device).cpu()
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    k = 0
    for s, n in enumerate(pages_needed):
        bt[s, :n] = perm[k:k + n].to(torch.int32)
        k += n
    sl = torch.tensor(seq_lens, dtype=torch.int32)

    k_cache = _randn_bf16((num_pages, block_size, hkv, head_dim), gen, device)
    v_cache = _randn_bf16((num_pages, block_size, hkv, head_dim), gen, device)
    _peak_rows(k_cache, peaked_frac, peaked_factor, gen)

    case = PagedCase(q=None, k_cache=k_cache, v_cache=v_cache, block_table=bt.to(device),
                     seq_lens=sl.to(device), block_size=block_size,
                     scale=1.0 / math.sqrt(head_dim), q_start=int(q_start))
    if q_rows is None:
        case.q = _randn_bf16((S, hq, head_dim), gen, device)
        if new_tokens:
            case.positions = (sl - 1).to(torch.int32).to(device)
            case.seq_idx = torch.arange(S, dtype=torch.int32, device=device)
    elif isinstance(q_rows, (list, tuple)):
        if len(q_rows) != S or any(not 0 <= r <= L for r, L in zip(q_rows, seq_lens)):
            raise ValueError("one chunk length per sequence, at most its key count")
        cu = np.concatenate([[0], np.cumsum(q_rows)]).astype(np.int32)
        case.q = _randn_bf16((int(cu[-1]), hq, head_dim), gen, device)
        case.positions = torch.cat([torch.arange(L - r, L, dtype=torch.int32)
                                    for r, L in zip(q_rows, seq_lens)]).to(device)
        case.seq_idx = torch.cat([torch.full((r,), s, dtype=torch.int32)
                                  for s, r in enumerate(q_rows)]).to(device)
    else:
        if S != 1 or q_start + q_rows != seq_lens[0]:
            raise ValueError("a prefill chunk is one sequence with q_start + q_rows keys")
        case.q = _randn_bf16((q_rows, hq, head_dim), gen, device)
        case.positions = torch.arange(q_start, q_start + q_rows, dtype=torch.int32,
                                      device=device)
        case.seq_idx = torch.zeros(q_rows, dtype=torch.int32, device=device)
    if case.positions is not None:
        T = case.positions.numel()
        case.new_k = _randn_bf16((T, hkv, head_dim), gen, device)
        case.new_v = _randn_bf16((T, hkv, head_dim), gen, device)
        if peaked_frac > 0:
            sel = torch.rand((T, hkv), generator=gen, device=device) < peaked_frac
            case.new_k[sel] = case.new_k[sel] * peaked_factor
    if poison:
        # Slots the new tokens will occupy start as NaN too: they must be written first.
        lens_before = sl.clone()
        if case.positions is not None:
            if q_rows is None:
                lens_before = sl - 1
            elif isinstance(q_rows, (list, tuple)):
                lens_before = sl - torch.tensor(q_rows, dtype=torch.int32)
            else:
                lens_before = torch.tensor([q_start], dtype=torch.int32)
        _poison(k_cache, bt, lens_before.clamp(min=0), block_size, num_pages)
        _poison(v_cache, bt, lens_before.clamp(min=0), block_size, num_pages)
    case.meta = dict(seed=int(seed), seq_lens=seq_lens, block_size=block_size,
                     num_pages=num_pages, peaked_frac=peaked_frac, hq=hq, hkv=hkv,
                     head_dim=head_dim)
    if isinstance(q_rows, (list, tuple)):
        case.meta["cu_seqlens_q"] = [int(x) for x in np.concatenate([[0], np.cumsum(q_rows)])]
    return case


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw BF16 bit patterns of a tensor as a host numpy uint16 array (a view-copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


# --------------------------------------------------------------------------------------
# The named workloads (sizes from the pages' serving tiers and profile).
# --------------------------------------------------------------------------------------
GIB = 1 << 30


def pool_pages_for_bytes(nbytes, block_size, hkv=HKV, head_dim=HEAD_DIM):
    """Pages of K+V that fit in nbytes: each page holds BS*Hkv*D BF16 for K and for V."""
    return nbytes // (2 * block_size * hkv * head_dim * 2)


def tiny_decode(device="cpu"):
    """1 sequence, 1700 prior tokens + the new token at position 1700 (1701 keys),
    BS 832 (3 logical pages) over a seeded permutation of an 8-page pool."""
    return paged_case(1001, [1701], 832, 8, new_tokens=1, device=device)


def decode_8k(block_size=832, device="cpu"):
    """1 sequence of 8192 keys over a shuffled 64-page pool, BS 832 or 784."""
    return paged_case(1002, [8192], block_size, 64, device=device)


def decode_sweep(context, device="cpu", block_size=832):
    """1 sequence of `context` keys in a 1 GiB K+V pool, 5% of K rows scaled x8."""
    npg = pool_pages_for_bytes(GIB, block_size)
    return paged_case(1003, [context], block_size, npg, peaked_frac=0.05, device=device)


def decode_sweep_rotation(context, device="cpu", block_size=832, max_seqs=64):
    """As decode_sweep, with as many sequences of `context` keys as the 1 GiB pool holds
    on disjoint pages (at most max_seqs): a timing loop that decodes them one per step in
    turn reads each sequence's K/V again only after the others', more than L2 holds."""
    npg = pool_pages_for_bytes(GIB, block_size)
    n = min(max_seqs, npg // -(-context // block_size))
    return paged_case(1003, [context] * n, block_size, npg, peaked_frac=0.05, device=device)


def prefill_chunk(device="cpu", q_len=4096, q_start=4096, block_size=832, num_pages=64):
    """q=4096 causal chunk at positions 4096..8191 over 4096 prior paged tokens."""
    return paged_case(1004, [q_start + q_len], block_size, num_pages, q_rows=q_len,
                      q_start=q_start, device=device)


def prefill_tail(device="cpu", block_size=832, num_pages=24):
    """The prompt's last, shorter chunk: q=1685 causal rows at positions 12288..13972 over
    12288 prior paged tokens (three q=4096 chunks before it)."""
    return paged_case(1006, [12288 + 1685], block_size, num_pages, q_rows=1685,
                      q_start=12288, device=device)


def prefill_first(device="cpu", block_size=832, num_pages=16):
    """The prompt's first chunk: q=4096 causal rows at positions 0..4095, no prior tokens."""
    return paged_case(1007, [4096], block_size, num_pages, q_rows=4096, q_start=0,
                      device=device)


def prefill_mixed(device="cpu", block_size=832, num_pages=96):
    """A mixed batch of chunked prefills, as a serving step schedules them: four
    sequences whose chunks (1024, 4096, 1685 and 512 rows) sit at the end of 3072, 8192,
    13973 and 512 keys."""
    return paged_case(1008, [3072, 8192, 13973, 512], block_size, num_pages,
                      q_rows=[1024, 4096, 1685, 512], device=device)


def batched_decode(device="cpu", num_seqs=16, lo=4096, hi=32768, block_size=832,
                   num_pages=640, seed=1005):
    """16 sequences with lengths uniform in [4096, 32768], one new token each, block
    tables drawn without replacement from a shared shuffled pool of 640 pages.  The
    lengths always come from seed 1005; `seed` draws the data and the pages."""
    rng = np.random.default_rng(1005)
    lens = rng.integers(lo, hi + 1, size=num_seqs).tolist()
    return paged_case(seed, lens, block_size, num_pages, new_tokens=1, device=device)
