"""Seeded synthetic inputs for the DSA indexer paged MQA-logits.

This module generates input bytes only.  It holds none of the indexer's
arithmetic (no dot products, no ReLU, no head weighting, no scaling, no
masking): it draws random numbers with a CPU ``torch.Generator`` and lays them
out in the cache formats the pages describe.  The CUDA path and the fp64
oracle both consume exactly these bytes.

Layouts (per physical page of P = 64 positions, D = 128):
  * fp8 keys: P*D e4m3 bytes, position-major, then P fp32 scales; one page is
    8,448 bytes.  "The Dispatch Wire: Connecting a Triton Indexer Kernel to
    Production Inference", section "The Reasoning and Decision-Making".
  * bf16 keys: P*D bf16 values, 256 bytes per position, no scale section;
    one page is 16,384 bytes.  "The Dispatch Decision: Wiring a Triton Kernel
    into Production", section "The Problem That Led Here".

Value distributions: q ~ N(0,1) rounded to bf16; w ~ N(0,1)/8 in fp32; fp8
keys are the round-to-nearest-even, saturating e4m3 cast of N(0,1)/s with a
per-position scale s ~ U[0.5, 2] stored beside them; bf16 keys are N(0,1)
rounded to bf16.  The five validation shapes printed on "The Final Gate:
Validating a Custom Triton Indexer Kernel Before Production Deployment",
section "What the Test Output Reveals", are available as extra decode cases.

Pages that no valid position references are filled with a poison pattern
(NaN keys and NaN scales) so that a stray read shows up as NaN in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

KV_E4M3 = 0
KV_BF16 = 1
H = 64
D = 128
P = 64
FP8_PAGE_BYTES = P * D + P * 4          # 8,448
FP8_SCALE_OFFSET = P * D                # 8,192
BF16_PAGE_BYTES = P * D * 2             # 16,384
POISON_E4M3 = 0x7F                      # e4m3 NaN code
POISON_BF16 = 0x7FC0                    # bf16 quiet NaN
POISON_F32 = 0x7FC00000                 # fp32 quiet NaN


@dataclass
class Workload:
    """One call's worth of inputs, host-resident (numpy)."""
    name: str
    kind: str                   # "decode", "prefill" or "topk" (decode + top-k selection)
    kv_dtype: int               # KV_E4M3 or KV_BF16
    R: int                      # rows: requests (decode) or queries (prefill)
    W: int                      # block-table width in pages
    q_bits: np.ndarray          # uint16 [R, H, D], bf16 bit patterns
    w: np.ndarray               # float32 [R, H]
    kcache: np.ndarray          # uint8 [num_pages * page_stride]
    page_stride: int            # bytes between consecutive physical pages
    num_pages: int
    kscale_offset: int | None   # byte offset of page 0's scales, None = 1.0
    block_table: np.ndarray     # int32 [rows_bt, W]
    bt_stride: int              # W, or 0 when all rows share one row
    seqlens: np.ndarray         # int32 [R]
    H: int = H
    D: int = D
    P: int = P
    meta: dict = field(default_factory=dict)

    @property
    def valid_positions(self) -> int:
        return int(np.clip(self.seqlens.astype(np.int64), 0, self.W * self.P).sum())

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move (read + write) for one call.

        Keys and scales of every valid position, q and w of every row, the
        block-table entries of valid pages, the row lengths, and 4 bytes of
        output for every position of the fixed [R, W*P] output (the -inf fill
        is part of the contract).  Prefill rows of one request share its
        block table and key stream: the keys of its longest row are read
        once.
        """
        per_pos = D + 4 if self.kv_dtype == KV_E4M3 else 2 * D
        L = np.clip(self.seqlens.astype(np.int64), 0, self.W * self.P)
        if self.kind == "prefill" and self.bt_stride == 0:
            key_bytes = int(L.max(initial=0)) * per_pos
            bt_bytes = int(math.ceil(L.max(initial=0) / self.P)) * 4
        elif self.kind == "prefill" and "groups" in self.meta:
            # the query tokens of one request share its keys: read once
            lmax = [int(L[a:a + n].max(initial=0)) for a, n in self.meta["groups"]]
            key_bytes = sum(lmax) * per_pos
            bt_bytes = sum(int(math.ceil(m / self.P)) for m in lmax) * 4
        else:
            key_bytes = int(L.sum()) * per_pos
            bt_bytes = int(np.ceil(L / self.P).sum()) * 4
        row_bytes = self.R * (H * D * 2 + H * 4 + 4)
        if self.kind == "topk":      # k positions and their logits per row
            out_bytes = self.R * self.meta["k_top"] * 8
        else:
            out_bytes = self.R * self.W * self.P * 4
        return key_bytes + bt_bytes + row_bytes + out_bytes

    def flops(self) -> int:
        """2*H*D per valid (row, position) pair: the q.k contraction."""
        return 2 * self.H * self.D * self.valid_positions


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _loguniform_int(g: torch.Generator, n: int, lo: int, hi: int) -> torch.Tensor:
    u = torch.rand(n, generator=g, dtype=torch.float64)
    v = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return v.floor().to(torch.int64).clamp(lo, hi)


def _fp8_pool(g: torch.Generator, num_pages: int, used: np.ndarray) -> np.ndarray:
    """Pool of fused fp8 pages; pages listed in `used` get data, others poison."""
    pool = np.empty((num_pages, FP8_PAGE_BYTES), dtype=np.uint8)
    pool[:, :FP8_SCALE_OFFSET] = POISON_E4M3
    pool[:, FP8_SCALE_OFFSET:].view(np.uint32)[:] = POISON_F32
    n = len(used)
    if n:
        s = torch.rand(n, P, generator=g) * 1.5 + 0.5          # U[0.5, 2]
        x = (torch.randn(n, P, D, generator=g) / s[:, :, None]).clamp(-448.0, 448.0)
        vals = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        pool[used, :FP8_SCALE_OFFSET] = vals.reshape(n, P * D)
        pool[used, FP8_SCALE_OFFSET:] = s.numpy().astype(np.float32).view(np.uint8).reshape(n, P * 4)
    return pool.reshape(-1)


def _bf16_pool(g: torch.Generator, num_pages: int, used: np.ndarray) -> np.ndarray:
    pool = np.empty((num_pages, P * D), dtype=np.uint16)
    pool[:] = POISON_BF16
    n = len(used)
    if n:
        pool[used] = _bf16_bits(torch.randn(n, P * D, generator=g))
    return pool.view(np.uint8).reshape(-1)


def _rows(g: torch.Generator, R: int) -> tuple[np.ndarray, np.ndarray]:
    q = _bf16_bits(torch.randn(R, H, D, generator=g))
    w = (torch.randn(R, H, generator=g) / 8).numpy().astype(np.float32)
    return q, w


def wide_range_queries(R: int, seed: int, outlier_d: int | None = None) -> np.ndarray:
    """bf16 query bits [R, H, D] whose heads span a wide dynamic range:
    every head has a magnitude m = 2^U{-3..3} and one outlier element of
    magnitude 256 * m with a random sign (at a random index, or at
    `outlier_d` in every head); the other elements are sign * m * 2^U[-6, 0],
    so they reach down to 2^-14 of the head's largest, one in eight of them
    exactly zero; every 16th head is all zero."""
    g = _gen(seed)
    mag = 2.0 ** torch.randint(-3, 4, (R, H, 1), generator=g).double()
    sign = torch.sign(torch.randn(R, H, D, generator=g, dtype=torch.float64))
    x = sign * mag * 2.0 ** (-6.0 * torch.rand(R, H, D, generator=g, dtype=torch.float64))
    x[torch.rand(R, H, D, generator=g) < 0.125] = 0.0
    if outlier_d is None:
        idx = torch.randint(0, D, (R, H, 1), generator=g)
    else:
        idx = torch.full((R, H, 1), int(outlier_d), dtype=torch.int64)
    osign = torch.sign(torch.randn(R, H, 1, generator=g, dtype=torch.float64))
    x.scatter_(2, idx, osign * mag * 256.0)
    x[:, ::16, :] = 0.0
    return _bf16_bits(x.float())


def zero_key_dim(w: "Workload", d: int) -> None:
    """Set element d of every key in w's pool to zero (in place)."""
    pool = w.kcache.reshape(w.num_pages, w.page_stride)
    if w.kv_dtype == KV_E4M3:
        pool[:, :FP8_SCALE_OFFSET].reshape(w.num_pages, P, D)[:, :, d] = 0
    else:
        pool.view(np.uint16).reshape(w.num_pages, P, D)[:, :, d] = 0


def _used_pages(bt: np.ndarray, seqlens: np.ndarray, bt_stride: int) -> np.ndarray:
    used = []
    for r in range(len(seqlens)):
        row = bt[0] if bt_stride == 0 else bt[r]
        n = int(math.ceil(max(int(seqlens[r]), 0) / P))
        used.append(row[:min(n, row.shape[0])])
    if not used:
        return np.zeros(0, dtype=np.int64)
    return np.unique(np.concatenate(used)).astype(np.int64)


def _assemble(name, kind, kv_dtype, g, W, bt, seqlens, num_pages, bt_stride,
              R=None, meta=None) -> Workload:
    R = len(seqlens) if R is None else R
    used = _used_pages(bt, seqlens, bt_stride)
    # rows are drawn before the pool so that a row's q/w do not depend on the
    # pool size
    q, w = _rows(g, R)
    if kv_dtype == KV_E4M3:
        kc, stride, koff = _fp8_pool(g, num_pages, used), FP8_PAGE_BYTES, FP8_SCALE_OFFSET
    else:
        kc, stride, koff = _bf16_pool(g, num_pages, used), BF16_PAGE_BYTES, None
    return Workload(name=name, kind=kind, kv_dtype=kv_dtype, R=R, W=W,
                    q_bits=q, w=w, kcache=kc, page_stride=stride,
                    num_pages=num_pages, kscale_offset=koff,
                    block_table=np.ascontiguousarray(bt, dtype=np.int32),
                    bt_stride=bt_stride,
                    seqlens=np.ascontiguousarray(seqlens, dtype=np.int32),
                    meta=dict(meta or {}))


def decode_uniform(name: str, B: int, W: int, max_len: int, pool: int,
                   seed: int = 0, kv_dtype: int = KV_E4M3) -> Workload:
    """B requests, L ~ U{1..max_len}, block table = a random permutation of a
    pool of `pool` pages (first B*W entries), as in the pages' validation."""
    g = _gen(seed)
    seqlens = torch.randint(1, max_len + 1, (B,), generator=g).numpy()
    bt = torch.randperm(pool, generator=g)[: B * W].numpy().reshape(B, W)
    return _assemble(name, "decode", kv_dtype, g, W, bt, seqlens, pool, W)


def decode_with_lengths(name: str, lengths, W: int, seed: int = 0,
                        kv_dtype: int = KV_E4M3, pool: int | None = None) -> Workload:
    """Requests with the given lengths; the block table is a random
    permutation of a pool of `pool` pages (default len(lengths) * W)."""
    g = _gen(seed)
    seqlens = np.asarray(lengths, dtype=np.int64)
    B = len(seqlens)
    pool = B * W if pool is None else pool
    bt = torch.randperm(pool, generator=g)[: B * W].numpy().reshape(B, W)
    return _assemble(name, "decode", kv_dtype, g, W, bt, seqlens, pool, W)


def decode_loguniform(name: str, B: int, W: int, lo: int, hi: int,
                      pages_per_req: int, seed: int = 0,
                      kv_dtype: int = KV_E4M3, seqlens: np.ndarray | None = None,
                      poison_tail: bool = True) -> Workload:
    """B requests with L = floor(exp(U[ln lo, ln hi])).  Each request owns
    `pages_per_req` pages of a shuffled pool; entries past its valid pages
    point at one poison page (index B*pages_per_req) when `poison_tail`,
    else at the rest of its own (unreferenced, poisoned) pages."""
    g = _gen(seed)
    if seqlens is None:
        seqlens = _loguniform_int(g, B, lo, hi).numpy()
    else:
        _loguniform_int(g, B, lo, hi)         # keep the stream aligned
    n_data = B * pages_per_req
    perm = torch.randperm(n_data, generator=g).numpy().reshape(B, pages_per_req)
    poison = n_data
    bt = np.full((B, W), poison, dtype=np.int64)
    for b in range(B):
        n = int(math.ceil(int(seqlens[b]) / P))
        if poison_tail:
            bt[b, :n] = perm[b, :n]
        else:
            m = min(W, pages_per_req)
            bt[b, :m] = perm[b, :m]
    return _assemble(name, "decode", kv_dtype, g, W, bt, seqlens, n_data + 1, W,
                     meta={"lo": lo, "hi": hi})


def prefill_causal(name: str, n_q: int, W: int, first_limit: int, seed: int = 0,
                   kv_dtype: int = KV_BF16) -> Workload:
    """n_q query tokens of one request sharing one block table (a random
    permutation of W pages); query i may see positions 0..first_limit+i, so
    its length is first_limit + i + 1."""
    g = _gen(seed)
    bt = torch.randperm(W, generator=g).numpy().reshape(1, W)
    seqlens = (first_limit + 1 + np.arange(n_q)).astype(np.int32)
    return _assemble(name, "prefill", kv_dtype, g, W, bt, seqlens, W, 0, R=n_q,
                     meta={"first_limit": first_limit})


def prefill_varlen(name: str, requests, seed: int = 0, kv_dtype: int = KV_BF16) -> Workload:
    """Several requests' prefill chunks in one call: request r brings n_r
    query tokens at the end of a context of c_r positions (query j of it may
    see positions 0..c_r - n_r + j), over its own pages of a shuffled pool.
    Every query token has a block-table row of its own (a copy of its
    request's row), so bt_stride = W; entries past a request's pages point
    at one poison page."""
    g = _gen(seed)
    reqs = [(int(n), int(c)) for n, c in requests]
    W = max(int(math.ceil(c / P)) for _, c in reqs)
    npages = [int(math.ceil(c / P)) for _, c in reqs]
    n_data = sum(npages)
    perm = torch.randperm(n_data, generator=g).numpy()
    poison = n_data
    rows, lens, groups, off, start = [], [], [], 0, 0
    for (n, c), k in zip(reqs, npages):
        row = np.full(W, poison, dtype=np.int64)
        row[:k] = perm[off:off + k]
        off += k
        for j in range(n):
            rows.append(row)
            lens.append(c - n + j + 1)
        groups.append((start, n))
        start += n
    bt = np.stack(rows)
    return _assemble(name, "prefill", kv_dtype, g, W, bt, np.asarray(lens), n_data + 1, W,
                     meta={"requests": reqs, "groups": groups})


def request_tables(w: Workload):
    """The request offsets (cu_q, host ints) and one block-table row per
    request of a several-request prefill workload (its per-query rows are
    copies of their request's row)."""
    groups = w.meta["groups"]
    cu = [0]
    for _, n in groups:
        cu.append(cu[-1] + n)
    rows = []
    for b, (a, n) in enumerate(groups):
        if n > 0:
            rows.append(w.block_table[a])
        else:                                   # no query token carries its row: any valid row
            rows.append(np.full(w.W, w.num_pages - 1, dtype=w.block_table.dtype))
    return cu, np.stack(rows)


# ---------------------------------------------------------------------------
# The named workloads.

def cfg1() -> Workload:
    """Decode fp8, B=1, W=8, L ~ U{1..512}, pool of 16 pages, seed 0."""
    g = _gen(0)
    seqlens = torch.randint(1, 513, (1,), generator=g).numpy()
    bt = torch.randperm(16, generator=g)[:8].numpy().reshape(1, 8)
    return _assemble("decode_fp8_B1_W8", "decode", KV_E4M3, g, 8, bt, seqlens, 16, 8)


def cfg2a() -> Workload:
    """Decode fp8, B=16, W=32 (8K-token cap: 2,048 positions), L ~ U{1..2048}."""
    return decode_uniform("decode_fp8_B16_W32", 16, 32, 2048, 512, seed=0)


def cfg2b() -> Workload:
    """Decode fp8, B=32, W=16, L ~ U{1..1024}."""
    return decode_uniform("decode_fp8_B32_W16", 32, 16, 1024, 512, seed=0)


def cfg3(W: int = 4097) -> Workload:
    """Decode fp8, B=64, L log-uniform 512..32768; table width W (4097 =
    262,208 positions uncapped; 512 = the smallest width that holds the
    same lengths)."""
    return decode_loguniform(f"decode_fp8_B64_W{W}", 64, W, 512, 32768, 512, seed=0)


def cfg3_short(W: int = 4097) -> Workload:
    """Decode fp8, B=64, L log-uniform 512..2048, width W (4097 vs 32):
    the same lengths under the uncapped and the 8K-token-capped table."""
    return decode_loguniform(f"decode_fp8_B64_short_W{W}", 64, W, 512, 2048, 32, seed=1)


def cfg4() -> Workload:
    """Decode bf16, B=64, W=2048, L log-uniform 4096..131072, scale 1."""
    return decode_loguniform("decode_bf16_B64_W2048", 64, 2048, 4096, 131072, 2048,
                             seed=0, kv_dtype=KV_BF16, poison_tail=False)


def cfg4_small() -> Workload:
    """Config 4's kernel at a size for detailed profiling: decode bf16, B=64,
    W=512, L log-uniform 1024..32768 (a 537 MB pool; the call moves more
    than L2 holds)."""
    return decode_loguniform("decode_bf16_B64_W512", 64, 512, 1024, 32768, 512,
                             seed=0, kv_dtype=KV_BF16, poison_tail=False)


def cfg5() -> Workload:
    """Prefill bf16: 4,096 queries of one request, 352 pages (22,528
    positions), causal limit of query i = 18432 + i."""
    return prefill_causal("prefill_bf16_q4096_W352", 4096, 352, 18432, seed=0)


def pages_validation_cases() -> list[Workload]:
    """The five (B, pages, max length) shapes of the pages' validation run,
    fp8 keys, with a shuffled pool twice the table size."""
    shapes = [(1, 8, 512), (16, 32, 2048), (32, 16, 1024), (4, 64, 4096), (8, 4, 256)]
    out = []
    for i, (B, W, Lmax) in enumerate(shapes):
        out.append(decode_uniform(f"pages_val_B{B}_W{W}", B, W, Lmax, 2 * B * W, seed=100 + i))
    return out


@dataclass
class StoreWorkload:
    """One key-cache store call: n new key rows and their slots, plus the
    pool they go into (host-resident; unwritten slots keep their poison)."""
    name: str
    kv_dtype: int
    k_bits: np.ndarray          # uint16 [n, D], bf16 bit patterns
    slots: np.ndarray           # int32 [n]: page * P + slot, < 0 = skip
    kcache: np.ndarray          # uint8 [num_pages * page_stride]
    page_stride: int
    num_pages: int
    kind: str = "store"
    D: int = D
    P: int = P
    meta: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.slots.shape[0])

    @property
    def valid_positions(self) -> int:
        """Rows actually stored (the store's unit of work)."""
        return int(((self.slots >= 0) & (self.slots < self.num_pages * self.P)).sum())

    def algorithmic_bytes(self) -> int:
        """Every row's 256 bytes of bf16 and 4-byte slot are read; each stored
        row writes D codes + a 4-byte scale (fp8) or 2*D bytes (bf16)."""
        written = (self.D + 4) if self.kv_dtype == KV_E4M3 else 2 * self.D
        return self.n * (2 * self.D + 4) + self.valid_positions * written

    def flops(self) -> int:
        return 0


def store_rows(name: str, n: int, num_pages: int, seed: int = 0, kv_dtype: int = KV_E4M3,
               n_skip: int = 0, n_bad: int = 0) -> StoreWorkload:
    """n key rows of N(0, 1) x a per-row factor U[0.01, 50] (bf16), stored to
    distinct random slots of a pool of num_pages pages; n_skip of them carry
    slot -1 and n_bad a slot past the pool."""
    g = _gen(seed)
    x = torch.randn(n, D, generator=g) * (torch.rand(n, 1, generator=g) * 49.99 + 0.01)
    k = _bf16_bits(x).reshape(n, D)
    slots = torch.randperm(num_pages * P, generator=g)[:n].numpy().astype(np.int32)
    pick = torch.randperm(n, generator=g).numpy()
    slots[pick[:n_skip]] = -1
    slots[pick[n_skip:n_skip + n_bad]] = num_pages * P + pick[n_skip:n_skip + n_bad]
    stride = FP8_PAGE_BYTES if kv_dtype == KV_E4M3 else BF16_PAGE_BYTES
    pool = np.full(num_pages * stride, 0xA5, dtype=np.uint8)
    return StoreWorkload(name=name, kv_dtype=kv_dtype, k_bits=k, slots=slots, kcache=pool,
                         page_stride=stride, num_pages=num_pages)


def cfg8() -> StoreWorkload:
    """Key-cache store, bf16 rows to fp8 pages: 65,536 rows (a long prefill
    chunk) into random slots of a 2,048-page pool."""
    return store_rows("store_fp8_n65536", 65536, 2048, seed=0)


def cfg9(k: int = 2048) -> Workload:
    """Config 3's decode call (fp8, B=64, W=4097) with top-k selection (k =
    2,048 by default): the positions and logits of each request's k best
    positions instead of the [64, 262,208] logits."""
    w = cfg3(4097)
    w.name = f"decode_topk{k}_fp8_B64_W4097"
    w.kind = "topk"
    w.meta["k_top"] = k
    return w


def cfg6() -> Workload:
    """Prefill bf16, four requests in one call with per-query table rows:
    (query tokens, context) = (256, 6144), (512, 12288), (128, 3072),
    (1024, 20480)."""
    return prefill_varlen("prefill_bf16_varlen4_q1920",
                          [(256, 6144), (512, 12288), (128, 3072), (1024, 20480)], seed=0)


def cfg6v() -> Workload:
    """Config 6's four requests called with one block-table row per request
    and the request offsets: all requests' query tiles in one launch."""
    w = cfg6()
    w.name = "prefill_bf16_varlen4_q1920_reqrows"
    w.meta["varlen"] = True
    return w


def cfg7() -> Workload:
    """Prefill with fp8 keys: 1,024 query tokens of one request over 128
    pages (8,192 positions), causal limit of query i = 7168 + i."""
    return prefill_causal("prefill_fp8_q1024_W128", 1024, 128, 7168, seed=0, kv_dtype=KV_E4M3)


NAMED = {
    "1": lambda: [cfg1()],
    "2": lambda: [cfg2a(), cfg2b()],
    "2a": lambda: [cfg2a()],
    "2b": lambda: [cfg2b()],
    "3": lambda: [cfg3(4097)],
    "3ref": lambda: [cfg3(512)],
    "3short": lambda: [cfg3_short(4097)],
    "3short_capped": lambda: [cfg3_short(32)],
    "4": lambda: [cfg4()],
    "4s": lambda: [cfg4_small()],
    "5": lambda: [cfg5()],
    "6": lambda: [cfg6()],
    "6v": lambda: [cfg6v()],
    "7": lambda: [cfg7()],
    "8": lambda: [cfg8()],
    "9": lambda: [cfg9()],
    "9k256": lambda: [cfg9(256)],
    "9k512": lambda: [cfg9(512)],
}
