"""Seeded synthetic inputs for the PagedAttention hot path.

This module only draws inputs: request lengths, block tables, copy-on-write
pairs, and N(0,1) tensors.  It holds none of the method's arithmetic (no slot
mapping, no attention, no copy); both the CUDA path and the oracle consume what
it produces, and neither is imported here.

The named workloads follow the shapes the pages' subject implies (16-token
blocks, per-request block tables drawn from one physical pool, shared prefix
blocks, continuous batches that mix chunked prefills and decodes):

1. ``tiny``   -- fp32, 4 requests, seq_lens {5, 16, 17, 40}, one query token
   each, 2 query heads over 1 KV head, head_dim 64, pool of 16 blocks assigned
   by a seeded permutation, scale 1/sqrt(64).
2. ``decode`` -- bf16, 64 requests, seq_lens uniform in [128, 4096], one query
   token, 32/8 heads, head_dim 128, pool of 20000 blocks drawn by seeded shuffle.
3. ``prefix`` -- bf16, 256 requests sharing one 1024-token prefix (the same 64
   physical blocks) plus unique suffixes uniform in [64, 512]; the block that
   holds each request's newest position is copied (copy-on-write) to a fresh
   block and the table repointed at the copy; pool of 20000.
4. ``mixed``  -- bf16 continuous-batching step with an 8192-token budget:
   8 chunked-prefill chunks of 512 query tokens after a cached context uniform in
   [0, 3072], then 4096 decode requests with seq_lens uniform in [256, 2048];
   pool = ceil(1.1 x blocks needed).
5. ``long``   -- bf16, 32 requests of 32768 tokens (2048 blocks each), 64/8
   heads, head_dim 128, pool of 70000.
6. ``prefill`` -- the chunk half of ``mixed`` on its own: 8 chunked-prefill chunks
   of 512 query tokens after a cached context uniform in [0, 3072]; pool =
   ceil(1.1 x blocks needed).  Used to measure the prefill kernel alone.

Every draw is seeded (``seed = 248000 + index`` by default); uniform integer
ranges are inclusive.  Lengths, permutations and pairs come from a numpy
generator on the host; bulk tensors from a torch generator on the device they
are made on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16
NAMES = ("tiny", "decode", "prefix", "mixed", "long", "prefill")
BASE_SEED = 248000


@dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray            # int32 [num_seqs]; context incl. this step's query tokens
    query_start_loc: np.ndarray     # int32 [num_seqs + 1]
    block_tables: np.ndarray        # int32 [num_seqs, max_blocks]; -1 past each request's blocks
    seed: int
    cow_src: np.ndarray | None = None
    cow_dst: np.ndarray | None = None
    block_tables_before_cow: np.ndarray | None = None
    notes: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def torch_dtype(self):
        import torch
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def make_tensors(self, device="cpu", gen_device=None, cache_chunk_blocks: int = 4096) -> dict:
        """Draw q, the new tokens' k/v and a fully populated K/V pool, all N(0,1).

        ``gen_device`` is where the random numbers are drawn (default: ``device``);
        drawing on the host and moving to the GPU gives both sides the same
        values for small cases, drawing on the GPU keeps large pools fast.
        """
        import torch
        dev = torch.device(device)
        gdev = torch.device(gen_device) if gen_device is not None else dev
        g = torch.Generator(device=gdev)
        g.manual_seed(self.seed)
        dt = self.torch_dtype()
        hkv, hq, d = self.num_kv_heads, self.num_q_heads, self.head_dim
        shape = (self.num_blocks, hkv, BLOCK, d)
        out = {}
        for name in ("k_cache", "v_cache"):
            cache = torch.empty(shape, dtype=dt, device=dev)
            for b0 in range(0, self.num_blocks, cache_chunk_blocks):
                b1 = min(self.num_blocks, b0 + cache_chunk_blocks)
                x = torch.randn((b1 - b0, hkv, BLOCK, d), generator=g, device=gdev, dtype=torch.float32)
                cache[b0:b1].copy_(x.to(dt))
            out[name] = cache
        T = self.num_tokens
        out["q"] = torch.randn((T, hq, d), generator=g, device=gdev, dtype=torch.float32).to(dt).to(dev)
        out["k_new"] = torch.randn((T, hkv, d), generator=g, device=gdev, dtype=torch.float32).to(dt).to(dev)
        out["v_new"] = torch.randn((T, hkv, d), generator=g, device=gdev, dtype=torch.float32).to(dt).to(dev)
        return out


def _tables(lengths, pool_ids, max_blocks=None):
    """Hand each request ceil(L / 16) ids from ``pool_ids`` in order; pad with -1."""
    nblk = [(int(L) + BLOCK - 1) // BLOCK for L in lengths]
    mb = max(nblk) if max_blocks is None else max_blocks
    bt = np.full((len(lengths), max(mb, 1)), -1, dtype=np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        bt[i, :n] = pool_ids[pos:pos + n]
        pos += n
    return bt, pos


def _qsl(q_lens):
    return np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)


def make(name: str, seed: int | None = None) -> Workload:
    """One of the named workloads (host-side metadata; tensors via make_tensors)."""
    idx = NAMES.index(name)
    seed = BASE_SEED + idx if seed is None else seed
    rng = np.random.default_rng(seed)
    if name == "tiny":
        L = np.array([5, 16, 17, 40], dtype=np.int32)
        pool = 16
        perm = rng.permutation(pool).astype(np.int32)
        bt, _ = _tables(L, perm)
        return Workload(name, "f32", 2, 1, 64, pool, 1.0 / math.sqrt(64), L, _qsl(np.ones(4, np.int32)),
                        bt, seed)
    if name == "decode":
        L = rng.integers(128, 4096, size=64, endpoint=True).astype(np.int32)
        pool = 20000
        bt, _ = _tables(L, rng.permutation(pool).astype(np.int32))
        return Workload(name, "bf16", 32, 8, 128, pool, 1.0 / math.sqrt(128), L,
                        _qsl(np.ones(64, np.int32)), bt, seed)
    if name == "prefix":
        n, prefix_tokens = 256, 1024
        s = rng.integers(64, 512, size=n, endpoint=True).astype(np.int32)
        L = (prefix_tokens + s).astype(np.int32)
        pool = 20000
        perm = rng.permutation(pool).astype(np.int32)
        n_prefix = prefix_tokens // BLOCK
        prefix_ids = perm[:n_prefix]
        suffix_bt, used = _tables(s, perm[n_prefix:])
        mb = n_prefix + suffix_bt.shape[1]
        before = np.full((n, mb), -1, dtype=np.int32)
        before[:, :n_prefix] = prefix_ids
        before[:, n_prefix:] = suffix_bt
        # copy-on-write: the block that holds each request's newest position is
        # copied into a fresh block and the table entry repointed at the copy
        fresh = perm[n_prefix + used:n_prefix + used + n]
        last_logical = (L - 1) // BLOCK
        cow_src = before[np.arange(n), last_logical].copy()
        cow_dst = fresh.astype(np.int32)
        after = before.copy()
        after[np.arange(n), last_logical] = cow_dst
        return Workload(name, "bf16", 32, 8, 128, pool, 1.0 / math.sqrt(128), L,
                        _qsl(np.ones(n, np.int32)), after, seed, cow_src=cow_src, cow_dst=cow_dst,
                        block_tables_before_cow=before,
                        notes={"prefix_blocks": n_prefix, "shared_prefix_ids": prefix_ids})
    if name == "mixed":
        n_chunks, chunk, n_dec = 8, 512, 4096
        ctx = rng.integers(0, 3072, size=n_chunks, endpoint=True).astype(np.int32)
        L_pre = ctx + chunk
        L_dec = rng.integers(256, 2048, size=n_dec, endpoint=True).astype(np.int32)
        L = np.concatenate([L_pre, L_dec]).astype(np.int32)
        q = np.concatenate([np.full(n_chunks, chunk, np.int32), np.ones(n_dec, np.int32)])
        need = int(sum((int(x) + BLOCK - 1) // BLOCK for x in L))
        pool = int(math.ceil(1.1 * need))
        bt, _ = _tables(L, rng.permutation(pool).astype(np.int32))
        return Workload(name, "bf16", 32, 8, 128, pool, 1.0 / math.sqrt(128), L, _qsl(q), bt, seed,
                        notes={"prefill_chunks": n_chunks, "chunk": chunk, "decodes": n_dec})
    if name == "long":
        n, ctx = 32, 32768
        L = np.full(n, ctx, dtype=np.int32)
        pool = 70000
        bt, _ = _tables(L, rng.permutation(pool).astype(np.int32))
        return Workload(name, "bf16", 64, 8, 128, pool, 1.0 / math.sqrt(128), L,
                        _qsl(np.ones(n, np.int32)), bt, seed)
    if name == "prefill":
        n_chunks, chunk = 8, 512
        ctx = rng.integers(0, 3072, size=n_chunks, endpoint=True).astype(np.int32)
        L = (ctx + chunk).astype(np.int32)
        need = int(sum((int(x) + BLOCK - 1) // BLOCK for x in L))
        pool = int(math.ceil(1.1 * need))
        bt, _ = _tables(L, rng.permutation(pool).astype(np.int32))
        return Workload(name, "bf16", 32, 8, 128, pool, 1.0 / math.sqrt(128), L,
                        _qsl(np.full(n_chunks, chunk, np.int32)), bt, seed,
                        notes={"prefill_chunks": n_chunks, "chunk": chunk})
    raise KeyError(name)


def shared_prefix_case(seed: int, prefix_blocks=(5, 33, 70), members=(9, 40, 3), num_kv_heads: int = 2,
                       group: int = 4, max_suffix: int = 300, bystanders: int = 6, bad_hints: bool = True,
                       long_suffix: int = 0) -> tuple[Workload, dict]:
    """A decode batch with shared-prefix groups, and the group hints for it.

    Group g's ``members[g]`` decode requests all start with the same
    ``prefix_blocks[g]`` physical blocks, then a suffix of U[1, max_suffix] tokens in
    blocks of their own (``long_suffix`` > 0 gives the first member of each group that
    many suffix tokens instead).  ``bystanders`` more requests -- decodes and
    prefill chunks -- have tables of their own.  Requests are shuffled.  With
    ``bad_hints`` the hint lists also name requests that must not be treated as
    members: a prefill chunk and a decode whose context ends inside the prefix (both
    with tables that start with the prefix), a request listed in two groups, and a
    decode whose table does not start with the prefix.  Returns the workload and
    ``{"prefix_block_tables", "prefix_num_blocks", "member_start", "member_seqs"}``.
    """
    rng = np.random.default_rng(seed)
    G = len(prefix_blocks)
    reqs = []  # (q_len, L, group or -1, table_is_prefixed, hint_groups)
    for g in range(G):
        P = prefix_blocks[g] * BLOCK
        for m in range(members[g]):
            sfx = long_suffix if (long_suffix and m == 0) else int(rng.integers(1, max_suffix, endpoint=True))
            reqs.append((1, P + sfx, g, True, [g]))
    for b in range(bystanders):
        if b % 2 == 0:
            reqs.append((1, int(rng.integers(1, 1500, endpoint=True)), -1, False, []))
        else:
            q = int(rng.integers(2, 150, endpoint=True))
            reqs.append((q, q + int(rng.integers(0, 400, endpoint=True)), -1, False, []))
    if bad_hints:
        P0 = prefix_blocks[0] * BLOCK
        reqs.append((37, P0 + 60, 0, True, [0]))                    # a prefill chunk after the prefix
        reqs.append((1, max(1, P0 - 3), 0, True, [0]))             # context ends inside the prefix
        g1 = 1 % G
        reqs.append((1, prefix_blocks[g1] * BLOCK + 20, g1, True, [g1, 0]))  # listed in two groups
        reqs.append((1, prefix_blocks[g1] * BLOCK + 50, -1, False, [g1]))   # its table is its own
    order = rng.permutation(len(reqs))
    reqs = [reqs[k] for k in order]
    n = len(reqs)
    q_lens = np.array([r[0] for r in reqs], np.int32)
    L = np.array([r[1] for r in reqs], np.int32)
    need_own = sum((int(r[1]) + BLOCK - 1) // BLOCK for r in reqs)
    pool = sum(prefix_blocks) + need_own + 11
    ids = rng.permutation(pool).astype(np.int32)
    prefix_ids, pos = [], 0
    for g in range(G):
        prefix_ids.append(ids[pos:pos + prefix_blocks[g]])
        pos += prefix_blocks[g]
    mb = max((int(x) + BLOCK - 1) // BLOCK for x in L) + 1
    bt = np.full((n, mb), -1, np.int32)
    for i, (q, Li, g, prefixed, _) in enumerate(reqs):
        nb = (Li + BLOCK - 1) // BLOCK
        k = 0
        if prefixed:
            k = min(nb, prefix_blocks[g])
            bt[i, :k] = prefix_ids[g][:k]
        bt[i, k:nb] = ids[pos:pos + nb - k]
        pos += nb - k
    lists = [[] for _ in range(G)]
    for i, r in enumerate(reqs):
        for g in r[4]:
            lists[g].append(i)
    member_start = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
    member_seqs = np.array([i for x in lists for i in x], np.int32)
    mpb = max(prefix_blocks)
    ptab = np.full((G, mpb), -1, np.int32)
    for g in range(G):
        ptab[g, :prefix_blocks[g]] = prefix_ids[g]
    w = Workload(f"shared{seed}", "bf16", group * num_kv_heads, num_kv_heads, 128, pool, 1.0 / math.sqrt(128), L,
                 _qsl(q_lens), bt, seed)
    return w, {"prefix_block_tables": ptab, "prefix_num_blocks": np.array(prefix_blocks, np.int32),
               "member_start": member_start, "member_seqs": member_seqs}


def random_case(seed: int, num_seqs: int = 5, max_ctx: int = 80, max_q: int = 40,
                group: int = 2, num_kv_heads: int = 2, head_dim: int = 64, dtype: str = "f32",
                decode_frac: float = 0.4, pool_slack: int = 7, extra_table_cols: int = 2) -> Workload:
    """A small mixed batch for tests: random context lengths and query counts
    (some decodes with one query token, some prefill chunks with a prior
    context), tables drawn from a shuffled pool with spare blocks."""
    rng = np.random.default_rng(seed)
    q_lens, L = [], []
    for _ in range(num_seqs):
        if rng.random() < decode_frac:
            q = 1
        else:
            q = int(rng.integers(1, max_q, endpoint=True))
        ctx = int(rng.integers(0, max(0, max_ctx - q), endpoint=True))
        q_lens.append(q)
        L.append(ctx + q)
    L = np.array(L, dtype=np.int32)
    need = int(sum((int(x) + BLOCK - 1) // BLOCK for x in L))
    pool = need + pool_slack
    mb = max((int(x) + BLOCK - 1) // BLOCK for x in L) + extra_table_cols
    bt, _ = _tables(L, rng.permutation(pool).astype(np.int32), max_blocks=mb)
    scale = 1.0 / math.sqrt(head_dim)
    return Workload(f"random{seed}", dtype, group * num_kv_heads, num_kv_heads, head_dim, pool, scale, L,
                    _qsl(np.array(q_lens, np.int32)), bt, seed)


def sized_case(seed: int, seq_lens, q_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
               dtype: str, pool: int | None = None, scale: float | None = None) -> Workload:
    """A batch with given lengths; tables drawn from a shuffled pool."""
    rng = np.random.default_rng(seed)
    L = np.asarray(seq_lens, dtype=np.int32)
    q = np.asarray(q_lens, dtype=np.int32)
    need = int(sum((int(x) + BLOCK - 1) // BLOCK for x in L))
    pool = need + 3 if pool is None else pool
    bt, _ = _tables(L, rng.permutation(pool).astype(np.int32))
    scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
    return Workload(f"sized{seed}", dtype, num_q_heads, num_kv_heads, head_dim, pool, scale, L, _qsl(q), bt,
                    seed)
