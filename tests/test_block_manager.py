"""Host block manager (libpkv, include/pkv_blocks.h) against what the pages state.

"vLLM's PagedAttention" teardown, section "PagedAttention: the KV cache is paged":
  * a request gets ceil(new tokens / 16) blocks, or none at all (None) if the pool is
    short;
  * block i's hash depends on blocks 0..i, so a second request with the same first
    tokens finds the first one's physical blocks and uses them too (one more user,
    nothing copied);
  * a block with no users is free again; freed blocks that still carry a hash are
    reused only after blocks that never did.
Section "What happens when the blocks run out": a freed request's blocks are queued
last block first, so its first blocks survive longest.
"The 1960s Operating System Trick ..." page, Technical Details: samples of one prompt
use the same blocks; only the block about to change is copied.
"""
import numpy as np
import pytest

BLOCK = 16


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_248_gb300 import _build
    _build.build()
    import paged_kv_cache_248_gb300 as m
    return m


def toks(seed, n):
    return np.random.default_rng(seed).integers(0, 50000, size=n).astype(np.int32)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 31, 32, 33, 2000])
def test_allocate_takes_ceil_tokens_over_16(pkv, n):
    bm = pkv.BlockManager(200)
    assert bm.get_computed_blocks(1, toks(0, n)) == 0
    assert bm.allocate_slots(1, n) == (n + BLOCK - 1) // BLOCK
    assert len(bm.block_table(1)) == (n + BLOCK - 1) // BLOCK
    assert bm.num_free == 200 - (n + BLOCK - 1) // BLOCK
    # growing within the last block takes nothing; crossing a boundary takes one
    last = (n + BLOCK - 1) // BLOCK * BLOCK
    assert bm.allocate_slots(1, last) == 0
    assert bm.allocate_slots(1, last + 1) == 1


def test_allocate_returns_none_and_takes_nothing_when_short(pkv):
    bm = pkv.BlockManager(5)
    bm.get_computed_blocks(1, [])
    assert bm.allocate_slots(1, 3 * BLOCK) == 3
    bm.get_computed_blocks(2, [])
    assert bm.allocate_slots(2, 3 * BLOCK) is None        # needs 3, only 2 free
    assert bm.num_free == 2 and bm.block_table(2) == []
    assert bm.allocate_slots(2, 2 * BLOCK) == 2
    assert bm.num_free == 0


def test_shared_prefix_reuses_physical_blocks(pkv):
    bm = pkv.BlockManager(64)
    system = toks(1, 3 * BLOCK)
    a = np.concatenate([system, toks(2, 10)])
    assert bm.get_computed_blocks(1, a) == 0
    bm.allocate_slots(1, a.size)
    assert bm.cache_full_blocks(1, a) == 3                 # three full blocks hashed
    free_before = bm.num_free
    b = np.concatenate([system, toks(3, 25)])
    assert bm.get_computed_blocks(2, b) == 3               # the system prompt is a hit
    assert bm.block_table(2) == bm.block_table(1)[:3]      # the same physical blocks
    assert bm.num_free == free_before                       # no copy, nothing taken
    bm.allocate_slots(2, b.size)
    assert bm.block_table(2)[:3] == bm.block_table(1)[:3]
    assert set(bm.block_table(2)[3:]).isdisjoint(bm.block_table(1))


def test_hash_chains_the_whole_prefix(pkv):
    bm = pkv.BlockManager(64)
    x, y, z = toks(4, BLOCK), toks(5, BLOCK), toks(6, BLOCK)
    h_x = bm.block_hash(0, x)
    assert bm.block_hash(0, x) == h_x                       # deterministic
    assert bm.block_hash(h_x, z) != bm.block_hash(bm.block_hash(0, y), z)  # same block, other parent
    assert bm.block_hash(h_x, z, 1) != bm.block_hash(h_x, z, 0)            # extra key counts
    # a request whose third block matches but whose first does not gets no hit
    a = np.concatenate([x, y, z])
    bm.get_computed_blocks(1, a)
    bm.allocate_slots(1, a.size)
    bm.cache_full_blocks(1, a)
    b = np.concatenate([toks(7, BLOCK), y, z])
    assert bm.get_computed_blocks(2, b) == 0
    c = np.concatenate([x, y, toks(8, BLOCK)])
    assert bm.get_computed_blocks(3, c) == 2


def test_block_returns_to_pool_at_refcount_zero(pkv):
    bm = pkv.BlockManager(32)
    p = toks(9, 2 * BLOCK)
    bm.get_computed_blocks(1, p)
    bm.allocate_slots(1, p.size)
    bm.cache_full_blocks(1, p)
    bm.get_computed_blocks(2, p)                            # shares both blocks
    assert bm.num_free == 30
    bm.free(1)
    assert bm.num_free == 30                                # still referenced by request 2
    bm.free(2)
    assert bm.num_free == 32


def test_cached_free_blocks_revive_and_tail_evicted_first(pkv):
    n = 8
    bm = pkv.BlockManager(n)
    p = toks(10, 4 * BLOCK)
    bm.get_computed_blocks(1, p)
    bm.allocate_slots(1, p.size)                            # blocks 0..3
    table = bm.block_table(1)
    bm.cache_full_blocks(1, p)
    bm.free(1)                                              # cached-but-free, tail first into the queue
    assert bm.num_free == n
    # a new request with the same prompt revives them without any copy
    assert bm.get_computed_blocks(2, p) == 4 and bm.block_table(2) == table
    bm.free(2)
    # never-used blocks are taken first; then the freed request's tail before its prefix
    bm.get_computed_blocks(3, [])
    bm.allocate_slots(3, (n - 4) * BLOCK)                   # the 4 never-used blocks
    assert set(bm.block_table(3)).isdisjoint(table)
    bm.allocate_slots(3, (n - 4 + 1) * BLOCK)               # evicts one cached block
    assert bm.block_table(3)[-1] == table[-1]               # the request's last block went first
    q = np.concatenate([p[:3 * BLOCK], toks(11, BLOCK)])
    assert bm.get_computed_blocks(4, q) == 3                # the prefix survived


def test_fork_and_copy_on_write(pkv):
    bm = pkv.BlockManager(16)
    p = toks(12, 40)                                        # 3 blocks, the last partial
    bm.get_computed_blocks(1, p)
    bm.allocate_slots(1, p.size)
    parent = bm.block_table(1)
    bm.fork(1, 2)                                           # a parallel sample: shares everything
    assert bm.block_table(2) == parent and bm.num_free == 13
    src_dst = bm.cow(2, 2)                                  # the sample writes into the shared last block
    assert src_dst[0] == parent[2] and src_dst[1] not in parent
    assert bm.block_table(2) == parent[:2] + [src_dst[1]]
    assert bm.block_table(1) == parent                      # the parent keeps its block
    assert bm.cow(2, 2) == ()                               # now private: no further copy
    assert bm.cow(1, 2) == ()                               # and the parent's is private again
    assert bm.cow(2, 0) != ()                               # the first block is still shared
    full = pkv.BlockManager(3)
    full.get_computed_blocks(1, [])
    full.allocate_slots(1, 48)
    full.fork(1, 2)
    assert full.cow(2, 1) is None                           # no free block for the copy


def test_waste_is_only_the_last_partial_block(pkv):
    # paging wastes at most the tail of each request's last block (< 16 slots)
    rng = np.random.default_rng(13)
    bm = pkv.BlockManager(100000)
    lens = rng.integers(1, 5000, size=200)
    for i, L in enumerate(lens):
        bm.get_computed_blocks(i, [])
        bm.allocate_slots(i, int(L))
    u = bm.usage()
    assert u["tokens_held"] == lens.sum()
    assert u["unused_slots"] == int(sum((-L) % BLOCK for L in lens))
    assert u["unused_slots"] < BLOCK * len(lens)
    assert u["blocks_in_use"] == sum((int(L) + BLOCK - 1) // BLOCK for L in lens)


def test_errors(pkv):
    bm = pkv.BlockManager(4)
    with pytest.raises(ValueError):
        bm.allocate_slots(7, 10)                            # unknown request
    bm.get_computed_blocks(1, [])
    with pytest.raises(ValueError):
        bm.get_computed_blocks(1, [])                       # already exists
    with pytest.raises(ValueError):
        pkv.BlockManager(0)


def test_prefix_groups_from_shared_blocks(pkv):
    bm = pkv.BlockManager(64)
    system = toks(20, 3 * BLOCK)
    a = np.concatenate([system, toks(21, 10)])
    bm.get_computed_blocks(1, a)
    bm.allocate_slots(1, a.size)
    bm.cache_full_blocks(1, a)
    b = np.concatenate([system, toks(22, 30)])
    assert bm.get_computed_blocks(2, b) == 3
    bm.allocate_slots(2, b.size)
    bm.get_computed_blocks(3, toks(23, 40))       # an unrelated request
    bm.allocate_slots(3, 40)
    tables, nblk, start, members = bm.prefix_groups([3, 1, 2], max_prefix_blocks=8)
    assert nblk.tolist() == [3] and start.tolist() == [0, 2]
    assert members.tolist() == [1, 2]                 # batch indices of requests 1 and 2
    assert tables[0, :3].tolist() == bm.block_table(1)[:3]
    assert (tables[0, 3:] == -1).all()


def test_prefix_groups_take_the_shortest_common_run(pkv):
    bm = pkv.BlockManager(64)
    p = toks(24, 5 * BLOCK)
    bm.get_computed_blocks(1, p)
    bm.allocate_slots(1, p.size)
    bm.fork(1, 2)                                     # shares all 5 blocks
    bm.fork(1, 3)
    src, dst = bm.cow(3, 2)                           # request 3 diverges at block 2
    tables, nblk, start, members = bm.prefix_groups([1, 2, 3], max_prefix_blocks=8)
    assert nblk.tolist() == [2] and members.tolist() == [0, 1, 2]
    tables, nblk, _, _ = bm.prefix_groups([1, 2], max_prefix_blocks=8)
    assert nblk.tolist() == [5]
    tables, nblk, _, _ = bm.prefix_groups([1, 2], max_prefix_blocks=3)   # capped
    assert nblk.tolist() == [3] and tables[0].tolist() == bm.block_table(1)[:3]


def test_prefix_groups_limits_and_errors(pkv):
    bm = pkv.BlockManager(64)
    for g in range(3):                                # three pairs, each sharing a block
        p = toks(30 + g, BLOCK)
        bm.get_computed_blocks(10 * g, p)
        bm.allocate_slots(10 * g, p.size + 1)
        bm.fork(10 * g, 10 * g + 1)
    reqs = [0, 1, 10, 11, 20, 21]
    tables, nblk, start, members = bm.prefix_groups(reqs, max_prefix_blocks=4)
    assert len(nblk) == 3 and start.tolist() == [0, 2, 4, 6]
    tables, nblk, start, members = bm.prefix_groups(reqs, max_prefix_blocks=4, max_groups=2)
    assert len(nblk) == 2 and members.tolist() == [0, 1, 2, 3]
    single = bm.prefix_groups([0], max_prefix_blocks=4)
    assert len(single[1]) == 0 and single[2].tolist() == [0]
    with pytest.raises(ValueError):
        bm.prefix_groups([0, 99], max_prefix_blocks=4)


def _check_pool(bm, live, n_blocks):
    """Invariants of the pool against the model ``live`` (request -> its token ids)."""
    refs = {}
    unused = 0
    for r, toks in live.items():
        table = bm.block_table(r)
        assert len(table) == (toks.size + BLOCK - 1) // BLOCK, r
        assert len(set(table)) == len(table), r                      # no block twice in one table
        unused += len(table) * BLOCK - toks.size
        for k, b in enumerate(table):
            assert 0 <= b < n_blocks
            refs.setdefault(b, []).append((r, k))
    # blocks in use are exactly the referenced ones; every other block is in the free queue
    assert bm.num_free == n_blocks - len(refs)
    u = bm.usage()
    assert u["blocks_in_use"] == len(refs)
    assert u["tokens_held"] == sum(t.size for t in live.values())
    assert u["unused_slots"] == unused
    # every reference to a block sees the same token ids in the slots it has filled
    for b, holders in refs.items():
        first = None
        for r, k in holders:
            content = live[r][k * BLOCK:(k + 1) * BLOCK]
            if first is None:
                first = content
            m = min(first.size, content.size)
            assert np.array_equal(first[:m], content[:m]), (b, holders)
    return refs


@pytest.mark.parametrize("seed", [21, 22, 23, 24])
def test_random_walk_keeps_the_pool_consistent(pkv, seed):
    # New requests (often extending a known prompt, so prefix hashes hit), appends,
    # forks, copy-on-write and frees, in a seeded random order on a small pool so that
    # allocation also fails; the pool is checked against a model after every operation.
    rng = np.random.default_rng(seed)
    n_blocks = 48
    bm = pkv.BlockManager(n_blocks)
    vocab = 5  # few distinct token ids: equal blocks are common
    prompts = [rng.integers(0, vocab, size=int(rng.integers(1, 90))).astype(np.int32) for _ in range(6)]
    live, next_id, hits = {}, 0, 0
    for _ in range(600):
        op = rng.random()
        if op < 0.35 or not live:
            base = prompts[int(rng.integers(len(prompts)))]
            toks = np.concatenate([base[:int(rng.integers(0, base.size + 1))],
                                   rng.integers(0, vocab, size=int(rng.integers(0, 40)))]).astype(np.int32)
            if toks.size == 0:
                continue
            r, next_id = next_id, next_id + 1
            hit = bm.get_computed_blocks(r, toks)
            assert 0 <= hit <= toks.size // BLOCK
            hits += hit
            if bm.allocate_slots(r, toks.size) is None:
                bm.free(r)                                    # gives back the blocks it hit
            else:
                bm.cache_full_blocks(r, toks)
                live[r] = toks
        elif op < 0.55:
            r = list(live)[int(rng.integers(len(live)))]
            toks = live[r]
            add = rng.integers(0, vocab, size=int(rng.integers(1, 24))).astype(np.int32)
            table = bm.block_table(r)
            shared = sum(table[-1] in bm.block_table(o) for o in live if o != r) > 0
            if toks.size % BLOCK and shared:                  # the write would land in a shared block
                if bm.cow(r, len(table) - 1) is None:
                    continue
            if bm.allocate_slots(r, toks.size + add.size) is None:
                continue
            live[r] = np.concatenate([toks, add])
            bm.cache_full_blocks(r, live[r])
        elif op < 0.68:
            p = list(live)[int(rng.integers(len(live)))]
            c, next_id = next_id, next_id + 1
            bm.fork(p, c)
            live[c] = live[p].copy()
            assert bm.block_table(c) == bm.block_table(p)
        elif op < 0.8:
            r = list(live)[int(rng.integers(len(live)))]
            before = bm.block_table(r)
            k = int(rng.integers(len(before)))
            others = [o for o in live if o != r]
            shared = any(before[k] in bm.block_table(o) for o in others)
            free_before = bm.num_free
            res = bm.cow(r, k)
            after = bm.block_table(r)
            if not shared:
                assert res == () and after == before
            elif res is None:
                assert free_before == 0 and after == before
            else:
                src, dst = res
                assert src == before[k] and after[k] == dst and after[:k] == before[:k] and after[k + 1:] == before[k + 1:]
                assert all(dst not in bm.block_table(o) for o in others)
                assert bm.num_free == free_before - 1
        else:
            r = list(live)[int(rng.integers(len(live)))]
            bm.free(r)
            del live[r]
        _check_pool(bm, live, n_blocks)
    assert hits > 0                                           # prefix reuse was exercised
    for r in list(live):
        bm.free(r)
    assert bm.num_free == n_blocks


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_prefix_groups_properties_on_random_batches(pkv, seed):
    # Sharing made by prefix-cache hits and forks; for random batches, the groups must
    # be exactly the batch's requests that share a first block (in order of first
    # appearance), each group's prefix the longest run of leading blocks all its
    # members share (capped), and the member lists a partition of those requests.
    rng = np.random.default_rng(seed)
    bm = pkv.BlockManager(4000)
    prompts = [rng.integers(0, 3, size=int(rng.integers(16, 200))).astype(np.int32) for _ in range(5)]
    live = []
    for r in range(120):
        if live and rng.random() < 0.3:
            p = live[int(rng.integers(len(live)))]
            bm.fork(p, r)
        else:
            base = prompts[int(rng.integers(len(prompts)))]
            toks = np.concatenate([base[:int(rng.integers(1, base.size + 1))],
                                   rng.integers(0, 3, size=int(rng.integers(0, 50)))]).astype(np.int32)
            bm.get_computed_blocks(r, toks)
            assert bm.allocate_slots(r, toks.size) is not None
            bm.cache_full_blocks(r, toks)
        live.append(r)
    tables = {r: bm.block_table(r) for r in live}
    formed = 0
    for trial in range(20):
        batch = [live[i] for i in rng.choice(len(live), size=int(rng.integers(1, 60)), replace=False)]
        cap = int(rng.integers(1, 16))
        max_groups = int(rng.integers(1, 12))
        pt, pn, ms, mseq = bm.prefix_groups(batch, cap, max_groups)
        G = len(pn)
        formed += G
        assert G <= max_groups and ms[0] == 0 and len(ms) == G + 1
        first = [tables[batch[k]][0] for k in range(len(batch))]
        # groups in order of their first member's batch position, distinct first blocks
        firsts_seen = []
        for k, b in enumerate(first):
            if b not in firsts_seen:
                firsts_seen.append(b)
        shared = [b for b in firsts_seen if first.count(b) >= 2]
        assert G == min(len(shared), max_groups)
        for g in range(G):
            members = list(mseq[ms[g]:ms[g + 1]])
            assert members == [k for k, b in enumerate(first) if b == shared[g]]   # all of them, batch order
            n = int(pn[g])
            assert 1 <= n <= cap
            pre = list(pt[g][:n])
            assert all(x == -1 for x in pt[g][n:])
            for k in members:
                assert tables[batch[k]][:n] == pre
            # longest: at the cap, or some member ends there, or two members differ there
            if n < cap:
                nxt = [tables[batch[k]][n] if len(tables[batch[k]]) > n else None for k in members]
                assert None in nxt or len(set(nxt)) > 1
    assert formed > 0
