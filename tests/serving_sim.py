"""A small continuous-batching loop on top of the host block manager (test helper).

Each step packs the running requests -- decodes and prefill chunks alike -- into one
batch under a token budget ("vLLM's PagedAttention" teardown, section "Continuous
batching"), grows their block tables with allocate_slots, and asks copy-on-write for
the first block each request writes into, which a forked parallel sample may still
share ("The 1960s Operating System Trick ..." page, Technical Details).  A second
request with the same system prompt is admitted later and finds the prompt's full
blocks by their chained hashes (section "PagedAttention: the KV cache is paged").

The loop yields one ``Step`` per iteration: the block copies to make first, then
the block tables, lengths and new tokens' K/V rows of the batch.  A token's K/V rows
are a fixed function of (token id, position), so requests that share a prompt prefix
also share its K/V rows, as a model would produce them.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 16


def kv_rows(token_ids, positions, hkv, d):
    """bf16 K and V rows [n, hkv, d], a fixed function of (token id, position)."""
    ks, vs = [], []
    for t, p in zip(token_ids, positions):
        g = torch.Generator().manual_seed(int(t) * 100003 + int(p))
        ks.append(torch.randn((hkv, d), generator=g))
        vs.append(torch.randn((hkv, d), generator=g))
    if not ks:
        return torch.empty((0, hkv, d), dtype=torch.bfloat16), torch.empty((0, hkv, d), dtype=torch.bfloat16)
    return torch.stack(ks).bfloat16(), torch.stack(vs).bfloat16()


class Req:
    def __init__(self, rid, prompt, gen):
        self.rid, self.tokens, self.gen_left = rid, [int(x) for x in prompt], gen
        self.done = 0                                     # tokens whose K/V rows are in the pool


@dataclass
class Step:
    index: int
    cow_src: np.ndarray                                   # int32, copies to make before the writes
    cow_dst: np.ndarray
    block_tables: np.ndarray                              # int32 [B, max_blocks], -1 padded
    seq_lens: np.ndarray                                  # int32 [B]
    query_start_loc: np.ndarray                           # int32 [B + 1]
    k_new: torch.Tensor                                   # bf16 [T, hkv, d]
    v_new: torch.Tensor
    live: dict = field(default_factory=dict)              # rid -> (block table, tokens in the pool)
    rids: list = field(default_factory=list)              # request ids in batch order

    @property
    def num_tokens(self):
        return int(self.query_start_loc[-1])


def run(bm, hkv, d, steps=14, budget=160, seed=7, events=None):
    """Drive ``bm`` (a BlockManager) through ``steps`` iterations; yields Step objects.

    After the consumer has processed a step, every request in ``Step.live`` holds the
    K/V rows of its first n tokens in the listed blocks.  ``events`` (a dict), if
    given, records the prefix-cache hit and the copy-on-write count.
    """
    rng = np.random.default_rng(seed)
    events = {} if events is None else events
    events.update(prefix_hit=0, cow=0, finished=0, forked=False)
    system = rng.integers(1, 30000, size=3 * BLOCK + 5)
    reqs, next_id = {}, 0

    def admit(prompt, gen):
        nonlocal next_id
        r = Req(next_id, prompt, gen)
        hit = bm.get_computed_blocks(r.rid, np.asarray(prompt, np.int32))
        r.done = min(hit * BLOCK, len(r.tokens) - 1)      # at least one token to compute
        reqs[r.rid] = r
        next_id += 1
        return r, hit

    a, _ = admit(np.concatenate([system, rng.integers(1, 30000, size=40)]), 6)
    for step in range(steps):
        if step == 2:   # same system prompt: its three full blocks are found by hash
            b, hit = admit(np.concatenate([system, rng.integers(1, 30000, size=23)]), 5)
            events["prefix_hit"] = hit
            events["shared_with_a"] = bm.block_table(b.rid)[:hit] == bm.block_table(a.rid)[:hit]
        if step == 5 and a.rid in reqs:   # a parallel sample of request a: shares all of a's blocks
            child = Req(next_id, a.tokens, 4)
            child.done = a.done
            bm.fork(a.rid, child.rid)
            reqs[child.rid] = child
            next_id += 1
            events["forked"] = True
        batch, left = [], budget
        for r in reqs.values():
            n = min(len(r.tokens) - r.done, left)
            if n <= 0:
                continue
            batch.append((r, n))
            left -= n
        if not batch:
            return
        cows = []
        for r, n in batch:
            if bm.allocate_slots(r.rid, r.done + n) is None:
                raise RuntimeError("pool exhausted")
            # only the block receiving the first new token can be shared: later ones are fresh
            cw = bm.cow(r.rid, r.done // BLOCK)
            if cw is None:
                raise RuntimeError("no free block for copy-on-write")
            if cw:
                cows.append(cw)
        events["cow"] += len(cows)
        tables = [bm.block_table(r.rid) for r, _ in batch]
        bt = np.full((len(batch), max(len(t) for t in tables)), -1, np.int32)
        new_tok, new_pos, q_lens = [], [], []
        for i, ((r, n), tab) in enumerate(zip(batch, tables)):
            bt[i, :len(tab)] = tab
            q_lens.append(n)
            new_tok += r.tokens[r.done:r.done + n]
            new_pos += list(range(r.done, r.done + n))
        k_new, v_new = kv_rows(new_tok, new_pos, hkv, d)
        seq_lens = np.asarray([r.done + n for r, n in batch], np.int32)
        live = {r.rid: (bm.block_table(r.rid), r.tokens[:r.done]) for r in reqs.values()}
        for (r, n), L in zip(batch, seq_lens):
            live[r.rid] = (bm.block_table(r.rid), r.tokens[:int(L)])
        yield Step(step, np.asarray([c[0] for c in cows], np.int32), np.asarray([c[1] for c in cows], np.int32),
                   bt, seq_lens, np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32), k_new, v_new, live,
                   [r.rid for r, _ in batch])
        # chunks complete; a request whose tokens are all in the pool emits the next one
        for r, n in batch:
            r.done += n
            if r.done == len(r.tokens):
                if r.gen_left == 0:
                    bm.free(r.rid)
                    del reqs[r.rid]
                    events["finished"] += 1
                    continue
                r.tokens.append(int(rng.integers(1, 30000)))
                r.gen_left -= 1
            bm.cache_full_blocks(r.rid, np.asarray(r.tokens[:r.done], np.int32))
        if not reqs:
            return


def gather(pool_bits: np.ndarray, table, n: int) -> np.ndarray:
    """The first n token rows [n, hkv, d] of a request, read through its block table."""
    if n == 0:
        return pool_bits[:0, :, 0, :]
    rows = [pool_bits[table[p // BLOCK], :, p % BLOCK, :] for p in range(n)]
    return np.stack(rows)
