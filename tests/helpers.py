"""Shared helpers for the parity tests: run one step on the GPU through the C ABI,
run the same step through the oracle, and compare.

A step is: slot mapping of the new tokens, scatter of their K/V into the pool,
then attention over the mixed batch.  The oracle gets the same seeded inputs
(the pool as drawn, before the GPU writes into it) and performs its own slot
mapping and scatter; nothing it reads comes from the CUDA path.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle

# tolerances: bf16 inputs, fp32 accumulation vs fp64 -> max-abs 2e-2, mean-abs 2e-3;
# fp32 inputs -> max-abs 1e-4
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-4, 1e-4)}


def bits(x: torch.Tensor) -> np.ndarray:
    """CPU copy as the oracle reads it: fp32 array or bf16 bit patterns (int16)."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().copy()
    return x.numpy().copy()


def to_gpu_meta(w, bt=None):
    dev = torch.device("cuda")
    return dict(
        block_tables=torch.from_numpy(np.ascontiguousarray(w.block_tables if bt is None else bt)).to(dev),
        seq_lens=torch.from_numpy(w.seq_lens).to(dev),
        query_start_loc=torch.from_numpy(w.query_start_loc).to(dev),
    )


def gpu_step(pkv, w, t: dict, bt=None, cow: bool = False):
    """Run copy (optional) + slot mapping + write + attention on the GPU; tensors in
    ``t`` must already be on the GPU (the caches are modified in place)."""
    m = to_gpu_meta(w, bt)
    if cow:
        pkv.pkv_copy_blocks(torch.from_numpy(w.cow_src).cuda(), torch.from_numpy(w.cow_dst).cuda(),
                            t["k_cache"], t["v_cache"])
    slots = pkv.pkv_slot_mapping(m["block_tables"], m["seq_lens"], m["query_start_loc"], w.num_tokens)
    pkv.pkv_write(t["k_new"], t["v_new"], slots, t["k_cache"], t["v_cache"])
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"],
                              m["query_start_loc"], w.scale, max(1, w.max_query_len), max(1, w.max_seq_len))
    st = pkv.pkv_get_last_error()
    return out, slots, st


def oracle_step(w, t_cpu: dict, bt=None, rows=None, cow: bool = False):
    """The same step by the oracle, from host copies of the drawn inputs."""
    kc, vc = bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"])
    table = w.block_tables if bt is None else bt
    if cow:
        oracle.copy_blocks(w.cow_src, w.cow_dst, kc, vc)
    slots = oracle.slot_mapping(table, w.seq_lens, w.query_start_loc)
    oracle.write(bits(t_cpu["k_new"]), bits(t_cpu["v_new"]), slots, kc, vc)
    out = oracle.attention(bits(t_cpu["q"]), kc, vc, table, w.seq_lens, w.query_start_loc, w.scale, rows=rows)
    return out, slots, kc, vc


def compare(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    max_tol, mean_tol = TOL[dtype]

    def where():
        rows = err.reshape(err.shape[0], -1).max(axis=1) if err.ndim > 1 else err
        bad = np.nonzero(rows > max_tol)[0]
        heads = sorted(set(np.nonzero(err[bad].max(axis=-1) > max_tol)[1].tolist())) if err.ndim == 3 and len(bad) else []
        return f" ({len(bad)} rows over tolerance, first {bad[:12].tolist()}, heads {heads[:16]})"

    assert np.isfinite(g).all(), f"{what}: non-finite output" + where()
    assert err.max() <= max_tol, f"{what}: max-abs {err.max():.3e} > {max_tol}" + where()
    assert err.mean() <= mean_tol, f"{what}: mean-abs {err.mean():.3e} > {mean_tol}"
    return float(err.max()), float(err.mean())


def sub_batch(w, t_gpu, seq_ids):
    """Requests ``seq_ids`` of a large batch, with only their blocks, copied to the host
    before the GPU step writes into the pool (block ids renumbered: the oracle's
    result does not depend on physical ids)."""
    seq_ids = np.asarray(seq_ids)
    bt = w.block_tables[seq_ids]
    used = np.unique(bt[bt >= 0])
    remap = np.full(w.num_blocks, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    qsl = w.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seq_ids]).astype(np.int64)
    q_lens = np.array([qsl[i + 1] - qsl[i] for i in seq_ids], np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    ridx = torch.from_numpy(rows).cuda()
    t_sub = {"k_cache": t_gpu["k_cache"].index_select(0, idx).cpu(),
             "v_cache": t_gpu["v_cache"].index_select(0, idx).cpu(),
             "q": t_gpu["q"].index_select(0, ridx).cpu(),
             "k_new": t_gpu["k_new"].index_select(0, ridx).cpu(),
             "v_new": t_gpu["v_new"].index_select(0, ridx).cpu()}
    w2 = dataclasses.replace(w, num_blocks=len(used), seq_lens=w.seq_lens[seq_ids].copy(),
                             query_start_loc=np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                             block_tables=bt2)
    return w2, t_sub, rows


def host_requests(w, pool_k, pool_v, t_gpu, seq_ids):
    """Requests ``seq_ids`` of a batch as a self-contained host batch for the oracle.

    Only the blocks those requests reference (their tables, and the sources of their
    copy-on-write pairs) are copied from ``pool_k``/``pool_v`` -- device pools as
    they were before the GPU step -- and renumbered 0..n-1; the oracle's result does
    not depend on physical ids.  Returns (workload, host tensors, the requests' query
    rows in the full batch, the original ids of the copied blocks)."""
    seq_ids = np.asarray(seq_ids, np.int64)
    bt = w.block_tables[seq_ids]
    ids = [bt[bt >= 0]]
    cow = w.cow_src is not None
    if cow:
        ids += [w.cow_src[seq_ids], w.cow_dst[seq_ids]]
    used = np.unique(np.concatenate(ids)).astype(np.int64)
    remap = np.full(w.num_blocks, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    qsl = w.query_start_loc
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seq_ids]).astype(np.int64)
    q_lens = (qsl[seq_ids + 1] - qsl[seq_ids]).astype(np.int32)
    idx = torch.from_numpy(used).to(pool_k.device)
    ridx = torch.from_numpy(rows).to(pool_k.device)
    t_sub = {"k_cache": pool_k.index_select(0, idx).cpu(),
             "v_cache": pool_v.index_select(0, idx).cpu(),
             "q": t_gpu["q"].index_select(0, ridx).cpu(),
             "k_new": t_gpu["k_new"].index_select(0, ridx).cpu(),
             "v_new": t_gpu["v_new"].index_select(0, ridx).cpu()}
    extra = {}
    if cow:
        extra = dict(cow_src=remap[w.cow_src[seq_ids]].astype(np.int32),
                     cow_dst=remap[w.cow_dst[seq_ids]].astype(np.int32))
    w2 = dataclasses.replace(w, num_blocks=len(used), seq_lens=w.seq_lens[seq_ids].copy(),
                             query_start_loc=np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                             block_tables=bt2, block_tables_before_cow=None, **extra)
    return w2, t_sub, rows, used
