"""Writes tests/golden/tiny_decode.npz from the oracle alone.

Run from the repository root: ``python tests/golden/make_golden.py``.  The
inputs are the seeded tiny fp32 decode workload (4 requests, seq_lens
{5, 16, 17, 40}, 2 query heads over 1 KV head, head_dim 64), drawn on the host;
the stored output is the fp64 oracle's.  The fixture guards the oracle and the
input generator against silent drift.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as wl  # noqa: E402


def compute():
    w = wl.make("tiny")
    t = w.make_tensors("cpu")
    kc, vc = t["k_cache"].numpy().copy(), t["v_cache"].numpy().copy()
    slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc)
    oracle.write(t["k_new"].numpy(), t["v_new"].numpy(), slots, kc, vc)
    out = oracle.attention(t["q"].numpy(), kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.scale)
    return dict(out=out, slots=slots, block_tables=w.block_tables, seq_lens=w.seq_lens,
                q_first=t["q"].numpy()[:, :, :4].copy())


if __name__ == "__main__":
    np.savez(os.path.join(HERE, "tiny_decode.npz"), **compute())
