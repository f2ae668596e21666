"""Oracle outputs of full-size MoE tokens in worker processes.

The oracle is single-threaded plain C; checking dozens of tokens of the
full-size prefill layer (each token runs six experts of 25M weights in
double precision, and each expert must first be regenerated and quantised)
takes minutes in one process.  The tokens are split over a pool of processes
started with the `spawn` method (never forked from a process that has
initialised CUDA); each worker quantises the experts its tokens need.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _moe_tokens_worker(task):
    name, toks, x, idx, w, dw = task
    import oracle
    from synth import recipes
    r = recipes.MOES[name]
    og, ou, od = [None] * r.E, [None] * r.E, [None] * r.E
    for e in sorted(set(int(v) for v in idx.reshape(-1))):
        og[e] = oracle.quantize(recipes.moe_expert_rows(r, "gate", e), r.bits, r.group)
        ou[e] = oracle.quantize(recipes.moe_expert_rows(r, "up", e), r.bits, r.group)
        od[e] = oracle.quantize(recipes.moe_expert_rows(r, "down", e), r.bits, r.group)
    y, b = oracle.moe_ffn(x, idx, w, og, ou, od, dw=dw)
    return toks, y, b


def moe_tokens(recipe_name: str, toks, x, idx, w, dw: float = 0.0, workers: int | None = None):
    """Oracle outputs (y, bound) of the given tokens (rows of x / idx / w) of
    a full-size MoE recipe, in the order of `toks`."""
    toks = np.asarray(toks)
    workers = workers or max(1, min(len(toks), (os.cpu_count() or 2) - 1, 16))
    chunks = [c for c in np.array_split(np.arange(len(toks)), workers) if len(c)]
    tasks = [(recipe_name, toks[c], np.ascontiguousarray(x[c]), np.ascontiguousarray(idx[c]),
              np.ascontiguousarray(w[c]), dw) for c in chunks]
    with mp.get_context("spawn").Pool(len(tasks)) as pool:
        res = pool.map(_moe_tokens_worker, tasks, chunksize=1)
    H = x.shape[1]
    y = np.empty((len(toks), H))
    b = np.empty((len(toks), H))
    pos = {int(t): i for i, t in enumerate(toks)}
    for tt, yy, bb in res:
        for j, t in enumerate(tt):
            y[pos[int(t)]] = yy[j]
            b[pos[int(t)]] = bb[j]
    return y, b
