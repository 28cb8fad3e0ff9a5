"""The oracle's row-independent steps at full batch size, spread over a pool of spawned processes
(spawned, not forked: the parent holds a CUDA context). Every function here only calls oracle/
on slices of its inputs; the results are the oracle's own, concatenated in row order.

  route_all   routing of every row (logits, sigmoid, top-k, weights per row chunk), then the
              oracle's plan over the whole batch
  quant_all   MXFP8 codes and scales of every row
  weights     MXFP4 codes and scales of the experts asked for (the rest stay zero)
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import moe as M


def _route_chunk(args):
    x, wr, bias, k = args
    r = M.route(x, wr, bias, k)
    return r.topk_idx, r.topk_w


def _quant_chunk(x):
    return M.quant_mxfp8(x)


def _quant_expert(args):
    e, w = args
    q, s = M.quant_mxfp4(w)
    return e, q, s


def _workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


class Pool:
    def __init__(self):
        self.n = _workers()
        self.pool = mp.get_context("spawn").Pool(self.n)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.pool.close()
        self.pool.join()

    def _chunks(self, T):
        return [c for c in np.array_split(np.arange(T), 4 * self.n) if len(c)]

    def route_all(self, x: np.ndarray, wr: np.ndarray, bias: np.ndarray, k: int, dead=None) -> M.Routing:
        parts = self.pool.map(_route_chunk, [(x[c], wr, bias, k) for c in self._chunks(x.shape[0])])
        idx = np.concatenate([p[0] for p in parts])
        w = np.concatenate([p[1] for p in parts])
        return M.plan(None, None, None, idx, w, wr.shape[0], dead)

    def quant_all(self, x: np.ndarray):
        parts = self.pool.map(_quant_chunk, [x[c] for c in self._chunks(x.shape[0])])
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])

    def weights(self, w_of_expert, E: int, R: int, K: int, experts) -> M.ExpertWeights:
        """w_of_expert(e) -> fp32 [R, K] numpy array; only `experts` are quantised."""
        codes = np.zeros((E, R, K // 2), dtype=np.uint8)
        scales = np.zeros((E, R, K // 32), dtype=np.uint8)
        jobs = ((int(e), w_of_expert(int(e))) for e in experts)
        for e, q, s in self.pool.imap_unordered(_quant_expert, jobs):
            codes[e], scales[e] = q, s
        return M.ExpertWeights(codes, scales, cache=16)
