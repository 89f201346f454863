"""Times the fp64 oracle on the host's cores, for the benchmark's CPU baseline.

TEST INFRASTRUCTURE ONLY: the CPU-baseline leg of ``bench.py`` is the one user. It
runs the oracle functions of ``oracle/attention.py`` unchanged, over independent
units of work ((sequence, KV head) for decode, (batch, head) for prefill, a request for
the shared-prefix decode), either in
this process (one core) or spread over worker processes started with ``spawn``, each
with one BLAS thread. The inputs are placed once in shared memory, so the workers
read them without a copy. Nothing here changes what the oracle computes or how.
"""
from __future__ import annotations

import multiprocessing as mp
import time
from multiprocessing import shared_memory

import numpy as np

from . import attention as _att

_W = {}  # worker state: name -> array view on shared memory


def _share(arrays):
    """Copies each array into a new shared-memory block; returns (blocks, specs)."""
    blocks, specs = [], {}
    for name, a in arrays.items():
        a = np.ascontiguousarray(a)
        shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
        np.ndarray(a.shape, a.dtype, buffer=shm.buf)[...] = a
        blocks.append(shm)
        specs[name] = (shm.name, a.shape, a.dtype.str)
    return blocks, specs


def _attach(specs, extra):
    _W.clear()
    _W["_shm"] = []
    for name, (shm_name, shape, dt) in specs.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _W["_shm"].append(shm)
        _W[name] = np.ndarray(shape, np.dtype(dt), buffer=shm.buf)
    _W.update(extra)


def _decode_units(units):
    q, kp, vp, bt, lens = _W["q"], _W["k_pages"], _W["v_pages"], _W["block_table"], _W["kv_lens"]
    G = q.shape[1] // kp.shape[1]
    for b, g in units:
        rows = [(b, h) for h in range(g * G, (g + 1) * G)]
        _att.decode_paged(q[b:b + 1], kp, vp, bt[b:b + 1], lens[b:b + 1], _W["scale"],
                          rows=[(0, h) for _, h in rows])
    return len(units)


def _prefill_units(units):
    q, k, v = _W["q"], _W["k"], _W["v"]
    G = q.shape[2] // k.shape[2]
    for b, h in units:
        _att.prefill_causal(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h // G:h // G + 1],
                            v[b:b + 1, :, h // G:h // G + 1], _W["scale"])
    return len(units)


def _cascade_units(units):
    q, kp, vp = _W["q"], _W["k_pages"], _W["v_pages"]
    for r in units:
        _att.cascade_decode(q[r:r + 1], kp, vp, _W["prefix_table"], _W["prefix_len"],
                            _W["suffix_table"][r:r + 1], _W["suffix_lens"][r:r + 1], _W["scale"])
    return len(units)


def _balanced(units, weights, n):
    """Splits the units into n lists of about equal total weight (largest first, greedy)."""
    order = sorted(range(len(units)), key=lambda i: -weights[i])
    bins, load = [[] for _ in range(n)], [0.0] * n
    for i in order:
        j = min(range(n), key=lambda x: load[x])
        bins[j].append(units[i])
        load[j] += weights[i]
    return [b for b in bins if b]


class _Runner:
    """Runs a unit function over a fixed list of units, in-process or in a spawn pool."""

    def __init__(self, fn, arrays, extra, units, weights, workers):
        self.fn, self.units, self.workers = fn, units, workers
        self.pool, self.blocks = None, []
        if workers <= 1:
            _attach({}, extra)
            _W.update(arrays)
            self.chunks = [units]
        else:
            self.blocks, specs = _share(arrays)
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(workers, initializer=_attach, initargs=(specs, extra))
            # a few chunks per worker, balanced by weight
            self.chunks = _balanced(units, weights, 4 * workers)

    def one_pass(self):
        if self.pool is None:
            return self.fn(self.chunks[0])
        return sum(self.pool.map(self.fn, self.chunks, chunksize=1))

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
        for shm in self.blocks:
            shm.close()
            shm.unlink()
        _W.clear()


def time_passes(runner, budget_s, min_passes=1):
    """Whole passes until ``budget_s`` has elapsed (at least ``min_passes``); (passes, seconds)."""
    runner.one_pass()  # warm-up: worker start-up and first touches are not timed
    passes, t0 = 0, time.perf_counter()
    while True:
        runner.one_pass()
        passes += 1
        el = time.perf_counter() - t0
        if passes >= min_passes and el >= budget_s:
            return passes, el


def decode_runner(q, k_pages, v_pages, block_table, kv_lens, scale, workers):
    """The paged-decode oracle over every (sequence, KV head) unit of the batch."""
    B = q.shape[0]
    Hkv = k_pages.shape[1]
    units = [(b, g) for b in range(B) for g in range(Hkv)]
    weights = [float(kv_lens[b]) for b, _ in units]
    arrays = dict(q=np.asarray(q, np.float64), k_pages=np.asarray(k_pages, np.float32),
                  v_pages=np.asarray(v_pages, np.float32), block_table=np.asarray(block_table, np.int32),
                  kv_lens=np.asarray(kv_lens, np.int32))
    return _Runner(_decode_units, arrays, {"scale": float(scale)}, units, weights, workers)


def prefill_runner(q, k, v, scale, workers):
    """The causal-prefill oracle over every (batch, query head) unit."""
    B, _, Hq, _ = q.shape
    units = [(b, h) for b in range(B) for h in range(Hq)]
    arrays = dict(q=np.asarray(q, np.float32), k=np.asarray(k, np.float32), v=np.asarray(v, np.float32))
    return _Runner(_prefill_units, arrays, {"scale": float(scale)}, units, [1.0] * len(units), workers)


def cascade_runner(q, k_pages, v_pages, prefix_table, prefix_len, suffix_table, suffix_lens, scale,
                   workers):
    """The shared-prefix decode oracle over every request (each call attends the prefix and
    the request's suffix for all of its heads)."""
    R = q.shape[0]
    units = list(range(R))
    weights = [float(prefix_len + suffix_lens[r]) for r in units]
    arrays = dict(q=np.asarray(q, np.float64), k_pages=np.asarray(k_pages, np.float32),
                  v_pages=np.asarray(v_pages, np.float32), prefix_table=np.asarray(prefix_table, np.int32),
                  suffix_table=np.asarray(suffix_table, np.int32), suffix_lens=np.asarray(suffix_lens, np.int32))
    return _Runner(_cascade_units, arrays, {"scale": float(scale), "prefix_len": int(prefix_len)}, units,
                   weights, workers)
