"""The oracle's paged decode spread over the host cores -- BASELINE INFRASTRUCTURE ONLY.

Used by bench.py's CPU-baseline leg to time the oracle (oracle/kvc_oracle.py,
unchanged) on all host cores: one process per core, started with "spawn" (a
process forked after CUDA is initialised can hang), each evaluating whole
sequences.  The inputs -- each sequence's cache blocks, as raw 16-bit patterns,
and its query row -- are written once to a scratch directory and memory-mapped
by the workers, so nothing large passes through the process pipes.  Nothing
here computes attention: the workers call kvc_oracle.paged_decode.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile
import time

import numpy as np

_STATE = {}


def _to_f64(bits16: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (bits16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits16.view(np.float16).astype(np.float64)


def _init(folder: str, dtype: str):
    _STATE["k"] = np.load(os.path.join(folder, "k.npy"), mmap_mode="r")
    _STATE["v"] = np.load(os.path.join(folder, "v.npy"), mmap_mode="r")
    _STATE["q"] = np.load(os.path.join(folder, "q.npy"), mmap_mode="r")
    _STATE["meta"] = np.load(os.path.join(folder, "meta.npy"))
    _STATE["dtype"] = dtype


def _decode(task):
    from oracle import kvc_oracle as O
    b, scale = task
    start, nblk, L = (int(x) for x in _STATE["meta"][b])
    dt = _STATE["dtype"]
    k = _to_f64(np.asarray(_STATE["k"][start:start + nblk]), dt)
    v = _to_f64(np.asarray(_STATE["v"][start:start + nblk]), dt)
    q = _to_f64(np.asarray(_STATE["q"][b:b + 1]), dt)
    O.paged_decode(q, k, v, np.arange(nblk)[None], [L], scale)
    return b


class OraclePool:
    """A pool of `workers` spawned processes holding one decode workload.

    k_blocks / v_blocks: per sequence, its blocks in logical order as 16-bit
    patterns [nblk, block_size, Hkv, D] (int16); q: [B, Hq, D] int16.
    """

    def __init__(self, k_blocks, v_blocks, q_bits, lens, dtype: str, workers: int):
        self.folder = tempfile.mkdtemp(prefix="kvc_oracle_pool_")
        starts, at = [], 0
        for kb in k_blocks:
            starts.append(at)
            at += kb.shape[0]
        np.save(os.path.join(self.folder, "k.npy"), np.concatenate(k_blocks))
        np.save(os.path.join(self.folder, "v.npy"), np.concatenate(v_blocks))
        np.save(os.path.join(self.folder, "q.npy"), np.ascontiguousarray(q_bits))
        meta = np.array([[s, kb.shape[0], L] for s, kb, L in zip(starts, k_blocks, lens)],
                        dtype=np.int64)
        np.save(os.path.join(self.folder, "meta.npy"), meta)
        self.n = len(lens)
        self.workers = workers
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(workers, initializer=_init, initargs=(self.folder, dtype))

    def run(self, order, scale: float) -> float:
        """Evaluate the sequences `order` (indices, repeats allowed); wall seconds."""
        t0 = time.perf_counter()
        list(self.pool.imap_unordered(_decode, [(int(b), scale) for b in order], chunksize=1))
        return time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.folder, ignore_errors=True)
