"""The fp64 oracle over many sequences at once, for the parity tests at the
workloads' stated round counts.

A pool of spawned worker processes (one per host core) attaches shared-memory
arrays that hold a batch of sequences' target and draft rows; the test copies
each batch straight from the GPU into them and maps sequence indices over the
pool.  Workers run ``oracle.verify_sample_seq`` unchanged.  The pool is
started with ``spawn`` so that no process holding a CUDA context is forked.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_W = None


def _init(names, shapes, dtypes):
    global _W
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    shms = [shared_memory.SharedMemory(name=n) for n in names]
    arrs = [np.ndarray(s, dtype=np.dtype(d), buffer=m.buf) for m, s, d in zip(shms, shapes, dtypes)]
    _W = (shms, arrs)


def _rows(a):
    """Logit rows as float64 (uint16 arrays hold bf16 bit patterns)."""
    import oracle
    return oracle.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _verify(task):
    import oracle
    b, toks, T, ua, ur = task
    tgt, dft = _W[1]
    return oracle.verify_sample_seq(tgt[b], dft[b], toks, T, ua, ur)


def _greedy(task):
    import oracle
    b, toks = task
    return oracle.verify_greedy_seq(_W[1][0][b], toks)


def _alpha(task):
    """alpha_j = sum_x min(p_j(x), q_j(x)) for the draft positions of sequence
    b (empty for a greedy sequence)."""
    import oracle
    b, T = task
    if not T > 0:
        return []
    tgt, dft = _W[1]
    return [float(np.minimum(oracle.row_probs(_rows(tgt[b, j]), T), oracle.row_probs(_rows(dft[b, j]), T)).sum())
            for j in range(dft.shape[1])]


class OraclePool:
    """Workers plus shared arrays target [n, gamma+1, V] and draft [n, gamma, V]
    of numpy dtype ``tdtype`` / ``ddtype`` (uint16 = bf16 bits)."""

    def __init__(self, n, gamma, V, tdtype, ddtype=None, cores=None):
        ddtype = tdtype if ddtype is None else ddtype
        self.cores = cores or os.cpu_count() or 1
        self.shms, shapes, dtypes, self.arrs = [], [], [], []
        for shape, dt in (((n, gamma + 1, V), np.dtype(tdtype)), ((n, gamma, V), np.dtype(ddtype))):
            m = shared_memory.SharedMemory(create=True, size=int(np.prod(shape)) * dt.itemsize)
            self.shms.append(m)
            shapes.append(shape)
            dtypes.append(dt.str)
            self.arrs.append(np.ndarray(shape, dtype=dt, buffer=m.buf))
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_init,
                                                 initargs=([m.name for m in self.shms], shapes, dtypes))

    @property
    def target(self):
        return self.arrs[0]

    @property
    def draft(self):
        return self.arrs[1]

    def fill(self, target, draft=None):
        """Copy a batch of torch tensors (on any device) into the shared arrays."""
        import torch
        for dst, src in ((self.arrs[0], target), (self.arrs[1], draft)):
            if src is None:
                continue
            t = torch.from_numpy(dst[:src.shape[0]].view(np.int16) if dst.dtype == np.uint16 else dst[:src.shape[0]])
            if src.dtype == torch.bfloat16:
                t = t.view(torch.bfloat16)
            t.copy_(src)

    def _chunk(self, n):
        return max(1, n // (4 * self.cores))

    def verify(self, draft_tokens, temperature, u_accept, u_resample):
        n = len(draft_tokens)
        tasks = [(b, draft_tokens[b], float(temperature[b]), u_accept[b], float(u_resample[b])) for b in range(n)]
        return self.pool.map(_verify, tasks, chunksize=self._chunk(n))

    def greedy(self, draft_tokens):
        n = len(draft_tokens)
        return self.pool.map(_greedy, [(b, draft_tokens[b]) for b in range(n)], chunksize=self._chunk(n))

    def alphas(self, temperature):
        n = len(temperature)
        out = self.pool.map(_alpha, [(b, float(temperature[b])) for b in range(n)], chunksize=self._chunk(n))
        return [a for seq in out for a in seq]

    def close(self):
        self.pool.close()
        self.pool.join()
        for m in self.shms:
            m.close()
            m.unlink()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
