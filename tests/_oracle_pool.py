"""Runs the float64 oracle on all host cores for the full-size parity tests.

The oracle is single-threaded outside its BLAS calls. Its row blocks are independent
(each is the same whole-row computation the oracle does, and the gradient terms of
disjoint query-row blocks add up to the whole: pinned in tests/test_oracle_pins.py),
so the tests run them in a pool of worker processes. The pool is started with
"spawn": the parent holds a CUDA context, and a child forked from such a process
must not touch it. Inputs reach the workers as .npy files that they map read-only;
each worker runs single-threaded BLAS. The number of workers is bounded by the host's
cores and by its available memory (each worker's row chunks hold at most 2^24 score
entries, about 1 GB of temporaries).
"""

from __future__ import annotations

import math
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

WORKER_BYTES = 2 << 30   # memory budget per worker


def _mem_available():
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            v = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            cur = int(f.read().strip())
        if v != "max":
            lim = int(v) - cur
            avail = lim if avail is None else min(avail, lim)
    except (OSError, ValueError):
        pass
    return avail if avail is not None else 8 << 30


def _scratch_dir():
    """Where the workers' input files go: LWM_ORACLE_TMP, else /dev/shm (memory-backed)
    when it has room, else the default temporary directory."""
    d = os.environ.get("LWM_ORACLE_TMP")
    if d:
        return d
    try:
        st = os.statvfs("/dev/shm")
        if st.f_bavail * st.f_frsize > (8 << 30):
            return "/dev/shm"
    except OSError:
        pass
    return None


def default_workers():
    cpus = len(os.sched_getaffinity(0))
    by_mem = int(0.6 * _mem_available()) // WORKER_BYTES
    return max(1, min(cpus, by_mem))


# ----------------------------------------------------------------------------- worker side
_ARRAYS = {}


def _load(d):
    if d not in _ARRAYS:
        _ARRAYS.clear()
        _ARRAYS[d] = {n[:-4]: np.load(os.path.join(d, n), mmap_mode="r") for n in os.listdir(d) if n.endswith(".npy")}
    return _ARRAYS[d]


def _fwd_task(args):
    import oracle
    d, b, h, r0, r1 = args
    A = _load(d)
    out, lse = oracle.forward_row_block(A["q"], A["k"], A["v"], A["seg"], b, h, np.arange(r0, r1))
    return b, h, r0, r1, out, lse


def _bwd_task(args):
    import oracle
    from oracle import attention as OA
    d, b, h, r0, r1 = args
    A = _load(d)
    S = A["q"].shape[1]
    dq = np.zeros((r1 - r0, A["q"].shape[3]))
    lo, hi, dk, dv = S, 0, None, None
    parts = []
    for rows in OA._chunks(np.arange(r0, r1), OA._chunk_rows(r1)):
        g, j0, gk, gv = oracle.backward_row_block(A["q"], A["k"], A["v"], A["dout"], A["seg"], b, h, rows)
        dq[rows - r0] = g
        parts.append((j0, gk, gv))
        lo, hi = min(lo, j0), max(hi, j0 + gk.shape[0])
    dk = np.zeros((max(hi - lo, 0), dq.shape[1]))
    dv = np.zeros_like(dk)
    for j0, gk, gv in parts:
        dk[j0 - lo:j0 - lo + gk.shape[0]] += gk
        dv[j0 - lo:j0 - lo + gv.shape[0]] += gv
    return b, h, r0, r1, dq, lo, dk, dv


def _keys_task(args):
    import oracle
    d, b, h, keys, r0, r1 = args
    A = _load(d)
    dk, dv = oracle.attention_key_grads(A["q"], A["k"], A["v"], A["dout"], A["seg"], b, h, keys, row_range=(r0, r1))
    return h, dk, dv


# ----------------------------------------------------------------------------- parent side
def _row_groups(seg_row, n_groups):
    """Contiguous row ranges of about equal oracle cost (cost of row i ~ the window of
    keys it needs: i - start of its document + 1)."""
    S = len(seg_row)
    start = np.zeros(S, np.int64)
    change = np.flatnonzero(np.diff(seg_row)) + 1
    start[change] = change
    start = np.maximum.accumulate(start)
    cost = np.cumsum(np.arange(S) - start + 1, dtype=np.float64)
    cuts = [0]
    for g in range(1, n_groups):
        cuts.append(int(np.searchsorted(cost, cost[-1] * g / n_groups)))
    cuts.append(S)
    cuts = sorted(set(cuts))
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


class OraclePool:
    """Oracle legs over selected heads of one workload, in spawned worker processes.

    ``tensors``: name -> float32 array [B, S, Hs, D] (the bf16 values), for names among
    q, k, v, dout; ``seg``: int [B, S]. Head index h below is an index into Hs.
    """

    def __init__(self, tensors, seg, workers=None):
        self.dir = tempfile.mkdtemp(prefix="lwm_oracle_", dir=_scratch_dir())
        for n, a in tensors.items():
            np.save(os.path.join(self.dir, n + ".npy"), np.ascontiguousarray(a, dtype=np.float32))
        np.save(os.path.join(self.dir, "seg.npy"), np.ascontiguousarray(seg, dtype=np.int64))
        self.B, self.S, self.Hs, self.D = next(iter(tensors.values())).shape
        self.seg = np.asarray(seg)
        self.workers = workers or default_workers()
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _groups(self, b, per_head):
        return _row_groups(self.seg[b], per_head)

    def forward(self):
        """(out [B, S, Hs, D], lse [B, Hs, S]) over every row of every selected head."""
        from oracle import attention as OA
        step = OA._chunk_rows(self.S)
        tasks = [(self.dir, b, h, r0, min(r0 + step, self.S))
                 for b in range(self.B) for h in range(self.Hs) for r0 in range(0, self.S, step)]
        out = np.zeros((self.B, self.S, self.Hs, self.D))
        lse = np.zeros((self.B, self.Hs, self.S))
        for b, h, r0, r1, o, l in self.pool.imap_unordered(_fwd_task, tasks):
            out[b, r0:r1, h] = o
            lse[b, h, r0:r1] = l
        return out, lse

    def backward(self):
        """(dq, dk, dv), each [B, S, Hs, D], over every row of every selected head."""
        per_head = max(1, math.ceil(2 * self.workers / (self.B * self.Hs)))
        tasks = [(self.dir, b, h, r0, r1) for b in range(self.B) for h in range(self.Hs)
                 for r0, r1 in self._groups(b, per_head)]
        dq, dk, dv = (np.zeros((self.B, self.S, self.Hs, self.D)) for _ in range(3))
        for b, h, r0, r1, g, lo, gk, gv in self.pool.imap_unordered(_bwd_task, tasks):
            dq[b, r0:r1, h] = g
            dk[b, lo:lo + len(gk), h] += gk
            dv[b, lo:lo + len(gv), h] += gv
        return dq, dk, dv

    def key_grads(self, b, heads, keys, per_head=None):
        """{h: (dk [K, D], dv [K, D])} for the selected keys of batch row b."""
        keys = np.asarray(keys, dtype=np.int64)
        per_head = per_head or max(1, math.ceil(2 * self.workers / len(heads)))
        seg_row = self.seg[b].copy()
        seg_row[: int(keys.min())] = -2   # rows before the first key contribute nothing
        groups = [(r0, r1) for r0, r1 in _row_groups(seg_row, per_head) if r1 > int(keys.min())]
        tasks = [(self.dir, b, h, keys, r0, r1) for h in heads for r0, r1 in groups]
        res = {h: (np.zeros((len(keys), self.D)), np.zeros((len(keys), self.D))) for h in heads}
        for h, gk, gv in self.pool.imap_unordered(_keys_task, tasks):
            res[h][0][:] += gk
            res[h][1][:] += gv
        return res
