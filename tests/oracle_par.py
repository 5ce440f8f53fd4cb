"""Independent oracle recurrences run in parallel worker processes.

The workers are spawned (never forked), so none inherits the CUDA context of
a test process that has already used the GPU; they import only numpy and the
oracle."""
import multiprocessing as mp
import os

from oracle import gdn_oracle as O


def _recurrent(args):
    return O.gdn_recurrent(*args)


def recurrent_many(tasks, procs=None):
    """[(S0, q, k, v, g, beta), ...] -> [(S_T, o), ...] in order."""
    procs = procs or min(16, os.cpu_count() or 1, len(tasks))
    if procs <= 1:
        return [_recurrent(t) for t in tasks]
    with mp.get_context("spawn").Pool(procs) as pool:
        return pool.map(_recurrent, tasks, chunksize=1)
