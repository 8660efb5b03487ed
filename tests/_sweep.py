"""Every fp32 bit pattern through a GPU quantiser, checked against the oracle.

The 2^32 patterns go in 256 chunks of 2^24 (chunk t holds the patterns whose
top byte is t), each with the format's largest finite value and zero padding
appended (so that a chunk whose values stay within range is quantised with
qscale == 1 and tests the cast alone, and so that the row length is a
multiple of four: the 16-byte path every aligned tensor takes).  The oracle's
side of each chunk runs in worker processes started with `spawn` (never
forked from a process that holds a CUDA context), the GPU side in the test's
own process; the two meet chunk by chunk.
"""

import multiprocessing as mp
import os

import numpy as np

FMAX = {"e4m3": 448.0, "e5m2": 57344.0}


def chunk_input(fmt, top):
    lo = np.uint64(top) << np.uint64(24)
    bits = (np.arange(1 << 24, dtype=np.uint64) + lo).astype(np.uint32)
    tail = np.array([FMAX[fmt], 0.0, 0.0, 0.0], np.float32)
    return np.concatenate([bits.view(np.float32), tail])[None, :]


def _oracle_chunk(task):
    import oracle
    fmt, top = task
    q, amax, scale = oracle.quantize_pertensor(chunk_input(fmt, top), fmt=fmt)
    return top, q, np.float32(amax).tobytes(), np.float32(scale).tobytes()


def sweep_all(fmt, gpu_quantize):
    """gpu_quantize(x) -> (codes, amax, scale) for a [1][n] fp32 array."""
    workers = max(1, min(8, (os.cpu_count() or 2) - 1))
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        tasks = [(fmt, t) for t in range(256)]
        for top, rq, ramax, rscale in pool.imap(_oracle_chunk, tasks):
            x = chunk_input(fmt, top)
            q, amax, scale = gpu_quantize(x)
            assert np.float32(amax).tobytes() == ramax, "amax, chunk %#x" % top
            assert np.float32(scale).tobytes() == rscale, "scale, chunk %#x" % top
            diff = np.flatnonzero(q.reshape(-1) != rq.reshape(-1))
            assert diff.size == 0, (
                "%s: chunk %#x: codes differ at %d places, first: got %#x want %#x (x=%r)"
                % (fmt, top, diff.size, q.reshape(-1)[diff[0]], rq.reshape(-1)[diff[0]],
                   x.reshape(-1)[diff[0]]))
