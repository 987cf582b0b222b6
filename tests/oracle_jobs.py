"""Oracle work for the full-size GPU tests, run in worker processes started with `spawn` (no CUDA
in them).  Each worker runs single-threaded numpy; the pool spreads rows, weight blocks and experts
over the host's cores.  numpy is imported after the thread limits are set."""

import os

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def init_worker():
    for v in _THREAD_VARS:
        os.environ[v] = "1"


def quantize_rows(x):
    from oracle import quantize_1x128

    return quantize_1x128(x)


def quantize_weights(w):
    from oracle import quantize_128x128

    return quantize_128x128(w)


def gemm(qa, sa, qb, sb):
    from oracle import gemm_nt

    return gemm_nt(qa, sa, qb, sb)


def pool():
    """A process pool of spawned workers (safe after CUDA has been initialised in this process)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    n = max(1, min(16, os.cpu_count() or 1))
    return ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"), initializer=init_worker)
