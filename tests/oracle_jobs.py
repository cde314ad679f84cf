"""Background runs of the CPU oracle for the full-size parity tests.

A full-size oracle decode takes minutes of host time (the 720p clip's first
two latent frames are five 704x1280 frames at about 16.6 TFLOP each), so the
GPU session starts these runs in a pool of spawned worker processes as soon
as it has collected a full-size parity test, and the tests collect the
results when they need them; meanwhile the other GPU tests run.  Workers are
spawned, never forked, and import NumPy only after their BLAS thread count is
set, so each one uses its share of the host cores.

Each job draws its own seeded weights and latents (``wan_synth``), rounds them
to bf16 (the bf16 decode's contract, section "Precision" of the page
"wan22_vae_decode/reference.py") and runs ``oracle.decode``, the page's frame
loop, on the first ``n_latent`` latent frames.
"""

from __future__ import annotations

import multiprocessing
import os

# (workload name, latent frames): the oracle decodes of the full-size tests
JOBS = (("720p", 2), ("portrait", 2), ("480p_b2", 1), ("wan21_720p", 1))
WORKERS = 3

_pool = None
_futures: dict = {}


def jobs_for(nodeids) -> tuple:
    """The jobs that the selected full-size tests need (by test id)."""
    need = []
    for job in JOBS:
        tag = {"720p": "[720p]", "portrait": "[portrait]", "480p_b2": "480p", "wan21_720p": "wan21"}[job[0]]
        if any("test_gpu_fullsize.py" in n and tag in n for n in nodeids):
            need.append(job)
    return tuple(need)


def _init_worker(threads: int) -> None:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = str(threads)


def run_job(name: str, n_latent: int):
    """The oracle's bf16-contract decode of latent frames [0, n_latent) of a
    workload (fp32 arithmetic on bf16-rounded inputs)."""
    import numpy as np

    import oracle
    import wan_synth
    cfg = wan_synth.CONFIGS[name]
    z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
    w = wan_synth.make_weights(base=cfg["base"], seed=cfg["weight_seed"], variant=cfg.get("variant", "ti2v"))
    wr = {k: oracle.round_bf16(v) for k, v in w.items()}
    zr = oracle.round_bf16(np.ascontiguousarray(z[:, :, :n_latent]))
    return oracle.decode(zr, wr)


def start(jobs=JOBS) -> None:
    """Submits the jobs (once per process); returns at once."""
    global _pool
    if _pool is not None:
        return
    cores = os.cpu_count() or 4
    _pool = multiprocessing.get_context("spawn").Pool(
        processes=WORKERS, initializer=_init_worker, initargs=(max(1, cores // WORKERS),))
    for name, n in jobs:
        _futures[(name, n)] = _pool.apply_async(run_job, (name, n))


def result(name: str, n_latent: int):
    """The job's video (starting the pool if nobody has); blocks until done."""
    if _pool is None:
        start(((name, n_latent),))
    if (name, n_latent) not in _futures:
        _futures[(name, n_latent)] = _pool.apply_async(run_job, (name, n_latent))
    return _futures[(name, n_latent)].get()


def shutdown() -> None:
    """Stops the workers, including any still computing."""
    global _pool
    if _pool is not None:
        _pool.terminate()
        _pool.join()
        _pool = None
        _futures.clear()
