"""The background oracle runs of the full-size parity tests (CPU): which jobs
a selection of tests needs, that the spawned workers return the oracle's
result, and that shutting the pool down stops a job still computing."""

import time

import numpy as np

import oracle
import wan_synth
from tests import oracle_jobs


def test_jobs_follow_the_selected_tests():
    ids = ["tests/test_gpu_fullsize.py::test_full_size_first_two_latent_frames[720p]",
           "tests/test_gpu_fullsize.py::test_full_size_wan21_720p_first_frame",
           "tests/test_gpu_decode.py::test_tiny_decode[1]"]
    assert oracle_jobs.jobs_for(ids) == (("720p", 2), ("wan21_720p", 1))
    assert oracle_jobs.jobs_for(["tests/test_gpu_fullsize.py::test_full_size_480p_batch2"]) == (("480p_b2", 1),)
    assert oracle_jobs.jobs_for(ids[2:]) == ()


def test_worker_result_equals_the_oracle_and_shutdown_stops_the_pool():
    try:
        oracle_jobs.start(jobs=(("tiny", 2), ("small", 3)))
        got = oracle_jobs.result("tiny", 2)
        cfg = wan_synth.CONFIGS["tiny"]
        z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
        w = wan_synth.make_weights(base=cfg["base"], seed=cfg["weight_seed"])
        ref = oracle.decode(oracle.round_bf16(z), {k: oracle.round_bf16(v) for k, v in w.items()})
        np.testing.assert_array_equal(got, ref)
    finally:
        t0 = time.perf_counter()
        oracle_jobs.shutdown()  # the full-width job is still running: terminated, not awaited
        assert time.perf_counter() - t0 < 30.0
    assert oracle_jobs._pool is None
