import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def tiny_weights():
    import wan_synth
    return wan_synth.make_weights(base=16, seed=0)


def pytest_collection_finish(session):
    """Starts the background oracle runs of the full-size parity tests as soon
    as one of them is selected, so they overlap the other GPU tests."""
    if session.config.option.collectonly:
        return
    from tests import oracle_jobs
    jobs = oracle_jobs.jobs_for([item.nodeid for item in session.items])
    if jobs:
        oracle_jobs.start(jobs)


def pytest_sessionfinish(session, exitstatus):
    from tests import oracle_jobs
    oracle_jobs.shutdown()
