"""Shared fixtures.  GPU tests carry the ``gpu`` marker and need a CUDA device
plus the built library; everything else runs on the CPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built sm_103a library")
    config.addinivalue_line("markers", "slow: full-size cases (minutes)")


@pytest.fixture(scope="session")
def tiny_layer():
    """The tiny workload's layer: shape, records, router weights and bias."""
    import synth
    shape = synth.TINY
    seed = synth.WORKLOADS["tiny_t8"][1]
    routed = [synth.expert_record(shape, seed, 0, "routed", e) for e in range(shape.n_experts)]
    shared = [synth.expert_record(shape, seed, 0, "shared", s) for s in range(shape.n_shared)]

    def get_record(kind, e):
        return routed[e] if kind == "routed" else shared[e]

    return dict(shape=shape, seed=seed, routed=routed, shared=shared, get_record=get_record,
                router_w=synth.router_weight(shape, seed), bias=synth.router_bias(shape, seed))
