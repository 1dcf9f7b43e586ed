"""Host cost per call of the small, launch-bound workload (fp32 1024 x 768
softmax), measured from C by tests/native/host_cost.c (the C ABI alone) and
through the Python binding. The bounds are loose (they catch a regression
such as a per-call environment scan or device query coming back, not the
last microsecond); bench.py reports the measured figures."""
import json

import pytest
import torch

from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]


def test_host_cost_from_c():
    import bench

    r = bench.host_cost_c()
    if r is None:
        pytest.skip("no host C compiler to build the driver")
    print(json.dumps(r))
    assert r["host_us_per_call"] < 10.0
    assert r["graph_us_per_call"] < r["events_us_per_call"] + 1.0


def test_host_cost_through_python():
    import bench

    us = bench.host_cost_python(torch.device("cuda"))
    print(f"python binding: {us:.2f} us per call")
    assert us < 20.0
