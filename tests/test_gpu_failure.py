"""Failure detection without a GPU fault: a bounded in-kernel wait that runs
out is reported through the device error flag, and the handle recovers.

The streaming kernel's grid barrier counts arrivals on one 64-bit counter and
ends each barrier at the next multiple of the grid.  Offsetting that count by
grid - 1 before a single-launch forward leaves all but one CTA waiting for an
arrival that never comes: their waits give up after about 2 s, set the
timeout flag and the launch returns.  get_device_error reports the flag and
resets the counters; the next forward is again correct."""
import time

import numpy as np
import pytest

from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import make_layer, run_forward

pytestmark = pytest.mark.gpu


def test_barrier_wait_times_out_reports_and_recovers():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.generate("decode-1")
    layer = make_layer(wl, dev)
    good = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    layer.debug_offset_grid_barrier(grid - 1)
    t0 = time.time()
    run_forward(layer, wl, dev)  # output undefined: the barrier gave up
    elapsed = time.time() - t0
    flags = layer.device_error()
    assert flags & api.DEVFLAG_TIMEOUT, flags
    assert 1.0 < elapsed < 60.0, elapsed
    again = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    assert np.array_equal(again, good)
    layer.close()
