"""The seeded generator gives the same bytes on the GPU as on the host, for
every distribution the workloads use (Box-Muller normals with and without
outliers, uniforms), over whole slabs, so that an input generated on the
device is the oracle's input bit for bit."""
import numpy as np
import pytest
import torch

from tests import gpu_helpers as H
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("start,count", [(0, 1 << 22), (3_000_000_001, 1_000_003)])
def test_device_slabs_equal_host_slabs(start, count):
    dev = H.device()
    cases = [(C.CFG2.dist, C.CFG2.key(3)), (C.CFG1.dist, C.CFG1.key(1)),
             (C.CFG4.dist, syn.stream_key(C.CFG4.seed, 0, 0, 0))]
    for dist, key in cases:
        host = syn.bf16_bits(dist.fill(start, count, key))
        gpu = syn.bf16_bits(dist.fill(start, count, key, device=dev))
        assert np.array_equal(host, gpu), (dist, start)
