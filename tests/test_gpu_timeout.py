"""The bounded-wait failure path of the decode kernels, driven without a GPU
fault: in the library's test mode every consumer warp first waits a few
microseconds on a barrier that nothing completes.  The wait runs out, the
kernel reports KV_ETIMEOUT through the status word, the producer stops and
lets its copies in flight land, and the call ends quickly (the producer
notices the consumers' abort instead of sitting out its own limit).  After
the mode is turned off and the workspace reset, the same workspace decodes
correctly again."""
import os
import time

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, assert_decode_close

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))


@pytest.mark.parametrize("engine", [0, kv.KV_DECODE_TENSOR_CORE], ids=["fused", "tensor_core"])
def test_consumer_wait_runs_out(engine):
    x = W.small_decode(81, 4, 32, 8, 128, [3000, 17, 0, 1200])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16,
                                                        engine))
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    out, lse, rc = dd.run(pages_per_split=engine, ws=ws)   # warm: kernels set up
    assert rc == 0
    try:
        kv.kv_test_consumer_timeout(2000)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        out, lse, rc = dd.run(pages_per_split=engine, ws=ws)
        dt = time.perf_counter() - t0
    finally:
        kv.kv_test_consumer_timeout(0)
    assert rc == kv.KV_ETIMEOUT
    assert dt < 1.0, dt   # far below the 4 s limit of the producer's own waits
    kv.kv_workspace_reset(ws)
    out, lse, rc = dd.run(pages_per_split=engine, ws=ws)
    assert rc == 0
    assert_decode_close(x, out, lse, ref_out, ref_lse)
