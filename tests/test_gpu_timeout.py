"""A bounded wait of the tcgen05 kernel runs out: the kernel returns, reports
NVFP4KV_FLAG_COPY_TIMEOUT, and the context stays usable.

The failure is made in a separate build of the library (test defines): the
first dequant warp of CTA (0, 0) withholds its arrival for the first tile, so
the product issuer never sees that tile's inputs; its idle bound (shortened
to about a millisecond in this build, like every wait's) runs out, it raises
the CTA's abort word and flag 0x4, and every other wait of the CTA returns at
once; copies and products in flight are drained before the tensor memory is
released.  Nothing faults or hangs: a wait that runs out is the designed end
of the kernel.  The production library then runs the same case clean and
correct."""
import contextlib
import ctypes as C
import os

import pytest
import torch

import gpu_harness as H
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import _lib
from nvfp4_paged_kv_nvfp4kv_gb300 import build as B
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TEST_DEFINES = ["NVFP4KV_TG5_TEST_SKIP_ARRIVE=1", "NVFP4KV_TG5_POLLS=50",
                "NVFP4KV_TG5_IDLE_POLLS=20000"]


@pytest.fixture(scope="module")
def timeout_lib():
    path = B.build(defines=TEST_DEFINES,
                   out=os.path.join(B.BUILD, "timeout", "libnvfp4kv.so"))
    L = C.CDLL(path)
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


@contextlib.contextmanager
def using(lib):
    prod = _lib.load()
    _lib._lib = lib
    try:
        yield
    finally:
        _lib._lib = prod


def extend_batch():
    cfg = W.custom_workload(seed=61, batch=3, kv_lens=(40, 300, 1000), qo_len=16,
                            num_qo_heads=8, num_kv_heads=2, causal=True)
    return W.make_batch(cfg)


def test_tcgen05_wait_runs_out_and_reports(timeout_lib):
    batch = extend_batch()
    with using(timeout_lib):
        g = H.GpuCase(batch, kernel=3)
        assert g.plan.info.kernel == 3
        out, lse = g.run()            # returns: the synchronise inside completes
        flags = N.nvfp4kv_workspace_flags(g.plan, clear=True)
    assert flags & _lib.FLAG_COPY_TIMEOUT, flags
    # the context is still usable
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 499500.0


def test_production_library_runs_the_same_case_clean():
    batch = extend_batch()
    g = H.GpuCase(batch, kernel=3)
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    oc, pt = H.oracle_cache(batch)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)
