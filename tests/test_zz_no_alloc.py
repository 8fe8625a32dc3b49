"""w4_gemv_levels_noalloc: the one-launch multi-level GEMV for callers that cannot allocate device
memory (code inside an allocator callback, processes whose device memory a caching allocator
reserved up front, serving loops that forbid allocation after warm-up, plugins that only receive
their input and output buffers).  Its level counters live in a fixed array inside libw4 instead of
a caller workspace.

Checked through the C ABI: two calls in a row give the same outputs, within the GEMV tolerance of
the other tests, as the existing workspace-based entry point (w4_step_create + w4_step_launch);
sizes beyond the fixed array are refused with W4_ERR_LIMIT before anything is launched.  This file
is collected last so that a run stopping at the first failure has already run everything else.
"""
import numpy as np
import pytest

import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import _lib

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(libw4):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def _close(y, y_ref):
    y = y.astype(np.float64)
    y_ref = y_ref.astype(np.float64)
    err = y - y_ref
    rel = np.linalg.norm(err) / np.linalg.norm(y_ref)
    assert np.all(np.isfinite(y)) and rel <= 1e-3
    assert np.max(np.abs(err)) <= 2e-2 * np.sqrt(np.mean(y_ref ** 2))


@pytest.mark.parametrize("fmt", ["nf4", "int4"])
def test_noalloc_matches_workspace_step_twice(dev, fmt):
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep(fmt, batch=1, device=str(dev), layers=2, lm_head=False).build().capture()
    stream = torch.cuda.Stream(dev)
    w4.check(step.launch(stream))                   # existing entry point, caller workspace
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    ref = [step.y_of(i).cpu().numpy().copy() for i in range(len(step.gemvs))]
    descs = step.descriptors()
    for call in range(2):                           # the array keeps the previous call's contents
        step.y.fill_(float("nan"))
        w4.check(w4.w4_gemv_levels_noalloc(descs, stream), f"no-alloc call {call}")
        torch.cuda.synchronize()
        assert w4.w4_device_check(stream) == 0
        for i in range(len(step.gemvs)):
            _close(step.y_of(i).cpu().numpy(), ref[i])
    step.close()


def test_noalloc_refuses_sizes_beyond_its_array(dev):
    x = torch.zeros(1536, dtype=torch.float16, device=dev)
    y = torch.zeros(256, dtype=torch.float16, device=dev)
    packed = torch.zeros((256, 768), dtype=torch.uint8, device=dev)
    scale = torch.zeros((256, 12), dtype=torch.float16, device=dev)
    n = _lib.W4_NOALLOC_MAX_LEVELS + 1
    descs = [dict(format=_lib.W4_FMT_INT4, packed=packed, scales=scale, codebook=None, x=x, y=y,
                  M=1, N=256, K=1536, blocksize=128, level=i) for i in range(n)]
    assert w4.w4_gemv_levels_noalloc(descs) == _lib.W4_ERR_LIMIT
