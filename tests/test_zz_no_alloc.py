"""w4_gemv_levels_noalloc: the one-launch multi-level GEMV for callers that cannot allocate device
memory (code inside an allocator callback, processes whose device memory a caching allocator
reserved up front, serving loops that forbid allocation after warm-up, plugins that only receive
their input and output buffers).  Its level counters live in a fixed array inside libw4 instead of
a caller workspace.

Checked through the C ABI: two calls in a row give the same bits as the existing workspace-based
entry point (w4_step_create + w4_step_launch), which runs the same kernel with the same tiling, and
sampled rows agree with the oracle; a call whose waits ran out (test hook) reports W4_ERR_TIMEOUT
and the next call is right again (each call clears its counters first); a chain whose levels read
the previous level's output in the same launch matches the workspace step bit for bit; sizes
beyond the fixed arrays are refused with W4_ERR_LIMIT before anything is launched.  This file is
collected last so that a run stopping at the first failure has already run everything else.
"""
import numpy as np
import pytest

import oracle
import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import _lib, synth

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


def _oracle_rows(step, i, rows):
    layer, proj, n, k = step.gemvs[i]
    w = synth.weights_rows(synth.weight_seed(layer, proj), n, k, rows, outlier_frac=step.outlier_frac)
    x = step.x_of(i)
    if step.fmt == "nf4":
        code = oracle.nf4_codebook()
        p, s = oracle.quantize_nf4(w, code, step.bs)
        return oracle.gemv_nf4(p, s, code, x, step.bs)
    if step.fmt == "int4":
        p, s = oracle.quantize_int4(w, step.bs)
        return oracle.gemv_int4(p, s, x, step.bs)
    p, s = oracle.quantize_fp4(w, step.bs)
    return oracle.gemv_fp4(p, s, x, step.bs)


@pytest.mark.parametrize("fmt,batch", [("nf4", 1), ("int4", 1), ("fp4", 4)])
def test_noalloc_matches_workspace_step_twice(dev, fmt, batch):
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep(fmt, batch=batch, device=str(dev), layers=2, lm_head=False).build().capture()
    stream = torch.cuda.Stream(dev)
    w4.check(step.launch(stream))                   # existing entry point, caller workspace
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    ref = step.y.clone()
    rng = np.random.default_rng(11)
    for i in range(len(step.gemvs)):
        n = step.gemvs[i][2]
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 6)]))
        _close(step.y_of(i).cpu().numpy()[:, rows], _oracle_rows(step, i, rows))
    descs = step.descriptors()
    for call in range(2):                           # the arrays keep the previous call's contents
        step.y.fill_(float("nan"))
        w4.check(w4.w4_gemv_levels_noalloc(descs, stream), f"no-alloc call {call}")
        torch.cuda.synchronize()
        assert w4.w4_device_check(stream) == 0
        assert torch.equal(step.y.view(torch.int16), ref.view(torch.int16))
    step.close()


def test_noalloc_after_a_timed_out_call(dev):
    """The test hook makes the next launch's producer issue nothing: the no-alloc call's waits run
    out and leave its counters wherever they stopped; the next call clears them and is exact."""
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep("nf4", batch=1, device=str(dev), layers=1, lm_head=False).build().capture()
    stream = torch.cuda.Stream(dev)
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    ref = step.y.clone()
    descs = step.descriptors()
    w4.w4_inject_timeout_once()
    w4.check(w4.w4_gemv_levels_noalloc(descs, stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == _lib.W4_ERR_TIMEOUT
    step.y.fill_(float("nan"))
    w4.check(w4.w4_gemv_levels_noalloc(descs, stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    assert torch.equal(step.y.view(torch.int16), ref.view(torch.int16))
    step.close()


@pytest.mark.parametrize("fmt", ["nf4", "int4"])
def test_noalloc_chained_levels(dev, fmt):
    """Level L+1's x is level L's y, written by other CTAs in the same launch (with a fan-out level):
    the no-alloc call gives the workspace step's bits, twice."""
    bs = 64 if fmt == "nf4" else 128
    fmt_id = _lib.W4_FMT_NF4 if fmt == "nf4" else _lib.W4_FMT_INT4
    shapes = [(1536, 1536, 0), (2048, 1536, 1), (1536, 2048, 2), (640, 1536, 3), (1536, 1536, 3)]
    codebook = torch.tensor(oracle.nf4_codebook(), dtype=torch.float32, device=dev)
    x0 = torch.from_numpy(synth.activations(778, 1, 1536)).to(dev)
    ys, packs, scales = [], [], []
    for i, (n, k, lev) in enumerate(shapes):
        W = torch.from_numpy(synth.weights(5100 + i, n, k)).to(dev)
        p = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        if fmt == "nf4":
            s = torch.empty((n, k // bs), dtype=torch.float32, device=dev)
            w4.check(w4.w4_quantize_nf4(W, p, s, codebook, n, k, bs))
        else:
            s = torch.empty((n, k // bs), dtype=torch.float16, device=dev)
            w4.check(w4.w4_quantize_int4(W, p, s, n, k, bs))
        packs.append(p)
        scales.append(s)
        ys.append(torch.full((1, n), float("nan"), dtype=torch.float16, device=dev))
    xs = [x0, ys[0], ys[1], ys[2], ys[2]]
    descs = [dict(format=fmt_id, packed=packs[i], scales=scales[i], codebook=codebook, x=xs[i], y=ys[i],
                  M=1, N=n, K=k, blocksize=bs, level=lev) for i, (n, k, lev) in enumerate(shapes)]
    torch.cuda.synchronize()
    workspace = torch.zeros(w4.w4_step_workspace_bytes(len(descs)) // 4, dtype=torch.int32, device=dev)
    st, h = w4.w4_step_create(descs, workspace)
    w4.check(st, "step create")
    stream = torch.cuda.Stream(dev)
    w4.check(w4.w4_step_launch(h, stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    ref = [y.clone() for y in ys]
    for call in range(2):
        for y in ys:
            y.fill_(float("nan"))
        w4.check(w4.w4_gemv_levels_noalloc(descs, stream), f"no-alloc call {call}")
        torch.cuda.synchronize()
        assert w4.w4_device_check(stream) == 0
        for y, r in zip(ys, ref):
            assert torch.equal(y.view(torch.int16), r.view(torch.int16))
    w4.check(w4.w4_step_destroy(h))


def test_noalloc_refuses_sizes_beyond_its_array(dev):
    x = torch.zeros(1536, dtype=torch.float16, device=dev)
    y = torch.zeros(256, dtype=torch.float16, device=dev)
    packed = torch.zeros((256, 768), dtype=torch.uint8, device=dev)
    scale = torch.zeros((256, 12), dtype=torch.float16, device=dev)
    n = _lib.W4_NOALLOC_MAX_LEVELS + 1
    descs = [dict(format=_lib.W4_FMT_INT4, packed=packed, scales=scale, codebook=None, x=x, y=y,
                  M=1, N=256, K=1536, blocksize=128, level=i) for i in range(n)]
    assert w4.w4_gemv_levels_noalloc(descs) == _lib.W4_ERR_LIMIT
