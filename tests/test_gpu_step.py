"""The decode-step driver: all 197 GEMVs captured in one CUDA graph with programmatic dependent
launch; every GEMV's sampled output rows checked against the oracle, and the graph replay equal
bit for bit to the eager back-to-back sequence."""
import numpy as np
import pytest

import oracle
import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(libw4):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def _check_step(step, rows_per_gemv=8, seed=0):
    rng = np.random.default_rng(seed)
    code = oracle.nf4_codebook()
    for i, (layer, proj, n, k) in enumerate(step.gemvs):
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, rows_per_gemv)]))
        w = synth.weights_rows(synth.weight_seed(layer, proj), n, k, rows, outlier_frac=step.outlier_frac)
        x = step.x_of(i)
        if step.fmt == "nf4":
            p, s = oracle.quantize_nf4(w, code, step.bs)
            y_ref = oracle.gemv_nf4(p, s, code, x, step.bs)
        elif step.fmt == "int4":
            p, s = oracle.quantize_int4(w, step.bs)
            y_ref = oracle.gemv_int4(p, s, x, step.bs)
        else:
            p, s = oracle.quantize_fp4(w, step.bs)
            y_ref = oracle.gemv_fp4(p, s, x, step.bs)
        y = step.y_of(i).cpu().numpy()[:, rows].astype(np.float64)
        rms = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
        assert np.all(np.abs(y - y_ref) <= 2e-2 * rms), (layer, proj)
        rel = np.linalg.norm(y - y_ref, axis=1) / np.linalg.norm(y_ref, axis=1)
        assert np.all(rel <= 1e-3), (layer, proj, rel)


@pytest.mark.parametrize("fmt,levels", [("nf4", "grouped"), ("nf4", "strict"), ("int4", "grouped"),
                                        ("fp4", "grouped")])
def test_full_step_graph(dev, fmt, levels):
    """The whole 197-GEMV step (113 levels grouped, 197 strict) in one persistent launch."""
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep(fmt, batch=1, device=str(dev), levels=levels).build().capture()
    assert len(step.gemvs) == 197
    assert step.levels[-1] == (112 if levels == "grouped" else 196)
    stream = torch.cuda.Stream(dev)
    l0 = w4.w4_launch_count()
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_launch_count() - l0 == 1                  # the whole step is one persistent launch
    assert torch.all(step.counters() == 0)                 # counters left at zero for the next launch
    assert w4.w4_device_check(stream) == 0
    g = step.y.clone()
    _check_step(step)
    # the eager back-to-back sequence gives the same bits
    step.y.fill_(float("nan"))
    w4.check(step.enqueue_eager(stream))
    torch.cuda.synchronize()
    assert torch.equal(step.y.view(torch.int16), g.view(torch.int16))
    # replaying back to back (programmatic launch overlap between replays) changes nothing
    step.y.fill_(float("nan"))
    for _ in range(5):
        w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    assert torch.equal(step.y.view(torch.int16), g.view(torch.int16))
    assert torch.all(step.counters() == 0)
    step.close()


def test_step_with_host_buffers(dev):
    """w4_step_run_host: x copied in from pinned host memory, the step, y copied out; the host y
    equals the device y of a plain launch bit for bit, and a changed host x reaches the kernels."""
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep("nf4", batch=1, device=str(dev), layers=1, lm_head=False).build().capture()
    stream = torch.cuda.Stream(dev)
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    ref = step.y.cpu().clone()
    x_pin = torch.from_numpy(step.x_host.copy()).pin_memory()
    y_pin = torch.full((step.y_elems,), float("nan"), dtype=torch.float16).pin_memory()
    step.x.zero_()
    w4.check(step.run_host(x_pin, y_pin, stream))
    stream.synchronize()
    assert w4.w4_device_check(stream) == 0
    assert torch.equal(y_pin.view(torch.int16), ref.view(torch.int16))
    x_pin.mul_(2)                                  # exact in FP16: every y doubles exactly
    w4.check(step.run_host(x_pin, y_pin, stream))
    stream.synchronize()
    assert torch.equal(y_pin.view(torch.int16), (ref.float() * 2).half().view(torch.int16))
    assert w4.w4_step_run_host(None, x_pin, step.x, 2, y_pin, step.y, 2) == w4._lib.W4_ERR_NULL
    assert w4.w4_step_run_host(step.step, x_pin, step.x, -1, y_pin, step.y, 2) == w4._lib.W4_ERR_SHAPE
    step.close()


@pytest.mark.parametrize("fmt,batch", [("int4", 1), ("nf4", 3), ("nf4", 8), ("int4", 8), ("nf4", 32), ("fp4", 2),
                                       ("fp4", 8), ("fp4", 32)])
def test_reduced_steps(dev, fmt, batch):
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep(fmt, batch=batch, device=str(dev), layers=2, lm_head=False,
                      outlier_frac=0.001).build().capture()
    stream = torch.cuda.Stream(dev)
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    _check_step(step, rows_per_gemv=16, seed=1)
    step.close()


@pytest.mark.parametrize("levels", ["strict", "grouped"])
def test_one_layer_steps_replayed_back_to_back(dev, levels):
    """A one-layer step replayed several times in a row: every level's first tile must reach the
    ring even while the stream gate is closed (the consumers wait for it before they wait for the
    previous level), so no bounded wait may run out."""
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep("nf4", batch=1, device=str(dev), layers=1, lm_head=False, levels=levels).build().capture()
    stream = torch.cuda.Stream(dev)
    for _ in range(4):
        w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    assert torch.all(step.counters() == 0)
    _check_step(step, rows_per_gemv=16, seed=3)
    step.close()


def test_step_timeout_path_recovers(dev):
    """The injected producer failure inside a multi-level persistent step: every bounded wait ends,
    the host reads W4_ERR_TIMEOUT, the counters are left at zero and the next replay is right."""
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep("nf4", batch=1, device=str(dev), layers=1, lm_head=False)
    step.build()
    stream = torch.cuda.Stream(dev)
    w4.w4_inject_timeout_once()
    step.capture()                       # the hook applies to the captured launch
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == w4._lib.W4_ERR_TIMEOUT
    assert torch.all(step.counters() == 0)
    step.close()
    step.capture()
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    _check_step(step, rows_per_gemv=16, seed=2)
    step.close()


@pytest.mark.parametrize("fmt,batch", [("nf4", 1), ("int4", 1), ("nf4", 3), ("int4", 8)])
def test_chained_levels_read_previous_outputs(dev, fmt, batch):
    """A chain in ONE persistent launch where level L+1's x IS level L's y (written by other CTAs
    during the same launch), with a fan-out level (two GEMVs on one x) and a long-K level.  Equal
    bit for bit to one launch per GEMV (stream order), and every level within tolerance of the
    oracle applied to the x the GPU actually read."""
    code = oracle.nf4_codebook()
    bs = 64 if fmt == "nf4" else 128
    # (N, K) per GEMV and its level; level 3 has two GEMVs reading level 2's output
    shapes = [(1536, 1536, 0), (2048, 1536, 1), (1536, 2048, 2), (640, 1536, 3), (1536, 1536, 3)]
    codebook = torch.tensor(code, dtype=torch.float32, device=dev)
    x0 = torch.from_numpy(synth.activations(777, batch, 1536)).to(dev)
    ys, packs, scales, ws = [], [], [], []
    for i, (n, k, lev) in enumerate(shapes):
        w = synth.weights(5000 + i, n, k, outlier_frac=0.001)
        ws.append(w)
        W = torch.from_numpy(w).to(dev)
        p = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        if fmt == "nf4":
            s = torch.empty((n, k // bs), dtype=torch.float32, device=dev)
            w4.check(w4.w4_quantize_nf4(W, p, s, codebook, n, k, bs))
        else:
            s = torch.empty((n, k // bs), dtype=torch.float16, device=dev)
            w4.check(w4.w4_quantize_int4(W, p, s, n, k, bs))
        packs.append(p)
        scales.append(s)
        ys.append(torch.full((batch, n), float("nan"), dtype=torch.float16, device=dev))
    # level 0 reads x0; GEMV i > 0 reads the output of the last GEMV of the level before
    xs = [x0, ys[0], ys[1], ys[2], ys[2]]
    fmt_id = w4._lib.W4_FMT_NF4 if fmt == "nf4" else w4._lib.W4_FMT_INT4
    descs = [dict(format=fmt_id, packed=packs[i], scales=scales[i], codebook=codebook, x=xs[i], y=ys[i],
                  M=batch, N=n, K=k, blocksize=bs, level=lev) for i, (n, k, lev) in enumerate(shapes)]
    torch.cuda.synchronize()
    ws_bytes = w4.w4_step_workspace_bytes(len(descs))
    workspace = torch.zeros(ws_bytes // 4, dtype=torch.int32, device=dev)
    st, h = w4.w4_step_create(descs, workspace)
    w4.check(st, "step create")
    stream = torch.cuda.Stream(dev)
    l0 = w4.w4_launch_count()
    w4.check(w4.w4_step_launch(h, stream))
    torch.cuda.synchronize()
    assert w4.w4_launch_count() - l0 == 1
    assert w4.w4_device_check(stream) == 0
    got = [y.clone() for y in ys]
    # each level against the oracle, fed the x the GPU read
    for i, (n, k, lev) in enumerate(shapes):
        x = xs[i].cpu().numpy().astype(np.float64)
        if fmt == "nf4":
            p, s = oracle.quantize_nf4(ws[i], code, bs)
            y_ref = oracle.gemv_nf4(p, s, code, x, bs)
        else:
            p, s = oracle.quantize_int4(ws[i], bs)
            y_ref = oracle.gemv_int4(p, s, x, bs)
        y = got[i].cpu().numpy().astype(np.float64)
        rms = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
        assert np.all(np.abs(y - y_ref) <= 2e-2 * rms), i
        rel = np.linalg.norm(y - y_ref, axis=1) / np.linalg.norm(y_ref, axis=1)
        assert np.all(rel <= 1e-3), (i, rel)
    # one launch per GEMV in stream order gives the same bits
    for y in ys:
        y.fill_(float("nan"))
    w4.check(w4.w4_gemv_sequence(descs, stream))
    torch.cuda.synchronize()
    for a, b in zip(got, ys):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # and replays of the step keep giving them
    for _ in range(3):
        w4.check(w4.w4_step_launch(h, stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    for a, b in zip(got, ys):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.all(workspace[: len(descs) + 1] == 0)          # the level counters
    w4.check(w4.w4_step_destroy(h))


@pytest.mark.parametrize("batch", [1, 3])
def test_step_with_mixed_block_sizes(dev, batch):
    """GEMVs with different NF4 block sizes (64, 128, 256) and a K that is not a multiple of 128 in
    one persistent launch: the general unit (scales looked up per k block) serves every span, and
    the results equal the oracle and, bit for bit, one launch per GEMV (each of which compiles its
    block size in)."""
    code = oracle.nf4_codebook()
    codebook = torch.tensor(code, dtype=torch.float32, device=dev)
    # (N, K, blocksize, level)
    shapes = [(1536, 1536, 64, 0), (700, 1536, 128, 0), (300, 1600, 64, 1), (900, 1024, 256, 2)]
    descs, ws, xs, ys = [], [], [], []
    for i, (n, k, bs, lev) in enumerate(shapes):
        w = synth.weights(6100 + i, n, k, outlier_frac=0.001)
        x = synth.activations(6200 + i, batch, k)
        p = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        s = torch.empty((n, k // bs), dtype=torch.float32, device=dev)
        w4.check(w4.w4_quantize_nf4(torch.from_numpy(w).to(dev), p, s, codebook, n, k, bs))
        X = torch.from_numpy(x).to(dev)
        y = torch.full((batch, n), float("nan"), dtype=torch.float16, device=dev)
        ws.append(w); xs.append(X); ys.append(y)
        descs.append(dict(format=w4._lib.W4_FMT_NF4, packed=p, scales=s, codebook=codebook, x=X, y=y,
                          M=batch, N=n, K=k, blocksize=bs, level=lev))
    torch.cuda.synchronize()
    workspace = torch.zeros(w4.w4_step_workspace_bytes(len(descs)) // 4, dtype=torch.int32, device=dev)
    st, h = w4.w4_step_create(descs, workspace)
    w4.check(st, "step create")
    stream = torch.cuda.Stream(dev)
    w4.check(w4.w4_step_launch(h, stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    got = [y.clone() for y in ys]
    for i, (n, k, bs, lev) in enumerate(shapes):
        p, s = oracle.quantize_nf4(ws[i], code, bs)
        y_ref = oracle.gemv_nf4(p, s, code, xs[i].cpu().numpy().astype(np.float64), bs)
        y = got[i].cpu().numpy().astype(np.float64)
        rms = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
        assert np.all(np.abs(y - y_ref) <= 2e-2 * rms), i
        rel = np.linalg.norm(y - y_ref, axis=1) / np.linalg.norm(y_ref, axis=1)
        assert np.all(rel <= 1e-3), (i, rel)
    for y in ys:
        y.fill_(float("nan"))
    w4.check(w4.w4_gemv_sequence(descs, stream))
    torch.cuda.synchronize()
    for a, b in zip(got, ys):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    w4.check(w4.w4_step_destroy(h))
