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
        else:
            p, s = oracle.quantize_int4(w, step.bs)
            y_ref = oracle.gemv_int4(p, s, x, step.bs)
        y = step.y_of(i).cpu().numpy()[:, rows].astype(np.float64)
        rms = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
        assert np.all(np.abs(y - y_ref) <= 2e-2 * rms), (layer, proj)
        rel = np.linalg.norm(y - y_ref, axis=1) / np.linalg.norm(y_ref, axis=1)
        assert np.all(rel <= 1e-3), (layer, proj, rel)


@pytest.mark.parametrize("levels", ["grouped", "strict"])
def test_full_nf4_step_graph(dev, levels):
    from weight_only_bit_gb300.step import DecodeStep
    step = DecodeStep("nf4", batch=1, device=str(dev), levels=levels).build().capture()
    assert len(step.gemvs) == 197
    assert step.levels[-1] == (112 if levels == "grouped" else 196)
    stream = torch.cuda.Stream(dev)
    l0 = w4.w4_launch_count()
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_launch_count() - l0 == 1                  # the whole step is one persistent launch
    assert torch.all(step.workspace == 0)                  # counters left at zero for the next launch
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
    assert torch.all(step.workspace == 0)
    step.close()


@pytest.mark.parametrize("fmt,batch", [("int4", 1), ("nf4", 3), ("nf4", 8), ("int4", 8), ("nf4", 32)])
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
    assert torch.all(step.workspace == 0)
    step.close()
    step.capture()
    w4.check(step.launch(stream))
    torch.cuda.synchronize()
    assert w4.w4_device_check(stream) == 0
    _check_step(step, rows_per_gemv=16, seed=2)
    step.close()
