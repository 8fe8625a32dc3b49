"""Full-size parity of the lm_head shape (151936 x 1536) at the batches of the sweep configuration,
through the C ABI, with weights N(0, 0.02) plus 0.1 % outliers at 10 sigma ("Do Quantization and
Sparsity make LLM Inference Faster ?", section "What we did": the eight shapes at batches 1, 8,
32 and 128).

The weights are quantised on the GPU (bit-exact against the oracle on the sampled rows); the
sampled output rows are checked one by one against the oracle at the GEMV tolerance.  At batches
above 8 the lm_head runs on the tcgen05 kernel with 1187 row tiles over 152 CTAs, so every CTA
takes 7 or 8 tiles: the sample holds rows of each CTA's 1st ... 8th tile for several CTAs, which
covers both tensor-memory accumulators (one at 256 batch columns), their release phases and the
scale slots' reuse.
"""
import numpy as np
import pytest

import oracle
import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N, K = synth.shape_of("lm_head")
OUTLIERS = 0.001
SEED = synth.weight_seed(28, "lm_head")


@pytest.fixture(scope="module")
def dev(libw4):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


@pytest.fixture(scope="module", params=["nf4", "int4"])
def lm_head(request, dev):
    fmt = request.param
    bs = 64 if fmt == "nf4" else 128
    w = synth.weights(SEED, N, K, outlier_frac=OUTLIERS)
    W = torch.from_numpy(w).to(dev)
    del w
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    code = torch.from_numpy(oracle.nf4_codebook()).to(dev)
    if fmt == "nf4":
        sc = torch.empty((N, K // bs), dtype=torch.float32, device=dev)
        w4.check(w4.w4_quantize_nf4(W, packed, sc, code, N, K, bs))
    else:
        sc = torch.empty((N, K // bs), dtype=torch.float16, device=dev)
        w4.check(w4.w4_quantize_int4(W, packed, sc, N, K, bs))
    del W
    torch.cuda.synchronize()
    yield fmt, bs, packed, sc, code
    del packed, sc
    torch.cuda.empty_cache()


def sample_rows(ctas=(0, 1, 37, 75, 76, 150, 151), per_tile=3, seed=0):
    """Rows of the k-th tile (k = 0 ... 7) of several CTAs: tile t = cta + 152 k covers rows
    128 t ... 128 t + 127; plus the first and last rows and random ones."""
    rng = np.random.default_rng(seed)
    rows = [0, N - 1]
    ntiles = (N + 127) // 128
    for cta in ctas:
        for k in range(8):
            t = cta + 152 * k
            if t < ntiles:
                lo, hi = 128 * t, min(N, 128 * t + 128)
                rows.extend(rng.integers(lo, hi, per_tile).tolist())
                rows.append(hi - 1)
    rows.extend(rng.integers(0, N, 32).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))


@pytest.mark.parametrize("m", [9, 32, 128, 256, 300])
def test_lm_head_full_size_batches(dev, lm_head, m):
    """Batches 256 and 300 are prefill-sized: tiles of 256 batch rows on one 256-column accumulator
    (the weights decoded once per 256 rows), 300 = 256 + a 44-row tile."""
    fmt, bs, packed, sc, code = lm_head
    st, plan = w4.w4_gemv_plan(w4._lib.W4_FMT_NF4 if fmt == "nf4" else w4._lib.W4_FMT_INT4, m, N, K, bs)
    assert st == 0 and plan["kernel"] == w4.W4_KERNEL_TCGEN05 and plan["grid"] == 152 and plan["cluster"] == 1
    assert plan["batch_tile"] == (256 if m > 128 else 128 if m > 64 else 64 if m > 32 else 32 if m > 16 else 16)
    x = synth.activations(synth.x_seed(28, 0, m), m, K)
    X = torch.from_numpy(x).to(dev)
    y = torch.full((m, N), float("nan"), dtype=torch.float16, device=dev)
    if fmt == "nf4":
        w4.check(w4.w4_gemv_nf4(packed, sc, code, X, y, m, N, K, bs))
    else:
        w4.check(w4.w4_gemv_int4(packed, sc, X, y, m, N, K, bs))
    torch.cuda.synchronize()
    assert w4.w4_device_check() == 0
    rows = sample_rows(seed=m)
    w_rows = synth.weights_rows(SEED, N, K, rows, outlier_frac=OUTLIERS)
    if fmt == "nf4":
        p_ref, s_ref = oracle.quantize_nf4(w_rows, oracle.nf4_codebook(), bs)
        y_ref = oracle.gemv_nf4(p_ref, s_ref, oracle.nf4_codebook(), x, bs)
    else:
        p_ref, s_ref = oracle.quantize_int4(w_rows, bs)
        y_ref = oracle.gemv_int4(p_ref, s_ref, x, bs)
    idx = torch.from_numpy(rows).to(dev)
    assert np.array_equal(packed[idx].cpu().numpy(), p_ref)
    assert np.array_equal(sc[idx].cpu().numpy().view(np.uint8), s_ref.view(np.uint8))
    got = y[:, idx].cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    for b in range(m):
        err = got[b] - y_ref[b]
        rms = np.sqrt(np.mean(y_ref[b] ** 2))
        assert np.max(np.abs(err)) <= 2e-2 * rms, (b, np.max(np.abs(err)), rms)
        assert np.linalg.norm(err) <= 1e-3 * np.linalg.norm(y_ref[b]), b
