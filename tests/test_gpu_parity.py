"""CUDA path against the oracle, through the C ABI, on seeded synthetic inputs.

Bars (from the target's stated criteria):
  * packing, codes, absmax, FP16 scales and dequantised weights: bit-exact;
  * GEMV: per output vector, relative L2 error <= 1e-3 and max |error| <= 2e-2 * RMS(y_ref)
    against the float64 oracle.
"""
import numpy as np
import pytest

import oracle
import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
MAX_ABS_RMS = 2e-2


@pytest.fixture(scope="module")
def dev(libw4):
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return torch.device("cuda:0")


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _code(dev):
    return _t(oracle.nf4_codebook(), dev)


def gpu_quantize(fmt, w, bs, dev):
    n, k = w.shape
    W = _t(w, dev)
    packed = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
    if fmt == "nf4":
        sc = torch.empty((n, k // bs), dtype=torch.float32, device=dev)
        w4.check(w4.w4_quantize_nf4(W, packed, sc, _code(dev), n, k, bs))
    else:
        sc = torch.empty((n, k // bs), dtype=torch.float16, device=dev)
        quant = w4.w4_quantize_int4 if fmt == "int4" else w4.w4_quantize_fp4
        w4.check(quant(W, packed, sc, n, k, bs))
    return packed, sc


def gpu_gemv(fmt, packed, sc, x, n, k, bs, dev, y=None):
    m = x.shape[0]
    X = _t(x, dev)
    if y is None:
        y = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
    launch_gemv(fmt, packed, sc, X, y, m, n, k, bs, dev)
    torch.cuda.synchronize()
    return y


def launch_gemv(fmt, packed, sc, X, y, m, n, k, bs, dev):
    if fmt == "nf4":
        w4.check(w4.w4_gemv_nf4(packed, sc, _code(dev), X, y, m, n, k, bs))
    elif fmt == "int4":
        w4.check(w4.w4_gemv_int4(packed, sc, X, y, m, n, k, bs))
    else:
        w4.check(w4.w4_gemv_fp4(packed, sc, X, y, m, n, k, bs))


# default block / group size of each format
BS = {"nf4": 64, "int4": 128, "fp4": 32}


def oracle_quantize(fmt, w, bs):
    if fmt == "nf4":
        return oracle.quantize_nf4(w, oracle.nf4_codebook(), bs)
    if fmt == "int4":
        return oracle.quantize_int4(w, bs)
    return oracle.quantize_fp4(w, bs)


def oracle_dequantize(fmt, packed, sc, bs):
    if fmt == "nf4":
        return oracle.dequantize_nf4(packed, sc, oracle.nf4_codebook(), bs)
    if fmt == "int4":
        return oracle.dequantize_int4(packed, sc, bs)
    return oracle.dequantize_fp4(packed, sc, bs)


def oracle_gemv(fmt, packed, sc, x, bs, rows=None):
    if fmt == "nf4":
        return oracle.gemv_nf4(packed, sc, oracle.nf4_codebook(), x, bs, rows=rows)
    if fmt == "int4":
        return oracle.gemv_int4(packed, sc, x, bs, rows=rows)
    return oracle.gemv_fp4(packed, sc, x, bs, rows=rows)


def assert_gemv_close(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y))
    for m in range(y_ref.shape[0]):
        err = y[m] - y_ref[m]
        rms = np.sqrt(np.mean(y_ref[m] ** 2))
        rel = np.linalg.norm(err) / max(np.linalg.norm(y_ref[m]), 1e-300)
        assert rel <= REL_L2, f"row {m}: relative L2 {rel:.3e}"
        assert np.max(np.abs(err)) <= MAX_ABS_RMS * rms, f"row {m}: max abs {np.max(np.abs(err)):.3e} rms {rms:.3e}"


QUANT_CASES = [
    # (fmt, N, K, bs)
    ("nf4", 1, 64, 64), ("nf4", 3, 128, 64), ("nf4", 257, 1536, 64), ("nf4", 16, 8960, 64),
    ("nf4", 5, 256, 32), ("nf4", 7, 512, 128), ("nf4", 2, 512, 256),
    ("int4", 1, 128, 128), ("int4", 3, 256, 128), ("int4", 257, 1536, 128), ("int4", 16, 8960, 128),
    ("int4", 5, 256, 32), ("int4", 7, 512, 64), ("int4", 2, 512, 256),
    ("fp4", 1, 32, 32), ("fp4", 3, 128, 32), ("fp4", 257, 1536, 32), ("fp4", 16, 8960, 32),
    ("fp4", 5, 256, 64), ("fp4", 7, 512, 128), ("fp4", 2, 512, 256),
]


@pytest.mark.parametrize("fmt,n,k,bs", QUANT_CASES)
def test_quantize_bit_exact(dev, fmt, n, k, bs):
    w = synth.weights(1000 + n + k + bs, n, k, outlier_frac=0.01)
    w[0, : min(k, bs)] = 0.0                                   # an all-zero block
    packed, sc = gpu_quantize(fmt, w, bs, dev)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    got = sc.cpu().numpy()
    assert got.dtype == s_ref.dtype and np.array_equal(got.view(np.uint8), s_ref.view(np.uint8))


@pytest.mark.parametrize("fmt,bs", [("nf4", 64), ("int4", 128), ("fp4", 32)])
def test_quantize_ties_and_grid_points(dev, fmt, bs):
    """Values exactly on code points and exactly at rounding boundaries."""
    code = oracle.nf4_codebook()
    rows = []
    if fmt == "nf4":
        a = np.float32(2.0 ** -5)
        q = np.arange(64) % 16
        rows.append((code[q] * a).astype(np.float32))
        mids = ((code[:-1].astype(np.float64) + code[1:]) / 2 * float(a)).astype(np.float32)
        r = np.zeros(64, np.float32); r[:15] = mids; r[15] = a
        rows.append(r)
    elif fmt == "int4":
        s = 2.0 ** -6
        t = np.array([2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 6.5, -6.5], np.float64)
        r = np.zeros(128, np.float32); r[: len(t)] = (t * s).astype(np.float32); r[127] = 7 * s
        rows.append(r)
        rows.append(((np.arange(128) % 15 - 7) * s).astype(np.float32))
    else:
        s = 2.0 ** -4
        grid = oracle.fp4_grid()
        mids = (grid[:-1] + grid[1:]) / 2
        r = np.zeros(32, np.float32)
        r[:7] = mids * s; r[7:14] = -mids * s; r[31] = 6 * s
        r[14:21] = np.nextafter((mids * s).astype(np.float32), np.float32(1))
        r[21:28] = np.nextafter((mids * s).astype(np.float32), np.float32(0))
        rows.append(r)
        rows.append(np.concatenate([grid, -grid[1:], grid, -grid[1:], [6.0, -6.0]]).astype(np.float32) * np.float32(s))
    w = np.stack(rows)
    packed, sc = gpu_quantize(fmt, w, bs, dev)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint8), s_ref.view(np.uint8))


@pytest.mark.parametrize("fmt,n,k,bs", [c for c in QUANT_CASES if c[1] > 1])
def test_dequantize_bit_exact(dev, fmt, n, k, bs):
    w = synth.weights(2000 + n + k, n, k)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    packed, sc = _t(p_ref, dev), _t(s_ref, dev)
    out = torch.empty((n, k), dtype=torch.float32, device=dev)
    if fmt == "nf4":
        w4.check(w4.w4_dequantize_nf4(packed, sc, _code(dev), out, n, k, bs))
    elif fmt == "int4":
        w4.check(w4.w4_dequantize_int4(packed, sc, out, n, k, bs))
    else:
        w4.check(w4.w4_dequantize_fp4(packed, sc, out, n, k, bs))
    ref = oracle_dequantize(fmt, p_ref, s_ref, bs)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


GEMV_CASES = [
    # (fmt, M, N, K, bs): tiny, ragged, several tiles, both K of the decode step
    ("nf4", 1, 1, 64, 64), ("nf4", 1, 3, 128, 64), ("nf4", 1, 257, 1536, 64), ("nf4", 1, 256, 1536, 64),
    ("nf4", 1, 1536, 1536, 64), ("nf4", 1, 100, 8960, 64), ("nf4", 2, 333, 1536, 64), ("nf4", 3, 64, 8960, 64),
    ("nf4", 4, 1000, 1536, 64), ("nf4", 5, 129, 1536, 64), ("nf4", 8, 777, 1536, 64), ("nf4", 8, 61, 8960, 64),
    ("nf4", 1, 70, 512, 32), ("nf4", 1, 70, 512, 128), ("nf4", 2, 70, 1024, 256),
    ("int4", 1, 1, 128, 128), ("int4", 1, 3, 256, 128), ("int4", 1, 257, 1536, 128), ("int4", 1, 256, 1536, 128),
    ("int4", 1, 1536, 1536, 128), ("int4", 1, 100, 8960, 128), ("int4", 2, 333, 1536, 128), ("int4", 3, 64, 8960, 128),
    ("int4", 4, 1000, 1536, 128), ("int4", 5, 129, 1536, 128), ("int4", 8, 777, 1536, 128), ("int4", 8, 61, 8960, 128),
    ("int4", 1, 70, 512, 32), ("int4", 1, 70, 512, 64), ("int4", 2, 70, 1024, 256),
    # an odd number of chunks per row and of batch rows x chunks (shared-memory layouts whose
    # parts are not multiples of 16 bytes)
    ("nf4", 1, 45, 96, 32), ("int4", 1, 45, 96, 32), ("int4", 3, 40, 160, 32), ("nf4", 3, 40, 160, 32),
    ("fp4", 1, 1, 64, 32), ("fp4", 1, 257, 1536, 32), ("fp4", 1, 1536, 1536, 32), ("fp4", 1, 100, 8960, 32),
    ("fp4", 2, 333, 1536, 32), ("fp4", 3, 64, 8960, 32), ("fp4", 4, 1000, 1536, 32), ("fp4", 8, 777, 1536, 32),
    ("fp4", 8, 61, 8960, 32), ("fp4", 1, 70, 512, 64), ("fp4", 2, 70, 1024, 128), ("fp4", 1, 45, 96, 32),
    ("fp4", 3, 40, 160, 32), ("fp4", 5, 129, 1536, 256),
    # batch 1 keeps a tile's partial sums in the 64 KB table's 128-byte gaps (32 spans each): a
    # row's spans filling one gap exactly (K 4096), spilling into a second (K 4224, also an odd
    # box count), three gaps at the largest K, and tiles capped at 128 rows by the gaps (K 512,
    # more rows than 152 tiles of 128)
    ("nf4", 1, 300, 4096, 64), ("nf4", 1, 300, 4224, 64), ("fp4", 1, 257, 4224, 32),
    ("int4", 1, 200, 10240, 128), ("nf4", 1, 40000, 512, 64),
]


@pytest.mark.parametrize("fmt,m,n,k,bs", GEMV_CASES)
def test_gemv_parity(dev, fmt, m, n, k, bs):
    w = synth.weights(3000 + n + k + m, n, k, outlier_frac=0.001)
    x = synth.activations(4000 + n + k + m, m, k)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    y = gpu_gemv(fmt, _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv(fmt, p_ref, s_ref, x, bs))


TC_CASES = [
    # (fmt, M, N, K, bs): the tensor-core paths (batch >= 9), ragged rows and batches, split-K
    # over a cluster (few row tiles), persistent tiles (many), a partial last 256-k super-chunk,
    # and shapes the tcgen05 kernel does not take (K % 64 != 0: mma.sync or CUDA cores)
    ("nf4", 16, 256, 1536, 64), ("int4", 16, 1000, 1600, 32), ("nf4", 24, 200, 320, 64), ("int4", 20, 8960, 1536, 128),
    ("nf4", 17, 128, 64, 64), ("int4", 24, 1536, 8960, 128), ("nf4", 40, 100, 96, 32), ("int4", 20, 100, 160, 32),
    ("int4", 128, 384, 768, 256), ("nf4", 64, 1536, 8960, 64), ("nf4", 9, 8960, 1536, 64), ("int4", 13, 300, 8960, 128),
    # prefill-sized batches: 128-row batch tiles (a remainder of 2 rows on the CUDA cores)
    ("nf4", 300, 640, 1536, 64), ("int4", 130, 257, 1024, 128),
    ("nf4", 32, 8960, 1536, 64), ("nf4", 32, 1536, 8960, 64), ("nf4", 33, 257, 1536, 64), ("nf4", 64, 129, 512, 32),
    ("nf4", 100, 300, 1536, 128), ("nf4", 128, 1536, 1536, 64), ("nf4", 128, 70, 8960, 256),
    ("int4", 32, 8960, 1536, 128), ("int4", 32, 1536, 8960, 128), ("int4", 47, 257, 1536, 64),
    ("int4", 128, 1536, 1536, 128), ("int4", 96, 130, 8960, 32),
    ("fp4", 16, 256, 1536, 32), ("fp4", 9, 8960, 1536, 32), ("fp4", 32, 1536, 8960, 32), ("fp4", 64, 129, 512, 64),
    ("fp4", 128, 1536, 1536, 32), ("fp4", 130, 257, 1024, 32), ("fp4", 20, 100, 160, 32), ("fp4", 40, 100, 96, 32),
    # prefill-sized batches on weight matrices with enough row tiles: 256-row batch tiles on one
    # 256-column accumulator (ragged rows, a ragged batch, several tiles per CTA)
    ("nf4", 256, 20000, 1536, 64), ("int4", 200, 19700, 768, 128), ("fp4", 300, 19500, 512, 32),
    ("nf4", 129, 19460, 1024, 32),
]


@pytest.mark.parametrize("fmt,m,n,k,bs", TC_CASES)
def test_tensor_core_batches(dev, fmt, m, n, k, bs):
    w = synth.weights(8000 + n + k + m, n, k, outlier_frac=0.001)
    x = synth.activations(8100 + n + k + m, m, k)
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(m).integers(0, n, 96)]))
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    packed, sc = _t(p_ref, dev), _t(s_ref, dev)
    y = gpu_gemv(fmt, packed, sc, x, n, k, bs, dev).cpu().numpy()
    assert_gemv_close(y[:, rows], oracle_gemv(fmt, p_ref, s_ref, x, bs, rows=rows))
    # the split-K sums run in a fixed order: a second launch gives the same bits
    y2 = gpu_gemv(fmt, packed, sc, x, n, k, bs, dev).cpu().numpy()
    assert np.array_equal(y.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
@pytest.mark.parametrize("m", [12, 20, 32, 64, 128])
def test_gemv_parity_larger_batches(dev, fmt, m):
    bs = BS[fmt]
    n, k = 300, 1536
    w = synth.weights(5000 + m, n, k)
    x = synth.activations(5100 + m, m, k)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    y = gpu_gemv(fmt, _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv(fmt, p_ref, s_ref, x, bs))


@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
def test_gemv_one_hot_zero_linearity_idempotence(dev, fmt):
    bs = BS[fmt]
    n, k = 96, 1536
    w = synth.weights(6000, n, k)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    packed, sc = _t(p_ref, dev), _t(s_ref, dev)
    wh = oracle_dequantize(fmt, p_ref, s_ref, bs)
    # one-hot x picks column k of w_hat: pins nibble order, block index and orientation
    for kk in (0, 1, 63, 64, 1535):
        x = np.zeros((1, k), np.float16)
        x[0, kk] = 1.0
        y = gpu_gemv(fmt, packed, sc, x, n, k, bs, dev).cpu().numpy()[0]
        exp = wh[:, kk].astype(np.float16)
        if fmt != "nf4":
            # exact path: equal values (bit for bit except that -0 and +0 are both accepted: an
            # FP4 code 8 decodes to -0, and a sum starting from +0 gives +0)
            assert np.array_equal(y, exp)
        else:
            assert np.allclose(y.astype(np.float64), wh[:, kk], rtol=2 ** -10, atol=0)
    # zero input gives exactly zero
    y0 = gpu_gemv(fmt, packed, sc, np.zeros((2, k), np.float16), n, k, bs, dev).cpu().numpy()
    assert np.all(y0 == 0)
    # linearity: doubling x doubles y bit for bit (power-of-two scaling commutes with rounding)
    x = synth.activations(6100, 2, k)
    y1 = gpu_gemv(fmt, packed, sc, x, n, k, bs, dev).cpu().numpy()
    y2 = gpu_gemv(fmt, packed, sc, (2 * x.astype(np.float32)).astype(np.float16), n, k, bs, dev).cpu().numpy()
    assert np.array_equal((2 * y1.astype(np.float32)).astype(np.float16).view(np.uint16), y2.view(np.uint16))
    # idempotence: a second launch into the same (dirty) y gives identical bits
    X = _t(x, dev)
    ya = torch.full((2, n), 7.0, dtype=torch.float16, device=dev)
    for _ in range(2):
        launch_gemv(fmt, packed, sc, X, ya, 2, n, k, bs, dev)
        torch.cuda.synchronize()
        assert np.array_equal(ya.cpu().numpy().view(np.uint16), y1.view(np.uint16))


@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
def test_gemv_writes_nothing_outside_y(dev, fmt):
    bs = BS[fmt]
    n, k, m = 131, 1536, 3
    w = synth.weights(7000, n, k)
    x = synth.activations(7001, m, k)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    guard = 2048
    buf = torch.full((guard + m * n + guard,), 1234.0, dtype=torch.float16, device=dev)
    y = buf[guard: guard + m * n].view(m, n)
    gpu_gemv(fmt, _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev, y=y)
    b = buf.cpu().numpy()
    assert np.all(b[:guard] == 1234.0) and np.all(b[guard + m * n:] == 1234.0)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv(fmt, p_ref, s_ref, x, bs))


@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
def test_decode_shapes_full_size_sampled(dev, fmt):
    """Every decode-step shape at full size, quantised on the GPU; sampled output rows checked
    one by one against the oracle (which quantises those rows itself)."""
    bs = BS[fmt]
    rng = np.random.default_rng(8)
    for name, n, k, _ in synth.DECODE_SHAPES:
        w = synth.weights(synth.weight_seed(0 if name != "lm_head" else 28, name), n, k)
        x = synth.activations(synth.x_seed(0, synth.X_SLOT[name], 1), 1, k)
        packed, sc = gpu_quantize(fmt, w, bs, dev)
        y = gpu_gemv(fmt, packed, sc, x, n, k, bs, dev).cpu().numpy()
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 64)]))
        p_ref, s_ref = oracle_quantize(fmt, w[rows], bs)
        assert np.array_equal(packed.cpu().numpy()[rows], p_ref)
        y_ref = oracle_gemv(fmt, p_ref, s_ref, x, bs)
        err = y[0, rows].astype(np.float64) - y_ref[0]
        # per-element bound of the criteria (the RMS over the sampled rows)
        rms = np.sqrt(np.mean(y_ref[0] ** 2))
        assert np.max(np.abs(err)) <= MAX_ABS_RMS * rms, name
        assert np.linalg.norm(err) <= REL_L2 * np.linalg.norm(y_ref[0]), name


def test_timeout_is_reported_and_context_survives(dev):
    """A producer that issues nothing (host-set test hook) makes every bounded wait run out after
    about a second; the kernel returns, the host reads W4_ERR_TIMEOUT, and the next GEMV is right."""
    n, k, bs = 64, 1536, 64
    w = synth.weights(9000, n, k)
    x = synth.activations(9001, 1, k)
    p_ref, s_ref = oracle_quantize("nf4", w, bs)
    packed, sc = _t(p_ref, dev), _t(s_ref, dev)
    assert w4.w4_device_check() == 0
    w4.w4_inject_timeout_once()
    gpu_gemv("nf4", packed, sc, x, n, k, bs, dev)
    assert w4.w4_device_check() == w4._lib.W4_ERR_TIMEOUT
    assert w4.w4_device_check() == 0                      # cleared after reading
    y = gpu_gemv("nf4", packed, sc, x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv("nf4", p_ref, s_ref, x, bs))


@pytest.mark.parametrize("n,k", [(1024, 1536), (8960, 1536)])
def test_tensor_core_timeout_is_reported_and_context_survives(dev, n, k):
    """The same host-set hook on the tcgen05 kernel (batch 32): its packed producer issues no
    copies, so the decoders', scale warps', MMA issuer's and epilogue's bounded waits run out; the
    kernel still waits for the x copies it issued, frees its tensor memory and returns.  The host
    reads W4_ERR_TIMEOUT from the tensor-core kernel's own error word, and the next call matches
    the oracle.  (1024 rows: split-K over a thread-block cluster; 8960 rows: no split.)"""
    bs, m = 64, 32
    st, plan = w4.w4_gemv_plan(w4._lib.W4_FMT_NF4, m, n, k, bs)
    assert st == 0 and plan["kernel"] == w4.W4_KERNEL_TCGEN05
    w = synth.weights(9100 + n, n, k)
    x = synth.activations(9101 + n, m, k)
    p_ref, s_ref = oracle_quantize("nf4", w, bs)
    packed, sc = _t(p_ref, dev), _t(s_ref, dev)
    assert w4.w4_device_check() == 0
    w4.w4_inject_timeout_once()
    gpu_gemv("nf4", packed, sc, x, n, k, bs, dev)
    assert w4.w4_device_check() == w4._lib.W4_ERR_TIMEOUT
    assert w4.w4_device_check() == 0
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n).integers(0, n, 64)]))
    y = gpu_gemv("nf4", packed, sc, x, n, k, bs, dev).cpu().numpy()
    assert_gemv_close(y[:, rows], oracle_gemv("nf4", p_ref, s_ref, x, bs, rows=rows))


# ----------------------------------------------------------------------------- precision conditions
@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
@pytest.mark.parametrize("m", [1, 8])
def test_small_batch_small_magnitude_blocks(dev, fmt, m):
    """Batches 1 ... 8 carry the block scale in FP32 (NF4) or as the stored FP16 scale, applied to
    the FP32 partial sums: blocks far below the FP16 normal range (absmax about 5e-6) still meet the
    bar.  x is scaled by 64 (exact in FP16) so that y stays in the FP16 normal range."""
    bs = BS[fmt]
    n, k = 300, 1536
    w = (synth.weights(9100 + m, n, k) * np.float32(1e-4)).astype(np.float32)
    x = (synth.activations(9101 + m, m, k).astype(np.float32) * 64).astype(np.float16)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    if fmt == "nf4":
        assert float(s_ref.max()) < 6.1e-5                      # every block below the FP16 normal range
    y = gpu_gemv(fmt, _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv(fmt, p_ref, s_ref, x, bs))


@pytest.mark.parametrize("m", [16, 64])
def test_tensor_core_nf4_absmax_at_the_low_end_of_the_stated_range(dev, m):
    """The tcgen05 path rounds the NF4 absmax to FP16: blocks with absmax just above the FP16 normal
    minimum (6.1e-5) meet the bar."""
    n, k, bs = 640, 1536, 64
    w = (synth.weights(9200 + m, n, k) * np.float32(4e-3)).astype(np.float32)
    x = (synth.activations(9201 + m, m, k).astype(np.float32) * 16).astype(np.float16)
    p_ref, s_ref = oracle_quantize("nf4", w, bs)
    assert float(s_ref.min()) >= 6.1e-5 and float(s_ref.max()) < 1e-3
    st, plan = w4.w4_gemv_plan(w4.W4_FMT_NF4, m, n, k, bs, 152)
    assert st == 0 and plan["kernel"] == w4.W4_KERNEL_TCGEN05
    y = gpu_gemv("nf4", _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv("nf4", p_ref, s_ref, x, bs))


@pytest.mark.parametrize("fmt", ["nf4", "int4", "fp4"])
@pytest.mark.parametrize("m", [1, 8, 16, 64])
def test_activation_outliers_at_100_sigma(dev, fmt, m):
    """0.1 % of the activations at +-100 (100 sigma of the N(0, 1) draws), the rest ordinary: every
    path (small-batch kernel, tcgen05) meets the bar."""
    bs = BS[fmt]
    n, k = 512, 1536
    w = synth.weights(9300 + m, n, k, outlier_frac=0.001)
    x = synth.activations(9301 + m, m, k).astype(np.float32)
    rng = np.random.default_rng(9302 + m)
    idx = rng.choice(m * k, size=max(1, round(0.001 * m * k)), replace=False)
    x.ravel()[idx] = np.where(rng.random(len(idx)) < 0.5, -100.0, 100.0)
    x = x.astype(np.float16)
    p_ref, s_ref = oracle_quantize(fmt, w, bs)
    y = gpu_gemv(fmt, _t(p_ref, dev), _t(s_ref, dev), x, n, k, bs, dev)
    assert_gemv_close(y.cpu().numpy(), oracle_gemv(fmt, p_ref, s_ref, x, bs))
