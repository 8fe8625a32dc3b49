"""The C ABI on the host: the library loads without a GPU, exports every symbol include/w4.h
declares, validates arguments before touching CUDA, and its host-side code book matches the
oracle's construction bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import weight_only_bit_gb300 as w4
from weight_only_bit_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "w4.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(_lib.SYMBOLS) == _declared()


def test_every_declared_symbol_is_exported(libw4):
    for name in _declared():
        assert hasattr(libw4, name), name


def test_codebook_matches_oracle_bit_for_bit(libw4):
    st, c = w4.w4_nf4_codebook()
    assert st == w4.W4_OK if hasattr(w4, "W4_OK") else st == 0
    lib_c = np.array(c, dtype=np.float32)
    assert np.array_equal(lib_c.view(np.uint32), oracle.nf4_codebook().view(np.uint32))
    assert libw4.w4_nf4_codebook(None) == _lib.W4_ERR_NULL


# fake, never dereferenced device addresses (validation returns before any CUDA call)
A = 1 << 20


def test_gemv_validation(libw4):
    g = libw4.w4_gemv_nf4
    ok = (A, A, A, A, A)
    assert g(None, A, A, A, A, 1, 256, 1536, 64, None) == _lib.W4_ERR_NULL
    assert g(A, A, None, A, A, 1, 256, 1536, 64, None) == _lib.W4_ERR_NULL          # NF4 needs a code book
    assert g(*ok, 1, 256, 1536, 48, None) == _lib.W4_ERR_BLOCKSIZE                  # not a power of two
    assert g(*ok, 1, 256, 1536, 16, None) == _lib.W4_ERR_BLOCKSIZE                  # below 32
    assert g(*ok, 1, 256, 1536, 512, None) == _lib.W4_ERR_BLOCKSIZE                 # above 256
    assert g(*ok, 1, 256, 1568, 64, None) == _lib.W4_ERR_SHAPE                      # K % bs != 0
    assert g(*ok, 0, 256, 1536, 64, None) == _lib.W4_ERR_SHAPE                      # empty batch
    assert g(*ok, 1, 0, 1536, 64, None) == _lib.W4_ERR_SHAPE                        # empty output
    assert g(*ok, 4097, 256, 1536, 64, None) == _lib.W4_ERR_UNSUPPORTED             # beyond the batch limit
    assert g(*ok, 1, 256, _lib.W4_MAX_K + 64, 64, None) == _lib.W4_ERR_UNSUPPORTED  # beyond the K limit
    assert g(A + 8, A, A, A, A, 1, 256, 1536, 64, None) == _lib.W4_ERR_ALIGN          # packed
    assert g(A, A + 4, A, A, A, 1, 256, 1536, 64, None) == _lib.W4_ERR_ALIGN          # absmax
    assert g(A, A, A, A + 2, A, 1, 256, 1536, 64, None) == _lib.W4_ERR_ALIGN          # x
    assert g(A, A, A, A, A + 1, 1, 256, 1536, 64, None) == _lib.W4_ERR_ALIGN          # y (2-byte rule)
    gi = libw4.w4_gemv_int4
    assert gi(A, None, A, A, 1, 256, 1536, 128, None) == _lib.W4_ERR_NULL
    assert gi(A, A, A, A, 1, 256, 1536, 96, None) == _lib.W4_ERR_BLOCKSIZE


def test_quantize_and_dequantize_validation(libw4):
    assert libw4.w4_quantize_nf4(None, A, A, A, 4, 64, 64, None) == _lib.W4_ERR_NULL
    assert libw4.w4_quantize_nf4(A, A, A, A, 4, 100, 64, None) == _lib.W4_ERR_SHAPE
    assert libw4.w4_quantize_nf4(A + 4, A, A, A, 4, 64, 64, None) == _lib.W4_ERR_ALIGN
    assert libw4.w4_quantize_int4(A, A, A, 4, 128, 100, None) == _lib.W4_ERR_BLOCKSIZE
    assert libw4.w4_dequantize_nf4(A, A, A, None, 4, 64, 64, None) == _lib.W4_ERR_NULL
    assert libw4.w4_dequantize_int4(A, A, A + 4, 4, 128, 128, None) == _lib.W4_ERR_ALIGN


def test_sequence_and_step_validation(libw4):
    d = (_lib.GemvDesc * 2)()
    d[0] = _lib.GemvDesc(_lib.W4_FMT_NF4, A, A, A, A, A, 1, 256, 1536, 64, 0)
    d[1] = _lib.GemvDesc(_lib.W4_FMT_INT4, A, A, 0, A, A, 1, 256, 1536, 100, 1)   # bad group
    assert libw4.w4_gemv_sequence(d, 2, None) == _lib.W4_ERR_BLOCKSIZE            # nothing enqueued
    assert libw4.w4_gemv_sequence(None, 2, None) == _lib.W4_ERR_NULL
    h = ctypes.c_void_p()
    assert libw4.w4_step_create(d, 2, A, ctypes.byref(h)) == _lib.W4_ERR_BLOCKSIZE and h.value is None
    d[1] = _lib.GemvDesc(_lib.W4_FMT_NF4, A, A, A, A, A, 1, 256, 1536, 64, 2)      # level jumps by 2
    assert libw4.w4_gemv_sequence(d, 2, None) == _lib.W4_ERR_SHAPE
    d[1].level = 0
    d[0].level = 1                                                                # first level must be 0
    assert libw4.w4_gemv_sequence(d, 2, None) == _lib.W4_ERR_SHAPE
    d[0].level = 0
    assert libw4.w4_step_create(d, 2, None, ctypes.byref(h)) == _lib.W4_ERR_NULL    # persistent needs workspace
    assert libw4.w4_step_create(d, 2, A + 4, ctypes.byref(h)) == _lib.W4_ERR_ALIGN
    assert libw4.w4_step_workspace_bytes(197) >= 4 * 198 and libw4.w4_step_workspace_bytes(0) == 0
    assert libw4.w4_step_launch(None, None) == _lib.W4_ERR_NULL
    assert libw4.w4_step_destroy(None) == _lib.W4_ERR_NULL
    d[0].format = 7
    assert libw4.w4_gemv_sequence(d, 1, None) == _lib.W4_ERR_UNSUPPORTED


def test_status_strings(libw4):
    for code in range(-8, 1):
        assert libw4.w4_status_str(code)
    assert w4.w4_status_str(_lib.W4_ERR_ALIGN) != w4.w4_status_str(_lib.W4_ERR_SHAPE)
    with pytest.raises(w4.W4Error):
        w4.check(_lib.W4_ERR_SHAPE, "shape")


# ---------------------------------------------------------------- dispatch and launch geometry
# w4_gemv_plan is the host half of w4_gemv_nf4 / w4_gemv_int4's dispatch (the same functions
# size the real launches), so these checks pin the batch-driven path choice and the tcgen05
# kernel's resource use without a GPU.  152 SMs: a GB300.

SMS = 152
DECODE = {"q": (1536, 1536), "k": (256, 1536), "gate": (8960, 1536), "down": (1536, 8960), "lm_head": (151936, 1536)}


def _plan(fmt, m, n, k, bs, sms=SMS):
    st, p = w4.w4_gemv_plan(fmt, m, n, k, bs, sms)
    assert st == w4.W4_OK, (fmt, m, n, k, bs, st)
    return p


@pytest.mark.parametrize("fmt,bs", [(w4.W4_FMT_NF4, 64), (w4.W4_FMT_INT4, 128), (w4.W4_FMT_FP4, 32)])
def test_plan_batches_up_to_8_stay_on_the_small_batch_kernel(libw4, fmt, bs):
    for m in range(1, 9):
        for n, k in DECODE.values():
            p = _plan(fmt, m, n, k, bs)
            assert p["kernel"] == w4.W4_KERNEL_SMALL_BATCH and p["launches"] == 1 and p["batch_tile"] == m
            assert p["cluster"] == 1 and p["smem_bytes"] <= 227 * 1024 and p["stages"] >= 2


@pytest.mark.parametrize("fmt,bs", [(w4.W4_FMT_NF4, 64), (w4.W4_FMT_INT4, 128), (w4.W4_FMT_FP4, 32)])
def test_plan_batch_1_every_k_fits(libw4, fmt, bs):
    # batch 1 takes the 64 KB byte-pair table with the partial sums in its gaps wherever the ring
    # keeps its stage budget: every K up to the limit must still give a launch within the shared
    # memory of one CTA, with at least two ring stages, and the decode shapes must get the table
    # (more than 64 KB of shared memory beside their ring stages)
    for k in range(max(bs, 64), w4.W4_MAX_K + 1, 64):
        if k % bs:
            continue
        for n in (1, 300, 40000, 151936):
            p = _plan(fmt, 1, n, k, bs)
            assert p["kernel"] == w4.W4_KERNEL_SMALL_BATCH and p["launches"] == 1
            assert p["smem_bytes"] <= 227 * 1024 and p["stages"] >= 2, (k, n, p)
    for n, k in DECODE.values():
        assert _plan(fmt, 1, n, k, bs)["smem_bytes"] > 64 * 1024 + 2 * 8 * 1024


@pytest.mark.parametrize("fmt,bs", [(w4.W4_FMT_NF4, 64), (w4.W4_FMT_INT4, 128), (w4.W4_FMT_NF4, 32),
                                    (w4.W4_FMT_INT4, 256), (w4.W4_FMT_FP4, 32)])
def test_plan_tcgen05_resources(libw4, fmt, bs):
    for m in list(range(9, 129, 7)) + [16, 17, 32, 33, 64, 65, 128]:
        for n, k in list(DECODE.values()) + [(1, 256), (129, 64), (300, 320), (70, 8960)]:
            if k % bs:
                continue
            p = _plan(fmt, m, n, k, bs)
            assert p["kernel"] == w4.W4_KERNEL_TCGEN05
            nb = p["batch_tile"]
            assert nb in (16, 32, 64, 128) and nb >= m and (nb == 16 or nb // 2 < m)
            assert p["threads"] == 864 and p["launches"] == 1
            assert p["smem_bytes"] <= 227 * 1024 and 4 <= p["stages"] <= 8
            # tensor memory: two accumulators of max(32, NB) columns, then 32 columns per A stage
            assert 2 * max(32, nb) <= 256 and 256 + 32 * p["stages"] <= 512
            nrb = -(-n // 128)
            if p["cluster"] > 1:
                assert p["cluster"] <= 8 and p["cluster"] <= -(-k // 256)
                assert p["grid"] == nrb * p["cluster"] <= SMS and 2 * nrb <= SMS
                # the FP32 partial tile [128][NB + 4] fits in the x stages (NB x 128 bytes each)
                assert 128 * (nb + 4) * 4 <= p["stages"] * nb * 128
            else:
                assert p["grid"] == min(nrb, SMS)


@pytest.mark.parametrize("fmt,bs", [(w4.W4_FMT_NF4, 64), (w4.W4_FMT_INT4, 128), (w4.W4_FMT_FP4, 32)])
def test_plan_prefill_batch_tiles(libw4, fmt, bs):
    """Above 128 rows: tiles of 256 batch rows (one 256-column accumulator, the weights decoded once
    per 256 rows) where the weight matrix has enough 128-row tiles for the SMs, else tiles of 128."""
    n, k = DECODE["lm_head"]
    for m in (129, 200, 256):
        p = _plan(fmt, m, n, k, bs)
        assert p["kernel"] == w4.W4_KERNEL_TCGEN05 and p["batch_tile"] == 256 and p["launches"] == 1
        assert p["cluster"] == 1 and p["grid"] == SMS and p["smem_bytes"] <= 227 * 1024
        # tensor memory: one accumulator of 256 columns, then 32 columns per A stage
        assert p["stages"] >= 4 and 256 + 32 * p["stages"] <= 512
    p = _plan(fmt, 512, n, k, bs)
    assert p["batch_tile"] == 256 and p["launches"] == 2
    p = _plan(fmt, 300, n, k, bs)
    assert p["batch_tile"] == 256 and p["launches"] == 2          # 256 + 44
    # a short weight matrix keeps 128-row batch tiles (its row tiles alone would leave SMs idle)
    p = _plan(fmt, 256, *DECODE["q"], bs)
    assert p["batch_tile"] == 128 and p["launches"] == 2


def test_plan_split_choices_on_the_decode_shapes(libw4):
    nf4 = w4.W4_FMT_NF4
    # few row tiles and enough K: split over a cluster sized to cover the SMs
    assert _plan(nf4, 32, *DECODE["q"], 64)["cluster"] == 6           # 12 tiles x 6 super-chunks
    assert _plan(nf4, 32, *DECODE["q"], 64)["grid"] == 72
    assert _plan(nf4, 16, *DECODE["k"], 64)["cluster"] == 6           # 2 tiles
    assert _plan(nf4, 32, *DECODE["down"], 64)["cluster"] == 8        # 35 super-chunks, 8 at most
    assert _plan(nf4, 128, *DECODE["down"], 64)["cluster"] == 8
    # the split does not pay: gate at batch >= 32 (70 tiles, 2-way split), q at batch 128
    assert _plan(nf4, 32, *DECODE["gate"], 64)["cluster"] == 1
    assert _plan(nf4, 128, *DECODE["gate"], 64)["cluster"] == 1
    assert _plan(nf4, 128, *DECODE["q"], 64)["cluster"] == 1
    # many row tiles: persistent, one CTA per SM
    p = _plan(nf4, 32, *DECODE["lm_head"], 64)
    assert p["cluster"] == 1 and p["grid"] == SMS
    # a one-super-chunk K cannot be split
    assert _plan(nf4, 32, 128, 256, 64)["cluster"] == 1
    # fewer SMs: smaller clusters, never more CTAs than SMs
    p = _plan(nf4, 32, *DECODE["q"], 64, sms=36)
    assert p["cluster"] == 3 and p["grid"] == 36


def test_plan_shapes_the_tensor_cores_do_not_take(libw4):
    # K not a multiple of 64: CUDA-core launches of at most 8 batch rows
    p = _plan(w4.W4_FMT_NF4, 40, 100, 96, 32)
    assert p["kernel"] == w4.W4_KERNEL_SMALL_BATCH and p["launches"] == 5 and p["batch_tile"] == 8
    p = _plan(w4.W4_FMT_INT4, 20, 100, 160, 32)
    assert p["kernel"] == w4.W4_KERNEL_SMALL_BATCH and p["launches"] == 3


def test_plan_validation(libw4):
    out = w4.GemvPlan()
    ref = ctypes.byref(out)
    assert libw4.w4_gemv_plan(0, 1, 16, 64, 64, SMS, None) == w4.W4_ERR_NULL
    assert libw4.w4_gemv_plan(3, 1, 16, 64, 64, SMS, ref) == w4.W4_ERR_UNSUPPORTED
    assert libw4.w4_gemv_plan(w4.W4_FMT_FP4, 1, 16, 64, 32, SMS, ref) == w4.W4_OK
    assert libw4.w4_gemv_plan(0, 0, 16, 64, 64, SMS, ref) == w4.W4_ERR_SHAPE
    assert libw4.w4_gemv_plan(0, 4097, 16, 64, 64, SMS, ref) == w4.W4_ERR_UNSUPPORTED
    assert libw4.w4_gemv_plan(0, 1, 0, 64, 64, SMS, ref) == w4.W4_ERR_SHAPE
    assert libw4.w4_gemv_plan(0, 1, 16, 96, 64, SMS, ref) == w4.W4_ERR_SHAPE
    assert libw4.w4_gemv_plan(0, 1, 16, 96, 48, SMS, ref) == w4.W4_ERR_BLOCKSIZE
    assert libw4.w4_gemv_plan(0, 1, 16, 64, 64, 0, ref) == w4.W4_ERR_SHAPE
    assert libw4.w4_gemv_plan(0, 1, 16, w4.W4_MAX_K + 64, 64, SMS, ref) == w4.W4_ERR_UNSUPPORTED


def test_plan_prefill_batches_run_as_128_row_tiles(libw4):
    nf4 = w4.W4_FMT_NF4
    p = _plan(nf4, 300, *DECODE["gate"], 64)
    assert p["kernel"] == w4.W4_KERNEL_TCGEN05 and p["batch_tile"] == 128 and p["launches"] == 3
    assert _plan(nf4, 256, *DECODE["q"], 64)["launches"] == 2
    assert _plan(nf4, 4096, *DECODE["q"], 64)["launches"] == 32
    # a remainder of 8 rows or fewer goes to the CUDA cores: one more launch
    assert _plan(nf4, 130, *DECODE["q"], 64)["launches"] == 2
    # K not a multiple of 64: CUDA-core launches of 8 rows throughout
    assert _plan(nf4, 300, 100, 96, 32)["launches"] == 38


def test_step_run_host_validates_on_the_host(libw4):
    """w4_step_run_host rejects a missing step, missing buffers of a non-empty copy and negative
    sizes before any CUDA call (no GPU needed)."""
    L = libw4
    assert L.w4_step_run_host(None, None, None, 0, None, None, 0, None) == w4.W4_ERR_NULL
    fake = ctypes.c_void_p(0)
    assert L.w4_step_run_host(fake, None, None, 0, None, None, 0, None) == w4.W4_ERR_NULL   # no graph
