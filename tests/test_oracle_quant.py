"""Pins of the block-quantization oracle (oracle/quant.py): the library's own q8b32 and
q4b32 formats (the audio.cpp plan's Task 8 names Q8_0 / Q4_K_M packages without defining
them), against the error bound of round-to-nearest, exact codes for representable blocks,
the zero block, nibble packing and the storage arithmetic."""
import numpy as np
import pytest

from oracle import quant as Q


@pytest.mark.parametrize("fmt", ["q8b32", "q4b32"])
def test_round_trip_error_is_within_half_a_step(fmt):
    rng = np.random.default_rng(0)
    w = rng.normal(size=(16, 256)) * 0.02
    q, d = Q.quantize(w, fmt)
    back = Q.dequantize(q, d)
    step = np.repeat(d.astype(np.float64), 32, axis=1)
    # half a step from rounding, plus the fp16 rounding of the scale scaled by |q| <= qmax
    bound = 0.5 * step + Q.QMAX[fmt] * step * 2.0 ** -10
    assert np.all(np.abs(back - w) <= bound + 1e-18)
    assert q.min() >= -Q.QMAX[fmt] and q.max() <= Q.QMAX[fmt]
    # the largest magnitude of each block maps to +-qmax
    blocks = np.abs(w).reshape(16, 8, 32)
    qb = np.abs(q.astype(np.int64)).reshape(16, 8, 32)
    np.testing.assert_array_equal(qb[np.arange(16)[:, None], np.arange(8)[None, :], blocks.argmax(axis=2)],
                                  Q.QMAX[fmt])


def test_representable_block_is_exact_and_zero_block_is_zero():
    d = np.float16(0.0078125)   # 2^-7, exact in fp16
    codes = np.arange(-127, 128, dtype=np.float64)[:32]
    codes[5] = 127.0            # max |code| = 127 so the block's scale is exactly d
    w = np.stack([codes * float(d), np.zeros(32)])
    q, s = Q.quantize(w, "q8b32")
    np.testing.assert_array_equal(q[0], codes.astype(np.int8))
    assert s[0, 0] == d and s[1, 0] == 0
    np.testing.assert_array_equal(q[1], 0)
    np.testing.assert_array_equal(Q.dequantize(q, s), w)


def test_q4_nibble_packing_round_trip_and_order():
    rng = np.random.default_rng(1)
    codes = rng.integers(-7, 8, size=(3, 64)).astype(np.int8)
    packed = Q.pack_q4(codes)
    assert packed.shape == (3, 32) and packed.dtype == np.uint8
    np.testing.assert_array_equal(Q.unpack_q4(packed), codes)
    assert Q.pack_q4(np.array([[-7, 7]], dtype=np.int8))[0, 0] == (1 | (15 << 4))   # lower nibble first


def test_storage_arithmetic():
    assert Q.bytes_per_weight("q8b32") == 34 / 32
    assert Q.bytes_per_weight("q4b32") == 18 / 32
    # the 0.6B decoder's 596M weights: bf16 1.19 GB -> q8b32 0.63 GB, q4b32 0.34 GB
    from qwen3_prefill_kv_gb300 import synth
    n = synth.QWEN3_06B.weight_params()
    assert n == 596_049_920
    assert abs(n * 2 / (n * Q.bytes_per_weight("q8b32")) - 1.88) < 0.01
    assert abs(n * 2 / (n * Q.bytes_per_weight("q4b32")) - 3.56) < 0.01
