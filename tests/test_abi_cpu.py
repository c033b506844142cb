"""The C ABI without a GPU: the library builds, loads, exports every symbol the
headers declare, and rejects bad arguments on the host before any CUDA call."""
import ctypes as C
import os
import re

import pytest

from qwen3_prefill_kv_gb300 import build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(qdec_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    bound = {s[0] for s in _lib.SIGNATURES}
    assert set(names) == bound, f"binding and headers disagree: {set(names) ^ bound}"


def test_strerror_and_status_codes(lib):
    assert lib.qdec_strerror(0) == b"ok"
    for code in range(-7, 0):
        assert lib.qdec_strerror(code) not in (b"", b"unknown status")


def _cfg(**kw):
    base = dict(hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32, ffn=384, vocab=1024,
                rope_theta=1e6, rms_eps=1e-6, max_seq=64)
    base.update(kw)
    return _lib.QdecConfig(*[base[k] for k, _ in _lib.QdecConfig._fields_])


def _create(lib, cfg, weights=True):
    w = _lib.QdecWeights()
    h = C.c_void_p()
    return lib.qdec_create(C.byref(cfg), C.byref(w) if weights else None, None, C.byref(h))


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=48), -7), (dict(n_q_heads=6, n_kv_heads=4), -7), (dict(hidden=100), -7),
    (dict(n_q_heads=24, n_kv_heads=2), -7), (dict(vocab=0), -1), (dict(max_seq=0), -1),
    (dict(rms_eps=0.0), -1),
])
def test_create_rejects_bad_shapes_on_host(lib, kw, code):
    assert _create(lib, _cfg(**kw)) == code
    assert lib.qdec_last_error()


def test_create_rejects_null_weights(lib):
    assert _create(lib, _cfg()) == -1          # weight pointers are NULL
    assert _create(lib, _cfg(), weights=False) == -1


def test_null_context_calls(lib):
    assert lib.qdec_position(None) == -1
    assert lib.qdec_decode_step(None, 0, None, None) == -1
    assert lib.qdec_prefill(None, None, 1, None, 0, 0, None, None) == -1
    assert lib.qdec_read_kv(None, 0, 0, 0, 1, None) == -1
    assert lib.qdec_sync(None) == -1
    lib.qdec_destroy(None)
    h = C.c_void_p()
    assert lib.qdec_clone(None, C.byref(h)) == -1
    assert lib.qdec_decode_step_batch(None, 0, None, None, None) == -1


def test_op_entry_points_validate_on_host(lib):
    assert lib.qdec_op_gemm(None, 64, None, 1, 1, 64, 0, 0, None, 1, 0, None) == -1
    assert lib.qdec_op_attention_prefill(None, 1, 4, 2, 32, 8, 0, None, None, None, 0, None) == -1
    assert lib.qdec_op_lm_head_scratch_bytes(1024) > 16
    assert lib.qdec_op_lm_head_argmax(None, 1024, 128, None, None, 1e-6, None, None, None, 0, None) == -1


def test_gemm_tile_width_setting_without_a_gpu(lib):
    """qdec_op_gemm_tile_width only sets the process-wide choice: 0, 128 and 256 are taken
    and the previous value returned; anything else is INVALID_ARG and changes nothing."""
    assert lib.qdec_op_gemm_tile_width(256) == 0
    assert lib.qdec_op_gemm_tile_width(128) == 256
    assert lib.qdec_op_gemm_tile_width(192) == -1
    assert lib.qdec_op_gemm_tile_width(0) == 128
    assert lib.qdec_op_gemm_tile_width(0) == 0


def test_fake_token_len_through_the_abi(lib):
    """The adaptor's row count on the host, against the oracle's definition and the page's
    worked example (183 frames -> 23 rows)."""
    import oracle
    assert _lib.fake_token_len(183) == 23
    for n in list(range(1, 70)) + [390, 1000, 3120, 4095]:
        assert _lib.fake_token_len(n) == oracle.fake_token_len(n), n
    assert _lib.fake_token_len(0) == 0


def test_adaptor_create_rejects_bad_arguments_on_host(lib):
    h = C.c_void_p()
    w = _lib.QdecAdaptorWeights()
    cfg = _lib.QdecAdaptorConfig(512, 2048, 1024, 8, 256, 2, 1e-12)
    assert lib.qdec_adaptor_create(None, C.byref(w), None, C.byref(h)) == -1
    assert lib.qdec_adaptor_create(C.byref(cfg), C.byref(w), None, C.byref(h)) == -1   # null weights
    bad = _lib.QdecAdaptorConfig(512, 2048, 1000, 8, 256, 2, 1e-12)                     # head_dim 125
    assert lib.qdec_adaptor_create(C.byref(bad), C.byref(w), None, C.byref(h)) == -7
    zero = _lib.QdecAdaptorConfig(512, 2048, 1024, 8, 256, 2, 0.0)
    assert lib.qdec_adaptor_create(C.byref(zero), C.byref(w), None, C.byref(h)) == -1
    assert lib.qdec_adaptor_run(None, None, 1, None, None) == -1
