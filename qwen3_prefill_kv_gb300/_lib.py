"""ctypes binding of the qdec C ABI (include/qdec.h, include/qdec_ops.h).

Argument marshalling only: every step of the decoder runs in the CUDA library.
There is no CPU fallback: if libqdec.so is missing, loading raises.
PyTorch tensors are accepted for buffers (their data_ptr is passed through).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqdec.so")

QDEC_OK = 0
STATUS = {-1: "INVALID_ARG", -2: "CAPACITY", -3: "STATE", -4: "CUDA", -5: "OOM", -6: "TIMEOUT",
          -7: "UNSUPPORTED"}

GEMM_STORE_F32, GEMM_ADD_F32, GEMM_SWIGLU_BF16, GEMM_STORE_BF16, GEMM_ATOMIC_F32 = 0, 1, 2, 3, 4
OPT_DECODE_KERNEL = 1
OPT_TRACE = 2
OPT_PREFILL_IMPL = 3
OPT_ATTN_UNIT_KEYS = 4
OPT_SPIN_LIMIT = 5
OPT_SHARED_PREFIX = 7
OPT_WEIGHTS = 8
WEIGHTS_BF16, WEIGHTS_Q8B32, WEIGHTS_Q4B32 = 0, 1, 2
PREFILL_TCGEN05, PREFILL_SIMT = 0, 1
DECODE_PERSISTENT, DECODE_GRAPH = 0, 1
IMPL_SIMT, IMPL_TCGEN05 = 0, 1


class QdecError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class QdecConfig(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_layers", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("rope_theta", C.c_float), ("rms_eps", C.c_float),
                ("max_seq", C.c_int32)]


_PP = C.POINTER(C.c_void_p)


class QdecWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("wqkv", _PP), ("wo", _PP),
                ("wgu", _PP), ("wd", _PP), ("g_in", _PP), ("g_post", _PP), ("g_q", _PP), ("g_k", _PP)]


_lib = None

# Every symbol include/qdec.h, include/qdec_ops.h and include/qdec_adaptor.h declare:
# (name, restype, argtypes).
_VP, _I32, _F, _SZ = C.c_void_p, C.c_int32, C.c_float, C.c_size_t
SIGNATURES = [
    ("qdec_create", C.c_int, [C.POINTER(QdecConfig), C.POINTER(QdecWeights), _VP, C.POINTER(_VP)]),
    ("qdec_prefill", C.c_int, [_VP, _VP, _I32, _VP, _I32, _I32, _VP, _VP]),
    ("qdec_decode_step", C.c_int, [_VP, _I32, _VP, _VP]),
    ("qdec_decode_step_batch", C.c_int, [_VP, _I32, _VP, _VP, _VP]),
    ("qdec_clone", C.c_int, [_VP, C.POINTER(_VP)]),
    ("qdec_position", C.c_int, [_VP]),
    ("qdec_read_kv", C.c_int, [_VP, _I32, _I32, _I32, _I32, _VP]),
    ("qdec_read_history", C.c_int, [_VP, _VP, _I32]),
    ("qdec_sync", C.c_int, [_VP]),
    ("qdec_set_option", C.c_int, [_VP, _I32, _I32]),
    ("qdec_get_option", C.c_int, [_VP, _I32]),
    ("qdec_read_trace", C.c_int, [_VP, _VP, _I32]),
    ("qdec_destroy", None, [_VP]),
    ("qdec_strerror", C.c_char_p, [C.c_int]),
    ("qdec_last_error", C.c_char_p, []),
    ("qdec_kernel_launches", C.c_uint64, []),
    ("qdec_op_gemm", C.c_int, [_VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32, _VP, _I32, _I32, _VP]),
    ("qdec_op_device_error", C.c_int, []),
    ("qdec_op_gemm_tile_width", C.c_int, [C.c_int32]),
    ("qdec_op_gemm_tile_rows", C.c_int, [C.c_int32]),
    ("qdec_op_programmatic_launch", C.c_int, [C.c_int32]),
    ("qdec_op_sample", C.c_int, [_VP, _I32, _VP, _I32, _F, _I32, _F, _F, C.c_uint64, _I32, _VP, _VP]),
    ("qdec_set_sampling", C.c_int, [_VP, _F, _I32, _F, _F, C.c_uint64]),
    ("qdec_op_gemm_splitk", C.c_int, [_VP, _I32, _VP, _I32, _I32, _I32, _I32, _VP, _I32, _VP]),
    ("qdec_op_attention_prefill", C.c_int, [_VP, _I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _I32, _VP]),
    ("qdec_op_lm_head_scratch_bytes", _SZ, [_I32]),
    ("qdec_op_lm_head_argmax", C.c_int, [_VP, _I32, _I32, _VP, _VP, _F, _VP, _VP, _VP, _SZ, _VP]),
    ("qdec_op_lm_head_argmax_static", C.c_int, [_VP, _I32, _I32, _VP, _VP, _F, _VP, _VP, _VP]),
    ("qdec_op_quantize", C.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _VP]),
    ("qdec_op_gemv_q", C.c_int, [_VP, _VP, _I32, _I32, _I32, _VP, _VP, _F, _I32, _I32, _VP, _VP]),
    ("qdec_fake_token_len", C.c_int32, [_I32]),
    ("qdec_adaptor_create", C.c_int, [_VP, _VP, _VP, C.POINTER(_VP)]),
    ("qdec_adaptor_run", C.c_int, [_VP, _VP, _I32, _VP, _VP]),
    ("qdec_adaptor_destroy", None, [_VP]),
]

LM_HEAD_STATIC_MAX_VOCAB = 262144


def load(path: str = LIB_PATH):
    """Loads libqdec.so (built by ``qwen3_prefill_kv_gb300.build``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m qwen3_prefill_kv_gb300.build` "
                          "(the decoder has no CPU fallback)")
    lib = C.CDLL(path)
    for name, res, args in SIGNATURES:
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != QDEC_OK:
        raise QdecError(rc, (_lib.qdec_last_error() or b"").decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Decoder:
    """One decoding context (KV cache + state) over borrowed device weights.

    ``weights`` is a ``synth.Weights`` (or any object with the same fields)
    whose tensors live on the GPU; the object is kept alive by the Decoder."""

    def __init__(self, shape, weights, max_seq: int, stream=None, _handle=None):
        self.lib = load()
        self.shape = shape
        self.weights = weights
        self.max_seq = max_seq
        self._stream = stream
        if _handle is not None:
            self.handle = _handle
            return
        cfg = QdecConfig(shape.hidden, shape.n_layers, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                         shape.ffn, shape.vocab, shape.rope_theta, shape.rms_eps, max_seq)
        nl = shape.n_layers
        arrs = {}
        for k in ("wqkv", "wo", "wgu", "wd", "g_in", "g_post", "g_q", "g_k"):
            arrs[k] = (C.c_void_p * nl)(*[l[k].data_ptr() for l in weights.layers])
        self._arrs = arrs
        w = QdecWeights(weights.embed.data_ptr(), weights.final_norm.data_ptr(),
                        *[C.cast(arrs[k], _PP) for k in ("wqkv", "wo", "wgu", "wd", "g_in", "g_post", "g_q", "g_k")])
        h = C.c_void_p()
        _check(self.lib.qdec_create(C.byref(cfg), C.byref(w), _stream_handle(stream), C.byref(h)))
        self.handle = h

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.qdec_destroy(self.handle)
            self.handle = None

    __del__ = close

    @property
    def position(self) -> int:
        r = self.lib.qdec_position(self.handle)
        if r < 0:
            _check(r)
        return r

    def prefill(self, ids, audio=None, audio_offset: int = 0, logits=None, want_argmax: bool = True):
        ids_np = np.ascontiguousarray(np.asarray(ids if not hasattr(ids, "numpy") else ids.cpu().numpy(),
                                                 dtype=np.int32))
        n_audio = 0 if audio is None else int(audio.shape[0])
        out = np.zeros(1, dtype=np.int32)
        _check(self.lib.qdec_prefill(self.handle, _ptr(ids_np), int(ids_np.size), _ptr(audio), n_audio,
                                     int(audio_offset), _ptr(logits), _ptr(out) if want_argmax else None))
        return int(out[0]) if want_argmax else None

    def decode_step(self, token: int = -1, logits=None, want_argmax: bool = True):
        out = np.zeros(1, dtype=np.int32)
        _check(self.lib.qdec_decode_step(self.handle, int(token), _ptr(logits), _ptr(out) if want_argmax else None))
        return int(out[0]) if want_argmax else None

    def clone(self) -> "Decoder":
        h = C.c_void_p()
        _check(self.lib.qdec_clone(self.handle, C.byref(h)))
        return Decoder(self.shape, self.weights, self.max_seq, self._stream, _handle=h)

    @staticmethod
    def decode_step_batch(decoders: Sequence["Decoder"], tokens, logits=None, want_argmax: bool = True):
        n = len(decoders)
        lib = decoders[0].lib
        hs = (C.c_void_p * n)(*[d.handle.value if isinstance(d.handle, C.c_void_p) else d.handle for d in decoders])
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        out = np.zeros(n, dtype=np.int32)
        _check(lib.qdec_decode_step_batch(C.cast(hs, C.c_void_p), n, _ptr(toks), _ptr(logits),
                                          _ptr(out) if want_argmax else None))
        return out if want_argmax else None

    def read_kv(self, layer: int, kind: int, pos0: int, n_pos: int) -> np.ndarray:
        """bf16 bits (uint16) [n_kv_heads, n_pos, head_dim] of one layer's K (kind 0) or V (kind 1)."""
        out = np.zeros((self.shape.n_kv_heads, n_pos, self.shape.head_dim), dtype=np.uint16)
        _check(self.lib.qdec_read_kv(self.handle, layer, kind, pos0, n_pos, _ptr(out)))
        return out

    def read_history(self, n: Optional[int] = None) -> np.ndarray:
        n = self.position if n is None else n
        out = np.zeros(n, dtype=np.int32)
        _check(self.lib.qdec_read_history(self.handle, _ptr(out), n))
        return out

    def sync(self) -> None:
        _check(self.lib.qdec_sync(self.handle))

    def set_option(self, option: int, value: int) -> None:
        _check(self.lib.qdec_set_option(self.handle, int(option), int(value)))

    def set_sampling(self, temperature: float = 0.0, top_k: int = 0, top_p: float = 1.0,
                     repetition_penalty: float = 1.0, seed: int = 0) -> None:
        """Token choice of prefill and decode steps (qdec_set_sampling); defaults are greedy."""
        _check(self.lib.qdec_set_sampling(self.handle, float(temperature), int(top_k), float(top_p),
                                          float(repetition_penalty), int(seed) & ((1 << 64) - 1)))

    def get_option(self, option: int) -> int:
        r = self.lib.qdec_get_option(self.handle, int(option))
        if r < 0:
            _check(r)
        return r

    def set_trace(self, on: bool) -> None:
        _check(self.lib.qdec_set_option(self.handle, OPT_TRACE, 1 if on else 0))

    def read_trace(self) -> np.ndarray:
        """[grid, 11 * n_layers + 8] trace of the last persistent step (see qdec_read_trace)."""
        n = self.lib.qdec_read_trace(self.handle, None, 0)
        if n < 0:
            _check(n)
        out = np.zeros(n, dtype=np.uint64)
        r = self.lib.qdec_read_trace(self.handle, _ptr(out), n)
        if r < 0:
            _check(r)
        return out.reshape(-1, 11 * self.shape.n_layers + 8)

    @property
    def decode_kernel(self) -> int:
        r = self.lib.qdec_get_option(self.handle, OPT_DECODE_KERNEL)
        if r < 0:
            _check(r)
        return r

    @decode_kernel.setter
    def decode_kernel(self, value: int) -> None:
        _check(self.lib.qdec_set_option(self.handle, OPT_DECODE_KERNEL, int(value)))


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().qdec_kernel_launches())


# ------------------------------------------------------------------ per-kernel entry points
def gemm(A, W, M, N, K, mode, C_out, lda=None, ldc=None, up_off=0, impl=IMPL_SIMT, stream=None) -> None:
    lib = load()
    _check(lib.qdec_op_gemm(_ptr(A), lda if lda is not None else K, _ptr(W), M, N, K, mode, up_off, _ptr(C_out),
                            ldc if ldc is not None else N, impl, _stream_handle(stream)))


def gemm_splitk(A, W, M, N, K, splits, C_out, lda=None, ldc=None, stream=None) -> None:
    """C += A . W^T on the tensor cores with K split over `splits` CTAs (fp32 atomics)."""
    lib = load()
    _check(lib.qdec_op_gemm_splitk(_ptr(A), lda if lda is not None else K, _ptr(W), M, N, K, splits, _ptr(C_out),
                                   ldc if ldc is not None else N, _stream_handle(stream)))


def gemm_tile_width(bn: int) -> int:
    """Forces the tcgen05 GEMM tile width (128 or 256; 0 = per shape); returns the previous one."""
    rc = int(load().qdec_op_gemm_tile_width(int(bn)))
    _check(min(rc, 0))
    return rc


def sample(logits, V, history, temperature, top_k, top_p, repetition_penalty, seed, pos, token_out,
           stream=None) -> None:
    """qdec_op_sample: the token choice on one logits vector into token_out (device int32)."""
    n = 0 if history is None else int(history.numel())
    _check(load().qdec_op_sample(_ptr(logits), int(V), _ptr(history) if n else None, n, float(temperature),
                                 int(top_k), float(top_p), float(repetition_penalty), int(seed) & ((1 << 64) - 1),
                                 int(pos), _ptr(token_out), _stream_handle(stream)))


def gemm_tile_rows(bm: int) -> int:
    """Forces the height of the 256-wide tcgen05 GEMM tiles (128: one CTA, 256: a CTA pair;
    0 = per shape); returns the previous setting."""
    rc = int(load().qdec_op_gemm_tile_rows(int(bm)))
    _check(min(rc, 0))
    return rc


def programmatic_launch(on: int) -> int:
    """Switches programmatic dependent launch of the prefill chain (1 = on, the default);
    returns the previous setting."""
    rc = int(load().qdec_op_programmatic_launch(int(on)))
    _check(min(rc, 0))
    return rc


def device_error() -> None:
    """Raises QdecError(TIMEOUT) if a tensor-core kernel gave up on a bounded wait."""
    _check(load().qdec_op_device_error())


def attention_prefill(Q, T, HQ, HKV, D, max_seq, pos0, k_cache, v_cache, O, impl=IMPL_SIMT, stream=None) -> None:
    lib = load()
    _check(lib.qdec_op_attention_prefill(_ptr(Q), T, HQ, HKV, D, max_seq, pos0, _ptr(k_cache), _ptr(v_cache),
                                         _ptr(O), impl, _stream_handle(stream)))


def quantize(W, N, K, fmt, codes, scales, stream=None) -> None:
    """qdec_op_quantize: bf16 W [N, K] -> codes (int8 [N, K] or uint8 [N, K / 2]) and fp16 scales."""
    _check(load().qdec_op_quantize(_ptr(W), int(N), int(K), int(fmt), _ptr(codes), _ptr(scales),
                                   _stream_handle(stream)))


def gemv_q(codes, scales, fmt, rows, K, x, norm_g, eps, mode, y, up_off=0, stream=None) -> None:
    """qdec_op_gemv_q: the decode GEMV on quantized weights."""
    _check(load().qdec_op_gemv_q(_ptr(codes), _ptr(scales), int(fmt), int(rows), int(K), _ptr(x), _ptr(norm_g),
                                 float(eps), int(mode), int(up_off), _ptr(y), _stream_handle(stream)))


def lm_head_scratch_bytes(V: int) -> int:
    return int(load().qdec_op_lm_head_scratch_bytes(V))


def lm_head_argmax_static(E, V, H, x, g_final, eps, logits, argmax, stream=None) -> None:
    """The lm_head + argmax that allocates nothing (library-owned static scratch)."""
    lib = load()
    _check(lib.qdec_op_lm_head_argmax_static(_ptr(E), V, H, _ptr(x), _ptr(g_final), float(eps), _ptr(logits),
                                             _ptr(argmax), _stream_handle(stream)))


def lm_head_argmax(E, V, H, x, g_final, eps, logits, argmax, scratch, stream=None) -> None:
    lib = load()
    nbytes = scratch.numel() * scratch.element_size()
    _check(lib.qdec_op_lm_head_argmax(_ptr(E), V, H, _ptr(x), _ptr(g_final), float(eps), _ptr(logits),
                                      _ptr(argmax), _ptr(scratch), nbytes, _stream_handle(stream)))


# ------------------------------------------------------------------ audio adaptor
class QdecAdaptorConfig(C.Structure):
    _fields_ = [("enc_dim", C.c_int32), ("proj_dim", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("ffn", C.c_int32), ("n_blocks", C.c_int32), ("ln_eps", C.c_float)]


class QdecAdaptorWeights(C.Structure):
    _fields_ = [("w1", C.c_void_p), ("w2", C.c_void_p), ("b1", C.c_void_p), ("b2", C.c_void_p),
                ("ln1_g", _PP), ("ln1_b", _PP), ("ln2_g", _PP), ("ln2_b", _PP),
                ("wqkv", _PP), ("wo", _PP), ("fc1", _PP), ("fc2", _PP),
                ("bqkv", _PP), ("bo", _PP), ("fc1_b", _PP), ("fc2_b", _PP)]


def fake_token_len(n_frames: int) -> int:
    """qdec_fake_token_len: rows the adaptor keeps for n_frames encoder frames."""
    return int(load().qdec_fake_token_len(int(n_frames)))


class Adaptor:
    """The projector + bidirectional adaptor (include/qdec_adaptor.h) over borrowed device
    weights: ``weights`` maps w1, b1, w2, b2 and ``blocks`` (a list of mappings with ln1_g,
    ln1_b, wqkv, bqkv, wo, bo, ln2_g, ln2_b, fc1, fc1_b, fc2, fc2_b) to CUDA tensors (bf16
    matrices, fp32 vectors); the object keeps them alive."""

    def __init__(self, shape, weights, stream=None):
        self.lib = load()
        self.shape = shape
        self.weights = weights
        cfg = QdecAdaptorConfig(shape.enc_dim, shape.proj_dim, shape.hidden, shape.n_heads, shape.ffn,
                                shape.n_blocks, shape.ln_eps)
        nb = shape.n_blocks
        keys = ("ln1_g", "ln1_b", "ln2_g", "ln2_b", "wqkv", "wo", "fc1", "fc2", "bqkv", "bo", "fc1_b", "fc2_b")
        self._arrs = {k: (C.c_void_p * max(nb, 1))(*[b[k].data_ptr() for b in weights["blocks"]]) for k in keys}
        w = QdecAdaptorWeights(weights["w1"].data_ptr(), weights["w2"].data_ptr(), weights["b1"].data_ptr(),
                               weights["b2"].data_ptr(), *[C.cast(self._arrs[k], _PP) for k in keys])
        h = C.c_void_p()
        _check(self.lib.qdec_adaptor_create(C.byref(cfg), C.byref(w), _stream_handle(stream), C.byref(h)))
        self.handle = h

    def run(self, frames, rows_out) -> int:
        """frames bf16 [T, enc_dim] (host or device) -> rows_out bf16 [fake_token_len(T), hidden]
        (host or device); returns the row count."""
        n = C.c_int32(0)
        _check(self.lib.qdec_adaptor_run(self.handle, _ptr(frames), int(frames.shape[0]), _ptr(rows_out),
                                         C.byref(n)))
        return int(n.value)

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.qdec_adaptor_destroy(self.handle)
            self.handle = None

    __del__ = close
