"""GB300 (sm_103a) forward pass of a GGUF (Q8_0 / Q4_0 / Q4_K / Q5_K / Q6_K) Llama-style decoder.

Thin ctypes binding over ``libaf.so`` (C ABI in ``include/af.h``): the
functions below only marshal arguments; every step of the forward pass runs in
the library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no CPU path: importing this package raises if the library is missing.
"""
import ctypes
import os

from ._build import LIB_PATH, build  # noqa: F401

AF_OK, AF_EINVAL, AF_ERANGE, AF_ENOMEM, AF_ECUDA, AF_ETIMEOUT, AF_ENOTIMPL = range(7)
AF_Q4_0, AF_Q8_0, AF_Q4_K, AF_Q5_K, AF_Q6_K = 2, 8, 12, 13, 14
AF_F32, AF_F16, AF_KV_Q8_0, AF_KV_Q4_0 = 0, 1, 2, 3
WTYPE = {"q4_0": AF_Q4_0, "q8_0": AF_Q8_0, "q4_k": AF_Q4_K, "q5_k": AF_Q5_K, "q6_k": AF_Q6_K}
KVTYPE = {"f32": AF_F32, "f16": AF_F16, "q8_0": AF_KV_Q8_0, "q4_0": AF_KV_Q4_0}
STATUS_NAMES = {0: "AF_OK", 1: "AF_EINVAL", 2: "AF_ERANGE", 3: "AF_ENOMEM", 4: "AF_ECUDA", 5: "AF_ETIMEOUT",
                6: "AF_ENOTIMPL"}


class AfError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class af_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "n_embd", "n_heads", "n_kv_heads", "head_dim", "n_ff",
                                               "n_vocab", "wtype", "kv_dtype", "max_ctx", "native_ctx",
                                               "max_chunk")] + \
               [("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("out_wtype", ctypes.c_int32),
                ("kv_window", ctypes.c_int32)]


class af_weights(ctypes.Structure):
    _fields_ = [("layer_blob", ctypes.POINTER(ctypes.c_void_p)), ("token_embd", ctypes.c_void_p),
                ("output_norm", ctypes.c_void_p), ("output", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libaf.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libaf.so not found at {LIB_PATH}: run __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64
        P = ctypes.POINTER
        L.af_last_error.restype = ctypes.c_char_p
        L.af_layer_offsets.argtypes = [P(af_config), P(u64)]
        L.af_kv_bytes.argtypes = [P(af_config)]
        L.af_kv_bytes.restype = u64
        L.af_model_create.argtypes = [P(af_config), P(af_weights), vp, P(vp)]
        L.af_prefill.argtypes = [vp, vp, i32, i32, vp]
        L.af_prefill_dev.argtypes = [vp, vp, i32, i32, vp]
        L.af_decode_step.argtypes = [vp, i32, i32, vp, vp]
        L.af_model_next_token_dev.argtypes = [vp]
        L.af_model_next_token_dev.restype = vp
        L.af_reset.argtypes = [vp]
        L.af_model_sync.argtypes = [vp, vp]
        L.af_model_kv_cache.argtypes = [vp, P(vp), P(vp)]
        L.af_model_kv_store.argtypes = [vp, P(vp), P(vp), P(vp), P(vp)]
        L.af_model_stream.argtypes = [vp]
        L.af_model_stream.restype = vp
        L.af_debug_capture.argtypes = [vp, vp]
        L.af_debug_trace.argtypes = [vp, vp]
        L.af_set_decode_graph.argtypes = [vp, ctypes.c_int]
        L.af_set_decode_mode.argtypes = [vp, ctypes.c_int]
        L.af_get_decode_mode.argtypes = [vp]
        L.af_model_destroy.argtypes = [vp]
        L.af_model_destroy.restype = None
        L.af_qweight_create.argtypes = [i32, vp, i32, i32, vp, P(vp)]
        L.af_qgemv.argtypes = [vp, vp, vp, vp]
        L.af_qgemm.argtypes = [vp, vp, i32, vp, vp]
        L.af_qweight_destroy.argtypes = [vp]
        L.af_qweight_destroy.restype = None
        L.af_attention_decode.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        L.af_attention_decode_static.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        L.af_attention_prefill.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        L.af_debug_stall.argtypes = [vp, ctypes.c_uint32]
        L.af_qweight_status.argtypes = [vp, vp]
        L.af_qweight_debug_stall.argtypes = [vp, ctypes.c_uint32, vp]
        f32 = ctypes.c_float
        L.af_sample.argtypes = [vp, i32, vp, i32, f32, f32, f32, f32, vp, vp]
        L.af_model_sample.argtypes = [vp, vp, vp, i32, f32, f32, f32, f32, vp]
        _lib = L
    return _lib


def check(rc):
    if rc != AF_OK:
        raise AfError(rc, lib().af_last_error().decode())
    return rc


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_config(cfg, max_chunk: int = 512) -> af_config:
    """af_config from a ModelConfig-like object (fields as in synth.configs)."""
    return af_config(cfg.n_layers, cfg.n_embd, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ff, cfg.n_vocab,
                     WTYPE[cfg.wtype], KVTYPE[cfg.kv_dtype], cfg.max_ctx, cfg.native_ctx, max_chunk, cfg.rms_eps,
                     cfg.rope_base, WTYPE[getattr(cfg, "out_wtype", "") or cfg.wtype], getattr(cfg, "kv_window", 0))


# ---------------------------------------------------------------- same-name entry points

def af_layer_offsets(cfg: af_config):
    off = (ctypes.c_uint64 * 10)()
    check(lib().af_layer_offsets(ctypes.byref(cfg), off))
    return [int(v) for v in off]


def af_kv_bytes(cfg: af_config) -> int:
    return int(lib().af_kv_bytes(ctypes.byref(cfg)))


def af_model_create(cfg: af_config, layer_blobs, token_embd, output_norm, output, stream=None):
    arr = (ctypes.c_void_p * cfg.n_layers)(*[_ptr(b) for b in layer_blobs])
    w = af_weights(arr, _ptr(token_embd), _ptr(output_norm), _ptr(output))
    h = ctypes.c_void_p()
    check(lib().af_model_create(ctypes.byref(cfg), ctypes.byref(w), _stream(stream), ctypes.byref(h)))
    return h.value


def af_prefill(m, tokens_host, n: int, start_pos: int, logits_dev=None):
    """tokens_host: a C-contiguous int32 numpy array (or host pointer)."""
    p = tokens_host if isinstance(tokens_host, int) else tokens_host.ctypes.data
    return check(lib().af_prefill(m, p, n, start_pos, _ptr(logits_dev)))


def af_prefill_dev(m, tokens_dev, n: int, start_pos: int, logits_dev=None):
    return check(lib().af_prefill_dev(m, _ptr(tokens_dev), n, start_pos, _ptr(logits_dev)))


def af_decode_step(m, token: int, pos: int, logits_dev=None, want_next: bool = False):
    nxt = ctypes.c_int32(-1)
    check(lib().af_decode_step(m, token, pos, _ptr(logits_dev), ctypes.byref(nxt) if want_next else None))
    return nxt.value if want_next else None


def af_model_next_token_dev(m) -> int:
    return lib().af_model_next_token_dev(m)


def af_model_sync(m, want_next: bool = False):
    nxt = ctypes.c_int32(-1)
    check(lib().af_model_sync(m, ctypes.byref(nxt) if want_next else None))
    return nxt.value if want_next else None


def af_model_stream(m) -> int:
    return lib().af_model_stream(m) or 0


def af_model_kv_cache(m):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    check(lib().af_model_kv_cache(m, ctypes.byref(k), ctypes.byref(v)))
    return k.value, v.value


def af_model_kv_store(m):
    """(k_codes, k_scales, v_codes, v_scales) device pointers of a quantized cache's store."""
    p = [ctypes.c_void_p() for _ in range(4)]
    check(lib().af_model_kv_store(m, *[ctypes.byref(x) for x in p]))
    return tuple(x.value for x in p)


def af_reset(m):
    return check(lib().af_reset(m))


def af_debug_capture(m, hidden_dev):
    return check(lib().af_debug_capture(m, _ptr(hidden_dev)))


AF_DECODE_PERSISTENT, AF_DECODE_KERNELS = 0, 1


def af_set_decode_mode(m, mode: int):
    return check(lib().af_set_decode_mode(m, mode))


def af_get_decode_mode(m) -> int:
    return lib().af_get_decode_mode(m)


def af_debug_trace(m, trace_dev):
    return check(lib().af_debug_trace(m, _ptr(trace_dev)))


def af_set_decode_graph(m, enable: bool):
    return check(lib().af_set_decode_graph(m, 1 if enable else 0))


def af_model_destroy(m):
    lib().af_model_destroy(m)


def af_qweight_create(wtype: int, blocks_dev, N: int, K: int, stream=None):
    h = ctypes.c_void_p()
    check(lib().af_qweight_create(wtype, _ptr(blocks_dev), N, K, _stream(stream), ctypes.byref(h)))
    return h.value


def af_qgemv(w, x_dev, y_dev, stream=None):
    return check(lib().af_qgemv(w, _ptr(x_dev), _ptr(y_dev), _stream(stream)))


def af_qgemm(w, X_dev, M: int, Y_dev, stream=None):
    return check(lib().af_qgemm(w, _ptr(X_dev), M, _ptr(Y_dev), _stream(stream)))


def af_qweight_destroy(w):
    lib().af_qweight_destroy(w)


def af_qweight_status(w, stream=None):
    return check(lib().af_qweight_status(w, _stream(stream)))


def af_qweight_debug_stall(w, polls: int, stream=None):
    return check(lib().af_qweight_debug_stall(w, polls, _stream(stream)))


def af_debug_stall(m, polls: int):
    return check(lib().af_debug_stall(m, polls))


def af_attention_decode(q_dev, k_dev, v_dev, kv_dtype: int, n_heads: int, n_kv_heads: int, head_dim: int, ctx: int,
                        pos: int, out_dev, stream=None):
    return check(lib().af_attention_decode(_ptr(q_dev), _ptr(k_dev), _ptr(v_dev), kv_dtype, n_heads, n_kv_heads,
                                           head_dim, ctx, pos, _ptr(out_dev), _stream(stream)))


def af_attention_decode_static(q_dev, k_dev, v_dev, kv_dtype: int, n_heads: int, n_kv_heads: int, head_dim: int,
                               ctx: int, pos: int, out_dev, stream=None):
    return check(lib().af_attention_decode_static(_ptr(q_dev), _ptr(k_dev), _ptr(v_dev), kv_dtype, n_heads,
                                                  n_kv_heads, head_dim, ctx, pos, _ptr(out_dev), _stream(stream)))


def af_attention_prefill(q_dev, k_dev, v_dev, kv_dtype: int, n_heads: int, n_kv_heads: int, head_dim: int, ctx: int,
                         start_pos: int, n: int, out_dev, stream=None):
    return check(lib().af_attention_prefill(_ptr(q_dev), _ptr(k_dev), _ptr(v_dev), kv_dtype, n_heads, n_kv_heads,
                                            head_dim, ctx, start_pos, n, _ptr(out_dev), _stream(stream)))


def af_sample(logits_dev, n_vocab: int, recent_dev, n_recent: int, repeat_penalty: float, temperature: float,
              top_p: float, u: float, token_dev, stream=None):
    return check(lib().af_sample(_ptr(logits_dev), n_vocab, _ptr(recent_dev), n_recent, repeat_penalty, temperature,
                                 top_p, u, _ptr(token_dev), _stream(stream)))


def af_model_sample(m, logits_dev, recent_dev, n_recent: int, repeat_penalty: float, temperature: float,
                    top_p: float, u: float, want_token: bool = False):
    """Sampler chain over the model's logits into its next-token word; returns the token if want_token."""
    out = ctypes.c_int32(-1)
    check(lib().af_model_sample(m, _ptr(logits_dev), _ptr(recent_dev), n_recent, repeat_penalty, temperature, top_p,
                                u, ctypes.byref(out) if want_token else None))
    return out.value if want_token else None


def af_last_error() -> str:
    return lib().af_last_error().decode()


# ---------------------------------------------------------------- convenience wrapper

class Model:
    """Owns an af_model; weights are device tensors in the layer-blob format."""

    def __init__(self, cfg, layer_blobs, token_embd, output_norm, output, max_chunk: int = 512, stream=None):
        self.cfg = cfg
        self.c = make_config(cfg, max_chunk)
        self.h = af_model_create(self.c, layer_blobs, token_embd, output_norm, output, stream)

    def prefill(self, tokens_host, start_pos: int, logits_dev=None):
        import numpy as np
        t = np.ascontiguousarray(tokens_host, dtype=np.int32)
        return af_prefill(self.h, t, t.size, start_pos, logits_dev)

    def decode(self, token: int, pos: int, logits_dev=None, want_next: bool = False):
        return af_decode_step(self.h, token, pos, logits_dev, want_next)

    def close(self):
        if getattr(self, "h", None):
            af_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
