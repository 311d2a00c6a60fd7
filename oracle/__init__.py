"""CPU oracle (fp64) for the GGUF-quantized Llama-style decoder — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It wraps ``liboracle.so`` (plain C++, fp64, built with
``-ffp-contract=off`` so x86 and Arm give the same roundings) through ctypes and
shares no code with the CUDA library.  See ``oracle.h`` for what each function
computes and which page section it follows.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

WTYPE_ID = {"q8_0": 8, "q4_0": 2, "q4_k": 12, "q5_k": 13, "q6_k": 14}
KV_ID = {"f32": 0, "f16": 1, "q8_0": 2, "q4_0": 3}


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "n_embd", "n_heads", "n_kv_heads", "head_dim", "n_ff",
                                               "n_vocab", "wtype", "kv_f16", "max_ctx", "native_ctx")] + \
               [("rms_eps", ctypes.c_double), ("rope_base", ctypes.c_double), ("out_wtype", ctypes.c_int32),
                ("kv_window", ctypes.c_int32)]


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-fPIC", "-shared", "-std=c++17", "-ffp-contract=off", "-pthread",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_double.restype = dbl
            L.orc_round_f16.argtypes = [dbl]
            L.orc_round_f16.restype = dbl
            L.orc_round_f32.argtypes = [dbl]
            L.orc_round_f32.restype = dbl
            L.orc_dequant_row.argtypes = [i32, vp, i64, vp]
            L.orc_qgemv.argtypes = [i32, vp, i64, i64, vp, vp, ctypes.c_int]
            L.orc_qgemv_rows.argtypes = [i32, vp, i64, vp, i64, vp, vp, ctypes.c_int]
            L.orc_qgemm.argtypes = [i32, vp, i64, i64, vp, i64, vp, ctypes.c_int]
            L.orc_rmsnorm.argtypes = [vp, vp, i64, dbl, vp]
            L.orc_rmsnorm.restype = None
            L.orc_yarn_scale.argtypes = [i32, i32]
            L.orc_yarn_scale.restype = dbl
            L.orc_rope_theta.argtypes = [i64, i32, i32, dbl, dbl]
            L.orc_rope_theta.restype = dbl
            L.orc_rope.argtypes = [vp, i32, i32, i64, dbl, dbl]
            L.orc_rope.restype = None
            L.orc_silu.argtypes = [dbl]
            L.orc_silu.restype = dbl
            L.orc_softmax.argtypes = [vp, i64]
            L.orc_softmax.restype = None
            L.orc_attention.argtypes = [vp, i32, i32, i32, vp, vp, i64, i64, vp]
            L.orc_attention.restype = None
            L.orc_layer_offsets.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(ctypes.c_uint64)]
            L.orc_kv_bytes.argtypes = [ctypes.POINTER(OrcConfig)]
            L.orc_kv_bytes.restype = ctypes.c_uint64
            L.orc_model_create.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(vp), vp, vp, vp, i64]
            L.orc_model_create.restype = vp
            L.orc_forward.argtypes = [vp, vp, i64, i64, vp, vp, ctypes.c_int]
            L.orc_kv_read.argtypes = [vp, i32, i32, i64, vp, vp]
            L.orc_kv_write.argtypes = [vp, i32, i32, i64, i64, vp, vp]
            L.orc_model_destroy.argtypes = [vp]
            L.orc_model_destroy.restype = None
            L.orc_argmax.argtypes = [vp, i64]
            L.orc_sample.argtypes = [vp, i64, vp, i64, dbl, dbl, dbl, dbl, vp, vp]
            L.orc_sample.restype = i64
            L.orc_sample_interval.argtypes = [vp, i64, vp, i64, dbl, dbl, dbl, i64, vp, vp, vp, vp]
            L.orc_argmax.restype = i64
            L.orc_quant_kv_row.argtypes = [i32, vp, i64]
            _lib = L
    return _lib


def _p(a):
    return a.ctypes.data


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def f16_to_double(bits: int) -> float:
    return lib().orc_f16_to_double(bits)


def round_f16(x: float) -> float:
    return lib().orc_round_f16(x)


def quant_kv_row(kv_dtype: str, v) -> np.ndarray:
    """A quantized cache's Q8_0 / Q4_0 replacement of one row of fp16 values."""
    out = np.array(v, dtype=np.float64)
    if lib().orc_quant_kv_row(KV_ID[kv_dtype], _p(out), out.size):
        raise ValueError("bad kv dtype or row length")
    return out


def dequant_row(wtype: str, blocks: np.ndarray, k: int) -> np.ndarray:
    out = np.empty(k, dtype=np.float64)
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    if lib().orc_dequant_row(WTYPE_ID[wtype], _p(b), k, _p(out)):
        raise ValueError("bad block type or k")
    return out


def qgemv(wtype: str, W: np.ndarray, n: int, k: int, x, nthreads: int = 0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(n, dtype=np.float64)
    if lib().orc_qgemv(WTYPE_ID[wtype], _p(W), n, k, _p(x), _p(y), nthreads or threads()):
        raise ValueError("bad args")
    return y


def qgemv_rows(wtype: str, W: np.ndarray, k: int, rows, x, nthreads: int = 0) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(len(rows), dtype=np.float64)
    if lib().orc_qgemv_rows(WTYPE_ID[wtype], _p(W), k, _p(rows), len(rows), _p(x), _p(y), nthreads or threads()):
        raise ValueError("bad args")
    return y


def qgemm(wtype: str, W: np.ndarray, n: int, k: int, X, nthreads: int = 0) -> np.ndarray:
    X = np.ascontiguousarray(X, dtype=np.float64)
    M = X.shape[0]
    Y = np.empty((M, n), dtype=np.float64)
    if lib().orc_qgemm(WTYPE_ID[wtype], _p(W), n, k, _p(X), M, _p(Y), nthreads or threads()):
        raise ValueError("bad args")
    return Y


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(w), x.size, eps, _p(y))
    return y


def yarn_scale(max_ctx: int, native_ctx: int) -> float:
    return lib().orc_yarn_scale(max_ctx, native_ctx)


def rope_theta(t: int, i: int, head_dim: int, base: float, ys: float) -> float:
    return lib().orc_rope_theta(t, i, head_dim, base, ys)


def rope(v, n_heads: int, head_dim: int, t: int, base: float, ys: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    lib().orc_rope(_p(v), n_heads, head_dim, t, base, ys)
    return v


def silu(g: float) -> float:
    return lib().orc_silu(g)


def softmax(s) -> np.ndarray:
    s = np.array(s, dtype=np.float64, copy=True)
    lib().orc_softmax(_p(s), s.size)
    return s


def attention(q, kc, vc, n_heads: int, n_kv_heads: int, head_dim: int, n_keys: int) -> np.ndarray:
    """q [H*D]; kc, vc [KVH, slots, D] (fp64); keys 0..n_keys-1."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    kc = np.ascontiguousarray(kc, dtype=np.float64)
    vc = np.ascontiguousarray(vc, dtype=np.float64)
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    lib().orc_attention(_p(q), n_heads, n_kv_heads, head_dim, _p(kc), _p(vc), kc.shape[1] * head_dim, n_keys,
                        _p(out))
    return out


def sample(logits, recent, repeat_penalty: float, temperature: float, top_p: float, u: float):
    """Sampler chain; returns (token, lo, hi): the token's cumulative-mass interval within the nucleus."""
    v = np.ascontiguousarray(logits, dtype=np.float64)
    r = np.ascontiguousarray(recent, dtype=np.int32)
    lo, hi = ctypes.c_double(), ctypes.c_double()
    t = lib().orc_sample(_p(v), v.size, _p(r) if r.size else None, r.size, repeat_penalty, temperature, top_p, u,
                         ctypes.byref(lo), ctypes.byref(hi))
    return int(t), lo.value, hi.value


def sample_interval(logits, recent, repeat_penalty: float, temperature: float, top_p: float, token: int):
    """(in_nucleus, lo, hi, p_token, p_boundary) of `token` under the sampler's distribution (temperature > 0)."""
    v = np.ascontiguousarray(logits, dtype=np.float64)
    r = np.ascontiguousarray(recent, dtype=np.int32)
    out = [ctypes.c_double() for _ in range(4)]
    rc = lib().orc_sample_interval(_p(v), v.size, _p(r) if r.size else None, r.size, repeat_penalty, temperature,
                                   top_p, token, *[ctypes.byref(o) for o in out])
    if rc < 0:
        raise ValueError("bad arguments")
    return bool(rc), out[0].value, out[1].value, out[2].value, out[3].value


def argmax(v) -> int:
    v = np.ascontiguousarray(v, dtype=np.float64)
    return int(lib().orc_argmax(_p(v), v.size))


def config_of(cfg) -> OrcConfig:
    """OrcConfig from a synth.ModelConfig-like object."""
    return OrcConfig(cfg.n_layers, cfg.n_embd, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ff, cfg.n_vocab,
                     WTYPE_ID[cfg.wtype], KV_ID[cfg.kv_dtype], cfg.max_ctx, cfg.native_ctx,
                     cfg.rms_eps, cfg.rope_base, WTYPE_ID[getattr(cfg, "out_wtype", "") or cfg.wtype],
                     getattr(cfg, "kv_window", 0))


def layer_offsets(cfg):
    off = (ctypes.c_uint64 * 10)()
    c = config_of(cfg)
    if lib().orc_layer_offsets(ctypes.byref(c), off):
        raise ValueError("bad shape")
    return [int(v) for v in off]


def kv_bytes(cfg) -> int:
    c = config_of(cfg)
    return int(lib().orc_kv_bytes(ctypes.byref(c)))


class Model:
    """fp64 reference model over host blobs (kept alive by this object)."""

    def __init__(self, cfg, layers, token_embd, output_norm, output, kv_slots: int = 0):
        self.cfg = cfg
        self._keep = (list(layers), token_embd, output_norm, output)
        self._c = config_of(cfg)
        arr = (ctypes.c_void_p * cfg.n_layers)(*[b.ctypes.data for b in layers])
        self._arr = arr
        self.h = lib().orc_model_create(ctypes.byref(self._c), arr, _p(token_embd), _p(output_norm), _p(output),
                                        kv_slots)
        if not self.h:
            raise ValueError("orc_model_create failed")

    @classmethod
    def from_host(cls, hm, kv_slots: int = 0):
        return cls(hm.cfg, hm.layers, hm.token_embd, hm.output_norm, hm.output, kv_slots)

    def forward(self, tokens, start_pos: int, want_logits=True, capture=False, nthreads: int = 0):
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.size
        logits = np.empty(self.cfg.n_vocab, dtype=np.float64) if want_logits else None
        cap = np.empty((self.cfg.n_layers + 1, n, self.cfg.n_embd), dtype=np.float64) if capture else None
        rc = lib().orc_forward(self.h, _p(tok), n, start_pos, _p(logits) if logits is not None else None,
                               _p(cap) if cap is not None else None, nthreads or threads())
        if rc:
            raise ValueError(f"orc_forward rc={rc}")
        return logits, cap

    def kv_read(self, layer: int, kvh: int, pos: int):
        D = self.cfg.head_dim
        k = np.empty(D, dtype=np.float64)
        v = np.empty(D, dtype=np.float64)
        if lib().orc_kv_read(self.h, layer, kvh, pos, _p(k), _p(v)):
            raise IndexError("slot out of range")
        return k, v

    def kv_write(self, layer: int, kvh: int, pos0: int, k, v):
        """Set slots pos0.. of (layer, kv head) to k, v [n][head_dim] (values of the cache's element type)."""
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        if k.shape != v.shape or k.ndim != 2 or k.shape[1] != self.cfg.head_dim:
            raise ValueError("k, v must be [n][head_dim]")
        if lib().orc_kv_write(self.h, layer, kvh, pos0, k.shape[0], _p(k), _p(v)):
            raise IndexError("slots out of range")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib().orc_model_destroy(h)
            self.h = None
