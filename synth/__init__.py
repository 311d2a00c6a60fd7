"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

A thin ctypes wrapper over ``synth.c`` (counter-based normals, GGUF Q8_0/Q4_0/
Q4_K/Q6_K block encoder, layer-blob packer).  It holds input generation only: nothing in
this package decodes a block or computes any step of the forward pass.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import (CONFIGS, KQUANT_CONFIGS, ModelConfig, Q4_0, Q8_0, Q4_K, Q5_K, Q6_K, BASE_SEED,  # noqa: F401
                      seed_of, kquant_seed_of)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

WTYPE_ID = {Q8_0: 8, Q4_0: 2, Q4_K: 12, Q5_K: 13, Q6_K: 14}
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_K: 144, Q5_K: 176, Q6_K: 210}
BLOCK_ELEMS = {Q8_0: 32, Q4_0: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256}

# tensor ids outside the per-layer range 1 + 16*layer + section
TID_TOKEN_EMBD = 0x100000
TID_OUTPUT_NORM = 0x100001
TID_OUTPUT = 0x100002
TID_PROMPT = 0x100003
TID_TEST_BASE = 0x200000


def build(force: bool = False) -> str:
    """Compile libsynth.so in place (gcc, portable C, no arch flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float
            vp = ctypes.c_void_p
            lib.syn_layer_offsets.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(u64)]
            lib.syn_gen_matrix.argtypes = [ctypes.c_int, u64, u64, i64, i64, f32, f32, vp, ctypes.c_int]
            lib.syn_gen_f32.argtypes = [u64, u64, i64, f32, f32, vp]
            lib.syn_gen_f32.restype = None
            lib.syn_gen_tokens.argtypes = [u64, u64, i64, ctypes.c_int, vp]
            lib.syn_gen_tokens.restype = None
            lib.syn_gen_layer.argtypes = [ctypes.c_int] * 6 + [u64, ctypes.c_int, f32, f32, vp, ctypes.c_int]
            lib.syn_f32_to_f16_bits.argtypes = [f32]
            lib.syn_f32_to_f16_bits.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def layer_offsets(cfg: ModelConfig):
    off = (ctypes.c_uint64 * 10)()
    rc = _load().syn_layer_offsets(cfg.n_embd, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ff,
                                   WTYPE_ID[cfg.wtype], off)
    if rc:
        raise ValueError(f"shape not blockable by {BLOCK_ELEMS[cfg.wtype]}")
    return [int(v) for v in off]


def matrix(wtype: str, seed: int, tid: int, n: int, k: int, sigma: float = 0.02, mean: float = 0.0,
           threads: int = 0) -> np.ndarray:
    """Random [n, k] matrix encoded as GGUF blocks: uint8 array of n*(k/block elements)*block bytes."""
    if k % BLOCK_ELEMS[wtype]:
        raise ValueError(f"k must be a multiple of {BLOCK_ELEMS[wtype]}")
    out = np.empty(n * (k // BLOCK_ELEMS[wtype]) * BLOCK_BYTES[wtype], dtype=np.uint8)
    rc = _load().syn_gen_matrix(WTYPE_ID[wtype], seed, tid, n, k, mean, sigma, out.ctypes.data,
                                threads or default_threads())
    if rc:
        raise ValueError("bad matrix shape")
    return out


def normals(seed: int, tid: int, n: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().syn_gen_f32(seed, tid, n, mean, sigma, out.ctypes.data)
    return out


def tokens(seed: int, n: int, vocab: int, tid: int = TID_PROMPT) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().syn_gen_tokens(seed, tid, n, vocab, out.ctypes.data)
    return out


def f16_bits(x: float) -> int:
    return int(_load().syn_f32_to_f16_bits(x))


def layer_blob(cfg: ModelConfig, seed: int, layer: int, threads: int = 0) -> np.ndarray:
    off = layer_offsets(cfg)
    out = np.empty(off[9], dtype=np.uint8)
    rc = _load().syn_gen_layer(cfg.n_embd, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ff,
                               WTYPE_ID[cfg.wtype], seed, layer, cfg.w_sigma, cfg.norm_sigma, out.ctypes.data,
                               threads or default_threads())
    if rc:
        raise ValueError("bad shape")
    return out


class HostModel:
    """All synthetic weights of one model, as host numpy arrays in the blob format."""

    def __init__(self, cfg: ModelConfig, seed: int, threads: int = 0):
        self.cfg, self.seed = cfg, seed
        self.offsets = layer_offsets(cfg)
        self.layers = [layer_blob(cfg, seed, l, threads) for l in range(cfg.n_layers)]
        self.token_embd = matrix(cfg.wtype, seed, TID_TOKEN_EMBD, cfg.n_vocab, cfg.n_embd, cfg.w_sigma,
                                 threads=threads)
        self.output_norm = normals(seed, TID_OUTPUT_NORM, cfg.n_embd, 1.0, cfg.norm_sigma)
        self.output = matrix(cfg.head_wtype, seed, TID_OUTPUT, cfg.n_vocab, cfg.n_embd, cfg.w_sigma,
                             threads=threads)

    def prompt(self, n: int = 0) -> np.ndarray:
        return tokens(self.seed, n or self.cfg.prompt_len, self.cfg.n_vocab)

    def nbytes(self) -> int:
        return sum(b.nbytes for b in self.layers) + self.token_embd.nbytes + self.output.nbytes + \
            self.output_norm.nbytes
