"""The C-ABI library loads and exports every symbol include/af.h declares;
host-only entry points agree with the oracle; validation errors come back as
status codes before anything touches a GPU.  No GPU needed."""
import ctypes
import os
import re

import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _af():
    import gguf_quantized_transformer_gb300 as af
    af.build()
    return af


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "af.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(af_[a-z_0-9]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported():
    af = _af()
    L = af.lib()
    syms = declared_symbols()
    assert "af_model_create" in syms and "af_qgemv" in syms and "af_qgemm" in syms
    assert "af_prefill" in syms and "af_decode_step" in syms
    for s in syms:
        assert hasattr(L, s), s


def test_python_binding_has_same_names():
    af = _af()
    for s in declared_symbols():
        assert hasattr(af, s), s


@pytest.mark.parametrize("idx", range(5))
def test_layer_offsets_and_kv_bytes_match_oracle(idx):
    af = _af()
    cfg = synth.CONFIGS[idx]
    c = af.make_config(cfg)
    assert af.af_layer_offsets(c) == oracle.layer_offsets(cfg) == synth.layer_offsets(cfg)
    assert af.af_kv_bytes(c) == oracle.kv_bytes(cfg)


@pytest.mark.parametrize("idx", range(len(synth.KQUANT_CONFIGS)))
def test_kquant_layer_offsets_match_oracle(idx):
    af = _af()
    cfg = synth.KQUANT_CONFIGS[idx]
    c = af.make_config(cfg)
    assert c.out_wtype == af.AF_Q6_K
    assert af.af_layer_offsets(c) == oracle.layer_offsets(cfg) == synth.layer_offsets(cfg)


def test_kquant_config_validation_without_gpu():
    af = _af()
    L = af.lib()
    out = ctypes.c_void_p()
    c = af.make_config(synth.KQUANT_CONFIGS[0])
    c.n_ff = 1408  # not a whole number of 256-weight super-blocks
    assert L.af_model_create(ctypes.byref(c), None, None, ctypes.byref(out)) == af.AF_EINVAL
    c = af.make_config(synth.KQUANT_CONFIGS[0])
    c.out_wtype = 7
    assert L.af_model_create(ctypes.byref(c), None, None, ctypes.byref(out)) == af.AF_EINVAL
    assert "out_wtype" in af.af_last_error()
    c = af.make_config(synth.CONFIGS[0])  # a Q8_0 body with a Q6_K head: n_embd 512 is whole super-blocks
    c.out_wtype = af.AF_Q6_K
    c.n_embd = 500
    assert L.af_model_create(ctypes.byref(c), None, None, ctypes.byref(out)) == af.AF_EINVAL
    assert out.value is None


def test_tinyllama_kv_bytes_worked_example():
    af = _af()
    assert af.af_kv_bytes(af.make_config(synth.CONFIGS[1])) == 92274688


def test_validation_errors_without_gpu():
    af = _af()
    L = af.lib()
    out = ctypes.c_void_p()
    assert L.af_model_create(None, None, None, ctypes.byref(out)) == af.AF_EINVAL
    c = af.make_config(synth.CONFIGS[0])
    c.wtype = 99
    assert L.af_model_create(ctypes.byref(c), None, None, ctypes.byref(out)) == af.AF_EINVAL
    assert "wtype" in af.af_last_error()
    c = af.make_config(synth.CONFIGS[0])
    c.n_kv_heads = 3
    assert L.af_model_create(ctypes.byref(c), None, None, ctypes.byref(out)) == af.AF_EINVAL
    c = af.make_config(synth.CONFIGS[0])
    c.head_dim = 96  # valid but not implemented
    c.n_heads = 8
    w = af.af_weights()
    assert L.af_model_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(out)) == af.AF_ENOTIMPL
    assert out.value is None
    assert L.af_qweight_create(af.AF_Q8_0, None, 4, 32, None, ctypes.byref(out)) == af.AF_EINVAL
    assert L.af_qweight_create(af.AF_Q8_0, 1, 4, 48, None, ctypes.byref(out)) == af.AF_EINVAL
    assert L.af_prefill(None, None, 1, 0, None) == af.AF_EINVAL
    assert L.af_decode_step(None, 0, 0, None, None) == af.AF_EINVAL
    assert L.af_attention_decode(None, None, None, 0, 8, 4, 64, 16, 0, None, None) == af.AF_EINVAL
    assert L.af_attention_decode_static(None, None, None, 0, 8, 4, 64, 16, 0, None, None) == af.AF_EINVAL


def test_sampler_validation():
    # host-side checks only (no launch)
    af = pytest.importorskip("gguf_quantized_transformer_gb300")
    L = af.lib()
    assert L.af_sample(None, 10, None, 0, 1.0, 1.0, 1.0, 0.5, 1, None) == af.AF_EINVAL
    assert L.af_sample(1, 0, None, 0, 1.0, 1.0, 1.0, 0.5, 1, None) == af.AF_ERANGE
    assert L.af_sample(1, 300000, None, 0, 1.0, 1.0, 1.0, 0.5, 1, None) == af.AF_ERANGE
    assert L.af_sample(1, 10, None, 3, 1.0, 1.0, 1.0, 0.5, 1, None) == af.AF_EINVAL
    assert L.af_sample(1, 10, None, 0, 1.0, -1.0, 1.0, 0.5, 1, None) == af.AF_EINVAL
    assert L.af_sample(1, 10, None, 0, 1.0, 1.0, 1.0, 1.0, 1, None) == af.AF_ERANGE
    assert L.af_sample(1, 10, None, 0, 1.0, 1.0, 1.0, -0.1, 1, None) == af.AF_ERANGE


def test_model_sample_validation():
    # host-side checks only: a null model and bad arguments return before any launch
    af = pytest.importorskip("gguf_quantized_transformer_gb300")
    L = af.lib()
    assert L.af_model_sample(None, None, None, 0, 1.0, 0.8, 0.9, 0.5, None) == af.AF_EINVAL
    assert "null model" in af.af_last_error()


def test_static_attention_rejects_oversize():
    # host-side capacity checks of the fixed scratch; they return before any launch
    # (the pointers are never dereferenced on the host)
    af = pytest.importorskip("gguf_quantized_transformer_gb300")
    L = af.lib()
    # (caches above 2048 slots: the split path, the only one that uses the fixed scratch)
    # more kv heads than arrival counters
    assert L.af_attention_decode_static(1, 1, 1, af.AF_F16, 1028, 1028, 64, 16384, 0, 1, None) == af.AF_ERANGE
    assert "n_kv_heads" in af.af_last_error()
    # partials: 8192 heads x >= 1 split x 132 floats > 2^20
    assert L.af_attention_decode_static(1, 1, 1, af.AF_F16, 8192, 1024, 128, 16384, 0, 1, None) == af.AF_ERANGE
    assert "partials" in af.af_last_error()
    assert af.af_kv_bytes(af.af_config()) == 0


def test_new_entry_points_validate_on_the_host():
    # argument checks that return before any launch (the pointers are never dereferenced on the host)
    af = pytest.importorskip("gguf_quantized_transformer_gb300")
    L = af.lib()
    ok = dict(kv=af.AF_F16, H=32, KVH=8, D=128, ctx=1024)
    def pf(q=1, start=0, n=4, ctx=1024, kv=af.AF_F16, H=32, KVH=8, D=128, out=16):
        return L.af_attention_prefill(q, 16, 16, kv, H, KVH, D, ctx, start, n, out, None)
    assert pf(q=None) == af.AF_EINVAL
    assert pf(out=None) == af.AF_EINVAL
    assert pf(kv=7) == af.AF_EINVAL
    assert pf(n=0) == af.AF_ERANGE and pf(n=513) == af.AF_ERANGE
    assert pf(start=1022, n=4) == af.AF_ERANGE and pf(start=-1) == af.AF_ERANGE
    assert pf(D=96) == af.AF_ENOTIMPL and pf(H=24, KVH=8) == af.AF_ENOTIMPL
    assert pf(q=8) == af.AF_EINVAL  # not 16-byte aligned
    assert ok
    assert L.af_qweight_status(None, None) == af.AF_EINVAL
    assert L.af_qweight_debug_stall(None, 1, None) == af.AF_EINVAL
    assert L.af_debug_stall(None, 1) == af.AF_EINVAL


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_quantized_kv_bytes_match_oracle(kvt):
    af = _af()
    cfg = synth.CONFIGS[3].with_(kv_dtype=kvt, kv_window=512)
    assert af.af_kv_bytes(af.make_config(cfg)) == oracle.kv_bytes(cfg)


def test_quantized_kv_config_validation():
    # host-side checks in af_model_create, before any device work (dummy pointers are never dereferenced)
    af = _af()
    L = af.lib()
    cfg = synth.CONFIGS[0].with_(kv_dtype="q8_0", kv_window=8)
    blobs = (ctypes.c_void_p * cfg.n_layers)(*([16] * cfg.n_layers))
    w = af.af_weights(blobs, 16, 16, 16)
    h = ctypes.c_void_p()
    c = af.make_config(cfg, max_chunk=16)  # window shorter than a chunk
    assert L.af_model_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == af.AF_EINVAL
    assert "kv_window" in af.af_last_error()
    c = af.make_config(cfg.with_(max_ctx=66), max_chunk=8)  # slots not a multiple of 4
    assert L.af_model_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == af.AF_ENOTIMPL
    c = af.make_config(cfg, max_chunk=8)
    c.kv_dtype = 9
    assert L.af_model_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == af.AF_EINVAL
    assert L.af_model_kv_store(None, None, None, None, None) == af.AF_EINVAL


def test_product_path_has_no_cpu_fallback():
    # the package must not import the oracle or any CPU implementation
    pkg = os.path.join(ROOT, "gguf_quantized_transformer_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f
