"""The algorithmic bytes and flops behind bench.py's roofline figures, against hand-computed values.

`achieved` in the bench line is these counts divided by measured time, so an error here would misstate every
roofline fraction.  Worked by hand for the synthetic shapes (GGUF bytes per weight: Q4_0 and Q4_K 4.5 bits,
Q8_0 8.5 bits, Q6_K 6.5625 bits):
  Llama-3-8B shape: per layer 4096*6144 + 4096*4096 + 3*14336*4096 = 218,103,808 weights, x 32 layers
  x 0.5625 B = 3.926 GB; LM head 128256*4096*0.5625 = 0.2955 GB; KV read 2*32*8*128*(p+1)*2 B
  (0.537 GB at p = 4096); norms and one embedding row are a few hundred KB.
  Prefill flops: 2 * 6.98e9 weights * tokens for the GEMMs, 4*H*D*L*sum_t(t+1) for causal attention, and
  2*V*E for the one LM-head row.
No GPU needed.
"""
import importlib.util
import os

import pytest

import synth

_spec = importlib.util.spec_from_file_location(
    "bench", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

LAYER_W_8B = 4096 * 6144 + 4096 * 4096 + 3 * 14336 * 4096  # 218,103,808


def test_layer_weight_count_8b_shape():
    assert LAYER_W_8B == 218103808


@pytest.mark.parametrize("p", [4096, 4351])
def test_decode_bytes_8b_q4_0(p):
    cfg = synth.CONFIGS[3]
    weights = 32 * LAYER_W_8B * 18 / 32 + 128256 * 4096 * 18 / 32
    kv = 2 * 32 * 8 * 128 * (p + 1) * 2
    small = 32 * 2 * 4096 * 4 + 4096 * 4 + 4096 * 18 / 32  # norm weights, final norm, one embedding row
    assert bench.decode_bytes_per_token(cfg, p) == pytest.approx(weights + kv + small, rel=1e-12)
    assert weights / 1e9 == pytest.approx(3.926 + 0.2955, abs=2e-3)


def test_decode_bytes_8b_q4_k_m_counts_the_q6_k_head():
    cfg = synth.KQUANT_CONFIGS[1]
    p = 4096
    weights = 32 * LAYER_W_8B * 144 / 256 + 128256 * 4096 * 210 / 256
    kv = 2 * 32 * 8 * 128 * (p + 1) * 2
    small = 32 * 2 * 4096 * 4 + 4096 * 4 + 4096 * 144 / 256
    assert bench.decode_bytes_per_token(cfg, p) == pytest.approx(weights + kv + small, rel=1e-12)


def test_decode_bytes_long_context_q8_0():
    cfg = synth.CONFIGS[4]  # f32 cache at p = 30720: the KV read alone is 8.05 GB
    kv = 2 * 32 * 8 * 128 * 30721 * 4
    assert kv / 1e9 == pytest.approx(8.05, abs=0.01)
    assert bench.decode_bytes_per_token(cfg, 30720) / 1e9 == pytest.approx(16.03, abs=0.01)


@pytest.mark.parametrize("idx,tokens,tflop", [(3, 4096, 61.57), (4, 30720, 676.2), (1, 2048, 4.347), (2, 1024, 2.062)])
def test_prefill_flops(idx, tokens, tflop):
    cfg = synth.CONFIGS[idx]
    total, gemm = bench.prefill_flops(cfg, tokens, 512)
    assert total / 1e12 == pytest.approx(tflop, rel=1e-3)
    L, H, D = cfg.n_layers, cfg.n_heads, cfg.head_dim
    attn = 4.0 * H * D * L * tokens * (tokens + 1) / 2
    assert total == pytest.approx(gemm + attn + 2.0 * cfg.n_vocab * cfg.n_embd, rel=1e-12)


def test_gemm_flops_per_token_8b():
    assert bench.gemm_flops(synth.CONFIGS[3], 1) == 2.0 * 32 * LAYER_W_8B
