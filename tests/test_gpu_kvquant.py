"""Quantized KV cache (Q8_0 / Q4_0 with an fp16 window) on the GPU against the oracle.

dotLLM, "CUDA components", names a quantized KV cache "Q8_0/Q4_0 + FP16 window"; the reading (oracle.cpp,
include/af.h): a slot is written in fp16 and, once it lies more than kv_window positions behind a step's last
position, is replaced by the Q8_0 / Q4_0 quantization of its fp16 values (decisions in fp32).  Checked:
  * whole-model parity (every layer's residual stream and the logits within 2e-2 * RMS, greedy ids where the
    margin allows) on the tiny model with a window of 8 slots (most slots retired) and on a 2-layer
    Llama-3-8B shape with a 512-slot window over two 512-token chunks and decode steps (decode attention reads
    the retired slots from the quantized store);
  * the retired codes bit-exact: the store and the fp16 copy of every retired slot equal the oracle's
    quantization of the GPU's own fp16 row from before it retired.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import device_array, gpu_model, run_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def af():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_quantized_transformer_gb300 as af
    af.build()
    af.lib()
    return af


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_tiny_small_window_parity(af, kvt):
    cfg = synth.CONFIGS[0].with_(kv_dtype=kvt, kv_window=8)
    run_parity(af, cfg, synth.seed_of(0), [8, 8, 8, 5], 10, 0, max_chunk=8)


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_tiny_window_covering_the_sequence(af, kvt):
    cfg = synth.CONFIGS[0].with_(kv_dtype=kvt, kv_window=64)
    run_parity(af, cfg, synth.seed_of(0), [32], 8, 0, max_chunk=64)


def test_llama3_8b_shape_q8_0_window_512(af):
    cfg = synth.CONFIGS[3].with_(n_layers=2, kv_dtype="q8_0", kv_window=512)
    worst = run_parity(af, cfg, synth.seed_of(3), [512, 512], 4, 1024 + 4)
    print(f"\n{cfg.name} kv q8_0 window 512, 2 layers, 2 x 512 + 4: worst layer {worst['layer']:.2e}, "
          f"logits {worst['logits']:.2e}")


def _dequant_store(kvt, codes, scales):
    """Values of store rows: codes [..., CB] uint8, scales [..., D/32] fp16 -> [..., D] float64."""
    d = scales.astype(np.float64)
    if kvt == "q8_0":
        q = codes.view(np.int8).astype(np.float64)
    else:
        lo = (codes & 15).astype(np.int64) - 8
        hi = (codes >> 4).astype(np.int64) - 8
        q = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2).astype(np.float64)
    D = q.shape[-1]
    return q * np.repeat(d, 32, axis=-1)[..., :D]


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_retired_rows_bit_exact(af, kvt):
    W = 8
    cfg = synth.CONFIGS[0].with_(kv_dtype=kvt, kv_window=W)
    hm = synth.HostModel(cfg, synth.seed_of(0))
    gm = gpu_model(hm, max_chunk=W)
    L, KVH, ctx, D = cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim
    kp, vp = af.af_model_kv_cache(gm.h)
    kc, vc = device_array(kp, (L, KVH, ctx, D), "<f2"), device_array(vp, (L, KVH, ctx, D), "<f2")
    prompt = hm.prompt(2 * W)
    gm.prefill(prompt[:W], 0)
    torch.cuda.synchronize()
    before = [kc[:, :, :W].double().cpu().numpy(), vc[:, :, :W].double().cpu().numpy()]
    gm.prefill(prompt[W:], W)  # slots 0..W-1 leave the window and retire before this chunk's attention
    torch.cuda.synchronize()
    kq, ks, vq, vs = af.af_model_kv_store(gm.h)
    cb = D if kvt == "q8_0" else D // 2
    for (cp, sp, fp16, rows) in [(kq, ks, kc, before[0]), (vq, vs, vc, before[1])]:
        codes = device_array(cp, (L, KVH, ctx, cb), "|u1")[:, :, :W].cpu().numpy()
        scales = device_array(sp, (L, KVH, ctx, D // 32), "<f2")[:, :, :W].cpu().numpy()
        got = _dequant_store(kvt, codes, scales)
        want = np.stack([oracle.quant_kv_row(kvt, r) for r in rows.reshape(-1, D)]).reshape(rows.shape)
        assert np.array_equal(got, want)
        # the fp16 copy of a retired slot: fp16(d q)
        copy = fp16[:, :, :W].double().cpu().numpy()
        assert np.array_equal(copy, want.astype(np.float16).astype(np.float64))
        # slots still in the window keep their fp16 values (not retired)
    gm.close()


def test_window_must_cover_a_chunk(af):
    cfg = synth.CONFIGS[0].with_(kv_dtype="q8_0", kv_window=8)
    hm = synth.HostModel(cfg, synth.seed_of(0))
    with pytest.raises(af.AfError) as e:
        gpu_model(hm, max_chunk=16)
    assert e.value.code == af.AF_EINVAL
