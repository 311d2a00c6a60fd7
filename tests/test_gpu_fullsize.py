"""Parity at the sizes the prefill kernels run at in the full workloads.

The prefill runs 512-row chunks: the tensor-core GEMM then spans four 128-row
M tiles with its fused epilogues (RoPE + KV write at start_pos + row, SwiGLU,
residual), and the tensor-core attention streams hundreds of key tiles per
query tile (Airframe "GPU_PIPELINE.md", Prefill: 512-token chunks filling KV
slots start_pos..; "Shimmy v2.0 Architecture", Extended Context (YaRN)).

  * standalone prefill attention (af_attention_prefill) against the oracle's
    attention, row by row: n = 512 at start_pos 0, 512 and 3584 over an fp16
    cache (Llama-3-8B shape), at 30208 over an fp32 cache (the 32768-slot
    long-context shape), at 1536 with head_dim 64 and group 8 (TinyLlama
    shape), and a ragged n = 300 at 700;
  * 2-layer versions of the Llama-3-8B Q4_0 and Q8_0/YaRN shapes through the
    whole model: two 512-token chunks then decode steps, and a 512-token chunk
    at start_pos 29696 over a cache prefix both sides hold (YaRN theta at
    t ~ 30k, ~460 key tiles per query tile);
  * the same decode steps through the persistent decode kernel
    (AF_DECODE_PERSISTENT): its streamed attention over an fp16 cache after
    1024 positions, and over an fp32 cache at t ~ 30k (about a hundred
    stages per split).

Tolerances: attention outputs within 1e-3 normwise per row (the standalone
bar); layer outputs and logits within 2e-2 * RMS(oracle).  The worst errors
seen are printed (run with -s to see them).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import normwise_rel_err, run_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ATTN_TOL = 1e-3


@pytest.fixture(scope="module")
def af():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_quantized_transformer_gb300 as af
    af.build()
    af.lib()
    return af


def _prefill_case(seed, H, KVH, D, ctx, n, kvt, qscale=1.0):
    q = synth.normals(seed, synth.TID_TEST_BASE + 70, n * H * D, sigma=qscale).reshape(n, H * D)
    kc = synth.normals(seed, synth.TID_TEST_BASE + 71, KVH * ctx * D, sigma=1.3).reshape(KVH, ctx, D)
    vc = synth.normals(seed, synth.TID_TEST_BASE + 72, KVH * ctx * D, sigma=1.3).reshape(KVH, ctx, D)
    dt = torch.float16 if kvt == "f16" else torch.float32
    kd, vd = torch.from_numpy(kc).to(dt).cuda(), torch.from_numpy(vc).to(dt).cuda()
    # the oracle reads the cache as stored (rounded to its element type)
    return torch.from_numpy(q).cuda(), kd, vd, q.astype(np.float64), kd.double().cpu().numpy(), vd.double().cpu().numpy()


PREFILL_CASES = [  # H, KVH, D, start_pos, n, kv dtype, rows checked (None = all), q scale
    (32, 8, 128, 0, 512, "f16", None, 1.0),
    (32, 8, 128, 512, 512, "f16", None, 1.0),
    (32, 8, 128, 3584, 512, "f16", [0, 1, 31, 32, 127, 128, 255, 300, 383, 384, 510, 511], 1.0),
    (32, 8, 128, 3584, 512, "f16", [0, 77, 200, 511], 4.0),  # peaky softmax
    (32, 8, 128, 30208, 512, "f32", [0, 63, 64, 255, 256, 511], 1.0),
    (32, 4, 64, 1536, 512, "f32", [0, 15, 16, 63, 64, 100, 255, 256, 400, 511], 1.0),
    (32, 8, 128, 700, 300, "f16", None, 1.0),
]


@pytest.mark.parametrize("H,KVH,D,start,n,kvt,rows,qscale", PREFILL_CASES)
def test_attention_prefill_parity(af, H, KVH, D, start, n, kvt, rows, qscale):
    ctx = start + n
    qd, kd, vd, q, kc, vc = _prefill_case(start + n, H, KVH, D, ctx, n, kvt, qscale)
    out = torch.full((n, H * D), float("nan"), dtype=torch.float32, device="cuda")
    af.af_attention_prefill(qd, kd, vd, af.KVTYPE[kvt], H, KVH, D, ctx, start, n, out)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    worst = 0.0
    for r in (range(n) if rows is None else rows):
        ref = oracle.attention(q[r], kc, vc, H, KVH, D, start + r + 1)  # row r attends to slots 0..start+r
        err = normwise_rel_err(got[r], ref)
        worst = max(worst, err)
        assert err <= ATTN_TOL, f"row {r} (position {start + r}): {err:.3e}"
    print(f"\nprefill attention H{H}/KVH{KVH}/D{D} {kvt} start {start} n {n}: worst row error {worst:.2e}")


def test_attention_prefill_rejects_bad_sizes(af):
    q = torch.zeros(4, 32 * 128, device="cuda")
    k = torch.zeros(8, 16, 128, dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    for start, n in [(0, 0), (14, 4), (-1, 2), (0, 513)]:
        with pytest.raises(af.AfError) as e:
            af.af_attention_prefill(q, k, k, af.AF_F16, 32, 8, 128, 16, start, n, out)
        assert e.value.code == af.AF_ERANGE


def test_llama3_8b_shape_two_full_chunks(af):
    """Two 512-token chunks (start 0 and 512) then 4 decode steps, Q4_0, fp16 cache, 2 layers."""
    cfg = synth.CONFIGS[3].with_(n_layers=2)
    worst = run_parity(af, cfg, synth.seed_of(3), [512, 512], 4, 1024 + 4)
    print(f"\n{cfg.name} 2 layers, 2 x 512 + 4: worst layer {worst['layer']:.2e}, logits {worst['logits']:.2e}")


def test_long_context_shape_two_full_chunks(af):
    """The Q8_0 / YaRN x4 / fp32-cache shape, 2 layers: two 512-token chunks then 4 decode steps."""
    cfg = synth.CONFIGS[4].with_(n_layers=2)
    worst = run_parity(af, cfg, synth.seed_of(4), [512, 512], 4, 1024 + 4)
    print(f"\n{cfg.name} 2 layers, 2 x 512 + 4: worst layer {worst['layer']:.2e}, logits {worst['logits']:.2e}")


def test_llama3_8b_shape_persistent_decode(af):
    """Two 512-token chunks, then 4 decode steps through the persistent kernel (Q4_0, fp16 cache, 2 layers)."""
    cfg = synth.CONFIGS[3].with_(n_layers=2)
    worst = run_parity(af, cfg, synth.seed_of(3), [512, 512], 4, 1024 + 4, decode_mode=af.AF_DECODE_PERSISTENT)
    print(f"\n{cfg.name} 2 layers, persistent decode: worst layer {worst['layer']:.2e}, logits {worst['logits']:.2e}")


def test_long_context_chunk_at_29696(af):
    """A 512-token chunk at start_pos 29696 over a seeded cache prefix (slots 0..29695, fp32 values both sides
    hold), then 2 decode steps from 30208: RoPE with the YaRN scale at t ~ 30k, attention over ~30k keys."""
    cfg = synth.CONFIGS[4].with_(n_layers=2)
    start = 29696
    KVH, D, L = cfg.n_kv_heads, cfg.head_dim, cfg.n_layers

    def prefix(om, gm):
        kc_dev, vc_dev = af.af_model_kv_cache(gm.h)
        nbytes = L * KVH * cfg.max_ctx * D * 4
        kc = _wrap_f32(kc_dev, nbytes).view(L, KVH, cfg.max_ctx, D)
        vc = _wrap_f32(vc_dev, nbytes).view(L, KVH, cfg.max_ctx, D)
        for l in range(L):
            for g in range(KVH):
                tid = synth.TID_TEST_BASE + 80 + 2 * (l * KVH + g)
                k = synth.normals(4, tid, start * D, sigma=1.3).reshape(start, D)
                v = synth.normals(4, tid + 1, start * D, sigma=1.3).reshape(start, D)
                kc[l, g, :start] = torch.from_numpy(k).cuda()
                vc[l, g, :start] = torch.from_numpy(v).cuda()
                om.kv_write(l, g, 0, k.astype(np.float64), v.astype(np.float64))
        torch.cuda.synchronize()

    for mode in (af.AF_DECODE_KERNELS, af.AF_DECODE_PERSISTENT):
        worst = run_parity(af, cfg, synth.seed_of(4), [512], 2, start + 512 + 2, start=start, prefix=prefix,
                           decode_mode=mode)
        print(f"\n{cfg.name} 2 layers, 512 at {start} + 2 (decode mode {mode}): worst layer {worst['layer']:.2e}, "
              f"logits {worst['logits']:.2e}")


def _wrap_f32(ptr, nbytes):
    """A torch float32 view of device memory the library owns (the model outlives the view)."""
    class _Cuda:
        def __init__(self, p, n):
            self.__cuda_array_interface__ = {"shape": (n // 4,), "typestr": "<f4", "data": (p, False), "version": 3}
    return torch.as_tensor(_Cuda(ptr, nbytes), device="cuda")
