"""Kernel-level parity through the C ABI: af_qgemv / af_qgemm / af_attention_decode
against the fp64 oracle on the same seeded inputs.

Bars: block decode is bit-exact (one-hot x extracts a weight column exactly);
qgemv / qgemm within 1e-3 normwise relative error; attention within 1e-3
normwise (fp32 path over an fp32/fp16 cache).  Full-size shapes are checked on
sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import QMM_TOL, normwise_rel_err

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _qweight(af, wtype, W, N, K):
    Wd = _dev(W)
    h = af.af_qweight_create(af.WTYPE[wtype], Wd, N, K)
    torch.cuda.synchronize()
    return h


# ---------------------------------------------------------------- block decode: bit-exact

@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_dequant_bit_exact_via_onehot(af, wtype):
    N, K = 64, 1024 + 64 if wtype == "q4_0" else 576
    W = synth.matrix(wtype, 11, synth.TID_TEST_BASE + 1, N, K)
    # hand-built first row: negative, zero and unit scales
    bb = synth.BLOCK_BYTES[wtype]
    W[0:2] = np.frombuffer(np.uint16(0xBC00).tobytes(), np.uint8)     # d = -1.0
    W[bb:bb + 2] = np.frombuffer(np.uint16(0x0000).tobytes(), np.uint8)  # d = 0
    h = _qweight(af, wtype, W, N, K)
    rb = (K // 32) * bb
    ref = np.stack([oracle.dequant_row(wtype, W[r * rb:(r + 1) * rb], K) for r in range(N)])  # [N, K]
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    for j in [0, 1, 15, 16, 17, 31, 32, 100, K - 33, K - 1]:
        x = torch.zeros(K, dtype=torch.float32, device="cuda")
        x[j] = 1.0
        af.af_qgemv(h, x, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.array_equal(got, ref[:, j].astype(np.float32)), (j, np.abs(got - ref[:, j]).max())
    af.af_qweight_destroy(h)


# ---------------------------------------------------------------- qgemv

GEMV_SHAPES = [(2, 32), (6, 96), (64, 1024), (1024, 512), (2816, 512), (512, 1408), (2560, 2048), (130, 5632)]


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", GEMV_SHAPES)
def test_qgemv_parity(af, wtype, N, K):
    W = synth.matrix(wtype, 21, synth.TID_TEST_BASE + 2, N, K)
    x = synth.normals(21, synth.TID_TEST_BASE + 3, K)
    h = _qweight(af, wtype, W, N, K)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    ref = oracle.qgemv(wtype, W, N, K, x.astype(np.float64))
    got = y.cpu().numpy()
    assert normwise_rel_err(got, ref) <= QMM_TOL
    # repeated calls reuse the scratch counters: same answer (deterministic order)
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), got)
    af.af_qweight_destroy(h)


FULL_SHAPES = [(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336), (128256, 4096)]


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", FULL_SHAPES)
def test_qgemv_full_size_sampled_rows(af, wtype, N, K):
    W = synth.matrix(wtype, 31, synth.TID_TEST_BASE + 4, N, K)
    x = synth.normals(31, synth.TID_TEST_BASE + 5, K)
    h = _qweight(af, wtype, W, N, K)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, 1, N - 2, N - 1], rng.integers(0, N, 300)]))
    ref = oracle.qgemv_rows(wtype, W, K, rows, x.astype(np.float64))
    got = y.cpu().numpy()[rows]
    assert normwise_rel_err(got, ref) <= QMM_TOL
    af.af_qweight_destroy(h)


# ---------------------------------------------------------------- qgemm

GEMM_CASES = [(1, 64, 64), (3, 2, 32), (7, 130, 96), (64, 256, 512), (130, 1024, 512), (512, 512, 1408),
              (200, 2816, 512), (512, 2560, 2048)]


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M,N,K", GEMM_CASES)
def test_qgemm_parity(af, wtype, M, N, K):
    W = synth.matrix(wtype, 41, synth.TID_TEST_BASE + 6, N, K)
    X = synth.normals(41, synth.TID_TEST_BASE + 7, M * K).reshape(M, K)
    h = _qweight(af, wtype, W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    ref = oracle.qgemm(wtype, W, N, K, X.astype(np.float64))
    got = Y.cpu().numpy()
    for m in range(M):
        assert normwise_rel_err(got[m], ref[m]) <= QMM_TOL, m
    af.af_qweight_destroy(h)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_qgemm_near_fp32(af, wtype):
    """The tensor-core GEMM splits X and W into fp16 hi + lo parts; with all three
    cross products kept the result is within a few fp32 roundings of the exact sum,
    far inside the 1e-3 bar (a dropped lo term would show up as ~1e-4)."""
    M, N, K = 130, 512, 2048
    W = synth.matrix(wtype, 43, synth.TID_TEST_BASE + 6, N, K)
    X = synth.normals(43, synth.TID_TEST_BASE + 7, M * K).reshape(M, K)
    h = _qweight(af, wtype, W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    ref = oracle.qgemm(wtype, W, N, K, X.astype(np.float64))
    got = Y.cpu().numpy()
    worst = max(normwise_rel_err(got[m], ref[m]) for m in range(M))
    assert worst <= 2e-5, worst
    af.af_qweight_destroy(h)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", [(6144, 4096), (28672, 4096), (4096, 14336)])
def test_qgemm_full_size_sampled(af, wtype, N, K):
    M = 512
    W = synth.matrix(wtype, 51, synth.TID_TEST_BASE + 8, N, K)
    X = synth.normals(51, synth.TID_TEST_BASE + 9, M * K).reshape(M, K)
    h = _qweight(af, wtype, W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 64)]))
    for m in [0, 1, 255, 510, 511]:
        ref = oracle.qgemv_rows(wtype, W, K, rows, X[m].astype(np.float64))
        assert normwise_rel_err(got[m, rows], ref) <= QMM_TOL, m
    af.af_qweight_destroy(h)


# ---------------------------------------------------------------- attention (decode)

ATTN_CASES = [  # H, KVH, D, ctx, pos, kv dtype
    (8, 4, 64, 64, 0, "f32"), (8, 4, 64, 64, 31, "f32"), (8, 4, 64, 64, 63, "f32"),
    (32, 4, 64, 2048, 2047, "f32"), (32, 8, 64, 4096, 1000, "f16"), (32, 8, 128, 8192, 4351, "f16"),
    (32, 8, 128, 32768, 30720, "f32"), (32, 8, 128, 32768, 30783, "f32"), (16, 16, 128, 300, 299, "f16"),
    # one kv head: many splits, split length not dividing the sequence; ragged last tile
    (8, 1, 64, 10000, 9728, "f16"), (8, 1, 128, 4096, 4000, "f32"), (2, 2, 64, 200, 130, "f32"),
    # group 8 with head_dim 128 and group 2 on either path; a cache just above the cluster path's
    (64, 8, 128, 8192, 5000, "f16"), (64, 8, 128, 2048, 1500, "f16"), (16, 8, 64, 3000, 2999, "f32"),
    (16, 8, 64, 1024, 1000, "f16"), (32, 8, 128, 2049, 2048, "f16"),
]


@pytest.mark.parametrize("H,KVH,D,ctx,pos,kvt", ATTN_CASES)
def test_attention_decode_parity(af, H, KVH, D, ctx, pos, kvt):
    seed = 61 + pos
    q = synth.normals(seed, synth.TID_TEST_BASE + 10, H * D)
    n = pos + 1
    k = synth.normals(seed, synth.TID_TEST_BASE + 11, KVH * n * D).reshape(KVH, n, D)
    v = synth.normals(seed, synth.TID_TEST_BASE + 12, KVH * n * D).reshape(KVH, n, D)
    dt = np.float16 if kvt == "f16" else np.float32
    kc = np.zeros((KVH, ctx, D), dt)
    vc = np.zeros((KVH, ctx, D), dt)
    kc[:, :n] = k.astype(dt)
    vc[:, :n] = v.astype(dt)
    kc[:, n:] = 1e4 if kvt == "f32" else 6e4  # slots past pos must be ignored
    out = torch.empty(H * D, dtype=torch.float32, device="cuda")
    af.af_attention_decode(_dev(q), _dev(kc), _dev(vc), af.KVTYPE[kvt], H, KVH, D, ctx, pos, out)
    ref = oracle.attention(q.astype(np.float64), kc[:, :n].astype(np.float64), vc[:, :n].astype(np.float64),
                           H, KVH, D, n)
    got = out.cpu().numpy()
    assert normwise_rel_err(got, ref) <= 1e-3
    if pos == 0:  # a single position returns V_0 (exactly, up to fp32 rounding of 1*v)
        want = np.repeat(vc[:, 0].astype(np.float32), H // KVH, axis=0).reshape(-1)
        assert np.allclose(got, want, rtol=1e-6, atol=0)


def test_attention_errors(af):
    q = torch.zeros(8 * 64, device="cuda")
    kv = torch.zeros(4 * 16 * 64, device="cuda")
    with pytest.raises(af.AfError) as e:
        af.af_attention_decode(q, kv, kv, af.AF_F32, 8, 4, 64, 16, 16, q)
    assert e.value.code == af.AF_ERANGE
    with pytest.raises(af.AfError) as e:
        af.af_attention_decode(q, kv, kv, af.AF_F32, 8, 4, 96, 16, 3, q)
    assert e.value.code == af.AF_ENOTIMPL
