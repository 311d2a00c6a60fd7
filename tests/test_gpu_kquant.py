"""K-quant (Q4_K, Q5_K, Q6_K) kernels through the C ABI against the fp64 oracle.

Same bars as the Q4_0 / Q8_0 kernels: the GEMV's decode of a weight is bit-exact (a one-hot x extracts
a weight column exactly, since d s_j n - dmin m_j and d c (q - 32) are formed with one rounding); qgemv
and qgemm within 1e-3 normwise; full-size shapes on sampled rows.  K is a whole number of 256-weight
super-blocks, and shapes whose K is not a whole GEMV chunk exercise the zero padding.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import QMM_TOL, normwise_rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KTYPES = ["q4_k", "q5_k", "q6_k"]


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
    h = af.af_qweight_create(af.WTYPE[wtype], _dev(W), N, K)
    torch.cuda.synchronize()
    return h


def _rows(wtype, W, N, K):
    rb = (K // 256) * synth.BLOCK_BYTES[wtype]
    return np.stack([oracle.dequant_row(wtype, W[r * rb:(r + 1) * rb], K) for r in range(N)])


@pytest.mark.parametrize("wtype", KTYPES)
def test_kquant_decode_bit_exact_via_onehot(af, wtype):
    N, K = 64, 1280  # five super-blocks: the row is padded to 2048 weights
    W = synth.matrix(wtype, 61, synth.TID_TEST_BASE + 20, N, K)
    # hand-edited first super-block of row 0: a negative d; of row 1: zero d (and dmin)
    if wtype in ("q4_k", "q5_k"):
        bb = synth.BLOCK_BYTES[wtype]
        W[0:2] = np.frombuffer(np.uint16(0xBC00).tobytes(), np.uint8)
        W[bb:bb + 4] = 0
    else:
        W[208:210] = np.frombuffer(np.uint16(0xBC00).tobytes(), np.uint8)
        W[(K // 256) * 210 + 208:(K // 256) * 210 + 210] = 0
    h = _qweight(af, wtype, W, N, K)
    ref = _rows(wtype, W, N, K)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    for j in [0, 1, 15, 16, 17, 31, 32, 63, 64, 100, 127, 128, 255, 256, 700, K - 33, K - 1]:
        x = torch.zeros(K, dtype=torch.float32, device="cuda")
        x[j] = 1.0
        af.af_qgemv(h, x, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.array_equal(got, ref[:, j].astype(np.float32)), (j, np.abs(got - ref[:, j]).max())
    af.af_qweight_destroy(h)


GEMV_SHAPES = [(2, 256), (6, 768), (64, 1024), (1024, 512), (2816, 512), (512, 1536), (2560, 2048), (130, 5632)]


@pytest.mark.parametrize("wtype", KTYPES)
@pytest.mark.parametrize("N,K", GEMV_SHAPES)
def test_kquant_qgemv_parity(af, wtype, N, K):
    W = synth.matrix(wtype, 71, synth.TID_TEST_BASE + 21, N, K)
    x = synth.normals(71, synth.TID_TEST_BASE + 22, K)
    h = _qweight(af, wtype, W, N, K)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    ref = oracle.qgemv(wtype, W, N, K, x.astype(np.float64))
    got = y.cpu().numpy()
    assert normwise_rel_err(got, ref) <= QMM_TOL
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), got)
    af.af_qweight_destroy(h)


@pytest.mark.parametrize("wtype,N,K", [("q4_k", 6144, 4096), ("q4_k", 28672, 4096), ("q4_k", 4096, 14336),
                                       ("q4_k", 128256, 4096), ("q6_k", 128256, 4096), ("q6_k", 4096, 14336),
                                       ("q5_k", 28672, 4096), ("q5_k", 4096, 14336)])
def test_kquant_qgemv_full_size_sampled_rows(af, wtype, N, K):
    W = synth.matrix(wtype, 81, synth.TID_TEST_BASE + 23, N, K)
    x = synth.normals(81, synth.TID_TEST_BASE + 24, K)
    h = _qweight(af, wtype, W, N, K)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    af.af_qgemv(h, _dev(x), y)
    torch.cuda.synchronize()
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, 1, N - 2, N - 1], rng.integers(0, N, 300)]))
    ref = oracle.qgemv_rows(wtype, W, K, rows, x.astype(np.float64))
    assert normwise_rel_err(y.cpu().numpy()[rows], ref) <= QMM_TOL
    af.af_qweight_destroy(h)


GEMM_CASES = [(1, 64, 256), (3, 2, 256), (7, 130, 512), (64, 256, 512), (130, 1024, 512), (512, 512, 1536),
              (200, 2816, 512), (512, 2560, 2048)]


@pytest.mark.parametrize("wtype", KTYPES)
@pytest.mark.parametrize("M,N,K", GEMM_CASES)
def test_kquant_qgemm_parity(af, wtype, M, N, K):
    W = synth.matrix(wtype, 91, synth.TID_TEST_BASE + 25, N, K)
    X = synth.normals(91, synth.TID_TEST_BASE + 26, M * K).reshape(M, K)
    h = _qweight(af, wtype, W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    ref = oracle.qgemm(wtype, W, N, K, X.astype(np.float64))
    got = Y.cpu().numpy()
    for m in range(M):
        assert normwise_rel_err(got[m], ref[m]) <= QMM_TOL, m
    af.af_qweight_destroy(h)


@pytest.mark.parametrize("wtype", KTYPES)
def test_kquant_qgemm_near_fp32(af, wtype):
    """K-quant weights are formed in fp32 and split into fp16 hi + rounded lo (relative error ~2^-22): the
    GEMM stays within a few fp32 roundings of the exact sum."""
    M, N, K = 130, 512, 2048
    W = synth.matrix(wtype, 93, synth.TID_TEST_BASE + 25, N, K)
    X = synth.normals(93, synth.TID_TEST_BASE + 26, M * K).reshape(M, K)
    h = _qweight(af, wtype, W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    ref = oracle.qgemm(wtype, W, N, K, X.astype(np.float64))
    got = Y.cpu().numpy()
    worst = max(normwise_rel_err(got[m], ref[m]) for m in range(M))
    assert worst <= 2e-5, worst
    af.af_qweight_destroy(h)


@pytest.mark.parametrize("N,K", [(6144, 4096), (28672, 4096), (4096, 14336)])
def test_q4_k_qgemm_full_size_sampled(af, N, K):
    M = 512
    W = synth.matrix("q4_k", 95, synth.TID_TEST_BASE + 27, N, K)
    X = synth.normals(95, synth.TID_TEST_BASE + 28, M * K).reshape(M, K)
    h = _qweight(af, "q4_k", W, N, K)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    af.af_qgemm(h, _dev(X), M, Y)
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 64)]))
    for m in [0, 1, 255, 510, 511]:
        ref = oracle.qgemv_rows("q4_k", W, K, rows, X[m].astype(np.float64))
        assert normwise_rel_err(got[m, rows], ref) <= QMM_TOL, m
    af.af_qweight_destroy(h)


def test_kquant_rejects_partial_super_blocks(af):
    W = _dev(np.zeros(4 * 144, np.uint8))
    with pytest.raises(af.AfError) as ei:
        af.af_qweight_create(af.AF_Q4_K, W, 4, 128)
    assert ei.value.code == af.AF_EINVAL
