"""Pins of the oracle's K-quant decoders (Q4_K, Q5_K, Q6_K super-blocks of 256 elements).

The pages name these formats (Shimmy v2.0 Architecture, "Quantization": "Q4_K_M super-block with row scales",
"Q6_K super-block, 6-bit"; the Airframe GPU pipeline's output head stored as Q6_K; dotLLM's Q4_K at about 4.5
bits per parameter) but leave the byte layout to a document they do not include, so the published GGUF layout is
the reading.  What pins it here, besides the layout itself:
  - the pages' sizes: 4.5 bits per weight for Q4_K, and the Airframe output head's ~210 MB, which is exactly
    twice the Q6_K bytes of a 32768 x 4096 matrix at 6.5625 bits per weight;
  - probes that set one field of a hand-built block and check that exactly the elements it belongs to change;
  - brute force on integer-valued matrices (exact in fp64);
  - the round trip through the generator's separately written encoder.
No GPU needed.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_worked_numbers.json")))
ONE = (0x00, 0x3C)  # fp16 1.0, little-endian
ZERO = (0x00, 0x00)


def test_kquant_sizes_match_pages():
    # Q4_K: 144 bytes per 256 weights is the page's 4.5 bits per weight
    assert synth.BLOCK_BYTES["q4_k"] * 8 / 256 == GOLD["q4_k_bits_per_weight"]["bits_per_weight"]
    assert synth.matrix("q4_k", 1, synth.TID_TEST_BASE, 3, 512).nbytes == 3 * 2 * 144
    # Q6_K: twice the bytes of the page's output head is its printed 210 (MiB)
    g = GOLD["output_weight_q6_k_32k_x_4096"]
    q6k_bytes = g["rows"] * g["cols"] // 256 * synth.BLOCK_BYTES["q6_k"]
    assert 2 * q6k_bytes == g["mib"] * 2 ** 20
    assert synth.matrix("q6_k", 1, synth.TID_TEST_BASE, 2, 768).nbytes == 2 * 3 * 210


# ---------------------------------------------------------------- Q4_K

def _q4k_block(d, dmin, s, m, nibbles):
    """One Q4_K block from 6-bit scales s[8], mins m[8] and 256 nibbles (element order)."""
    b = np.zeros(144, np.uint8)
    b[0:2], b[2:4] = d, dmin
    sc = np.zeros(12, np.int64)
    # bytes 0-3: s0..s3 (bits 0-5) + top bits of s4..s7; bytes 4-7: m0..m3 + top bits of m4..m7;
    # bytes 8-11: low nibbles of s4..s7 | low nibbles of m4..m7 << 4
    for j in range(4):
        sc[j] = s[j] + ((s[j + 4] >> 4) << 6)
        sc[4 + j] = m[j] + ((m[j + 4] >> 4) << 6)
        sc[8 + j] = (s[j + 4] & 15) + ((m[j + 4] & 15) << 4)
    b[4:16] = sc
    n = np.asarray(nibbles, np.int64).reshape(4, 2, 32)  # [group of 64][low / high half][32]
    b[16:] = (n[:, 0, :] + (n[:, 1, :] << 4)).reshape(128)
    return b


S = [1, 17, 33, 63, 5, 21, 48, 60]
M = [0, 63, 2, 40, 63, 1, 30, 16]


def test_q4_k_scale_and_min_unpacking():
    # nibbles 0: every element of sub-block j is -dmin m_j; nibbles 1: d s_j - dmin m_j (d = dmin = 1)
    v0 = oracle.dequant_row("q4_k", _q4k_block(ONE, ONE, S, M, [0] * 256), 256)
    v1 = oracle.dequant_row("q4_k", _q4k_block(ONE, ONE, S, M, [1] * 256), 256)
    for j in range(8):
        assert np.all(v0[32 * j:32 * j + 32] == -M[j])
        assert np.all(v1[32 * j:32 * j + 32] == S[j] - M[j])


@pytest.mark.parametrize("c,l", [(0, 0), (0, 31), (1, 7), (2, 20), (3, 31)])
def test_q4_k_nibble_locality(c, l):
    # d = 1, dmin = 0, all scales 1: byte 32c + l = 0xA5 sets element 64c + l to 5 and 64c + 32 + l to 10
    nib = [0] * 256
    nib[64 * c + l], nib[64 * c + 32 + l] = 5, 10
    blk = _q4k_block(ONE, ZERO, [1] * 8, [0] * 8, nib)
    assert blk[16 + 32 * c + l] == 0xA5 and np.count_nonzero(blk[16:]) == 1
    v = oracle.dequant_row("q4_k", blk, 256)
    want = np.zeros(256)
    want[64 * c + l], want[64 * c + 32 + l] = 5, 10
    assert np.array_equal(v, want)


# ---------------------------------------------------------------- Q5_K

def _q5k_block(d, dmin, s, m, codes):
    """One Q5_K block: Q4_K's header and nibble placement for the low 4 bits, the high bits in their plane."""
    codes = np.asarray(codes, np.int64)
    b4 = _q4k_block(d, dmin, s, m, codes & 15)
    qh = np.zeros(32, np.int64)
    for e in range(256):
        c, r = e // 64, e % 64
        qh[r % 32] += (codes[e] >> 4) << (2 * c + (1 if r >= 32 else 0))
    return np.concatenate([b4[:16], qh.astype(np.uint8), b4[16:]])


def test_q5_k_size_is_5_5_bits():
    assert synth.BLOCK_BYTES["q5_k"] * 8 / 256 == 5.5
    assert synth.matrix("q5_k", 1, synth.TID_TEST_BASE, 2, 512).nbytes == 2 * 2 * 176


def test_q5_k_scales_mins_and_codes():
    # codes 17 everywhere (nibble 1, high bit 1): value = 17 s_j - m_j with d = dmin = 1
    v = oracle.dequant_row("q5_k", _q5k_block(ONE, ONE, S, M, [17] * 256), 256)
    for j in range(8):
        assert np.all(v[32 * j:32 * j + 32] == 17 * S[j] - M[j])


@pytest.mark.parametrize("e", [0, 31, 32, 63, 64, 100, 150, 191, 192, 255])
def test_q5_k_high_bit_locality(e):
    # one element's high bit set (code 16): exactly that element changes (d = 1, dmin = 0, scales 1)
    codes = [0] * 256
    codes[e] = 16
    blk = _q5k_block(ONE, ZERO, [1] * 8, [0] * 8, codes)
    assert np.count_nonzero(blk[16:48]) == 1 and np.count_nonzero(blk[48:]) == 0
    want = np.zeros(256)
    want[e] = 16
    assert np.array_equal(oracle.dequant_row("q5_k", blk, 256), want)


# ---------------------------------------------------------------- Q6_K

def _q6k_block(d, scales, q):
    """One Q6_K block from 16 int8 scales and 256 six-bit codes (element order)."""
    q = np.asarray(q, np.int64)
    ql = np.zeros(128, np.int64)
    qh = np.zeros(64, np.int64)
    for e in range(256):
        h, k, l = e // 128, (e % 128) // 32, e % 32
        ql[64 * h + 32 * (k & 1) + l] += (q[e] & 15) << (0 if k < 2 else 4)
        qh[32 * h + l] += (q[e] >> 4) << (2 * k)
    return np.concatenate([ql.astype(np.uint8), qh.astype(np.uint8), np.asarray(scales, np.int8).view(np.uint8),
                           np.array(d, np.uint8)])


SC6 = [-8, -7, -6, -5, -4, -3, -2, -1, 3, 1, 2, 5, 4, 127, -128, 6]


def test_q6_k_scales_per_16_elements():
    # every code 33 (q - 32 = 1): the value is the sub-block's scale
    blk = _q6k_block(ONE, SC6, [33] * 256)
    assert np.all(blk[:128] == 0x11) and np.all(blk[128:192] == 0xAA)  # nibble 1 everywhere, high bits 2
    v = oracle.dequant_row("q6_k", blk, 256)
    assert np.array_equal(v, np.repeat(np.array(SC6, np.float64), 16))


@pytest.mark.parametrize("e", [0, 31, 32, 63, 64, 100, 127, 128, 161, 200, 255])
def test_q6_k_code_locality(e):
    # raising one element's code changes exactly that element; the low and the high parts separately
    for code in (37, 49, 0, 63):  # 37: low nibble 5; 49: high part 3; 0 and 63: the extremes
        q = [33] * 256
        q[e] = code
        v = oracle.dequant_row("q6_k", _q6k_block(ONE, SC6, q), 256)
        want = np.repeat(np.array(SC6, np.float64), 16)
        want[e] = SC6[e // 16] * (code - 32)
        assert np.array_equal(v, want), (e, code)


# ---------------------------------------------------------------- matmuls and round trip

def _int_matrix_blocks(wtype, Wi):
    """K-quant blocks whose values are the integer matrix Wi (Q4_K: 0..15, Q6_K: -32..31)."""
    N, K = Wi.shape
    out = []
    for r in range(N):
        for b in range(K // 256):
            v = Wi[r, 256 * b:256 * b + 256]
            if wtype == "q4_k":
                out.append(_q4k_block(ONE, ZERO, [1] * 8, [0] * 8, v))
            elif wtype == "q5_k":
                out.append(_q5k_block(ONE, ZERO, [1] * 8, [0] * 8, v))
            else:
                out.append(_q6k_block(ONE, [1] * 16, v + 32))
    return np.concatenate(out)


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("N,K,M", [(1, 256, 1), (3, 512, 2)])
def test_kquant_qgemm_brute_force_integers(wtype, N, K, M):
    rng = np.random.default_rng(N * 10 + K + M)
    lim = {"q4_k": (0, 16), "q5_k": (0, 32), "q6_k": (-32, 32)}[wtype]
    Wi = rng.integers(*lim, size=(N, K))
    X = rng.integers(-50, 51, size=(M, K)).astype(np.float64)
    blocks = _int_matrix_blocks(wtype, Wi)
    want = np.array([[sum(int(X[m, j]) * int(Wi[i, j]) for j in range(K)) for i in range(N)] for m in range(M)])
    assert np.array_equal(oracle.qgemm(wtype, blocks, N, K, X), want.astype(np.float64))
    assert np.array_equal(oracle.qgemv(wtype, blocks, N, K, X[0]), want[0].astype(np.float64))


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
def test_kquant_encoder_decoder_roundtrip(wtype):
    # the generator's encoder and the oracle's decoder were written separately: each decoded element lies within
    # two quantisation steps of its source (half a step of code rounding plus the rounding of the 6- or 8-bit
    # sub-block scale); a misplaced nibble, bit or scale errs by the whole value range, 15 or more steps
    N, K, sigma = 6, 512, 0.02
    W = synth.matrix(wtype, 11, synth.TID_TEST_BASE + 5, N, K, sigma=sigma)
    src = np.array([synth.normals(11, synth.TID_TEST_BASE + 5, N * K)]).reshape(N, K).astype(np.float64) * sigma
    rb = (K // 256) * synth.BLOCK_BYTES[wtype]
    err = []
    for r in range(N):
        row = oracle.dequant_row(wtype, W[r * rb:(r + 1) * rb], K)
        for sb in range(K // 32):
            w = src[r, 32 * sb:32 * sb + 32]
            if wtype in ("q4_k", "q5_k"):
                step = (w.max() - min(0.0, w.min())) / (15 if wtype == "q4_k" else 31)
            else:
                step = np.max(np.abs(w)) / 32
            assert np.max(np.abs(row[32 * sb:32 * sb + 32] - w)) <= 2 * step + 1e-7, (r, sb)
        err.append(row - src[r])
    rel_rms = np.sqrt(np.mean(np.square(err))) / sigma
    assert rel_rms < {"q4_k": 0.15, "q5_k": 0.08, "q6_k": 0.05}[wtype]


def test_kquant_layer_offsets_agree_with_generator():
    for cfg in synth.KQUANT_CONFIGS:
        assert oracle.layer_offsets(cfg) == synth.layer_offsets(cfg)


@pytest.mark.parametrize("idx", [0, 2])
def test_kquant_model_chunked_prefill_equals_unchunked(idx):
    cfg = synth.KQUANT_CONFIGS[idx]
    host = synth.HostModel(cfg, synth.kquant_seed_of(idx))
    assert host.output.nbytes == cfg.n_vocab * (cfg.n_embd // 256) * 210  # the Q6_K head
    toks = host.prompt()
    lf, _ = oracle.Model.from_host(host).forward(toks, 0)
    ch = oracle.Model.from_host(host)
    ch.forward(toks[:11], 0, want_logits=False)
    lc, _ = ch.forward(toks[11:], 11)
    assert np.array_equal(lf, lc)
    assert np.all(np.isfinite(lf)) and np.std(lf) > 0
