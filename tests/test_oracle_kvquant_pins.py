"""Pins of the oracle's quantized KV cache (Q8_0 / Q4_0 with an fp16 window).

dotLLM's CUDA components name a quantized KV cache "Q8_0/Q4_0 + FP16 window" and nothing more; the reading
(stated in oracle.cpp): a slot is written in fp16, and once it lies more than kv_window positions behind a
step's last position it is replaced by the Q8_0 / Q4_0 quantization of those fp16 values, per 32-element block
along head_dim; a step is never longer than the window.  Pinned here by rows on the quantization grid (reproduced exactly), the quantization-step bound,
a window that covers the whole sequence (bit-exact equality with the fp16 cache), and the slot-by-slot state of
layer 0, whose K/V rows do not depend on attention.  No GPU needed.
"""
import numpy as np
import pytest

import oracle
import synth


def f16(x):
    return np.asarray(x, np.float16).astype(np.float64)


def test_q8_0_row_on_grid_is_exact():
    q = np.array([127, -127, 5, 0, -64] + [3] * 27, np.float64)
    v = np.concatenate([q, -q]) * 2.0 ** -7  # max |v| / 127 = 2^-7, exact in fp16
    assert np.array_equal(oracle.quant_kv_row("q8_0", v), v)


def test_q4_0_row_on_grid_is_exact():
    c = np.array([-8, 7, 0, 3, -1] + [2] * 27, np.float64)  # the extreme element -8 d sets d = 0.25
    v = np.concatenate([c, c[::-1]]) * 0.25
    assert np.array_equal(oracle.quant_kv_row("q4_0", v), v)


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_zero_rows_stay_zero(kvt):
    assert np.array_equal(oracle.quant_kv_row(kvt, np.zeros(64)), np.zeros(64))


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_quantization_step_bound(kvt):
    rng = np.random.default_rng(5)
    for _ in range(50):
        v = f16(rng.standard_normal(128) * rng.uniform(0.01, 10))
        out = oracle.quant_kv_row(kvt, v)
        for b in range(0, 128, 32):
            blk, got = v[b:b + 32], out[b:b + 32]
            if kvt == "q8_0":
                d = float(np.float16(np.float32(np.max(np.abs(blk))) / np.float32(127)))
                assert np.max(np.abs(got - blk)) <= 0.56 * d  # half a step, plus the fp16 rounding of d
            else:
                m = blk[np.argmax(np.abs(blk))]
                d = abs(float(np.float16(np.float32(m) / np.float32(-8))))
                assert np.max(np.abs(got - blk)) <= 1.01 * d  # the far end of the range clamps within one step


def _model(kv_dtype, kv_window, slots=48):
    cfg = synth.CONFIGS[0].with_(kv_dtype=kv_dtype, kv_window=kv_window)
    hm = synth.HostModel(cfg, synth.seed_of(0))
    return hm, oracle.Model.from_host(hm, kv_slots=slots)


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_window_covering_the_sequence_equals_fp16_cache(kvt):
    hm, q = _model(kvt, 64)
    _, f = _model("f16", 0)
    toks = hm.prompt(20)
    lq, cq = q.forward(toks, 0, capture=True)
    lf, cf = f.forward(toks, 0, capture=True)
    assert np.array_equal(lq, lf) and np.array_equal(cq, cf)


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_layer0_slots_quantized_exactly_outside_the_window(kvt):
    W = 5
    hm, q = _model(kvt, W)
    _, f = _model("f16", 0)
    toks = hm.prompt(21)
    for p in range(0, 20, 5):  # chunks no longer than the window
        q.forward(toks[p:p + 5], p)
        f.forward(toks[p:p + 5], p)
    b = 19
    for s in range(20):
        for g in range(hm.cfg.n_kv_heads):
            kq, vq = q.kv_read(0, g, s)
            kf, vf = f.kv_read(0, g, s)  # layer 0's K/V rows do not depend on attention
            if s <= b - W:
                assert np.array_equal(kq, oracle.quant_kv_row(kvt, kf)), (s, g)
                assert np.array_equal(vq, oracle.quant_kv_row(kvt, vf)), (s, g)
            else:
                assert np.array_equal(kq, kf) and np.array_equal(vq, vf), (s, g)
    # the next step retires exactly one more slot, quantized once (from its fp16 values)
    q.forward(toks[20:21], 20)
    f.forward(toks[20:21], 20)
    s = 20 - W
    kq, _ = q.kv_read(0, 0, s)
    kf, _ = f.kv_read(0, 0, s)
    assert np.array_equal(kq, oracle.quant_kv_row(kvt, kf))
    kq, _ = q.kv_read(0, 0, s + 1)
    kf, _ = f.kv_read(0, 0, s + 1)
    assert np.array_equal(kq, kf)


def test_small_window_deviation_grows_with_coarser_codes():
    # with a 2-slot window (chunks of 2, then decode steps) most slots are quantized: the logits move away from
    # the fp16 cache's, less for the 8-bit codes than for the 4-bit ones
    hm, _ = _model("q8_0", 2)
    toks = hm.prompt(24)

    def run(kvt):
        _, m = _model(kvt, 2 if kvt != "f16" else 0)
        for p in range(0, 20, 2):
            m.forward(toks[p:p + 2], p, want_logits=False)
        for p in range(20, 24):
            lg, _ = m.forward(toks[p:p + 1], p)
        return lg
    lf = run("f16")
    dev = {kvt: np.max(np.abs(run(kvt) - lf)) / np.sqrt(np.mean(lf ** 2)) for kvt in ("q8_0", "q4_0")}
    assert 0 < dev["q8_0"] < dev["q4_0"] < 1.0, dev


@pytest.mark.parametrize("kvt", ["q8_0", "q4_0"])
def test_step_longer_than_the_window_is_refused(kvt):
    hm, q = _model(kvt, 4)
    with pytest.raises(ValueError):
        q.forward(hm.prompt(5), 0)
    q.forward(hm.prompt(4), 0)  # a chunk of exactly the window is fine


def test_quantized_kv_bytes():
    # Llama-3-8B shape, 8192 slots: 32 layers x 8 kv heads x (K, V) rows of 128 values per slot, each slot held
    # in fp16 (256 B) and in the Q8_0 store (4 blocks of 34 B: "Shimmy v2.0 Architecture", Quantization) or the
    # Q4_0 store (4 blocks of 18 B).  Hand-computed: 512 rows x 8192 slots x (256 + 136) B and x (256 + 72) B.
    cfg = synth.CONFIGS[3].with_(kv_dtype="q8_0", kv_window=512)
    assert oracle.kv_bytes(cfg) == 1_644_167_168
    assert oracle.kv_bytes(cfg.with_(kv_dtype="q4_0")) == 1_375_731_712
