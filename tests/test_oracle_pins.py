"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks an oracle function against something other than itself:
values the pages print (tests/golden/page_worked_numbers.json), blocks whose
values are known by construction, closed forms, invariants and brute force on
integer-valued inputs (exact in fp64).  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_worked_numbers.json")))


# ---------------------------------------------------------------- formats

@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14),
                                      (0x7BFF, 65504.0), (0x3555, 0.333251953125), (0x8000, -0.0),
                                      (0x03FF, 1023 * 2.0 ** -24)])
def test_f16_decode_known_values(bits, val):
    assert oracle.f16_to_double(bits) == val


def test_f16_rounding_matches_numpy():
    # numpy's double->half conversion is a correctly rounded library routine
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(2000) * s for s in (1e-7, 1e-5, 1e-3, 1.0, 100.0, 3e4)])
    xs = np.concatenate([xs, [1 + 2 ** -11, 1 + 3 * 2 ** -11, 65519.0, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    for x in xs:
        assert oracle.round_f16(float(x)) == float(np.float16(x)), x


def test_encoder_scale_rounding_matches_numpy():
    # the generator stores block scales as fp16 RNE from fp32
    rng = np.random.default_rng(2)
    for x in (rng.standard_normal(500) * 1e-3).astype(np.float32):
        assert synth.f16_bits(float(x)) == int(np.float16(x).view(np.uint16))


# ---------------------------------------------------------------- dequant

def test_q8_0_identity_block():
    d = 0x3C00  # 1.0
    q = np.array(list(range(-127, -127 + 32)), dtype=np.int8)
    blk = np.concatenate([np.frombuffer(np.uint16(d).tobytes(), np.uint8), q.view(np.uint8)])
    assert np.array_equal(oracle.dequant_row("q8_0", blk, 32), q.astype(np.float64))


@pytest.mark.parametrize("name,wtype", [("q8_0_block_example", "q8_0"), ("q4_0_block_example", "q4_0")])
def test_dequant_worked_blocks(name, wtype):
    g = GOLD[name]
    blk = np.frombuffer(bytes.fromhex(g["block_hex"]), dtype=np.uint8)
    assert np.array_equal(oracle.dequant_row(wtype, blk, 32), np.array(g["values"], dtype=np.float64))


def test_q4_0_nibble_order_and_offset():
    # low nibble of byte j -> element j; high nibble -> element j + 16; value d * (n - 8)
    d = 0x4000  # 2.0
    lo = np.arange(16, dtype=np.uint8)            # elements 0..15 get n = 0..15
    hi = (15 - np.arange(16)).astype(np.uint8)    # elements 16..31 get n = 15..0
    blk = np.concatenate([np.frombuffer(np.uint16(d).tobytes(), np.uint8), lo | (hi << 4)])
    want = 2.0 * (np.concatenate([np.arange(16), 15 - np.arange(16)]) - 8)
    assert np.array_equal(oracle.dequant_row("q4_0", blk, 32), want)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_negative_and_zero_scale(wtype):
    qb = 32 if wtype == "q8_0" else 16
    body = (np.arange(qb) * 7 % 256).astype(np.uint8)
    for dbits, dval in ((0xBC00, -1.0), (0x0000, 0.0), (0x8000, -0.0)):
        blk = np.concatenate([np.frombuffer(np.uint16(dbits).tobytes(), np.uint8), body])
        out = oracle.dequant_row(wtype, blk, 32)
        if wtype == "q8_0":
            want = dval * body.view(np.int8).astype(np.float64)
        else:
            n = np.concatenate([body & 15, body >> 4]).astype(np.float64)
            want = dval * (n - 8)
        assert np.array_equal(out, want)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_encoder_decoder_roundtrip_bound(wtype):
    # the generator's encoder and the oracle's decoder were written separately:
    # decoded values must sit within half a quantisation step of the source
    K, N = 256, 8
    W = synth.matrix(wtype, 7, synth.TID_TEST_BASE, N, K, sigma=0.02)
    bb = synth.BLOCK_BYTES[wtype]
    for r in range(N):
        row = oracle.dequant_row(wtype, W[r * (K // 32) * bb:(r + 1) * (K // 32) * bb], K)
        for b in range(K // 32):
            blk = W[(r * (K // 32) + b) * bb:(r * (K // 32) + b + 1) * bb]
            d = abs(oracle.f16_to_double(int(blk[0]) | (int(blk[1]) << 8)))
            vals = row[b * 32:(b + 1) * 32]
            if wtype == "q8_0":
                assert np.max(np.abs(vals)) <= 127 * d * (1 + 1e-12)
            else:
                # the extreme element maps to nibble 0: value -8 * d_signed = the extreme
                assert np.max(np.abs(vals)) == pytest.approx(8 * d, rel=0, abs=0)


# ---------------------------------------------------------------- matmuls

def _int_blocks(q_int, wtype):
    """GGUF blocks with d = 1.0 holding the given integer matrix (values fixed by construction)."""
    N, K = q_int.shape
    out = []
    one = np.frombuffer(np.uint16(0x3C00).tobytes(), np.uint8)
    for r in range(N):
        for b in range(K // 32):
            v = q_int[r, b * 32:(b + 1) * 32]
            if wtype == "q8_0":
                out += [one, v.astype(np.int8).view(np.uint8)]
            else:
                n = (v + 8).astype(np.uint8)
                out += [one, (n[:16] | (n[16:] << 4)).astype(np.uint8)]
    return np.concatenate(out)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K,M", [(1, 32, 1), (3, 32, 2), (4, 64, 3), (2, 96, 1)])
def test_qgemm_brute_force_integers(wtype, N, K, M):
    rng = np.random.default_rng(N * 100 + K + M)
    lim = (-127, 128) if wtype == "q8_0" else (-8, 8)
    Wi = rng.integers(*lim, size=(N, K))
    X = rng.integers(-50, 51, size=(M, K)).astype(np.float64)
    blocks = _int_blocks(Wi, wtype)
    Y = oracle.qgemm(wtype, blocks, N, K, X)
    want = np.array([[sum(int(X[m, j]) * int(Wi[i, j]) for j in range(K)) for i in range(N)] for m in range(M)])
    assert np.array_equal(Y, want.astype(np.float64))
    y = oracle.qgemv(wtype, blocks, N, K, X[0])
    assert np.array_equal(y, want[0].astype(np.float64))
    rows = np.array([N - 1, 0])
    assert np.array_equal(oracle.qgemv_rows(wtype, blocks, K, rows, X[0]), want[0][rows].astype(np.float64))


# ---------------------------------------------------------------- norm, rope, silu, softmax, attention

def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, 0.3, 1e-5
    w = (1.0 + 0.01 * np.arange(n)).astype(np.float32)
    y = oracle.rmsnorm(np.full(n, c), w, eps)
    want = w.astype(np.float64) * c / math.sqrt(c * c + eps)
    assert np.allclose(y, want, rtol=1e-15, atol=0)


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(512)
    w = np.ones(512, np.float32)
    y = oracle.rmsnorm(x, w, 0.0)
    assert math.isclose(np.sqrt(np.mean(y * y)), 1.0, rel_tol=1e-13)
    assert np.allclose(oracle.rmsnorm(1000 * x, w, 0.0), y, rtol=1e-13)


def test_yarn_scale():
    assert oracle.yarn_scale(32768, 8192) == 4.0
    assert oracle.yarn_scale(2048, 2048) == 1.0
    assert oracle.yarn_scale(1024, 2048) == 1.0


def test_rope_theta_worked_values():
    for cs in GOLD["rope_theta_yarn"]["cases"]:
        ys = oracle.yarn_scale(cs["max_ctx"], cs["native_ctx"])
        th = oracle.rope_theta(cs["t"], cs["i"], cs["head_dim"], cs["base"], ys)
        assert th == pytest.approx(cs["theta"], rel=1e-14, abs=1e-300)


def test_rope_identity_at_t0_and_norm_preserving():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(4 * 64)
    assert np.array_equal(oracle.rope(v, 4, 64, 0, 10000.0, 1.0), v)
    r = oracle.rope(v, 4, 64, 777, 10000.0, 1.0)
    assert np.allclose(np.hypot(r[0::2], r[1::2]), np.hypot(v[0::2], v[1::2]), rtol=1e-14)
    assert not np.allclose(r, v)


def test_rope_pair_rotation_closed_form():
    # one head, D = 2: the single pair rotates by theta(t, 0) = t / yarn_scale
    t, ys = 3, 2.0
    r = oracle.rope([1.0, 0.0], 1, 2, t, 10000.0, ys)
    assert r[0] == pytest.approx(math.cos(1.5), abs=1e-15) and r[1] == pytest.approx(math.sin(1.5), abs=1e-15)


def test_rope_relative_position():
    # rot(q, t) . rot(k, s) depends on (t - s) / yarn_scale only
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for ys in (1.0, 4.0):
        a = oracle.rope(q, 1, 64, 100, 500000.0, ys) @ oracle.rope(k, 1, 64, 90, 500000.0, ys)
        b = oracle.rope(q, 1, 64, 1010, 500000.0, ys) @ oracle.rope(k, 1, 64, 1000, 500000.0, ys)
        assert a == pytest.approx(b, rel=1e-10)
    # yarn_scale 4 at t equals scale 1 at t / 4
    assert np.allclose(oracle.rope(q, 1, 64, 400, 500000.0, 4.0), oracle.rope(q, 1, 64, 100, 500000.0, 1.0),
                       rtol=1e-13, atol=1e-15)


def test_silu_properties():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    for g in (-3.0, -0.5, 0.25, 2.0, 7.0):
        assert oracle.silu(g) - oracle.silu(-g) == pytest.approx(g, rel=1e-14)  # g*s(g) + g*s(-g) = g
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_softmax_properties():
    rng = np.random.default_rng(6)
    s = rng.standard_normal(1000) * 10
    p = oracle.softmax(s)
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.allclose(oracle.softmax(s + 1234.5), p, rtol=1e-9)
    assert np.allclose(oracle.softmax(np.zeros(7)), np.full(7, 1 / 7), rtol=1e-15)
    two = oracle.softmax([0.7, -0.3])
    assert two[0] == pytest.approx(1 / (1 + math.exp(-1.0)), rel=1e-15)


def test_attention_single_key_returns_v0():
    rng = np.random.default_rng(7)
    H, KVH, D, S = 8, 4, 64, 5
    q = rng.standard_normal(H * D)
    kc, vc = rng.standard_normal((KVH, S, D)), rng.standard_normal((KVH, S, D))
    out = oracle.attention(q, kc, vc, H, KVH, D, 1).reshape(H, D)
    for h in range(H):
        assert np.array_equal(out[h], vc[h // (H // KVH), 0])


def test_attention_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(8)
    H, KVH, D, S = 4, 2, 32, 9
    q = rng.standard_normal(H * D)
    kc = np.broadcast_to(rng.standard_normal((KVH, 1, D)), (KVH, S, D)).copy()
    vc = rng.standard_normal((KVH, S, D))
    out = oracle.attention(q, kc, vc, H, KVH, D, S).reshape(H, D)
    for h in range(H):
        assert np.allclose(out[h], vc[h // 2].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_attention_two_keys_closed_form():
    D = 16
    q = np.zeros(D); q[0] = 2.0
    kc = np.zeros((1, 2, D)); kc[0, 0, 0] = 1.0; kc[0, 1, 0] = -1.0   # scores +-2/sqrt(D) = +-0.5
    vc = np.zeros((1, 2, D)); vc[0, 0, 1] = 1.0; vc[0, 1, 2] = 1.0
    out = oracle.attention(q, kc, vc, 1, 1, D, 2)
    a0 = 1 / (1 + math.exp(-1.0))
    assert out[1] == pytest.approx(a0, rel=1e-15) and out[2] == pytest.approx(1 - a0, rel=1e-15)


def test_gqa_equals_mha_with_duplicated_kv():
    rng = np.random.default_rng(9)
    H, KVH, D, S = 8, 2, 16, 6
    q = rng.standard_normal(H * D)
    kc, vc = rng.standard_normal((KVH, S, D)), rng.standard_normal((KVH, S, D))
    gqa = oracle.attention(q, kc, vc, H, KVH, D, S)
    mha = oracle.attention(q, np.repeat(kc, H // KVH, 0), np.repeat(vc, H // KVH, 0), H, H, D, S)
    assert np.array_equal(gqa, mha)


def test_attention_causal_prefix_only():
    # keys beyond n_keys must not influence the result
    rng = np.random.default_rng(10)
    H, KVH, D, S = 2, 1, 8, 10
    q = rng.standard_normal(H * D)
    kc, vc = rng.standard_normal((KVH, S, D)), rng.standard_normal((KVH, S, D))
    a = oracle.attention(q, kc, vc, H, KVH, D, 4)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, 4:] = 99.0; vc2[:, 4:] = -99.0
    assert np.array_equal(a, oracle.attention(q, kc2, vc2, H, KVH, D, 4))


# ---------------------------------------------------------------- sizes the pages print

def test_kv_bytes_worked_examples():
    for key in ("kv_cache_tinyllama_2048_f32", "kv_cache_llama3_8b_f16_maxseq4096"):
        g = GOLD[key]
        cfg = synth.CONFIGS[1].with_(n_layers=g["n_layers"], n_kv_heads=g["n_kv_heads"], max_ctx=g["max_ctx"],
                                     head_dim=g["head_dim"], n_heads=32,
                                     kv_dtype="f32" if g["elem_bytes"] == 4 else "f16")
        assert oracle.kv_bytes(cfg) == g["bytes"]
    assert oracle.kv_bytes(synth.CONFIGS[1]) == 92274688
    assert oracle.kv_bytes(synth.CONFIGS[3]) == 1073741824
    assert oracle.kv_bytes(synth.CONFIGS[2]) == 134217728


def test_layer_offsets_agree_with_generator():
    for cfg in synth.CONFIGS:
        assert oracle.layer_offsets(cfg) == synth.layer_offsets(cfg)
        off = oracle.layer_offsets(cfg)
        assert all(o % 256 == 0 for o in off)


# ---------------------------------------------------------------- whole model invariants

@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS[0]
    return synth.HostModel(cfg, synth.seed_of(0))


def test_chunked_prefill_equals_unchunked_bit_exact(tiny):
    toks = tiny.prompt()
    full = oracle.Model.from_host(tiny)
    lf, cf = full.forward(toks, 0, capture=True)
    ch = oracle.Model.from_host(tiny)
    ch.forward(toks[:8], 0, want_logits=False)
    ch.forward(toks[8:20], 8, want_logits=False)
    lc, cc = ch.forward(toks[20:], 20, capture=True)
    assert np.array_equal(lf, lc)
    assert np.array_equal(cf[:, 20:], cc)


def test_decode_after_prefill_equals_full_prefill(tiny):
    toks = tiny.prompt()
    a = oracle.Model.from_host(tiny)
    la, _ = a.forward(toks, 0)
    b = oracle.Model.from_host(tiny)
    b.forward(toks[:-1], 0, want_logits=False)
    lb, _ = b.forward(toks[-1:], len(toks) - 1)
    assert np.array_equal(la, lb)


def test_thread_count_does_not_change_results(tiny):
    toks = tiny.prompt()[:9]
    l1, c1 = oracle.Model.from_host(tiny).forward(toks, 0, capture=True, nthreads=1)
    l8, c8 = oracle.Model.from_host(tiny).forward(toks, 0, capture=True, nthreads=7)
    assert np.array_equal(l1, l8) and np.array_equal(c1, c8)


def test_embedding_capture_is_dequantized_row(tiny):
    cfg = tiny.cfg
    toks = tiny.prompt()[:3]
    _, cap = oracle.Model.from_host(tiny).forward(toks, 0, want_logits=False, capture=True)
    rb = (cfg.n_embd // 32) * synth.BLOCK_BYTES[cfg.wtype]
    for r, t in enumerate(toks):
        assert np.array_equal(cap[0, r], oracle.dequant_row(cfg.wtype, tiny.token_embd[t * rb:(t + 1) * rb],
                                                            cfg.n_embd))


def test_kv_slots_written_exactly_and_rounded(tiny):
    cfg = tiny.cfg.with_(kv_dtype="f16")
    m = oracle.Model(cfg, tiny.layers, tiny.token_embd, tiny.output_norm, tiny.output)
    toks = tiny.prompt()[:5]
    m.forward(toks, 3, want_logits=False)  # slots 3..7 written, the rest stay zero
    for l in range(cfg.n_layers):
        for g in range(cfg.n_kv_heads):
            for p in range(cfg.max_ctx):
                k, v = m.kv_read(l, g, p)
                written = 3 <= p < 8
                assert bool(np.any(k != 0)) == written and bool(np.any(v != 0)) == written
                if written:
                    assert all(oracle.round_f16(x) == x for x in k)


def test_kv_write_sets_the_slots_forward_reads(tiny):
    """A cache prefix set with kv_write is the one the next chunk attends to: copying the slots a real prefill
    wrote into a fresh model gives the same continuation, bit for bit (and kv_read returns what was set)."""
    cfg = tiny.cfg
    toks = tiny.prompt()
    a = oracle.Model.from_host(tiny)
    a.forward(toks[:20], 0, want_logits=False)
    la, ca = a.forward(toks[20:], 20, capture=True)
    b = oracle.Model.from_host(tiny)
    for l in range(cfg.n_layers):
        for g in range(cfg.n_kv_heads):
            kv = [a.kv_read(l, g, p) for p in range(20)]
            k = np.stack([x[0] for x in kv])
            v = np.stack([x[1] for x in kv])
            b.kv_write(l, g, 0, k, v)
            assert all(np.array_equal(b.kv_read(l, g, p)[0], k[p]) for p in range(20))
    lb, cb = b.forward(toks[20:], 20, capture=True)
    assert np.array_equal(la, lb) and np.array_equal(ca, cb)
    # a different prefix changes the continuation (the setter is not a no-op)
    b.kv_write(0, 0, 3, np.ones((1, cfg.head_dim)), np.ones((1, cfg.head_dim)))
    lc, _ = b.forward(toks[20:], 20)
    assert not np.array_equal(la, lc)
    with pytest.raises(IndexError):
        b.kv_write(0, 0, cfg.max_ctx - 1, np.ones((2, cfg.head_dim)), np.ones((2, cfg.head_dim)))


def test_rope_position_matters_in_model(tiny):
    # same token at two different positions with an empty cache otherwise: K differs only by the rotation
    cfg = tiny.cfg
    m1 = oracle.Model.from_host(tiny)
    m2 = oracle.Model.from_host(tiny)
    tok = tiny.prompt()[:1]
    m1.forward(tok, 0, want_logits=False)
    m2.forward(tok, 5, want_logits=False)
    k0, v0 = m1.kv_read(0, 0, 0)
    k5, v5 = m2.kv_read(0, 0, 5)
    assert np.array_equal(v0, v5)                       # V is position-free
    ys = oracle.yarn_scale(cfg.max_ctx, cfg.native_ctx)
    rot = oracle.rope(k0, 1, cfg.head_dim, 5, cfg.rope_base, ys)  # k0 is unrotated at t = 0
    assert np.allclose(rot, k5, rtol=0, atol=1e-6)      # f32 cache rounding


def test_dispatch_count_arithmetic():
    g = GOLD["dispatch_count_tinyllama"]
    assert g["n_layers"] * 6 == g["matmul_dispatches"]
    assert g["matmul_dispatches"] + 4 * g["n_layers"] == g["total_dispatches"]


# ---------------------------------------------------------------- sampler chain (Airframe GPU pipeline)

def test_sample_uniform_logits_picks_floor_u_v():
    # equal logits, no nucleus cut: the order is by index and each token has mass 1/V
    V = 10
    for u, want in [(0.0, 0), (0.05, 0), (0.15, 1), (0.47, 4), (0.999, 9)]:
        t, lo, hi = oracle.sample(np.zeros(V), [], 1.0, 1.0, 1.0, u)
        assert t == want, (u, t)
        assert lo <= u <= hi


def test_sample_greedy_at_zero_temperature_with_penalty():
    logits = np.arange(10, dtype=np.float64)
    assert oracle.sample(logits, [], 1.0, 0.0, 1.0, 0.7)[0] == 9
    # token 9 divided by 2 -> 4.5: token 8 wins; duplicates in the recent list divide once
    assert oracle.sample(logits, [9], 2.0, 0.0, 1.0, 0.7)[0] == 8
    assert oracle.sample(logits, [9, 9, 9, 8], 2.0, 0.0, 1.0, 0.7)[0] == 7  # 9 -> 4.5, 8 -> 4, 7 wins
    # penalty <= 1 is off
    assert oracle.sample(logits, [9], 1.0, 0.0, 1.0, 0.7)[0] == 9


def test_sample_two_tokens_closed_form():
    a, b, T = 1.3, 0.4, 0.7
    p0 = 1.0 / (1.0 + np.exp((b - a) / T))  # token 0 is the more probable one
    assert oracle.sample(np.array([a, b]), [], 1.0, T, 1.0, p0 - 1e-9)[0] == 0
    assert oracle.sample(np.array([a, b]), [], 1.0, T, 1.0, p0 + 1e-9)[0] == 1


def test_sample_nucleus_cut_and_renormalization():
    probs = np.array([0.2, 0.5, 0.3])
    logits = np.log(probs)
    # sorted: 1 (0.5), 2 (0.3), 0 (0.2); top_p 0.75 keeps {1, 2} (0.5 < 0.75 <= 0.8), mass 0.8
    assert oracle.sample(logits, [], 1.0, 1.0, 0.75, 0.6)[0] == 1   # target 0.48 <= 0.5
    assert oracle.sample(logits, [], 1.0, 1.0, 0.75, 0.7)[0] == 2   # target 0.56 in (0.5, 0.8]
    assert oracle.sample(logits, [], 1.0, 1.0, 0.75, 0.999)[0] == 2  # token 0 is never drawn
    # a tiny top_p keeps only the most probable token
    for u in (0.0, 0.5, 0.999):
        assert oracle.sample(logits, [], 1.0, 1.0, 1e-9, u)[0] == 1


def test_sample_high_temperature_approaches_uniform():
    logits = np.array([3.0, 0.0, -2.0, 1.0])
    t, lo, hi = oracle.sample(logits, [], 1.0, 1e6, 1.0, 0.6)
    # near-equal masses, still ordered by probability: 0, 3, 1, 2 -> the third one
    assert t == 1 and abs(lo - 0.5) < 1e-5 and abs(hi - 0.75) < 1e-5


def test_sample_interval_contains_the_draw():
    logits = synth.normals(9, synth.TID_TEST_BASE + 32, 500) * 2.0
    for top_p in (1.0, 0.9, 0.3):
        for u in (0.0, 0.2, 0.61, 0.97):
            t, lo, hi = oracle.sample(logits, [3, 4], 1.2, 0.9, top_p, u)
            inn, lo2, hi2, pt, pb = oracle.sample_interval(logits, [3, 4], 1.2, 0.9, top_p, t)
            assert inn and (lo2, hi2) == (lo, hi) and lo <= u <= hi and pt >= pb
