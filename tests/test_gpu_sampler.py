"""The on-device sampler chain (af_sample) against the oracle.

Where the draw is decided by floating point (the nucleus boundary, the crossing
of u times the nucleus mass) the GPU sums in fp32 and the oracle in fp64, so the
GPU's token must be the oracle's token for u or top_p moved by a hair; where the
result is fixed exactly (equal logits, greedy with clear margins) it must match.
"""
import numpy as np
import pytest

import oracle
import synth

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


def _run(af, logits, recent, pen, temp, top_p, u):
    ld = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    r = np.ascontiguousarray(recent, dtype=np.int32)
    rd = torch.from_numpy(r).cuda() if r.size else None
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    af.af_sample(ld, ld.numel(), rd, r.size, pen, temp, top_p, u, tok)
    torch.cuda.synchronize()
    return int(tok.item())


def test_equal_logits_pick_by_index(af):
    V = 128256
    for u in (0.0, 0.123456, 0.5, 0.987654):
        # token k has cumulative mass (k + 1) / V: the first with (k + 1) >= u V (u as the float32 passed)
        want = oracle.sample(np.zeros(V), [], 1.0, 1.0, 1.0, float(np.float32(u)))[0]
        assert want == max(0, int(np.ceil(float(np.float32(u)) * V)) - 1)
        assert _run(af, np.zeros(V), [], 1.0, 1.0, 1.0, u) == want


def test_greedy_with_penalty_matches_oracle(af):
    rng = np.random.default_rng(3)
    for V in (1000, 128256):
        logits = synth.normals(5, synth.TID_TEST_BASE + 30 + V % 7, V).astype(np.float32) * 3
        top = np.argsort(-logits)[:8]
        recent = np.concatenate([top[:3], top[:2], rng.integers(0, V, 20)])
        want = oracle.sample(logits.astype(np.float64), recent, 1.7, 0.0, 1.0, 0.3)[0]
        assert _run(af, logits, recent, 1.7, 0.0, 1.0, 0.3) == want
        # ties at the maximum go to the lowest index
        tied = logits.copy()
        tied[[5, 9, 700]] = tied.max() + 1.0
        assert _run(af, tied, [], 1.0, 0.0, 0.9, 0.3) == 5


CASES = [  # penalty, temperature, top_p
    (1.0, 1.0, 1.0), (1.3, 0.8, 0.95), (1.1, 0.5, 0.5), (1.0, 2.0, 0.99), (1.5, 0.7, 0.1), (1.0, 1.0, 1e-6),
]


@pytest.mark.parametrize("pen,temp,top_p", CASES)
def test_sampling_matches_oracle(af, pen, temp, top_p):
    V = 128256
    logits = synth.normals(7, synth.TID_TEST_BASE + 31, V).astype(np.float32) * 2.5
    recent = np.argsort(-logits)[:16][::2].astype(np.int32)
    l64 = logits.astype(np.float64)
    for u in (0.0, 0.01, 0.3, 0.5, 0.77, 0.9999):
        got = _run(af, logits, recent, pen, temp, top_p, u)
        if got == oracle.sample(l64, recent, pen, temp, top_p, u)[0]:
            continue
        # otherwise the GPU's token must sit where fp32 sums can move the crossing: its cumulative interval
        # (oracle, fp64) within 1e-4 of u, and inside the nucleus up to the same slack at its boundary
        inn, lo, hi, pt, pb = oracle.sample_interval(l64, recent, pen, temp, top_p, got)
        assert lo - 1e-4 <= u <= hi + 1e-4, (u, got, lo, hi)
        inn_wide = oracle.sample_interval(l64, recent, pen, temp, min(top_p + 1e-4, 1.0), got)[0]
        assert inn or inn_wide, (u, got, pt, pb)


@pytest.mark.parametrize("V", [1, 5, 9, 1000, 32003, 262144])
def test_vocab_sizes_and_ragged_slices(af, V):
    """Vocabularies smaller than the CTA count (empty slices), ragged slice ends and the maximum size."""
    logits = synth.normals(9, synth.TID_TEST_BASE + 32, V).astype(np.float32) * 2.0
    l64 = logits.astype(np.float64)
    recent = np.arange(0, V, max(1, V // 5))[:8].astype(np.int32)
    assert _run(af, logits, recent, 1.2, 0.0, 1.0, 0.5) == oracle.sample(l64, recent, 1.2, 0.0, 1.0, 0.5)[0]
    for top_p, u in ((1.0, 0.61), (0.9, 0.2), (0.9, 0.999)):
        got = _run(af, logits, recent, 1.2, 0.9, top_p, u)
        assert 0 <= got < V
        if got == oracle.sample(l64, recent, 1.2, 0.9, top_p, u)[0]:
            continue
        inn, lo, hi, _, _ = oracle.sample_interval(l64, recent, 1.2, 0.9, top_p, got)
        assert lo - 1e-4 <= u <= hi + 1e-4, (V, u, got, lo, hi)
        assert inn or oracle.sample_interval(l64, recent, 1.2, 0.9, min(top_p + 1e-4, 1.0), got)[0]
    # equal logits over a ragged vocabulary: the tie group spans every non-empty slice
    for u in (0.0, 0.4, 0.9999):
        want = max(0, int(np.ceil(float(np.float32(u)) * V)) - 1)
        got = _run(af, np.zeros(V), [], 1.0, 1.0, 1.0, u)
        assert abs(got - want) <= max(1, V // 100000), (V, u, got, want)


def test_on_device_sampled_decode_loop(af):
    """Prefill, then decode steps fed by af_model_sample: the drawn token goes into the model's next-token word
    and af_decode_step(-1) consumes it from the device.  Each token is a valid draw from that step's logits,
    and every step's logits match the oracle fed the same tokens."""
    from helpers import LAYER_TOL, gpu_model, rms_rel_err
    cfg = synth.CONFIGS[0]
    hm = synth.HostModel(cfg, synth.seed_of(0))
    gm = gpu_model(hm)
    om = oracle.Model.from_host(hm)
    prompt = hm.prompt()
    logits = torch.empty(cfg.n_vocab, dtype=torch.float32, device="cuda")
    gm.prefill(prompt, 0, logits)
    ref, _ = om.forward(prompt, 0)
    p = len(prompt)
    rec = prompt[-8:].astype(np.int32)
    recent = torch.from_numpy(rec).cuda()
    for u in (0.1, 0.5, 0.9, 0.33, 0.77, 0.05):
        tok = af.af_model_sample(gm.h, logits, recent, 8, 1.1, 0.8, 0.95, u, want_token=True)
        got = logits.cpu().numpy().astype(np.float64)
        assert rms_rel_err(got, ref) <= LAYER_TOL
        inn, lo, hi, _, _ = oracle.sample_interval(got, rec, 1.1, 0.8, 0.95, tok)
        assert lo - 1e-4 <= u <= hi + 1e-4, (u, tok, lo, hi)
        assert inn or oracle.sample_interval(got, rec, 1.1, 0.8, 0.95 + 1e-4, tok)[0]
        gm.decode(-1, p, logits)  # the drawn token, fed from the device
        ref, _ = om.forward([tok], p)
        p += 1
    gm.close()
