"""af_attention_decode_static (the allocation-free decode attention entry point)
against af_attention_decode, through the C ABI.

Both run the same kernel with the same split count, so results must be
bit-identical.  Two calls in a row with different inputs check that the fixed
scratch (arrival counters) is left ready for the next call; two calls queued
back to back on one stream, with no synchronisation between them, check the
documented use (the second launch may start while the first still runs, and
waits for it before it touches the shared scratch).  Kept in a file of its
own, collected last, so it also runs after every other GPU test in one
process.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import normwise_rel_err

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


def _case(seed, H, KVH, D, ctx, kvt):
    q = synth.normals(seed, synth.TID_TEST_BASE + 20, H * D)
    kc = synth.normals(seed, synth.TID_TEST_BASE + 21, KVH * ctx * D).reshape(KVH, ctx, D)
    vc = synth.normals(seed, synth.TID_TEST_BASE + 22, KVH * ctx * D).reshape(KVH, ctx, D)
    dt = torch.float16 if kvt == "f16" else torch.float32
    return (torch.from_numpy(q).cuda(), torch.from_numpy(kc).to(dt).cuda(), torch.from_numpy(vc).to(dt).cuda(),
            q, kc, vc)


CALLS = [  # two calls in a row each: H, KVH, D, ctx, pos, kv dtype (above 2048 slots: the split path, which uses
    # the fixed scratch; up to 2048: the cluster path)
    [(32, 8, 128, 12288, 12287, "f16"), (32, 8, 128, 12288, 1000, "f16")],
    [(8, 4, 64, 512, 511, "f32"), (64, 8, 128, 2048, 2047, "f32")],
    [(32, 4, 64, 3000, 2999, "f32"), (32, 8, 128, 2048, 2047, "f16")],
]


@pytest.mark.parametrize("calls", CALLS)
def test_static_matches_allocating_entry_point(af, calls):
    for i, (H, KVH, D, ctx, pos, kvt) in enumerate(calls):
        qd, kd, vd, q, kc, vc = _case(61 + i, H, KVH, D, ctx, kvt)
        want = torch.empty(H * D, dtype=torch.float32, device="cuda")
        got = torch.full((H * D,), float("nan"), dtype=torch.float32, device="cuda")
        af.af_attention_decode(qd, kd, vd, af.KVTYPE[kvt], H, KVH, D, ctx, pos, want)
        af.af_attention_decode_static(qd, kd, vd, af.KVTYPE[kvt], H, KVH, D, ctx, pos, got)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {i}"
        # and both against the oracle at the attention bar (slots 0..pos of the cache as stored)
        n = pos + 1
        kq = kd.float().cpu().numpy()[:, :n].astype(np.float64)
        vq = vd.float().cpu().numpy()[:, :n].astype(np.float64)
        ref = oracle.attention(q.astype(np.float64), kq, vq, H, KVH, D, n)
        assert normwise_rel_err(got.cpu().numpy(), ref) <= 1e-3, f"call {i}"


def test_static_back_to_back_on_one_stream(af):
    """Two split-path calls (caches above 2048 slots) with different inputs and kv-head counts queued on one
    stream with no synchronisation between them; one sync, then both against the allocating entry point and the
    oracle."""
    calls = [(32, 8, 128, 4096, 4000, "f16"), (32, 4, 64, 3072, 3071, "f32")]
    cases, outs = [], []
    s = torch.cuda.Stream()
    for i, (H, KVH, D, ctx, pos, kvt) in enumerate(calls):
        cases.append(_case(71 + i, H, KVH, D, ctx, kvt))
        outs.append(torch.full((H * D,), float("nan"), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    for (H, KVH, D, ctx, pos, kvt), (qd, kd, vd, *_), o in zip(calls, cases, outs):
        af.af_attention_decode_static(qd, kd, vd, af.KVTYPE[kvt], H, KVH, D, ctx, pos, o, s)
    s.synchronize()
    for (H, KVH, D, ctx, pos, kvt), (qd, kd, vd, q, kc, vc), got in zip(calls, cases, outs):
        want = torch.empty(H * D, dtype=torch.float32, device="cuda")
        af.af_attention_decode(qd, kd, vd, af.KVTYPE[kvt], H, KVH, D, ctx, pos, want)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        n = pos + 1
        kq = kd.float().cpu().numpy()[:, :n].astype(np.float64)
        vq = vd.float().cpu().numpy()[:, :n].astype(np.float64)
        ref = oracle.attention(q.astype(np.float64), kq, vq, H, KVH, D, n)
        assert normwise_rel_err(got.cpu().numpy(), ref) <= 1e-3


def test_static_scratch_limit_applies_to_the_split_path_only(af):
    """The cluster path (caches of up to 2048 slots) uses none of the fixed scratch, so a kv-head count above its
    counters is accepted there and refused on the split path."""
    H, KVH, D = 1032, 1032, 64
    q = torch.zeros(H * D, device="cuda")
    out = torch.empty(H * D, device="cuda")
    k = torch.zeros(KVH * 2049 * D, dtype=torch.float16, device="cuda")
    af.af_attention_decode_static(q, k, k, af.AF_F16, H, KVH, D, 2048, 5, out)
    torch.cuda.synchronize()
    with pytest.raises(af.AfError) as e:
        af.af_attention_decode_static(q, k, k, af.AF_F16, H, KVH, D, 2049, 5, out)
    assert e.value.code == af.AF_ERANGE
