"""af_attention_decode_static (the allocation-free decode attention entry point)
against af_attention_decode, through the C ABI.

Both run the same kernel with the same split count, so results must be
bit-identical.  Two calls in a row with different inputs check that the fixed
scratch (arrival counters) is left ready for the next call.  Kept in a file of
its own, collected last, so it also runs after every other GPU test in one
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


CALLS = [  # two calls in a row each: H, KVH, D, ctx, pos, kv dtype
    [(32, 8, 128, 4096, 4095, "f16"), (32, 8, 128, 4096, 1000, "f16")],
    [(8, 4, 64, 512, 511, "f32"), (64, 8, 128, 2048, 2047, "f32")],
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
