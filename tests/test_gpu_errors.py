"""Error reporting and host-buffer ownership of the C ABI, on the GPU.

  * A bounded device-side wait that gives up comes back as AF_ETIMEOUT on the
    host, with no fault and no hang, and the context stays usable: the test
    hook (af_debug_stall / af_qweight_debug_stall) makes the first wait of the
    decode GEMVs poll an mbarrier that nothing arrives on, so the kernels take
    their real timeout path (error word, drain of the bulk copies in flight,
    early return).  The report clears the word: the next calls succeed and
    match the oracle again.
  * af_prefill copies its host token ids before it returns: a caller that
    overwrites its page-locked buffer right after the call gets the result of
    the ids it passed.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import QMM_TOL, gpu_model, normwise_rel_err, rms_rel_err

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


def test_qgemv_timeout_is_reported_and_cleared(af):
    N, K = 4096, 4096
    W = synth.matrix("q4_0", 3, synth.TID_TEST_BASE + 90, N, K)
    x = synth.normals(3, synth.TID_TEST_BASE + 91, K)
    h = af.af_qweight_create(af.AF_Q4_0, torch.from_numpy(W).cuda(), N, K)
    xd, y = torch.from_numpy(x).cuda(), torch.empty(N, device="cuda")
    af.af_qgemv(h, xd, y)
    assert af.af_qweight_status(h) == af.AF_OK
    af.af_qweight_debug_stall(h, 64)
    for _ in range(3):  # every launch times out; the word reports once
        af.af_qgemv(h, xd, y)
    with pytest.raises(af.AfError) as e:
        af.af_qweight_status(h)
    assert e.value.code == af.AF_ETIMEOUT
    assert af.af_qweight_status(h) == af.AF_OK  # cleared by the report
    af.af_qweight_debug_stall(h, 0)
    af.af_qgemv(h, xd, y)
    assert af.af_qweight_status(h) == af.AF_OK
    ref = oracle.qgemv("q4_0", W, N, K, x.astype(np.float64))
    assert normwise_rel_err(y.cpu().numpy(), ref) <= QMM_TOL
    af.af_qweight_destroy(h)


def test_model_timeout_is_reported_cleared_and_recovers(af):
    cfg = synth.CONFIGS[0]
    hm = synth.HostModel(cfg, synth.seed_of(0))
    gm = gpu_model(hm)
    prompt = hm.prompt(8)
    logits = torch.empty(cfg.n_vocab, device="cuda")
    gm.prefill(prompt, 0, logits)
    tok = af.af_model_sync(gm.h, want_next=True)
    af.af_debug_stall(gm.h, 64)
    with pytest.raises(af.AfError) as e:
        gm.decode(tok, 8, logits, want_next=True)
    assert e.value.code == af.AF_ETIMEOUT
    assert af.af_model_sync(gm.h) is None  # the report cleared the word
    # recovery: stall off, cache cleared, the same prompt and step again against the oracle
    af.af_debug_stall(gm.h, 0)
    af.af_reset(gm.h)
    gm.prefill(prompt, 0, logits)
    om = oracle.Model.from_host(hm)
    ref, _ = om.forward(prompt, 0)
    tok = oracle.argmax(ref)
    gm.decode(tok, 8, logits, want_next=True)
    ref, _ = om.forward([tok], 8)
    assert rms_rel_err(logits.cpu().numpy(), ref) <= 2e-2
    gm.close()


def test_prefill_host_ids_are_copied_before_return(af):
    cfg = synth.CONFIGS[0]
    hm = synth.HostModel(cfg, synth.seed_of(0))
    prompt = hm.prompt(32)
    a, b = gpu_model(hm), gpu_model(hm)
    la = torch.empty(cfg.n_vocab, device="cuda")
    lb = torch.empty(cfg.n_vocab, device="cuda")
    pinned = torch.from_numpy(prompt.copy()).pin_memory()
    buf = pinned.numpy()
    for p in range(0, 32, 8):  # each chunk's ids are overwritten right after the call returns
        buf[p:p + 8] = prompt[p:p + 8]
        af.af_prefill(a.h, buf[p:p + 8], 8, p, la if p == 24 else None)
        buf[p:p + 8] = (prompt[p:p + 8] + 7) % cfg.n_vocab
    for p in range(0, 32, 8):
        b.prefill(prompt[p:p + 8], p, lb if p == 24 else None)
    torch.cuda.synchronize()
    assert torch.equal(la, lb)
    a.close()
    b.close()
