"""Shared helpers for the parity tests: device upload of synthetic models and
the tolerances stated for this path.

Tolerances (numbers, as stated for the method):
  * standalone qgemv / qgemm: max|y - y_ref| / max|y_ref| <= 1e-3
  * layer outputs (residual stream after each layer) and logits:
      max|y - y_ref| <= 2e-2 * RMS(y_ref)
  * greedy token: equal to the oracle's wherever the oracle's top-2 logit
    margin exceeds 1e-2
  * integer work (block decode to fp32, KV slot indexing): bit-exact
"""
import numpy as np

QMM_TOL = 1e-3
LAYER_TOL = 2e-2
ARGMAX_MARGIN = 1e-2


def normwise_rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(y - ref)) / np.max(np.abs(ref)))


def rms_rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(y - ref)) / np.sqrt(np.mean(ref * ref)))


def top2_margin(logits):
    s = np.sort(np.asarray(logits, np.float64))
    return float(s[-1] - s[-2])


def to_device(hm):
    """Upload a synth.HostModel: returns dict of torch CUDA tensors (uint8 blobs, f32 norms)."""
    import torch
    dev = torch.device("cuda:0")
    return {
        "layers": [torch.from_numpy(b).to(dev) for b in hm.layers],
        "token_embd": torch.from_numpy(hm.token_embd).to(dev),
        "output_norm": torch.from_numpy(hm.output_norm).to(dev),
        "output": torch.from_numpy(hm.output).to(dev),
    }


def gpu_model(hm, max_chunk=512):
    import gguf_quantized_transformer_gb300 as af
    import torch
    d = to_device(hm)
    m = af.Model(hm.cfg, d["layers"], d["token_embd"], d["output_norm"], d["output"], max_chunk=max_chunk)
    torch.cuda.synchronize()
    del d  # the model holds its own repacked copy
    return m


def check_capture(got, ref, what, worst=None):
    """Residual stream after the embedding and after every layer: got, ref [L+1, n, E]."""
    for l in range(ref.shape[0]):
        err = rms_rel_err(got[l], ref[l])
        if worst is not None:
            worst["layer"] = max(worst.get("layer", 0.0), err)
        assert err <= LAYER_TOL, f"{what}: layer {l} err {err:.3e}"


def check_logits(got, ref, what, worst=None):
    import oracle
    err = rms_rel_err(got, ref)
    if worst is not None:
        worst["logits"] = max(worst.get("logits", 0.0), err)
    assert err <= LAYER_TOL, f"{what}: logits err {err:.3e}"
    if top2_margin(ref) > ARGMAX_MARGIN:
        assert int(np.argmax(got)) == oracle.argmax(ref), what


def run_parity(af, cfg, seed, chunks, n_decode, kv_slots, start=0, prefix=None, max_chunk=512, decode_mode=None):
    """Prefill the prompt in `chunks` from position `start`, then n_decode greedy steps under teacher forcing,
    comparing every layer's residual stream and the logits with the oracle.  prefix(om, gm), if given, fills
    cache slots [0, start) of both models before the first chunk; decode_mode, if given, is set on the GPU
    model (af_set_decode_mode).  Returns the worst errors seen."""
    import torch

    import oracle
    import synth
    hm = synth.HostModel(cfg, seed)
    prompt = hm.prompt(sum(chunks) + start)[start:]
    om = oracle.Model.from_host(hm, kv_slots=kv_slots)
    gm = gpu_model(hm, max_chunk=max_chunk)
    if decode_mode is not None:
        af.af_set_decode_mode(gm.h, decode_mode)
    if prefix is not None:
        prefix(om, gm)
    L, E, V = cfg.n_layers, cfg.n_embd, cfg.n_vocab
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    worst = {}
    p, i = start, 0
    for ci, n in enumerate(chunks):
        last = ci == len(chunks) - 1
        ref_logits, ref_cap = om.forward(prompt[i:i + n], p, want_logits=last, capture=True)
        cap = torch.empty(L + 1, n, E, dtype=torch.float32, device="cuda")
        af.af_debug_capture(gm.h, cap)
        gm.prefill(prompt[i:i + n], p, logits if last else None)
        torch.cuda.synchronize()
        check_capture(cap.cpu().numpy(), ref_cap, f"{cfg.name} prefill chunk {ci}", worst)
        if last:
            check_logits(logits.cpu().numpy(), ref_logits, f"{cfg.name} prefill logits", worst)
        p += n
        i += n
    tok = oracle.argmax(ref_logits)
    for step in range(n_decode):
        ref_logits, ref_cap = om.forward([tok], p, capture=True)
        cap = torch.empty(L + 1, 1, E, dtype=torch.float32, device="cuda")
        af.af_debug_capture(gm.h, cap)
        nxt = gm.decode(tok, p, logits, want_next=True)
        got = logits.cpu().numpy()
        check_capture(cap.cpu().numpy(), ref_cap, f"{cfg.name} decode step {step}", worst)
        check_logits(got, ref_logits, f"{cfg.name} decode step {step}", worst)
        assert nxt == int(np.argmax(got))  # device argmax = argmax of the device logits
        tok = oracle.argmax(ref_logits)  # teacher forcing
        p += 1
    gm.close()
    return worst


def device_array(ptr, shape, typestr):
    """A torch view of device memory the library owns (the owner must outlive the view)."""
    import torch

    class _Cuda:
        def __init__(self):
            n = int(np.prod(shape))
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False), "version": 3}
    return torch.as_tensor(_Cuda(), device="cuda").view(*shape)
