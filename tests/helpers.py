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
