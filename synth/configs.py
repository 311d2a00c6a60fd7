"""Model shapes and workloads of the five synthetic decoders.

Shapes follow the models the cited pages run: a tiny 2-layer decoder, a
TinyLlama-1.1B shape (the Airframe GPU-pipeline page's KV-cache example), a
Llama-3.2-1B shape and a Llama-3-8B shape (the dotLLM "GPU Inference" page's
VRAM-estimation table), plus the 8B shape with the YaRN extended context of the
Shimmy v2.0 Architecture page ("Extended Context (YaRN)").

Pure data: no arithmetic of the method lives here.
"""
from dataclasses import dataclass, asdict, replace

Q8_0 = "q8_0"
Q4_0 = "q4_0"
Q4_K = "q4_k"
Q5_K = "q5_k"
Q6_K = "q6_k"
BASE_SEED = 20261202


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    n_embd: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    n_ff: int
    n_vocab: int
    wtype: str          # "q8_0" | "q4_0" | "q4_k" | "q5_k" | "q6_k": every layer matrix and token_embd
    kv_dtype: str       # "f32" | "f16" (and, for the oracle, "q8_0" | "q4_0": quantized with an fp16 window)
    max_ctx: int
    native_ctx: int     # == max_ctx means no YaRN scaling
    rope_base: float
    rms_eps: float = 1e-5
    # workload
    prompt_len: int = 0
    chunk: int = 512
    n_decode: int = 0
    w_sigma: float = 0.02
    norm_sigma: float = 0.1
    out_wtype: str = ""  # the LM head's block type ("" = wtype)
    kv_window: int = 0   # quantized caches: slots kept fp16 behind a step's last position

    @property
    def head_wtype(self) -> str:
        return self.out_wtype or self.wtype

    def as_dict(self):
        return asdict(self)

    def with_(self, **kw):
        return replace(self, **kw)


CONFIGS = [
    ModelConfig("tiny-2L-q8_0", 2, 512, 8, 4, 64, 1408, 2048, Q8_0, "f32", 64, 64, 10000.0,
                prompt_len=32, chunk=512, n_decode=16),
    ModelConfig("tinyllama-1.1b-shape-q8_0", 22, 2048, 32, 4, 64, 5632, 32000, Q8_0, "f32", 2048, 2048, 10000.0,
                prompt_len=2048, chunk=512, n_decode=128),
    ModelConfig("llama-3.2-1b-shape-q4_0", 16, 2048, 32, 8, 64, 8192, 128256, Q4_0, "f16", 4096, 4096, 500000.0,
                prompt_len=1024, chunk=512, n_decode=256),
    ModelConfig("llama-3-8b-shape-q4_0", 32, 4096, 32, 8, 128, 14336, 128256, Q4_0, "f16", 8192, 8192, 500000.0,
                prompt_len=4096, chunk=512, n_decode=256),
    ModelConfig("llama-3-8b-shape-q8_0-yarn4", 32, 4096, 32, 8, 128, 14336, 128256, Q8_0, "f32", 32768, 8192,
                500000.0, prompt_len=30720, chunk=512, n_decode=64),
]


# K-quant models in the Q4_K_M mix the pages run (dotLLM, VRAM Estimation: "Llama 3 8B, Q4_K_M"): Q4_K
# layer matrices and embedding, a Q6_K LM head (Airframe GPU pipeline, output head stored as Q6_K).
KQUANT_CONFIGS = [
    ModelConfig("tiny-2L-q4_k_m", 2, 512, 8, 4, 64, 1536, 2048, Q4_K, "f32", 64, 64, 10000.0,
                prompt_len=32, chunk=512, n_decode=16, out_wtype=Q6_K),
    ModelConfig("llama-3-8b-shape-q4_k_m", 32, 4096, 32, 8, 128, 14336, 128256, Q4_K, "f16", 8192, 8192, 500000.0,
                prompt_len=4096, chunk=512, n_decode=256, out_wtype=Q6_K),
    # the Q5_K_M mix (Shimmy v2.0 Architecture, Quantization: "Q5_K_M super-block, 5-bit with high-bit plane")
    ModelConfig("tiny-2L-q5_k_m", 2, 512, 8, 4, 64, 1536, 2048, Q5_K, "f16", 64, 64, 10000.0,
                prompt_len=32, chunk=512, n_decode=16, out_wtype=Q6_K),
]


def seed_of(index: int) -> int:
    return BASE_SEED + index


def kquant_seed_of(index: int) -> int:
    return BASE_SEED + 100 + index
