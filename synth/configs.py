"""Draft-model shapes and workload recipes.

Each entry is a draft model shape (the DFlash draft: shared embedding, fc +
RMSNorm context fusion, a few Qwen3-style decoder layers, shared LM head) plus
the workload it is exercised with: batch size, context-length mix, how many
newly accepted positions each step injects, and the probability with which the
synthetic target agrees with the draft's argmax.

The five named workloads are:
  tiny_f32   fp32, hidden 256, 2 layers, 4/2 heads x 64, SwiGLU 768, vocab 2048,
             3 features (768 -> 256 fc), batch 1, context 64, K=7
  q8b_b1     Qwen3-8B-shaped bf16 draft (5 layers, hidden 4096, 32/8 heads x 128,
             SwiGLU 12288, vocab 151936, 5 features 20480 -> 4096), batch 1,
             context 2048, K=15
  q8b_b32    the same draft, batch 32, ragged contexts U[512, 8192], K=15,
             1..16 newly injected positions per request per step, 64-token pages
  q4b_b128   Qwen3-4B-shaped bf16 draft (hidden 2560, 32/8 heads x 128, SwiGLU
             9728, 5 features 12800 -> 2560), batch 128, context 1024, K=7
  q27b_b8    27B-target-shaped bf16 draft (hidden 5120, 40/8 heads x 128, SwiGLU
             17408, 5 features 25600 -> 5120), batch 8, context 32768, K=15,
             full prefill then 64 draft+verify steps
plus `mini_bf16`, a small bf16 shape (ragged vocabulary, ragged contexts) that the
oracle finishes in seconds, used for element-by-element parity.
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class DraftConfig:
    name: str
    dtype: str              # "f32" or "bf16": storage / GEMM operand type
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    n_feat: int             # number of target layers whose hidden states are fused
    target_hidden: int      # width of each target hidden state
    block_k: int            # K mask positions; the query block has K+1 rows
    topk: int = 16
    mask_token_id: int = -1  # -1 -> vocab - 1
    qk_norm: int = 1
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    input_embedding_scale: float = 1.0
    # variants the pages mention besides the default path
    block_causal: int = 0           # 1: causal mask inside the query block
    output_multiplier: float = 1.0  # logits scale
    logit_softcap: float = 0.0      # > 0: logits = c * tanh(logits / c) after the scale
    mask_embedding: int = 0         # 1: a trained mask embedding replaces E[mask_id]
    dyn_conv: int = 0               # 1: DFlash 2 two-tap dynamic convolutions in every layer
    selector_rank: int = 0          # r > 0: DFlash 2 path selector with rank-r codebooks
    # workload
    batch: int = 1
    ctx_min: int = 64
    ctx_max: int = 64
    n_new_max: int = 16      # newly accepted positions per request per step: U[1, n_new_max]
    accept_p: float = 0.6    # synthetic target agrees with the draft argmax with this probability
    steps: int = 1           # consecutive draft+verify steps in one workload
    verify_driven: bool = False  # n_new = accept_len + 1 from the real verify (else drawn)

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_token_id < 0 else self.mask_token_id

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def feat_dim(self) -> int:
        return self.n_feat * self.target_hidden

    def layer_params(self) -> int:
        h, q, kv, i = self.hidden, self.q_dim, self.kv_dim, self.intermediate
        return h * (q + 2 * kv) + q * h + 3 * h * i + 2 * h + 2 * self.head_dim


CONFIGS = {
    "tiny_f32": DraftConfig(
        name="tiny_f32", dtype="f32", hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2,
        head_dim=64, intermediate=768, vocab=2048, n_feat=3, target_hidden=256, block_k=7,
        mask_token_id=2047, batch=1, ctx_min=64, ctx_max=64, n_new_max=8, accept_p=0.7),
    "mini_bf16": DraftConfig(
        name="mini_bf16", dtype="bf16", hidden=512, n_layers=2, n_q_heads=8, n_kv_heads=2,
        head_dim=128, intermediate=1408, vocab=5000, n_feat=3, target_hidden=384, block_k=15,
        batch=3, ctx_min=50, ctx_max=300, n_new_max=16, accept_p=0.6),
    "q8b_b1": DraftConfig(
        name="q8b_b1", dtype="bf16", hidden=4096, n_layers=5, n_q_heads=32, n_kv_heads=8,
        head_dim=128, intermediate=12288, vocab=151936, n_feat=5, target_hidden=4096,
        block_k=15, batch=1, ctx_min=2048, ctx_max=2048, n_new_max=16, accept_p=0.6),
    "q8b_b32": DraftConfig(
        name="q8b_b32", dtype="bf16", hidden=4096, n_layers=5, n_q_heads=32, n_kv_heads=8,
        head_dim=128, intermediate=12288, vocab=151936, n_feat=5, target_hidden=4096,
        block_k=15, batch=32, ctx_min=512, ctx_max=8192, n_new_max=16, accept_p=0.6),
    "q4b_b128": DraftConfig(
        name="q4b_b128", dtype="bf16", hidden=2560, n_layers=5, n_q_heads=32, n_kv_heads=8,
        head_dim=128, intermediate=9728, vocab=151936, n_feat=5, target_hidden=2560,
        block_k=7, batch=128, ctx_min=1024, ctx_max=1024, n_new_max=8, accept_p=0.6),
    "q27b_b8": DraftConfig(
        name="q27b_b8", dtype="bf16", hidden=5120, n_layers=5, n_q_heads=40, n_kv_heads=8,
        head_dim=128, intermediate=17408, vocab=151936, n_feat=5, target_hidden=5120,
        block_k=15, batch=8, ctx_min=32768, ctx_max=32768, n_new_max=16, accept_p=0.6,
        steps=64, verify_driven=True),
}


def get_config(name: str, **overrides) -> DraftConfig:
    cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg
