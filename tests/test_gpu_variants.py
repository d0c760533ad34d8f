"""GPU parity of the variants the pages mention besides the default path: the causal mask
inside the query block, a trained mask embedding, and the LM head's output scale and logit
soft cap. Whole draft + verify steps against the oracle, on the tensor-core path (bf16, with
the fused top-k LM head at 2 requests and the logits + row top-k LM head at 3) and on the
FFMA path (fp32)."""
import pytest

from synth import get_config

from test_gpu_parity import _limits, _run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_speculative_inject_gb300 import build
    build.build()


ALL = dict(block_causal=1, mask_embedding=1, output_multiplier=2.0, logit_softcap=3.0)


@pytest.mark.parametrize("lens", [[120, 37], [50, 173, 300]])
def test_variants_bf16(lens):
    cfg = get_config("mini_bf16", **ALL)
    _run_steps(cfg, _limits(max_batch=4, max_pages=32, max_positions=512, max_inject_rows=100), lens, steps=2)


def test_variants_f32():
    cfg = get_config("tiny_f32", **ALL)
    _run_steps(cfg, _limits(max_batch=1, max_pages=8, max_positions=256, max_inject_rows=64), [64], steps=2)


@pytest.mark.parametrize("var", [dict(block_causal=1), dict(mask_embedding=1),
                                 dict(output_multiplier=0.5, logit_softcap=0.2)])
def test_each_variant_alone(var):
    cfg = get_config("mini_bf16", n_layers=1, **var)
    _run_steps(cfg, _limits(max_batch=4, max_pages=16, max_positions=512, max_inject_rows=64), [90, 64], steps=1)
