"""The C-ABI library loads, exports every symbol include/dflash.h declares, and its
host-only logic (config validation, status names) works without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import block_diffusion_speculative_inject_gb300 as pkg
    from block_diffusion_speculative_inject_gb300 import build as b
    b.build()
    return pkg.library()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("dflash_create", "dflash_destroy", "dflash_inject_context", "dflash_draft_step",
              "dflash_verify_greedy", "dflash_release", "dflash_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from block_diffusion_speculative_inject_gb300 import _ffi
    out = subprocess.run(["nm", "-D", "--defined-only", _ffi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dflash_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def _cfg_struct(**over):
    from block_diffusion_speculative_inject_gb300 import Limits, make_config
    from synth import get_config
    c = make_config(get_config("tiny_f32"), Limits(max_batch=2, max_pages=8, max_positions=256,
                                                   max_inject_rows=64))
    for k, v in over.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    (None, None, 0),
    ("hidden", 200, -6), ("head_dim", 96, -6), ("n_kv_heads", 3, -1), ("block_k", 0, -6),
    ("block_k", 32, -6), ("topk", 33, -6), ("topk", 0, -6), ("page_size", 32, -6),
    ("mask_token_id", 2048, -1), ("mask_token_id", -1, -1), ("max_batch", 0, -1),
    ("max_positions", 5, -1), ("dtype", 7, -1), ("n_layers", 9, -6), ("target_hidden", 96, -6),
    ("intermediate", 700, -6), ("rms_eps", -1.0, -1),
    ("block_causal", 2, -1), ("output_multiplier", -1.0, -1), ("logit_softcap", -0.5, -1),
    ("dyn_conv", 2, -1), ("selector_rank", 48, -6), ("selector_rank", 544, -6), ("selector_rank", 16, -6),
    ("selector_rank", 64, 0), ("dyn_conv", 1, 0), ("block_causal", 1, 0), ("logit_softcap", 30.0, 0),
])
def test_validate_config(lib, field, value, status):
    c = _cfg_struct(**({field: value} if field else {}))
    buf = ctypes.create_string_buffer(256)
    st = lib.dflash_validate_config(ctypes.byref(c), buf, 256)
    assert st == status, buf.value
    if status:
        assert buf.value   # a reason is given


def test_status_strings(lib):
    for s, name in [(0, b"DFLASH_OK"), (-2, b"DFLASH_ERR_OUT_OF_PAGES"), (-5, b"DFLASH_ERR_DEVICE")]:
        assert lib.dflash_status_string(s) == name


def test_null_context_calls_are_rejected(lib):
    assert lib.dflash_release(None, 1) == -1
    assert lib.dflash_truncate(None, 1, 0) == -1
    assert lib.dflash_last_error(None) == b""
    assert lib.dflash_free_pages(None) == 0
    assert lib.dflash_inject_blocks(None, None, 1, None, None, 16, None) == -1
    out = ctypes.c_void_p()
    assert lib.dflash_create(None, None, 0, ctypes.byref(out)) == -1
    assert not out.value


def test_package_fails_loudly_without_the_library(tmp_path):
    from block_diffusion_speculative_inject_gb300 import _ffi
    with pytest.raises(ImportError):
        _ffi.load(str(tmp_path / "missing.so"))


def test_context_free_calls_check_their_arguments_first(lib):
    """The tree, selector and top-k calls reject bad sizes on the host, before any CUDA call
    (so this runs without a GPU), and accept zero requests as a no-op."""
    P = None
    # dflash_ddtree_build(stream, n, L, kc, budget, ...): L in 1..31, kc in 1..32, budget in 1..1024
    for n, L, kc, budget in [(1, 0, 4, 8), (1, 32, 4, 8), (1, 7, 0, 8), (1, 7, 33, 8), (1, 7, 4, 0), (1, 7, 4, 1025),
                             (-1, 7, 4, 8)]:
        assert lib.dflash_ddtree_build(P, n, L, kc, budget, P, P, P, P, P, P, P, P, P) == -1
    assert lib.dflash_ddtree_build(P, 0, 7, 4, 8, P, P, P, P, P, P, P, P, P) == 0
    assert lib.dflash_ddtree_build(P, 2, 7, 4, 8, P, P, P, P, P, P, P, P, P) == -1      # NULL buffers
    assert lib.dflash_ddtree_walk(P, 1, 0, 8, P, P, P, P, P, P, P) == -1
    assert lib.dflash_ddtree_walk(P, 0, 7, 8, P, P, P, P, P, P, P) == 0
    # dflash_select_path(stream, n, K, kc, r, vocab, dtype, ...): r a multiple of 32 in [32, 512]
    for n, K, kc, r, V, dt in [(1, 7, 16, 48, 100, 1), (1, 7, 16, 544, 100, 1), (1, 0, 16, 64, 100, 1),
                               (1, 32, 16, 64, 100, 1), (1, 7, 33, 64, 100, 1), (1, 7, 16, 64, 0, 1),
                               (1, 7, 16, 64, 100, 5)]:
        assert lib.dflash_select_path(P, n, K, kc, r, V, dt, P, P, P, P, P, P, P, P) == -1
    assert lib.dflash_select_path(P, 0, 7, 16, 64, 100, 1, P, P, P, P, P, P, P, P) == 0
    assert lib.dflash_select_sample(P, 1, 7, 16, 64, 100, 1, ctypes.c_float(0.0), P, P, P, P, P, P, P, P, P, P, P) == -1
    assert lib.dflash_select_sample(P, 1, 7, 16, 64, 100, 1, ctypes.c_float(1.0), P, P, P, P, P, P, P, P, P, P, P) == -1
    assert lib.dflash_select_sample(P, 0, 7, 16, 64, 100, 1, ctypes.c_float(1.0), P, P, P, P, P, P, P, P, P, P, P) == 0
