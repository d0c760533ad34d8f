"""ctypes declarations of include/dflash.h (argument marshalling only)."""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash.so")

OK = 0
STATUS = {0: "DFLASH_OK", -1: "DFLASH_ERR_INVALID_ARG", -2: "DFLASH_ERR_OUT_OF_PAGES",
          -3: "DFLASH_ERR_UNKNOWN_REQUEST", -4: "DFLASH_ERR_CUDA", -5: "DFLASH_ERR_DEVICE",
          -6: "DFLASH_ERR_UNSUPPORTED"}
F32, BF16 = 0, 1


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab",
        "n_feat", "target_hidden", "block_k", "topk", "mask_token_id", "qk_norm", "max_batch",
        "max_requests", "max_pages", "page_size", "max_positions", "max_inject_rows")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("input_embedding_scale", ctypes.c_float), ("dtype", ctypes.c_int32),
        ("block_causal", ctypes.c_int32), ("output_multiplier", ctypes.c_float),
        ("logit_softcap", ctypes.c_float), ("dyn_conv", ctypes.c_int32), ("selector_rank", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm", "w_gate", "w_up",
        "w_down", "conv_base", "conv_proj")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("fc", ctypes.c_void_p),
                ("fc_norm", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights)), ("mask_embedding", ctypes.c_void_p),
                ("sel_pred_codebook", ctypes.c_void_p), ("sel_succ_codebook", ctypes.c_void_p),
                ("sel_hidden_proj", ctypes.c_void_p)]


class DraftOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("argmax", "topk_idx", "topk_val", "logits", "lse", "selected")] + [
        ("sel_temperature", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("sel_uniform", "sel_q_tok", "sel_q_p", "sel_q_n")]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I32P = ctypes.POINTER(ctypes.c_int32)

SIGNATURES = {
    "dflash_validate_config": (_I32, [ctypes.POINTER(Config), ctypes.c_char_p, _I32]),
    "dflash_create": (_I32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), _I32, ctypes.POINTER(_P)]),
    "dflash_destroy": (None, [_P]),
    "dflash_inject_context": (_I32, [_P, _P, _I32, _I32P, _I32P, _I32, ctypes.POINTER(_P)]),
    "dflash_inject_blocks": (_I32, [_P, _P, _I32, _I32P, _I32P, _I32, ctypes.POINTER(_P)]),
    "dflash_draft_step": (_I32, [_P, _P, _I32, _I32P, _P, _P, _P, _P, _P]),
    "dflash_verify_greedy": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P]),
    "dflash_sample_tokens": (_I32, [_P, _P, _I32, _P, _P, _P, _P]),
    "dflash_draft_step_lse": (_I32, [_P, _P, _I32, _I32P, _P, _P, _P, _P, _P, _P]),
    "dflash_draft_step_ex": (_I32, [_P, _P, _I32, _I32P, _P, ctypes.POINTER(DraftOut)]),
    "dflash_select_path": (_I32, [_P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_ddtree_build": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_ddtree_walk": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_verify_sample": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_verify_sample_q": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_select_sample": (_I32, [_P, _I32, _I32, _I32, _I32, _I32, _I32, ctypes.c_float, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _P]),
    "dflash_release": (_I32, [_P, _I32]),
    "dflash_truncate": (_I32, [_P, _I32, _I32]),
    "dflash_context_len": (_I32, [_P, _I32, _I32P]),
    "dflash_export_kv": (_I32, [_P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "dflash_free_pages": (_I32, [_P]),
    "dflash_last_error": (ctypes.c_char_p, [_P]),
    "dflash_status_string": (ctypes.c_char_p, [_I32]),
    "dflash_launch_count": (ctypes.c_int64, [_P]),
    "dflash_topk_noalloc": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, ctypes.c_char_p, _I32]),
    "dflash_timing_enable": (_I32, [_P, _I32]),
    "dflash_timing_classes": (_I32, []),
    "dflash_timing_class_name": (ctypes.c_char_p, [_I32]),
    "dflash_timing_read": (_I32, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), _I32]),
}

class Sampling(ctypes.Structure):
    """dflash_sampling: temperature > 0, 1 <= top_k <= 32, 0 < top_p <= 1."""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


_lib = None


def load(path=None):
    """Loads libdflash.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libdflash.so not found at {p}; build it with "
                          "`python -m block_diffusion_speculative_inject_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib
