"""ctypes declarations of include/jepa.h (argument marshalling only).

Loading fails loudly when libjepa_gb300.so has not been built: there is no fallback path.
"""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjepa_gb300.so")

# jepa_status
OK, E_INVALID_ARG, E_UNSUPPORTED, E_BUDGET, E_OOM, E_CUDA, E_TIMEOUT = range(7)
STATUS_NAMES = {0: "JEPA_OK", 1: "JEPA_E_INVALID_ARG", 2: "JEPA_E_UNSUPPORTED", 3: "JEPA_E_BUDGET",
                4: "JEPA_E_OOM", 5: "JEPA_E_CUDA", 6: "JEPA_E_TIMEOUT"}
FP32, BF16 = 0, 1
POS_NONE, POS_LEARNED, POS_ROPE3D, POS_SINCOS2D, POS_SINCOS3D = 0, 1, 2, 3, 4
RESIZE_TRILINEAR, RESIZE_BICUBIC = 0, 1
POOL_MEAN, POOL_CLS = 0, 1
ROPE_TILED, ROPE_INTERLEAVED = 0, 1
ATTN_FULL, ATTN_BLOCK_CAUSAL = 0, 1
LAYOUT_TCHW, LAYOUT_CTHW = 0, 1
EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL, EPI_QKV_ROPE, EPI_PATCH_EMBED = range(5)


class HParams(ctypes.Structure):
    _fields_ = [
        ("embed_dim", ctypes.c_int32), ("n_layer", ctypes.c_int32), ("n_head", ctypes.c_int32),
        ("ffn_dim", ctypes.c_int32), ("patch_size", ctypes.c_int32), ("tubelet_size", ctypes.c_int32),
        ("img_size", ctypes.c_int32), ("n_frames", ctypes.c_int32), ("in_chans", ctypes.c_int32),
        ("ln_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("pos_type", ctypes.c_int32), ("rope_layout", ctypes.c_int32), ("rope_interpolate", ctypes.c_int32),
        ("rope_ref_grid", ctypes.c_int32), ("cls_token", ctypes.c_int32), ("modality_embed", ctypes.c_int32),
        ("attn_mode", ctypes.c_int32), ("n_pos_rows", ctypes.c_int32),
        ("sincos_w_first", ctypes.c_int32), ("sincos_uniform_power", ctypes.c_int32),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Epilogue(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("d_bias", ctypes.c_void_p), ("d_out", ctypes.c_void_p),
        ("d_rope", ctypes.c_void_p), ("rows_per_item", ctypes.c_int32), ("prefix", ctypes.c_int32),
        ("n_head", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("rope_layout", ctypes.c_int32),
        ("patches_per_item", ctypes.c_int32), ("d_pos", ctypes.c_void_p), ("d_vec", ctypes.c_void_p),
        ("d_rope_ids", ctypes.c_void_p),
    ]


class PredHParams(ctypes.Structure):
    _fields_ = [
        ("embed_dim", ctypes.c_int32), ("n_layer", ctypes.c_int32), ("n_head", ctypes.c_int32),
        ("ffn_dim", ctypes.c_int32), ("enc_dim", ctypes.c_int32), ("out_dim", ctypes.c_int32),
        ("n_mask_tokens", ctypes.c_int32), ("mask_index", ctypes.c_int32), ("ln_eps", ctypes.c_float),
        ("rope_theta", ctypes.c_float), ("rope_layout", ctypes.c_int32),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class HeadHParams(ctypes.Structure):
    _fields_ = [("embed_dim", ctypes.c_int32), ("n_head", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("n_pool_layers", ctypes.c_int32), ("n_classes", ctypes.c_int32), ("ln_eps", ctypes.c_float)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_float),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


# name -> (restype, argtypes); the exported surface of include/jepa.h
_P, _I, _U64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float
_HP = ctypes.POINTER(HParams)
_PHP = ctypes.POINTER(PredHParams)
_HHP = ctypes.POINTER(HeadHParams)
SIGNATURES = {
    "jepa_preset": (_I, [ctypes.c_char_p, _HP]),
    "jepa_hparams_validate": (_I, [_HP]),
    "jepa_n_tokens": (_I, [_HP, _I, _I, _I, ctypes.POINTER(ctypes.c_int32)]),
    "jepa_model_load": (_I, [_HP, _U64, _I, _I, ctypes.POINTER(_P)]),
    "jepa_model_free": (None, [_P]),
    "jepa_gguf_hparams": (_I, [ctypes.c_char_p, _HP]),
    "jepa_model_load_gguf": (_I, [ctypes.c_char_p, _I, _I, ctypes.POINTER(_P)]),
    "jepa_model_hparams": (_I, [_P, _HP]),
    "jepa_model_tensor": (_I, [_P, ctypes.c_char_p, _P, _SZ]),
    "jepa_context_new": (_I, [_P, _I, _I, _I, _I, _SZ, ctypes.POINTER(_P)]),
    "jepa_context_free": (None, [_P]),
    "jepa_context_set_stream": (_I, [_P, _P]),
    "jepa_context_set_graph": (_I, [_P, _I]),
    "jepa_context_set_pdl": (_I, [_P, _I]),
    "jepa_context_workspace_bytes": (_I, [_P, ctypes.POINTER(_SZ)]),
    "jepa_context_max_batch": (_I, [_P, ctypes.POINTER(_I)]),
    "jepa_context_launches": (_I, [_P, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int32)]),
    "jepa_encode": (_I, [_P, _P, _I, _I, _I, _I, _I, _P]),
    "jepa_encode_host": (_I, [_P, _P, _I, _I, _I, _I, _I, _P]),
    "jepa_encode_host_async": (_I, [_P, _P, _I, _I, _I, _I, _I, _P]),
    "jepa_context_sync": (_I, [_P]),
    "jepa_context_set_profiling": (_I, [_P, _I]),
    "jepa_context_profile": (_I, [_P, ctypes.POINTER(KernelStat), _I, ctypes.POINTER(ctypes.c_int32), _I]),
    "jepa_op_patchify": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "jepa_op_layernorm": (_I, [_P, _I, _I, _P, _P, _F, _I, _P, _P]),
    "jepa_op_linear": (_I, [_I, _P, _I, _I, _P, _I, ctypes.POINTER(Epilogue), _P]),
    "jepa_op_rope_table": (_I, [_HP, _I, _I, _I, _P, _P]),
    "jepa_op_sincos_table": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "jepa_op_pos_resize": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P]),
    "jepa_op_attention": (_I, [_I, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "jepa_device_status": (_I, []),
    "jepa_debug_wait_timeout": (_I, [_I]),
    "jepa_encode_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "jepa_pred_preset": (_I, [ctypes.c_char_p, _PHP]),
    "jepa_pred_hparams_validate": (_I, [_PHP]),
    "jepa_pred_load": (_I, [_PHP, _U64, _I, _I, ctypes.POINTER(_P)]),
    "jepa_pred_free": (None, [_P]),
    "jepa_pred_tensor": (_I, [_P, ctypes.c_char_p, _P, _SZ]),
    "jepa_pred_context_new": (_I, [_P, _I, _I, _I, _SZ, ctypes.POINTER(_P)]),
    "jepa_pred_context_free": (None, [_P]),
    "jepa_pred_context_set_stream": (_I, [_P, _P]),
    "jepa_pred_context_set_graph": (_I, [_P, _I]),
    "jepa_pred_context_set_profiling": (_I, [_P, _I]),
    "jepa_pred_context_profile": (_I, [_P, ctypes.POINTER(KernelStat), _I, ctypes.POINTER(ctypes.c_int32), _I]),
    "jepa_pred_context_launches": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int32)]),
    "jepa_predict": (_I, [_P, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I, _P]),
    "jepa_pred_context_sync": (_I, [_P]),
    "jepa_head_preset": (_I, [ctypes.c_char_p, _HHP]),
    "jepa_head_hparams_validate": (_I, [_HHP]),
    "jepa_head_load": (_I, [_HHP, _U64, _I, _I, ctypes.POINTER(_P)]),
    "jepa_head_free": (None, [_P]),
    "jepa_head_tensor": (_I, [_P, ctypes.c_char_p, _P, _SZ]),
    "jepa_head_context_new": (_I, [_P, _I, _I, _SZ, ctypes.POINTER(_P)]),
    "jepa_head_context_free": (None, [_P]),
    "jepa_head_context_set_stream": (_I, [_P, _P]),
    "jepa_head_context_set_graph": (_I, [_P, _I]),
    "jepa_head_context_set_profiling": (_I, [_P, _I]),
    "jepa_head_context_profile": (_I, [_P, ctypes.POINTER(KernelStat), _I, ctypes.POINTER(ctypes.c_int32), _I]),
    "jepa_head_context_launches": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int32)]),
    "jepa_head_forward": (_I, [_P, _P, _I, _I, _P, _P]),
    "jepa_head_context_sync": (_I, [_P]),
    "jepa_op_pool": (_I, [_I, _P, _I, _I, _I, _I, _P, _P]),
    "jepa_error_text": (ctypes.c_char_p, []),
    "jepa_error_reset": (None, []),
}

_lib = None


class JepaError(RuntimeError):
    def __init__(self, status, text):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {text}")
        self.status = status
        self.text = text


def lib():
    """The loaded library; raises if it was not built (run __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build the CUDA extension first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(status):
    if status != OK:
        text = lib().jepa_error_text()
        raise JepaError(status, text.decode() if text else "")
    return status
