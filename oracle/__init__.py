"""Oracle: plain fp64 CPU reference of the shared ViT encoder forward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
(``jepa_vision_encoder_gb300``) never does. It shares no code with the GPU path
except the seeded input generator (``synth``).

The arithmetic lives in ``oracle.cpp`` (compiled to ``liboracle.so``); this
module only marshals numpy arrays through ctypes.
"""
import ctypes
import os
import subprocess
from dataclasses import dataclass, asdict

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SYNTH_H = os.path.join(os.path.dirname(_HERE), "synth", "jepa_synth.h")
_lib = None


class OracleHParams(ctypes.Structure):
    _fields_ = [
        ("embed_dim", ctypes.c_int), ("n_layer", ctypes.c_int), ("n_head", ctypes.c_int),
        ("ffn_dim", ctypes.c_int), ("patch_size", ctypes.c_int), ("tubelet_size", ctypes.c_int),
        ("in_chans", ctypes.c_int), ("ln_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
        ("pos_type", ctypes.c_int), ("rope_layout", ctypes.c_int), ("rope_interpolate", ctypes.c_int),
        ("rope_ref_grid", ctypes.c_int), ("cls_token", ctypes.c_int), ("modality_embed", ctypes.c_int),
        ("attn_mode", ctypes.c_int), ("n_pos_rows", ctypes.c_int), ("img_size", ctypes.c_int),
        ("n_frames", ctypes.c_int), ("sincos_w_first", ctypes.c_int), ("sincos_uniform_power", ctypes.c_int),
        ("q_weight_scale", ctypes.c_double), ("k_weight_scale", ctypes.c_double),
    ]


@dataclass
class Config:
    """Encoder hyper-parameters in the jepa.enc.* vocabulary (one item's geometry is T, H, W)."""
    embed_dim: int
    n_layer: int
    n_head: int
    ffn_dim: int
    patch_size: int
    tubelet_size: int
    in_chans: int = 3
    ln_eps: float = 1e-6
    rope_theta: float = 10000.0
    pos_type: int = 0          # 0 none, 1 learned, 2 rope3d, 3 sincos2d, 4 sincos3d
    rope_layout: int = 0       # 0 tiled, 1 interleaved
    rope_interpolate: int = 0
    rope_ref_grid: int = 0
    cls_token: int = 0
    modality_embed: int = 0
    attn_mode: int = 0         # 0 full, 1 block_causal
    n_pos_rows: int = 0
    img_size: int = 0          # training crop and frames: the grid a sin-cos table is baked for
    n_frames: int = 0
    sincos_w_first: int = 0    # sincos2d halves [w | h] (HF I-JEPA order)
    sincos_uniform_power: int = 0
    # test input option, not part of the method: the synthetic q / k rows of every attn_qkv.weight
    # are multiplied by these factors in float (bf16 weights: rounded to bf16 again), for peaked
    # attention
    q_weight_scale: float = 1.0
    k_weight_scale: float = 1.0

    def struct(self) -> OracleHParams:
        return OracleHParams(**asdict(self))

    @property
    def head_dim(self) -> int:
        return self.embed_dim // self.n_head


class OraclePredHParams(ctypes.Structure):
    _fields_ = [
        ("embed_dim", ctypes.c_int), ("n_layer", ctypes.c_int), ("n_head", ctypes.c_int),
        ("ffn_dim", ctypes.c_int), ("enc_dim", ctypes.c_int), ("out_dim", ctypes.c_int),
        ("n_mask_tokens", ctypes.c_int), ("mask_index", ctypes.c_int), ("ln_eps", ctypes.c_double),
        ("rope_theta", ctypes.c_double), ("rope_layout", ctypes.c_int),
    ]


@dataclass
class PredConfig:
    """Masked-predictor hyper-parameters in the jepa.pred.* vocabulary."""
    embed_dim: int
    n_layer: int
    n_head: int
    ffn_dim: int
    enc_dim: int
    out_dim: int
    n_mask_tokens: int = 10
    mask_index: int = 1
    ln_eps: float = 1e-6
    rope_theta: float = 10000.0
    rope_layout: int = 0

    def struct(self) -> OraclePredHParams:
        return OraclePredHParams(**asdict(self))

    @property
    def head_dim(self) -> int:
        return self.embed_dim // self.n_head


class OracleHeadHParams(ctypes.Structure):
    _fields_ = [("embed_dim", ctypes.c_int), ("n_head", ctypes.c_int), ("ffn_dim", ctypes.c_int),
                ("n_pool_layers", ctypes.c_int), ("n_classes", ctypes.c_int), ("ln_eps", ctypes.c_double)]


@dataclass
class HeadConfig:
    """Attentive-pool head hyper-parameters in the jepa.head.* vocabulary."""
    embed_dim: int
    n_head: int
    ffn_dim: int
    n_pool_layers: int = 3
    n_classes: int = 174
    ln_eps: float = 1e-6

    def struct(self) -> OracleHeadHParams:
        return OracleHeadHParams(**asdict(self))


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (g++, OpenMP, contraction off for the generator)."""
    src = os.path.join(_HERE, "oracle.cpp")
    hdr = os.path.join(_HERE, "oracle.h")
    newest = max(os.path.getmtime(p) for p in (src, hdr, _SYNTH_H))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O3", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", tmp, src])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        hp = ctypes.POINTER(OracleHParams)
        L.oracle_n_tokens.argtypes = [hp, I, I, I]
        L.oracle_n_tokens.restype = I
        L.oracle_patchify.argtypes = [hp, P, I, I, I, I, I, P]
        L.oracle_conv3d.argtypes = [hp, P, I, I, I, I, I, P, P, P]
        L.oracle_linear.argtypes = [P, I, I, P, P, I, P]
        L.oracle_linear.restype = None
        L.oracle_layernorm.argtypes = [P, I, I, P, P, ctypes.c_double, P]
        L.oracle_layernorm.restype = None
        L.oracle_gelu.argtypes = [P, ctypes.c_size_t, P]
        L.oracle_gelu.restype = None
        L.oracle_rope_positions.argtypes = [hp, I, I, I, P]
        L.oracle_rope_tables.argtypes = [hp, I, I, I, P, P]
        L.oracle_rope_apply.argtypes = [P, I, I, I, P, P, P]
        L.oracle_rope_apply.restype = None
        L.oracle_sincos_2d.argtypes = [I, I, I, I, P]
        L.oracle_sincos_3d.argtypes = [I, I, I, I, I, P]
        L.oracle_interp_trilinear.argtypes = [P, I, I, I, I, I, I, I, P]
        L.oracle_interp_bicubic.argtypes = [P, I, I, I, I, I, P]
        L.oracle_pos_table.argtypes = [hp, I, I, I, P]
        L.oracle_rope_tables_pos.argtypes = [I, ctypes.c_double, I, P, I, P, P]
        L.oracle_rope_tables_pos.restype = None
        L.oracle_predict.argtypes = [ctypes.POINTER(OraclePredHParams), ctypes.c_uint64, I, P, I, I, P, I, P, I,
                                     I, I, P]
        L.oracle_cross_attention.argtypes = [P, I, P, P, I, I, I, P]
        L.oracle_cross_attention.restype = None
        L.oracle_attentive_head.argtypes = [ctypes.POINTER(OracleHeadHParams), ctypes.c_uint64, I, P, I, I, P, P]
        L.oracle_pool.argtypes = [P, I, I, I, I, I, P]
        L.oracle_mask_allow.argtypes = [I, I, I, I, I, I]
        L.oracle_attention.argtypes = [P, P, P, I, I, I, I, I, I, P]
        L.oracle_attention.restype = None
        L.oracle_encode.argtypes = [hp, ctypes.c_uint64, I, P, I, I, I, I, I, I, P]
        L.oracle_num_threads.argtypes = []
        _lib = L
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def n_tokens(cfg: Config, T: int, H: int, W: int) -> int:
    s = cfg.struct()
    return int(lib().oracle_n_tokens(ctypes.byref(s), T, H, W))


def geometry(cfg: Config, T: int, H: int, W: int):
    gt, gh, gw = T // cfg.tubelet_size, H // cfg.patch_size, W // cfg.patch_size
    K = cfg.in_chans * cfg.tubelet_size * cfg.patch_size ** 2
    return gt, gh, gw, K


def patchify(cfg: Config, pix, layout: int = 0) -> np.ndarray:
    pix = _f32(pix)
    B = pix.shape[0]
    T, H, W = (pix.shape[1], pix.shape[3], pix.shape[4]) if layout == 0 else (pix.shape[2], pix.shape[3], pix.shape[4])
    gt, gh, gw, K = geometry(cfg, T, H, W)
    out = np.empty((B * gt * gh * gw, K), dtype=np.float64)
    s = cfg.struct()
    rc = lib().oracle_patchify(ctypes.byref(s), pix.ctypes.data, B, T, H, W, layout, out.ctypes.data)
    assert rc == 0
    return out


def conv3d(cfg: Config, pix, w, bias, layout: int = 0) -> np.ndarray:
    pix = _f32(pix)
    B = pix.shape[0]
    T, H, W = (pix.shape[1], pix.shape[3], pix.shape[4]) if layout == 0 else (pix.shape[2], pix.shape[3], pix.shape[4])
    gt, gh, gw, K = geometry(cfg, T, H, W)
    w = _f64(w)
    bias = _f64(bias)
    out = np.empty((B, gt, gh, gw, cfg.embed_dim), dtype=np.float64)
    s = cfg.struct()
    rc = lib().oracle_conv3d(ctypes.byref(s), pix.ctypes.data, B, T, H, W, layout, w.ctypes.data,
                             bias.ctypes.data, out.ctypes.data)
    assert rc == 0
    return out


def linear(x, w, b=None) -> np.ndarray:
    x, w = _f64(x), _f64(w)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    bp = None
    if b is not None:
        b = _f64(b)
        bp = b.ctypes.data
    lib().oracle_linear(x.ctypes.data, M, K, w.ctypes.data, bp, N, y.ctypes.data)
    return y


def layernorm(x, gamma, beta, eps) -> np.ndarray:
    x, gamma, beta = _f64(x), _f64(gamma), _f64(beta)
    M, D = x.shape
    y = np.empty_like(x)
    lib().oracle_layernorm(x.ctypes.data, M, D, gamma.ctypes.data, beta.ctypes.data, float(eps), y.ctypes.data)
    return y


def gelu(x) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().oracle_gelu(x.ctypes.data, x.size, y.ctypes.data)
    return y


def rope_positions(cfg: Config, T, H, W) -> np.ndarray:
    gt, gh, gw, _ = geometry(cfg, T, H, W)
    pos = np.empty((gt * gh * gw, 3), dtype=np.float64)
    s = cfg.struct()
    assert lib().oracle_rope_positions(ctypes.byref(s), T, H, W, pos.ctypes.data) == 0
    return pos


def rope_tables(cfg: Config, T, H, W):
    N = n_tokens(cfg, T, H, W)
    hd = cfg.head_dim
    c = np.empty((N, hd), dtype=np.float64)
    s_ = np.empty((N, hd), dtype=np.float64)
    s = cfg.struct()
    assert lib().oracle_rope_tables(ctypes.byref(s), T, H, W, c.ctypes.data, s_.ctypes.data) == 0
    return c, s_


def rope_apply(x, n_head, cos_t, sin_t) -> np.ndarray:
    """x: [N, n_head*hd]."""
    x = _f64(x)
    cos_t, sin_t = _f64(cos_t), _f64(sin_t)
    N = x.shape[0]
    hd = x.shape[1] // n_head
    out = np.empty_like(x)
    lib().oracle_rope_apply(x.ctypes.data, N, n_head, hd, cos_t.ctypes.data, sin_t.ctypes.data, out.ctypes.data)
    return out


def sincos_2d(gh, gw, D, w_first=False) -> np.ndarray:
    """2-D sin-cos table [gh*gw, D], halves [h | w] (or [w | h] when w_first)."""
    out = np.empty((gh * gw, D), dtype=np.float64)
    if lib().oracle_sincos_2d(gh, gw, D, int(w_first), out.ctypes.data) != 0:
        raise ValueError(f"sincos_2d refused width {D}")
    return out


def sincos_3d(gt, gh, gw, D, uniform_power=False) -> np.ndarray:
    """3-D sin-cos table [gt*gh*gw, D], parts [t | h | w]."""
    out = np.empty((gt * gh * gw, D), dtype=np.float64)
    if lib().oracle_sincos_3d(gt, gh, gw, D, int(uniform_power), out.ctypes.data) != 0:
        raise ValueError(f"sincos_3d refused width {D}")
    return out


def interp_trilinear(src, size) -> np.ndarray:
    """src [st, sh, sw, D] -> [dt, dh, dw, D] (pixel-centre aligned)."""
    src = _f64(src)
    st, sh, sw, D = src.shape
    dt, dh, dw = size
    out = np.empty((dt, dh, dw, D), dtype=np.float64)
    assert lib().oracle_interp_trilinear(src.ctypes.data, st, sh, sw, D, dt, dh, dw, out.ctypes.data) == 0
    return out


def interp_bicubic(src, size) -> np.ndarray:
    """src [sh, sw, D] -> [dh, dw, D] (pixel-centre aligned, Keys a = -0.75)."""
    src = _f64(src)
    sh, sw, D = src.shape
    dh, dw = size
    out = np.empty((dh, dw, D), dtype=np.float64)
    assert lib().oracle_interp_bicubic(src.ctypes.data, sh, sw, D, dh, dw, out.ctypes.data) == 0
    return out


def pos_table(cfg: Config, T, H, W) -> np.ndarray:
    """The sin-cos table a T x H x W clip adds to its patch rows, [Np, D]."""
    gt, gh, gw, _ = geometry(cfg, T, H, W)
    out = np.empty((gt * gh * gw, cfg.embed_dim), dtype=np.float64)
    s = cfg.struct()
    rc = lib().oracle_pos_table(ctypes.byref(s), T, H, W, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_pos_table refused the configuration (code {rc})")
    return out


def rope_tables_pos(hd, theta, layout, pos):
    """cos / signed-sin tables [n, hd] at explicit positions pos [n, 3]."""
    pos = _f64(pos)
    n = pos.shape[0]
    c = np.empty((n, hd), dtype=np.float64)
    s_ = np.empty((n, hd), dtype=np.float64)
    lib().oracle_rope_tables_pos(hd, float(theta), layout, pos.ctypes.data, n, c.ctypes.data, s_.ctypes.data)
    return c, s_


def predict(pcfg: PredConfig, seed: int, bf16_weights: bool, enc, ctx_ids, tgt_ids, grid) -> np.ndarray:
    """Masked predictor: enc [B, n_enc, enc_dim], ctx_ids [B, n_ctx], tgt_ids [B, n_tgt], grid (gh, gw)
    -> [B, n_tgt, out_dim] fp64."""
    enc = _f64(enc)
    B, n_enc, _ = enc.shape
    ctx = np.ascontiguousarray(ctx_ids, dtype=np.int32).reshape(B, -1)
    tgt = np.ascontiguousarray(tgt_ids, dtype=np.int32).reshape(B, -1)
    out = np.empty((B, tgt.shape[1], pcfg.out_dim), dtype=np.float64)
    s = pcfg.struct()
    rc = lib().oracle_predict(ctypes.byref(s), seed, int(bf16_weights), enc.ctypes.data, B, n_enc, ctx.ctypes.data,
                              ctx.shape[1], tgt.ctypes.data, tgt.shape[1], grid[0], grid[1], out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_predict refused the configuration (code {rc})")
    return out


def cross_attention(q, k, v, n_head) -> np.ndarray:
    """q [Nq, H*hd], k, v [Nk, H*hd] -> [Nq, H*hd]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    hd = q.shape[1] // n_head
    o = np.empty_like(q)
    lib().oracle_cross_attention(q.ctypes.data, q.shape[0], k.ctypes.data, v.ctypes.data, k.shape[0], n_head, hd,
                                 o.ctypes.data)
    return o


def attentive_head(hcfg: HeadConfig, seed: int, bf16_weights: bool, tokens):
    """tokens [B, N, D] -> (pooled [B, D], logits [B, n_classes]) fp64."""
    tokens = _f64(tokens)
    B, N, D = tokens.shape
    pooled = np.empty((B, D), dtype=np.float64)
    logits = np.empty((B, hcfg.n_classes), dtype=np.float64)
    s = hcfg.struct()
    rc = lib().oracle_attentive_head(ctypes.byref(s), seed, int(bf16_weights), tokens.ctypes.data, B, N,
                                     pooled.ctypes.data, logits.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_attentive_head refused the configuration (code {rc})")
    return pooled, logits


def pool(tokens, prefix: int, mode: int) -> np.ndarray:
    """tokens [B, N, D] -> [B, D]: mode 0 mean of the patch tokens, mode 1 the CLS row."""
    tokens = _f64(tokens)
    B, N, D = tokens.shape
    out = np.empty((B, D), dtype=np.float64)
    if lib().oracle_pool(tokens.ctypes.data, B, N, D, prefix, mode, out.ctypes.data) != 0:
        raise ValueError("oracle_pool refused the arguments")
    return out


def mask_allow(attn_mode, prefix, frame_tokens, N, q, k) -> bool:
    return bool(lib().oracle_mask_allow(attn_mode, prefix, frame_tokens, N, q, k))


def attention(q, k, v, n_head, attn_mode=0, prefix=0, frame_tokens=1) -> np.ndarray:
    """q, k, v: [N, n_head*hd] -> o [N, n_head*hd]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N = q.shape[0]
    hd = q.shape[1] // n_head
    o = np.empty_like(q)
    lib().oracle_attention(q.ctypes.data, k.ctypes.data, v.ctypes.data, N, n_head, hd, attn_mode, prefix,
                           frame_tokens, o.ctypes.data)
    return o


def encode(cfg: Config, seed: int, bf16_weights: bool, pix, layout: int = 0, final_norm: bool = True) -> np.ndarray:
    """Whole encoder on pixels [B,T,C,H,W] (layout 0) or [B,C,T,H,W] (layout 1) -> [B, N, D] fp64."""
    pix = _f32(pix)
    B = pix.shape[0]
    T, H, W = (pix.shape[1], pix.shape[3], pix.shape[4]) if layout == 0 else (pix.shape[2], pix.shape[3], pix.shape[4])
    N = n_tokens(cfg, T, H, W)
    assert N > 0
    out = np.empty((B, N, cfg.embed_dim), dtype=np.float64)
    s = cfg.struct()
    rc = lib().oracle_encode(ctypes.byref(s), seed, int(bf16_weights), pix.ctypes.data, B, T, H, W, layout,
                             int(final_norm), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_encode refused the configuration (code {rc})")
    return out
