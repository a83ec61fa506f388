"""GB300 (sm_103a) forward pass of the shared ViT encoder of the JEPA family.

A thin Python layer over the C ABI of include/jepa.h (libjepa_gb300.so): it passes torch
tensors' device pointers and a CUDA stream; every step of the encoder runs in the library's
CUDA kernels. Importing works without a GPU; calls that launch kernels need one.

    import jepa_vision_encoder_gb300 as jv
    model = jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16")
    ctx = jv.Context(model, max_batch=1, frames=16, height=256, width=256)
    tokens = ctx.encode(pixels)          # pixels: float32 CUDA tensor [B, T, 3, H, W]
"""
import ctypes
import os

import torch

from . import _lib
from ._lib import (ATTN_BLOCK_CAUSAL, ATTN_FULL, BF16, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL,
                   EPI_PATCH_EMBED, EPI_QKV_ROPE, FP32, LAYOUT_CTHW, LAYOUT_TCHW, POS_LEARNED, POS_NONE,
                   POS_ROPE3D, POS_SINCOS2D, POS_SINCOS3D, RESIZE_BICUBIC, RESIZE_TRILINEAR, ROPE_INTERLEAVED,
                   ROPE_TILED, POOL_CLS, POOL_MEAN, Epilogue, HeadHParams, HParams, JepaError, PredHParams, check,
                   lib)

__all__ = ["Model", "Context", "HParams", "JepaError", "preset", "hparams", "gguf_hparams", "n_tokens", "ops", "lib", "Predictor",
           "PredContext", "PredHParams", "pred_preset", "Head", "HeadContext", "HeadHParams", "head_preset"]

PRESETS = ("hfvit_ti14", "vjepa2_vitl16", "vjepa2_1_vitl16", "levjepa_vitl16", "vjepa2_vitg16", "vjepa_vitl16",
           "ijepa_vitl16")


def _dtype_code(dtype) -> int:
    if dtype in (BF16, "bf16", torch.bfloat16):
        return BF16
    if dtype in (FP32, "fp32", "f32", torch.float32):
        return FP32
    raise ValueError(f"unknown dtype {dtype!r}")


def preset(name: str) -> HParams:
    hp = HParams()
    check(lib().jepa_preset(name.encode(), ctypes.byref(hp)))
    return hp


def gguf_hparams(path: str) -> HParams:
    """The checked encoder hyper-parameters of a GGUF file (no weights are read; no GPU needed)."""
    hp = HParams()
    check(lib().jepa_gguf_hparams(os.fsencode(path), ctypes.byref(hp)))
    return hp


def hparams(**kw) -> HParams:
    hp = HParams()
    hp.in_chans = 3
    hp.ln_eps = 1e-6
    hp.rope_theta = 10000.0
    for k, v in kw.items():
        setattr(hp, k, v)
    return hp


def n_tokens(hp: HParams, T: int, H: int, W: int) -> int:
    n = ctypes.c_int32()
    check(lib().jepa_n_tokens(ctypes.byref(hp), T, H, W, ctypes.byref(n)))
    return n.value


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _clip_dims(pixels: torch.Tensor, layout: int):
    if layout == LAYOUT_TCHW:
        return pixels.shape[0], pixels.shape[1], pixels.shape[3], pixels.shape[4]
    return pixels.shape[0], pixels.shape[2], pixels.shape[3], pixels.shape[4]


class Model:
    """Synthetic-weight encoder resident on one GPU (immutable; shareable across threads)."""

    def __init__(self, hp: HParams, seed: int = 0, dtype="bf16", device: int = 0):
        self.hp = hp
        self.seed = seed
        self.dtype = _dtype_code(dtype)
        self.device = device
        h = ctypes.c_void_p()
        check(lib().jepa_model_load(ctypes.byref(hp), seed, self.dtype, device, ctypes.byref(h)))
        self._h = h

    @classmethod
    def from_gguf(cls, path: str, dtype="bf16", device: int = 0):
        """An encoder loaded from a GGUF file (checked as jepa_gguf_hparams describes)."""
        self = cls.__new__(cls)
        self.hp = gguf_hparams(path)
        self.seed = None
        self.dtype = _dtype_code(dtype)
        self.device = device
        h = ctypes.c_void_p()
        check(lib().jepa_model_load_gguf(os.fsencode(path), self.dtype, device, ctypes.byref(h)))
        self._h = h
        return self

    @classmethod
    def preset(cls, name: str, seed: int = 0, dtype="bf16", device: int = 0, **overrides):
        hp = preset(name)
        for k, v in overrides.items():
            setattr(hp, k, v)
        return cls(hp, seed=seed, dtype=dtype, device=device)

    def tensor(self, name: str, shape) -> torch.Tensor:
        """An enc.* tensor copied to host memory as float32."""
        n = 1
        for s in shape:
            n *= s
        out = torch.empty(n, dtype=torch.float32)
        check(lib().jepa_model_tensor(self._h, name.encode(), ctypes.c_void_p(out.data_ptr()), n))
        return out.reshape(shape)

    def n_tokens(self, T, H, W) -> int:
        return n_tokens(self.hp, T, H, W)

    def encode_noalloc(self, pixels: torch.Tensor, out: torch.Tensor, layout: int = LAYOUT_TCHW) -> torch.Tensor:
        """Encode into the caller's `out` with the library's fixed scratch array as workspace
        (no device allocation); synchronous on torch's current stream. Calls must not overlap."""
        assert pixels.is_cuda and pixels.dtype == torch.float32 and pixels.is_contiguous()
        assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
        B, T, H, W = _clip_dims(pixels, layout)
        assert out.numel() == B * self.n_tokens(T, H, W) * self.hp.embed_dim
        check(lib().jepa_encode_noalloc(self._h, _ptr(pixels), B, T, H, W, layout, _ptr(out), _stream_ptr()))
        return out

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_model_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """Workspace for clips up to (max_batch, frames, height, width); one thread at a time.

    Kernels run on `stream` if one is given (the caller orders its own work around it), else
    on a side stream the context owns: encode() then waits for torch's current stream before
    launching and makes the current stream wait for the encode, so torch code before and after
    is ordered with it (and CUDA-graph capture never touches the legacy default stream).
    """

    def __init__(self, model: Model, max_batch: int, frames: int, height: int, width: int,
                 max_workspace_bytes: int = 0, stream=None, graph: bool = False):
        self.model = model
        h = ctypes.c_void_p()
        check(lib().jepa_context_new(model._h, max_batch, frames, height, width, max_workspace_bytes,
                                     ctypes.byref(h)))
        self._h = h
        self._own = stream is None
        self.stream = torch.cuda.Stream(device=model.device) if stream is None else stream
        check(lib().jepa_context_set_stream(self._h, ctypes.c_void_p(self.stream.cuda_stream)))
        if graph:
            check(lib().jepa_context_set_graph(self._h, 1))

    def _enter(self):
        if self._own:
            self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))

    def _leave(self):
        if self._own:
            torch.cuda.current_stream(self.stream.device).wait_stream(self.stream)

    def set_graph(self, enable: bool):
        check(lib().jepa_context_set_graph(self._h, int(enable)))

    def set_pdl(self, enable: bool):
        """Programmatic dependent launches between the encode's kernels (on by default)."""
        check(lib().jepa_context_set_pdl(self._h, int(enable)))

    @property
    def workspace_bytes(self) -> int:
        n = ctypes.c_size_t()
        check(lib().jepa_context_workspace_bytes(self._h, ctypes.byref(n)))
        return n.value

    @property
    def max_batch(self) -> int:
        """Items one encode call folds together at most (the max_batch the context was made for)."""
        n = ctypes.c_int32()
        check(lib().jepa_context_max_batch(self._h, ctypes.byref(n)))
        return n.value

    def launches(self, B, T, H, W) -> int:
        n = ctypes.c_int32()
        check(lib().jepa_context_launches(self._h, B, T, H, W, ctypes.byref(n)))
        return n.value

    def encode(self, pixels: torch.Tensor, out: torch.Tensor = None, layout: int = LAYOUT_TCHW) -> torch.Tensor:
        """pixels: contiguous float32 CUDA tensor [B,T,C,H,W] (layout 0) or [B,C,T,H,W] (layout 1)."""
        assert pixels.is_cuda and pixels.dtype == torch.float32 and pixels.is_contiguous()
        B, T, H, W = _clip_dims(pixels, layout)
        N = self.model.n_tokens(T, H, W)
        if out is None:
            out = torch.empty((B, N, self.model.hp.embed_dim), dtype=torch.float32, device=pixels.device)
        self._enter()
        check(lib().jepa_encode(self._h, _ptr(pixels), B, T, H, W, layout, _ptr(out)))
        self._leave()
        return out

    def encode_host(self, pixels: torch.Tensor, out: torch.Tensor = None, layout: int = LAYOUT_TCHW) -> torch.Tensor:
        """Host (CPU, ideally pinned) float32 pixels in, host tokens out; synchronous."""
        assert not pixels.is_cuda and pixels.dtype == torch.float32 and pixels.is_contiguous()
        B, T, H, W = _clip_dims(pixels, layout)
        N = self.model.n_tokens(T, H, W)
        if out is None:
            out = torch.empty((B, N, self.model.hp.embed_dim), dtype=torch.float32)
        check(lib().jepa_encode_host(self._h, _ptr(pixels), B, T, H, W, layout, _ptr(out)))
        return out

    def encode_host_async(self, pixels: torch.Tensor, out: torch.Tensor, layout: int = LAYOUT_TCHW) -> torch.Tensor:
        """Pipelined host encode: enqueues upload, encode and download and returns at once; the copies
        overlap the neighbouring calls' encodes (pinned buffers). `pixels` and `out` must stay alive
        and untouched until sync()."""
        assert not pixels.is_cuda and pixels.dtype == torch.float32 and pixels.is_contiguous()
        assert not out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
        B, T, H, W = _clip_dims(pixels, layout)
        check(lib().jepa_encode_host_async(self._h, _ptr(pixels), B, T, H, W, layout, _ptr(out)))
        return out

    def sync(self):
        check(lib().jepa_context_sync(self._h))

    def set_profiling(self, enable: bool):
        check(lib().jepa_context_set_profiling(self._h, int(enable)))

    def profile(self, reset: bool = True) -> dict:
        """Per-kernel-class event timings accumulated since the last reset:
        {name: {"launches", "total_ms", "flops", "bytes"}} (synchronises the context stream)."""
        buf = (_lib.KernelStat * 16)()
        n = ctypes.c_int32()
        check(lib().jepa_context_profile(self._h, buf, 16, ctypes.byref(n), int(reset)))
        return {buf[i].name.decode(): {"launches": buf[i].launches, "total_ms": buf[i].total_ms,
                                       "flops": buf[i].flops, "bytes": buf[i].bytes} for i in range(n.value)}

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_context_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pred_preset(name: str) -> PredHParams:
    hp = PredHParams()
    check(lib().jepa_pred_preset(name.encode(), ctypes.byref(hp)))
    return hp


class Predictor:
    """Synthetic-weight masked-latent predictor (pred.* tensors) resident on one GPU, bf16."""

    def __init__(self, hp: PredHParams, seed: int = 0, dtype="bf16", device: int = 0):
        self.hp = hp
        self.seed = seed
        self.device = device
        h = ctypes.c_void_p()
        check(lib().jepa_pred_load(ctypes.byref(hp), seed, _dtype_code(dtype), device, ctypes.byref(h)))
        self._h = h

    @classmethod
    def preset(cls, name: str, seed: int = 0, dtype="bf16", device: int = 0, **overrides):
        hp = pred_preset(name)
        for k, v in overrides.items():
            setattr(hp, k, v)
        return cls(hp, seed=seed, dtype=dtype, device=device)

    def tensor(self, name: str, shape) -> torch.Tensor:
        """A pred.* tensor copied to host memory as float32."""
        n = 1
        for s in shape:
            n *= s
        out = torch.empty(n, dtype=torch.float32)
        check(lib().jepa_pred_tensor(self._h, name.encode(), ctypes.c_void_p(out.data_ptr()), n))
        return out.reshape(shape)

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_pred_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PredContext:
    """Workspace for up to max_batch items of max_ctx context and max_tgt target tokens; streams
    as Context (an own side stream ordered with torch's current stream, or the given `stream`)."""

    def __init__(self, pred: Predictor, max_batch: int, max_ctx: int, max_tgt: int, max_workspace_bytes: int = 0,
                 stream=None, graph: bool = False):
        self.pred = pred
        h = ctypes.c_void_p()
        check(lib().jepa_pred_context_new(pred._h, max_batch, max_ctx, max_tgt, max_workspace_bytes, ctypes.byref(h)))
        self._h = h
        self._own = stream is None
        self.stream = torch.cuda.Stream(device=pred.device) if stream is None else stream
        check(lib().jepa_pred_context_set_stream(self._h, ctypes.c_void_p(self.stream.cuda_stream)))
        if graph:
            check(lib().jepa_pred_context_set_graph(self._h, 1))

    def set_graph(self, enable: bool):
        check(lib().jepa_pred_context_set_graph(self._h, int(enable)))

    def set_profiling(self, enable: bool):
        check(lib().jepa_pred_context_set_profiling(self._h, int(enable)))

    def launches(self, n_ctx: int) -> int:
        n = ctypes.c_int32()
        check(lib().jepa_pred_context_launches(self._h, n_ctx, ctypes.byref(n)))
        return n.value

    def predict(self, enc: torch.Tensor, ctx_ids: torch.Tensor, tgt_ids: torch.Tensor, grid, out: torch.Tensor = None):
        """enc: float32 CUDA [B, n_enc, enc_dim]; ctx_ids / tgt_ids: int32 CUDA [B, n]; grid (gt, gh, gw)."""
        assert enc.is_cuda and enc.dtype == torch.float32 and enc.is_contiguous()
        assert tgt_ids.dtype == torch.int32 and tgt_ids.is_contiguous()
        assert ctx_ids.dtype == torch.int32 and ctx_ids.is_contiguous()
        B, n_enc, _ = enc.shape
        n_ctx, n_tgt = ctx_ids.shape[-1], tgt_ids.shape[-1]
        if out is None:
            out = torch.empty((B, n_tgt, self.pred.hp.out_dim), dtype=torch.float32, device=enc.device)
        if self._own:
            self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        ctx_ptr = ctypes.c_void_p(ctx_ids.data_ptr() if n_ctx else 0)
        check(lib().jepa_predict(self._h, _ptr(enc), B, n_enc, ctx_ptr, n_ctx, _ptr(tgt_ids), n_tgt, grid[0], grid[1],
                                 grid[2], _ptr(out)))
        if self._own:
            torch.cuda.current_stream(self.stream.device).wait_stream(self.stream)
        return out

    def sync(self):
        check(lib().jepa_pred_context_sync(self._h))

    def profile(self, reset: bool = True) -> dict:
        """Per-kernel-class event timings (profiling on: eager launches), as Context.profile."""
        buf = (_lib.KernelStat * 16)()
        n = ctypes.c_int32()
        check(lib().jepa_pred_context_profile(self._h, buf, 16, ctypes.byref(n), int(reset)))
        return {buf[i].name.decode(): {"launches": buf[i].launches, "total_ms": buf[i].total_ms,
                                       "flops": buf[i].flops, "bytes": buf[i].bytes} for i in range(n.value)}

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_pred_context_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def head_preset(name: str) -> HeadHParams:
    hp = HeadHParams()
    check(lib().jepa_head_preset(name.encode(), ctypes.byref(hp)))
    return hp


class Head:
    """Synthetic-weight attentive-pool head + classifier (head.* tensors) on one GPU, bf16."""

    def __init__(self, hp: HeadHParams, seed: int = 0, dtype="bf16", device: int = 0):
        self.hp = hp
        self.seed = seed
        self.device = device
        h = ctypes.c_void_p()
        check(lib().jepa_head_load(ctypes.byref(hp), seed, _dtype_code(dtype), device, ctypes.byref(h)))
        self._h = h

    @classmethod
    def preset(cls, name: str, seed: int = 0, dtype="bf16", device: int = 0, **overrides):
        hp = head_preset(name)
        for k, v in overrides.items():
            setattr(hp, k, v)
        return cls(hp, seed=seed, dtype=dtype, device=device)

    def tensor(self, name: str, shape) -> torch.Tensor:
        """A head.* tensor copied to host memory as float32."""
        n = 1
        for s in shape:
            n *= s
        out = torch.empty(n, dtype=torch.float32)
        check(lib().jepa_head_tensor(self._h, name.encode(), ctypes.c_void_p(out.data_ptr()), n))
        return out.reshape(shape)

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_head_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HeadContext:
    """Workspace for up to max_batch items of max_tokens tokens; streams as Context."""

    def __init__(self, head: Head, max_batch: int, max_tokens: int, max_workspace_bytes: int = 0, stream=None,
                 graph: bool = False):
        self.head = head
        h = ctypes.c_void_p()
        check(lib().jepa_head_context_new(head._h, max_batch, max_tokens, max_workspace_bytes, ctypes.byref(h)))
        self._h = h
        self._own = stream is None
        self.stream = torch.cuda.Stream(device=head.device) if stream is None else stream
        check(lib().jepa_head_context_set_stream(self._h, ctypes.c_void_p(self.stream.cuda_stream)))
        if graph:
            check(lib().jepa_head_context_set_graph(self._h, 1))

    def set_graph(self, enable: bool):
        check(lib().jepa_head_context_set_graph(self._h, int(enable)))

    def set_profiling(self, enable: bool):
        check(lib().jepa_head_context_set_profiling(self._h, int(enable)))

    def launches(self, with_logits: bool = True) -> int:
        n = ctypes.c_int32()
        check(lib().jepa_head_context_launches(self._h, int(with_logits), ctypes.byref(n)))
        return n.value

    def forward(self, tokens: torch.Tensor, pooled: torch.Tensor = None, logits: torch.Tensor = None,
                want_pooled: bool = True, want_logits: bool = True):
        """tokens: float32 CUDA [B, N, D] -> (pooled [B, D], logits [B, n_classes])."""
        assert tokens.is_cuda and tokens.dtype == torch.float32 and tokens.is_contiguous()
        B, N, D = tokens.shape
        if pooled is None and want_pooled:
            pooled = torch.empty((B, D), dtype=torch.float32, device=tokens.device)
        if logits is None and want_logits:
            logits = torch.empty((B, self.head.hp.n_classes), dtype=torch.float32, device=tokens.device)
        if self._own:
            self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        check(lib().jepa_head_forward(self._h, _ptr(tokens), B, N,
                                      ctypes.c_void_p(pooled.data_ptr() if pooled is not None else 0),
                                      ctypes.c_void_p(logits.data_ptr() if logits is not None else 0)))
        if self._own:
            torch.cuda.current_stream(self.stream.device).wait_stream(self.stream)
        return pooled, logits

    def sync(self):
        check(lib().jepa_head_context_sync(self._h))

    def profile(self, reset: bool = True) -> dict:
        buf = (_lib.KernelStat * 16)()
        n = ctypes.c_int32()
        check(lib().jepa_head_context_profile(self._h, buf, 16, ctypes.byref(n), int(reset)))
        return {buf[i].name.decode(): {"launches": buf[i].launches, "total_ms": buf[i].total_ms,
                                       "flops": buf[i].flops, "bytes": buf[i].bytes} for i in range(n.value)}

    def close(self):
        if getattr(self, "_h", None):
            lib().jepa_head_context_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ops:
    """The encoder's kernels one at a time (same kernels the encode path launches)."""

    @staticmethod
    def patchify(pixels: torch.Tensor, tubelet: int, patch: int, layout: int = LAYOUT_TCHW, dtype="bf16"):
        if layout == LAYOUT_TCHW:
            B, T, C, H, W = pixels.shape
        else:
            B, C, T, H, W = pixels.shape
        rows = B * (T // tubelet) * (H // patch) * (W // patch)
        K = C * tubelet * patch * patch
        code = _dtype_code(dtype)
        out = torch.empty((rows, K), dtype=torch.bfloat16 if code == BF16 else torch.float32, device=pixels.device)
        check(lib().jepa_op_patchify(_ptr(pixels), B, T, C, H, W, tubelet, patch, layout, code, _ptr(out),
                                     _stream_ptr()))
        return out

    @staticmethod
    def layernorm(x: torch.Tensor, gamma, beta, eps: float, dtype="fp32"):
        M, D = x.shape
        code = _dtype_code(dtype)
        y = torch.empty((M, D), dtype=torch.bfloat16 if code == BF16 else torch.float32, device=x.device)
        check(lib().jepa_op_layernorm(_ptr(x), M, D, _ptr(gamma), _ptr(beta), eps, code, _ptr(y), _stream_ptr()))
        return y

    @staticmethod
    def linear(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor, out: torch.Tensor, kind: int = EPI_BIAS,
               rope: torch.Tensor = None, rows_per_item: int = 1, prefix: int = 0, n_head: int = 0,
               head_dim: int = 0, rope_layout: int = 0, patches_per_item: int = 1, pos: torch.Tensor = None,
               vec: torch.Tensor = None, rope_ids: torch.Tensor = None):
        M, K = x.shape
        N = w.shape[0]
        code = BF16 if x.dtype == torch.bfloat16 else FP32
        e = Epilogue()
        e.kind = kind
        e.d_bias = bias.data_ptr()
        e.d_out = out.data_ptr()
        e.d_rope = rope.data_ptr() if rope is not None else None
        e.rows_per_item = rows_per_item
        e.prefix = prefix
        e.n_head = n_head
        e.head_dim = head_dim
        e.rope_layout = rope_layout
        e.patches_per_item = patches_per_item
        e.d_pos = pos.data_ptr() if pos is not None else None
        e.d_vec = vec.data_ptr() if vec is not None else None
        e.d_rope_ids = rope_ids.data_ptr() if rope_ids is not None else None
        check(lib().jepa_op_linear(code, _ptr(x), M, K, _ptr(w), N, ctypes.byref(e), _stream_ptr()))
        return out

    @staticmethod
    def rope_table(hp: HParams, T: int, H: int, W: int, device="cuda"):
        hd = hp.embed_dim // hp.n_head
        d = 2 * ((hd // 3) // 2)
        gt, gh, gw = T // hp.tubelet_size, H // hp.patch_size, W // hp.patch_size
        table = torch.empty((gt * gh * gw, 3, d // 2, 2), dtype=torch.float32, device=device)
        check(lib().jepa_op_rope_table(ctypes.byref(hp), T, H, W, _ptr(table), _stream_ptr()))
        return table

    @staticmethod
    def sincos_table(kind: int, gt: int, gh: int, gw: int, D: int, w_first: bool = False,
                     uniform_power: bool = False, device="cuda"):
        """Fixed sin-cos position table [gt*gh*gw, D] (kind POS_SINCOS2D with gt == 1, or POS_SINCOS3D)."""
        table = torch.empty((gt * gh * gw, D), dtype=torch.float32, device=device)
        check(lib().jepa_op_sincos_table(kind, gt, gh, gw, D, int(w_first), int(uniform_power), _ptr(table),
                                         _stream_ptr()))
        return table

    @staticmethod
    def pos_resize(table: torch.Tensor, src_grid, dst_grid, mode: int = RESIZE_TRILINEAR):
        """Resize a [st*sh*sw, D] float table to [dt*dh*dw, D] (trilinear, or bicubic per frame)."""
        st, sh, sw = src_grid
        dt, dh, dw = dst_grid
        D = table.shape[-1]
        out = torch.empty((dt * dh * dw, D), dtype=torch.float32, device=table.device)
        check(lib().jepa_op_pos_resize(_ptr(table), st, sh, sw, D, mode, _ptr(out), dt, dh, dw, _stream_ptr()))
        return out

    @staticmethod
    def attention(qkv: torch.Tensor, B: int, N: int, n_head: int, head_dim: int = 64, attn_mode: int = ATTN_FULL,
                  prefix: int = 0, frame_tokens: int = 1):
        code = BF16 if qkv.dtype == torch.bfloat16 else FP32
        out = torch.empty((B * N, n_head * head_dim), dtype=qkv.dtype, device=qkv.device)
        check(lib().jepa_op_attention(code, _ptr(qkv), B, N, n_head, head_dim, attn_mode, prefix, frame_tokens,
                                      _ptr(out), _stream_ptr()))
        return out

    @staticmethod
    def pool(tokens: torch.Tensor, prefix: int = 0, mode: int = POOL_MEAN):
        """tokens float32 CUDA [B, N, D] -> [B, D]: the mean of rows [prefix, N), or row 0 (POOL_CLS)."""
        B, N, D = tokens.shape
        out = torch.empty((B, D), dtype=torch.float32, device=tokens.device)
        check(lib().jepa_op_pool(mode, _ptr(tokens), B, N, D, prefix, _ptr(out), _stream_ptr()))
        return out

    @staticmethod
    def device_status():
        return lib().jepa_device_status()

    @staticmethod
    def wait_timeout_probe(limit_us: int) -> int:
        return lib().jepa_debug_wait_timeout(limit_us)
