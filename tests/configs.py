"""The workloads of the encoder (synthetic inputs), in the jepa.enc.* vocabulary.

Shapes follow the pages' ViT-Ti/L/g image and video workloads:
  hfvit Ti/14 224^2 image (fp32), V-JEPA 2 ViT-L/16 16x256^2 video (bf16, batch 1 and 8),
  V-JEPA 2.1 ViT-L/16 16x384^2 (interleaved RoPE + interpolate_rope + modality vector),
  LeVJEPA ViT-L/16 16x256^2 tubelet 1 (CLS + block-causal), V-JEPA 2 ViT-g/16 64x256^2,
  and the two fixed-table families at ViT-L/16 width: V-JEPA with its 3-D sin-cos table baked
  for 16x224^2 and resized (trilinear) to a 16x256^2 clip, I-JEPA with its [w | h] 2-D table
  baked for 224^2 and resized (bicubic) to 256^2 images, 8 per call.
`small()` shrinks a workload (frames, image size, depth) so the oracle finishes in
seconds while the geometry still spans several 128-row tiles with a ragged tail.
"""
from dataclasses import replace

from oracle import Config

HFVIT_TI14 = Config(embed_dim=192, n_layer=12, n_head=3, ffn_dim=768, patch_size=14, tubelet_size=1,
                    pos_type=1, cls_token=1, n_pos_rows=257)
VJEPA2_L16 = Config(embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, patch_size=16, tubelet_size=2,
                    pos_type=2, rope_layout=0)
VJEPA2_1_L16 = Config(embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, patch_size=16, tubelet_size=2,
                      pos_type=2, rope_layout=1, rope_interpolate=1, rope_ref_grid=16, modality_embed=1)
LEVJEPA_L16 = Config(embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, patch_size=16, tubelet_size=1,
                     pos_type=2, rope_layout=0, cls_token=1, attn_mode=1)
VJEPA_L16 = Config(embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, patch_size=16, tubelet_size=2,
                   pos_type=4, img_size=224, n_frames=16, sincos_uniform_power=1)
IJEPA_L16 = Config(embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, patch_size=16, tubelet_size=1,
                   pos_type=3, img_size=224, n_frames=1, sincos_w_first=1)
VJEPA2_G16 = Config(embed_dim=1408, n_layer=40, n_head=22, ffn_dim=6144, patch_size=16, tubelet_size=2,
                    pos_type=2, rope_layout=0)

# name -> (config, dtype, batches, (T, H, W), library preset name)
WORKLOADS = {
    "hfvit_ti14_224": (HFVIT_TI14, "fp32", (1,), (1, 224, 224)),
    "vjepa2_vitl16_16x256": (VJEPA2_L16, "bf16", (1, 8), (16, 256, 256)),
    "vjepa2_1_vitl16_16x384": (VJEPA2_1_L16, "bf16", (1,), (16, 384, 384)),
    "levjepa_vitl16_16x256": (LEVJEPA_L16, "bf16", (2,), (16, 256, 256)),
    "vjepa2_vitg16_64x256": (VJEPA2_G16, "bf16", (1,), (64, 256, 256)),
    "vjepa_vitl16_16x256": (VJEPA_L16, "bf16", (1,), (16, 256, 256)),
    "ijepa_vitl16_256": (IJEPA_L16, "bf16", (8,), (1, 256, 256)),
}


def small(name: str, n_layer: int = 2):
    """A reduced workload: same family and widths, few layers, a clip of a few hundred tokens."""
    cfg, dtype, batches, _ = WORKLOADS[name]
    if name == "hfvit_ti14_224":
        return replace(cfg, n_layer=n_layer), dtype, (1, 224, 224)
    if name == "vjepa2_vitl16_16x256":
        return replace(cfg, n_layer=n_layer), dtype, (4, 192, 176)      # 2x12x11 = 264 tokens
    if name == "vjepa2_1_vitl16_16x384":
        return replace(cfg, n_layer=n_layer), dtype, (4, 208, 160)      # 2x13x10 = 260 tokens, scale 15/12, 15/9
    if name == "levjepa_vitl16_16x256":
        return replace(cfg, n_layer=n_layer), dtype, (3, 160, 144)      # 3x10x9 + CLS = 271 tokens
    if name == "vjepa2_vitg16_64x256":
        return replace(cfg, n_layer=n_layer), dtype, (4, 160, 192)      # 2x10x12 = 240 tokens
    if name == "vjepa_vitl16_16x256":   # table baked for 2x12x12, resized to 2x13x11 = 286 tokens
        return replace(cfg, n_layer=n_layer, n_frames=4, img_size=192), dtype, (4, 208, 176)
    if name == "ijepa_vitl16_256":      # table baked for 14x14, resized to 17x15 = 255 tokens
        return replace(cfg, n_layer=n_layer), dtype, (1, 272, 240)
    raise KeyError(name)

# The V-JEPA 2 ViT-L masked predictor (jepa.pred.*): 12 layers of width 384, 12 heads of 32,
# over the 8 x 16 x 16 position grid of a 16 x 256^2 clip; the pages' worked predictor example
# takes the first half of the tokens as context and the second half as targets.
from oracle import PredConfig  # noqa: E402

PRED_VJEPA2_L16 = PredConfig(embed_dim=384, n_layer=12, n_head=12, ffn_dim=1536, enc_dim=1024, out_dim=1024,
                             n_mask_tokens=10, mask_index=1)
PRED_WORKLOAD = dict(grid=(8, 16, 16), n_ctx=1024, n_tgt=1024, batches=(1, 8))

# The V-JEPA 2 ViT-L SSv2 classifier head (jepa.head.*): 3 pooler layers, 174 classes, over the
# 2048 tokens of a 16 x 256^2 clip's encoder output.
from oracle import HeadConfig  # noqa: E402

HEAD_VJEPA2_L16_SSV2 = HeadConfig(embed_dim=1024, n_head=16, ffn_dim=4096, n_pool_layers=3, n_classes=174)
HEAD_WORKLOAD = dict(tokens=2048, batches=(1, 8))
