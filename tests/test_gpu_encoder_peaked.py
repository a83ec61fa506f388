"""Whole-encoder parity with peaked attention at the full token counts (GPU only).

With the plain N(0, 0.02) recipe the encoder's attention is nearly uniform (score std about 0.4),
so its output is close to the mean of V and barely depends on the RoPE layout or the mask: a key
range or tile-index error past the first few thousand keys could hide under the bf16 bar. Here the
q and k rows of every attn_qkv.weight are scaled by 2.5 and 2 (score std about 2.0), written in f32
into a forged GGUF file that the library loads as bf16, and drawn the same way by the oracle (its
test input option, which rounds the scaled weights to bf16 like the load does). At each workload's full token count (2048,
4608, 4097 x 2 clips, 8192 with 22 heads), two layers deep, every token must meet the bf16 bar
(per-token cosine >= 0.9999, max |d| <= 3e-2), and the control -- the same file with the other
RoPE layout, or without the block-causal mask -- must miss it ("Architecture", 3-D RoPE: the wrong
layout loses accuracy; Block-causal attention: the unmasked graph gives other tokens).
"""
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import gguf_forge as gf
import oracle
import synth
from configs import LEVJEPA_L16, VJEPA2_1_L16, VJEPA2_G16, VJEPA2_L16

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu

PEAKED = dict(n_layer=2, q_weight_scale=2.5, k_weight_scale=2.0)
# name -> (config, clips, (T, H, W), control: the hyper-parameter change that must fail the bar)
CASES = {
    "vjepa2_vitl16_16x256": (VJEPA2_L16, 1, (16, 256, 256), dict(rope_layout=1)),
    "vjepa2_1_vitl16_16x384": (VJEPA2_1_L16, 1, (16, 384, 384), dict(rope_layout=0)),
    "levjepa_vitl16_16x256": (LEVJEPA_L16, 2, (16, 256, 256), dict(attn_mode=0)),
    "vjepa2_vitg16_64x256": (VJEPA2_G16, 1, (64, 256, 256), dict(rope_layout=1)),
}


def bar(got, ref):
    got = got.reshape(-1, got.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    return float(cos.min()), float(np.abs(got - ref).max())


def encode_file(path, pix, T, H, W):
    model = jv.Model.from_gguf(path, dtype="bf16")
    ctx = jv.Context(model, pix.shape[0], T, H, W)
    out = ctx.encode(torch.from_numpy(pix).cuda())
    ctx.sync()
    res = out.cpu().double().numpy()
    ctx.close()
    return res


@pytest.mark.parametrize("name", list(CASES))
def test_peaked_attention_full_token_count(tmp_path, name):
    base, B, (T, H, W), control = CASES[name]
    cfg = replace(base, img_size=H, n_frames=T, **PEAKED)
    path = os.path.join(tmp_path, "peaked.gguf")
    tensors = gf.encoder_tensors(cfg)
    gf.write_gguf(path, gf.encoder_kvs(cfg), tensors)
    pix = synth.pixels(70, (B, T, 3, H, W))
    ref = oracle.encode(cfg, 0, True, pix)
    got = encode_file(path, pix, T, H, W)
    assert got.shape == ref.shape
    cos, err = bar(got, ref)
    d = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(d), d.shape)
    where = (f"worst element (item, token, column) {tuple(int(i) for i in worst)}, error quantiles 99/99.99 % "
             f"{np.quantile(d, 0.99):.2e} / {np.quantile(d, 0.9999):.2e}")
    assert cos >= 0.9999 and err <= 3e-2, f"{name}: min token cosine {cos:.6f}, max abs {err:.3e}; {where}"
    # the control file: same weights, the other layout or no mask
    gf.write_gguf(path, gf.encoder_kvs(replace(cfg, **control)), tensors)
    c_cos, c_err = bar(encode_file(path, pix, T, H, W), ref)
    assert c_cos < 0.9999 or c_err > 3e-2, f"{name} control {control}: cosine {c_cos:.6f}, max abs {c_err:.3e}"
    print(f"{name}: cos {cos:.7f} err {err:.2e} ({where}); control {control}: cos {c_cos:.5f} err {c_err:.2e}")
