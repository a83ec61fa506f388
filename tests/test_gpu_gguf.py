"""Encoders loaded from forged GGUF files, on the GPU (GPU only).

A file written from the generator's weights (bf16 matrices as bf16 or f32, fused or split q / k /
v) loads to the same model as the synthetic preset, so the two encode bit for bit alike; f16
matrices load as their exact f16 values; a sin-cos file's stored table is used as stored (and
resized for other grids), checked against the oracle under the encoder's bf16 bar.
"""
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import gguf_forge as gf
import oracle
import synth
from configs import HFVIT_TI14, VJEPA2_L16, VJEPA_L16

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu


def write(tmp_path, cfg, **kw):
    path = os.path.join(tmp_path, "m.gguf")
    gf.write_gguf(path, gf.encoder_kvs(cfg), gf.encoder_tensors(cfg, **kw))
    return path


def encode(model, pix, T, H, W):
    ctx = jv.Context(model, pix.shape[0], T, H, W)
    out = ctx.encode(torch.from_numpy(pix).cuda())
    ctx.sync()
    return out.cpu()


@pytest.mark.parametrize("matrix_type,fused", [(gf.GGML_BF16, True), (gf.GGML_F32, True), (gf.GGML_BF16, False)])
def test_file_model_encodes_like_the_synthetic_model(tmp_path, matrix_type, fused):
    cfg = replace(VJEPA2_L16, n_layer=2, img_size=256, n_frames=16)
    path = write(tmp_path, cfg, matrix_type=matrix_type, fused=fused)
    if not fused:
        kvs = gf.set_kv(gf.encoder_kvs(cfg), "jepa.enc.qkv_fused", gf.BOOL, False)
        gf.write_gguf(path, kvs, gf.encoder_tensors(cfg, matrix_type=matrix_type, fused=False))
    from_file = jv.Model.from_gguf(path, dtype="bf16")
    synthetic = jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16", n_layer=2)
    pix = synth.pixels(40, (2, 4, 3, 192, 176))
    assert torch.equal(encode(from_file, pix, 4, 192, 176), encode(synthetic, pix, 4, 192, 176))
    name = "enc.blk.1.attn_qkv.weight"
    assert torch.equal(from_file.tensor(name, (3072, 1024)), synthetic.tensor(name, (3072, 1024)))


def test_fp32_model_from_f32_file_and_f16_matrices(tmp_path):
    cfg = replace(HFVIT_TI14, n_layer=2, img_size=224, n_frames=1)
    path = write(tmp_path, cfg, matrix_type=gf.GGML_F32, round_bf16=False)
    pix = synth.pixels(41, (1, 1, 3, 224, 224))
    a = encode(jv.Model.from_gguf(path, dtype="fp32"), pix, 1, 224, 224)
    b = encode(jv.Model.preset("hfvit_ti14", seed=0, dtype="fp32", n_layer=2), pix, 1, 224, 224)
    assert torch.equal(a, b)
    path16 = write(tmp_path, cfg, matrix_type=gf.GGML_F16, round_bf16=False)
    m16 = jv.Model.from_gguf(path16, dtype="fp32")
    w = synth.param(0, "enc.blk.0.ffn_up.weight", (768, 192), False)
    assert np.array_equal(m16.tensor("enc.blk.0.ffn_up.weight", (768, 192)).numpy(), w.astype(np.float16).astype(np.float32))


def test_sincos_file_table_is_used_and_resized(tmp_path):
    cfg = replace(VJEPA_L16, n_layer=2, n_frames=4, img_size=192)         # table for 2 x 12 x 12
    table = oracle.sincos_3d(2, 12, 12, 1024, True).astype(np.float32)
    path = write(tmp_path, cfg, pos_table=table)
    model = jv.Model.from_gguf(path, dtype="bf16")
    assert np.array_equal(model.tensor("enc.pos_embed", (288, 1024)).numpy(), table)
    for T, H, W in [(4, 192, 192), (4, 208, 176)]:
        pix = synth.pixels(42, (1, T, 3, H, W))
        got = encode(model, pix, T, H, W).double().numpy().reshape(-1, 1024)
        ref = oracle.encode(cfg, 0, True, pix).reshape(-1, 1024)
        cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
        assert cos.min() >= 0.9999 and np.abs(got - ref).max() <= 3e-2
