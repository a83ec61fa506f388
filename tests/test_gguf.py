"""The GGUF encoder reader and its checks ("Architecture", Robustness: what the loader validates),
on forged files (CPU only: jepa_gguf_hparams reads no weights and makes no CUDA call).

Every row of the pages' validation table has a case here: header and counts, tensor extent
(a truncated file), architecture / family, integer and float ranges, enum strings,
block_causal on a family without a mask, derived invariants, tensor dtype, tensor shape and
required tensors; plus what this build cannot run (family lewm, other activations, register
tokens, layer scale, quantized weights), refused as unsupported.
"""
import ctypes
import os
from dataclasses import replace

import numpy as np
import pytest

import gguf_forge as gf
import oracle
from configs import HFVIT_TI14, IJEPA_L16, LEVJEPA_L16, VJEPA2_1_L16, VJEPA2_L16, VJEPA_L16

jv = pytest.importorskip("jepa_vision_encoder_gb300")
E_INVALID, E_UNSUP = jv._lib.E_INVALID_ARG, jv._lib.E_UNSUPPORTED

SMALL = {
    "vjepa2": replace(VJEPA2_L16, n_layer=1, img_size=256, n_frames=16),
    "vjepa2_1": replace(VJEPA2_1_L16, n_layer=1, img_size=384, n_frames=16),
    "levjepa": replace(LEVJEPA_L16, n_layer=1, img_size=256, n_frames=16),
    "hfvit": replace(HFVIT_TI14, n_layer=1, img_size=224, n_frames=1),
    "vjepa": replace(VJEPA_L16, n_layer=1),
    "ijepa": replace(IJEPA_L16, n_layer=1),
    "tiny": replace(VJEPA2_L16, n_layer=1, embed_dim=256, n_head=4, ffn_dim=512, img_size=256, n_frames=16),
}


def table_of(cfg):
    """The sin-cos table a converter bakes: the oracle's, rounded to float32."""
    g = cfg.img_size // cfg.patch_size
    if cfg.pos_type == 3:
        return oracle.sincos_2d(g, g, cfg.embed_dim, bool(cfg.sincos_w_first)).astype(np.float32)
    return oracle.sincos_3d(cfg.n_frames // cfg.tubelet_size, g, g, cfg.embed_dim,
                            bool(cfg.sincos_uniform_power)).astype(np.float32)


def forge(tmp_path, name, kvs=None, tensors=None, **kw):
    cfg = SMALL[name]
    kvs = gf.encoder_kvs(cfg) if kvs is None else kvs
    if tensors is None:
        tensors = gf.encoder_tensors(cfg, pos_table=table_of(cfg) if cfg.pos_type in (3, 4) else None)
    path = os.path.join(tmp_path, f"{name}.gguf")
    gf.write_gguf(path, kvs, tensors, **kw)
    return path


def refused(path, status, fragment):
    with pytest.raises(jv.JepaError) as e:
        jv.gguf_hparams(path)
    assert e.value.status == status, e.value
    assert fragment in e.value.text, e.value.text


@pytest.mark.parametrize("name", [n for n in SMALL if n != "tiny"])
def test_forged_files_give_their_hyper_parameters(tmp_path, name):
    cfg = SMALL[name]
    hp = jv.gguf_hparams(forge(tmp_path, name))
    for k in ("embed_dim", "n_layer", "n_head", "ffn_dim", "patch_size", "tubelet_size", "in_chans", "pos_type",
              "cls_token", "modality_embed", "attn_mode", "n_pos_rows"):
        assert getattr(hp, k) == getattr(cfg, k), k
    if cfg.pos_type == 2:
        assert (hp.rope_layout, hp.rope_interpolate, hp.rope_ref_grid) == (cfg.rope_layout, cfg.rope_interpolate,
                                                                          cfg.rope_ref_grid)
    assert jv.lib().jepa_hparams_validate(ctypes.byref(hp)) == 0


def test_split_qkv_projections_are_accepted(tmp_path):
    cfg = SMALL["tiny"]
    kvs = gf.set_kv(gf.encoder_kvs(cfg), "jepa.enc.qkv_fused", gf.BOOL, False)
    assert jv.gguf_hparams(forge(tmp_path, "tiny", kvs=kvs, tensors=gf.encoder_tensors(cfg, fused=False))).n_layer == 1
    refused(forge(tmp_path, "tiny", kvs=kvs), E_INVALID, "enc.blk.0.attn_q.weight is missing")


def test_header_and_extent(tmp_path):
    refused(forge(tmp_path, "tiny", magic=b"GGUX"), E_INVALID, "not a GGUF file")
    refused(forge(tmp_path, "tiny", version=1), E_INVALID, "version 1")
    refused(forge(tmp_path, "tiny", truncate=100), E_INVALID, "extends past the end of the file")
    path = os.path.join(tmp_path, "short.gguf")
    with open(path, "wb") as f:
        f.write(b"GGUF\x03\x00\x00\x00\x01")
    refused(path, E_INVALID, "truncated header")
    refused(forge(tmp_path, "tiny", alignment=24), E_INVALID, "offset not aligned")


KV_CASES = [
    ("general.architecture", gf.STRING, "llama", E_INVALID, "not jepa"),
    ("jepa.family", gf.STRING, "dinov9", E_INVALID, "not one of the seven families"),
    ("jepa.family", gf.STRING, "lewm", E_UNSUP, "lewm"),
    ("jepa.enc.embed_dim", gf.U32, 0, E_INVALID, "jepa.enc.embed_dim"),
    ("jepa.enc.embed_dim", gf.U32, 70000, E_INVALID, "jepa.enc.embed_dim"),
    ("jepa.enc.n_layer", gf.I32, -2, E_INVALID, "jepa.enc.n_layer"),
    ("jepa.enc.n_head", gf.U32, 15, E_INVALID, "not divisible by n_head"),
    ("jepa.enc.ffn_dim", gf.U64, 1 << 40, E_INVALID, "jepa.enc.ffn_dim"),
    ("jepa.enc.patch_size", gf.STRING, "16", E_INVALID, "not an integer"),
    ("jepa.enc.ln_eps", gf.F32, float("nan"), E_INVALID, "not finite"),
    ("jepa.enc.ln_eps", gf.F32, 2.0, E_INVALID, "ln_eps"),
    ("jepa.enc.rope_theta", gf.F32, 0.0, E_INVALID, "rope_theta"),
    ("jepa.enc.act", gf.STRING, "silu", E_UNSUP, "gelu_erf"),
    ("jepa.enc.act", gf.STRING, "relu6", E_INVALID, "unknown"),
    ("jepa.enc.pos_type", gf.STRING, "alibi", E_INVALID, "unknown"),
    ("jepa.enc.rope_freq_layout", gf.STRING, "zigzag", E_INVALID, "unknown"),
    ("jepa.enc.attn_mode", gf.STRING, "block_causal", E_INVALID, "has no mask"),
    ("jepa.enc.attn_mode", gf.STRING, "sliding", E_INVALID, "unknown"),
    ("jepa.enc.rope_interpolate", gf.BOOL, True, E_INVALID, "rope_ref_grid"),
    ("jepa.enc.n_registers", gf.U32, 4, E_UNSUP, "register"),
    ("jepa.enc.layer_scale", gf.BOOL, True, E_UNSUP, "layer scale"),
    ("jepa.enc.cls_token", gf.U32, 1, E_INVALID, "not a bool"),
    ("jepa.enc.img_size", None, None, E_INVALID, "required key jepa.enc.img_size"),
]


@pytest.mark.parametrize("key,t,v,status,fragment", KV_CASES)
def test_keys_are_checked(tmp_path, key, t, v, status, fragment):
    cfg = SMALL["tiny"]
    kvs = gf.encoder_kvs(cfg)
    if key == "jepa.enc.rope_interpolate":
        kvs = gf.set_kv(kvs, "jepa.enc.rope_ref_grid", gf.U32, None)
    kvs = gf.set_kv(kvs, key, t, v)
    refused(forge(tmp_path, "tiny", kvs=kvs), status, fragment)


def test_odd_head_width_on_a_rope_family(tmp_path):
    cfg = replace(SMALL["tiny"], embed_dim=90, n_head=6, ffn_dim=64)     # head width 15
    refused(forge(tmp_path, "tiny", kvs=gf.encoder_kvs(cfg), tensors=[]), E_INVALID, "odd head width")


def test_tensors_are_checked(tmp_path):
    cfg = SMALL["tiny"]
    ts = gf.encoder_tensors(cfg)

    def edit(name, fn):
        return [fn(t) if t[0] == name else t for t in ts]
    refused(forge(tmp_path, "tiny", tensors=[t for t in ts if t[0] != "enc.norm.bias"]), E_INVALID,
            "enc.norm.bias is missing")
    refused(forge(tmp_path, "tiny", tensors=edit("enc.blk.0.ln1.weight", lambda t: (t[0], t[1], gf.GGML_F16))),
            E_INVALID, "must be f32")
    refused(forge(tmp_path, "tiny", tensors=edit("enc.blk.0.ffn_up.weight", lambda t: (t[0], t[1][:-64], t[2]))),
            E_INVALID, "has shape [448, 256]")
    refused(forge(tmp_path, "tiny", tensors=edit("enc.blk.0.attn_out.weight", lambda t: (t[0], t[1], gf.GGML_Q8_0))),
            E_UNSUP, "q8_0")
    refused(forge(tmp_path, "tiny", tensors=ts + [ts[0]]), E_INVALID, "appears twice")


def test_matrix_types_f32_f16_bf16_are_accepted(tmp_path):
    cfg = SMALL["hfvit"]
    for mt in (gf.GGML_F32, gf.GGML_F16, gf.GGML_BF16):
        p = forge(tmp_path, "hfvit", tensors=gf.encoder_tensors(cfg, matrix_type=mt))
        assert jv.gguf_hparams(p).embed_dim == 192


def test_validation_comes_before_any_device_use(tmp_path):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    bad = forge(tmp_path, "tiny", kvs=gf.set_kv(gf.encoder_kvs(SMALL["tiny"]), "jepa.family", gf.STRING, "x"))
    assert jv.lib().jepa_model_load_gguf(bad.encode(), 1, 0, ctypes.byref(h)) == E_INVALID
    good = forge(tmp_path, "tiny")
    assert jv.lib().jepa_model_load_gguf(good.encode(), 1, 0, ctypes.byref(h)) == jv._lib.E_CUDA
