"""CPU-only checks of the C ABI: the library loads, exports every entry point include/jepa.h
declares, and its host-side logic (presets, validation, token geometry, argument refusal)
behaves as the pages' robustness rules say. No kernel is launched here."""
import ctypes
import os
import re
import threading

import pytest

import jepa_vision_encoder_gb300 as jv
from jepa_vision_encoder_gb300 import _lib
from configs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(?:jepa_status|void|const char\s*\*|int32_t|int)\s+\**\s*(jepa_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    L = jv.lib()
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    # the Python binding covers the whole surface
    assert names <= set(_lib.SIGNATURES), names - set(_lib.SIGNATURES)


PRESET_OF = {
    "hfvit_ti14_224": "hfvit_ti14",
    "vjepa2_vitl16_16x256": "vjepa2_vitl16",
    "vjepa2_1_vitl16_16x384": "vjepa2_1_vitl16",
    "levjepa_vitl16_16x256": "levjepa_vitl16",
    "vjepa2_vitg16_64x256": "vjepa2_vitg16",
    "vjepa_vitl16_16x256": "vjepa_vitl16",
    "ijepa_vitl16_256": "ijepa_vitl16",
}


@pytest.mark.parametrize("workload", list(WORKLOADS))
def test_presets_match_workloads(workload):
    cfg, dtype, batches, (T, H, W) = WORKLOADS[workload]
    hp = jv.preset(PRESET_OF[workload])
    for k in ("embed_dim", "n_layer", "n_head", "ffn_dim", "patch_size", "tubelet_size", "in_chans", "pos_type",
              "rope_layout", "rope_interpolate", "rope_ref_grid", "cls_token", "modality_embed", "attn_mode",
              "n_pos_rows", "sincos_w_first", "sincos_uniform_power"):
        assert getattr(hp, k) == getattr(cfg, k), k
    if cfg.pos_type in (_lib.POS_SINCOS2D, _lib.POS_SINCOS3D):   # the grid the table is baked for
        assert (hp.img_size, hp.n_frames) == (cfg.img_size, cfg.n_frames)
    assert abs(hp.ln_eps - cfg.ln_eps) < 1e-12 and hp.rope_theta == cfg.rope_theta
    assert jv.lib().jepa_hparams_validate(ctypes.byref(hp)) == 0
    import oracle
    assert jv.n_tokens(hp, T, H, W) == oracle.n_tokens(cfg, T, H, W)


def test_predictor_preset_matches_its_config():
    from configs import PRED_VJEPA2_L16
    hp = jv.pred_preset("vjepa2_vitl16")
    for k in ("embed_dim", "n_layer", "n_head", "ffn_dim", "enc_dim", "out_dim", "n_mask_tokens", "mask_index",
              "rope_layout"):
        assert getattr(hp, k) == getattr(PRED_VJEPA2_L16, k), k
    assert jv.lib().jepa_pred_hparams_validate(ctypes.byref(hp)) == 0
    L = jv.lib()
    for kw, frag in [(dict(n_head=7), "not divisible"), (dict(embed_dim=33 * 12), "odd"), (dict(mask_index=-1), "mask_index"),
                     (dict(rope_layout=3), "rope_layout"), (dict(n_layer=0), "n_layer")]:
        bad = jv.pred_preset("vjepa2_vitl16")
        for k, v in kw.items():
            setattr(bad, k, v)
        expect(L.jepa_pred_hparams_validate(ctypes.byref(bad)), _lib.E_INVALID_ARG, frag)
    expect(L.jepa_pred_preset(b"nope", ctypes.byref(hp)), _lib.E_INVALID_ARG, "unknown preset")
    expect(L.jepa_predict(None, None, 1, 1, None, 0, None, 1, 1, 1, 1, None), _lib.E_INVALID_ARG)


def test_head_preset_matches_its_config():
    from configs import HEAD_VJEPA2_L16_SSV2
    hp = jv.head_preset("vjepa2_vitl16_ssv2")
    for k in ("embed_dim", "n_head", "ffn_dim", "n_pool_layers", "n_classes"):
        assert getattr(hp, k) == getattr(HEAD_VJEPA2_L16_SSV2, k), k
    L = jv.lib()
    assert L.jepa_head_hparams_validate(ctypes.byref(hp)) == 0
    for kw, frag in [(dict(n_head=7), "not divisible"), (dict(n_classes=0), "n_classes"),
                     (dict(n_pool_layers=-1), "n_pool_layers"), (dict(ln_eps=-1.0), "ln_eps")]:
        bad = jv.head_preset("vjepa2_vitl16_ssv2")
        for k, v in kw.items():
            setattr(bad, k, v)
        expect(L.jepa_head_hparams_validate(ctypes.byref(bad)), _lib.E_INVALID_ARG, frag)
    expect(L.jepa_head_forward(None, None, 1, 1, None, None), _lib.E_INVALID_ARG)
    expect(L.jepa_op_pool(0, None, 1, 1, 4, 0, None, None), _lib.E_INVALID_ARG)


def test_token_counts():
    assert jv.n_tokens(jv.preset("vjepa2_vitg16"), 64, 256, 256) == 8192
    hp = jv.preset("levjepa_vitl16")
    assert jv.n_tokens(hp, 16, 224, 224) == 3137
    assert jv.n_tokens(hp, 16, 256, 256) == 4097
    assert jv.n_tokens(jv.preset("vjepa2_1_vitl16"), 16, 384, 384) == 4608


def expect(status, code, fragment=None):
    assert status == code, (status, jv.lib().jepa_error_text())
    if fragment:
        assert fragment in jv.lib().jepa_error_text().decode()


def test_refusals_by_name():
    L = jv.lib()
    hp = jv.preset("vjepa2_vitl16")
    n = ctypes.c_int32()
    expect(L.jepa_n_tokens(ctypes.byref(hp), 15, 256, 256, ctypes.byref(n)), _lib.E_INVALID_ARG, "not divisible")
    expect(L.jepa_n_tokens(ctypes.byref(hp), 16, 250, 256, ctypes.byref(n)), _lib.E_INVALID_ARG, "not divisible")
    expect(L.jepa_n_tokens(ctypes.byref(hp), 0, 256, 256, ctypes.byref(n)), _lib.E_INVALID_ARG)
    expect(L.jepa_preset(b"no_such_model", ctypes.byref(hp)), _lib.E_INVALID_ARG, "unknown preset")
    cases = [
        ("vjepa2_vitl16", dict(n_head=15), "not divisible by n_head"),
        ("vjepa2_vitl16", dict(embed_dim=75, n_head=5), "odd head width"),
        ("vjepa2_1_vitl16", dict(rope_ref_grid=0), "rope_ref_grid"),
        ("vjepa2_vitl16", dict(ln_eps=float("nan")), "ln_eps"),
        ("vjepa2_vitl16", dict(n_layer=0), "n_layer"),
        ("hfvit_ti14", dict(n_pos_rows=0), "n_pos_rows"),
        ("vjepa2_vitl16", dict(attn_mode=7), "attn_mode"),
        ("vjepa2_vitl16", dict(rope_theta=-1.0), "rope_theta"),
        ("vjepa2_vitl16", dict(pos_type=5), "pos_type"),
        ("vjepa_vitl16", dict(img_size=200), "multiple of patch"),
        ("vjepa_vitl16", dict(n_frames=15), "multiple of tubelet"),
        ("vjepa_vitl16", dict(embed_dim=1028, n_head=4, sincos_uniform_power=0), "sin-cos axes"),
        ("ijepa_vitl16", dict(embed_dim=1026, n_head=18), "sin-cos axes"),
    ]
    for name, kw, frag in cases:
        bad = jv.preset(name)
        for k, v in kw.items():
            setattr(bad, k, v)
        expect(L.jepa_hparams_validate(ctypes.byref(bad)), _lib.E_INVALID_ARG, frag)


def test_null_arguments_refused():
    L = jv.lib()
    expect(L.jepa_encode(None, None, 1, 16, 256, 256, 0, None), _lib.E_INVALID_ARG)
    expect(L.jepa_context_sync(None), _lib.E_INVALID_ARG)
    expect(L.jepa_model_tensor(None, b"enc.norm.weight", None, 0), _lib.E_INVALID_ARG)
    expect(L.jepa_op_attention(1, None, 1, 1, 1, 64, 0, 0, 1, None, None), _lib.E_INVALID_ARG)
    L.jepa_error_reset()
    assert L.jepa_error_text() == b""


def test_error_text_is_thread_local():
    L = jv.lib()
    L.jepa_error_reset()
    seen = {}

    def worker():
        hp = jv.preset("vjepa2_vitl16")
        hp.n_layer = 0
        L.jepa_hparams_validate(ctypes.byref(hp))
        seen["other"] = L.jepa_error_text()

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert b"n_layer" in seen["other"]
    assert L.jepa_error_text() == b""


def test_model_load_without_gpu_is_refused_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    hp = jv.preset("hfvit_ti14")
    h = ctypes.c_void_p()
    st = jv.lib().jepa_model_load(ctypes.byref(hp), 0, 0, 0, ctypes.byref(h))
    assert st == _lib.E_CUDA and not h.value
