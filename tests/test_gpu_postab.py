"""Fixed sin-cos position tables and their resizing on the GPU, against the oracle (GPU only).

Bars: the table kernel computes in double and stores float, so each entry is within one float
rounding (2^-24 relative, values in [-1, 1]) of the oracle's; the resize kernel computes in float
with at most 16 taps, so max |d| <= 1e-5 * max |src|. The encoder cases check the whole forward
with a baked table at the training grid and a resized one, through one context that switches
between the two.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from configs import IJEPA_L16, VJEPA_L16
from dataclasses import replace

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    yield
    torch.cuda.synchronize()
    assert jv.ops.device_status() == 0


TABLES = [
    (jv.POS_SINCOS2D, (1, 14, 14), 1024, True, False),
    (jv.POS_SINCOS2D, (1, 16, 16), 1280, False, False),
    (jv.POS_SINCOS2D, (1, 5, 9), 64, True, False),
    (jv.POS_SINCOS3D, (8, 14, 14), 1024, False, True),
    (jv.POS_SINCOS3D, (8, 14, 14), 1024, False, False),
    (jv.POS_SINCOS3D, (3, 7, 5), 1026, False, True),
    (jv.POS_SINCOS3D, (2, 4, 6), 1408, False, False),
]


@pytest.mark.parametrize("kind,grid,D,w_first,uniform", TABLES)
def test_sincos_table_matches_oracle(kind, grid, D, w_first, uniform):
    gt, gh, gw = grid
    got = jv.ops.sincos_table(kind, gt, gh, gw, D, w_first, uniform).cpu().double().numpy()
    ref = oracle.sincos_2d(gh, gw, D, w_first) if kind == jv.POS_SINCOS2D else oracle.sincos_3d(gt, gh, gw, D, uniform)
    assert np.abs(got - ref).max() <= 2.0 ** -24


RESIZES = [
    (jv.RESIZE_TRILINEAR, (8, 14, 14), (8, 16, 16)),
    (jv.RESIZE_TRILINEAR, (2, 12, 12), (2, 13, 11)),
    (jv.RESIZE_TRILINEAR, (8, 16, 16), (4, 7, 9)),
    (jv.RESIZE_TRILINEAR, (8, 14, 14), (32, 16, 16)),
    (jv.RESIZE_TRILINEAR, (1, 3, 3), (2, 1, 5)),
    (jv.RESIZE_BICUBIC, (1, 14, 14), (1, 16, 16)),
    (jv.RESIZE_BICUBIC, (1, 14, 14), (1, 17, 15)),
    (jv.RESIZE_BICUBIC, (1, 16, 16), (1, 12, 9)),
    (jv.RESIZE_BICUBIC, (1, 1, 5), (1, 4, 5)),
    (jv.RESIZE_BICUBIC, (2, 6, 4), (2, 9, 11)),
]


@pytest.mark.parametrize("mode,src_grid,dst_grid", RESIZES)
@pytest.mark.parametrize("D", [64, 1024])
def test_pos_resize_matches_oracle(mode, src_grid, dst_grid, D):
    src = np.random.default_rng(7).standard_normal(src_grid + (D,)).astype(np.float32)
    got = jv.ops.pos_resize(torch.from_numpy(src.reshape(-1, D)).cuda(), src_grid, dst_grid, mode)
    got = got.cpu().double().numpy().reshape(dst_grid + (D,))
    if mode == jv.RESIZE_TRILINEAR:
        ref = oracle.interp_trilinear(src, dst_grid)
    else:
        ref = np.stack([oracle.interp_bicubic(src[t], dst_grid[1:]) for t in range(src_grid[0])])
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(src).max()


def test_equal_grids_copy_exactly():
    src = torch.randn(3 * 5 * 7, 32, device="cuda")
    assert torch.equal(jv.ops.pos_resize(src, (3, 5, 7), (3, 5, 7), jv.RESIZE_TRILINEAR), src)
    assert torch.equal(jv.ops.pos_resize(src, (3, 5, 7), (3, 5, 7), jv.RESIZE_BICUBIC), src)


@pytest.mark.parametrize("name,grid,rows", [("vjepa_vitl16", (8, 14, 14), 1568), ("ijepa_vitl16", (1, 14, 14), 196)])
def test_model_holds_the_table_of_its_training_grid(name, grid, rows):
    model = jv.Model.preset(name, seed=0, dtype="bf16", n_layer=1)
    got = model.tensor("enc.pos_embed", (rows, 1024)).double().numpy()
    ref = (oracle.sincos_3d(*grid, 1024, True) if name == "vjepa_vitl16"
           else oracle.sincos_2d(grid[1], grid[2], 1024, True))
    assert np.abs(got - ref).max() <= 2.0 ** -24


def check_tokens(got, ref, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    assert cos.min() >= 0.9999, f"{what}: min token cosine {cos.min():.7f}"
    assert np.abs(got - ref).max() <= 3e-2, f"{what}: max abs err {np.abs(got - ref).max():.3e}"


def test_vjepa_encoder_native_and_resized_grids_through_one_context():
    cfg = replace(VJEPA_L16, n_layer=2, n_frames=4, img_size=192)       # table baked for 2 x 12 x 12
    model = jv.Model.preset("vjepa_vitl16", seed=0, dtype="bf16", n_layer=2, n_frames=4, img_size=192)
    ctx = jv.Context(model, 2, 4, 208, 192)
    shapes = [(4, 192, 192), (4, 208, 176), (4, 192, 192)]               # native, resized, native again
    outs = []
    for i, (T, H, W) in enumerate(shapes):
        pix = synth.pixels(20 + i, (2, T, 3, H, W))
        out = ctx.encode(torch.from_numpy(pix).cuda()).cpu().numpy()
        outs.append(out)
        check_tokens(out, oracle.encode(cfg, 0, True, pix), f"{T}x{H}x{W}")


def test_fp32_sincos2d_encoder():
    cfg = replace(IJEPA_L16, embed_dim=192, n_head=3, ffn_dim=768, n_layer=2, patch_size=14, img_size=224)
    model = jv.Model(jv.hparams(**{k: getattr(cfg, k) for k in (
        "embed_dim", "n_layer", "n_head", "ffn_dim", "patch_size", "tubelet_size", "pos_type", "img_size",
        "n_frames", "sincos_w_first")}), seed=0, dtype="fp32")
    for H, W in [(224, 224), (252, 196)]:                                 # 16 x 16 baked; 18 x 14 resized
        ctx = jv.Context(model, 1, 1, H, W)
        pix = synth.pixels(30, (1, 1, 3, H, W))
        out = ctx.encode(torch.from_numpy(pix).cuda()).cpu().double().numpy()
        ref = oracle.encode(cfg, 0, False, pix)
        assert np.abs(out - ref).max() / np.abs(ref).max() <= 1e-4


def test_sincos_refusals():
    L = jv.lib()
    t = torch.empty(64, device="cuda")
    assert L.jepa_op_sincos_table(jv.POS_SINCOS2D, 2, 2, 2, 8, 0, 0, t.data_ptr(), None) == jv._lib.E_INVALID_ARG
    assert L.jepa_op_sincos_table(jv.POS_SINCOS3D, 1, 2, 2, 12, 0, 0, t.data_ptr(), None) == jv._lib.E_INVALID_ARG
    assert L.jepa_op_sincos_table(jv.POS_LEARNED, 1, 2, 2, 8, 0, 0, t.data_ptr(), None) == jv._lib.E_INVALID_ARG
    u = torch.empty(4096, device="cuda")
    assert L.jepa_op_pos_resize(t.data_ptr(), 1, 2, 2, 16, jv.RESIZE_BICUBIC, u.data_ptr(), 2, 2, 2,
                                None) == jv._lib.E_INVALID_ARG
    assert L.jepa_op_pos_resize(t.data_ptr(), 1, 2, 2, 16, 3, u.data_ptr(), 1, 2, 2, None) == jv._lib.E_INVALID_ARG
    assert L.jepa_op_pos_resize(t.data_ptr(), 1, 2, 2, 16, 0, t.data_ptr() + 64, 1, 2, 2,
                                None) == jv._lib.E_INVALID_ARG   # overlapping
    with pytest.raises(jv.JepaError) as e:
        jv.Model.preset("vjepa_vitl16", seed=0, dtype="bf16", n_layer=1, cls_token=1)
    assert e.value.status == jv._lib.E_UNSUPPORTED
    model = jv.Model.preset("ijepa_vitl16", seed=0, dtype="bf16", n_layer=1)
    ctx = jv.Context(model, 1, 2, 64, 64)
    with pytest.raises(jv.JepaError) as e:    # a 2-D table has no time axis
        ctx.encode(torch.zeros((1, 2, 3, 64, 64), dtype=torch.float32, device="cuda"))
    assert e.value.status == jv._lib.E_UNSUPPORTED
