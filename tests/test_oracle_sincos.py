"""Pins of the oracle's fixed sin-cos position tables and their resizing (CPU only).

What fixes each function, other than the oracle itself:
  * the tables: the origin row, the unit circle of every (sin, cos) column pair, the frequency
    ladder read back from the table (1 down to 1/10000 in d/2 geometric steps), translation
    invariance of row dot products, the 3-D table reducing to the 2-D one on a single frame,
    the uniform-power cut, and the pages' own worked example (jepa.cpp "Converter", ijepa: the
    [w | h] and [h | w] orderings of the 16 x 16 x 1280 table differ by up to 2.0);
  * the resizing: PyTorch's interpolate (trilinear / bicubic, align_corners off) as the library
    routine the pages' runtime follows ("as HF does"), the identity at equal sizes, constants
    kept, and a hand-worked 2 -> 3 sample.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def axis_parts(D, kind, uniform=False):
    """Column ranges of the per-axis parts of a table row."""
    if kind == 2:
        return [(0, D // 2), (D // 2, D)]
    d = 2 * math.ceil(D / 6) if uniform else None
    widths = [d, d, d] if uniform else [D // 2, D // 4, D // 4]
    parts, o = [], 0
    for w in widths:
        parts.append((o, min(o + w, D)))
        o += w
    return parts


@pytest.mark.parametrize("w_first", [False, True])
def test_sincos_2d_origin_row_is_zero_sines_and_unit_cosines(w_first):
    t = oracle.sincos_2d(5, 7, 64, w_first)
    for a, b in axis_parts(64, 2):
        half = (b - a) // 2
        assert np.array_equal(t[0, a:a + half], np.zeros(half))
        assert np.array_equal(t[0, a + half:b], np.ones(half))


def test_sincos_pairs_lie_on_the_unit_circle():
    for t, parts in [(oracle.sincos_2d(6, 9, 96), axis_parts(96, 2)),
                     (oracle.sincos_3d(4, 5, 6, 128), axis_parts(128, 3)),
                     (oracle.sincos_3d(3, 4, 5, 126, True), axis_parts(126, 3, True))]:
        for a, b in parts:
            half = (b - a) // 2
            s, c = t[:, a:a + half], t[:, a + half:a + 2 * half]
            assert np.abs(s * s + c * c - 1.0).max() < 1e-14


@pytest.mark.parametrize("d_axis", [8, 32, 640])
def test_frequency_ladder_read_back_from_the_table(d_axis):
    # position 1 on the w axis: angle_k = w_k, recovered with atan2 (every w_k <= 1 < pi)
    t = oracle.sincos_2d(1, 2, 2 * d_axis, w_first=False)
    half = d_axis // 2
    s, c = t[1, d_axis:d_axis + half], t[1, d_axis + half:]
    w = np.arctan2(s, c)
    assert abs(w[0] - 1.0) < 1e-15
    ratio = w[1:] / w[:-1]
    assert np.abs(ratio - ratio[0]).max() < 1e-12          # geometric ladder
    assert abs(ratio[0] ** half - 1e-4) < 1e-15            # d/2 steps span 1 -> 1/10000
    # the h half of the same row is the origin
    assert np.array_equal(t[1, :half], np.zeros(half))


def test_row_dot_products_depend_only_on_the_offset():
    t = oracle.sincos_2d(1, 40, 64, w_first=True)   # one row of 40 positions: the w part is [0, 32)
    e = t[:, :32]
    g = e @ e.T
    for off in (0, 1, 5, 17):
        diag = np.diag(g, off)
        assert np.abs(diag - diag[0]).max() < 1e-12


def test_the_two_2d_orderings_swap_halves():
    a = oracle.sincos_2d(4, 6, 48, w_first=False)
    b = oracle.sincos_2d(4, 6, 48, w_first=True)
    assert np.array_equal(a[:, :24], b[:, 24:]) and np.array_equal(a[:, 24:], b[:, :24])


def test_ijepa_orderings_differ_by_up_to_two():
    # the pages' worked example: 16 x 16 x 1280, [w | h] against [h | w], "differs by up to 2.0"
    d = np.abs(oracle.sincos_2d(16, 16, 1280, True) - oracle.sincos_2d(16, 16, 1280, False)).max()
    assert 1.99 < d <= 2.0


def test_sincos_3d_on_one_frame_is_a_time_origin_and_the_2d_table():
    D = 256
    t3 = oracle.sincos_3d(1, 6, 5, D)
    t2 = oracle.sincos_2d(6, 5, D // 2, w_first=False)
    assert np.array_equal(t3[:, :D // 4], np.zeros((30, D // 4)))
    assert np.array_equal(t3[:, D // 4:D // 2], np.ones((30, D // 4)))
    assert np.abs(t3[:, D // 2:] - t2).max() < 1e-15


def test_sincos_3d_time_part_follows_the_frame_only():
    t = oracle.sincos_3d(3, 4, 5, 64).reshape(3, 4, 5, 64)
    tp = t[..., :32]
    assert np.array_equal(tp, np.broadcast_to(tp[:, :1, :1], tp.shape))
    wp = t[..., 48:]
    assert np.array_equal(wp, np.broadcast_to(wp[:1, :1, :], wp.shape))


def test_uniform_power_cuts_the_last_axis():
    # 1024 and 1026 both give axis width 2 ceil(D/6) = 342; the 1024 table is the 1026 one cut
    a = oracle.sincos_3d(2, 3, 4, 1024, True)
    b = oracle.sincos_3d(2, 3, 4, 1026, True)
    assert np.array_equal(a, b[:, :1024])
    # the h part of width 342 starts at column 342 and follows the row h alone
    h = a.reshape(2, 3, 4, 1024)[..., 342:684]
    assert np.array_equal(h, np.broadcast_to(h[:1, :, :1], h.shape))


def test_widths_the_split_cannot_take_are_refused():
    with pytest.raises(ValueError):
        oracle.sincos_2d(2, 2, 66)
    with pytest.raises(ValueError):
        oracle.sincos_3d(2, 2, 2, 68)        # D/4 = 17 is odd


def torch_resize(x, size, mode):
    xt = torch.from_numpy(np.ascontiguousarray(x))
    if mode == "trilinear":
        y = torch.nn.functional.interpolate(xt.permute(3, 0, 1, 2)[None], size=size, mode=mode, align_corners=False)
        return y[0].permute(1, 2, 3, 0).numpy()
    y = torch.nn.functional.interpolate(xt.permute(2, 0, 1)[None], size=size, mode=mode, align_corners=False)
    return y[0].permute(1, 2, 0).numpy()


@pytest.mark.parametrize("src,size", [((8, 14, 14), (8, 16, 16)), ((8, 16, 16), (8, 12, 20)), ((8, 14, 14), (4, 7, 9)),
                                      ((2, 3, 3), (5, 1, 6)), ((1, 4, 4), (3, 4, 4))])
def test_trilinear_matches_the_library_routine(src, size):
    x = np.random.default_rng(1).standard_normal(src + (24,))
    got = oracle.interp_trilinear(x, size)
    assert np.abs(got - torch_resize(x, size, "trilinear")).max() < 1e-13


@pytest.mark.parametrize("src,size", [((16, 16), (20, 18)), ((14, 14), (16, 16)), ((16, 16), (12, 9)), ((3, 2), (7, 1)),
                                      ((1, 5), (4, 5)), ((16, 16), (32, 32))])
def test_bicubic_matches_the_library_routine(src, size):
    x = np.random.default_rng(2).standard_normal(src + (20,))
    got = oracle.interp_bicubic(x, size)
    assert np.abs(got - torch_resize(x, size, "bicubic")).max() < 1e-13


def test_equal_sizes_are_the_identity_and_constants_stay():
    x = np.random.default_rng(3).standard_normal((3, 5, 7, 8))
    assert np.array_equal(oracle.interp_trilinear(x, (3, 5, 7)), x)
    assert np.array_equal(oracle.interp_bicubic(x[0], (5, 7)), x[0])
    c = np.full((4, 6, 3), 2.5)
    assert np.abs(oracle.interp_bicubic(c, (9, 5)) - 2.5).max() < 1e-14
    assert np.abs(oracle.interp_trilinear(c[None], (2, 9, 5)) - 2.5).max() < 1e-14


def test_linear_resize_of_two_samples_to_three_by_hand():
    # n_in 2 -> n_out 3: c = (o + 1/2) 2/3 - 1/2 = -1/6 (clamped to 0), 1/2, 7/6 (past the end)
    x = np.array([1.0, 4.0]).reshape(1, 1, 2, 1)
    got = oracle.interp_trilinear(x, (1, 1, 3)).ravel()
    assert np.allclose(got, [1.0, 2.5, 4.0], rtol=0, atol=1e-15)
    # cubic at c = 1/2 between samples 1, 4 with clamped outer taps: Keys weights at 3/2, 1/2, 1/2, 3/2
    w_out, w_in = -0.09375, 0.59375
    got = oracle.interp_bicubic(x[0], (1, 3)).ravel()
    assert abs(got[1] - ((w_out + w_in) * 1.0 + (w_in + w_out) * 4.0)) < 1e-15


def test_pos_table_at_the_training_grid_is_the_baked_table():
    from configs import VJEPA_L16
    from dataclasses import replace
    cfg = replace(VJEPA_L16, embed_dim=128, n_head=2)
    t = oracle.pos_table(cfg, 16, 224, 224)
    assert np.array_equal(t, oracle.sincos_3d(8, 14, 14, 128, bool(cfg.sincos_uniform_power)))
    r = oracle.pos_table(cfg, 16, 256, 256)
    base = oracle.sincos_3d(8, 14, 14, 128, bool(cfg.sincos_uniform_power)).reshape(8, 14, 14, 128)
    assert np.array_equal(r, oracle.interp_trilinear(base, (8, 16, 16)).reshape(-1, 128))


def test_pos_table_2d_refuses_several_frames():
    from configs import IJEPA_L16
    from dataclasses import replace
    cfg = replace(IJEPA_L16, embed_dim=128, n_head=2)
    with pytest.raises(ValueError):
        oracle.pos_table(cfg, 2, 224, 224)
    t = oracle.pos_table(cfg, 1, 256, 256)
    base = oracle.sincos_2d(14, 14, cfg.embed_dim, True).reshape(14, 14, -1)
    assert np.array_equal(t, oracle.interp_bicubic(base, (16, 16)).reshape(-1, cfg.embed_dim))
