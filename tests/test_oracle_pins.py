"""Pins of the oracle to what the pages and the mathematics fix (CPU only).

Each test checks an oracle function against something other than itself: a value
the pages print (tests/golden/printed_values.json), a closed form, an invariant,
a special case that reduces to a library routine (torch conv3d / layer_norm /
scaled_dot_product_attention, numpy complex multiplication, math.erf), or brute
force on tiny inputs. A plausible slip in the oracle (dropped term, wrong sign or
index, transposed operand, wrong RoPE layout, wrong mask edge) fails one of them.
"""
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import Config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "printed_values.json")


def tiny_video(**kw):
    base = dict(embed_dim=24, n_layer=2, n_head=2, ffn_dim=40, patch_size=4, tubelet_size=2, pos_type=2)
    base.update(kw)
    return Config(**base)


# ---------------------------------------------------------------- patchify / embed
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("t", [1, 2])
def test_patch_embed_equals_strided_conv3d(layout, t):
    """Rearrangement + matmul == Conv3d with kernel = stride = (t, P, P) (Architecture, shared ViT graph)."""
    cfg = tiny_video(tubelet_size=t, embed_dim=12)
    B, T, C, H, W = 2, 4, 3, 12, 8
    rng = np.random.default_rng(1)
    pix_tchw = rng.uniform(-2, 2, size=(B, T, C, H, W)).astype(np.float32)
    pix = pix_tchw if layout == 0 else np.ascontiguousarray(pix_tchw.transpose(0, 2, 1, 3, 4))
    w = rng.normal(size=(12, C, t, 4, 4))
    b = rng.normal(size=12)
    # library routine: torch conv3d over [B, C, T, H, W]
    ref = torch.nn.functional.conv3d(torch.from_numpy(pix_tchw.transpose(0, 2, 1, 3, 4).astype(np.float64)),
                                     torch.from_numpy(w), torch.from_numpy(b), stride=(t, 4, 4))
    ref = ref.permute(0, 2, 3, 4, 1).numpy()  # [B, gt, gh, gw, D]
    patches = oracle.patchify(cfg, pix, layout)
    emb = oracle.linear(patches, w.reshape(12, -1), b).reshape(ref.shape)
    assert np.abs(emb - ref).max() < 1e-12
    brute = oracle.conv3d(cfg, pix, w, b, layout)
    assert np.abs(brute - ref).max() < 1e-12


def test_patch_element_and_token_order():
    """Element order (c, dt, dy, dx) and token order (t, h, w) (SkyVision V-JEPA 2 section; schema Token order)."""
    cfg = tiny_video(tubelet_size=2, patch_size=2)
    B, T, C, H, W = 1, 4, 3, 4, 6
    pix = np.arange(B * T * C * H * W, dtype=np.float32).reshape(B, T, C, H, W)
    p = oracle.patchify(cfg, pix, 0)
    gt, gh, gw = 2, 2, 3
    for tt in range(gt):
        for hh in range(gh):
            for ww in range(gw):
                i = tt * gh * gw + hh * gw + ww
                k = 0
                for c in range(C):
                    for dt in range(2):
                        for dy in range(2):
                            for dx in range(2):
                                assert p[i, k] == pix[0, tt * 2 + dt, c, hh * 2 + dy, ww * 2 + dx]
                                k += 1


def test_token_counts_printed():
    g = json.load(open(GOLDEN))
    for row in g["token_counts"]:
        cfg = tiny_video(patch_size=row["patch"], tubelet_size=row["tubelet"], cls_token=row["cls"])
        assert oracle.n_tokens(cfg, row["T"], row["H"], row["W"]) == row["N"], row["cite"]
    cfg = tiny_video(patch_size=16, tubelet_size=2)
    assert oracle.n_tokens(cfg, 16, 256, 256) == 2048
    assert oracle.n_tokens(cfg, 15, 256, 256) == -1  # not divisible by the tubelet


# ---------------------------------------------------------------- linear / LN / GELU
def test_linear_matches_matmul():
    rng = np.random.default_rng(2)
    x, w, b = rng.normal(size=(37, 29)), rng.normal(size=(13, 29)), rng.normal(size=13)
    assert np.abs(oracle.linear(x, w, b) - (x @ w.T + b)).max() < 1e-12
    # weights are [out, in]: using w un-transposed would not match
    sq = rng.normal(size=(13, 13))
    assert np.abs(oracle.linear(x[:, :13], sq) - x[:, :13] @ sq).max() > 1e-3


def test_layernorm_library_and_closed_forms():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(9, 33)) * 5 + 40.0  # offset rows: centred variance matters
    g, b = rng.normal(size=33), rng.normal(size=33)
    y = oracle.layernorm(x, g, b, 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), torch.from_numpy(b), 1e-6)
    assert np.abs(y - ref.numpy()).max() < 1e-12
    # constant row -> beta exactly
    yc = oracle.layernorm(np.full((2, 33), 7.25), g, b, 1e-6)
    assert np.abs(yc - b).max() < 1e-15
    # normalised row: mean 0, biased variance var/(var+eps)
    eps = 0.5
    yn = oracle.layernorm(x, np.ones(33), np.zeros(33), eps)
    var = x.var(axis=1)
    assert np.abs(yn.mean(axis=1)).max() < 1e-12
    assert np.abs(yn.var(axis=1) - var / (var + eps)).max() < 1e-12


def test_gelu_erf():
    xs = np.linspace(-8, 8, 161)
    y = oracle.gelu(xs)
    ref = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in xs])
    assert np.abs(y - ref).max() < 1e-15
    # not the tanh approximation
    tanh = 0.5 * xs * (1 + np.tanh(math.sqrt(2 / math.pi) * (xs + 0.044715 * xs ** 3)))
    assert np.abs(y - tanh).max() > 1e-4


# ---------------------------------------------------------------- RoPE
def rope_cfg(layout, hd=64, heads=2, **kw):
    return tiny_video(embed_dim=hd * heads, n_head=heads, rope_layout=layout, patch_size=2, **kw)


def test_rope_split_printed():
    g = json.load(open(GOLDEN))
    for key in ("rope_split", "rope_split_predictor"):
        hd, per = g[key]["head_dim"], g[key]["per_axis"]
        cfg = rope_cfg(0, hd=hd)
        c, s = oracle.rope_tables(cfg, 4, 8, 8)
        # a late token has every rotated dim away from cos 1 / sin 0, untouched dims exactly identity
        row = c.shape[0] - 1
        rotated = np.nonzero(s[row] != 0.0)[0]
        assert len(rotated) == 3 * per
        assert rotated.max() == 3 * per - 1
        if "untouched" in g[key]:
            assert hd - 3 * per == g[key]["untouched"]
            assert np.all(c[row, 3 * per:] == 1.0) and np.all(s[row, 3 * per:] == 0.0)


@pytest.mark.parametrize("layout", [0, 1])
def test_rope_identity_at_position_zero(layout):
    cfg = rope_cfg(layout)
    c, s = oracle.rope_tables(cfg, 4, 8, 8)
    x = np.random.default_rng(4).normal(size=(c.shape[0], cfg.embed_dim))
    y = oracle.rope_apply(x, cfg.n_head, c, s)
    assert np.array_equal(y[0], x[0])        # token 0 sits at (0, 0, 0)
    assert not np.allclose(y[-1], x[-1])


def test_rope_frequencies_closed_form():
    """omega_k = 1/10000^(2k/d): at d = 20, omega_0 = 1 and omega_5 = 10000^-1/2 = 0.01 exactly."""
    cfg = rope_cfg(1)  # interleaved: columns 2k, 2k+1 carry omega_k
    T, H, W = 2 * 7, 2, 2  # gt = 7 frames -> token with t = 3 exists
    c, s = oracle.rope_tables(cfg, T, H, W)
    pos = oracle.rope_positions(cfg, T, H, W)
    i = int(np.nonzero((pos[:, 0] == 3) & (pos[:, 1] == 0) & (pos[:, 2] == 0))[0][0])
    assert abs(c[i, 0] - math.cos(3.0)) < 1e-15 and abs(s[i, 1] - math.sin(3.0)) < 1e-15
    assert abs(s[i, 0] + math.sin(3.0)) < 1e-15          # even member carries -sin
    assert abs(c[i, 10] - math.cos(0.03)) < 1e-15        # k = 5 -> omega = 0.01
    assert abs(c[i, 20] - 1.0) == 0.0                    # h axis at h = 0


def test_rope_interleaved_is_complex_rotation():
    """Interleaved layout = textbook RoPE: each pair (x[2k], x[2k+1]) is multiplied by e^{i theta_k}."""
    cfg = rope_cfg(1, heads=1)
    T, H, W = 6, 10, 8
    c, s = oracle.rope_tables(cfg, T, H, W)
    pos = oracle.rope_positions(cfg, T, H, W)
    x = np.random.default_rng(5).normal(size=(c.shape[0], 64))
    y = oracle.rope_apply(x, 1, c, s)
    d = 20
    omega = 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    for i in range(c.shape[0]):
        for a in range(3):
            z = x[i, a * d:(a + 1) * d:2] + 1j * x[i, a * d + 1:(a + 1) * d:2]
            z = z * np.exp(1j * pos[i, a] * omega)
            assert np.abs(y[i, a * d:(a + 1) * d:2] - z.real).max() < 1e-13
            assert np.abs(y[i, a * d + 1:(a + 1) * d:2] - z.imag).max() < 1e-13
        assert np.array_equal(y[i, 60:], x[i, 60:])
    # norm preserved
    assert np.abs(np.linalg.norm(y, axis=1) - np.linalg.norm(x, axis=1)).max() < 1e-12


def test_rope_interleaved_scores_depend_on_offset_only():
    """A true rotation gives <R(p)q, R(p')k> = f(p - p'); the tiled quirk does not."""
    T, H, W = 8, 12, 12
    rng = np.random.default_rng(6)
    q, k = rng.normal(size=64), rng.normal(size=64)

    def score(layout, pa, pb):
        cfg = rope_cfg(layout, heads=1)
        c, s = oracle.rope_tables(cfg, T, H, W)
        pos = oracle.rope_positions(cfg, T, H, W)
        ia = int(np.nonzero((pos == pa).all(axis=1))[0][0])
        ib = int(np.nonzero((pos == pb).all(axis=1))[0][0])
        X = np.zeros((c.shape[0], 64))
        X[ia] = q
        Y = np.zeros((c.shape[0], 64))
        Y[ib] = k
        return oracle.rope_apply(X, 1, c, s)[ia] @ oracle.rope_apply(Y, 1, c, s)[ib]

    a1 = score(1, (1, 2, 3), (0, 0, 1))
    a2 = score(1, (3, 5, 5), (2, 3, 3))
    assert abs(a1 - a2) < 1e-12
    t1 = score(0, (1, 2, 3), (0, 0, 1))
    t2 = score(0, (3, 5, 5), (2, 3, 3))
    assert abs(t1 - t2) > 1e-6


def test_rope_tiled_is_the_repeat_expansion():
    """Tiled table = [f_0..f_{d/2-1}, f_0..f_{d/2-1}] per axis, applied as x cos + rot90(x) sin
    (Architecture 3-D RoPE; schema rope_freq_layout; SkyVision: repeat is tiling, not interleaving)."""
    cfg = rope_cfg(0, heads=1)
    T, H, W = 6, 10, 8
    c, s = oracle.rope_tables(cfg, T, H, W)
    pos = oracle.rope_positions(cfg, T, H, W)
    x = np.random.default_rng(7).normal(size=(c.shape[0], 64))
    y = oracle.rope_apply(x, 1, c, s)
    d = 20
    omega = 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    for i in range(c.shape[0]):
        for a in range(3):
            seg = x[i, a * d:(a + 1) * d]
            emb = np.tile(pos[i, a] * omega, 2)        # the repeat(1,1,1,2) expansion
            rot = np.stack([-seg[1::2], seg[0::2]], axis=-1).reshape(-1)
            ref = seg * np.cos(emb) + rot * np.sin(emb)
            assert np.abs(y[i, a * d:(a + 1) * d] - ref).max() < 1e-13
    # the two members of a pair see different angles: not norm-preserving
    assert np.abs(np.linalg.norm(y, axis=1) - np.linalg.norm(x, axis=1)).max() > 1e-3


def test_rope_layouts_related_by_fixed_permutation():
    """tiled column j carries omega_{j mod d/2}; interleaved column pi(j) = 2 (j mod d/2) + [j >= d/2] carries the same."""
    T, H, W = 6, 10, 8
    ct, st = oracle.rope_tables(rope_cfg(0, heads=1), T, H, W)
    ci, si = oracle.rope_tables(rope_cfg(1, heads=1), T, H, W)
    d, h = 20, 10
    for a in range(3):
        for j in range(d):
            pj = 2 * (j % h) + (1 if j >= h else 0)
            assert np.array_equal(ct[:, a * d + j], ci[:, a * d + pj])
            assert np.array_equal(np.abs(st[:, a * d + j]), np.abs(si[:, a * d + pj]))
    assert not np.array_equal(ct, ci)


def test_rope_layouts_coincide_at_one_frequency():
    """head_dim 6 -> d = 2, one frequency per axis: tiled and interleaved are the same rotation."""
    T, H, W = 4, 6, 6
    ct, st = oracle.rope_tables(rope_cfg(0, hd=6, heads=1), T, H, W)
    ci, si = oracle.rope_tables(rope_cfg(1, hd=6, heads=1), T, H, W)
    assert np.array_equal(ct, ci) and np.array_equal(st, si)


def test_interpolate_rope_positions():
    """V-JEPA 2.1: h, w scaled by (ref-1)/(g-1), t untouched (Architecture 3-D RoPE; schema rope_ref_grid)."""
    g = json.load(open(GOLDEN))
    assert 256 // g["rope_ref_grid"]["patch"] == g["rope_ref_grid"]["ref_grid"]
    assert 256 // g["rope_ref_grid_p14"]["patch"] == g["rope_ref_grid_p14"]["ref_grid"]
    cfg = tiny_video(patch_size=16, embed_dim=128, n_head=2, rope_layout=1, rope_interpolate=1, rope_ref_grid=16)
    pos = oracle.rope_positions(cfg, 4, 384, 384)   # 24 x 24 grid
    hs = np.unique(pos[:, 1])
    assert len(hs) == 24 and hs[0] == 0.0 and hs[-1] == 15.0
    assert np.abs(np.diff(hs) - 15.0 / 23.0).max() < 1e-14
    assert np.array_equal(np.unique(pos[:, 0]), [0.0, 1.0])
    # at the reference grid the scale is 1: same tables as without interpolation
    a = oracle.rope_tables(cfg, 4, 256, 256)
    b = oracle.rope_tables(replace(cfg, rope_interpolate=0), 4, 256, 256)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_cls_rows_are_identity():
    cfg = rope_cfg(0, cls_token=1)
    c, s = oracle.rope_tables(cfg, 4, 8, 8)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    assert not np.all(s[1:] == 0.0)
    # the first patch token (row 1) sits at position (0,0,0): identity as well
    assert np.all(c[1] == 1.0) and np.all(s[1] == 0.0)


# ---------------------------------------------------------------- mask / attention
def mask_matrix(attn_mode, prefix, F, N):
    return np.array([[oracle.mask_allow(attn_mode, prefix, F, N, q, k) for k in range(N)] for q in range(N)])


def test_block_causal_density_printed():
    g = json.load(open(GOLDEN))["block_causal_density"]
    F = g["gh"] * g["gw"]
    N = g["T"] * F + g["cls"]
    assert N == g["N"]
    # count visible pairs with the oracle's predicate, frame by frame (rows of one frame share a pattern)
    open_pairs = sum(F * sum(oracle.mask_allow(1, 1, F, N, 1 + f * F, k) for k in range(N)) for f in range(g["T"]))
    open_pairs += sum(oracle.mask_allow(1, 1, F, N, 0, k) for k in range(N))
    assert round(100.0 * open_pairs / N ** 2, 1) == g["percent"], g["cite"]


def test_block_causal_entries():
    F, N = 3, 1 + 3 * 3
    m = mask_matrix(1, 1, F, N)
    assert m[0].all()                      # CLS row open
    assert not m[1:, 0].any()              # CLS column closed to patch queries
    for q in range(1, N):
        for k in range(1, N):
            assert m[q, k] == ((q - 1) // F >= (k - 1) // F)
    assert mask_matrix(0, 1, F, N).all()


def sdpa(q, k, v, H, allow):
    N = q.shape[0]
    hd = q.shape[1] // H
    t = lambda a: torch.from_numpy(a.reshape(N, H, hd).transpose(1, 0, 2).copy())
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=torch.from_numpy(allow))
    return o.numpy().transpose(1, 0, 2).reshape(N, H * hd)


@pytest.mark.parametrize("attn_mode,prefix", [(0, 0), (1, 1), (1, 0)])
def test_attention_matches_library_sdpa(attn_mode, prefix):
    rng = np.random.default_rng(8)
    H, hd, F = 3, 16, 4
    N = prefix + 5 * F
    q, k, v = (rng.normal(size=(N, H * hd)) * 1.5 for _ in range(3))
    o = oracle.attention(q, k, v, H, attn_mode, prefix, F)
    ref = sdpa(q, k, v, H, mask_matrix(attn_mode, prefix, F, N))
    assert np.abs(o - ref).max() < 1e-12
    if attn_mode == 1:   # the unmasked control must disagree
        full = sdpa(q, k, v, H, np.ones((N, N), dtype=bool))
        assert np.abs(o - full).max() > 1e-2


def test_block_causal_single_frame():
    rng = np.random.default_rng(9)
    H, hd, F = 2, 8, 7
    q, k, v = (rng.normal(size=(F, H * hd)) for _ in range(3))
    assert np.abs(oracle.attention(q, k, v, H, 1, 0, F) - oracle.attention(q, k, v, H, 0, 0, F)).max() < 1e-15
    # with CLS: equal to full attention with key column 0 closed for rows >= 1
    N = F + 1
    q, k, v = (rng.normal(size=(N, H * hd)) for _ in range(3))
    allow = np.ones((N, N), dtype=bool)
    allow[1:, 0] = False
    assert np.abs(oracle.attention(q, k, v, H, 1, 1, F) - sdpa(q, k, v, H, allow)).max() < 1e-12


def test_attention_special_cases():
    rng = np.random.default_rng(10)
    H, hd, N = 2, 8, 11
    q, v = rng.normal(size=(N, H * hd)), rng.normal(size=(N, H * hd))
    k = np.tile(rng.normal(size=(1, H * hd)), (N, 1))       # identical keys -> mean of V
    o = oracle.attention(q, k, v, H)
    assert np.abs(o - v.mean(axis=0)).max() < 1e-14
    o = oracle.attention(q, k, v, H, 1, 0, 4)               # ... of the visible V under the mask
    for i in range(N):
        vis = (np.arange(N) // 4) <= i // 4
        assert np.abs(o[i] - v[vis].mean(axis=0)).max() < 1e-14
    # a dominant score selects its v row
    k = rng.normal(size=(N, H * hd)) * 0.01
    k[5] = q[3] * 100.0
    o = oracle.attention(q, k, v, H)
    assert np.abs(o[3] - v[5]).max() < 1e-10


# ---------------------------------------------------------------- whole encoder
def bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 (ties to even), as float32 (finite values)."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def torch_encoder(cfg: Config, seed, bf16, pix):
    """Independent composition of library routines (conv3d, layer_norm, sdpa, F.gelu) with the
    RoPE written as the pages' expansion; weights drawn from the shared generator."""
    B, T, C, Hh, Ww = pix.shape
    D, NH, F_ = cfg.embed_dim, cfg.n_head, cfg.ffn_dim
    hd = D // NH
    t, P = cfg.tubelet_size, cfg.patch_size
    gt, gh, gw = T // t, Hh // P, Ww // P
    K = C * t * P * P
    prm = lambda name, shape: torch.from_numpy(synth.param(seed, name, shape, bf16).astype(np.float64))
    w = prm("enc.patch_embed.weight", (D, K)).reshape(D, C, t, P, P)
    x = torch.nn.functional.conv3d(torch.from_numpy(pix.transpose(0, 2, 1, 3, 4).astype(np.float64)), w,
                                   prm("enc.patch_embed.bias", (D,)), stride=(t, P, P))
    x = x.flatten(2).transpose(1, 2)  # [B, Np, D], tokens t-major then h then w
    if cfg.cls_token:
        x = torch.cat([prm("enc.cls_token", (D,)).expand(B, 1, D), x], dim=1)
    if cfg.pos_type == 1:
        x = x + prm("enc.pos_embed", (cfg.n_pos_rows, D))
    if cfg.modality_embed:
        x = x + prm("enc.mod_embed_video", (D,))
    N = x.shape[1]
    pre = 1 if cfg.cls_token else 0
    if cfg.pos_type == 2:
        d = 2 * ((hd // 3) // 2)
        ii = np.arange(gt * gh * gw)
        tpos, hpos, wpos = ii // (gh * gw), (ii % (gh * gw)) // gw, ii % gw
        if cfg.rope_interpolate:
            hpos = hpos * ((cfg.rope_ref_grid - 1) / (gh - 1))
            wpos = wpos * ((cfg.rope_ref_grid - 1) / (gw - 1))
        omega = cfg.rope_theta ** (-np.arange(d // 2) * 2.0 / d)
        angles = []
        for p in (tpos, hpos, wpos):
            f = np.outer(p, omega)
            angles.append(np.tile(f, 2) if cfg.rope_layout == 0 else np.repeat(f, 2, axis=1))
        ang = np.concatenate(angles + [np.zeros((len(ii), hd - 3 * d))], axis=1)
        ang = np.concatenate([np.zeros((pre, hd)), ang], axis=0)
        cos_, sin_ = torch.from_numpy(np.cos(ang)), torch.from_numpy(np.sin(ang))

        def rope(z):  # z [B, H, N, hd]
            rot = torch.stack([-z[..., 1::2], z[..., 0::2]], dim=-1).flatten(-2)
            return z * cos_ + rot * sin_
    allow = torch.from_numpy(mask_matrix(cfg.attn_mode, pre, gh * gw, N))
    for l in range(cfg.n_layer):
        p = f"enc.blk.{l}."
        h = torch.nn.functional.layer_norm(x, (D,), prm(p + "ln1.weight", (D,)), prm(p + "ln1.bias", (D,)), cfg.ln_eps)
        wqkv = prm(p + "attn_qkv.weight", (3 * D, D))
        if cfg.q_weight_scale != 1.0 or cfg.k_weight_scale != 1.0:   # test input option: scaled q, k rows
            sc = np.ones((3 * D, 1), dtype=np.float32)
            sc[:D], sc[D:2 * D] = cfg.q_weight_scale, cfg.k_weight_scale
            w32 = (wqkv.numpy().astype(np.float32) * sc).astype(np.float32)
            wqkv = torch.from_numpy((bf16_round(w32) if bf16 else w32).astype(np.float64))
        qkv = h @ wqkv.T + prm(p + "attn_qkv.bias", (3 * D,))
        q, k, v = (qkv[..., i * D:(i + 1) * D].reshape(B, N, NH, hd).transpose(1, 2) for i in range(3))
        if cfg.pos_type == 2:
            q, k = rope(q), rope(k)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allow)
        o = o.transpose(1, 2).reshape(B, N, D)
        x = x + o @ prm(p + "attn_out.weight", (D, D)).T + prm(p + "attn_out.bias", (D,))
        h = torch.nn.functional.layer_norm(x, (D,), prm(p + "ln2.weight", (D,)), prm(p + "ln2.bias", (D,)), cfg.ln_eps)
        u = torch.nn.functional.gelu(h @ prm(p + "ffn_up.weight", (F_, D)).T + prm(p + "ffn_up.bias", (F_,)))
        x = x + u @ prm(p + "ffn_down.weight", (D, F_)).T + prm(p + "ffn_down.bias", (D,))
    return torch.nn.functional.layer_norm(x, (D,), prm("enc.norm.weight", (D,)), prm("enc.norm.bias", (D,)),
                                          cfg.ln_eps).numpy()


ENC_CASES = {
    "hfvit": (Config(embed_dim=48, n_layer=2, n_head=2, ffn_dim=80, patch_size=4, tubelet_size=1, pos_type=1,
                     cls_token=1, n_pos_rows=1 + 4 * 5), (1, 16, 20)),
    "vjepa2_tiled": (tiny_video(embed_dim=128, n_head=2, ffn_dim=96), (4, 12, 16)),
    "vjepa2_1_interleaved": (tiny_video(embed_dim=128, n_head=2, ffn_dim=96, rope_layout=1, rope_interpolate=1,
                                       rope_ref_grid=4, modality_embed=1), (4, 12, 20)),
    "levjepa_block_causal": (tiny_video(embed_dim=128, n_head=2, ffn_dim=96, tubelet_size=1, cls_token=1,
                                        attn_mode=1), (3, 12, 8)),
    # peaked attention: the q / k rows of attn_qkv.weight scaled by 4 and 2 (a test input option)
    "levjepa_peaked": (tiny_video(embed_dim=128, n_head=2, ffn_dim=96, tubelet_size=1, cls_token=1, attn_mode=1,
                                  q_weight_scale=2.5, k_weight_scale=2.0), (3, 12, 8)),
}


@pytest.mark.parametrize("name", list(ENC_CASES))
@pytest.mark.parametrize("bf16", [False, True])
def test_encoder_equals_library_composition(name, bf16):
    cfg, (T, H, W) = ENC_CASES[name]
    pix = synth.pixels(3, (2, T, 3, H, W))
    out = oracle.encode(cfg, 3, bf16, pix)
    ref = torch_encoder(cfg, 3, bf16, pix)
    assert out.shape == ref.shape
    assert np.abs(out - ref).max() < 1e-10
    # layout 1 (N C T H W) gives the same tokens
    out1 = oracle.encode(cfg, 3, bf16, np.ascontiguousarray(pix.transpose(0, 2, 1, 3, 4)), layout=1)
    assert np.array_equal(out, out1)


def test_wrong_layout_and_unmasked_controls_disagree():
    cfg, (T, H, W) = ENC_CASES["levjepa_block_causal"]
    pix = synth.pixels(4, (1, T, 3, H, W))
    ref = oracle.encode(cfg, 4, False, pix)
    assert np.abs(oracle.encode(replace(cfg, attn_mode=0), 4, False, pix) - ref).max() > 1e-3
    assert np.abs(oracle.encode(replace(cfg, rope_layout=1), 4, False, pix) - ref).max() > 1e-3


def test_batch_items_are_independent():
    cfg, (T, H, W) = ENC_CASES["vjepa2_tiled"]
    pix = synth.pixels(5, (3, T, 3, H, W))
    out = oracle.encode(cfg, 5, True, pix)
    for b in range(3):
        assert np.array_equal(out[b], oracle.encode(cfg, 5, True, pix[b:b + 1])[0])


def test_qk_weight_scale_touches_only_the_q_and_k_rows():
    """The scale option multiplies the q rows by its first factor and the k rows by its second:
    (a, b) and (b, a) swap nothing for scores (q.k scales by a*b either way) but do change the
    tokens, since the biases are not scaled; (1, 1) is the plain recipe."""
    cfg, (T, H, W) = ENC_CASES["vjepa2_tiled"]
    pix = synth.pixels(6, (1, T, 3, H, W))
    plain = oracle.encode(cfg, 6, True, pix)
    assert np.array_equal(oracle.encode(replace(cfg, q_weight_scale=1.0, k_weight_scale=1.0), 6, True, pix), plain)
    a = oracle.encode(replace(cfg, q_weight_scale=4.0, k_weight_scale=2.0), 6, True, pix)
    b = oracle.encode(replace(cfg, q_weight_scale=2.0, k_weight_scale=4.0), 6, True, pix)
    assert np.abs(a - plain).max() > 1e-3 and np.abs(a - b).max() > 1e-6
