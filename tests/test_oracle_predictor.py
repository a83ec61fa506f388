"""Pins of the oracle's masked-latent predictor (CPU only).

What fixes it, other than the oracle itself:
  * an independent composition of library routines in float64 (torch: gather, linear, stable
    argsort, layer_norm, scaled_dot_product_attention, erf GELU) with the pages' RoPE expansion
    (the per-axis cos / sin of pos * omega_k, tiled by `repeat`, applied as x cos + rot90(x) sin),
    on a width with head_dim 32, so the 5-frequency wrap is exercised;
  * the pages' statement that at head_dim 32 the odd member of pair u uses frequency
    (2u + 1) mod 5, read back from the RoPE table;
  * invariances: the listing order of the context and target ids does not matter (outputs follow
    the targets), a mask index counts modulo the number of mask tokens, a predictor without
    context depends on the positions alone.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
import synth

PC = oracle.PredConfig(embed_dim=96, n_layer=2, n_head=3, ffn_dim=384, enc_dim=64, out_dim=80, n_mask_tokens=4,
                       mask_index=1)
GRID = (4, 5)          # (gh, gw): ids decode as t = id // 20, h = (id % 20) // 5, w = id % 5
N_ENC = 2 * 4 * 5


def ids_case(seed, n_ctx, n_tgt, B=2, overlap=False):
    rng = np.random.default_rng(seed)
    ctx, tgt = [], []
    for _ in range(B):
        perm = rng.permutation(N_ENC)
        ctx.append(perm[:n_ctx])
        tgt.append(rng.permutation(N_ENC)[:n_tgt] if overlap else perm[n_ctx:n_ctx + n_tgt])
    return np.array(ctx, dtype=np.int32), np.array(tgt, dtype=np.int32)


def W(name, shape, bf16):
    return torch.from_numpy(synth.param(0, name, shape, bf16).astype(np.float64))


def rope_expand(x, pos, theta, d):
    """The pages' rotation on one axis segment: cos / sin of pos * omega_k (k < d/2) repeated to
    d columns ([f_0..f_{d/2-1}, f_0..f_{d/2-1}]), x cos + rot90(x) sin on (even, odd) pairs."""
    omega = 1.0 / theta ** (torch.arange(d // 2, dtype=torch.float64) / (d / 2))
    f = pos[:, None] * omega[None, :]
    cos, sin = f.cos().repeat(1, 2), f.sin().repeat(1, 2)
    y = x.unflatten(-1, (-1, 2))
    rot = torch.stack((-y[..., 1], y[..., 0]), dim=-1).flatten(-2)
    return x * cos + rot * sin


def torch_predict(pc, bf16, enc, ctx_ids, tgt_ids, grid):
    P, E, O, H, F = pc.embed_dim, pc.enc_dim, pc.out_dim, pc.n_head, pc.ffn_dim
    hd = P // H
    d = 2 * ((hd // 3) // 2)
    gh, gw = grid
    enc = torch.from_numpy(np.asarray(enc, dtype=np.float64))
    outs = []
    for b in range(enc.shape[0]):
        ctx = torch.from_numpy(ctx_ids[b].astype(np.int64))
        tgt = torch.from_numpy(tgt_ids[b].astype(np.int64))
        x_ctx = Fn.linear(enc[b, ctx], W("pred.embed.weight", (P, E), bf16), W("pred.embed.bias", (P,), bf16))
        tok = W("pred.mask_tokens", (pc.n_mask_tokens, P), bf16)[pc.mask_index % pc.n_mask_tokens]
        x = torch.cat([x_ctx, tok[None, :].expand(len(tgt), P)], dim=0)
        ids = torch.cat([ctx, tgt])
        order = torch.argsort(ids, stable=True)
        x, ids = x[order], ids[order]
        pos = [(ids // (gh * gw)).double(), ((ids % (gh * gw)) // gw).double(), (ids % gw).double()]
        for l in range(pc.n_layer):
            p = f"pred.blk.{l}."
            h = Fn.layer_norm(x, (P,), W(p + "ln1.weight", (P,), bf16), W(p + "ln1.bias", (P,), bf16), pc.ln_eps)
            qkv = Fn.linear(h, W(p + "attn_qkv.weight", (3 * P, P), bf16), W(p + "attn_qkv.bias", (3 * P,), bf16))
            q, k, v = (t.reshape(-1, H, hd).transpose(0, 1) for t in qkv.split(P, dim=-1))

            def rope(t):
                parts = [rope_expand(t[..., a * d:(a + 1) * d], pos[a], pc.rope_theta, d) for a in range(3)]
                return torch.cat(parts + [t[..., 3 * d:]], dim=-1)
            o = Fn.scaled_dot_product_attention(rope(q)[None], rope(k)[None], v[None])[0]
            o = o.transpose(0, 1).reshape(-1, P)
            x = x + Fn.linear(o, W(p + "attn_out.weight", (P, P), bf16), W(p + "attn_out.bias", (P,), bf16))
            h = Fn.layer_norm(x, (P,), W(p + "ln2.weight", (P,), bf16), W(p + "ln2.bias", (P,), bf16), pc.ln_eps)
            u = Fn.gelu(Fn.linear(h, W(p + "ffn_up.weight", (F, P), bf16), W(p + "ffn_up.bias", (F,), bf16)))
            x = x + Fn.linear(u, W(p + "ffn_down.weight", (P, F), bf16), W(p + "ffn_down.bias", (P,), bf16))
        y = Fn.layer_norm(x, (P,), W("pred.norm.weight", (P,), bf16), W("pred.norm.bias", (P,), bf16), pc.ln_eps)
        y = y[torch.argsort(order)]            # back to the input order
        outs.append(Fn.linear(y[len(ctx):], W("pred.proj.weight", (O, P), bf16), W("pred.proj.bias", (O,), bf16)))
    return torch.stack(outs).numpy()


@pytest.mark.parametrize("n_ctx,n_tgt,overlap", [(15, 10, False), (30, 10, False), (0, 12, False), (20, 20, True)])
@pytest.mark.parametrize("bf16", [False, True])
def test_predictor_equals_library_composition(n_ctx, n_tgt, overlap, bf16):
    ctx, tgt = ids_case(n_ctx + n_tgt, n_ctx, n_tgt, overlap=overlap)
    enc = np.random.default_rng(5).standard_normal((2, N_ENC, PC.enc_dim))
    got = oracle.predict(PC, 0, bf16, enc, ctx, tgt, GRID)
    ref = torch_predict(PC, bf16, enc, ctx, tgt, GRID)
    assert np.abs(got - ref).max() < 1e-11 * max(1.0, np.abs(ref).max())


def test_interleaved_layout_pairs_share_one_frequency():
    # the interleaved layout: frequency k on dims (2k, 2k+1); it is a different rotation from the tiled one
    pc = oracle.PredConfig(**{**PC.__dict__, "rope_layout": 1, "n_layer": 1})
    ctx, tgt = ids_case(3, 12, 6)
    enc = np.random.default_rng(6).standard_normal((2, N_ENC, PC.enc_dim))
    got = oracle.predict(pc, 0, False, enc, ctx, tgt, GRID)
    tiled = oracle.predict(oracle.PredConfig(**{**pc.__dict__, "rope_layout": 0}), 0, False, enc, ctx, tgt, GRID)
    assert np.abs(got - tiled).max() > 1e-6   # the two layouts are different rotations
    c_i, s_i = oracle.rope_tables_pos(32, 10000.0, 1, np.array([[1.0, 2.0, 3.0]]))
    for j in range(0, 30, 2):                  # interleaved: both members of pair u at frequency u
        assert c_i[0, j] == c_i[0, j + 1] and s_i[0, j] == -s_i[0, j + 1]


def test_head_dim_32_odd_members_wrap_the_five_frequencies():
    # the pages: at head_dim 32 each axis has d = 10, i.e. 5 frequencies; in the tiled layout the
    # odd member of pair u uses frequency (2u + 1) mod 5 (not the even member's + 1)
    cos_t, sin_t = oracle.rope_tables_pos(32, 10000.0, 0, np.array([[1.0, 0.0, 0.0]]))
    omega = 10000.0 ** (-np.arange(5) / 5.0)
    for u in range(5):
        ang_even = np.arctan2(-sin_t[0, 2 * u], cos_t[0, 2 * u])
        ang_odd = np.arctan2(sin_t[0, 2 * u + 1], cos_t[0, 2 * u + 1])
        assert abs(ang_even - omega[(2 * u) % 5]) < 1e-15
        assert abs(ang_odd - omega[(2 * u + 1) % 5]) < 1e-15
    assert np.all(cos_t[0, 10:] == 1.0) and np.all(sin_t[0, 10:] == 0.0)   # h, w at 0; dims 30, 31 pass


def test_listing_order_of_ids_does_not_matter():
    ctx, tgt = ids_case(11, 18, 9)
    enc = np.random.default_rng(7).standard_normal((2, N_ENC, PC.enc_dim))
    base = oracle.predict(PC, 0, False, enc, ctx, tgt, GRID)
    rng = np.random.default_rng(8)
    pc_, pt_ = rng.permutation(18), rng.permutation(9)
    got = oracle.predict(PC, 0, False, enc, ctx[:, pc_], tgt[:, pt_], GRID)
    assert np.abs(got - base[:, pt_]).max() < 1e-12


def test_mask_index_counts_modulo_the_tokens():
    ctx, tgt = ids_case(12, 10, 5)
    enc = np.random.default_rng(9).standard_normal((2, N_ENC, PC.enc_dim))
    a = oracle.predict(PC, 0, False, enc, ctx, tgt, GRID)
    b = oracle.predict(oracle.PredConfig(**{**PC.__dict__, "mask_index": 1 + PC.n_mask_tokens}), 0, False, enc, ctx,
                       tgt, GRID)
    c = oracle.predict(oracle.PredConfig(**{**PC.__dict__, "mask_index": 0}), 0, False, enc, ctx, tgt, GRID)
    assert np.array_equal(a, b)
    assert np.abs(a - c).max() > 1e-6


def test_without_context_only_positions_matter():
    _, tgt = ids_case(13, 0, 7)
    tgt[1] = tgt[0]
    enc = np.random.default_rng(10).standard_normal((2, N_ENC, PC.enc_dim))
    y = oracle.predict(PC, 0, False, enc, np.zeros((2, 0), dtype=np.int32), tgt, GRID)
    assert np.abs(y[0] - y[1]).max() < 1e-13


def test_bad_ids_are_refused():
    enc = np.zeros((1, N_ENC, PC.enc_dim))
    with pytest.raises(ValueError):
        oracle.predict(PC, 0, False, enc, np.array([[N_ENC]]), np.array([[1]]), GRID)
    with pytest.raises(ValueError):
        oracle.predict(PC, 0, False, enc, np.array([[0]]), np.array([[-1]]), GRID)
