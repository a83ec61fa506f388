"""The masked-latent predictor on the GPU, against the oracle (GPU only).

Stage tests feed seeded inputs to one kernel through the C ABI: the QKV epilogue with per-row
position ids and head_dim 32, and the flash attention on width-32 heads (64-byte tiles, scale
1/sqrt(32)), with sharp scores so that a wrong position or scale shows. Whole-predictor tests compare with oracle.predict
(fp64, the same bf16 weights): per-token cosine >= 0.9999 and max |d| <= 3e-2 * max |ref| (the
encoder's bf16 bar, relative because the projected outputs are not unit-scale). Full size: the
V-JEPA 2 ViT-L predictor over a 16 x 256^2 clip's 2048 tokens against tests/golden/
full_pred_vjepa2_vitl16.npz (written by tests/golden/make_pred_golden.py from the oracle alone).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from configs import PRED_VJEPA2_L16, PRED_WORKLOAD
from dataclasses import replace

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "full_pred_vjepa2_vitl16.npz")


@pytest.fixture(autouse=True)
def _clean_status():
    yield
    torch.cuda.synchronize()
    assert jv.ops.device_status() == 0


def bf16_exact(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.detach().cpu().double().numpy()


def positions(ids, gh, gw):
    ids = np.asarray(ids)
    return np.stack([ids // (gh * gw), (ids % (gh * gw)) // gw, ids % gw], axis=1).astype(np.float64)


# ------------------------------------------------------------------ stages
@pytest.mark.parametrize("layout", [0, 1])
def test_qkv_epilogue_with_position_ids_and_width_32_heads(layout):
    n_head, hd, M = 4, 32, 300                       # ragged: 300 rows = 2 tiles + 44
    P = n_head * hd
    gt, gh, gw = 3, 5, 7
    rng = np.random.default_rng(31)
    x = rng.standard_normal((M, P)).astype(np.float32)
    w = (rng.standard_normal((3 * P, P)) * 0.05).astype(np.float32)
    b = (rng.standard_normal(3 * P) * 0.1).astype(np.float32)
    ids = rng.integers(0, gt * gh * gw, M).astype(np.int32)
    hp = jv.hparams(embed_dim=P, n_layer=1, n_head=n_head, ffn_dim=64, patch_size=16, tubelet_size=2,
                    pos_type=jv.POS_ROPE3D, rope_layout=layout)
    table = jv.ops.rope_table(hp, 2 * gt, 16 * gh, 16 * gw)      # per-token table of the whole grid
    out = torch.zeros((M, 3 * P), dtype=torch.bfloat16, device="cuda")
    xt, wt = bf16_exact(x), bf16_exact(w)
    jv.ops.linear(xt.cuda(), wt.cuda(), torch.from_numpy(b).cuda(), out, jv.EPI_QKV_ROPE, rope=table,
                  rows_per_item=M, n_head=n_head, head_dim=hd, rope_layout=layout,
                  rope_ids=torch.from_numpy(ids).cuda())
    got = f64(out)
    qkv = oracle.linear(f64(xt), f64(wt), b)
    c, s = oracle.rope_tables_pos(hd, 10000.0, layout, positions(ids, gh, gw))
    ref = np.concatenate([oracle.rope_apply(qkv[:, :P], n_head, c, s), oracle.rope_apply(qkv[:, P:2 * P], n_head, c, s),
                          qkv[:, 2 * P:]], axis=1)
    bound = 2e-6 * np.sqrt(P) * np.abs(ref).max() + 2.0 ** -8 * np.abs(ref)   # fp32 sums + one bf16 rounding
    assert np.all(np.abs(got - ref) <= bound)
    # the same rows with positions in row order instead of the ids would differ
    c2, s2 = oracle.rope_tables_pos(hd, 10000.0, layout, positions(np.arange(M) % (gt * gh * gw), gh, gw))
    wrong = oracle.rope_apply(qkv[:, :P], n_head, c2, s2)
    assert np.abs(got[:, :P] - wrong).max() > 0.05 * np.abs(ref).max()


@pytest.mark.parametrize("B,N,H", [(1, 128, 2), (2, 300, 3), (1, 1100, 12)])
def test_attention_on_width_32_heads(B, N, H):
    rng = np.random.default_rng(40 + N)
    sharp = 3.0   # score std of q.k / sqrt(32)
    q = rng.standard_normal((B * N, H * 32)) * np.sqrt(sharp)
    k = rng.standard_normal((B * N, H * 32)) * np.sqrt(sharp)
    v = rng.standard_normal((B * N, H * 32))
    qkv = bf16_exact(np.concatenate([q, k, v], axis=1))
    got = f64(jv.ops.attention(qkv.cuda(), B, N, H, head_dim=32))
    e = f64(qkv)
    P = H * 32
    ref = np.concatenate([oracle.attention(e[b * N:(b + 1) * N, :P], e[b * N:(b + 1) * N, P:2 * P],
                                           e[b * N:(b + 1) * N, 2 * P:], H) for b in range(B)])
    assert np.abs(got - ref).max() <= 0.01 * np.abs(e[:, 2 * P:]).max()
    # the width-64 scale (1/8 instead of 1/sqrt(32)) would not pass
    wrong = np.concatenate([oracle.attention(e[b * N:(b + 1) * N, :P] / np.sqrt(2.0), e[b * N:(b + 1) * N, P:2 * P],
                                             e[b * N:(b + 1) * N, 2 * P:], H) for b in range(B)])
    assert np.abs(got - wrong).max() > 0.05


def test_block_causal_on_width_32_heads():
    # CLS + three frames of 256 rows (two tiles each): the frame-aligned tiling on 64-byte-swizzled
    # tiles and the prefix-row CTA on width-32 heads
    B, N, H, F = 1, 1 + 3 * 256, 2, 256
    rng = np.random.default_rng(44)
    q = rng.standard_normal((N, H * 32)) * np.sqrt(3.0)
    k = rng.standard_normal((N, H * 32)) * np.sqrt(3.0)
    v = rng.standard_normal((N, H * 32))
    qkv = bf16_exact(np.concatenate([q, k, v], axis=1))
    got = f64(jv.ops.attention(qkv.cuda(), B, N, H, 32, 1, 1, F))
    e = f64(qkv)
    P = H * 32
    ref = oracle.attention(e[:, :P], e[:, P:2 * P], e[:, 2 * P:], H, 1, 1, F)
    vmax = np.abs(e[:, 2 * P:]).max()
    assert np.abs(got - ref).max() <= 0.01 * vmax
    assert np.abs(got[:1] - ref[:1]).max() <= 0.01 * vmax  # the CLS row, which sees every key
    full = oracle.attention(e[:, :P], e[:, P:2 * P], e[:, 2 * P:], H)
    assert np.abs(got - full).max() > 0.01 * vmax


# ------------------------------------------------------------------ whole predictor
def check_pred(got, ref, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    err = np.abs(got - ref).max()
    assert cos.min() >= 0.9999, f"{what}: min token cosine {cos.min():.7f}"
    assert err <= 3e-2 * np.abs(ref).max(), f"{what}: max abs err {err:.3e} of {np.abs(ref).max():.3e}"


def small_case(seed, n_ctx, n_tgt, B=2, grid=(2, 12, 11), overlap=False):
    n_pos = grid[0] * grid[1] * grid[2]
    rng = np.random.default_rng(seed)
    ctx, tgt = [], []
    for _ in range(B):
        perm = rng.permutation(n_pos)
        ctx.append(perm[:n_ctx])
        tgt.append(rng.permutation(n_pos)[:n_tgt] if overlap else perm[n_ctx:n_ctx + n_tgt])
    enc = synth.fill(seed, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, n_pos, 1024))
    return enc, np.array(ctx, dtype=np.int32).reshape(B, n_ctx), np.array(tgt, dtype=np.int32), grid


def run_gpu(pred, enc, ctx, tgt, grid, graph=False):
    B = enc.shape[0]
    pc = jv.PredContext(pred, B, max(ctx.shape[1], 1), tgt.shape[1], graph=graph)
    out = pc.predict(torch.from_numpy(enc).cuda(), torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(), grid)
    pc.sync()
    return out.cpu().numpy(), pc


@pytest.mark.parametrize("n_ctx,n_tgt,overlap", [(150, 100, False), (0, 120, False), (264, 264, True), (200, 3, False)])
def test_small_predictor_matches_oracle(n_ctx, n_tgt, overlap):
    pc_cfg = replace(PRED_VJEPA2_L16, n_layer=2)
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0, n_layer=2)
    enc, ctx, tgt, grid = small_case(n_ctx + n_tgt, n_ctx, n_tgt, overlap=overlap)
    got, _ = run_gpu(pred, enc, ctx, tgt, grid)
    ref = oracle.predict(pc_cfg, 0, True, enc, ctx, tgt, grid[1:])
    check_pred(got, ref, f"ctx {n_ctx} tgt {n_tgt}")


def test_weights_are_the_generator_bits():
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0, n_layer=1)
    for name, shape in [("pred.embed.weight", (384, 1024)), ("pred.mask_tokens", (10, 384)),
                        ("pred.blk.0.attn_qkv.weight", (1152, 384)), ("pred.norm.weight", (384,)),
                        ("pred.proj.bias", (1024,))]:
        assert np.array_equal(pred.tensor(name, shape).numpy(), synth.param(0, name, shape, True)), name


def test_target_order_permutes_outputs_and_graph_replay_matches():
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0, n_layer=2)
    enc, ctx, tgt, grid = small_case(7, 120, 90)
    base, pc = run_gpu(pred, enc, ctx, tgt, grid)
    perm = np.random.default_rng(8).permutation(90)
    other, _ = run_gpu(pred, enc, ctx[:, ::-1].copy(), tgt[:, perm].copy(), grid)
    assert np.abs(other - base[:, perm]).max() <= 1e-2 * np.abs(base).max()
    pc.set_graph(True)
    e, c, t = (torch.from_numpy(a).cuda() for a in (enc, ctx, tgt))
    out = torch.empty((2, 90, 1024), device="cuda")
    for _ in range(3):
        pc.predict(e, c, t, grid, out)
    pc.sync()
    assert np.array_equal(out.cpu().numpy(), base)


def test_bad_ids_are_reported_and_the_context_recovers():
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0, n_layer=1)
    enc, ctx, tgt, grid = small_case(9, 40, 30)
    pc = jv.PredContext(pred, 2, 40, 30)
    bad = tgt.copy()
    bad[1, 3] = grid[0] * grid[1] * grid[2]          # one past the grid
    pc.predict(torch.from_numpy(enc).cuda(), torch.from_numpy(ctx).cuda(), torch.from_numpy(bad).cuda(), grid)
    with pytest.raises(jv.JepaError) as e:
        pc.sync()
    assert e.value.status == jv._lib.E_INVALID_ARG
    out = pc.predict(torch.from_numpy(enc).cuda(), torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(), grid)
    pc.sync()
    ref = oracle.predict(replace(PRED_VJEPA2_L16, n_layer=1), 0, True, enc, ctx, tgt, grid[1:])
    check_pred(out.cpu().numpy(), ref, "after a bad call")
    with pytest.raises(jv.JepaError) as e:      # over the context's maxima
        pc.predict(torch.from_numpy(enc).cuda(), torch.from_numpy(ctx).cuda(),
                   torch.zeros((2, 31), dtype=torch.int32, device="cuda"), grid)
    assert e.value.status == jv._lib.E_BUDGET
    with pytest.raises(jv.JepaError) as e:
        jv.Predictor.preset("vjepa2_vitl16", seed=0, dtype="fp32", n_layer=1)
    assert e.value.status == jv._lib.E_UNSUPPORTED


@pytest.mark.skipif(not os.path.exists(GOLDEN), reason="no full-size predictor golden")
def test_full_size_predictor_sampled_rows_match_oracle():
    g = np.load(GOLDEN)
    grid = tuple(int(x) for x in g["grid"])
    B = int(g["batch"])
    enc = synth.fill(int(g["seed"]), "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, int(np.prod(grid)), 1024))
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0)
    got, _ = run_gpu(pred, enc, g["ctx"], g["tgt"], grid)
    for j, b in enumerate(g["items"]):
        check_pred(got[int(b)][g["rows"]], g["out"][j].astype(np.float64), f"item {b}")
