"""Stage-by-stage parity of the CUDA kernels against the oracle (GPU only).

Every test feeds the same seeded inputs to one kernel (through the C ABI) and to the matching
oracle function, and compares element by element:
  - data movement (patchify) is bit-exact; bf16 storage equals round-to-nearest-even of the
    exact value (the same decision on both sides, made by torch's bf16 conversion);
  - fp32 kernels: max |d| <= 1e-5 * max |ref| (plus a few ulps);
  - bf16 kernels: the oracle gets the bf16-rounded inputs exactly; the bound is what fp32
    accumulation plus one bf16 rounding of the output allows (stated per test).
Sizes span several tiles and a ragged tail; every GEMM tile width and epilogue is exercised.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import Config

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_status():
    yield
    torch.cuda.synchronize()
    assert jv.ops.device_status() == 0


def bf16_exact(a: np.ndarray) -> torch.Tensor:
    """float array -> bf16 tensor (RNE), the values both sides then use exactly."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def rnd(shape, seed, scale=1.0, offset=0.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale + offset).astype(np.float32)


# ------------------------------------------------------------------ patchify
@pytest.mark.parametrize("t,P,T,H,W", [(2, 16, 4, 48, 64), (1, 16, 3, 32, 48), (1, 14, 1, 56, 42), (2, 8, 2, 24, 16)])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_patchify_bit_exact(t, P, T, H, W, layout, dtype):
    B, C = 2, 3
    pix = synth.pixels(11, (B, T, C, H, W))
    src = pix if layout == 0 else np.ascontiguousarray(pix.transpose(0, 2, 1, 3, 4))
    got = jv.ops.patchify(torch.from_numpy(src).to(DEV), t, P, layout, dtype)
    cfg = Config(embed_dim=8, n_layer=1, n_head=1, ffn_dim=8, patch_size=P, tubelet_size=t)
    ref = oracle.patchify(cfg, src, layout)
    if dtype == "fp32":
        assert np.array_equal(f64(got), ref)
    else:
        assert torch.equal(got.cpu(), bf16_exact(ref))


# ------------------------------------------------------------------ layernorm
@pytest.mark.parametrize("M,D", [(333, 192), (257, 1024), (130, 1408), (5, 2048), (1, 1024)])
def test_layernorm(M, D):
    x = rnd((M, D), 1, scale=3.0, offset=20.0)  # large offset: a one-pass variance would fail
    g, b = rnd(D, 2, 0.1, 1.0), rnd(D, 3, 0.01)
    xd, gd, bd = (torch.from_numpy(a).to(DEV) for a in (x, g, b))
    ref = oracle.layernorm(x, g, b, 1e-6)
    y32 = f64(jv.ops.layernorm(xd, gd, bd, 1e-6, "fp32"))
    assert np.abs(y32 - ref).max() <= 2e-5 * np.abs(ref).max()
    y16 = f64(jv.ops.layernorm(xd, gd, bd, 1e-6, "bf16"))
    assert np.all(np.abs(y16 - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


# ------------------------------------------------------------------ GEMM epilogue references
def ref_epilogue(kind, acc, bias, out_init=None, **kw):
    v = acc + bias
    if kind == jv.EPI_BIAS_GELU:
        return oracle.gelu(v)
    if kind == jv.EPI_BIAS_RESIDUAL:
        return out_init + v
    if kind == jv.EPI_QKV_ROPE:
        D = kw["n_head"] * kw["head_dim"]
        c, s = kw["tables"]
        rows = kw["rows_per_item"]
        out = v.copy()
        for i0 in range(0, v.shape[0], rows):
            blk = slice(i0, i0 + rows)
            out[blk, :D] = oracle.rope_apply(v[blk, :D], kw["n_head"], c, s)
            out[blk, D:2 * D] = oracle.rope_apply(v[blk, D:2 * D], kw["n_head"], c, s)
        return out
    return v


def bf16_bound(ref, K):
    # fp32 accumulation of K exact bf16 products + one bf16 rounding of the output
    return 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max() + 1e-6


# (M, N, K): tile widths 256 (many tiles, > 1 per CTA), 128, 64; ragged M. (2125, 3072), (4099, 4096)
# and (4099, 768) run on the 2-SM pair kernel; (4099, 1408) and (4099, 2368) on the pair kernel with a
# ragged last column tile (N % 256 = 128 and 64: the columns past N are loaded as zeros, not stored).
GEMM_SHAPES = [(2048 + 77, 3072, 256), (2048, 1024, 1024), (257, 256, 128), (128, 64, 64), (4096 + 3, 4096, 128),
               (4096 + 3, 768, 128), (4096 + 3, 1408, 128), (4096 + 3, 2368, 64),
               (1, 1024, 128), (129, 512, 64)]  # one row; one row past a tile


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("kind", [jv.EPI_BIAS, jv.EPI_BIAS_GELU, jv.EPI_BIAS_RESIDUAL])
def test_linear_bf16(M, N, K, kind):
    x = bf16_exact(rnd((M, K), 4))
    w = bf16_exact(rnd((N, K), 5, 0.05))
    bias = rnd(N, 6, 0.1)
    acc = oracle.linear(f64(x), f64(w))
    if kind == jv.EPI_BIAS_RESIDUAL:
        init = rnd((M, N), 7)
        out = torch.from_numpy(init).to(DEV)
        ref = ref_epilogue(kind, acc, bias, init)
    else:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        ref = ref_epilogue(kind, acc, bias)
    jv.ops.linear(x.to(DEV), w.to(DEV), torch.from_numpy(bias).to(DEV), out, kind)
    got = f64(out)
    bound = bf16_bound(ref, K) if kind != jv.EPI_BIAS_RESIDUAL else 2e-6 * np.sqrt(K) * np.abs(acc).max() + 1e-6
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside; first at {np.argwhere(bad)[:4].tolist()}"


@pytest.mark.parametrize("M,N,K", [(333, 1024, 192), (129, 64, 588)])
@pytest.mark.parametrize("kind", [jv.EPI_BIAS, jv.EPI_BIAS_GELU, jv.EPI_BIAS_RESIDUAL])
def test_linear_fp32(M, N, K, kind):
    x, w, bias = rnd((M, K), 8), rnd((N, K), 9, 0.05), rnd(N, 10, 0.1)
    acc = oracle.linear(x, w)
    init = rnd((M, N), 11)
    out = torch.from_numpy(init).to(DEV) if kind == jv.EPI_BIAS_RESIDUAL else torch.empty((M, N), dtype=torch.float32, device=DEV)
    ref = ref_epilogue(kind, acc, bias, init)
    jv.ops.linear(torch.from_numpy(x).to(DEV), torch.from_numpy(w).to(DEV), torch.from_numpy(bias).to(DEV), out, kind)
    assert np.abs(f64(out) - ref).max() <= 1e-5 * np.abs(ref).max()


ROPE_CASES = {
    "tiled": (dict(rope_layout=0), (4, 48, 64)),
    "interleaved_interp": (dict(rope_layout=1, rope_interpolate=1, rope_ref_grid=16), (4, 80, 96)),
    "tiled_cls": (dict(rope_layout=0, cls_token=1, tubelet_size=1), (3, 48, 32)),
}


def rope_cfgs(extra, n_head):
    base = dict(embed_dim=64 * n_head, n_layer=1, n_head=n_head, ffn_dim=64, patch_size=16, tubelet_size=2,
                pos_type=2)
    base.update(extra)
    return Config(**base), jv.hparams(**base)


@pytest.mark.parametrize("case", list(ROPE_CASES))
def test_rope_table(case):
    extra, (T, H, W) = ROPE_CASES[case]
    cfg, hp = rope_cfgs(extra, 2)
    tab = jv.ops.rope_table(hp, T, H, W).cpu().double().numpy()  # [Np, 3, 10, 2]
    pre = cfg.cls_token
    d = 20
    # interleaved oracle columns 2k / 2k+1 carry frequency k: compare cos and sin
    ci, si = oracle.rope_tables(Config(**{**cfg.__dict__, "rope_layout": 1}), T, H, W)
    for a in range(3):
        assert np.abs(tab[:, a, :, 0] - ci[pre:, a * d:(a + 1) * d:2]).max() < 2e-7
        assert np.abs(tab[:, a, :, 1] - si[pre:, a * d + 1:(a + 1) * d:2]).max() < 2e-7


@pytest.mark.parametrize("case", list(ROPE_CASES))
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_qkv_rope_epilogue(case, dtype, n_head=4, B=2):
    extra, (T, H, W) = ROPE_CASES[case]
    cfg, hp = rope_cfgs(extra, n_head)
    D = 64 * n_head
    N = oracle.n_tokens(cfg, T, H, W)
    M, K = B * N, 128
    x, w, bias = rnd((M, K), 12), rnd((3 * D, K), 13, 0.1), rnd(3 * D, 14, 0.1)
    if dtype == "bf16":
        xt, wt = bf16_exact(x), bf16_exact(w)
        out = torch.empty((M, 3 * D), dtype=torch.bfloat16, device=DEV)
    else:
        xt, wt = torch.from_numpy(x), torch.from_numpy(w)
        out = torch.empty((M, 3 * D), dtype=torch.float32, device=DEV)
    table = jv.ops.rope_table(hp, T, H, W)
    jv.ops.linear(xt.to(DEV), wt.to(DEV), torch.from_numpy(bias).to(DEV), out, jv.EPI_QKV_ROPE, rope=table,
                  rows_per_item=N, prefix=cfg.cls_token, n_head=n_head, head_dim=64, rope_layout=cfg.rope_layout)
    acc = oracle.linear(f64(xt), f64(wt))
    ref = ref_epilogue(jv.EPI_QKV_ROPE, acc, bias, n_head=n_head, head_dim=64, rows_per_item=N,
                       tables=oracle.rope_tables(cfg, T, H, W))
    got = f64(out)
    if dtype == "fp32":
        assert np.abs(got - ref).max() <= 2e-6 * np.abs(ref).max()
    else:
        assert not (np.abs(got - ref) > bf16_bound(ref, K) + 2.0 ** -8 * np.abs(acc + bias)).any()
    # control: the other layout is outside the bar
    other = Config(**{**cfg.__dict__, "rope_layout": 1 - cfg.rope_layout})
    wrong = ref_epilogue(jv.EPI_QKV_ROPE, acc, bias, n_head=n_head, head_dim=64, rows_per_item=N,
                         tables=oracle.rope_tables(other, T, H, W))
    assert np.abs(got - wrong).max() > 0.05 * np.abs(ref).max()


def test_qkv_rope_epilogue_ragged_pair_tile():
    # ViT-g's 22 heads: N = 3 * 1408 = 4224 = 16.5 pair tiles; 200 items of 24 tokens make M large
    # enough for the pair kernel, whose last column tile is half past N
    test_qkv_rope_epilogue("tiled", "bf16", n_head=22, B=200)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("prefix,use_pos,use_vec", [(0, False, True), (1, True, False), (0, True, True)])
def test_patch_embed_epilogue(dtype, prefix, use_pos, use_vec):
    B, Np, K, D = 3, 130, 192, 256
    N = Np + prefix
    x, w, bias = rnd((B * Np, K), 15), rnd((D, K), 16, 0.05), rnd(D, 17, 0.1)
    pos, vec = rnd((N, D), 18, 0.02), rnd(D, 19, 0.02)
    xt, wt = (bf16_exact(x), bf16_exact(w)) if dtype == "bf16" else (torch.from_numpy(x), torch.from_numpy(w))
    init = np.full((B * N, D), 7.0, dtype=np.float32)  # prefix rows must stay untouched
    X = torch.from_numpy(init).to(DEV)
    jv.ops.linear(xt.to(DEV), wt.to(DEV), torch.from_numpy(bias).to(DEV), X, jv.EPI_PATCH_EMBED,
                  rows_per_item=N, prefix=prefix, patches_per_item=Np,
                  pos=torch.from_numpy(pos).to(DEV) if use_pos else None,
                  vec=torch.from_numpy(vec).to(DEV) if use_vec else None)
    emb = oracle.linear(f64(xt), f64(wt), bias).reshape(B, Np, D)
    ref = init.reshape(B, N, D).astype(np.float64)
    ref[:, prefix:] = emb + (pos[prefix:] if use_pos else 0) + (vec if use_vec else 0)
    got = f64(X).reshape(B, N, D)
    assert np.abs(got - ref).max() <= 2e-6 * np.sqrt(K) * np.abs(ref).max()
    assert np.all(got[:, :prefix] == 7.0)


# ------------------------------------------------------------------ attention
def attn_inputs(B, N, H, seed, sharp=3.0):
    # q, k entries of std sqrt(sharp): scores q.k/8 have std `sharp`, a peaked softmax
    q = rnd((B * N, H * 64), seed, sharp ** 0.5)
    k = rnd((B * N, H * 64), seed + 1, sharp ** 0.5)
    v = rnd((B * N, H * 64), seed + 2)
    return np.concatenate([q, k, v], axis=1)


ATTN_CASES = [
    # B, N, H, mode, prefix, frame_tokens
    (1, 128, 2, 0, 0, 1),
    (3, 1, 2, 0, 0, 1),                # one token: the output is its own value row
    (1, 129, 1, 0, 0, 1),              # one key past a tile
    (2, 257, 3, 0, 0, 1),
    (1, 1000, 2, 0, 0, 1),
    (1, 2048, 2, 0, 0, 1),
    (2, 1 + 4 * 100, 2, 1, 1, 100),    # levjepa-style: CLS + frames straddling tiles
    (1, 1 + 3 * 256, 2, 1, 1, 256),    # frames of two tiles each, shifted by the CLS row
    (1, 5 * 96, 2, 1, 0, 96),          # block-causal without a prefix
    (1, 1 + 200, 1, 1, 1, 200),        # one frame: full attention with the CLS column closed
    (1, 2 + 2 * 256, 2, 1, 2, 256),    # two prefix rows
    (1, 1 + 32 * 256, 1, 1, 1, 256),   # 8193 tokens: the prefix row over 65 key tiles
]


def ref_attention(qkv, B, N, H, mode, prefix, F):
    D = H * 64
    out = np.empty((B * N, D))
    for b in range(B):
        blk = qkv[b * N:(b + 1) * N]
        out[b * N:(b + 1) * N] = oracle.attention(blk[:, :D], blk[:, D:2 * D], blk[:, 2 * D:], H, mode, prefix, F)
    return out


@pytest.mark.parametrize("B,N,H,mode,prefix,F", ATTN_CASES)
def test_attention_bf16(B, N, H, mode, prefix, F):
    qkv = bf16_exact(attn_inputs(B, N, H, 20 + N))
    got = f64(jv.ops.attention(qkv.to(DEV), B, N, H, 64, mode, prefix, F))
    x = f64(qkv)
    ref = ref_attention(x, B, N, H, mode, prefix, F)
    vmax = np.abs(x[:, 2 * H * 64:]).max()
    err = np.abs(got - ref).max()
    # bf16 P (2^-9 relative per weight) and bf16 output rounding: well inside 1 % of max |v|
    assert err <= 1e-2 * vmax, err
    # control: for multi-frame block-causal cases the unmasked result is outside the bar
    if mode == 1 and N - prefix > F:
        full = ref_attention(x, B, N, H, 0, prefix, F)
        assert np.abs(got - full).max() > 1e-2 * vmax


# The workloads' full attention geometries: V-JEPA 2.1 at 384 px (4608 tokens, 16 heads), LeVJEPA's
# two clips of 4097 tokens (CLS + 16 frames of 256, block-causal), ViT-g/16's 8192 tokens x 22 heads.
# Every head runs on the GPU; the oracle computes the listed heads (all queries and keys of each,
# the last head included), compared element by element under the same bar as above.
FULL_ATTN_CASES = [
    # name, B, N, H, mode, prefix, frame_tokens, heads checked
    ("vjepa2_1_16x384", 1, 4608, 16, 0, 0, 1, (0, 7, 15)),
    ("levjepa_16x256_2clips", 2, 4097, 16, 1, 1, 256, (0, 9, 15)),
    ("vitg16_64x256", 1, 8192, 22, 0, 0, 1, (0, 13, 21)),
]


def head_cols(H, heads):
    D = H * 64
    cols = [np.arange(h * 64, (h + 1) * 64) for h in heads]
    one = np.concatenate(cols)
    return one, np.concatenate([one, D + one, 2 * D + one])


@pytest.mark.parametrize("name,B,N,H,mode,prefix,F,heads", FULL_ATTN_CASES, ids=[c[0] for c in FULL_ATTN_CASES])
def test_attention_bf16_full_geometry(name, B, N, H, mode, prefix, F, heads):
    qkv = bf16_exact(attn_inputs(B, N, H, 90 + H))
    got = f64(jv.ops.attention(qkv.to(DEV), B, N, H, 64, mode, prefix, F))
    out_cols, in_cols = head_cols(H, heads)
    x = f64(qkv)[:, in_cols]
    ref = ref_attention(x, B, N, len(heads), mode, prefix, F)
    vmax = np.abs(x[:, 2 * len(heads) * 64:]).max()
    err = np.abs(got[:, out_cols] - ref).max()
    assert err <= 1e-2 * vmax, f"{name}: max |d| {err:.3e} against 1 % of max |v| {vmax:.3f}"
    if mode == 1:   # control: the unmasked result is outside the bar
        full = ref_attention(x, B, N, len(heads), 0, prefix, F)
        assert np.abs(got[:, out_cols] - full).max() > 1e-2 * vmax


@pytest.mark.parametrize("B,N,H,mode,prefix,F", [(1, 257, 3, 0, 0, 1), (2, 1 + 3 * 50, 2, 1, 1, 50),
                                                 (1, 300, 2, 1, 0, 75)])
def test_attention_fp32(B, N, H, mode, prefix, F):
    qkv = attn_inputs(B, N, H, 40 + N)
    got = f64(jv.ops.attention(torch.from_numpy(qkv).to(DEV), B, N, H, 64, mode, prefix, F))
    ref = ref_attention(qkv.astype(np.float64), B, N, H, mode, prefix, F)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_attention_identical_keys_give_mean_of_v():
    B, N, H = 1, 300, 2
    x = attn_inputs(B, N, H, 50)
    x[:, H * 64:2 * H * 64] = x[0, H * 64:2 * H * 64]
    qkv = bf16_exact(x)
    got = f64(jv.ops.attention(qkv.to(DEV), B, N, H))
    v = f64(qkv)[:, 2 * H * 64:]
    assert np.abs(got - v.mean(axis=0)).max() < 1e-2


# ------------------------------------------------------------------ failure path of the bounded waits
def test_bounded_wait_reports_timeout_and_device_stays_usable():
    assert jv.ops.wait_timeout_probe(20000) == jv._lib.E_TIMEOUT
    assert jv.ops.device_status() == 0   # the error word was cleared
    x = bf16_exact(rnd((128, 64), 60))
    w = bf16_exact(rnd((64, 64), 61))
    out = torch.empty((128, 64), dtype=torch.bfloat16, device=DEV)
    jv.ops.linear(x.to(DEV), w.to(DEV), torch.zeros(64, dtype=torch.float32, device=DEV), out)
    torch.cuda.synchronize()
    ref = oracle.linear(f64(x), f64(w))
    assert np.all(np.abs(f64(out) - ref) <= bf16_bound(ref, 64))
