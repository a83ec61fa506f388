"""The attentive-pool head, classifier and pooling on the GPU, against the oracle (GPU only).

Bars: pooled features and logits per item: cosine >= 0.9999 and max |d| <= 3e-2 * max |ref| (the
encoder's bf16 bar, relative since neither output is unit-scale); the pooler blocks run the
encoder's bf16 kernels, the one-row tail runs in fp32 with bf16 weights. Pooling: the CLS row is
copied bit for bit; the mean is an fp32 sum in a fixed order, within 1e-6 of max |x|. Full size:
the V-JEPA 2 ViT-L SSv2 head over 2048 tokens at 8 items per call against tests/golden/
full_head_vjepa2_vitl16_ssv2.npz (written by tests/golden/make_head_golden.py from the oracle).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from configs import HEAD_VJEPA2_L16_SSV2
from dataclasses import replace

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "full_head_vjepa2_vitl16_ssv2.npz")


@pytest.fixture(autouse=True)
def _clean_status():
    yield
    torch.cuda.synchronize()
    assert jv.ops.device_status() == 0


def check_rows(got, ref, what):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    err = np.abs(got - ref).max()
    assert cos.min() >= 0.9999, f"{what}: min cosine {cos.min():.7f}"
    assert err <= 3e-2 * np.abs(ref).max(), f"{what}: max abs err {err:.3e} of {np.abs(ref).max():.3e}"


def tokens_of(seed, B, N, D=1024):
    return synth.fill(seed, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, N, D))


@pytest.mark.parametrize("layers,N", [(0, 300), (1, 300), (2, 129), (0, 1)])
def test_small_head_matches_oracle(layers, N):
    hc = replace(HEAD_VJEPA2_L16_SSV2, n_pool_layers=layers)
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, n_pool_layers=layers)
    tok = tokens_of(layers * 1000 + N, 2, N)
    ctx = jv.HeadContext(head, 2, N)
    pooled, logits = ctx.forward(torch.from_numpy(tok).cuda())
    ctx.sync()
    rp, rl = oracle.attentive_head(hc, 0, True, tok)
    check_rows(pooled.cpu().numpy(), rp, f"pooled L{layers} N{N}")
    check_rows(logits.cpu().numpy(), rl, f"logits L{layers} N{N}")


def test_weights_are_the_generator_bits():
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, n_pool_layers=1)
    for name, shape in [("head.query", (1024,)), ("head.xattn.ln_kv.weight", (1024,)), ("head.xattn.k.weight", (1024, 1024)),
                        ("head.xattn.v.bias", (1024,)), ("head.blk.0.attn_qkv.weight", (3072, 1024)),
                        ("head.cls.weight", (174, 1024))]:
        assert np.array_equal(head.tensor(name, shape).numpy(), synth.param(0, name, shape, True)), name


def test_graph_replay_and_partial_outputs_match_eager():
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, n_pool_layers=1)
    tok = torch.from_numpy(tokens_of(11, 3, 200)).cuda()
    ctx = jv.HeadContext(head, 3, 200)
    p0, l0 = ctx.forward(tok)
    p0, l0 = p0.clone(), l0.clone()
    only_p, _ = ctx.forward(tok, want_logits=False)
    _, only_l = ctx.forward(tok, want_pooled=False)
    ctx.sync()
    assert torch.equal(only_p, p0) and torch.equal(only_l, l0)
    ctx.set_graph(True)
    pooled = torch.empty_like(p0)
    logits = torch.empty_like(l0)
    for _ in range(3):
        ctx.forward(tok, pooled, logits)
    ctx.sync()
    assert torch.equal(pooled, p0) and torch.equal(logits, l0)
    assert torch.equal(tok, torch.from_numpy(tokens_of(11, 3, 200)).cuda())   # the input is read only


def test_pooling_matches_oracle():
    x = tokens_of(12, 3, 2049, 1024)
    xt = torch.from_numpy(x).cuda()
    cls = jv.ops.pool(xt, prefix=1, mode=jv.POOL_CLS).cpu().numpy()
    assert np.array_equal(cls, x[:, 0])
    for prefix in (0, 1):
        got = jv.ops.pool(xt, prefix=prefix, mode=jv.POOL_MEAN).cpu().double().numpy()
        assert np.abs(got - oracle.pool(x, prefix, 0)).max() <= 1e-6 * np.abs(x).max()
    with pytest.raises(jv.JepaError):
        jv.ops.pool(xt, prefix=0, mode=jv.POOL_CLS)


def test_head_refusals():
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, n_pool_layers=0)
    ctx = jv.HeadContext(head, 2, 100)
    with pytest.raises(jv.JepaError) as e:
        ctx.forward(torch.zeros((3, 100, 1024), device="cuda"))
    assert e.value.status == jv._lib.E_BUDGET
    with pytest.raises(jv.JepaError) as e:
        jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, dtype="fp32")
    assert e.value.status == jv._lib.E_UNSUPPORTED
    with pytest.raises(jv.JepaError) as e:
        jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, n_head=8)     # head_dim 128 with pooler layers
    assert e.value.status == jv._lib.E_UNSUPPORTED


@pytest.mark.skipif(not os.path.exists(GOLDEN), reason="no full-size head golden")
def test_full_size_head_matches_oracle():
    g = np.load(GOLDEN)
    B, N = int(g["batch"]), int(g["tokens"])
    tok = tokens_of(int(g["seed"]), B, N)
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0)
    ctx = jv.HeadContext(head, B, N)
    pooled, logits = ctx.forward(torch.from_numpy(tok).cuda())
    ctx.sync()
    for j, b in enumerate(g["items"]):
        check_rows(pooled[int(b)].cpu().numpy()[None], g["pooled"][j][None].astype(np.float64), f"pooled item {b}")
        check_rows(logits[int(b)].cpu().numpy()[None], g["logits"][j][None].astype(np.float64), f"logits item {b}")
