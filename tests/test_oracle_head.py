"""Pins of the oracle's attentive-pool head, cross-attention and pooling (CPU only).

What fixes them, other than the oracle itself:
  * an independent float64 composition of library routines (torch: layer_norm, linear,
    scaled_dot_product_attention with one query, erf GELU) of the head as the pages' tensor
    table lays it out (self-attention blocks first, LN on keys / values only, no output
    projection, the raw query as the residual, no final norm before the classifier);
  * special cases: one token (the attention returns that token's value row), identical tokens,
    no pooler blocks; invariance to the order of the tokens (nothing in the head knows
    positions); cross_attention == torch's sdpa; pooling == numpy mean / row 0.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
import synth

HC = oracle.HeadConfig(embed_dim=128, n_head=2, ffn_dim=256, n_pool_layers=2, n_classes=10)


def W(name, shape, bf16):
    return torch.from_numpy(synth.param(0, name, shape, bf16).astype(np.float64))


def torch_head(hc, bf16, tokens):
    D, F, H, C = hc.embed_dim, hc.ffn_dim, hc.n_head, hc.n_classes
    hd = D // H
    pooled, logits = [], []
    for x in torch.from_numpy(np.asarray(tokens, dtype=np.float64)):
        for l in range(hc.n_pool_layers):
            p = f"head.blk.{l}."
            h = Fn.layer_norm(x, (D,), W(p + "ln1.weight", (D,), bf16), W(p + "ln1.bias", (D,), bf16), hc.ln_eps)
            qkv = Fn.linear(h, W(p + "attn_qkv.weight", (3 * D, D), bf16), W(p + "attn_qkv.bias", (3 * D,), bf16))
            q, k, v = (t.reshape(-1, H, hd).transpose(0, 1) for t in qkv.split(D, dim=-1))
            o = Fn.scaled_dot_product_attention(q[None], k[None], v[None])[0].transpose(0, 1).reshape(-1, D)
            x = x + Fn.linear(o, W(p + "attn_out.weight", (D, D), bf16), W(p + "attn_out.bias", (D,), bf16))
            h = Fn.layer_norm(x, (D,), W(p + "ln2.weight", (D,), bf16), W(p + "ln2.bias", (D,), bf16), hc.ln_eps)
            u = Fn.gelu(Fn.linear(h, W(p + "ffn_up.weight", (F, D), bf16), W(p + "ffn_up.bias", (F,), bf16)))
            x = x + Fn.linear(u, W(p + "ffn_down.weight", (D, F), bf16), W(p + "ffn_down.bias", (D,), bf16))
        query = W("head.query", (1, D), bf16)
        kv = Fn.layer_norm(x, (D,), W("head.xattn.ln_kv.weight", (D,), bf16), W("head.xattn.ln_kv.bias", (D,), bf16),
                           hc.ln_eps)
        q = Fn.linear(query, W("head.xattn.q.weight", (D, D), bf16), W("head.xattn.q.bias", (D,), bf16))
        k = Fn.linear(kv, W("head.xattn.k.weight", (D, D), bf16), W("head.xattn.k.bias", (D,), bf16))
        v = Fn.linear(kv, W("head.xattn.v.weight", (D, D), bf16), W("head.xattn.v.bias", (D,), bf16))
        split = lambda t: t.reshape(-1, H, hd).transpose(0, 1)  # noqa: E731
        o = Fn.scaled_dot_product_attention(split(q)[None], split(k)[None], split(v)[None])[0]
        y = query + o.transpose(0, 1).reshape(1, D)
        h = Fn.layer_norm(y, (D,), W("head.xattn.ln2.weight", (D,), bf16), W("head.xattn.ln2.bias", (D,), bf16),
                          hc.ln_eps)
        u = Fn.gelu(Fn.linear(h, W("head.xattn.ffn_up.weight", (F, D), bf16), W("head.xattn.ffn_up.bias", (F,), bf16)))
        y = y + Fn.linear(u, W("head.xattn.ffn_down.weight", (D, F), bf16), W("head.xattn.ffn_down.bias", (D,), bf16))
        pooled.append(y[0])
        logits.append(Fn.linear(y, W("head.cls.weight", (C, D), bf16), W("head.cls.bias", (C,), bf16))[0])
    return torch.stack(pooled).numpy(), torch.stack(logits).numpy()


@pytest.mark.parametrize("N,layers", [(37, 2), (130, 0), (1, 1)])
@pytest.mark.parametrize("bf16", [False, True])
def test_head_equals_library_composition(N, layers, bf16):
    hc = oracle.HeadConfig(**{**HC.__dict__, "n_pool_layers": layers})
    tokens = np.random.default_rng(N).standard_normal((2, N, hc.embed_dim))
    pooled, logits = oracle.attentive_head(hc, 0, bf16, tokens)
    rp, rl = torch_head(hc, bf16, tokens)
    assert np.abs(pooled - rp).max() < 1e-11 * np.abs(rp).max()
    assert np.abs(logits - rl).max() < 1e-11 * np.abs(rl).max()


def test_cross_attention_equals_sdpa_and_single_key_returns_its_value():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((3, 96)), rng.standard_normal((50, 96)), rng.standard_normal((50, 96))
    got = oracle.cross_attention(q, k, v, 3)
    split = lambda a: torch.from_numpy(a).reshape(a.shape[0], 3, 32).transpose(0, 1)  # noqa: E731
    ref = Fn.scaled_dot_product_attention(split(q), split(k), split(v)).transpose(0, 1).reshape(3, 96).numpy()
    assert np.abs(got - ref).max() < 1e-13
    one = oracle.cross_attention(q, k[:1], v[:1], 3)
    assert np.abs(one - v[:1]).max() < 1e-15
    same = oracle.cross_attention(q, np.repeat(k[:1], 7, 0), v[:7], 3)
    assert np.abs(same - v[:7].mean(0)).max() < 1e-14


def test_head_ignores_token_order():
    tokens = np.random.default_rng(4).standard_normal((1, 40, HC.embed_dim))
    a = oracle.attentive_head(HC, 0, False, tokens)
    b = oracle.attentive_head(HC, 0, False, tokens[:, np.random.default_rng(5).permutation(40)])
    assert np.abs(a[0] - b[0]).max() < 1e-12 and np.abs(a[1] - b[1]).max() < 1e-12


def test_identical_tokens_pool_like_one_token():
    hc = oracle.HeadConfig(**{**HC.__dict__, "n_pool_layers": 0})
    row = np.random.default_rng(6).standard_normal((1, 1, hc.embed_dim))
    one = oracle.attentive_head(hc, 0, False, row)
    many = oracle.attentive_head(hc, 0, False, np.repeat(row, 25, axis=1))
    assert np.abs(one[1] - many[1]).max() < 1e-12


def test_pooling():
    t = np.random.default_rng(7).standard_normal((3, 9, 5))
    assert np.abs(oracle.pool(t, 0, 0) - t.mean(1)).max() < 1e-15
    assert np.abs(oracle.pool(t, 1, 0) - t[:, 1:].mean(1)).max() < 1e-15
    assert np.array_equal(oracle.pool(t, 1, 1), t[:, 0])
    with pytest.raises(ValueError):
        oracle.pool(t, 0, 1)          # no CLS row to take
