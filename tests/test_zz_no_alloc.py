"""Allocation-free encode against the context encode (GPU only).

jepa_encode_noalloc runs the encoder with a fixed scratch array compiled into the library as its
workspace. Two calls in a row must each agree with jepa_encode on the same clip within the
encoder's parity bar (fp32: max |y - ref| / max |ref| <= 1e-4; bf16: per-token cosine >= 0.9999
and max |y - ref| <= 3e-2), the second call must leave the device's free memory unchanged, and a
batch whose workspace does not fit in the array is refused before anything is launched.
The file name sorts last so that it also runs after every other GPU test.
"""
import numpy as np
import pytest
import torch

import synth

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu


def bar(got, ref, dtype, what):
    got = got.double().cpu().numpy().reshape(-1, got.shape[-1])
    ref = ref.double().cpu().numpy().reshape(-1, ref.shape[-1])
    err = np.abs(got - ref)
    if dtype == "fp32":
        assert err.max() / np.abs(ref).max() <= 1e-4, f"{what}: max rel err {err.max() / np.abs(ref).max():.3e}"
    else:
        cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
        assert cos.min() >= 0.9999, f"{what}: min token cosine {cos.min():.7f}"
        assert err.max() <= 3e-2, f"{what}: max abs err {err.max():.3e}"


def clip(seed, B, T, H, W):
    return torch.from_numpy(synth.pixels(seed, (B, T, 3, H, W))).float().cuda().contiguous()


# (preset, dtype, n_layer, B, T, H, W): the largest clip the array holds for ViT-L/16 at full
# depth, and a small fp32 ViT whose call leaves different contents in the array in between.
CASES = [
    ("vjepa2_vitl16", "bf16", None, 1, 16, 256, 256),
    ("hfvit_ti14", "fp32", None, 2, 1, 224, 224),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_two_calls_match_context_encode(case):
    name, dtype, n_layer, B, T, H, W = case
    kw = {} if n_layer is None else {"n_layer": n_layer}
    model = jv.Model.preset(name, seed=0, dtype=dtype, **kw)
    ctx = jv.Context(model, B, T, H, W)
    N = model.n_tokens(T, H, W)
    D = model.hp.embed_dim
    outs, refs = [], []
    for seed in (11, 12):
        px = clip(seed, B, T, H, W)
        refs.append(ctx.encode(px).clone())
        out = torch.empty((B, N, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        model.encode_noalloc(px, out)
        free1 = torch.cuda.mem_get_info()[0]
        if seed == 12:  # the first call may include the one-time look-up of the array
            assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
        outs.append(out)
    torch.cuda.synchronize()
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert torch.isfinite(o).all()
        bar(o, r, dtype, f"{name} call {i + 1}")
    assert not torch.equal(outs[0], outs[1])  # two clips, two results
    assert jv.ops.device_status() == 0


def test_oversized_batch_is_refused():
    model = jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16", n_layer=1)
    B, T, H, W = 2, 16, 256, 256
    px = torch.zeros((B, T, 3, H, W), dtype=torch.float32, device="cuda")
    out = torch.full((B, model.n_tokens(T, H, W), model.hp.embed_dim), 7.0, device="cuda")
    with pytest.raises(jv.JepaError) as e:
        model.encode_noalloc(px, out)
    assert e.value.status == 3 and "scratch" in e.value.text
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing ran
