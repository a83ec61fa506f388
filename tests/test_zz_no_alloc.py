"""Allocation-free encode against the context encode (GPU only).

jepa_encode_noalloc is for callers that must not allocate device memory: code running inside
another framework's memory pool, a fixed-budget embedded service, or a loop where a cudaMalloc
(which can synchronise the device) is not allowed. It runs the encoder with a fixed scratch
array compiled into the library as its workspace.

The test makes one set-up call (the first call on a device looks up the array's address; the
first launches of each kernel may also load its module), then two calls in a row on two other
clips. Each of the two must equal jepa_encode on the same clip bit for bit: both run the same
launch sequence (one lane, the same tile widths, the same kernels), so any difference would mean
stale or aliased scratch. The device's free memory must be the same before the first of the two
calls and after the second: nothing is allocated and kept by either call. A batch whose
workspace does not fit in the array is refused before anything is launched.
The file name sorts last so that it also runs after every other GPU test.
"""
import pytest
import torch

import synth

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu


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
    clips = [clip(seed, B, T, H, W) for seed in (10, 11, 12)]
    refs = [ctx.encode(px).clone() for px in clips[1:]]
    outs = [torch.full((B, N, D), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    model.encode_noalloc(clips[0], outs[0])   # set-up call
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    model.encode_noalloc(clips[1], outs[1])
    model.encode_noalloc(clips[2], outs[2])
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, f"device free memory moved by {free_before - free_after} bytes"
    for i, (o, r) in enumerate(zip(outs[1:], refs)):
        assert torch.isfinite(o).all(), f"{name} call {i + 1}"
        assert torch.equal(o, r), f"{name} call {i + 1}: max |d| {(o - r).abs().max().item():.3e}"
    assert not torch.equal(outs[1], outs[2])  # two clips, two results
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
