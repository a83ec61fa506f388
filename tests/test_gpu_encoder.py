"""Whole-encoder parity of the GPU path against the oracle (GPU only).

Bars (per workload dtype):
  fp32: max |y - ref| / max |ref| <= 1e-4
  bf16: per-token cosine >= 0.9999 and max |y - ref| <= 3e-2 (outputs are unit-scale after the norm)
Small cases run the live oracle (2 layers, a few hundred tokens, several tiles + ragged tail);
full-size cases compare sampled rows with tests/golden/full_<workload>.npz, written by
tests/golden/make_full_goldens.py from the oracle alone.
"""
import os
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
from configs import WORKLOADS, small

jv = pytest.importorskip("jepa_vision_encoder_gb300")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PRESET = {
    "hfvit_ti14_224": "hfvit_ti14",
    "vjepa2_vitl16_16x256": "vjepa2_vitl16",
    "vjepa2_1_vitl16_16x384": "vjepa2_1_vitl16",
    "levjepa_vitl16_16x256": "levjepa_vitl16",
    "vjepa2_vitg16_64x256": "vjepa2_vitg16",
    "vjepa_vitl16_16x256": "vjepa_vitl16",
    "ijepa_vitl16_256": "ijepa_vitl16",
}


def check_bar(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    err = np.abs(got - ref)
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    if dtype == "fp32":
        rel = err.max() / np.abs(ref).max()
        assert rel <= 1e-4, f"{what}: max rel err {rel:.3e}"
    else:
        assert cos.min() >= 0.9999, f"{what}: min token cosine {cos.min():.7f}"
        assert err.max() <= 3e-2, f"{what}: max abs err {err.max():.3e}"
    return err.max(), cos.min()


def make(name, n_layer=None, batch=1, T=None, H=None, W=None, graph=False, cfg=None):
    cfg0, dtype, _, (T0, H0, W0) = WORKLOADS[name]
    kw = {} if n_layer is None else {"n_layer": n_layer}
    if cfg is not None and cfg.pos_type in (jv.POS_SINCOS2D, jv.POS_SINCOS3D):   # the grid the table is baked for
        kw.update(img_size=cfg.img_size, n_frames=cfg.n_frames)
    model = jv.Model.preset(PRESET[name], seed=0, dtype=dtype, **kw)
    ctx = jv.Context(model, batch, T or T0, H or H0, W or W0, graph=graph)
    return model, ctx


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_small_encoder_matches_oracle(name):
    cfg, dtype, (T, H, W) = small(name)
    B = 2
    model, ctx = make(name, n_layer=cfg.n_layer, batch=B, T=T, H=H, W=W, cfg=cfg)
    pix = synth.pixels(0, (B, T, 3, H, W))
    out = ctx.encode(torch.from_numpy(pix).cuda())
    ctx.sync()
    ref = oracle.encode(cfg, 0, dtype == "bf16", pix)
    check_bar(out.cpu().numpy(), ref, dtype, name)


# The degenerate clips: one patch per frame (one token per tubelet; with a CLS row, two tokens),
# so every kernel runs on a single row tile with one valid row and a 1 x 1 position grid.
@pytest.mark.parametrize("name,T,H,W", [("vjepa2_vitl16_16x256", 2, 16, 16), ("vjepa2_1_vitl16_16x384", 2, 16, 16),
                                        ("levjepa_vitl16_16x256", 1, 16, 16), ("levjepa_vitl16_16x256", 3, 16, 16)])
def test_one_patch_clips_match_oracle(name, T, H, W):
    cfg, dtype, _ = small(name)
    B = 2
    model, ctx = make(name, n_layer=cfg.n_layer, batch=B, T=T, H=H, W=W, cfg=cfg)
    pix = synth.pixels(5, (B, T, 3, H, W))
    out = ctx.encode(torch.from_numpy(pix).cuda())
    ctx.sync()
    ref = oracle.encode(cfg, 0, dtype == "bf16", pix)
    assert out.shape == ref.shape
    check_bar(out.cpu().numpy(), ref, dtype, f"{name} {T}x{H}x{W}")


def test_weights_are_the_generator_bits():
    model = jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16", n_layer=1)
    for name, shape in [("enc.blk.0.attn_qkv.weight", (3072, 1024)), ("enc.blk.0.ln1.weight", (1024,)),
                        ("enc.patch_embed.bias", (1024,))]:
        assert np.array_equal(model.tensor(name, shape).numpy(), synth.param(0, name, shape, True))


def test_layouts_agree_bit_exact():
    name = "vjepa2_vitl16_16x256"
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=2, batch=1, T=T, H=H, W=W)
    pix = synth.pixels(1, (1, T, 3, H, W))
    a = ctx.encode(torch.from_numpy(pix).cuda()).clone()
    b = ctx.encode(torch.from_numpy(np.ascontiguousarray(pix.transpose(0, 2, 1, 3, 4))).cuda(), layout=jv.LAYOUT_CTHW)
    ctx.sync()
    assert torch.equal(a, b)


# B = 5 (bf16) runs as two uneven halves (3 + 2 items) on two streams; graph replay captures both
@pytest.mark.parametrize("B,graph", [(3, False), (5, False), (5, True)])
@pytest.mark.parametrize("name", ["vjepa2_vitl16_16x256", "levjepa_vitl16_16x256", "hfvit_ti14_224"])
def test_batch_items_equal_single_calls(name, B, graph):
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=2, batch=B, T=T, H=H, W=W, graph=graph)
    pix = torch.from_numpy(synth.pixels(2, (B, T, 3, H, W))).cuda()
    full = ctx.encode(pix).clone()
    for b in range(B):
        one = ctx.encode(pix[b:b + 1].contiguous()).clone()
        assert torch.equal(full[b:b + 1], one), f"item {b}"
    ctx.sync()


def test_graph_replay_and_host_api_match_eager():
    name = "levjepa_vitl16_16x256"
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=2, batch=2, T=T, H=H, W=W)
    pix_h = torch.from_numpy(synth.pixels(3, (2, T, 3, H, W)))
    eager = ctx.encode(pix_h.cuda()).clone()
    ctx.set_graph(True)
    pix_d = pix_h.cuda()
    out = torch.empty_like(eager)
    for _ in range(3):
        ctx.encode(pix_d, out)
    ctx.sync()
    assert torch.equal(out, eager)
    host = ctx.encode_host(pix_h.pin_memory())
    assert torch.equal(host, eager.cpu())


def test_pipelined_host_encodes_match_the_synchronous_ones():
    """Several jepa_encode_host_async calls in flight (uploads and downloads overlapping other
    calls' encodes, the two device slots each reused) give the synchronous call's bits, per call."""
    name = "vjepa2_vitl16_16x256"
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=2, batch=2, T=T, H=H, W=W)
    ctx.set_graph(True)
    clips = [torch.from_numpy(synth.pixels(20 + i, (2, T, 3, H, W))).pin_memory() for i in range(5)]
    ref = [ctx.encode_host(c).clone() for c in clips]
    outs = [torch.empty_like(r).pin_memory() for r in ref]
    for c, o in zip(clips, outs):
        ctx.encode_host_async(c, o)
    ctx.sync()
    for i, (o, r) in enumerate(zip(outs, ref)):
        assert torch.equal(o, r), f"call {i}"
    # one clip of a different batch size through the same slots, then the first clip again
    small_out = torch.empty((1,) + ref[0].shape[1:]).pin_memory()
    ctx.encode_host_async(clips[1][:1].contiguous().pin_memory(), small_out)
    ctx.encode_host_async(clips[0], outs[0])
    ctx.sync()
    assert torch.equal(small_out, ref[1][:1]) and torch.equal(outs[0], ref[0])


def test_pipelined_host_refusals_and_mixing_with_the_synchronous_call():
    name = "vjepa2_vitl16_16x256"
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=1, batch=2, T=T, H=H, W=W)
    clip = torch.from_numpy(synth.pixels(30, (2, T, 3, H, W))).pin_memory()
    ref = ctx.encode_host(clip).clone()
    too_big = torch.from_numpy(synth.pixels(31, (3, T, 3, H, W))).pin_memory()
    out3 = torch.empty((3,) + ref.shape[1:]).pin_memory()
    with pytest.raises(jv.JepaError) as e:
        ctx.encode_host_async(too_big, out3)  # over the context's batch: refused, nothing enqueued
    assert e.value.status == jv._lib.E_BUDGET
    a, b = torch.empty_like(ref).pin_memory(), torch.empty_like(ref).pin_memory()
    ctx.encode_host_async(clip, a)
    mid = ctx.encode_host(clip)            # a synchronous call between pipelined ones
    ctx.encode_host_async(clip, b)
    ctx.sync()
    assert torch.equal(a, ref) and torch.equal(mid, ref) and torch.equal(b, ref)


@pytest.mark.parametrize("name", ["vjepa2_vitl16_16x256", "hfvit_ti14_224"])
def test_programmatic_launches_change_nothing(name):
    # the same kernels with and without programmatic dependent launch, eager and graph replay
    cfg, dtype, (T, H, W) = small(name)
    model, ctx = make(name, n_layer=cfg.n_layer, batch=2, T=T, H=H, W=W)
    pix = torch.from_numpy(synth.pixels(5, (2, T, 3, H, W))).cuda()
    ctx.set_pdl(False)
    ref = ctx.encode(pix).clone()
    ctx.set_pdl(True)
    out = ctx.encode(pix).clone()
    ctx.set_graph(True)
    for _ in range(2):
        graph_out = ctx.encode(pix).clone()
    ctx.sync()
    assert torch.equal(out, ref)
    assert torch.equal(graph_out, ref)


def test_two_threads_two_contexts_bit_identical():
    name = "vjepa2_1_vitl16_16x384"
    cfg, dtype, (T, H, W) = small(name)
    model = jv.Model.preset(PRESET[name], seed=0, dtype=dtype, n_layer=2)
    pix = torch.from_numpy(synth.pixels(4, (1, T, 3, H, W)))
    results = {}

    def run(i):
        ctx = jv.Context(model, 1, T, H, W)
        results[i] = ctx.encode_host(pix)
        ctx.close()

    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert torch.equal(results[0], results[1])


def test_refusals():
    model = jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16", n_layer=1)
    with pytest.raises(jv.JepaError) as e:
        jv.Context(model, 64, 64, 512, 512, max_workspace_bytes=1 << 30)
    assert e.value.status == jv._lib.E_BUDGET
    ctx = jv.Context(model, 1, 4, 64, 64)
    assert ctx.max_batch == 1 and jv.Context(model, 3, 4, 64, 64).max_batch == 3
    with pytest.raises(jv.JepaError) as e:   # more items than jepa_context_max_batch
        ctx.encode(torch.zeros((2, 4, 3, 64, 64), dtype=torch.float32, device="cuda"))
    assert e.value.status == jv._lib.E_BUDGET
    with pytest.raises(jv.JepaError) as e:
        ctx.encode(torch.zeros((1, 3, 3, 64, 64), dtype=torch.float32, device="cuda"))
    assert e.value.status == jv._lib.E_INVALID_ARG
    hf = jv.Model.preset("hfvit_ti14", seed=0, dtype="fp32", n_layer=1)
    c2 = jv.Context(hf, 1, 1, 112, 112)
    with pytest.raises(jv.JepaError) as e:   # learned table of 257 rows, clip of 65 tokens
        c2.encode(torch.zeros((1, 1, 3, 112, 112), dtype=torch.float32, device="cuda"))
    assert e.value.status == jv._lib.E_UNSUPPORTED
    with pytest.raises(jv.JepaError) as e:
        jv.Model.preset("vjepa2_vitl16", seed=0, dtype="bf16", n_layer=1, n_head=8)   # head_dim 128
    assert e.value.status == jv._lib.E_UNSUPPORTED


def golden_cases():
    return [n for n in WORKLOADS if os.path.exists(os.path.join(GOLDEN, f"full_{n}.npz"))]


@pytest.mark.parametrize("name", golden_cases())
def test_full_size_sampled_rows_match_oracle(name):
    g = np.load(os.path.join(GOLDEN, f"full_{name}.npz"))
    cfg, dtype, batches, (T, H, W) = WORKLOADS[name]
    B = int(g["batch"])
    model, ctx = make(name, batch=B)
    pix = torch.from_numpy(synth.pixels(int(g["seed"]), (B, T, 3, H, W))).cuda()
    out = ctx.encode(pix)
    ctx.sync()
    rows = torch.from_numpy(g["rows"]).long().cuda()
    for j, b in enumerate(g["items"]):
        got = out[int(b)][rows].cpu().numpy()
        check_bar(got, g["tokens"][j].astype(np.float64), dtype, f"{name} item {b}")
    if B > 1:   # every item of the full batch equals its single-item encode
        one = jv.Context(model, 1, T, H, W)
        for b in range(B):
            assert torch.equal(one.encode(pix[b:b + 1].contiguous()), out[b:b + 1]), f"item {b}"
