"""Forged GGUF encoder files for the loader tests (there are no real checkpoints here).

Writes the GGUF format (v3 unless asked otherwise): the magic "GGUF", u32 version, u64 tensor
and key/value counts, the key/value pairs, the tensor infos (name, n_dims, dims in ggml order --
innermost first --, ggml type, offset into the data section), padding to the alignment, and the
data. The encoder keys and tensor names are the jepa.enc.* / enc.* schema of the jepa.cpp pages;
the values are the shared generator's synthetic weights.
"""
import struct

import numpy as np

import synth

U8, I8, U16, I16, U32, I32, F32, BOOL, STRING, ARRAY, U64, I64, F64 = range(13)
GGML_F32, GGML_F16, GGML_Q8_0, GGML_BF16 = 0, 1, 8, 30
_FMT = {U8: "<B", I8: "<b", U16: "<H", I16: "<h", U32: "<I", I32: "<i", F32: "<f", U64: "<Q", I64: "<q", F64: "<d"}


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _value(t: int, v) -> bytes:
    if t == STRING:
        return _str(v)
    if t == BOOL:
        return struct.pack("<B", 1 if v else 0)
    if t == ARRAY:
        et, items = v
        return struct.pack("<IQ", et, len(items)) + b"".join(_value(et, x) for x in items)
    return struct.pack(_FMT[t], v)


def _bf16_bytes(a: np.ndarray) -> bytes:
    bits = np.ascontiguousarray(a, dtype="<f4").view("<u4").astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16   # round to nearest even (finite values)
    return rounded.astype("<u2").tobytes()


def _data(a: np.ndarray, gtype: int) -> bytes:
    if gtype == GGML_F32:
        return np.ascontiguousarray(a, dtype="<f4").tobytes()
    if gtype == GGML_F16:
        return np.ascontiguousarray(a, dtype="<f2").tobytes()
    if gtype == GGML_BF16:
        return _bf16_bytes(a)
    if gtype == GGML_Q8_0:   # blocks of 32 values in 34 bytes; the content is never decoded here
        return bytes(a.size // 32 * 34)
    raise ValueError(gtype)


def write_gguf(path, kvs, tensors, alignment=32, version=3, magic=b"GGUF", truncate=0):
    """kvs: [(key, type, value)]; tensors: [(name, array in PyTorch order, ggml type)]."""
    out = bytearray(magic + struct.pack("<IQQ", version, len(tensors), len(kvs)))
    for k, t, v in kvs:
        out += _str(k) + struct.pack("<I", t) + _value(t, v)
    blobs, off = [], 0
    for name, a, gtype in tensors:
        dims = list(reversed(a.shape))
        out += _str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        out += struct.pack("<IQ", gtype, off)
        data = _data(a, gtype)
        blobs.append(data)
        off += (len(data) + alignment - 1) // alignment * alignment
    out += bytes((-len(out)) % alignment)
    for data in blobs:
        out += data + bytes((-len(data)) % alignment)
    if truncate:
        out = out[:-truncate]
    with open(path, "wb") as f:
        f.write(out)


FAMILY_OF_POS = {1: "hfvit", 2: "vjepa2", 3: "ijepa", 4: "vjepa"}


def encoder_kvs(cfg, family=None):
    """The jepa.* keys of an oracle Config (jepa.enc.* vocabulary)."""
    pos = {1: "learned", 2: "rope3d", 3: "sincos2d", 4: "sincos3d"}[cfg.pos_type]
    if family is None:
        family = "levjepa" if cfg.attn_mode == 1 else ("vjepa2_1" if cfg.rope_layout == 1 and cfg.pos_type == 2
                                                       else FAMILY_OF_POS[cfg.pos_type])
    kvs = [("general.architecture", STRING, "jepa"), ("jepa.schema_version", U32, 1), ("jepa.family", STRING, family),
           ("jepa.enc.embed_dim", U32, cfg.embed_dim), ("jepa.enc.n_layer", U32, cfg.n_layer),
           ("jepa.enc.n_head", U32, cfg.n_head), ("jepa.enc.ffn_dim", U32, cfg.ffn_dim),
           ("jepa.enc.patch_size", U32, cfg.patch_size), ("jepa.enc.tubelet_size", U32, cfg.tubelet_size),
           ("jepa.enc.img_size", U32, cfg.img_size or 224), ("jepa.enc.n_frames", U32, cfg.n_frames or 16),
           ("jepa.enc.in_chans", U32, cfg.in_chans), ("jepa.enc.ln_eps", F32, cfg.ln_eps),
           ("jepa.enc.act", STRING, "gelu_erf"), ("jepa.enc.pos_type", STRING, pos),
           ("jepa.enc.cls_token", BOOL, bool(cfg.cls_token)), ("jepa.enc.n_registers", U32, 0),
           ("jepa.enc.qkv_fused", BOOL, True), ("jepa.enc.modality_embed", BOOL, bool(cfg.modality_embed))]
    if cfg.pos_type == 2:
        kvs += [("jepa.enc.rope_theta", F32, cfg.rope_theta),
                ("jepa.enc.rope_freq_layout", STRING, "interleaved" if cfg.rope_layout else "tiled"),
                ("jepa.enc.rope_interpolate", BOOL, bool(cfg.rope_interpolate)),
                ("jepa.enc.rope_ref_grid", U32, cfg.rope_ref_grid)]
    if cfg.attn_mode == 1:
        kvs.append(("jepa.enc.attn_mode", STRING, "block_causal"))
    return kvs


def encoder_tensors(cfg, seed=0, matrix_type=GGML_BF16, fused=True, pos_table=None, round_bf16=True):
    """The enc.* tensors of an oracle Config with the generator's values (matrices bf16-rounded, as
    the bf16 model holds them, unless round_bf16 is false; q / k rows of attn_qkv.weight scaled by
    the Config's q_weight_scale / k_weight_scale); pos_table: the table of a sin-cos model (rows of
    its training grid)."""
    D, F, L = cfg.embed_dim, cfg.ffn_dim, cfg.n_layer
    K = cfg.in_chans * cfg.tubelet_size * cfg.patch_size ** 2
    P = lambda name, shape: synth.param(seed, name, shape, round_bf16)  # noqa: E731
    ts = [("enc.patch_embed.weight", P("enc.patch_embed.weight", (D, K)), matrix_type),
          ("enc.patch_embed.bias", P("enc.patch_embed.bias", (D,)), GGML_F32)]
    if cfg.pos_type == 1:
        ts.append(("enc.pos_embed", P("enc.pos_embed", (cfg.n_pos_rows, D)), GGML_F32))
    if cfg.pos_type in (3, 4):
        ts.append(("enc.pos_embed", np.asarray(pos_table, dtype=np.float32), GGML_F32))
    if cfg.cls_token:
        ts.append(("enc.cls_token", P("enc.cls_token", (D,)), GGML_F32))
    if cfg.modality_embed:
        ts.append(("enc.mod_embed_video", P("enc.mod_embed_video", (D,)), GGML_F32))
    for l in range(L):
        p = f"enc.blk.{l}."
        ts += [(p + "ln1.weight", P(p + "ln1.weight", (D,)), GGML_F32), (p + "ln1.bias", P(p + "ln1.bias", (D,)), GGML_F32)]
        wqkv, bqkv = P(p + "attn_qkv.weight", (3 * D, D)), P(p + "attn_qkv.bias", (3 * D,))
        # the oracle's test input option: q and k rows scaled in float (a bf16 model rounds the
        # file's f32 value to bf16 at load, as the oracle does)
        wqkv[:D] *= np.float32(getattr(cfg, "q_weight_scale", 1.0))
        wqkv[D:2 * D] *= np.float32(getattr(cfg, "k_weight_scale", 1.0))
        if fused:
            ts += [(p + "attn_qkv.weight", wqkv, matrix_type), (p + "attn_qkv.bias", bqkv, GGML_F32)]
        else:
            for i, part in enumerate("qkv"):
                ts += [(p + f"attn_{part}.weight", wqkv[i * D:(i + 1) * D], matrix_type),
                       (p + f"attn_{part}.bias", bqkv[i * D:(i + 1) * D], GGML_F32)]
        ts += [(p + "attn_out.weight", P(p + "attn_out.weight", (D, D)), matrix_type),
               (p + "attn_out.bias", P(p + "attn_out.bias", (D,)), GGML_F32),
               (p + "ln2.weight", P(p + "ln2.weight", (D,)), GGML_F32), (p + "ln2.bias", P(p + "ln2.bias", (D,)), GGML_F32),
               (p + "ffn_up.weight", P(p + "ffn_up.weight", (F, D)), matrix_type),
               (p + "ffn_up.bias", P(p + "ffn_up.bias", (F,)), GGML_F32),
               (p + "ffn_down.weight", P(p + "ffn_down.weight", (D, F)), matrix_type),
               (p + "ffn_down.bias", P(p + "ffn_down.bias", (D,)), GGML_F32)]
    ts += [("enc.norm.weight", P("enc.norm.weight", (D,)), GGML_F32), ("enc.norm.bias", P("enc.norm.bias", (D,)), GGML_F32)]
    return ts


def set_kv(kvs, key, t, v):
    """A copy of kvs with key set (added if absent); v None removes it."""
    out = [kv for kv in kvs if kv[0] != key]
    if v is not None:
        out.append((key, t, v))
    return out
