/*
 * jepa.h -- C ABI of the GB300 (sm_103a) ViT encoder library (libjepa_gb300.so).
 *
 * The library runs the forward pass of the shared ViT encoder graph of the jepa.cpp
 * pages ("Architecture", section "The shared ViT graph"):
 *
 *   tokens = patch_embed(rearranged pixels) [+ pos_embed] [+ cls] [+ modality vec]
 *   for each block:  x += attn(ln1(x));  x += ffn(ln2(x))    (pre-LN, GELU(erf), qkv bias)
 *   x = norm(x)
 *
 * on hand-written CUDA kernels: a pixel->patch rearrangement, tcgen05/TMEM GEMMs fed by TMA
 * (patch embed, fused QKV with bias + 3-D RoPE, out-projection + residual, FFN up + GELU,
 * FFN down + residual), a tcgen05 flash-attention kernel (full or block-causal), LayerNorm,
 * and an fp32 SIMT path for the fp32 mode. Weights are synthetic (seeded), laid out under
 * the GGUF schema's enc.* names and shapes ("GGUF schema (v1)", Encoder tensors).
 *
 * Conventions (shared by every entry point):
 *  - Every function returns jepa_status; on failure a human-readable reason is kept in a
 *    thread-local buffer (jepa_error_text), and nothing is clamped or defaulted silently
 *    ("Architecture", Robustness).
 *  - Pointers named d_* are device pointers (cudaMalloc / torch CUDA memory) on the model's
 *    device; pointers named h_* are host pointers. The caller owns every buffer it passes;
 *    the library owns the weights (jepa_model) and the workspace (jepa_context).
 *  - Launches are asynchronous on the context's (or the op's) stream. Argument errors are
 *    returned synchronously. A bounded device-side wait that gives up (a kernel that could
 *    not make progress within its time limit) is reported as JEPA_E_TIMEOUT by the next
 *    jepa_context_sync / jepa_device_status.
 *  - Thread contract ("Architecture", Robustness): a jepa_model is immutable after load and
 *    may be shared by any number of threads; a jepa_context belongs to one thread at a time.
 *  - Layouts are row-major (C order). bf16 = bfloat16 stored as uint16_t bit patterns.
 */
#ifndef JEPA_H
#define JEPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct jepa_model jepa_model;
typedef struct jepa_context jepa_context;

typedef enum {
  JEPA_OK = 0,
  JEPA_E_INVALID_ARG = 1, /* a null pointer, a non-positive or non-divisible size */
  JEPA_E_UNSUPPORTED = 2, /* a valid request this build cannot run (e.g. head_dim not 64) */
  JEPA_E_BUDGET = 3,      /* the workspace would exceed the caller's byte budget, or the context's max shape */
  JEPA_E_OOM = 4,         /* cudaMalloc failed */
  JEPA_E_CUDA = 5,        /* a CUDA runtime call failed */
  JEPA_E_TIMEOUT = 6      /* a device-side bounded wait expired; the context is still usable */
} jepa_status;

typedef enum { JEPA_FP32 = 0, JEPA_BF16 = 1 } jepa_dtype;
typedef enum {
  JEPA_POS_NONE = 0,
  JEPA_POS_LEARNED = 1,
  JEPA_POS_ROPE3D = 2,
  JEPA_POS_SINCOS2D = 3, /* fixed 2-D sin-cos table (I-JEPA) */
  JEPA_POS_SINCOS3D = 4  /* fixed 3-D sin-cos table (V-JEPA) */
} jepa_pos_type;
typedef enum { JEPA_RESIZE_TRILINEAR = 0, JEPA_RESIZE_BICUBIC = 1 } jepa_resize_mode;
typedef enum { JEPA_ROPE_TILED = 0, JEPA_ROPE_INTERLEAVED = 1 } jepa_rope_layout;
typedef enum { JEPA_ATTN_FULL = 0, JEPA_ATTN_BLOCK_CAUSAL = 1 } jepa_attn_mode;
typedef enum { JEPA_LAYOUT_TCHW = 0, JEPA_LAYOUT_CTHW = 1 } jepa_pixel_layout;

/* Encoder hyper-parameters, mirroring the jepa.enc.* keys ("GGUF schema (v1)", Encoder).
 *  pos_type        JEPA_POS_LEARNED: enc.pos_embed [n_pos_rows, D], rows = [CLS?; patches]
 *                  JEPA_POS_ROPE3D : 3-D RoPE on q and k ("Architecture", 3-D RoPE)
 *                  JEPA_POS_SINCOS2D / SINCOS3D: enc.pos_embed is the fixed sin-cos table of the
 *                  training grid (img_size/P)^2 (x n_frames/t for 3-D), baked at load; a clip of
 *                  another grid adds that table resized to its own grid, bicubic for 2-D and
 *                  trilinear for 3-D ("GGUF schema (v1)", Encoder: sincos tables). Patch rows
 *                  only: no CLS token; a 2-D table serves single-frame clips only.
 *  rope_layout     tiled (V-JEPA 2) or interleaved (V-JEPA 2.1) cos/sin table layout
 *  rope_interpolate, rope_ref_grid   V-JEPA 2.1: h, w rescaled by (ref-1)/(grid-1)
 *  cls_token       prepend enc.cls_token (no position information for it)
 *  modality_embed  add enc.mod_embed_video to every token (V-JEPA 2.1)
 *  attn_mode       full, or LeVJEPA's block-causal mask ("Architecture", Block-causal attention)
 *  img_size, n_frames  training geometry: the grid a sin-cos table is baked for (otherwise
 *                  informational; jepa_encode takes the clip's own T,H,W)
 *  sincos_w_first  2-D table halves ordered [w | h] (the HF I-JEPA table) instead of [h | w]
 *  sincos_uniform_power  3-D table with three equal axis widths 2*ceil(D/6), cut to D, instead
 *                  of (D/2, D/4, D/4) ("Converter", sincos_3d(..., uniform_power)) */
typedef struct {
  int32_t embed_dim, n_layer, n_head, ffn_dim;
  int32_t patch_size, tubelet_size, img_size, n_frames, in_chans;
  float ln_eps, rope_theta;
  int32_t pos_type, rope_layout, rope_interpolate, rope_ref_grid;
  int32_t cls_token, modality_embed, attn_mode, n_pos_rows;
  int32_t sincos_w_first, sincos_uniform_power;
} jepa_hparams;

/* ------------------------------------------------------------------ configuration */

/* Fill *out with a named workload's hyper-parameters. Names:
 *  "hfvit_ti14"      ViT-Ti/14 image encoder, learned pos + CLS (hfvit / LeWM encoder shape)
 *  "vjepa2_vitl16"   V-JEPA 2 ViT-L/16, tubelet 2, tiled 3-D RoPE
 *  "vjepa2_1_vitl16" V-JEPA 2.1 ViT-L/16, interleaved RoPE, interpolate_rope (ref grid 16), modality vector
 *  "levjepa_vitl16"  LeVJEPA ViT-L/16, tubelet 1, CLS, tiled RoPE, block-causal
 *  "vjepa2_vitg16"   V-JEPA 2 ViT-g/16 (embed 1408, 40 layers, 22 heads, ffn 6144)
 *  "vjepa_vitl16"    V-JEPA ViT-L/16, tubelet 2, 3-D sin-cos table (uniform power) baked for 16x224^2
 *  "ijepa_vitl16"    I-JEPA-style image encoder at ViT-L/16 width, [w | h] 2-D sin-cos table baked
 *                    for 224^2 (the released I-JEPA widths have head_dim 80 / 88, which this
 *                    build refuses)
 * Unknown name -> JEPA_E_INVALID_ARG. */
jepa_status jepa_preset(const char* name, jepa_hparams* out);

/* Range and invariant checks of "Architecture", Robustness (what the loader validates):
 * sizes in range, embed_dim % n_head == 0, even head width on a RoPE model, rope_interpolate
 * with a ref grid, ln_eps in [0, 1], rope_theta > 0, a learned table with rows, a sin-cos table
 * with a training grid (img_size a multiple of the patch; for 3-D n_frames a multiple of the
 * tubelet) and a width its split can take (2-D: D % 4 == 0; 3-D: D % 8 == 0 unless uniform). */
jepa_status jepa_hparams_validate(const jepa_hparams* hp);

/* Tokens of one item of a T x H x W clip: (T/t)(H/P)(W/P) + cls ("GGUF schema (v1)", Token order).
 * Refuses sizes that are not divisible by the tubelet / patch (no cropping). */
jepa_status jepa_n_tokens(const jepa_hparams* hp, int32_t T, int32_t H, int32_t W, int32_t* n_out);

/* ------------------------------------------------------------------ model */

/* Synthesise every enc.* tensor of `hp` from `seed` (synth/jepa_synth.h recipe: matrices
 * N(0,0.02), biases 0.01 N(0,1), LN gamma 1+0.1 N(0,1), beta 0.01 N(0,1), cls/pos/modality
 * N(0,0.02)) and upload it to CUDA device `device`. dtype JEPA_BF16 stores the matrix weights
 * (patch_embed, attn_qkv, attn_out, ffn_up, ffn_down) as bf16 and computes in bf16 with fp32
 * accumulation; JEPA_FP32 keeps everything fp32. Norms, biases and vectors stay fp32 in both
 * ("GGUF schema (v1)", Quantization rules). The returned model is immutable. */
jepa_status jepa_model_load(const jepa_hparams* hp, uint64_t seed, int32_t dtype, int32_t device,
                            jepa_model** out);
void jepa_model_free(jepa_model* m);
jepa_status jepa_model_hparams(const jepa_model* m, jepa_hparams* out);

/* Read the encoder of a GGUF file (v2 / v3; the jepa.* keys and enc.* tensors of "GGUF schema
 * (v1)") and check it as the pages' loader does ("Architecture", Robustness: what the loader
 * validates), without loading any weight: header counts and lengths in range; every tensor's
 * bytes inside the file; general.architecture = jepa and a known jepa.family; every jepa.enc.*
 * integer in its range and every float finite and in range; enum strings known (act, pos_type,
 * rope_freq_layout, attn_mode); block_causal only on levjepa; the derived invariants of
 * jepa_hparams_validate; every required enc.* tensor present, f32 for the operands the graph adds
 * (norms, biases, tokens, tables) and f32 / f16 / bf16 for the matrices, each shape matching the
 * hyper-parameters (a learned table's rows are taken from the tensor). Absent flags (cls_token,
 * modality_embed, rope_interpolate, layer_scale) are off; an absent attn_mode is full (the pages:
 * no existing file carries it); qkv_fused false takes attn_q / attn_k / attn_v and fuses them.
 * Refused by name: JEPA_E_INVALID_ARG for a malformed or inconsistent file; JEPA_E_UNSUPPORTED for
 * a valid file this build cannot run (family lewm, act other than gelu_erf, register tokens, layer
 * scale, quantized weights). Host only: no CUDA call. */
jepa_status jepa_gguf_hparams(const char* path, jepa_hparams* out);
/* jepa_gguf_hparams, then load the file's enc.* tensors as a model on `device` (dtype as
 * jepa_model_load: bf16 rounds the matrices to nearest even; the file's position table is used
 * as stored, and resized for other grids). */
jepa_status jepa_model_load_gguf(const char* path, int32_t dtype, int32_t device, jepa_model** out);

/* Copy the enc.* tensor `name` (e.g. "enc.blk.3.attn_qkv.weight") to host memory as float:
 * n_elems must equal the tensor's element count (shape per the GGUF schema, PyTorch row-major).
 * Synchronous. Unknown name -> JEPA_E_INVALID_ARG. */
jepa_status jepa_model_tensor(const jepa_model* m, const char* name, float* h_dst, size_t n_elems);

/* ------------------------------------------------------------------ context */

/* Allocate a workspace for clips of up to max_batch items of max_frames x max_height x max_width
 * ("Architecture", The engine in one page: jepa_context_new allocates a compute arena).
 * max_workspace_bytes = 0 means 8 GiB. Over budget -> JEPA_E_BUDGET (refused, not allocated).
 * The context starts on its own non-blocking stream of the model's device. */
jepa_status jepa_context_new(const jepa_model* m, int32_t max_batch, int32_t max_frames, int32_t max_height,
                             int32_t max_width, size_t max_workspace_bytes, jepa_context** out);
void jepa_context_free(jepa_context* c);
/* Use `stream` (a cudaStream_t, e.g. torch.cuda.current_stream().cuda_stream) for all launches. */
jepa_status jepa_context_set_stream(jepa_context* c, void* stream);
/* enable != 0: capture the encode launch sequence of a (shape, pixel ptr, token ptr) key into a
 * CUDA graph on first use and replay it afterwards ("Architecture", GPU backend: graph replay).
 * The context stream must then not be the legacy default stream. */
jepa_status jepa_context_set_graph(jepa_context* c, int32_t enable);
/* enable != 0 (the default): the encode's kernels go out as programmatic dependent launches, so
 * each kernel's set-up (barriers, TMEM, tensor-map prefetch) overlaps the end of the previous
 * one; every kernel waits for its predecessor before touching shared data, so results do not
 * change. Launches are ordinary while per-kernel profiling is on. */
jepa_status jepa_context_set_pdl(jepa_context* c, int32_t enable);
jepa_status jepa_context_workspace_bytes(const jepa_context* c, size_t* out);
/* The largest number of items one jepa_encode call of this context folds into its launch sequence
 * ("Architecture", Batching: the encode folds up to jepa_context_max_batch() items, which never
 * mix): the max_batch given to jepa_context_new. A caller with more items splits them into calls
 * of at most this many. Null argument -> JEPA_E_INVALID_ARG. */
jepa_status jepa_context_max_batch(const jepa_context* c, int32_t* out);
/* Kernel launches one jepa_encode of this shape issues (graph replay counts the kernels inside; a
 * batch that runs as two halves counts each half's). */
jepa_status jepa_context_launches(const jepa_context* c, int32_t B, int32_t T, int32_t H, int32_t W,
                                  int32_t* n_out);

/* Encode B clips. d_pixels: float [B,T,C,H,W] (layout JEPA_LAYOUT_TCHW) or [B,C,T,H,W]
 * (JEPA_LAYOUT_CTHW, the NCTHW tensor of "Architecture", Video ingest), already normalised.
 * d_tokens: float [B, N, embed_dim], N from jepa_n_tokens, after the final norm. Items never
 * mix ("Architecture", Batching). Asynchronous on the context stream. In bf16, a batch of 4 or more
 * items runs as two halves, the second on a side stream the context owns, forked from and joined
 * back into the context stream (work queued after the call waits for both; each row's result is
 * the same as in one pass). Shapes beyond the context's max -> JEPA_E_BUDGET; not divisible ->
 * JEPA_E_INVALID_ARG. A 16-byte aligned d_pixels takes the vectorised rearrangement. */
jepa_status jepa_encode(jepa_context* c, const float* d_pixels, int32_t B, int32_t T, int32_t H, int32_t W,
                        int32_t layout, float* d_tokens);

/* Same with HOST buffers: copies h_pixels to the device, encodes, copies the tokens back and
 * waits. Pinned host memory makes the copies asynchronous DMA; pageable memory also works. */
jepa_status jepa_encode_host(jepa_context* c, const float* h_pixels, int32_t B, int32_t T, int32_t H,
                             int32_t W, int32_t layout, float* h_tokens);

/* Pipelined form of jepa_encode_host for streams of clips: enqueues the upload of h_pixels, the
 * encode and the download of the tokens into h_tokens, and returns without waiting. The context
 * holds two device slots for uploads and two for downloads on streams of their own, so the copies
 * of one call run under the encodes of its neighbours (pinned host memory is needed for that
 * overlap; pageable memory works but serialises). Both host buffers must stay valid and
 * untouched until jepa_context_sync returns; the tokens are bit-identical to jepa_encode_host's.
 * Argument errors are returned at once and enqueue nothing; JEPA_E_OOM if the four slots
 * (2 x (max pixels + max tokens) floats, allocated by the first call) do not fit. */
jepa_status jepa_encode_host_async(jepa_context* c, const float* h_pixels, int32_t B, int32_t T, int32_t H,
                                   int32_t W, int32_t layout, float* h_tokens);

/* Wait for the context stream (and the copies of jepa_encode_host_async) and report device-side
 * errors (JEPA_E_TIMEOUT) raised since the last check. */
jepa_status jepa_context_sync(jepa_context* c);

/* Per-kernel timing of the encode launch sequence (the measurement side of "Architecture",
 * Tools: jepa-bench). With profiling on, every launch of jepa_encode is bracketed by CUDA events
 * recorded on the context stream (graph replay is bypassed while it is on). */
typedef struct {
  char name[24];          /* kernel class: "patchify", "gemm_patch", "ln", "gemm_qkv", "attention", ... */
  int32_t launches;       /* launches accumulated since the last reset */
  float total_ms;         /* sum of their event-measured durations */
  double flops;           /* algorithmic flops of those launches (GEMMs: 2MNK; attention: 4 hd V) */
  double bytes;           /* algorithmic HBM bytes of those launches (memory-bound kernels) */
} jepa_kernel_stat;
jepa_status jepa_context_set_profiling(jepa_context* c, int32_t enable);
/* Synchronises the context stream, folds the recorded events into at most `max` classes of
 * out[], sets *n_out, and clears the accumulators when reset != 0. */
jepa_status jepa_context_profile(jepa_context* c, jepa_kernel_stat* out, int32_t max, int32_t* n_out,
                                 int32_t reset);

/* ------------------------------------------------------------------ stage entry points
 * The kernels the encoder runs, callable one at a time (tests compare each against the oracle).
 * `stream` is a cudaStream_t (NULL = legacy default stream). Device errors of these calls are
 * reported by jepa_device_status. */

/* Rearrange pixels into patch rows ("Architecture", The shared ViT graph; element order
 * (c, dt, dy, dx), token order (t, h, w)). d_out: [B*Np, C*t*P*P] float (out_dtype JEPA_FP32)
 * or bf16 (JEPA_BF16). */
jepa_status jepa_op_patchify(const float* d_pixels, int32_t B, int32_t T, int32_t C, int32_t H, int32_t W,
                             int32_t tubelet, int32_t patch, int32_t layout, int32_t out_dtype, void* d_out,
                             void* stream);

/* LayerNorm over rows with a centred two-pass variance ("Architecture", Attention and precision):
 * d_y = (x - mean) / sqrt(var + eps) * gamma + beta; d_x float [M, D]; d_y float or bf16 [M, D].
 * D must be a multiple of 4 and at most 2048. */
jepa_status jepa_op_layernorm(const float* d_x, int32_t M, int32_t D, const float* d_gamma,
                              const float* d_beta, float eps, int32_t out_dtype, void* d_y, void* stream);

/* What a GEMM does with its accumulator tile (the fused epilogues of the encoder). */
typedef enum {
  JEPA_EPI_BIAS = 0,          /* out[m,n] = acc + bias[n]                                   */
  JEPA_EPI_BIAS_GELU = 1,     /* out[m,n] = GELU_erf(acc + bias[n])                         */
  JEPA_EPI_BIAS_RESIDUAL = 2, /* out[m,n] += acc + bias[n]   (out is the fp32 residual X)    */
  JEPA_EPI_QKV_ROPE = 3,      /* out = acc + bias, then 3-D RoPE on the q and k columns      */
  JEPA_EPI_PATCH_EMBED = 4    /* X[b*rows_per_item + prefix + i] = acc + bias (+pos) (+vec)  */
} jepa_epi_kind;

typedef struct {
  int32_t kind;               /* jepa_epi_kind */
  const float* d_bias;        /* [N] fp32, required */
  void* d_out;                /* [M, N] (or the remapped rows of PATCH_EMBED); bf16 for BIAS, BIAS_GELU
                                 and QKV_ROPE in the bf16 path, fp32 otherwise */
  /* QKV_ROPE: rows are tokens of items of rows_per_item tokens whose first `prefix` rows are
   * not rotated; columns are [q | k | v] of n_head heads of head_dim each; d_rope is the table
   * of jepa_op_rope_table for the item's patch grid (NULL: no rotation). */
  const float* d_rope;
  int32_t rows_per_item, prefix, n_head, head_dim, rope_layout;
  /* PATCH_EMBED: input row m is patch i = m % patches_per_item of item b = m / patches_per_item. */
  int32_t patches_per_item;
  const float* d_pos;         /* [rows_per_item, N] learned table (rows = [prefix; patches]) or NULL */
  const float* d_vec;         /* [N] vector added to every patch row (modality) or NULL */
  /* QKV_ROPE, optional: d_rope_ids [M] gives every row's patch index (its position in d_rope's
   * grid) in place of its place in its item (token sequences that are not the grid in order). */
  const int32_t* d_rope_ids;
} jepa_epilogue;

/* out = epilogue(x w^T): d_x [M, K], d_w [N, K] (PyTorch Linear layout), both fp32 (dtype
 * JEPA_FP32, SIMT kernel) or both bf16 (JEPA_BF16, tcgen05 kernel: K % 64 == 0, N % 64 == 0,
 * 16-byte aligned operands). */
jepa_status jepa_op_linear(int32_t dtype, const void* d_x, int32_t M, int32_t K, const void* d_w, int32_t N,
                           const jepa_epilogue* epi, void* stream);

/* 3-D RoPE cos/sin table of one item's patch grid ("Architecture", 3-D RoPE):
 * d_table float [Np, 3, d/2, 2] with (cos, sin) of pos_axis * theta^(-2k/d), d = 2*((hd/3)/2),
 * positions (t, h, w) of patch i (h, w rescaled for rope_interpolate). */
jepa_status jepa_op_rope_table(const jepa_hparams* hp, int32_t T, int32_t H, int32_t W, float* d_table,
                               void* stream);

/* Fixed sin-cos position table ("GGUF schema (v1)", Encoder: sincos tables; "Converter",
 * sincos_2d / sincos_3d). One axis of even width d maps position p to
 * [sin(p w_0) .. sin(p w_{d/2-1}), cos(p w_0) .. cos(p w_{d/2-1})], w_k = 10000^(-k/(d/2)).
 *  kind JEPA_POS_SINCOS2D: gt must be 1; row i = h*gw + w holds [axis(h) | axis(w)], each D/2
 *       wide, or [axis(w) | axis(h)] when w_first. D % 4 == 0.
 *  kind JEPA_POS_SINCOS3D: row i = (t*gh + h)*gw + w holds [axis(t) | axis(h) | axis(w)] of
 *       widths (D/2, D/4, D/4) (D % 8 == 0), or 2*ceil(D/6) each when uniform_power, cut to D.
 * d_table: device float [gt*gh*gw, D], written on `stream` (values computed in double, stored
 * as float). Bad sizes or kind -> JEPA_E_INVALID_ARG. */
jepa_status jepa_op_sincos_table(int32_t kind, int32_t gt, int32_t gh, int32_t gw, int32_t D, int32_t w_first,
                                 int32_t uniform_power, float* d_table, void* stream);

/* Resize a position table to another grid ("GGUF schema (v1)", Encoder: the runtime interpolates
 * the training-grid table for other grids, as HF does), with pixel-centre alignment: output
 * index o of an axis of n_in -> n_out samples reads the input at c = (o + 1/2) n_in/n_out - 1/2.
 *  JEPA_RESIZE_TRILINEAR: src [st, sh, sw, D] -> dst [dt, dh, dw, D]; per axis c clamped at 0,
 *       samples floor(c) and floor(c)+1 (clamped to n_in-1) blended linearly.
 *  JEPA_RESIZE_BICUBIC: per frame (st == dt), [sh, sw, D] -> [dh, dw, D]; per axis the samples
 *       floor(c)-1 .. floor(c)+2 (clamped to the axis) weighted by Keys' cubic kernel, a = -0.75.
 * d_src, d_dst: device float, 16-byte aligned, D % 4 == 0, not overlapping; arithmetic in float.
 * Bad sizes, mode or alignment -> JEPA_E_INVALID_ARG. */
jepa_status jepa_op_pos_resize(const float* d_src, int32_t st, int32_t sh, int32_t sw, int32_t D, int32_t mode,
                               float* d_dst, int32_t dt, int32_t dh, int32_t dw, void* stream);

/* Softmax attention per (item, head): o = softmax(q k^T / sqrt(head_dim) + mask) v.
 * d_qkv: [B*N, 3*n_head*head_dim] ([q | k | v] columns, heads contiguous), d_out: [B*N, n_head*head_dim];
 * fp32 (dtype JEPA_FP32) or bf16 (JEPA_BF16: tcgen05 flash kernel); head_dim 64; d_qkv (and in fp32
 * d_out) 16-byte aligned, else JEPA_E_INVALID_ARG.
 * bf16 also takes head_dim 32 (the masked predictor's heads; 64-byte tiles, scale 1/sqrt(32)).
 * attn_mode JEPA_ATTN_BLOCK_CAUSAL: the first `prefix` rows see every key, prefix columns are
 * closed to the other rows, and patch key j is visible to patch query i iff
 * (i - prefix) / frame_tokens >= (j - prefix) / frame_tokens. */
jepa_status jepa_op_attention(int32_t dtype, const void* d_qkv, int32_t B, int32_t N, int32_t n_head,
                              int32_t head_dim, int32_t attn_mode, int32_t prefix, int32_t frame_tokens,
                              void* d_out, void* stream);

/* Device-side error word of the stage entry points: JEPA_OK, or JEPA_E_TIMEOUT if a bounded wait
 * gave up since the last call (the word is cleared). Synchronises the device. */
jepa_status jepa_device_status(void);

/* Runs one kernel whose mbarrier wait can never complete, with a wait limit of `limit_us`
 * microseconds, and returns what the host then reads (JEPA_E_TIMEOUT when the limit works).
 * Exercises the failure path of every bounded wait without faulting or hanging the GPU. */
jepa_status jepa_debug_wait_timeout(int32_t limit_us);

/* ------------------------------------------------------------------ allocation-free encode
 * The jepa.cpp pages have no counterpart to this entry point. It serves callers that cannot
 * allocate device memory at all: a host program whose device memory is owned by a fixed pool or
 * by another framework's allocator, or a loop where a cudaMalloc (which may synchronise the
 * whole device) is not allowed. It runs the same kernels as jepa_encode, but its workspace is
 * one scratch array of JEPA_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library, so every
 * GPU that loads the library holds that array until the process exits.
 *  - The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine);
 *    it uses the model from jepa_model_load and the caller's pixel and token buffers as given.
 *  - A clip batch whose workspace does not fit in the array is refused with JEPA_E_BUDGET before
 *    anything is launched (one 16 x 256 x 256 ViT-L/16 clip fits; jepa_context_new has no such cap).
 *  - The first call on a device looks up the array's address on that device (set-up); make that
 *    first call before any CUDA stream capture.
 *  - All calls share the one array, which keeps whatever the last call left in it; calls whose
 *    work overlaps on the GPU (other streams, other threads) race on it: serialise them.
 *  - The call is synchronous: it launches on `stream` (a cudaStream_t, NULL = legacy default),
 *    waits for it, and returns JEPA_E_TIMEOUT if a device-side bounded wait gave up.
 * Other arguments as jepa_encode. */
#define JEPA_NOALLOC_SCRATCH_BYTES (64ull << 20)
jepa_status jepa_encode_noalloc(const jepa_model* m, const float* d_pixels, int32_t B, int32_t T, int32_t H,
                                int32_t W, int32_t layout, float* d_tokens, void* stream);

/* Thread-local text of the last failure of this thread, and its reset. */
/* ------------------------------------------------------------------ masked predictor
 *
 * The masked-latent predictor of V-JEPA 2 ("GGUF schema (v1)", Predictor: pred.* tensors; the
 * SkyVision V-JEPA 2 notes, masked-latent predictor): per item, the encoder tokens at the context
 * ids are projected by pred.embed (enc_dim -> embed_dim), a mask token (row mask_index mod
 * n_mask_tokens of pred.mask_tokens) stands at each target id, the sequence runs through
 * n_layer pre-LN blocks of the encoder's layout (pred.blk.*) with 3-D RoPE at the ids'
 * positions and full attention, pred.norm, and the target rows are projected by pred.proj
 * (embed_dim -> out_dim). The pages order the tokens by position id before the blocks and
 * restore the order after pred.norm; with full attention and per-token positions that order
 * changes no result, so the library keeps the input order [context ; targets]. */
typedef struct jepa_predictor jepa_predictor;
typedef struct jepa_pred_context jepa_pred_context;

/* jepa.pred.* hyper-parameters. head_dim = embed_dim / n_head must be 32 or 64. */
typedef struct {
  int32_t embed_dim, n_layer, n_head, ffn_dim; /* V-JEPA 2: 384, 12, 12, 1536 */
  int32_t enc_dim, out_dim;                    /* pred.embed input width, pred.proj output width */
  int32_t n_mask_tokens, mask_index;           /* 10 (V-JEPA 2); the row the targets take (1 by default) */
  float ln_eps, rope_theta;
  int32_t rope_layout;                         /* JEPA_ROPE_TILED (V-JEPA 2) or JEPA_ROPE_INTERLEAVED */
} jepa_pred_hparams;

/* "vjepa2_vitl16": the V-JEPA 2 ViT-L predictor (384 wide, 12 layers, 12 heads of 32, ffn 1536,
 * enc and out 1024, 10 mask tokens, mask index 1: transformers never passes another index,
 * per the pages). Unknown name -> JEPA_E_INVALID_ARG. */
jepa_status jepa_pred_preset(const char* name, jepa_pred_hparams* out);
jepa_status jepa_pred_hparams_validate(const jepa_pred_hparams* hp);

/* Synthesise every pred.* tensor (the enc.* recipe of jepa_model_load) and upload it to `device`;
 * bf16 only (dtype JEPA_FP32 -> JEPA_E_UNSUPPORTED). Immutable, shareable. */
jepa_status jepa_pred_load(const jepa_pred_hparams* hp, uint64_t seed, int32_t dtype, int32_t device,
                           jepa_predictor** out);
void jepa_pred_free(jepa_predictor* p);
/* Copy pred.* tensor `name` to host floats (n_elems must match), as jepa_model_tensor. */
jepa_status jepa_pred_tensor(const jepa_predictor* p, const char* name, float* h_dst, size_t n_elems);

/* Workspace for up to max_batch items of max_ctx context and max_tgt target tokens
 * (max_workspace_bytes 0 = 8 GiB; over budget -> JEPA_E_BUDGET). Own non-blocking stream. */
jepa_status jepa_pred_context_new(const jepa_predictor* p, int32_t max_batch, int32_t max_ctx, int32_t max_tgt,
                                  size_t max_workspace_bytes, jepa_pred_context** out);
void jepa_pred_context_free(jepa_pred_context* c);
jepa_status jepa_pred_context_set_stream(jepa_pred_context* c, void* stream);
/* enable != 0: capture the launch sequence of a (shape, pointers) key into a CUDA graph on first
 * use and replay it afterwards. */
jepa_status jepa_pred_context_set_graph(jepa_pred_context* c, int32_t enable);
/* Events around every launch (eager launches only while on); jepa_pred_context_profile folds them
 * per kernel class as jepa_context_profile does. */
jepa_status jepa_pred_context_set_profiling(jepa_pred_context* c, int32_t enable);
jepa_status jepa_pred_context_profile(jepa_pred_context* c, jepa_kernel_stat* out, int32_t max, int32_t* n_out,
                                      int32_t reset);
/* Kernel launches of one jepa_predict of this shape. */
jepa_status jepa_pred_context_launches(const jepa_pred_context* c, int32_t n_ctx, int32_t* n_out);

/* Predict B items, asynchronously on the context stream.
 *  d_enc:     device float [B, n_enc, enc_dim], the encoder's output tokens (no prefix rows)
 *  d_ctx_ids: device int32 [B, n_ctx], context token indices in [0, n_enc) and < gt*gh*gw
 *  d_tgt_ids: device int32 [B, n_tgt], target positions in [0, gt*gh*gw); an id may repeat and
 *             may also be a context id (the pages' all-to-all default)
 *  gt, gh, gw: the position grid the ids index (id -> t = id / (gh gw), h = id % (gh gw) / gw,
 *             w = id % gw; the pages decode predictor ids on the fixed img_size/patch grid)
 *  d_out:     device float [B, n_tgt, out_dim], 16-byte aligned
 * n_ctx may be 0; n_tgt >= 1; enc_dim % 8 == 0. An id out of range is replaced by 0 on the device
 * and reported as JEPA_E_INVALID_ARG by the next jepa_pred_context_sync. */
jepa_status jepa_predict(jepa_pred_context* c, const float* d_enc, int32_t B, int32_t n_enc, const int32_t* d_ctx_ids,
                         int32_t n_ctx, const int32_t* d_tgt_ids, int32_t n_tgt, int32_t gt, int32_t gh, int32_t gw,
                         float* d_out);
/* Wait for the context stream; JEPA_E_INVALID_ARG if an id was out of range, JEPA_E_TIMEOUT if a
 * bounded wait gave up (the word is cleared). */
jepa_status jepa_pred_context_sync(jepa_pred_context* c);

/* ------------------------------------------------------------------ attentive-pool head, pooling
 *
 * The attentive-pool head and classifier of the V-JEPA 2 video classifiers ("GGUF schema (v1)",
 * Head: head.* tensors; the SkyVision V-JEPA 2 notes, attentive pooler and classifier):
 * n_pool_layers pre-LN self-attention blocks of the encoder's layout (head.blk.*, no RoPE, no mask)
 * over all tokens, then one learned query (head.query) attends to the tokens: keys and values
 * are projected from the tokens after head.xattn.ln_kv, the query from the raw query token, there
 * is no output projection and the query is the residual (x = query + attn); then
 * x += ffn_down(GELU(ffn_up(ln2(x)))). pooled = x (the head's embedding); logits = x head.cls^T
 * + bias, with no final norm. */
typedef struct jepa_head jepa_head;
typedef struct jepa_head_context jepa_head_context;

/* jepa.head.* hyper-parameters; head_dim = embed_dim / n_head is 32, 64 or 128 (64 when
 * n_pool_layers > 0). */
typedef struct {
  int32_t embed_dim, n_head, ffn_dim, n_pool_layers, n_classes;
  float ln_eps;
} jepa_head_hparams;

/* "vjepa2_vitl16_ssv2": the V-JEPA 2 ViT-L SSv2 classifier head (1024 wide, 16 heads, ffn 4096,
 * 3 pooler layers, 174 classes). Unknown name -> JEPA_E_INVALID_ARG. */
jepa_status jepa_head_preset(const char* name, jepa_head_hparams* out);
jepa_status jepa_head_hparams_validate(const jepa_head_hparams* hp);
/* Synthesise every head.* tensor (the enc.* recipe) and upload it to `device`; bf16 only. */
jepa_status jepa_head_load(const jepa_head_hparams* hp, uint64_t seed, int32_t dtype, int32_t device, jepa_head** out);
void jepa_head_free(jepa_head* h);
jepa_status jepa_head_tensor(const jepa_head* h, const char* name, float* h_dst, size_t n_elems);

/* Workspace for up to max_batch items of max_tokens tokens (at most 32768; budget 0 = 8 GiB). */
jepa_status jepa_head_context_new(const jepa_head* h, int32_t max_batch, int32_t max_tokens, size_t max_workspace_bytes,
                                  jepa_head_context** out);
void jepa_head_context_free(jepa_head_context* c);
jepa_status jepa_head_context_set_stream(jepa_head_context* c, void* stream);
jepa_status jepa_head_context_set_graph(jepa_head_context* c, int32_t enable);
jepa_status jepa_head_context_set_profiling(jepa_head_context* c, int32_t enable);
jepa_status jepa_head_context_profile(jepa_head_context* c, jepa_kernel_stat* out, int32_t max, int32_t* n_out,
                                      int32_t reset);
/* Kernel launches of one jepa_head_forward (with_logits != 0: the classifier too). */
jepa_status jepa_head_context_launches(const jepa_head_context* c, int32_t with_logits, int32_t* n_out);

/* Run the head on B items of N encoder tokens, asynchronously on the context stream.
 *  d_tokens: device float [B, N, embed_dim] (the encoder's output; read only), 16-byte aligned
 *  d_pooled: device float [B, embed_dim] or NULL;  d_logits: device float [B, n_classes] or NULL
 *  (at least one of the two). */
jepa_status jepa_head_forward(jepa_head_context* c, const float* d_tokens, int32_t B, int32_t N, float* d_pooled,
                              float* d_logits);
/* Wait for the context stream; JEPA_E_TIMEOUT if a bounded wait gave up. */
jepa_status jepa_head_context_sync(jepa_head_context* c);

/* Pooled features of encoder tokens: JEPA_POOL_MEAN = the mean of the patch tokens, rows
 * [prefix, N) ("GGUF schema (v1)", ijepa note: the feature is the mean of the patch tokens);
 * JEPA_POOL_CLS = row 0, the CLS token (hfvit / levjepa; needs prefix >= 1).
 * d_tokens: device float [B, N, D], d_out: device float [B, D], both 16-byte aligned, D % 4 == 0. */
typedef enum { JEPA_POOL_MEAN = 0, JEPA_POOL_CLS = 1 } jepa_pool_mode;
jepa_status jepa_op_pool(int32_t mode, const float* d_tokens, int32_t B, int32_t N, int32_t D, int32_t prefix,
                         float* d_out, void* stream);

const char* jepa_error_text(void);
void jepa_error_reset(void);

#ifdef __cplusplus
}
#endif
#endif /* JEPA_H */
