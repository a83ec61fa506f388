/*
 * oracle.h -- plain, slow, fp64 CPU reference of the shared ViT encoder forward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library includes, links or
 * calls this code; only the tests, the smoke check and the bench's CPU-baseline
 * leg use it. It shares no code with the GPU path except the seeded input
 * generator (synth/jepa_synth.h).
 *
 * Every function follows a passage of the jepa.cpp pages:
 *   [S] = jepa.cpp "GGUF schema (v1)"      (tensor table, token order, family notes)
 *   [A] = jepa.cpp "Architecture"          (shared ViT graph, 3-D RoPE, block-causal attention)
 *   [C] = jepa.cpp "Converter"             (conv flattening, qkv fusing, hfvit/levjepa maps)
 *   [K] = SkyVision.cpp README, V-JEPA 2 section (tubelet packing order, tiled-RoPE quirk)
 *   [R] = jepa.cpp "Converter" reference table (sincos_2d / sincos_3d helpers, ijepa table order)
 *
 * All arithmetic is double precision; bf16 inputs (weights of the bf16 mode)
 * enter as their exact values.
 */
#ifndef JEPA_ORACLE_H
#define JEPA_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Encoder hyper-parameters, mirroring the jepa.enc.* keys of [S] "Encoder". */
typedef struct {
  int embed_dim, n_layer, n_head, ffn_dim;
  int patch_size, tubelet_size, in_chans;
  double ln_eps, rope_theta;
  int pos_type;         /* 0 none, 1 learned table, 2 rope3d, 3 sincos2d, 4 sincos3d */
  int rope_layout;      /* 0 tiled (V-JEPA 2), 1 interleaved (V-JEPA 2.1) */
  int rope_interpolate; /* V-JEPA 2.1 interpolate_rope */
  int rope_ref_grid;    /* 256 / patch_size */
  int cls_token;        /* prepend enc.cls_token */
  int modality_embed;   /* add enc.mod_embed_video to every token */
  int attn_mode;        /* 0 full, 1 block_causal */
  int n_pos_rows;       /* rows of enc.pos_embed (learned only) */
  int img_size;         /* training crop: the sin-cos table covers (img/P) x (img/P) ... */
  int n_frames;         /* ... x (frames/t) positions */
  int sincos_w_first;   /* sincos2d halves ordered [w | h] (HF I-JEPA) instead of [h | w] */
  int sincos_uniform_power; /* sincos3d: three equal axis widths 2*ceil(D/6), cut to D */
  /* Test input, not part of the method: the synthetic q rows [0, D) and k rows [D, 2D) of every
   * enc.blk.*.attn_qkv.weight are multiplied by these factors (1 = the plain recipe), in float,
   * and with bf16 weights rounded to bf16 again (round to nearest even), which is the value a bf16
   * model holds when a file stores the scaled weight in f32. Larger q, k give peaked attention, so
   * that a test encoder's output depends strongly on the scores (RoPE layout, mask). */
  double q_weight_scale, k_weight_scale;
} oracle_hparams;

/* Number of tokens of one item: (T/t)(H/P)(W/P) + cls. Returns -1 if a size is not divisible. */
int oracle_n_tokens(const oracle_hparams* hp, int T, int H, int W);

/* Pixel -> patch rows ([A] "The shared ViT graph"; [S] "Token order"; [K] tubelet packing).
 * pix: [B,T,C,H,W] (layout 0) or [B,C,T,H,W] (layout 1), float.
 * out: [B*Np, C*t*P*P], element k = ((c*t + dt)*P + dy)*P + dx, token i = (tt*gh + hh)*gw + ww. */
int oracle_patchify(const oracle_hparams* hp, const float* pix, int B, int T, int H, int W, int layout,
                    double* out);

/* Brute-force strided 3-D convolution (kernel = stride = (t, P, P)), the operation the
 * rearrangement + matmul replaces ([A] "The shared ViT graph").
 * w: [D, C, t, P, P]; out: [B, gt, gh, gw, D]. */
int oracle_conv3d(const oracle_hparams* hp, const float* pix, int B, int T, int H, int W, int layout,
                  const double* w, const double* bias, double* out);

/* y = x w^T + b; x [M,K], w [N,K] (PyTorch row-major, [S] tensor table), b [N] or NULL. */
void oracle_linear(const double* x, int M, int K, const double* w, const double* b, int N, double* y);

/* LayerNorm over rows: centred two-pass biased variance, eps inside the sqrt ([A] "Attention and precision"). */
void oracle_layernorm(const double* x, int M, int D, const double* gamma, const double* beta, double eps,
                      double* y);

/* GELU(erf): 0.5 x (1 + erf(x / sqrt 2)) ([S] jepa.enc.act = gelu_erf). */
void oracle_gelu(const double* x, size_t n, double* y);

/* Per-patch-token RoPE positions (t, h, w) ([A] "3-D RoPE"), with interpolate_rope
 * scaling of h and w by (ref-1)/(g-1). pos: [Np, 3]. */
int oracle_rope_positions(const oracle_hparams* hp, int T, int H, int W, double* pos);

/* cos / signed-sin tables [N, hd] for all N tokens (prefix rows are identity), so that
 * rope(x)[j] = x[j] cos[j] + x[j^1] sin[j] for j < 3d and x[j] for the rest. */
int oracle_rope_tables(const oracle_hparams* hp, int T, int H, int W, double* cos_t, double* sin_t);

/* Apply the tables to x [N, H*hd] in place-free form (q and k of every head). */
void oracle_rope_apply(const double* x, int N, int n_head, int hd, const double* cos_t, const double* sin_t,
                       double* out);

/* Fixed sin-cos position tables ([S] "Encoder": sincos2d / sincos3d, baked at conversion for the
 * training grid; [R] sincos_2d, sincos_3d). One axis of even width d maps position p to
 * [sin(p w_0) .. sin(p w_{d/2-1}), cos(p w_0) .. cos(p w_{d/2-1})], w_k = 10000^(-k/(d/2)).
 * sincos_2d: rows i = h*gw + w, columns [axis(h) | axis(w)] of width D/2 each, or [axis(w) | axis(h)]
 *   when w_first (the order of the HF I-JEPA table). D % 4 == 0. out: [gh*gw, D].
 * sincos_3d: rows i = (t*gh + h)*gw + w, columns [axis(t) | axis(h) | axis(w)] of widths
 *   (D/2, D/4, D/4), or 2*ceil(D/6) each when uniform_power, the row then cut to its first D
 *   columns. out: [gt*gh*gw, D]. Returns -1 on a width the split cannot take. */
int oracle_sincos_2d(int gh, int gw, int D, int w_first, double* out);
int oracle_sincos_3d(int gt, int gh, int gw, int D, int uniform_power, double* out);

/* Resizing a position table to another grid ([S] "Encoder": the runtime interpolates the
 * training-grid table for other grids; [S] ijepa note: as HF does). Pixel-centre alignment
 * (align_corners off): output index o of an axis resized from n_in to n_out samples reads the
 * input at c = (o + 1/2) n_in / n_out - 1/2.
 * trilinear: src [st, sh, sw, D] -> dst [dt, dh, dw, D]; per axis c is clamped at 0 and the two
 *   neighbours floor(c), floor(c)+1 (the latter clamped to n_in-1) are blended linearly.
 * bicubic: src [sh, sw, D] -> dst [dh, dw, D]; per axis the four samples floor(c)-1 .. floor(c)+2
 *   (indices clamped to [0, n_in-1]) are weighted by Keys' cubic convolution kernel, a = -0.75.
 * Returns -1 on a non-positive size. */
int oracle_interp_trilinear(const double* src, int st, int sh, int sw, int D, int dt, int dh, int dw, double* dst);
int oracle_interp_bicubic(const double* src, int sh, int sw, int D, int dh, int dw, double* dst);

/* The position table one clip adds to its patch rows, [gt*gh*gw, D], for pos_type 3 / 4: the
 * sin-cos table of the training grid ((n_frames/t) x (img/P) x (img/P); one frame for sincos2d),
 * resized to the clip's grid when they differ (bicubic for sincos2d, trilinear for sincos3d).
 * Returns -1 on a bad size, -2 when the table cannot serve the clip (sincos2d on several frames). */
int oracle_pos_table(const oracle_hparams* hp, int T, int H, int W, double* out);

/* cos / signed-sin tables [n, hd] of n tokens at explicit (t, h, w) positions pos [n, 3], the
 * same rule as oracle_rope_tables (no prefix rows). */
void oracle_rope_tables_pos(int hd, double theta, int layout, const double* pos, int n, double* cos_t,
                            double* sin_t);

/* Is key k visible to query q? attn_mode 0: every k < N. attn_mode 1 (block-causal,
 * [S] levjepa note; [A] "Block-causal attention"): prefix rows see everything, prefix
 * columns are closed to patch queries, patch keys visible iff frame(q) >= frame(k). */
int oracle_mask_allow(int attn_mode, int prefix, int frame_tokens, int N, int q, int k);

/* Softmax attention per head: o = softmax(q k^T / sqrt(hd) + mask) v.
 * q, k, v, o: [N, H*hd], heads contiguous ([A] "Attention and precision"). */
void oracle_attention(const double* q, const double* k, const double* v, int N, int n_head, int hd,
                      int attn_mode, int prefix, int frame_tokens, double* o);

/* The whole encoder ([A] "The shared ViT graph") for B items with synthetic weights of
 * `seed` (bf16_weights != 0 rounds the matrix weights to bf16, as the bf16 model holds them).
 * out: [B, N, D]; final_norm = 0 returns the residual stream before enc.norm. */
int oracle_encode(const oracle_hparams* hp, uint64_t seed, int bf16_weights, const float* pix, int B, int T,
                  int H, int W, int layout, int final_norm, double* out);

/* Masked-latent predictor hyper-parameters (jepa.pred.* of [S] "Predictor"). */
typedef struct {
  int embed_dim, n_layer, n_head, ffn_dim; /* predictor width, depth, heads, ffn (V-JEPA 2: 384/12/12/1536) */
  int enc_dim, out_dim;                    /* pred.embed input width, pred.proj output width */
  int n_mask_tokens, mask_index;           /* rows of pred.mask_tokens; the row targets take (mod n) */
  double ln_eps, rope_theta;
  int rope_layout;                         /* 0 tiled (V-JEPA 2), 1 interleaved */
} oracle_pred_hparams;

/* The masked predictor ([S] "Predictor" tensor table; [K] V-JEPA 2 section, masked-latent
 * predictor): per item, the encoder tokens at the context ids are projected by pred.embed, a
 * mask token (row mask_index mod n_mask_tokens of pred.mask_tokens) stands at each target id,
 * the tokens are put in order of position id (stable), run through the pred.blk stack (the
 * encoder's block with 3-D RoPE at the ids' positions, full attention), normalised by
 * pred.norm, put back in their input order, and the target rows projected by pred.proj.
 * Position id -> (t, h, w) = (id / (gh gw), (id mod gh gw) / gw, id mod gw).
 * enc [B, n_enc, enc_dim]; ctx_ids [B, n_ctx] in [0, n_enc); tgt_ids [B, n_tgt] >= 0;
 * out [B, n_tgt, out_dim]. Returns -1 on a bad size or id. */
int oracle_predict(const oracle_pred_hparams* hp, uint64_t seed, int bf16_weights, const double* enc, int B,
                   int n_enc, const int* ctx_ids, int n_ctx, const int* tgt_ids, int n_tgt, int gh, int gw,
                   double* out);

/* Attention of Nq query rows over Nk key / value rows per head, o = softmax(q k^T / sqrt(hd)) v
 * (no mask): q [Nq, H*hd], k, v [Nk, H*hd], o [Nq, H*hd], heads contiguous. */
void oracle_cross_attention(const double* q, int Nq, const double* k, const double* v, int Nk, int n_head, int hd,
                            double* o);

/* Attentive-pool head hyper-parameters (jepa.head.* of [S] "Head"). */
typedef struct {
  int embed_dim, n_head, ffn_dim, n_pool_layers, n_classes;
  double ln_eps;
} oracle_head_hparams;

/* The attentive-pool head and classifier ([S] "Head" tensor table; [K] V-JEPA 2 section, the
 * attentive pooler and the classifier): n_pool_layers pre-LN self-attention blocks over all
 * tokens (the encoder block's layout, head.blk.*, no RoPE, no mask), then one learned query
 * (head.query) attends to the tokens: keys and values are projected (head.xattn.k / .v) from
 * the tokens after head.xattn.ln_kv, the query (head.xattn.q) from the raw query token, there is
 * no output projection, and the query is the residual: x = query + attn; x += down(GELU(up(
 * ln2(x)))) (head.xattn.ffn_*). pooled = x; logits = x head.cls^T + bias (no final norm).
 * tokens [B, N, D]; pooled [B, D] and logits [B, n_classes] (either may be NULL). */
int oracle_attentive_head(const oracle_head_hparams* hp, uint64_t seed, int bf16_weights, const double* tokens, int B,
                          int N, double* pooled, double* logits);

/* Pooled features of [B, N, D] tokens whose first `prefix` rows are prefix (CLS) tokens:
 * mode 0 = the mean of the N - prefix patch tokens ([S] ijepa note: the feature is the mean of
 * the patch tokens), mode 1 = row 0, the CLS token ([C] hfvit / levjepa: the CLS token).
 * out [B, D]. Returns -1 on a bad size or mode (mode 1 needs prefix >= 1). */
int oracle_pool(const double* tokens, int B, int N, int D, int prefix, int mode, double* out);

/* Number of OpenMP threads the oracle uses. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
