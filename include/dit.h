/*
 * dit.h -- C ABI of libdit.so: the forward pass of a non-causal joint video+audio diffusion
 * transformer (DiT) over a packed variable-length token sequence, and the rectified-flow Euler
 * step of the denoise loop around it, on one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited as page title then section:
 *   [H3] "feat(minimax-h3): port the MiniMax-H3 omni-modal video+audio DiT"
 *   [M3] "feat(MODEL-MUSIC-MUSIC3): the 2.4B fp32 DiT onto the device, staged once"
 *   [BF] "feat(minimax-h3): stream the ORIGINAL bf16 DiT to the device, one tensor at a time"
 *
 * Conventions shared by every call:
 *   - Array arguments are DEVICE pointers owned by the caller unless the name ends in _host.
 *     Nothing here frees or retains a caller pointer beyond the call, except bound weights
 *     (dit_bind_weights), which must outlive the handle.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All device
 *     work is enqueued on it; no call synchronises the device unless it says so.
 *   - Errors are return codes only: no exception, abort or exit crosses this boundary.  Host-side
 *     validation happens before any launch, so a call that returns an error launched nothing.
 *     Device-side failures (an invalid packed layout, a bounded wait that ran out) are recorded in
 *     a device status word and are read back by dit_get_stats / dit_sync_status.
 *   - Row-major everywhere.  A linear map's weight is [out, in] (the "MatmulBT" convention of
 *     [M3] "What moved": Y = X W^T).
 */
#ifndef DIT_H_
#define DIT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DIT_API __attribute__((visibility("default")))
#else
#define DIT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, negative size, bad enum */
  DIT_ERR_CONFIG = 2,         /* a dit_config field out of the supported range */
  DIT_ERR_UNBOUND = 3,        /* dit_forward before dit_bind_weights */
  DIT_ERR_MISSING_WEIGHT = 4, /* a required weight pointer is NULL; dit_last_error names it */
  DIT_ERR_LAYOUT = 5,         /* packed layout rejected (host checks, or the device validator) */
  DIT_ERR_CAPACITY = 6,       /* n_tokens > max_tokens, n_docs > max_docs, workspace too small */
  DIT_ERR_CUDA = 7,           /* a CUDA runtime call failed; dit_last_error has its message */
  DIT_ERR_DEVICE_TIMEOUT = 8, /* a kernel's bounded wait ran out; the kernel exited cleanly */
  DIT_ERR_UNSUPPORTED = 9,    /* shape outside what the kernels tile (see dit_create) */
  DIT_ERR_RANGE = 10          /* a weight or activation beyond the f16 operands' range (65504); see act_bf16 */
} dit_status;

enum { DIT_RMSNORM = 0, DIT_LAYERNORM = 1 };
enum { DIT_BF16 = 0, DIT_FP32 = 1 };
/* 16-bit operand type of the op-level tensor-core calls (A, B, and the 16-bit outputs they write). */
enum { DIT_ELEM_BF16 = 0, DIT_ELEM_F16 = 1 };

/* Model configuration.  [H3] "The device-resident forward (W2b)" for the modality-indexed AdaLN
 * DiT (adaln = 1, RMSNorm); [M3] "What moved" for the music DiT (adaln = 0, LayerNorm, partial
 * rotary, 1x1 pre/post convolutions). */
typedef struct {
  int n_blocks;       /* L */
  int hidden;         /* d */
  int n_heads;        /* H */
  int head_dim;       /* Dh, H * Dh == d */
  int ffn_hidden;     /* F: the FFN computes value * silu(gate) over an up projection 2F wide */
  int norm;           /* DIT_RMSNORM | DIT_LAYERNORM; either takes the per-channel gain / shift weights when given */
  float norm_eps;
  int adaln;          /* 1: modality-indexed AdaLN modulate + gated residuals; 0: plain residuals */
  int n_modalities;   /* tags index [0, n_modalities): 0 = video, 1 = audio */
  int t_embed_dim;    /* width of the sinusoidal timestep embedding (even) */
  int rope_axes;      /* 3 (t, h, w) or 1 (t) */
  int rope_dims[3];   /* rotary width per axis, in dims (even); their sum is rotary_dim */
  int rotary_dim;     /* R <= head_dim: NeoX rotate_half on the first R dims of each head */
  double rope_base;   /* inverse frequency base (10000) */
  int io_channels;    /* 0, or the channel count of 1x1 pre/post convolutions around the stack */
  int dtype;          /* DIT_BF16 (bf16 weights and GEMM operands, fp32 residual) | DIT_FP32 */
  int max_tokens;     /* capacity: largest n_tokens a forward may pass */
  int max_docs;       /* capacity: largest n_docs a forward may pass */
  /* The video-VAE ViT3D decoder block ([H3] "Update: video-VAE decoder block ported"): */
  int qk_norm;         /* 1: per-head RMS norm of q and k over head_dim, no affine, eps = norm_eps,
                          before RoPE */
  int qkv_interleaved; /* 1: w_qkv / b_qkv rows per head [q_h | k_h | v_h] (the ViT's
                          qkv.view(S, H, 3 Dh).chunk(3)); repacked at bind.  0: [q_all | k_all | v_all] */
  int final_norm;      /* without AdaLN, the final norm: 0 the blocks' norm, 1 RMSNorm, 2 LayerNorm */
  /* Operand precision of a DIT_BF16 model.  The weights are bf16 values; the tensor cores take both
   * operands in one 16-bit type.  act_bf16 = 0 (the default): f16 operands.  Each weight is copied to
   * f16 at bind (exact for magnitudes 2^-17 .. 65504; a larger one makes bind return DIT_ERR_RANGE)
   * and the norm outputs, q, k, v, the attention probabilities and output, and the FFN hidden state
   * are rounded to f16: 2^-11 relative instead of bf16's 2^-8, at the same tensor-core rate.  With
   * bf16 rounding the block outputs of the full-width models (d = 3072, F = 8192 and up) miss the
   * bf16 stream's 3e-3 x RMS tolerance; with f16 they meet it.  A norm output or FFN hidden value
   * beyond 65504 sets the status word to DIT_ERR_RANGE.  act_bf16 = 1: bf16 operands throughout
   * (bf16's range, coarser rounding). */
  int act_bf16;
  /* 1: the four linear maps of every block (qkv, out, FFN up, FFN down) have NVFP4 weights, bound
   * with dit_bind_nvfp4 ([H3] "What this push adds": the NVFP4 checkpoint's projections); the
   * weights' matrices in dit_bind_weights are then ignored (may be NULL), their biases used.  Needs
   * DIT_BF16 with act_bf16 = 0 (the GEMMs take f16 activations) and qkv_interleaved = 0. */
  int nvfp4;
} dit_config;

/* One block's weights (device pointers; matrices and biases in cfg.dtype, biases may be NULL = zero;
 * gains, shifts and residual scales always fp32).
 *   w_qkv  [3d, d]   fused rows in the order [q_all | k_all | v_all], heads contiguous
 *                    ([H3] "Update: video-VAE decoder block ported": the DiT's fused qkv order)
 *   w_o    [d, d]
 *   w_in   [2F, d]   rows 0..F-1 the value, rows F..2F-1 the gate ([M3] "Correctness")
 *   w_down [d, F]
 *   w_ada  [n_mod * 6d, t_embed_dim]  per modality six d-wide chunks:
 *          shift1, scale1, gate1, shift2, scale2, gate2           (adaln = 1 only)
 *   ln1_g/ln1_b/ln2_g/ln2_b [d]  the two norms' gains / shifts (LayerNorm; RMSNorm takes the gains,
 *                                the ViT's rms_norm affine); NULL = none
 *   res1/res2 [d]                per-channel residual scales without AdaLN: x += res1 * attention
 *                                branch, x += res2 * FFN branch (NULL = 1) */
typedef struct {
  const void *w_qkv, *b_qkv, *w_o, *b_o, *w_in, *b_in, *w_down, *b_down;
  const void *w_ada, *b_ada;
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
  const void *res1, *res2;
} dit_block_weights;

/* All weights.  `blocks` is a HOST array of n_blocks entries (read during the call only).
 *   w_ada_final [n_mod * 2d, t_embed_dim]: shift_f, scale_f        (adaln = 1)
 *   lnf_g, lnf_b [d]                                                 (LayerNorm)
 *   w_pre [d, io], w_post [io, d] with biases b_pre [d], b_post [io] (io_channels > 0) */
typedef struct {
  int n_blocks;
  const dit_block_weights* blocks;
  const void *w_ada_final, *b_ada_final;
  const void *lnf_g, *lnf_b;
  const void *w_pre, *b_pre, *w_post, *b_post;
} dit_weights;

typedef struct {
  int64_t forwards;             /* dit_forward calls that launched work */
  int64_t kernels_launched;     /* every kernel this handle launched */
  int64_t gemm_launches, attention_launches, norm_launches, other_launches;
  int64_t attention_tiles;      /* (query tile, head) work items of the last forward (device count), tiles of
                                   dit_attention_block_rows() rows */
  int64_t bound_bytes;          /* bytes of library-owned repacked weight copies */
  int32_t device_status;        /* last status word read back (0 = ok) */
  int32_t last_layout_error;    /* device validator's code for the last forward (0 = ok) */
} dit_stats;

typedef struct dit_handle dit_handle;

/* ---------------------------------------------------------------------------------------------
 * Model-level calls
 * ------------------------------------------------------------------------------------------- */

/* Validate `cfg` and create a handle.  No device memory is allocated here.  What the kernels tile:
 *   DIT_BF16: RMSNorm blocks, with modality AdaLN or without it (the ViT3D decoder block: qk_norm,
 *     qkv_interleaved, final_norm, RMS gains and residual scales); hidden a multiple of 256 with
 *     hidden / 128 in {1..6, 8, 10, 12, 16, 20, 24, 32, 40, 48, 64}; head_dim 64 or 128;
 *     ffn_hidden a multiple of 128; rotary_dim / 2 a multiple of 8 and head_dim - rotary_dim a
 *     multiple of 16; t_embed_dim a multiple of 8 (of 256 above 256); io_channels 0.
 *   DIT_FP32 (the music DiT, [M3] "What moved"): RMSNorm or LayerNorm blocks without AdaLN,
 *     head_dim 64 or 128, any even rotary_dim <= head_dim (partial rotary), hidden a multiple of 128
 *     (a width the norm kernel tiles), ffn_hidden a multiple of 64, and io_channels 0 or a multiple
 *     of 128 (1x1 pre/post convolutions around the stack).
 * Anything else returns DIT_ERR_CONFIG (not a valid model) or DIT_ERR_UNSUPPORTED (valid, not
 * tiled), dit_last_error(NULL) naming the field. */
DIT_API dit_status dit_create(const dit_config* cfg, dit_handle** out);

/* NVFP4 weights of one linear map [N, K] ([H3] "What this push adds"): q [N][K/2] E2M1 codes two
 * per byte (even k in the low nibble), s [N][K/16] E4M3 scales (one per 16 along K), g the fp32
 * global scale; the weight is code * scale * g.  Device pointers. */
typedef struct {
  const uint8_t* q;
  const uint8_t* s;
  float g;
} dit_nvfp4_linear;
typedef struct {
  dit_nvfp4_linear qkv;   /* [3d, d] in the order [q_all | k_all | v_all] */
  dit_nvfp4_linear o;     /* [d, d] */
  dit_nvfp4_linear in;    /* [2F, d]: value rows, then gate rows */
  dit_nvfp4_linear down;  /* [d, F] */
} dit_nvfp4_block;

/* Bind the NVFP4 linear maps of a handle created with nvfp4 = 1 (blocks: HOST array of n_blocks
 * entries; the device arrays are read during the call only).  Each weight is repacked once into
 * the library's tile-contiguous layout (N * K * 9 / 16 bytes, library-owned; the FFN up rows
 * interleaved for the SiLU-gate epilogue), and the forward's four GEMMs of every block read it,
 * expanding codes * scales to f16 in shared memory for the tensor cores.  Call after
 * dit_bind_weights (which binds the biases, AdaLN and norms); a forward before both returns
 * DIT_ERR_UNBOUND.  A NULL code or scale pointer returns DIT_ERR_MISSING_WEIGHT naming it.
 * Synchronises `stream`. */
DIT_API dit_status dit_bind_nvfp4(dit_handle* h, const dit_nvfp4_block* blocks, void* stream);

/* Release the handle and its repacked weight copies (synchronises the device first). */
DIT_API dit_status dit_destroy(dit_handle* h);

/* Message for the last error on this handle (h may be NULL for dit_create's error). */
DIT_API const char* dit_last_error(const dit_handle* h);

/* Bytes of caller-provided device workspace a forward of n_tokens tokens in n_docs documents needs
 * (activations, cos/sin cache, tile schedule, status word).  0 when cfg is invalid. */
DIT_API size_t dit_workspace_bytes(const dit_config* cfg, int n_tokens, int n_docs);

/* Bind the weights once ([M3] "Speed": staged once, never per forward).  Non-owning: the caller's
 * tensors must stay alive and unchanged while the handle is used.  The library makes these
 * repacked copies on the device (enqueued on `stream`, owned by the handle): fp32 biases, the
 * FFN up projection with value/gate rows interleaved per 128 features (the stage-time half swap of
 * [M3] "What moved"), and every block's AdaLN matrix concatenated into one.  The first NULL
 * required pointer returns DIT_ERR_MISSING_WEIGHT and dit_last_error names it ([H3] "Update:
 * quantized arms land": missing tensors are reported by name). */
DIT_API dit_status dit_bind_weights(dit_handle* h, const dit_weights* w, void* stream);

/* One DiT forward.  [H3] "The device-resident forward (W2b)": every activation stays on the
 * device; the block stack never round-trips through the host.
 *   x_tokens      fp32 [n_tokens, d] token-major (io_channels > 0: channel-major per document,
 *                 [io, len_j] blocks back to back)
 *   cu_seqlens    int32 [n_docs + 1], cu[0] = 0, strictly increasing, cu[n_docs] = n_tokens
 *   doc_ids       int32 [n_tokens], doc_ids[i] = j for cu[j] <= i < cu[j+1]
 *   modality_tags uint8 [n_tokens], < n_modalities
 *   pos_thw       fp64 [n_tokens, 3] (t, h, w) position grid ([H3] "Correctness gates")
 *   timestep      the flow time t = sigma in [0, 1]
 *   out           fp32, same layout and size as x_tokens (may not alias x_tokens)
 *   workspace     device buffer of at least dit_workspace_bytes(cfg, n_tokens, n_docs) bytes,
 *                 256-byte aligned; its contents on entry are ignored.
 * Attention is block-diagonal over cu_seqlens and non-causal ([H3] "Correctness gates":
 * DFlashBlockAttention(causal=false)); no mask tensor exists.  Asynchronous on `stream`.  The
 * device validator checks doc_ids/tags against cu_seqlens; if it rejects the layout every later
 * kernel of the forward returns early and the status word reads DIT_ERR_LAYOUT. */
DIT_API dit_status dit_forward(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                       const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw, int n_tokens,
                       float timestep, float* out, void* workspace, size_t workspace_bytes, void* stream);

/* dit_forward with one timestep per modality.  [H3] "Milestone: the whole t2va path composes end
 * to end": the joint loop runs separate sigma schedules for video (shift 12) and audio (shift 3),
 * so at one Euler step the two modalities sit at different flow times.  Every AdaLN row of
 * modality m (the per-block [m][6][d] rows and the final [m][2][d] rows) is computed from the
 * timestep embedding of timesteps[m].
 *   timesteps  host fp32 [n_modalities], each in [0, 1]; read before the call returns.
 * Every other argument, layout and error is that of dit_forward; with all timesteps equal the
 * result is bit-identical to dit_forward at that timestep.  n_modalities above 8 returns
 * DIT_ERR_UNSUPPORTED.  A handle built without AdaLN (the fp32 forward) has no timestep input:
 * timesteps[0] is range-checked and otherwise unused. */
DIT_API dit_status dit_forward_modal(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                             const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw,
                             int n_tokens, const float* timesteps, float* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Latent I/O: the steps either side of the block stack.  [H3] "What this push adds": both patch
 * projections and both output heads stay fp32 islands around the bf16 block stream.
 * ------------------------------------------------------------------------------------------- */

#define DIT_MAX_LATENT_MODALITIES 8

/* Per-modality patch projection (token features -> d) and output head (d -> token features).
 * Device pointers, fp32, row-major [out][in]; biases may be NULL (zero).
 *   width[m]    token feature width of modality m: C*pt*ph*pw for a patchified video latent,
 *               C for a packed audio latent (any width >= 1, at most 65536)
 *   w_patch[m]  [d][width[m]]     b_patch[m] [d]
 *   w_head[m]   [width[m]][d]     b_head[m]  [width[m]]
 * dit_bind_latent_io copies the weights into the library's split (tf32 hi, lo) form, padded to
 * the GEMM's tiles, and keeps its own copies of the biases: the caller's buffers may be freed
 * once the call returns.  Needs a DIT_BF16 handle with adaln = 1 and n_modalities equal to the
 * handle's (at most 8); otherwise DIT_ERR_UNSUPPORTED / DIT_ERR_INVALID_ARG.  Synchronises
 * `stream`.  Binding again replaces the previous set. */
typedef struct {
  int n_modalities;
  int width[DIT_MAX_LATENT_MODALITIES];
  const float* w_patch[DIT_MAX_LATENT_MODALITIES];
  const float* b_patch[DIT_MAX_LATENT_MODALITIES];
  const float* w_head[DIT_MAX_LATENT_MODALITIES];
  const float* b_head[DIT_MAX_LATENT_MODALITIES];
} dit_latent_io;
DIT_API dit_status dit_bind_latent_io(dit_handle* h, const dit_latent_io* io, void* stream);

/* Workspace of dit_forward_latent (the forward's, plus the final hidden state, the row maps and
 * the islands' GEMM scratch); 0 when no latent I/O is bound. */
DIT_API size_t dit_workspace_bytes_latent(const dit_handle* h, int n_tokens, int n_docs);

/* The forward between latent tokens, for one flow time per modality:
 *   x[row] = z[m][r] W_patch[m]^T + b_patch[m]   for the r-th token tagged m (packed order)
 *   out    = the forward of x (dit_forward_modal: blocks, final norm + modulate)
 *   v[m][r] = out[row] W_head[m]^T + b_head[m]
 * The projections and heads are fp32 GEMMs (3xTF32 on the tensor cores); the patch projection
 * writes straight into the fp32 residual stream, the heads read the final layer's fp32 output.
 *   z, v        HOST arrays of n_modalities DEVICE pointers: z[m] fp32 [n_rows[m]][width[m]],
 *               v[m] fp32 [n_rows[m]][width[m]] (written); either may be NULL where n_rows[m] = 0
 *   n_rows      HOST int [n_modalities]: the number of tokens tagged m; they must add up to
 *               n_tokens (else DIT_ERR_INVALID_ARG).  The device checks them against the tags:
 *               a mismatch sets the status word to DIT_ERR_LAYOUT (layout code 8) and no later
 *               kernel of the call does work.
 *   timesteps   HOST fp32 [n_modalities], each in [0, 1]
 *   workspace   at least dit_workspace_bytes_latent(h, n_tokens, n_docs) bytes, 256-byte aligned
 * The layout arguments are dit_forward's.  Asynchronous on `stream`. */
DIT_API dit_status dit_forward_latent(dit_handle* h, const float* const* z, const int* n_rows,
                              const int32_t* cu_seqlens, int n_docs, const int32_t* doc_ids,
                              const uint8_t* modality_tags, const double* pos_thw, int n_tokens,
                              const float* timesteps, float* const* v, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Latent <-> token packing, exact (values are moved, never computed).  [H3] "Correctness gates"
 * (patchify / unpatchify / audio pack / unpack, exact with a round-trip identity).
 *   latent  fp32 [C][T*pt][H*ph][W*pw] (T, H, W count patches, not latent frames or pixels)
 *   tokens  fp32 [T*H*W][C*pt*ph*pw], token (t, h, w) at row (t*H + h)*W + w; its features are
 *           the patch in (c, a, b, e) order, e fastest: the flattening of a Conv3d weight
 *           [d][C][pt][ph][pw], so the patch projection with kernel == stride is a plain linear
 *           ([H3] "Encoder complete").
 * All sizes >= 1 and C*pt*ph*pw <= 12287; device buffers that do not overlap.  The audio forms
 * move a [C][T] latent to [T][C] tokens and back (a 1x1x1 patch on an H = W = 1 latent). */
DIT_API dit_status dit_patchify(const float* latent, int C, int T, int H, int W, int pt, int ph, int pw,
                        float* tokens, void* stream);
DIT_API dit_status dit_unpatchify(const float* tokens, int C, int T, int H, int W, int pt, int ph, int pw,
                          float* latent, void* stream);
DIT_API dit_status dit_audio_pack(const float* latent, int C, int T, float* tokens, void* stream);
DIT_API dit_status dit_audio_unpack(const float* tokens, int C, int T, float* latent, void* stream);

/* RotaryEmbeddingND positions of the video-VAE decoder, for a T x H x W token grid (w fastest):
 * pos[(t*H + h)*W + w] = (p(t, T), p(h, H), p(w, W)), p(i, n) = (2 * ((i + 0.5) / n) - 1) * 2 pi,
 * in double.  [H3] "Update: video-VAE ViT3D decoder complete": length-normalised ids mapped into
 * [-1, 1), scaled by 2 pi.  With rope_axes 3, rope_base 100 (rope_theta) and rope_dims splitting
 * rotary_dim = 0.75 * head_dim over the axes, dit_forward's cos/sin cache then holds that RoPE's
 * angles.  Host only; pos HOST [T*H*W][3]. */
DIT_API dit_status dit_vit_positions(int T, int H, int W, double* pos);

/* The same forward from HOST buffers: copies the inputs in (cudaMemcpyAsync, one per array),
 * runs dit_forward and copies `out_host` back, all on `stream`, then synchronises the stream.
 * Use pinned host memory for full copy speed.  workspace must hold
 * dit_workspace_bytes_host(cfg, n_tokens, n_docs) bytes (forward workspace + staging). */
DIT_API size_t dit_workspace_bytes_host(const dit_config* cfg, int n_tokens, int n_docs);
DIT_API dit_status dit_forward_host(dit_handle* h, const float* x_host, const int32_t* cu_host, int n_docs,
                            const int32_t* doc_ids_host, const uint8_t* tags_host, const double* pos_host,
                            int n_tokens, float timestep, float* out_host, void* workspace,
                            size_t workspace_bytes, void* stream);

/* One Euler-ancestral (eta = 0) step of the rectified flow, in place on x, fp32, in this exact
 * order with no fused multiply-add ([H3] "Correctness gates": euler-ancestral eta0 scheduler +
 * rf_v_to_x0, gated exact):
 *   x0 = x - sigma * v;   x <- x0 + (sigma_next * (x - x0)) / sigma
 * x, v: fp32 [n] device.  sigma must be > 0.  Bit-identical to the same IEEE fp32 sequence on a
 * CPU.  Stateless: resuming a loop at step k with the saved x gives the uninterrupted result. */
DIT_API dit_status dit_euler_step(float* x, const float* v, int64_t n, float sigma, float sigma_next, void* stream);

/* dit_euler_step with each token's own modality schedule: row r of x [n_tokens][d] takes the
 * pair (sigma[tags[r]], sigma_next[tags[r]]) and the same fp32 operation order, so every row is
 * bit-identical to dit_euler_step on that row with that pair.  [H3] "Milestone: the whole t2va
 * path composes end to end" (separate video and audio schedules in one packed sequence).
 *   x, v        fp32 [n_tokens][d] device; x updated in place
 *   tags        uint8 [n_tokens] device; a row whose tag is >= n_modalities is left unchanged
 *   sigma, sigma_next  HOST fp32 [n_modalities]; every sigma must be > 0
 *   n_modalities in [1, 8].  Returns DIT_ERR_INVALID_ARG on a bad argument, before any launch. */
DIT_API dit_status dit_euler_step_modal(float* x, const float* v, int n_tokens, int d, const uint8_t* tags,
                                const float* sigma, const float* sigma_next, int n_modalities, void* stream);

/* The rectified-flow time shift of one sigma, s * sigma / (1 + (s - 1) * sigma), evaluated in
 * double and rounded to fp32.  [H3] "Milestone: the whole t2va path composes end to end" names
 * the shifts (video 12, audio 3); the pages give no formula, and this is the usual one for
 * sigma in [0, 1] (shift 1 is the identity; sigma 0 and 1 are fixed points).  Host only. */
DIT_API float dit_time_shift(float sigma, float shift);

/* Counters (asserted by the tests) and the device status word.  dit_sync_status synchronises
 * `stream`, reads the status word of `workspace` (the one the last forward used) and returns it
 * as a dit_status. */
DIT_API dit_status dit_get_stats(const dit_handle* h, dit_stats* out);
DIT_API dit_status dit_sync_status(dit_handle* h, const void* workspace, void* stream);

/* Failure-path self-test of the bounded waits.  Launches one kernel that waits on an mbarrier
 * nothing ever arrives at, through the same bounded wait the GEMM and attention pipelines use, with
 * a limit of limit_ns (0 < limit_ns <= 1e9).  The wait runs out, the kernel records the timeout in
 * *status_word (a caller-owned device int) and returns; the call synchronises `stream` and returns
 * DIT_ERR_DEVICE_TIMEOUT when that happened (DIT_OK would mean the wait ended some other way).  No
 * trap, no fault: the context stays usable for the next call. */
DIT_API dit_status dit_selftest_wait_timeout(uint64_t limit_ns, int* status_word, void* stream);

/* Per-block dumps for parity tests: when `dump` is non-NULL each later forward copies the fp32
 * residual after block l into dump + l * n_tokens * d (device, caller-owned, L * N * d floats). */
DIT_API dit_status dit_set_dump(dit_handle* h, float* dump);

/* Per-kernel-kind timing with CUDA events recorded on the forward's stream around every launch.
 * enable = 1 starts collecting (events are created lazily); dit_get_kernel_times synchronises and
 * returns, per kind, the summed milliseconds and launch count since the last reset.
 * Kinds: 0 gemm_qkv, 1 attention, 2 gemm_out, 3 gemm_ffn_up, 4 gemm_ffn_down, 5 norm_modulate,
 *        6 other (schedule, cos/sin cache, AdaLN, copies),
 *        7 latent_io (row maps, patch projections and output heads of dit_forward_latent). */
#define DIT_KERNEL_KINDS 8
DIT_API dit_status dit_set_kernel_timing(dit_handle* h, int enable);
DIT_API dit_status dit_get_kernel_times(dit_handle* h, double* ms_out, int64_t* launches_out);

/* ---------------------------------------------------------------------------------------------
 * Op-level calls: each runs one kernel of the forward on caller buffers, for parity testing and
 * for composing the forward differently.  Shapes and layouts are those the forward uses.
 * ------------------------------------------------------------------------------------------- */

/* Norm + indexed AdaLN modulate ([H3] "The device-resident forward (W2b)"):
 *   y[r] = N(x[r]) * (1 + scale[tag[r]]) + shift[tag[r]]
 * N = RMSNorm x / sqrt(mean(x^2) + eps) (norm = DIT_RMSNORM) or LayerNorm (DIT_LAYERNORM), either
 * followed by the per-channel gain ln_g and shift ln_b when given (NULL = none).  x fp32 [n, d]; shift/scale fp32 rows of d values, row m at
 * shift + m * mod_stride (NULL shift and scale = no modulation); tags uint8 [n] (may be NULL
 * when shift is NULL).  Output bf16 [n, d] (out_kind 0), fp32 [n, d] (1) or f16 [n, d] (2).
 * Requires d % 128 == 0 and d <= 8192. */
DIT_API dit_status dit_op_norm_modulate(const float* x, int n, int d, int norm, float eps, const float* ln_g,
                                const float* ln_b, const uint8_t* tags, const float* shift, const float* scale,
                                int64_t mod_stride, void* y, int out_kind, void* stream);

/* Per-row RoPE cos/sin cache from the fp64 grid ([BF] "What this enables": BuildRopeCosSin;
 * [H3] "The device-resident forward (W2b)": a per-row cos/sin cache fed from three axes of the
 * fp64 position grid).  inv[k] of axis a = (float) base^(-2k/dims[a]); theta = pos[r][axis] * inv
 * in fp64; cos/sin in fp64, stored fp32 [n, rotary_dim/2] with the axis blocks concatenated. */
DIT_API dit_status dit_op_rope_cache(const double* pos, int n, int n_axes, const int* dims_host, double base,
                             float* cos_out, float* sin_out, void* stream);

/* AdaLN conditioning: e = [cos(1000 t f_k) | sin(1000 t f_k)], f_k = exp(-ln(1e4) k / (t_dim/2));
 * mod[r] = W[r] . silu(e) + b[r] for r < rows.  W bf16 bits [rows, t_dim], b fp32 [rows] or NULL,
 * mod fp32 [rows].  t_dim % 256 == 0 or t_dim in {64, 128}. */
DIT_API dit_status dit_op_adaln(const void* w, const float* b, int rows, int t_dim, float t, float* mod, void* stream);

/* GEMM D = A B^T on the tcgen05 tensor cores, 16-bit operands, fp32 accumulation in TMEM.
 * A [M, K] row-major, B [N, K] row-major (the weight), both of the 16-bit type `elem`
 * (DIT_ELEM_BF16 or DIT_ELEM_F16), bias fp32 [N] or NULL.
 * M >= 1 any; N % 256 == 0; K % 64 == 0; A, B 16-byte aligned.  Epilogues:
 *   dit_op_gemm            out = A B^T + bias, stored bf16 (out_kind 0), fp32 (1) or f16 (2), [M, N]
 *   dit_op_gemm_qkv_rope   N = 3d: q, k get bias + NeoX rotate_half with cos/sin [M, R/2] on the
 *                          first R dims of each Dh-wide head and are stored as `elem` [M, d]; v is
 *                          stored TRANSPOSED, vt [d, n_pad] (vt[c * n_pad + row]) of type `elem`,
 *                          n_pad >= M, n_pad % 8 == 0; the padding columns [M, n_pad) are
 *                          written as zeros.
 *   dit_op_gemm_gated_residual  x[M, N] (fp32, in place) += gate[tag[r]] * (A B^T + bias);
 *                          gate rows at gate + m * gate_stride (NULL gate = plain residual add).
 *   dit_op_gemm_swiglu     B, bias in the interleaved layout of dit_op_pack_ffn_in (2F rows);
 *                          h [M, F] of type `elem` = (u + b_u) * silu(g + b_g). */
DIT_API dit_status dit_op_gemm(const void* a, const void* b, const float* bias, int M, int N, int K, void* out, int out_kind,
                       int elem, void* stream);
DIT_API dit_status dit_op_gemm_qkv_rope(const void* a, const void* b, const float* bias, int M, int d, int K, int n_heads,
                                int head_dim, int rotary_dim, const float* cos_cache, const float* sin_cache,
                                void* q, void* k, void* vt, int n_pad, int elem, void* stream);
DIT_API dit_status dit_op_gemm_gated_residual(const void* a, const void* b, const float* bias, int M, int N, int K,
                                      float* x, const float* gate, int64_t gate_stride, const uint8_t* tags,
                                      int elem, void* stream);
DIT_API dit_status dit_op_gemm_swiglu(const void* a, const void* b_packed, const float* bias_packed, int M, int F, int K,
                              void* h, int elem, void* stream);

/* GEMM with NVFP4 weights.  [H3] "What this push adds": the NVFP4 checkpoint's projections carry
 * a U8 weight with two FP4 (E2M1) codes per byte ([N][K/2]), an F8_E4M3 scale per group of 16
 * along K ([N][K/16]) and an F32 global scale; the logical weight is code * scale * global (even
 * k in the low nibble).  dit_op_pack_nvfp4 repacks q and s once into the tile-contiguous layout
 * the kernel streams (dit_nvfp4_packed_bytes(N, K) = N*K*9/16 bytes, 16-byte aligned).
 * dit_op_gemm_nvfp4 computes out = A W^T + bias with A f16 [M, K] (every code * scale product
 * is exact in f16, so the tensor cores run f16 x f16 with fp32 accumulation; the global scale
 * multiplies the accumulator).  out_kind 0 bf16, 1 fp32, 2 f16, [M, N].  N % 256 == 0,
 * K % 64 == 0, A 16-byte aligned; else DIT_ERR_INVALID_ARG before any launch. */
DIT_API size_t dit_nvfp4_packed_bytes(int N, int K);
DIT_API dit_status dit_op_pack_nvfp4(const uint8_t* q, const uint8_t* scales, int N, int K, void* packed,
                             void* stream);
DIT_API dit_status dit_op_gemm_nvfp4(const void* a_f16, const void* packed, float w_scale, const float* bias, int M,
                             int N, int K, void* out, int out_kind, void* stream);

/* fp32 GEMM y = x w^T + bias exactly as the fp32 forward computes its linear maps ([M3] "What
 * moved": every Linear is a MatmulBT with a rank-1 bias add; fp32 stays fp32): 3xTF32 on the
 * tcgen05 tensor cores (each operand split into tf32 hi + lo parts, three tf32 products per fp32
 * product, 32-deep accumulation chunks summed in fp32), split-K partial sums reduced in a fixed order.
 *   x fp32 [M, K] row-major, w fp32 [N, K] row-major, bias fp32 [N] or NULL, y fp32 [M, N] (written).
 *   M >= 1; N % 128 == 0; K % 32 == 0; x, w, y 16-byte aligned.
 *   workspace: device scratch of dit_gemm_f32_workspace_bytes(M, N, K) bytes, caller-owned (the hi/lo
 *   splits of x and w and the partial sums); not retained after the call's device work.
 *   Results are deterministic; calls on one stream are ordered.  Errors: DIT_ERR_INVALID_ARG for bad
 *   shapes or pointers (nothing launched), DIT_ERR_CUDA when a launch fails. */
DIT_API size_t dit_gemm_f32_workspace_bytes(int M, int N, int K);
DIT_API dit_status dit_op_gemm_f32(const float* x, const float* w, const float* bias, int M, int N, int K, float* y,
                           void* workspace, void* stream);

/* Interleave an FFN up projection [2F, d] (value rows then gate rows) into 128-feature groups:
 * packed rows [256 g, 256 g + 128) = value rows [128 g, +128), the next 128 = the gate rows
 * [F + 128 g, +128).  bias (fp32 [2F] or NULL) is interleaved the same way into bias_packed
 * (fp32 [2F]; zeros when bias is NULL).  F % 128 == 0. */
DIT_API dit_status dit_op_pack_ffn_in(const void* w_in, const float* b_in, int F, int d, void* w_packed, float* b_packed,
                              void* stream);

/* Varlen non-causal flash attention on the tcgen05 tensor cores ([H3] "Correctness gates":
 * DFlashBlockAttention(causal=false) over the packed sequence; [M3] "What moved": non-causal,
 * no bias).  Per document [cu[j], cu[j+1]) and head h:  o_i = softmax_j(q_i . k_j / sqrt(Dh)) v_j.
 * Every 16-bit array is of the type `elem` (DIT_ELEM_BF16 or DIT_ELEM_F16); the probabilities
 * take the same type as the PV operand.
 *   q, k  [n_tokens, H * Dh];  vt [H * Dh, n_pad] (n_pad % 8 == 0, n_pad >= n_tokens; its padding
 *         columns are never read into a result)
 * Key/value tiles are 128 tokens wide and 128-aligned, so a document's boundary tiles also load its
 * neighbours' keys and values: their scores are replaced by -inf and their V^T columns by zeros
 * before they are used, so every document's output is bit-independent of the other documents'
 * values, non-finite ones included.
 *   o     [n_tokens, H * Dh]
 * head_dim is 64 or 128.  The (document, query tile) work list is built on the device from
 * cu_seqlens into `workspace` (dit_attention_workspace_bytes(n_docs, n_tokens) bytes). */
DIT_API size_t dit_attention_workspace_bytes(int n_docs, int n_tokens);
/* Query rows per (document, query tile) work item of the attention: the unit of
 * dit_stats.attention_tiles. */
DIT_API int dit_attention_block_rows(void);
DIT_API dit_status dit_op_attention(const void* q, const void* k, const void* vt, int n_pad, const int32_t* cu_seqlens,
                            int n_docs, int n_tokens, int n_heads, int head_dim, void* o, void* workspace,
                            int elem, void* stream);

/* The same attention with no caller-provided scratch, for callers that cannot allocate device
 * memory: e.g. a plugin running inside another framework's executor that is handed no allocator, or
 * a latency-critical serving thread that cannot afford cudaMalloc's implicit device synchronisation.
 * The pages have no counterpart of this call; it exists for such callers only.
 *   Arguments, layouts and results are those of dit_op_attention, without `workspace`.
 *   Scratch: a fixed array inside libdit.so's device memory (256 bytes of status words plus
 *   DIT_ATTENTION_NOALLOC_MAX_TILES (document, 128-row q-tile) entries of 8 bytes, about 64 KB),
 *   held by every GPU that loads the library until the process exits.  Nothing is allocated or freed.
 *   Capacity: ceil(n_tokens / 128) + n_docs <= DIT_ATTENTION_NOALLOC_MAX_TILES, else
 *   DIT_ERR_CAPACITY with dit_last_error(NULL) saying so, before any work is enqueued.
 *   Errors found on the device: cu_seqlens is checked on the device, as in dit_op_attention; a
 *   rejected layout leaves `o` unwritten and the call still returns DIT_OK (the work is
 *   asynchronous).  dit_op_attention_noalloc_status reads the outcome back.
 *   Set-up: the first call in each CUDA context (per device; again after cudaDeviceReset) looks up
 *   the array's device address (cudaGetSymbolAddress) and caches it for that context; make that
 *   first call before any stream capture.
 *   Sharing: all calls use the same array, which keeps the last call's contents (the status words
 *   are cleared at the start of each call).  Calls whose device work overlaps (other streams, other
 *   host threads on the same device) race on it: serialise them. */
#define DIT_ATTENTION_NOALLOC_MAX_TILES 8192
DIT_API dit_status dit_op_attention_noalloc(const void* q, const void* k, const void* vt, int n_pad,
                                            const int32_t* cu_seqlens, int n_docs, int n_tokens, int n_heads,
                                            int head_dim, void* o, int elem, void* stream);

/* Outcome of the last dit_op_attention_noalloc call in the current context: synchronises `stream`,
 * reads the fixed array's status words (no allocation) and returns DIT_OK, DIT_ERR_LAYOUT
 * (cu_seqlens rejected; *layout_code, when layout_code is not NULL, gets the validator's code:
 * 1 no documents, 2 cu[0] != 0, 3 not strictly increasing, 4 cu[n_docs] != n_tokens),
 * DIT_ERR_DEVICE_TIMEOUT (a bounded wait ran out) or DIT_ERR_CUDA.  Shares the array, so it reads
 * whichever call's device work finished last. */
DIT_API dit_status dit_op_attention_noalloc_status(int* layout_code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DIT_H_ */
