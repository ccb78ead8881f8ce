// Internal launcher interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dit {

// Opt `func` into `bytes` of dynamic shared memory on the current device.  The attribute is per
// device, so the cache is a bitmask of the devices (0-63) already set, one mask per kernel.
inline cudaError_t opt_in_smem(const void* func, int bytes, unsigned long long* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return e;
}

// Epilogue kinds of the tcgen05 GEMM engine.
enum GemmEpilogue : int {
  kEpiStore = 0,        // out = acc + bias (bf16 or fp32)
  kEpiQkvRope = 1,      // q, k: + bias, NeoX RoPE, bf16 [M, d]; v: + bias, bf16 transposed [d, n_pad]
  kEpiGatedResid = 2,   // x += gate[tag] * (acc + bias), fp32 in place
  kEpiSwiglu = 3,       // h = (u + b_u) * silu(g + b_g), interleaved 128-feature groups, bf16 [M, F]
};

struct GemmArgs {
  int M, N, K;
  int f16 = 0;             // A, B and the 16-bit outputs of kEpiQkvRope / kEpiSwiglu are f16 (1) or bf16 (0)
  const float* bias;       // [N] or nullptr
  // kEpiStore
  void* out;
  int out_kind;            // 0 bf16, 1 fp32, 2 f16
  // kEpiQkvRope
  int d, head_dim, rot_half;
  int qk_norm;             // 1: per-head RMS norm of q and k (no affine) before the rotation
  float qk_eps;
  const float* cos_cache;  // [M, rot_half]
  const float* sin_cache;
  void* q;
  void* k;
  void* vt;
  int n_pad;
  // kEpiGatedResid
  float* x;
  const float* gate;
  long long gate_stride;
  const uint8_t* tags;
  // common
  int* status;             // device status word (may be null)
  int group_n;             // N-blocks per raster group (L2 reuse of B)
  // NVFP4 weights (gemm_nvfp4_launch): B is the tile-contiguous repack of nvfp4_pack_launch, A f16;
  // every epilogue takes acc * w_scale (the weight's global scale) in place of acc
  const uint8_t* b_packed = nullptr;
  float w_scale = 1.f;
};

// Launch D = A B^T with the given epilogue.  A bf16 [M, K], B bf16 [N, K].  Returns a CUDA error.
cudaError_t gemm_launch(int epilogue, const void* A, const void* B, const GemmArgs& args, cudaStream_t stream);
// The same with NVFP4 weights: A f16 [M, K]; B from args.b_packed (N % 256 == 0, K % 64 == 0).
cudaError_t gemm_nvfp4_launch(int epilogue, const void* A, const GemmArgs& args, cudaStream_t stream);
// NVFP4 weight repack: q [N][K/2] (two E2M1 per byte, even k low), s [N][K/16] (E4M3) ->
// [N/256][K/64] tiles of 9216 bytes: 256 rows x 32 bytes of codes, then 256 rows x 4 scales.
constexpr int kNvfp4TileBytes = 9216;
// ffn_F > 0 interleaves the rows of an FFN up projection [2F, K] into 128-feature value/gate groups.
cudaError_t nvfp4_pack_launch(const uint8_t* q, const uint8_t* s, int N, int K, uint8_t* packed, cudaStream_t st,
                              int ffn_F = 0);

// Attention: q, k bf16 [N, H*Dh], vt bf16 [H*Dh, n_pad], o bf16 [N, H*Dh].  `items` is the
// device tile list built by attention_schedule_launch (int2 {doc, q_start}), `count` its length.
struct AttnArgs {
  int n_tokens, n_heads, head_dim, n_pad, n_docs;
  const int32_t* cu;
  const int2* items;
  const int* count;
  int max_items;
  float scale_log2;   // log2(e) / sqrt(Dh)
  int* status;
  int f16 = 0;        // q, k, vt, P and o are f16 (1) or bf16 (0)
};
cudaError_t attention_launch(const void* q, const void* k, const void* vt, void* o, const AttnArgs& args,
                             cudaStream_t stream);

// Validates cu_seqlens (and doc_ids / tags when given) and writes the (doc, q_start) list of
// attention_item_rows()-row query tiles, longest documents first.  On a bad layout sets kDevLayout
// in *status and writes count = 0.
cudaError_t attention_schedule_launch(const int32_t* cu, int n_docs, int n_tokens, const int32_t* doc_ids,
                                      const uint8_t* tags, int n_mod, int2* items, int* count, int max_items,
                                      int* layout_code, int* status, cudaStream_t stream);
// A bound on the list length: ceil(n_tokens / 128) + n_docs.
int attention_max_items(int n_docs, int n_tokens);
int attention_item_rows();

// Elementwise / reduction kernels.
// out_kind: 0 bf16, 1 fp32, 2 f16 (values beyond f16's finite range set kDevRange in *status),
// 3 the 3xF16 GEMM's operand: f16 hi and lo parts of y * 2^kF16x3ActExp in the token-tiled layout of
// x3_xs_index (token tile x3_token_tile(n)).
cudaError_t norm_modulate_launch(const float* x, const float* x_lo, int n, int d, int norm, float eps, const float* ln_g,
                                 const float* ln_b, const uint8_t* tags, const float* shift, const float* scale,
                                 long long mod_stride, void* y, int out_kind, int* status, cudaStream_t s);
cudaError_t rope_cache_launch(const double* pos, int n, int n_axes, const int* dims, double base, float* cos_out,
                              float* sin_out, const int* status, cudaStream_t s);
// Timesteps of the AdaLN conditioning: one for every row (n_t = 1), or one per modality (n_t =
// n_mod <= kMaxModalTimesteps), the row's modality following the concatenated layout: L blocks of
// [n_mod][6d] rows (mod_block = n_mod * 6d rows each, block_rows = L * mod_block in all), then the
// final [n_mod][2d].
constexpr int kMaxModalTimesteps = 8;
struct AdaTimesteps {
  float t[kMaxModalTimesteps];
  int n_t, six_d, two_d, mod_block, block_rows;
};
cudaError_t adaln_launch(const void* w, const float* b, int rows, int t_dim, const AdaTimesteps& ts, float* mod,
                         const int* status, cudaStream_t s);
// Per-modality sigma pairs of the tagged Euler step (n_mod <= kMaxModalTimesteps).
struct ModalSigmas {
  float sigma[kMaxModalTimesteps];
  float sigma_next[kMaxModalTimesteps];
  int n;  // pairs in use; a row whose tag is >= n is left unchanged
};
cudaError_t euler_tagged_launch(float* x, const float* v, int n_tokens, int d, const uint8_t* tags,
                                const ModalSigmas& sg, cudaStream_t s);
cudaError_t euler_launch(float* x, const float* v, long long n, float sigma, float sigma_next, cudaStream_t s);
// Latent <-> token packing (inverse = 0: latent [C][T*pt][H*ph][W*pw] -> tokens [T*H*W][C*pt*ph*pw]).
cudaError_t patch_launch(const float* src, float* dst, int C, int T, int H, int W, int pt, int ph, int pw,
                         int inverse, cudaStream_t s);
// Per-modality row lists from the tags: rows[off[m] + k] = the k-th token tagged m, k < count[m].
struct ModalRows {
  int n;
  int count[kMaxModalTimesteps];
  int off[kMaxModalTimesteps];
};
cudaError_t row_map_launch(const uint8_t* tags, int n, const ModalRows& mr, int* rows, int* layout_code, int* status,
                           cudaStream_t s);
// Rows of the per-head interleaved qkv order [q_h | k_h | v_h] into [q_all | k_all | v_all].
cudaError_t qkv_deinterleave_launch(const void* src, void* dst, int H, int Dh, int row_bytes, cudaStream_t s);
cudaError_t pack_ffn_in_launch(const void* w_in, const float* b_in, int F, int d, void* w_packed, float* b_packed,
                               cudaStream_t s);
cudaError_t to_f32_launch(const void* src, int src_is_bf16, long long n, float* dst, cudaStream_t s);
// bf16 -> f16 (round to nearest even; exact for |v| >= 2^-17 and <= 65504); *flag |= kDevRange when a
// value is beyond f16's finite range.  src and dst may be the same buffer.
cudaError_t bf16_to_f16_launch(const void* src, void* dst, long long n, int* flag, cudaStream_t s);

int num_sms();
bool norm_width_supported(int d);
cudaError_t wait_timeout_selftest_launch(int* status, unsigned long long limit_ns, cudaStream_t s);

// fp32 path (csrc/fp32.cu): split-K 3xTF32 tensor-core GEMM D = X W^T (X [M, K], W [N, K], fp32 given
// as tf32 (hi, lo) pairs, N % 128 == 0, K % 32 == 0) into partials [S][M][N], then fixed-order
// reductions that apply the epilogues.
constexpr int kSgemmMaxSplits = 16;
int tf32x3_splits(int M, int N, int K);
int tf32x3_effective_splits(int K, int S);
cudaError_t tf32x3_partial_launch(const float* x_hi, const float* x_lo, const float* w_hi, const float* w_lo, int M,
                                  int N, int K, int S, float* part, const int* status, cudaStream_t s);
cudaError_t tf32_split_launch(const float* x, size_t n, float* hi, float* lo, cudaStream_t s);
// The 3xF16 GEMM (the fp32 forward's linear maps): operands as f16 (hi, lo) parts of x 2^e, K a
// multiple of kF16x3K, N a multiple of kTf32x3N; the partial sums are scaled back by 2^-(w_exp + x_exp).
constexpr int kF16x3K = 64;
constexpr int kF16x3ActExp = 4;  // the activations' fixed scale exponent
int f16x3_splits(int M, int N, int K);
int f16x3_effective_splits(int K, int S);
// With w_tiled, W is the bind-time weight-tile layout of f16_split_launch (kSplitWeightTiles; w_lo is
// unused); with x_tiled, x_hi is the token-tiled operand of x3_xs_index (x_lo unused).  Otherwise both
// are row-major [rows][K] hi and lo arrays.
cudaError_t f16x3_partial_launch(const uint16_t* x_hi, const uint16_t* x_lo, const uint16_t* w_hi,
                                 const uint16_t* w_lo, const int* w_exp, int x_exp, int M, int N, int K, int S,
                                 float* part, const int* status, cudaStream_t s, int w_tiled = 0, int x_tiled = 0);
// Largest |x| (as float bits) into *out (cleared first).
cudaError_t absmax_launch(const float* x, size_t n, unsigned int* out, cudaStream_t s);
// x [M][K] (stride ldx) -> f16 hi, lo parts of x 2^e, zero-padded to Kp columns: e from *max_bits (a
// weight's scale, also written to *e_out) when max_bits is given, else e_fixed; kDevRange in *status
// past 65504.  Layouts: kSplitRows, hi and lo [M][Kp]; kSplitWeightTiles, 128 x 32 tiles [M / 128][Kp /
// 32], each tile's hi part (4096 elements) followed by its lo part, pre-swizzled for the 64-byte
// swizzle (pass lo = hi + 4096); kSplitTokenTiles, the layout of x3_xs_index (lo unused).
enum F16SplitLayout : int { kSplitRows = 0, kSplitWeightTiles = 1, kSplitTokenTiles = 2 };
cudaError_t f16_split_launch(const float* x, long long ldx, int K, int M, int Kp, const unsigned int* max_bits,
                             int e_fixed, int* e_out, uint16_t* hi, uint16_t* lo, int* status, cudaStream_t s,
                             int layout = kSplitRows);
// The 3xTF32 GEMM's tiling: K a multiple of kTf32x3K, N (output features) a multiple of kTf32x3N.
constexpr int kTf32x3K = 32;
constexpr int kTf32x3N = 128;
// Split of rows (rows ? rows[r] : r) of x (stride ldx, K columns) into [M][Kp] hi/lo, zero-padded.
cudaError_t tf32_split_rows_launch(const float* x, long long ldx, int K, const int* rows, int M, int Kp, float* hi,
                                   float* lo, const int* status, cudaStream_t s);
// out[(rows ? rows[r] : r) * ld_out + n] = sum of the S partials [S][M][Np] + bias[n], for n < n_out.
cudaError_t sgemm_reduce_rows_launch(const float* part, int S, int M, int Np, int n_out, const float* bias,
                                     const int* rows, float* out, long long ld_out, const int* status,
                                     cudaStream_t s);
cudaError_t sgemm_reduce_store_launch(const float* part, int S, int M, int N, const float* bias, float* out, int add,
                                      float* lo, const int* status, cudaStream_t s);
// The residual-stream reduction fused with the norm that reads the stream next (d % 1024 == 0,
// d <= 8192): resid (+)= sum of the S partials + bias (compensated with resid_lo; add = 0 stores),
// then y = norm(resid + resid_lo) * g + b as out_kind 1 (fp32) or 3 (the 3xF16 operand).
bool reduce_norm_fusable(int d);
cudaError_t sgemm_reduce_resid_norm_launch(const float* part, int S, int M, int d, const float* bias, float* resid,
                                           float* resid_lo, int add, int norm, float eps, const float* g,
                                           const float* b, void* y, int out_kind, int* status, cudaStream_t s);
cudaError_t sgemm_reduce_qkv_launch(const float* part, int S, int M, int d, int Dh, int half, const float* bias,
                                    const float* cs, const float* sn, float* q, float* k, float* v, const int* status,
                                    cudaStream_t s);
// h_split: when given, h is written as the 3xF16 GEMM's token-tiled operand (x3_xs_index) of
// h * 2^kF16x3ActExp instead of fp32 into h.
cudaError_t sgemm_reduce_swiglu_launch(const float* part, int S, int M, int F, const float* bias, float* h,
                                       uint16_t* h_split, int* status, cudaStream_t s);
// Exact fp32 attention over the (document, 128-row q-tile) list of attention_schedule_launch.
// o_split: when given, o is written as the 3xF16 GEMM's token-tiled operand (x3_xs_index, n_tokens
// rows) of o * 2^kF16x3ActExp instead of fp32 into o.
cudaError_t attention_f32_launch(const float* q, const float* k, const float* v, const int32_t* cu, const int2* items,
                                 const int* count, int max_items, int n_tokens, int H, int Dh, float* o,
                                 uint16_t* o_split, int* status, cudaStream_t s);
cudaError_t io_transpose_launch(const float* src, float* dst, const int32_t* cu, const int32_t* doc_ids, int n, int io,
                                int to_frames, const int* status, cudaStream_t s);

}  // namespace dit
