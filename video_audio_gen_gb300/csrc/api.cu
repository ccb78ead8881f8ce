// C ABI of libdit.so (declared in include/dit.h): handle, validation, bind-time weight repacks,
// workspace layout and the orchestration of one DiT forward on a caller stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dit.h"
#include "common.cuh"
#include "kernels.h"

using namespace dit;

namespace {

thread_local std::string g_create_error;

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// An fp32 weight as the 3xTF32 GEMM reads it: tf32(w) and tf32(w - tf32(w)), library-owned.
struct SplitW {
  float* hi = nullptr;
  float* lo = nullptr;
};

// An fp32 weight as the 3xF16 GEMM reads it: f16 (hi, lo) parts of W 2^e and the exponent e (device).
struct SplitW16 {
  uint16_t* hi = nullptr;
  uint16_t* lo = nullptr;
  int* e = nullptr;
};

struct BlockDev {
  SplitW16 s_qkv, s_o, s_in, s_down;  // fp32 path
  const void* w_qkv = nullptr;
  const void* w_o = nullptr;
  const void* w_down = nullptr;
  const void* w_in = nullptr;      // fp32 path: value rows then gate rows, used as bound
  float* ln1_g = nullptr;          // fp32 path, LayerNorm gains / shifts (NULL = none)
  float* ln1_b = nullptr;
  float* ln2_g = nullptr;
  float* ln2_b = nullptr;
  void* w_in_packed = nullptr;
  float* b_qkv = nullptr;
  float* b_o = nullptr;
  float* b_in_packed = nullptr;
  float* b_down = nullptr;
  // NVFP4 linear maps (nvfp4 = 1): tile-contiguous repacks and global scales
  uint8_t *nv_qkv = nullptr, *nv_o = nullptr, *nv_in = nullptr, *nv_down = nullptr;
  float g_qkv = 1.f, g_o = 1.f, g_in = 1.f, g_down = 1.f;
  float* res1 = nullptr;           // per-channel residual scales without AdaLN (NULL = 1)
  float* res2 = nullptr;
};

// Workspace layout of one forward (offsets in bytes from the workspace base).
struct WsLayout {
  size_t status, items, mod, cosc, sinc, resid, y, q, k, vt, o, h, part = 0, resid_lo = 0, xs_hi = 0, xs_lo = 0,
      total;
  int n_pad, max_items, half, mod_rows;
};

struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};

}  // namespace

struct dit_handle {
  dit_config cfg;
  bool bound = false;
  bool nvfp4_bound = false;
  std::string err;
  std::vector<void*> allocs;
  std::vector<BlockDev> blocks;
  void* w_ada_all = nullptr;   // bf16 [ada_rows, t_dim]: L blocks x [n_mod * 6d], then final [n_mod * 2d]
  float* b_ada_all = nullptr;  // fp32 [ada_rows]
  int ada_rows = 0;
  // fp32 path: final LayerNorm and the 1x1 pre/post convolutions
  float *lnf_g = nullptr, *lnf_b = nullptr, *b_pre = nullptr, *b_post = nullptr;
  const float *w_pre = nullptr, *w_post = nullptr;
  SplitW16 s_pre, s_post;  // fp32 path: the 1x1 convolutions' weights split for the 3xF16 GEMM
  // latent I/O (dit_bind_latent_io): per modality the patch projection [d][kp] and the output head
  // [np][d] split for the 3xTF32 GEMM, zero-padded to the GEMM's K chunk and N tile
  int lat_n = 0;
  int lat_width[kMaxModalTimesteps] = {}, lat_kp[kMaxModalTimesteps] = {}, lat_np[kMaxModalTimesteps] = {};
  SplitW lat_patch[kMaxModalTimesteps], lat_head[kMaxModalTimesteps];
  float* lat_b_patch[kMaxModalTimesteps] = {};
  float* lat_b_head[kMaxModalTimesteps] = {};
  float* dump = nullptr;
  dit_stats stats;
  bool timing = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_next = 0;
  std::vector<TimedLaunch> timed;
  double ms_acc[DIT_KERNEL_KINDS];
  int64_t n_acc[DIT_KERNEL_KINDS];
};

namespace {

dit_status set_err(dit_handle* h, dit_status st, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
dit_status set_err(dit_handle* h, dit_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h)
    h->err = buf;
  else
    g_create_error = buf;
  return st;
}

dit_status cuda_err(dit_handle* h, cudaError_t e, const char* what) {
  return set_err(h, DIT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DIT_CK(h, call, what)                            \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_err((h), e_, (what)); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

dit_status validate_config(const dit_config* c) {
  if (!c) return set_err(nullptr, DIT_ERR_INVALID_ARG, "config is NULL");
  if (c->n_blocks < 1) return set_err(nullptr, DIT_ERR_CONFIG, "n_blocks must be >= 1");
  if (c->hidden < 1 || c->n_heads < 1 || c->head_dim < 1 || c->n_heads * c->head_dim != c->hidden)
    return set_err(nullptr, DIT_ERR_CONFIG, "hidden must equal n_heads * head_dim");
  if (c->ffn_hidden < 1) return set_err(nullptr, DIT_ERR_CONFIG, "ffn_hidden must be >= 1");
  if (c->norm != DIT_RMSNORM && c->norm != DIT_LAYERNORM) return set_err(nullptr, DIT_ERR_CONFIG, "bad norm");
  if (!(c->norm_eps > 0.f)) return set_err(nullptr, DIT_ERR_CONFIG, "norm_eps must be > 0");
  if (c->adaln != 0 && c->adaln != 1) return set_err(nullptr, DIT_ERR_CONFIG, "adaln must be 0 or 1");
  if (c->adaln && (c->n_modalities < 1 || c->n_modalities > 255))
    return set_err(nullptr, DIT_ERR_CONFIG, "n_modalities must be in [1, 255]");
  if (c->adaln && (c->t_embed_dim < 8 || c->t_embed_dim % 8 || (c->t_embed_dim > 256 && c->t_embed_dim % 256)))
    return set_err(nullptr, DIT_ERR_CONFIG, "t_embed_dim must be a multiple of 8 (and of 256 above 256)");
  if (c->rope_axes != 1 && c->rope_axes != 3) return set_err(nullptr, DIT_ERR_CONFIG, "rope_axes must be 1 or 3");
  int rsum = 0;
  for (int a = 0; a < c->rope_axes; ++a) {
    if (c->rope_dims[a] < 0 || c->rope_dims[a] % 2) return set_err(nullptr, DIT_ERR_CONFIG, "rope_dims must be even");
    rsum += c->rope_dims[a];
  }
  if (rsum != c->rotary_dim || c->rotary_dim > c->head_dim || c->rotary_dim < 0)
    return set_err(nullptr, DIT_ERR_CONFIG, "rotary_dim must equal sum(rope_dims) and be <= head_dim");
  if (!(c->rope_base > 1.0)) return set_err(nullptr, DIT_ERR_CONFIG, "rope_base must be > 1");
  if (c->io_channels < 0) return set_err(nullptr, DIT_ERR_CONFIG, "io_channels must be >= 0");
  if (c->max_tokens < 1 || c->max_docs < 1) return set_err(nullptr, DIT_ERR_CONFIG, "max_tokens/max_docs must be >= 1");
  if (c->dtype != DIT_BF16 && c->dtype != DIT_FP32) return set_err(nullptr, DIT_ERR_CONFIG, "bad dtype");
  if ((c->qk_norm != 0 && c->qk_norm != 1) || (c->qkv_interleaved != 0 && c->qkv_interleaved != 1))
    return set_err(nullptr, DIT_ERR_CONFIG, "qk_norm and qkv_interleaved must be 0 or 1");
  if (c->final_norm < 0 || c->final_norm > 2) return set_err(nullptr, DIT_ERR_CONFIG, "final_norm must be 0, 1 or 2");
  if (c->act_bf16 != 0 && c->act_bf16 != 1) return set_err(nullptr, DIT_ERR_CONFIG, "act_bf16 must be 0 or 1");
  if (c->nvfp4 != 0 && c->nvfp4 != 1) return set_err(nullptr, DIT_ERR_CONFIG, "nvfp4 must be 0 or 1");
  if (c->nvfp4 && (c->dtype != DIT_BF16 || c->act_bf16 || c->qkv_interleaved))
    return set_err(nullptr, DIT_ERR_UNSUPPORTED, "nvfp4 needs dtype DIT_BF16, act_bf16 = 0 and qkv_interleaved = 0");
  if (c->adaln && c->final_norm)
    return set_err(nullptr, DIT_ERR_CONFIG, "with AdaLN the final layer is RMSNorm + modulate (final_norm must be 0)");
  // What the sm_103a kernels tile.
  if (c->head_dim != 128 && c->head_dim != 64)
    return set_err(nullptr, DIT_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!norm_width_supported(c->hidden)) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "hidden width not tiled by the norm kernel");
  if (c->dtype == DIT_FP32) {
    if (c->adaln) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "the fp32 forward has no AdaLN (adaln must be 0)");
    if (c->qk_norm || c->qkv_interleaved || c->final_norm)
      return set_err(nullptr, DIT_ERR_UNSUPPORTED, "qk_norm / qkv_interleaved / final_norm need the bf16 forward");
    if (c->hidden % 128) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "fp32: hidden must be a multiple of 128");
    if (c->ffn_hidden % 64) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "fp32: ffn_hidden must be a multiple of 64");
    if (c->io_channels % 128) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "fp32: io_channels must be 0 or a multiple of 128");
    return DIT_OK;
  }
  if (c->hidden % 256) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "hidden must be a multiple of 256");
  if ((c->rotary_dim / 2) % 8 || (c->head_dim - c->rotary_dim) % 16)
    return set_err(nullptr, DIT_ERR_UNSUPPORTED, "rotary_dim/2 must be a multiple of 8 and head_dim-rotary_dim of 16");
  if (c->ffn_hidden % 128) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "ffn_hidden must be a multiple of 128");
  if (c->io_channels) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "pre/post convolutions need the fp32 forward");
  if (c->norm == DIT_LAYERNORM) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "LayerNorm blocks need the fp32 forward");
  return DIT_OK;
}

WsLayout ws_layout_fp32(const dit_config* c, int n, int n_docs);

WsLayout ws_layout(const dit_config* c, int n, int n_docs) {
  if (c->dtype == DIT_FP32) return ws_layout_fp32(c, n, n_docs);
  WsLayout w;
  const int d = c->hidden, F = c->ffn_hidden;
  w.n_pad = (n + 7) & ~7;
  w.max_items = attention_max_items(n_docs, n);
  w.half = c->rotary_dim / 2;
  w.mod_rows = c->adaln ? c->n_blocks * c->n_modalities * 6 * d + c->n_modalities * 2 * d : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  w.status = take(64);
  w.items = take((size_t)w.max_items * sizeof(int2));
  w.mod = take((size_t)w.mod_rows * 4);
  w.cosc = take((size_t)n * w.half * 4);
  w.sinc = take((size_t)n * w.half * 4);
  w.resid = take((size_t)n * d * 4);
  w.y = take((size_t)n * d * 2);
  w.q = take((size_t)n * d * 2);
  w.k = take((size_t)n * d * 2);
  w.vt = take((size_t)d * w.n_pad * 2);
  w.o = take((size_t)n * d * 2);
  w.h = take((size_t)n * F * 2);
  w.total = off;
  return w;
}

// fp32 forward: fp32 activations, split-K partial sums, frame-major staging for the 1x1 convolutions.
// Reuses WsLayout's fields: q/k hold fp32 q, k; vt holds fp32 v [N, d]; h fp32 [N, F]; mod the
// frame-major staging [N, io]; items the split-K partial buffer.
WsLayout ws_layout_fp32(const dit_config* c, int n, int n_docs) {
  WsLayout w;
  const int d = c->hidden, F = c->ffn_hidden, io = c->io_channels;
  w.n_pad = (n + 7) & ~7;
  w.max_items = attention_max_items(n_docs, n);
  w.half = c->rotary_dim / 2;
  w.mod_rows = 0;
  size_t widest = (size_t)3 * d;
  if ((size_t)2 * F > widest) widest = (size_t)2 * F;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  w.status = take(64);
  w.items = take((size_t)w.max_items * sizeof(int2));
  w.cosc = take((size_t)n * w.half * 4);
  w.sinc = take((size_t)n * w.half * 4);
  w.resid = take((size_t)n * d * 4);
  w.y = take((size_t)n * d * 4);
  w.q = take((size_t)n * d * 4);
  w.k = take((size_t)n * d * 4);
  w.vt = take((size_t)n * d * 4);
  w.o = take((size_t)n * d * 4);
  w.h = take((size_t)n * F * 4);
  w.mod = take((size_t)n * (io ? io : 1) * 4);
  w.part = take((size_t)kSgemmMaxSplits * n * widest * 4);
  w.resid_lo = take((size_t)n * d * 4);
  size_t widest_in = (size_t)d;  // the GEMM inputs: io (pre-conv), d, F (FFN down)
  if ((size_t)F > widest_in) widest_in = (size_t)F;
  if ((size_t)io > widest_in) widest_in = (size_t)io;
  // the 3xF16 operand: rows padded to whole token tiles, hi and lo parts
  const int x_nt = x3_token_tile(n > 0 ? n : 1);
  const size_t n_pad = (size_t)((n + x_nt - 1) / x_nt) * x_nt;
  w.xs_hi = take(n_pad * widest_in * 4);
  w.xs_lo = take((size_t)n * widest_in * 4);
  w.total = off;
  return w;
}

// status word layout at ws + status: [0] device status bits, [1] layout code, [2] attention item count
struct StatusWords {
  int bits, layout_code, count, pad;
};

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

void* dev_alloc(dit_handle* h, size_t bytes, cudaError_t* e) {
  void* p = nullptr;
  *e = cudaMalloc(&p, bytes ? bytes : 16);
  if (*e == cudaSuccess) {
    h->allocs.push_back(p);
    h->stats.bound_bytes += (int64_t)bytes;
  }
  return p;
}

cudaEvent_t next_event(dit_handle* h) {
  if (h->ev_next >= h->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->ev_pool.push_back(e);
  }
  return h->ev_pool[h->ev_next++];
}

// Record-around helper: kind < 0 means untimed.
struct Launch {
  dit_handle* h;
  cudaStream_t s;
  int kind;
  cudaEvent_t a = nullptr;
  Launch(dit_handle* h_, cudaStream_t s_, int k) : h(h_), s(s_), kind(k) {
    if (h && h->timing) {
      a = next_event(h);
      if (a) cudaEventRecord(a, s);
    }
  }
  // n: the kernels launched in this group (the stats count kernels)
  void done(int n = 1) {
    if (h && h->timing && a) {
      cudaEvent_t b = next_event(h);
      if (b) {
        cudaEventRecord(b, s);
        h->timed.push_back({kind, a, b});
      }
    }
    if (h) {
      h->stats.kernels_launched += n;
      if (kind == 0 || kind == 2 || kind == 3 || kind == 4) h->stats.gemm_launches += n;
      else if (kind == 1) h->stats.attention_launches += n;
      else if (kind == 5) h->stats.norm_launches += n;
      else h->stats.other_launches += n;
    }
  }
};


// ------------------------------------------------------------------------------------------------
// fp32 path (the music DiT shape): bind and forward
// ------------------------------------------------------------------------------------------------
dit_status bind_fp32(dit_handle* h, const dit_weights* w, cudaStream_t s) {
  const dit_config& c = h->cfg;
  const int d = c.hidden, F = c.ffn_hidden, io = c.io_channels;
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_block_weights& b = w->blocks[l];
    const struct {
      const void* p;
      const char* name;
    } req[] = {{b.w_qkv, "w_qkv"}, {b.w_o, "w_o"}, {b.w_in, "w_in"}, {b.w_down, "w_down"}};
    for (const auto& r : req) {
      if (!r.p) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: blocks[%d].%s", l, r.name);
      if (!aligned16(r.p)) return set_err(h, DIT_ERR_INVALID_ARG, "blocks[%d].%s is not 16-byte aligned", l, r.name);
    }
  }
  if (io && !w->w_pre) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: w_pre");
  if (io && !w->w_post) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: w_post");
  cudaStreamSynchronize(s);
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  h->blocks.assign(c.n_blocks, BlockDev());
  h->stats.bound_bytes = 0;
  h->bound = false;
  cudaError_t e = cudaSuccess;
  // fp32 copies of the small vectors (NULL stays NULL for LayerNorm parameters: no affine)
  auto vec = [&](const void* src, long long n, bool zero_if_null) -> float* {
    if (!src && !zero_if_null) return nullptr;
    float* dst = static_cast<float*>(dev_alloc(h, n * 4, &e));
    if (e != cudaSuccess) return nullptr;
    e = src ? to_f32_launch(src, 0, n, dst, s) : cudaMemsetAsync(dst, 0, n * 4, s);
    return e == cudaSuccess ? dst : nullptr;
  };
  // f16 (hi, lo) copies of every fp32 linear weight [rows, K] scaled by its own power of two, read by
  // the 3xF16 GEMM: 4 bytes per weight, as the fp32 weight itself
  unsigned int* maxbuf = static_cast<unsigned int*>(dev_alloc(h, 16, &e));
  if (e != cudaSuccess) return cuda_err(h, e, "bind: alloc");
  // (128 x 32 tiles, each tile's hi part followed by its lo part, in the GEMM's shared-memory image)
  auto split = [&](const void* src, long long rows, int K, SplitW16* out) -> bool {
    const size_t n = (size_t)rows * K;
    out->hi = static_cast<uint16_t*>(dev_alloc(h, n * 4, &e));
    if (e == cudaSuccess) out->lo = out->hi + (size_t)kTf32x3N * kTf32x3K;
    if (e == cudaSuccess) out->e = static_cast<int*>(dev_alloc(h, 16, &e));
    if (e == cudaSuccess) e = absmax_launch(static_cast<const float*>(src), n, maxbuf, s);
    if (e == cudaSuccess)
      e = f16_split_launch(static_cast<const float*>(src), K, K, (int)rows, K, maxbuf, 0, out->e, out->hi, out->lo,
                           nullptr, s, kSplitWeightTiles);
    return e == cudaSuccess;
  };
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_block_weights& b = w->blocks[l];
    BlockDev& bd = h->blocks[l];
    if (!split(b.w_qkv, 3ll * d, d, &bd.s_qkv) || !split(b.w_o, d, d, &bd.s_o) ||
        !split(b.w_in, 2ll * F, d, &bd.s_in) || !split(b.w_down, d, F, &bd.s_down))
      return cuda_err(h, e, "bind: split fp32 weights");
    bd.w_qkv = b.w_qkv;
    bd.w_o = b.w_o;
    bd.w_in = b.w_in;
    bd.w_down = b.w_down;
    if (!(bd.b_qkv = vec(b.b_qkv, 3ll * d, true))) return cuda_err(h, e, "bind b_qkv");
    if (!(bd.b_o = vec(b.b_o, d, true))) return cuda_err(h, e, "bind b_o");
    if (!(bd.b_in_packed = vec(b.b_in, 2ll * F, true))) return cuda_err(h, e, "bind b_in");
    if (!(bd.b_down = vec(b.b_down, d, true))) return cuda_err(h, e, "bind b_down");
    bd.ln1_g = vec(b.ln1_g, d, false);
    bd.ln1_b = vec(b.ln1_b, d, false);
    bd.ln2_g = vec(b.ln2_g, d, false);
    bd.ln2_b = vec(b.ln2_b, d, false);
    if (e != cudaSuccess) return cuda_err(h, e, "bind layer norm");
  }
  h->lnf_g = vec(w->lnf_g, d, false);
  h->lnf_b = vec(w->lnf_b, d, false);
  if (io) {
    h->w_pre = static_cast<const float*>(w->w_pre);
    h->w_post = static_cast<const float*>(w->w_post);
    if (!split(w->w_pre, d, io, &h->s_pre) || !split(w->w_post, io, d, &h->s_post))
      return cuda_err(h, e, "bind: split conv weights");
    h->b_pre = vec(w->b_pre, d, true);
    h->b_post = vec(w->b_post, io, true);
  }
  if (e != cudaSuccess) return cuda_err(h, e, "bind final / io weights");
  DIT_CK(h, cudaStreamSynchronize(s), "bind sync");
  h->bound = true;
  return DIT_OK;
}

// One fp32 GEMM of the forward: the 3xF16 partial sums of the activation operand in `xs` (f16 hi and
// lo parts of x 2^kF16x3ActExp in the token-tiled layout), then (by the caller) the fixed-order
// reduction that applies the epilogue.  The operand is written by the kernel that produces x (the norms, the
// attention, the SiLU-gate reduction); `run` splits an fp32 x first (the 1x1 convolutions' inputs).
struct Sgemm {
  dit_handle* h;
  cudaStream_t s;
  float* part;
  uint16_t* xs;
  int* status;
  int S;  // effective splits of the last partial launch
  cudaError_t run_split(const SplitW16& W, int M, int N, int K) {
    const int want = f16x3_splits(M, N, K);
    S = f16x3_effective_splits(K, want);
    return f16x3_partial_launch(xs, nullptr, W.hi, nullptr, W.e, kF16x3ActExp, M, N, K, want, part, status, s, 1,
                                1);
  }
  cudaError_t run(const float* X, const SplitW16& W, int M, int N, int K) {
    cudaError_t e =
        f16_split_launch(X, K, K, M, K, nullptr, kF16x3ActExp, nullptr, xs, nullptr, status, s, kSplitTokenTiles);
    return e == cudaSuccess ? run_split(W, M, N, K) : e;
  }
};

dit_status forward_fp32(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                        const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw, int N,
                        float* out, void* workspace, const WsLayout& L, cudaStream_t s) {
  const dit_config& c = h->cfg;
  const int d = c.hidden, F = c.ffn_hidden, H = c.n_heads, io = c.io_channels;
  StatusWords* sw = at<StatusWords>(workspace, L.status);
  int* status = &sw->bits;
  int2* items = at<int2>(workspace, L.items);
  float* cosc = at<float>(workspace, L.cosc);
  float* sinc = at<float>(workspace, L.sinc);
  float* resid = at<float>(workspace, L.resid);
  float* resid_lo = at<float>(workspace, L.resid_lo);
  float* y = at<float>(workspace, L.y);
  float* q = at<float>(workspace, L.q);
  float* k = at<float>(workspace, L.k);
  float* v = at<float>(workspace, L.vt);
  float* xt = at<float>(workspace, L.mod);
  Sgemm g{h, s, at<float>(workspace, L.part), at<uint16_t>(workspace, L.xs_hi), status, 1};
  {
    Launch ln(h, s, 6);
    DIT_CK(h, cudaMemsetAsync(sw, 0, sizeof(StatusWords), s), "status reset");
    DIT_CK(h, attention_schedule_launch(cu_seqlens, n_docs, N, doc_ids, modality_tags, 1, items, &sw->count,
                                        L.max_items, &sw->layout_code, status, s), "layout check");
    ln.done();
  }
  if (L.half > 0) {
    Launch ln(h, s, 6);
    DIT_CK(h, rope_cache_launch(pos_thw, N, c.rope_axes, c.rope_dims, c.rope_base, cosc, sinc, status, s), "rope cache");
    ln.done();
  }
  // The reductions that add into the residual stream are fused with the norm that reads it next
  // (one kernel instead of two) when the width allows it.
  const bool fuse = reduce_norm_fusable(d) && c.n_blocks > 0;
  bool norm1_done = false;  // block l's norm1 was written by the previous fused reduction
  if (io) {
    // 1x1 pre-convolution as MatmulBT on the frame-major activation ([M3] "What moved")
    Launch ln(h, s, 6);
    DIT_CK(h, io_transpose_launch(x_tokens, xt, cu_seqlens, doc_ids, N, io, 1, status, s), "to frames");
    DIT_CK(h, g.run(xt, h->s_pre, N, d, io), "pre-conv");
    if (fuse) {
      DIT_CK(h, sgemm_reduce_resid_norm_launch(g.part, g.S, N, d, h->b_pre, resid, resid_lo, 0, c.norm, c.norm_eps,
                                               h->blocks[0].ln1_g, h->blocks[0].ln1_b, g.xs, 3, status, s),
             "pre-conv reduce + norm1");
      norm1_done = true;
    } else {
      DIT_CK(h, sgemm_reduce_store_launch(g.part, g.S, N, d, h->b_pre, resid, 0, resid_lo, status, s),
             "pre-conv reduce");
    }
    ln.done(4);
  } else {
    DIT_CK(h, cudaMemcpyAsync(resid, x_tokens, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, s), "copy x");
    DIT_CK(h, cudaMemsetAsync(resid_lo, 0, (size_t)N * d * 4, s), "clear residual low part");
  }
  for (int l = 0; l < c.n_blocks; ++l) {
    const BlockDev& B = h->blocks[l];
    const bool last = l + 1 == c.n_blocks;
    if (!norm1_done) {
      Launch ln(h, s, 5);
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, B.ln1_g, B.ln1_b, nullptr, nullptr,
                                     nullptr, 0, g.xs, 3, status, s), "norm1");
      ln.done();
    }
    {
      Launch ln(h, s, 0);
      DIT_CK(h, g.run_split(B.s_qkv, N, 3 * d, d), "qkv");
      DIT_CK(h, sgemm_reduce_qkv_launch(g.part, g.S, N, d, c.head_dim, L.half, B.b_qkv, cosc, sinc, q, k, v, status, s),
             "qkv reduce");
      ln.done(2);
    }
    {
      Launch ln(h, s, 1);
      DIT_CK(h, attention_f32_launch(q, k, v, cu_seqlens, items, &sw->count, L.max_items, N, H, c.head_dim, nullptr,
                                     g.xs, status, s), "attention");
      ln.done();
    }
    {
      Launch ln(h, s, 2);
      DIT_CK(h, g.run_split(B.s_o, N, d, d), "out-proj");
      if (fuse)
        DIT_CK(h, sgemm_reduce_resid_norm_launch(g.part, g.S, N, d, B.b_o, resid, resid_lo, 1, c.norm, c.norm_eps,
                                                 B.ln2_g, B.ln2_b, g.xs, 3, status, s),
               "out-proj reduce + norm2");
      else
        DIT_CK(h, sgemm_reduce_store_launch(g.part, g.S, N, d, B.b_o, resid, 1, resid_lo, status, s),
               "out-proj reduce");
      ln.done(2);
    }
    if (!fuse) {
      Launch ln(h, s, 5);
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, B.ln2_g, B.ln2_b, nullptr, nullptr,
                                     nullptr, 0, g.xs, 3, status, s), "norm2");
      ln.done();
    }
    {
      Launch ln(h, s, 3);
      DIT_CK(h, g.run_split(B.s_in, N, 2 * F, d), "ffn up");
      DIT_CK(h, sgemm_reduce_swiglu_launch(g.part, g.S, N, F, B.b_in_packed, nullptr, g.xs, status, s),
             "ffn up reduce");
      ln.done(2);
    }
    {
      Launch ln(h, s, 4);
      DIT_CK(h, g.run_split(B.s_down, N, d, F), "ffn down");
      if (fuse) {
        // the next block's norm1, or after the last block the final norm
        const float* ng = last ? h->lnf_g : h->blocks[l + 1].ln1_g;
        const float* nb = last ? h->lnf_b : h->blocks[l + 1].ln1_b;
        DIT_CK(h, sgemm_reduce_resid_norm_launch(g.part, g.S, N, d, B.b_down, resid, resid_lo, 1, c.norm, c.norm_eps,
                                                 ng, nb, last ? (io ? static_cast<void*>(y) : out) : g.xs,
                                                 last ? 1 : 3, status, s),
               "ffn down reduce + norm");
        norm1_done = true;
      } else {
        DIT_CK(h, sgemm_reduce_store_launch(g.part, g.S, N, d, B.b_down, resid, 1, resid_lo, status, s),
               "ffn down reduce");
      }
      ln.done(2);
    }
    if (h->dump)
      DIT_CK(h, cudaMemcpyAsync(h->dump + (size_t)l * N * d, resid, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, s),
             "dump");
  }
  if (!fuse) {
    Launch ln(h, s, 5);
    DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, h->lnf_g, h->lnf_b, nullptr, nullptr, nullptr, 0,
                                   io ? y : out, 1, status, s), "final norm");
    ln.done();
  }
  if (io) {
    Launch ln(h, s, 6);
    DIT_CK(h, g.run(y, h->s_post, N, io, d), "post-conv");
    DIT_CK(h, sgemm_reduce_store_launch(g.part, g.S, N, io, h->b_post, xt, 0, nullptr, status, s), "post-conv reduce");
    DIT_CK(h, io_transpose_launch(xt, out, cu_seqlens, doc_ids, N, io, 0, status, s), "to channels");
    ln.done(4);
  }
  h->stats.forwards++;
  return DIT_OK;
}

}  // namespace

extern "C" {

const char* dit_last_error(const dit_handle* h) { return h ? h->err.c_str() : g_create_error.c_str(); }

dit_status dit_create(const dit_config* cfg, dit_handle** out) {
  if (!out) return set_err(nullptr, DIT_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  dit_status st = validate_config(cfg);
  if (st != DIT_OK) return st;
  dit_handle* h = new dit_handle();
  h->cfg = *cfg;
  memset(&h->stats, 0, sizeof h->stats);
  memset(h->ms_acc, 0, sizeof h->ms_acc);
  memset(h->n_acc, 0, sizeof h->n_acc);
  *out = h;
  g_create_error.clear();
  return DIT_OK;
}

dit_status dit_destroy(dit_handle* h) {
  if (!h) return DIT_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  for (void* p : h->allocs) cudaFree(p);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  delete h;
  return DIT_OK;
}

size_t dit_workspace_bytes(const dit_config* cfg, int n_tokens, int n_docs) {
  if (validate_config(cfg) != DIT_OK || n_tokens < 1 || n_docs < 1) return 0;
  return ws_layout(cfg, n_tokens, n_docs).total;
}

dit_status dit_bind_weights(dit_handle* h, const dit_weights* w, void* stream) {
  if (!h) return DIT_ERR_INVALID_ARG;
  if (!w || !w->blocks) return set_err(h, DIT_ERR_INVALID_ARG, "weights or weights->blocks is NULL");
  const dit_config& c = h->cfg;
  if (w->n_blocks != c.n_blocks)
    return set_err(h, DIT_ERR_INVALID_ARG, "weights.n_blocks %d != config n_blocks %d", w->n_blocks, c.n_blocks);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.dtype == DIT_FP32) return bind_fp32(h, w, s);
  const int d = c.hidden, F = c.ffn_hidden, nm = c.n_modalities, td = c.t_embed_dim;
  // Missing tensors are reported by name before anything is allocated.
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_block_weights& b = w->blocks[l];
    // with NVFP4 linear maps the four matrices come from dit_bind_nvfp4
    const bool lin = !c.nvfp4;
    const struct {
      const void* p;
      const char* name;
      bool need;
    } req[] = {{b.w_qkv, "w_qkv", lin}, {b.w_o, "w_o", lin}, {b.w_in, "w_in", lin}, {b.w_down, "w_down", lin},
               {b.w_ada, "w_ada", c.adaln != 0}};
    for (const auto& r : req) {
      if (!r.need) continue;
      if (!r.p) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: blocks[%d].%s", l, r.name);
      if (!aligned16(r.p)) return set_err(h, DIT_ERR_INVALID_ARG, "blocks[%d].%s is not 16-byte aligned", l, r.name);
    }
  }
  if (c.adaln && !w->w_ada_final) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: w_ada_final");

  // Free a previous binding.
  cudaStreamSynchronize(s);
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  h->blocks.assign(c.n_blocks, BlockDev());
  h->stats.bound_bytes = 0;
  h->bound = false;
  h->nvfp4_bound = false;

  cudaError_t e;
  const int is_bf16 = c.dtype == DIT_BF16;
  auto bias_f32 = [&](const void* src, long long n) -> float* {
    float* dst = static_cast<float*>(dev_alloc(h, n * 4, &e));
    if (e != cudaSuccess) return nullptr;
    if (src)
      e = to_f32_launch(src, is_bf16, n, dst, s);
    else
      e = cudaMemsetAsync(dst, 0, n * 4, s);
    return e == cudaSuccess ? dst : nullptr;
  };
  // fp32 vectors (gains, shifts, residual scales): library-owned copies, NULL stays NULL
  auto vec32 = [&](const void* src, long long n) -> float* {
    if (!src) return nullptr;
    float* dst = static_cast<float*>(dev_alloc(h, n * 4, &e));
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToDevice, s);
    return dst;
  };
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_block_weights& b = w->blocks[l];
    BlockDev& bd = h->blocks[l];
    bd.w_qkv = b.w_qkv;
    bd.w_o = b.w_o;
    bd.w_down = b.w_down;
    if (!(bd.b_qkv = bias_f32(b.b_qkv, 3ll * d))) return cuda_err(h, e, "bind b_qkv");
    if (c.qkv_interleaved) {
      // [q_h | k_h | v_h] per head -> the engine's [q_all | k_all | v_all]: a library-owned copy
      void* wq = dev_alloc(h, (size_t)3 * d * d * 2, &e);
      if (e != cudaSuccess) return cuda_err(h, e, "alloc w_qkv");
      DIT_CK(h, qkv_deinterleave_launch(b.w_qkv, wq, c.n_heads, c.head_dim, d * 2, s), "deinterleave w_qkv");
      float* bq = static_cast<float*>(dev_alloc(h, (size_t)3 * d * 4, &e));
      if (e != cudaSuccess) return cuda_err(h, e, "alloc b_qkv");
      DIT_CK(h, qkv_deinterleave_launch(bd.b_qkv, bq, c.n_heads, c.head_dim, 4, s), "deinterleave b_qkv");
      bd.w_qkv = wq;
      bd.b_qkv = bq;
    }
    bd.ln1_g = vec32(b.ln1_g, d);
    bd.ln1_b = vec32(b.ln1_b, d);
    bd.ln2_g = vec32(b.ln2_g, d);
    bd.ln2_b = vec32(b.ln2_b, d);
    bd.res1 = vec32(b.res1, d);
    bd.res2 = vec32(b.res2, d);
    if (e != cudaSuccess) return cuda_err(h, e, "bind gains / residual scales");
    if (!(bd.b_o = bias_f32(b.b_o, d))) return cuda_err(h, e, "bind b_o");
    if (!(bd.b_down = bias_f32(b.b_down, d))) return cuda_err(h, e, "bind b_down");
    float* b_in = nullptr;
    if (b.b_in && !(b_in = bias_f32(b.b_in, 2ll * F))) return cuda_err(h, e, "bind b_in");
    bd.w_in_packed = c.nvfp4 ? nullptr : dev_alloc(h, (size_t)2 * F * d * 2, &e);
    if (e != cudaSuccess) return cuda_err(h, e, "alloc w_in");
    bd.b_in_packed = static_cast<float*>(dev_alloc(h, (size_t)2 * F * 4, &e));
    if (e != cudaSuccess) return cuda_err(h, e, "alloc b_in");
    DIT_CK(h, pack_ffn_in_launch(c.nvfp4 ? nullptr : b.w_in, b_in, F, d, bd.w_in_packed, bd.b_in_packed, s),
           "pack w_in");
  }
  if (!c.act_bf16 && !c.nvfp4) {
    // f16 GEMM operands: the four linear maps' weights as library-owned f16 copies.  bf16 -> f16 is
    // exact for every value of magnitude 2^-17 .. 65504; a weight beyond 65504 is refused.
    int* range = static_cast<int*>(dev_alloc(h, 16, &e));
    if (e != cudaSuccess) return cuda_err(h, e, "alloc range flag");
    DIT_CK(h, cudaMemsetAsync(range, 0, 16, s), "range flag");
    auto to_f16 = [&](const void* src, long long n, bool in_place) -> const void* {
      void* dst = in_place ? const_cast<void*>(src) : dev_alloc(h, (size_t)n * 2, &e);
      if (e == cudaSuccess) e = bf16_to_f16_launch(src, dst, n, range, s);
      return dst;
    };
    for (int l = 0; l < c.n_blocks; ++l) {
      BlockDev& bd = h->blocks[l];
      bd.w_qkv = to_f16(bd.w_qkv, 3ll * d * d, c.qkv_interleaved != 0);  // the de-interleaved copy is ours
      if (e == cudaSuccess) bd.w_o = to_f16(bd.w_o, (long long)d * d, false);
      if (e == cudaSuccess) bd.w_down = to_f16(bd.w_down, (long long)d * F, false);
      if (e == cudaSuccess) to_f16(bd.w_in_packed, 2ll * F * d, true);
      if (e != cudaSuccess) return cuda_err(h, e, "bind: f16 weight copies");
    }
    int flag = 0;
    DIT_CK(h, cudaMemcpyAsync(&flag, range, sizeof flag, cudaMemcpyDeviceToHost, s), "read range flag");
    DIT_CK(h, cudaStreamSynchronize(s), "bind sync");
    if (flag & kDevRange)
      return set_err(h, DIT_ERR_RANGE, "a weight exceeds f16's range (65504); bind with act_bf16 = 1");
  }
  h->lnf_g = vec32(w->lnf_g, d);
  h->lnf_b = vec32(w->lnf_b, d);
  if (e != cudaSuccess) return cuda_err(h, e, "bind final norm");
  if (!c.adaln) {
    h->ada_rows = 0;
    DIT_CK(h, cudaStreamSynchronize(s), "bind sync");
    h->bound = true;
    return DIT_OK;
  }
  // AdaLN matrices of every block, then the final layer's, in one [rows, t_dim] matrix.
  const size_t blk_rows = (size_t)nm * 6 * d, fin_rows = (size_t)nm * 2 * d;
  h->ada_rows = (int)(c.n_blocks * blk_rows + fin_rows);
  h->w_ada_all = dev_alloc(h, (size_t)h->ada_rows * td * 2, &e);
  if (e != cudaSuccess) return cuda_err(h, e, "alloc w_ada");
  h->b_ada_all = static_cast<float*>(dev_alloc(h, (size_t)h->ada_rows * 4, &e));
  if (e != cudaSuccess) return cuda_err(h, e, "alloc b_ada");
  for (int l = 0; l < c.n_blocks; ++l) {
    DIT_CK(h, cudaMemcpyAsync(static_cast<char*>(h->w_ada_all) + (size_t)l * blk_rows * td * 2, w->blocks[l].w_ada,
                              blk_rows * td * 2, cudaMemcpyDeviceToDevice, s), "copy w_ada");
    if (w->blocks[l].b_ada)
      DIT_CK(h, to_f32_launch(w->blocks[l].b_ada, is_bf16, (long long)blk_rows, h->b_ada_all + l * blk_rows, s), "b_ada");
    else
      DIT_CK(h, cudaMemsetAsync(h->b_ada_all + l * blk_rows, 0, blk_rows * 4, s), "b_ada");
  }
  DIT_CK(h, cudaMemcpyAsync(static_cast<char*>(h->w_ada_all) + (size_t)c.n_blocks * blk_rows * td * 2, w->w_ada_final,
                            fin_rows * td * 2, cudaMemcpyDeviceToDevice, s), "copy w_ada_final");
  if (w->b_ada_final)
    DIT_CK(h, to_f32_launch(w->b_ada_final, is_bf16, (long long)fin_rows, h->b_ada_all + c.n_blocks * blk_rows, s),
           "b_ada_final");
  else
    DIT_CK(h, cudaMemsetAsync(h->b_ada_all + c.n_blocks * blk_rows, 0, fin_rows * 4, s), "b_ada_final");
  DIT_CK(h, cudaStreamSynchronize(s), "bind sync");
  h->bound = true;
  return DIT_OK;
}

dit_status dit_bind_nvfp4(dit_handle* h, const dit_nvfp4_block* blocks, void* stream) {
  if (!h) return DIT_ERR_INVALID_ARG;
  const dit_config& c = h->cfg;
  if (!c.nvfp4) return set_err(h, DIT_ERR_CONFIG, "dit_bind_nvfp4 needs a handle created with nvfp4 = 1");
  if (!h->bound) return set_err(h, DIT_ERR_UNBOUND, "dit_bind_nvfp4 before dit_bind_weights");
  if (!blocks) return set_err(h, DIT_ERR_INVALID_ARG, "blocks is NULL");
  const int d = c.hidden, F = c.ffn_hidden;
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_nvfp4_block& b = blocks[l];
    const struct {
      const dit_nvfp4_linear* w;
      const char* name;
    } lin[] = {{&b.qkv, "qkv"}, {&b.o, "o"}, {&b.in, "in"}, {&b.down, "down"}};
    for (const auto& x : lin) {
      if (!x.w->q) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: blocks[%d].%s.q", l, x.name);
      if (!x.w->s) return set_err(h, DIT_ERR_MISSING_WEIGHT, "missing weight: blocks[%d].%s.s", l, x.name);
      if (!(x.w->g > 0.f) || !isfinite(x.w->g))
        return set_err(h, DIT_ERR_INVALID_ARG, "blocks[%d].%s.g must be a finite positive scale", l, x.name);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  auto pack = [&](const dit_nvfp4_linear& w, int N, int K, int ffn_F, uint8_t** out, float* g) -> bool {
    *out = static_cast<uint8_t*>(dev_alloc(h, (size_t)N * K * 9 / 16, &e));
    if (e == cudaSuccess) e = nvfp4_pack_launch(w.q, w.s, N, K, *out, s, ffn_F);
    *g = w.g;
    return e == cudaSuccess;
  };
  for (int l = 0; l < c.n_blocks; ++l) {
    const dit_nvfp4_block& b = blocks[l];
    BlockDev& bd = h->blocks[l];
    if (!pack(b.qkv, 3 * d, d, 0, &bd.nv_qkv, &bd.g_qkv) || !pack(b.o, d, d, 0, &bd.nv_o, &bd.g_o) ||
        !pack(b.in, 2 * F, d, F, &bd.nv_in, &bd.g_in) || !pack(b.down, d, F, 0, &bd.nv_down, &bd.g_down))
      return cuda_err(h, e, "bind NVFP4 linear maps");
  }
  DIT_CK(h, cudaStreamSynchronize(s), "bind nvfp4 sync");
  h->nvfp4_bound = true;
  return DIT_OK;
}

// The latent forward's inputs and scratch, resolved on the host.
struct LatentArgs {
  const float* const* z;  // host array of device pointers, z[m] [count[m]][width[m]]
  ModalRows mr;           // row counts (the caller's) and their offsets into `rows`
  int* rows;              // device [N]: the rows of modality m at rows + off[m]
  float *xs_hi, *xs_lo, *part;
};

// Splits of an island GEMM: the 3xTF32 plan's, capped so that splits x M stays within the N rows
// the partial buffer holds.
static int island_splits(int M, int Nn, int K, int n_tokens) {
  int S = tf32x3_splits(M, Nn, K);
  const int cap = n_tokens / M > 1 ? n_tokens / M : 1;
  return S < cap ? S : cap;
}

// The patch projections: the row maps from the tags, then per modality x[rows_m] = z_m W_patch^T + b
// written straight into the fp32 residual.
static dit_status latent_embed(dit_handle* h, const LatentArgs& a, const uint8_t* tags, int N, float* resid,
                               int* layout_code, int* status, cudaStream_t s) {
  const int d = h->cfg.hidden;
  {
    Launch ln(h, s, 7);
    DIT_CK(h, row_map_launch(tags, N, a.mr, a.rows, layout_code, status, s), "row maps");
    ln.done();
  }
  for (int m = 0; m < a.mr.n; ++m) {
    const int M = a.mr.count[m];
    if (M == 0) continue;
    const int Kp = h->lat_kp[m];
    Launch ln(h, s, 7);
    DIT_CK(h, tf32_split_rows_launch(a.z[m], h->lat_width[m], h->lat_width[m], nullptr, M, Kp, a.xs_hi, a.xs_lo,
                                     status, s), "patch split");
    const int want = island_splits(M, d, Kp, N);
    DIT_CK(h, tf32x3_partial_launch(a.xs_hi, a.xs_lo, h->lat_patch[m].hi, h->lat_patch[m].lo, M, d, Kp, want, a.part,
                                    status, s), "patch projection");
    DIT_CK(h, sgemm_reduce_rows_launch(a.part, tf32x3_effective_splits(Kp, want), M, d, d, h->lat_b_patch[m],
                                       a.rows + a.mr.off[m], resid, d, status, s), "patch projection store");
    ln.done(3);
  }
  return DIT_OK;
}

// One of the forward's GEMMs: the 16-bit weight B, or its NVFP4 repack (then A is f16 and the global
// scale multiplies the accumulator in the epilogue).
static cudaError_t gemm_any(int epi, const void* A, const void* B, const uint8_t* nv, float g_scale, GemmArgs g,
                            cudaStream_t s) {
  if (!nv) return gemm_launch(epi, A, B, g, s);
  g.b_packed = nv;
  g.w_scale = g_scale;
  return gemm_nvfp4_launch(epi, A, g, s);
}

// The forward with its AdaLN timesteps: n_t = 1 (every modality at t[0]) or n_t = n_modalities.
// With `lat` the residual is filled by the patch projections instead of copied from x_tokens.
static dit_status forward_impl(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                               const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw,
                               int n_tokens, const float* t_in, int n_t, float* out, void* workspace,
                               size_t workspace_bytes, void* stream, const LatentArgs* lat = nullptr) {
  if (!h) return DIT_ERR_INVALID_ARG;
  if (!h->bound) return set_err(h, DIT_ERR_UNBOUND, "dit_forward before dit_bind_weights");
  const dit_config& c = h->cfg;
  if (c.nvfp4 && !h->nvfp4_bound) return set_err(h, DIT_ERR_UNBOUND, "nvfp4 = 1: dit_forward before dit_bind_nvfp4");
  if ((!x_tokens && !lat) || !cu_seqlens || !doc_ids || !modality_tags || !pos_thw || !out || !workspace)
    return set_err(h, DIT_ERR_INVALID_ARG, "a required pointer is NULL");
  if (n_tokens < 1 || n_docs < 1) return set_err(h, DIT_ERR_LAYOUT, "n_tokens and n_docs must be >= 1");
  if (n_tokens > c.max_tokens || n_docs > c.max_docs)
    return set_err(h, DIT_ERR_CAPACITY, "n_tokens %d / n_docs %d exceed max_tokens %d / max_docs %d", n_tokens,
                   n_docs, c.max_tokens, c.max_docs);
  if ((!lat && !aligned16(x_tokens)) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return set_err(h, DIT_ERR_INVALID_ARG, "x/out must be 16-byte and workspace 256-byte aligned");
  if (static_cast<const void*>(x_tokens) == static_cast<const void*>(out))
    return set_err(h, DIT_ERR_INVALID_ARG, "out may not alias x_tokens");
  const WsLayout L = ws_layout(&c, n_tokens, n_docs);
  if (workspace_bytes < L.total)
    return set_err(h, DIT_ERR_CAPACITY, "workspace %zu bytes < required %zu", workspace_bytes, L.total);
  for (int i = 0; i < n_t; ++i)
    if (!(t_in[i] >= 0.f && t_in[i] <= 1.f)) return set_err(h, DIT_ERR_INVALID_ARG, "timestep must be in [0, 1]");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.dtype == DIT_FP32)
    return forward_fp32(h, x_tokens, cu_seqlens, n_docs, doc_ids, modality_tags, pos_thw, n_tokens, out, workspace, L,
                        s);
  const int d = c.hidden, F = c.ffn_hidden, H = c.n_heads, nm = c.n_modalities;
  const int N = n_tokens;
  const int f16 = c.act_bf16 ? 0 : 1;     // 16-bit operand type: f16 unless the config asks for bf16
  const int y_kind = f16 ? 2 : 0;
  StatusWords* sw = at<StatusWords>(workspace, L.status);
  int* status = &sw->bits;
  int2* items = at<int2>(workspace, L.items);
  float* mod = at<float>(workspace, L.mod);
  float* cosc = at<float>(workspace, L.cosc);
  float* sinc = at<float>(workspace, L.sinc);
  float* resid = at<float>(workspace, L.resid);
  const float* resid_lo = nullptr;  // the bf16 forward keeps a plain fp32 residual
  void* y = at<void>(workspace, L.y);
  void* q = at<void>(workspace, L.q);
  void* k = at<void>(workspace, L.k);
  void* vt = at<void>(workspace, L.vt);
  void* o = at<void>(workspace, L.o);
  void* hbuf = at<void>(workspace, L.h);

  {
    Launch ln(h, s, 6);
    DIT_CK(h, cudaMemsetAsync(sw, 0, sizeof(StatusWords), s), "status reset");
    DIT_CK(h, attention_schedule_launch(cu_seqlens, n_docs, N, doc_ids, modality_tags, nm, items, &sw->count,
                                        L.max_items, &sw->layout_code, status, s), "schedule");
    ln.done();
  }
  {
    Launch ln(h, s, 6);
    DIT_CK(h, rope_cache_launch(pos_thw, N, c.rope_axes, c.rope_dims, c.rope_base, cosc, sinc, status, s), "rope cache");
    ln.done();
  }
  if (c.adaln) {
    Launch ln(h, s, 6);
    AdaTimesteps ts{};
    ts.n_t = n_t;
    for (int i = 0; i < n_t; ++i) ts.t[i] = t_in[i];
    ts.six_d = 6 * d;
    ts.two_d = 2 * d;
    ts.mod_block = nm * 6 * d;
    ts.block_rows = c.n_blocks * nm * 6 * d;
    DIT_CK(h, adaln_launch(h->w_ada_all, h->b_ada_all, h->ada_rows, c.t_embed_dim, ts, mod, status, s), "adaln");
    ln.done();
  }
  if (lat) {
    const dit_status st = latent_embed(h, *lat, modality_tags, N, resid, &sw->layout_code, status, s);
    if (st != DIT_OK) return st;
  } else {
    DIT_CK(h, cudaMemcpyAsync(resid, x_tokens, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, s), "copy x");
  }

  const long long mstride = 6ll * d;  // between modality rows of one block's [n_mod][6][d]
  AttnArgs aa;
  aa.n_tokens = N;
  aa.n_heads = H;
  aa.head_dim = c.head_dim;
  aa.n_pad = L.n_pad;
  aa.n_docs = n_docs;
  aa.cu = cu_seqlens;
  aa.items = items;
  aa.count = &sw->count;
  aa.max_items = L.max_items;
  aa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  aa.status = status;
  aa.f16 = f16;

  for (int l = 0; l < c.n_blocks; ++l) {
    const BlockDev& B = h->blocks[l];
    const float* ml = mod + (size_t)l * nm * 6 * d;
    {
      Launch ln(h, s, 5);
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, B.ln1_g, B.ln1_b, modality_tags,
                                     c.adaln ? ml + 0 * d : nullptr, c.adaln ? ml + 1 * d : nullptr, mstride, y,
                                     y_kind, status, s), "norm1");
      ln.done();
    }
    {
      Launch ln(h, s, 0);
      GemmArgs g{};
      g.M = N; g.N = 3 * d; g.K = d; g.bias = B.b_qkv;
      g.d = d; g.head_dim = c.head_dim; g.rot_half = c.rotary_dim / 2;
      g.cos_cache = cosc; g.sin_cache = sinc; g.q = q; g.k = k; g.vt = vt; g.n_pad = L.n_pad;
      g.qk_norm = c.qk_norm; g.qk_eps = c.norm_eps;
      g.status = status; g.f16 = f16;
      DIT_CK(h, gemm_any(kEpiQkvRope, y, B.w_qkv, B.nv_qkv, B.g_qkv, g, s), "gemm qkv");
      ln.done();
    }
    {
      Launch ln(h, s, 1);
      DIT_CK(h, attention_launch(q, k, vt, o, aa, s), "attention");
      ln.done();
    }
    {
      Launch ln(h, s, 2);
      GemmArgs g{};
      g.M = N; g.N = d; g.K = d; g.bias = B.b_o;
      g.x = resid; g.gate = c.adaln ? ml + 2 * d : B.res1; g.gate_stride = c.adaln ? mstride : 0;
      g.tags = modality_tags; g.status = status; g.f16 = f16;
      DIT_CK(h, gemm_any(kEpiGatedResid, o, B.w_o, B.nv_o, B.g_o, g, s), "gemm out");
      ln.done();
    }
    {
      Launch ln(h, s, 5);
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, B.ln2_g, B.ln2_b, modality_tags,
                                     c.adaln ? ml + 3 * d : nullptr, c.adaln ? ml + 4 * d : nullptr, mstride, y,
                                     y_kind, status, s), "norm2");
      ln.done();
    }
    {
      Launch ln(h, s, 3);
      GemmArgs g{};
      g.M = N; g.N = 2 * F; g.K = d; g.bias = B.b_in_packed; g.out = hbuf; g.status = status;
      g.f16 = f16; g.out_kind = y_kind;
      DIT_CK(h, gemm_any(kEpiSwiglu, y, B.w_in_packed, B.nv_in, B.g_in, g, s), "gemm ffn up");
      ln.done();
    }
    {
      Launch ln(h, s, 4);
      GemmArgs g{};
      g.M = N; g.N = d; g.K = F; g.bias = B.b_down;
      g.x = resid; g.gate = c.adaln ? ml + 5 * d : B.res2; g.gate_stride = c.adaln ? mstride : 0;
      g.tags = modality_tags; g.status = status; g.f16 = f16;
      DIT_CK(h, gemm_any(kEpiGatedResid, hbuf, B.w_down, B.nv_down, B.g_down, g, s), "gemm ffn down");
      ln.done();
    }
    if (h->dump)
      DIT_CK(h, cudaMemcpyAsync(h->dump + (size_t)l * N * d, resid, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, s),
             "dump");
  }
  {
    const float* mf = mod + (size_t)c.n_blocks * nm * 6 * d;
    Launch ln(h, s, 5);
    if (c.adaln)
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.norm, c.norm_eps, nullptr, nullptr, modality_tags, mf,
                                     mf + d, 2ll * d, out, 1, status, s), "final norm");
    else  // the final norm without modulation: the blocks' kind, or final_norm's
      DIT_CK(h, norm_modulate_launch(resid, resid_lo, N, d, c.final_norm ? c.final_norm - 1 : c.norm, c.norm_eps,
                                     h->lnf_g, h->lnf_b, nullptr, nullptr, nullptr, 0, out, 1, status, s),
             "final norm");
    ln.done();
  }
  h->stats.forwards++;
  return DIT_OK;
}

dit_status dit_forward(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                       const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw, int n_tokens,
                       float timestep, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(h, x_tokens, cu_seqlens, n_docs, doc_ids, modality_tags, pos_thw, n_tokens, &timestep, 1, out,
                      workspace, workspace_bytes, stream);
}

dit_status dit_forward_modal(dit_handle* h, const float* x_tokens, const int32_t* cu_seqlens, int n_docs,
                             const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw, int n_tokens,
                             const float* timesteps, float* out, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!h) return DIT_ERR_INVALID_ARG;
  if (!timesteps) return set_err(h, DIT_ERR_INVALID_ARG, "timesteps is NULL");
  const int nm = h->cfg.adaln ? h->cfg.n_modalities : 1;
  if (nm > kMaxModalTimesteps)
    return set_err(h, DIT_ERR_UNSUPPORTED, "per-modality timesteps support up to %d modalities", kMaxModalTimesteps);
  return forward_impl(h, x_tokens, cu_seqlens, n_docs, doc_ids, modality_tags, pos_thw, n_tokens, timesteps, nm, out,
                      workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------------------------------------
// Latent I/O
// ------------------------------------------------------------------------------------------------

namespace {

// dit_forward_latent's workspace: the forward's, then the final hidden state [N][d], the row maps
// [N], and the islands' split operands [N][kmax] x 2 and partial sums [N][nmax] (island_splits
// keeps splits x M <= N).
struct LatLayout {
  size_t out_h, rows, xs_hi, xs_lo, part, total;
};

LatLayout lat_layout(const dit_handle* h, int N, int n_docs) {
  LatLayout L{};
  const int d = h->cfg.hidden;
  size_t kmax = (size_t)d, nmax = (size_t)d;
  for (int m = 0; m < h->lat_n; ++m) {
    kmax = std::max(kmax, (size_t)h->lat_kp[m]);
    nmax = std::max(nmax, (size_t)h->lat_np[m]);
  }
  size_t off = align_up(ws_layout(&h->cfg, N, n_docs).total);
  L.out_h = off;
  off = align_up(off + (size_t)N * d * 4);
  L.rows = off;
  off = align_up(off + (size_t)N * 4);
  L.xs_hi = off;
  off = align_up(off + (size_t)N * kmax * 4);
  L.xs_lo = off;
  off = align_up(off + (size_t)N * kmax * 4);
  L.part = off;
  off = align_up(off + (size_t)N * nmax * 4);
  L.total = off;
  return L;
}

}  // namespace

dit_status dit_bind_latent_io(dit_handle* h, const dit_latent_io* io, void* stream) {
  if (!h || !io) return DIT_ERR_INVALID_ARG;
  const dit_config& c = h->cfg;
  if (c.dtype != DIT_BF16 || !c.adaln)
    return set_err(h, DIT_ERR_UNSUPPORTED, "latent I/O needs the bf16 model with AdaLN");
  const int nm = io->n_modalities;
  if (nm != c.n_modalities || nm < 1 || nm > kMaxModalTimesteps)
    return set_err(h, DIT_ERR_INVALID_ARG, "n_modalities %d must equal the model's (%d) and be at most %d", nm,
                   c.n_modalities, kMaxModalTimesteps);
  for (int m = 0; m < nm; ++m) {
    if (io->width[m] < 1 || io->width[m] > 65536)
      return set_err(h, DIT_ERR_INVALID_ARG, "width[%d] = %d outside [1, 65536]", m, io->width[m]);
    if (!io->w_patch[m] || !io->w_head[m]) return set_err(h, DIT_ERR_MISSING_WEIGHT, "w_patch/w_head[%d] is NULL", m);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const int d = c.hidden;
  int kp[kMaxModalTimesteps], np[kMaxModalTimesteps];
  SplitW patch[kMaxModalTimesteps], head[kMaxModalTimesteps];
  float* bp[kMaxModalTimesteps] = {};
  float* bh[kMaxModalTimesteps] = {};
  auto alloc = [&](size_t floats) -> float* { return static_cast<float*>(dev_alloc(h, floats * 4, &e)); };
  auto copy_bias = [&](const float* src, int n) -> float* {
    if (!src) return nullptr;
    float* dst = alloc((size_t)n);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, (size_t)n * 4, cudaMemcpyDeviceToDevice, s);
    return dst;
  };
  for (int m = 0; m < nm; ++m) {
    const int w = io->width[m];
    kp[m] = (w + kTf32x3K - 1) / kTf32x3K * kTf32x3K;
    np[m] = (w + kTf32x3N - 1) / kTf32x3N * kTf32x3N;
    // patch projection [d][width] -> [d][kp], columns past width zero
    patch[m].hi = alloc((size_t)d * kp[m]);
    if (e == cudaSuccess) patch[m].lo = alloc((size_t)d * kp[m]);
    if (e == cudaSuccess)
      e = tf32_split_rows_launch(io->w_patch[m], w, w, nullptr, d, kp[m], patch[m].hi, patch[m].lo, nullptr, s);
    // output head [width][d] -> [np][d], rows past width zero
    if (e == cudaSuccess) head[m].hi = alloc((size_t)np[m] * d);
    if (e == cudaSuccess) head[m].lo = alloc((size_t)np[m] * d);
    if (e == cudaSuccess) e = cudaMemsetAsync(head[m].hi, 0, (size_t)np[m] * d * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(head[m].lo, 0, (size_t)np[m] * d * 4, s);
    if (e == cudaSuccess)
      e = tf32_split_rows_launch(io->w_head[m], d, d, nullptr, w, d, head[m].hi, head[m].lo, nullptr, s);
    if (e == cudaSuccess) bp[m] = copy_bias(io->b_patch[m], d);
    if (e == cudaSuccess) bh[m] = copy_bias(io->b_head[m], w);
    if (e != cudaSuccess) return cuda_err(h, e, "bind latent io");
  }
  DIT_CK(h, cudaStreamSynchronize(s), "bind latent io sync");
  h->lat_n = nm;
  for (int m = 0; m < nm; ++m) {
    h->lat_width[m] = io->width[m];
    h->lat_kp[m] = kp[m];
    h->lat_np[m] = np[m];
    h->lat_patch[m] = patch[m];
    h->lat_head[m] = head[m];
    h->lat_b_patch[m] = bp[m];
    h->lat_b_head[m] = bh[m];
  }
  return DIT_OK;
}

size_t dit_workspace_bytes_latent(const dit_handle* h, int n_tokens, int n_docs) {
  if (!h || h->lat_n == 0 || n_tokens < 1 || n_docs < 1) return 0;
  return lat_layout(h, n_tokens, n_docs).total;
}

dit_status dit_forward_latent(dit_handle* h, const float* const* z, const int* n_rows, const int32_t* cu_seqlens,
                              int n_docs, const int32_t* doc_ids, const uint8_t* modality_tags, const double* pos_thw,
                              int n_tokens, const float* timesteps, float* const* v, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!h) return DIT_ERR_INVALID_ARG;
  if (!h->bound) return set_err(h, DIT_ERR_UNBOUND, "dit_forward_latent before dit_bind_weights");
  if (h->lat_n == 0) return set_err(h, DIT_ERR_UNBOUND, "dit_forward_latent before dit_bind_latent_io");
  if (!z || !n_rows || !v || !timesteps || !workspace)
    return set_err(h, DIT_ERR_INVALID_ARG, "a required pointer is NULL");
  if (n_tokens < 1 || n_docs < 1) return set_err(h, DIT_ERR_LAYOUT, "n_tokens and n_docs must be >= 1");
  if (n_tokens > h->cfg.max_tokens || n_docs > h->cfg.max_docs)
    return set_err(h, DIT_ERR_CAPACITY, "n_tokens %d / n_docs %d exceed the handle's capacity", n_tokens, n_docs);
  LatentArgs a{};
  a.z = z;
  a.mr.n = h->lat_n;
  long long sum = 0;
  for (int m = 0; m < h->lat_n; ++m) {
    if (n_rows[m] < 0) return set_err(h, DIT_ERR_INVALID_ARG, "n_rows[%d] < 0", m);
    if (n_rows[m] > 0 && (!z[m] || !v[m])) return set_err(h, DIT_ERR_INVALID_ARG, "z[%d] or v[%d] is NULL", m, m);
    a.mr.count[m] = n_rows[m];
    a.mr.off[m] = (int)sum;
    sum += n_rows[m];
  }
  if (sum != n_tokens)
    return set_err(h, DIT_ERR_INVALID_ARG, "n_rows add up to %lld, not n_tokens = %d", sum, n_tokens);
  if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))
    return set_err(h, DIT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const LatLayout LL = lat_layout(h, n_tokens, n_docs);
  if (workspace_bytes < LL.total)
    return set_err(h, DIT_ERR_CAPACITY, "workspace %zu bytes < required %zu", workspace_bytes, LL.total);
  a.rows = at<int>(workspace, LL.rows);
  a.xs_hi = at<float>(workspace, LL.xs_hi);
  a.xs_lo = at<float>(workspace, LL.xs_lo);
  a.part = at<float>(workspace, LL.part);
  float* out_h = at<float>(workspace, LL.out_h);
  dit_status st = forward_impl(h, nullptr, cu_seqlens, n_docs, doc_ids, modality_tags, pos_thw, n_tokens, timesteps,
                               h->lat_n, out_h, workspace, workspace_bytes, stream, &a);
  if (st != DIT_OK) return st;
  // the output heads: v_m = out[rows_m] W_head^T + b_head
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = &at<StatusWords>(workspace, ws_layout(&h->cfg, n_tokens, n_docs).status)->bits;
  const int d = h->cfg.hidden;
  for (int m = 0; m < h->lat_n; ++m) {
    const int M = n_rows[m];
    if (M == 0) continue;
    const int Np = h->lat_np[m];
    Launch ln(h, s, 7);
    DIT_CK(h, tf32_split_rows_launch(out_h, d, d, a.rows + a.mr.off[m], M, d, a.xs_hi, a.xs_lo, status, s),
           "head split");
    const int want = island_splits(M, Np, d, n_tokens);
    DIT_CK(h, tf32x3_partial_launch(a.xs_hi, a.xs_lo, h->lat_head[m].hi, h->lat_head[m].lo, M, Np, d, want, a.part,
                                    status, s), "output head");
    DIT_CK(h, sgemm_reduce_rows_launch(a.part, tf32x3_effective_splits(d, want), M, Np, h->lat_width[m],
                                       h->lat_b_head[m], nullptr, v[m], h->lat_width[m], status, s),
           "output head store");
    ln.done(3);
  }
  return DIT_OK;
}

static dit_status patch_call(const float* src, float* dst, int C, int T, int H, int W, int pt, int ph, int pw,
                             int inverse, void* stream) {
  if (!src || !dst) return set_err(nullptr, DIT_ERR_INVALID_ARG, "NULL latent or token buffer");
  if (C < 1 || T < 1 || H < 1 || W < 1 || pt < 1 || ph < 1 || pw < 1)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "every size must be >= 1");
  const long long P = (long long)C * pt * ph * pw;
  if (P > 12287) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "C*pt*ph*pw = %lld above 12287", P);
  const long long n = P * T * H * W;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(src), b0 = reinterpret_cast<uintptr_t>(dst);
  if (a0 < b0 + (uintptr_t)n * 4 && b0 < a0 + (uintptr_t)n * 4)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "latent and token buffers overlap");
  const cudaError_t e = patch_launch(src, dst, C, T, H, W, pt, ph, pw, inverse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, inverse ? "unpatchify" : "patchify");
}

dit_status dit_patchify(const float* latent, int C, int T, int H, int W, int pt, int ph, int pw, float* tokens,
                        void* stream) {
  return patch_call(latent, tokens, C, T, H, W, pt, ph, pw, 0, stream);
}

dit_status dit_unpatchify(const float* tokens, int C, int T, int H, int W, int pt, int ph, int pw, float* latent,
                          void* stream) {
  return patch_call(tokens, latent, C, T, H, W, pt, ph, pw, 1, stream);
}

dit_status dit_audio_pack(const float* latent, int C, int T, float* tokens, void* stream) {
  return patch_call(latent, tokens, C, T, 1, 1, 1, 1, 1, 0, stream);
}

dit_status dit_audio_unpack(const float* tokens, int C, int T, float* latent, void* stream) {
  return patch_call(tokens, latent, C, T, 1, 1, 1, 1, 1, 1, stream);
}

size_t dit_workspace_bytes_host(const dit_config* cfg, int n_tokens, int n_docs) {
  size_t base = dit_workspace_bytes(cfg, n_tokens, n_docs);
  if (!base) return 0;
  const size_t width = cfg->io_channels ? cfg->io_channels : cfg->hidden;
  size_t extra = align_up((size_t)n_tokens * width * 4) * 2 + align_up((size_t)(n_docs + 1) * 4) +
                 align_up((size_t)n_tokens * 4) + align_up((size_t)n_tokens) + align_up((size_t)n_tokens * 24);
  return align_up(base) + extra;
}

dit_status dit_forward_host(dit_handle* h, const float* x_host, const int32_t* cu_host, int n_docs,
                            const int32_t* doc_ids_host, const uint8_t* tags_host, const double* pos_host,
                            int n_tokens, float timestep, float* out_host, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!h) return DIT_ERR_INVALID_ARG;
  if (!x_host || !cu_host || !doc_ids_host || !tags_host || !pos_host || !out_host || !workspace)
    return set_err(h, DIT_ERR_INVALID_ARG, "a required pointer is NULL");
  if (n_tokens < 1 || n_docs < 1) return set_err(h, DIT_ERR_LAYOUT, "n_tokens and n_docs must be >= 1");
  const size_t need = dit_workspace_bytes_host(&h->cfg, n_tokens, n_docs);
  if (!need || workspace_bytes < need) return set_err(h, DIT_ERR_CAPACITY, "workspace too small for the host forward");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t base = align_up(dit_workspace_bytes(&h->cfg, n_tokens, n_docs));
  const size_t width = h->cfg.io_channels ? h->cfg.io_channels : h->cfg.hidden;
  const size_t xb = (size_t)n_tokens * width * 4;
  char* p = static_cast<char*>(workspace) + base;
  float* x_d = reinterpret_cast<float*>(p); p += align_up(xb);
  float* out_d = reinterpret_cast<float*>(p); p += align_up(xb);
  int32_t* cu_d = reinterpret_cast<int32_t*>(p); p += align_up((size_t)(n_docs + 1) * 4);
  int32_t* ids_d = reinterpret_cast<int32_t*>(p); p += align_up((size_t)n_tokens * 4);
  uint8_t* tags_d = reinterpret_cast<uint8_t*>(p); p += align_up((size_t)n_tokens);
  double* pos_d = reinterpret_cast<double*>(p);
  DIT_CK(h, cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, s), "h2d x");
  DIT_CK(h, cudaMemcpyAsync(cu_d, cu_host, (size_t)(n_docs + 1) * 4, cudaMemcpyHostToDevice, s), "h2d cu");
  DIT_CK(h, cudaMemcpyAsync(ids_d, doc_ids_host, (size_t)n_tokens * 4, cudaMemcpyHostToDevice, s), "h2d doc_ids");
  DIT_CK(h, cudaMemcpyAsync(tags_d, tags_host, (size_t)n_tokens, cudaMemcpyHostToDevice, s), "h2d tags");
  DIT_CK(h, cudaMemcpyAsync(pos_d, pos_host, (size_t)n_tokens * 24, cudaMemcpyHostToDevice, s), "h2d pos");
  dit_status st = dit_forward(h, x_d, cu_d, n_docs, ids_d, tags_d, pos_d, n_tokens, timestep, out_d, workspace,
                              base, stream);
  if (st != DIT_OK) return st;
  DIT_CK(h, cudaMemcpyAsync(out_host, out_d, xb, cudaMemcpyDeviceToHost, s), "d2h out");
  DIT_CK(h, cudaStreamSynchronize(s), "host forward sync");
  return DIT_OK;
}

dit_status dit_euler_step(float* x, const float* v, int64_t n, float sigma, float sigma_next, void* stream) {
  if (n < 0 || (n > 0 && (!x || !v))) return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad euler arguments");
  if (!(sigma > 0.f)) return set_err(nullptr, DIT_ERR_INVALID_ARG, "sigma must be > 0");
  cudaError_t e = euler_launch(x, v, n, sigma, sigma_next, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "euler");
}

dit_status dit_euler_step_modal(float* x, const float* v, int n_tokens, int d, const uint8_t* tags,
                                const float* sigma, const float* sigma_next, int n_modalities, void* stream) {
  if (n_tokens < 0 || d < 1 || (n_tokens > 0 && (!x || !v || !tags)) || !sigma || !sigma_next || n_modalities < 1 ||
      n_modalities > kMaxModalTimesteps)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad tagged euler arguments");
  ModalSigmas sg{};
  sg.n = n_modalities;
  for (int m = 0; m < n_modalities; ++m) {
    if (!(sigma[m] > 0.f)) return set_err(nullptr, DIT_ERR_INVALID_ARG, "sigma must be > 0");
    sg.sigma[m] = sigma[m];
    sg.sigma_next[m] = sigma_next[m];
  }
  cudaError_t e = euler_tagged_launch(x, v, n_tokens, d, tags, sg, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "euler tagged");
}

dit_status dit_vit_positions(int T, int H, int W, double* pos) {
  if (T < 1 || H < 1 || W < 1 || !pos) return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad vit_positions arguments");
  const double two_pi = 6.283185307179586476925;  // 2 pi
  const int n[3] = {T, H, W};
  for (int t = 0; t < T; ++t)
    for (int hh = 0; hh < H; ++hh)
      for (int w = 0; w < W; ++w) {
        const int id[3] = {t, hh, w};
        double* p = pos + ((size_t)(t * H + hh) * W + w) * 3;
        for (int a = 0; a < 3; ++a) p[a] = (2.0 * ((id[a] + 0.5) / (double)n[a]) - 1.0) * two_pi;
      }
  return DIT_OK;
}

float dit_time_shift(float sigma, float shift) {
  const double s = (double)shift, x = (double)sigma;
  return (float)(s * x / (1.0 + (s - 1.0) * x));
}

dit_status dit_get_stats(const dit_handle* h, dit_stats* out) {
  if (!h || !out) return DIT_ERR_INVALID_ARG;
  *out = h->stats;
  return DIT_OK;
}

dit_status dit_sync_status(dit_handle* h, const void* workspace, void* stream) {
  if (!h || !workspace) return DIT_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StatusWords sw;
  DIT_CK(h, cudaStreamSynchronize(s), "sync");
  DIT_CK(h, cudaMemcpy(&sw, workspace, sizeof sw, cudaMemcpyDeviceToHost), "read status");
  h->stats.device_status = sw.bits;
  h->stats.last_layout_error = sw.layout_code;
  h->stats.attention_tiles = (int64_t)sw.count * h->cfg.n_heads;
  if (sw.bits & kDevLayout) return set_err(h, DIT_ERR_LAYOUT, "device validator rejected the layout (code %d)", sw.layout_code);
  if (sw.bits & kDevTimeout) return set_err(h, DIT_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out");
  if (sw.bits & kDevCapacity) return set_err(h, DIT_ERR_CAPACITY, "tile schedule overflow");
  if (sw.bits & kDevRange)
    return set_err(h, DIT_ERR_RANGE, "an f16 operand (norm output or FFN hidden) exceeded 65504; act_bf16 = 1 avoids it");
  return DIT_OK;
}

dit_status dit_selftest_wait_timeout(uint64_t limit_ns, int* status_word, void* stream) {
  if (!status_word || limit_ns == 0 || limit_ns > 1000000000ull)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "status_word must be a device int; 0 < limit_ns <= 1e9");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int bits = 0;
  cudaError_t e = cudaMemsetAsync(status_word, 0, sizeof(int), s);
  if (e == cudaSuccess) e = wait_timeout_selftest_launch(status_word, limit_ns, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&bits, status_word, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "wait self-test");
  return (bits & kDevTimeout) ? DIT_ERR_DEVICE_TIMEOUT : DIT_OK;
}

dit_status dit_set_dump(dit_handle* h, float* dump) {
  if (!h) return DIT_ERR_INVALID_ARG;
  h->dump = dump;
  return DIT_OK;
}

dit_status dit_set_kernel_timing(dit_handle* h, int enable) {
  if (!h) return DIT_ERR_INVALID_ARG;
  h->timing = enable != 0;
  h->timed.clear();
  h->ev_next = 0;
  memset(h->ms_acc, 0, sizeof h->ms_acc);
  memset(h->n_acc, 0, sizeof h->n_acc);
  return DIT_OK;
}

dit_status dit_get_kernel_times(dit_handle* h, double* ms_out, int64_t* launches_out) {
  if (!h || !ms_out || !launches_out) return DIT_ERR_INVALID_ARG;
  DIT_CK(h, cudaDeviceSynchronize(), "timing sync");
  for (const TimedLaunch& t : h->timed) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      h->ms_acc[t.kind] += ms;
      h->n_acc[t.kind] += 1;
    }
  }
  h->timed.clear();
  h->ev_next = 0;
  for (int i = 0; i < DIT_KERNEL_KINDS; ++i) {
    ms_out[i] = h->ms_acc[i];
    launches_out[i] = h->n_acc[i];
  }
  return DIT_OK;
}

// ------------------------------------------------------------------------------------------------
// op-level entry points
// ------------------------------------------------------------------------------------------------

dit_status dit_op_norm_modulate(const float* x, int n, int d, int norm, float eps, const float* ln_g, const float* ln_b,
                                const uint8_t* tags, const float* shift, const float* scale, int64_t mod_stride,
                                void* y, int out_kind, void* stream) {
  if (n < 0 || !x || !y || (shift && (!scale || !tags)) || out_kind < 0 || out_kind > 2 ||
      (norm != DIT_RMSNORM && norm != DIT_LAYERNORM))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad norm_modulate arguments");
  if (!norm_width_supported(d)) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "width %d not tiled by the norm kernel", d);
  if (!aligned16(x) || !aligned16(y) || (shift && (!aligned16(shift) || !aligned16(scale) || mod_stride % 4)))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "norm_modulate pointers must be 16-byte aligned");
  cudaError_t e = norm_modulate_launch(x, nullptr, n, d, norm, eps, ln_g, ln_b, tags, shift, scale, mod_stride, y, out_kind,
                                       nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "norm_modulate");
}

dit_status dit_op_rope_cache(const double* pos, int n, int n_axes, const int* dims_host, double base, float* cos_out,
                             float* sin_out, void* stream) {
  if (n < 0 || !pos || !cos_out || !sin_out || !dims_host || (n_axes != 1 && n_axes != 3))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad rope_cache arguments");
  cudaError_t e = rope_cache_launch(pos, n, n_axes, dims_host, base, cos_out, sin_out, nullptr,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "rope_cache");
}

dit_status dit_op_adaln(const void* w, const float* b, int rows, int t_dim, float t, float* mod, void* stream) {
  if (rows < 0 || !w || !mod || t_dim < 8 || t_dim % 8 || (t_dim > 256 && t_dim % 256) || !aligned16(w))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad adaln arguments");
  AdaTimesteps ts{};
  ts.n_t = 1;
  ts.t[0] = t;
  cudaError_t e = adaln_launch(w, b, rows, t_dim, ts, mod, nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "adaln");
}

static dit_status check_gemm(const void* a, const void* b, int M, int N, int K, int elem) {
  if (!a || !b || M < 0 || N <= 0 || K <= 0) return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad GEMM arguments");
  if (elem != DIT_ELEM_BF16 && elem != DIT_ELEM_F16)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "elem must be DIT_ELEM_BF16 or DIT_ELEM_F16");
  if (N % 256 || K % 64) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "GEMM needs N %% 256 == 0 and K %% 64 == 0");
  if (!aligned16(a) || !aligned16(b)) return set_err(nullptr, DIT_ERR_INVALID_ARG, "GEMM operands must be 16-byte aligned");
  return DIT_OK;
}

dit_status dit_op_gemm(const void* a, const void* b, const float* bias, int M, int N, int K, void* out, int out_kind,
                       int elem, void* stream) {
  dit_status st = check_gemm(a, b, M, N, K, elem);
  if (st != DIT_OK) return st;
  if (!out || out_kind < 0 || out_kind > 2) return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad GEMM output");
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.bias = bias; g.out = out; g.out_kind = out_kind; g.f16 = elem;
  cudaError_t e = gemm_launch(kEpiStore, a, b, g, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "gemm");
}

size_t dit_nvfp4_packed_bytes(int N, int K) {
  if (N <= 0 || K <= 0 || N % 256 || K % 64) return 0;
  return (size_t)N * K * 9 / 16;
}

dit_status dit_op_pack_nvfp4(const uint8_t* q, const uint8_t* scales, int N, int K, void* packed, void* stream) {
  if (!q || !scales || !packed || N <= 0 || K <= 0 || N % 256 || K % 64 || !aligned16(packed))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad NVFP4 pack arguments (N %% 256, K %% 64, 16-byte aligned out)");
  cudaError_t e = nvfp4_pack_launch(q, scales, N, K, static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "nvfp4 pack");
}

dit_status dit_op_gemm_nvfp4(const void* a_f16, const void* packed, float w_scale, const float* bias, int M, int N,
                             int K, void* out, int out_kind, void* stream) {
  if (!a_f16 || !packed || !out || M < 1 || N <= 0 || K <= 0 || N % 256 || K % 64 || !aligned16(a_f16) ||
      !aligned16(packed) || out_kind < 0 || out_kind > 2)
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad NVFP4 GEMM arguments");
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.bias = bias; g.out = out; g.out_kind = out_kind;
  g.b_packed = static_cast<const uint8_t*>(packed);
  g.w_scale = w_scale;
  cudaError_t e = gemm_nvfp4_launch(kEpiStore, a_f16, g, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "nvfp4 gemm");
}

dit_status dit_op_gemm_qkv_rope(const void* a, const void* b, const float* bias, int M, int d, int K, int n_heads,
                                int head_dim, int rotary_dim, const float* cos_cache, const float* sin_cache, void* q,
                                void* k, void* vt, int n_pad, int elem, void* stream) {
  dit_status st = check_gemm(a, b, M, 3 * d, K, elem);
  if (st != DIT_OK) return st;
  if (d % 256 || n_heads * head_dim != d || 256 % head_dim || rotary_dim > head_dim || (rotary_dim / 2) % 16 ||
      (head_dim - rotary_dim) % 16 || !q || !k || !vt || n_pad < M || n_pad % 8 ||
      (rotary_dim > 0 && (!cos_cache || !sin_cache)))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad qkv_rope arguments");
  GemmArgs g{};
  g.M = M; g.N = 3 * d; g.K = K; g.bias = bias; g.d = d; g.head_dim = head_dim; g.rot_half = rotary_dim / 2;
  g.cos_cache = cos_cache; g.sin_cache = sin_cache; g.q = q; g.k = k; g.vt = vt; g.n_pad = n_pad; g.f16 = elem;
  cudaError_t e = gemm_launch(kEpiQkvRope, a, b, g, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "gemm qkv");
}

dit_status dit_op_gemm_gated_residual(const void* a, const void* b, const float* bias, int M, int N, int K, float* x,
                                      const float* gate, int64_t gate_stride, const uint8_t* tags, int elem,
                                      void* stream) {
  dit_status st = check_gemm(a, b, M, N, K, elem);
  if (st != DIT_OK) return st;
  if (!x || (gate && (!tags || gate_stride % 4 || !aligned16(gate))) || !aligned16(x))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad gated_residual arguments");
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.bias = bias; g.x = x; g.gate = gate; g.gate_stride = gate_stride; g.tags = tags;
  g.f16 = elem;
  cudaError_t e = gemm_launch(kEpiGatedResid, a, b, g, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "gemm gated residual");
}

dit_status dit_op_gemm_swiglu(const void* a, const void* b_packed, const float* bias_packed, int M, int F, int K,
                              void* hout, int elem, void* stream) {
  dit_status st = check_gemm(a, b_packed, M, 2 * F, K, elem);
  if (st != DIT_OK) return st;
  if (!hout || F % 128) return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad swiglu arguments");
  GemmArgs g{};
  g.M = M; g.N = 2 * F; g.K = K; g.bias = bias_packed; g.out = hout; g.f16 = elem; g.out_kind = elem ? 2 : 0;
  cudaError_t e = gemm_launch(kEpiSwiglu, a, b_packed, g, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "gemm swiglu");
}

dit_status dit_op_pack_ffn_in(const void* w_in, const float* b_in, int F, int d, void* w_packed, float* b_packed,
                              void* stream) {
  if (!w_in || !w_packed || !b_packed || F <= 0 || F % 128 || d <= 0 || d % 8 || !aligned16(w_in) || !aligned16(w_packed))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad pack_ffn_in arguments");
  cudaError_t e = pack_ffn_in_launch(w_in, b_in, F, d, w_packed, b_packed, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "pack_ffn_in");
}

namespace {
struct GemmF32Ws {
  size_t x_hi, x_lo, w_hi, w_lo, part, maxbits, w_exp, total;
  int Kp;
};
GemmF32Ws gemm_f32_ws(int M, int N, int K) {
  GemmF32Ws w{};
  w.Kp = (K + kF16x3K - 1) / kF16x3K * kF16x3K;  // zero-padded to the GEMM's K step
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  w.x_hi = take((size_t)M * w.Kp * 2);
  w.x_lo = take((size_t)M * w.Kp * 2);
  w.w_hi = take((size_t)N * w.Kp * 2);
  w.w_lo = take((size_t)N * w.Kp * 2);
  w.part = take((size_t)kSgemmMaxSplits * M * N * 4);
  w.maxbits = take(16);
  w.w_exp = take(16);
  w.total = off;
  return w;
}
}  // namespace

size_t dit_gemm_f32_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  return gemm_f32_ws(M, N, K).total;
}

dit_status dit_op_gemm_f32(const float* x, const float* w, const float* bias, int M, int N, int K, float* y,
                           void* workspace, void* stream) {
  if (!x || !w || !y || !workspace || M < 1 || N < 128 || N % 128 || K < 32 || K % 32 || !aligned16(x) ||
      !aligned16(w) || !aligned16(y))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "fp32 GEMM needs M >= 1, N %% 128 == 0, K %% 32 == 0, aligned pointers");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const GemmF32Ws L = gemm_f32_ws(M, N, K);
  const int Kp = L.Kp;
  uint16_t* x_hi = at<uint16_t>(workspace, L.x_hi);
  uint16_t* x_lo = at<uint16_t>(workspace, L.x_lo);
  uint16_t* w_hi = at<uint16_t>(workspace, L.w_hi);
  uint16_t* w_lo = at<uint16_t>(workspace, L.w_lo);
  float* part = at<float>(workspace, L.part);
  unsigned int* maxbits = at<unsigned int>(workspace, L.maxbits);
  int* w_exp = at<int>(workspace, L.w_exp);
  cudaError_t e = f16_split_launch(x, K, K, M, Kp, nullptr, kF16x3ActExp, nullptr, x_hi, x_lo, nullptr, s);
  if (e == cudaSuccess) e = absmax_launch(w, (size_t)N * K, maxbits, s);
  if (e == cudaSuccess) e = f16_split_launch(w, K, K, N, Kp, maxbits, 0, w_exp, w_hi, w_lo, nullptr, s);
  const int want = f16x3_splits(M, N, Kp);
  if (e == cudaSuccess)
    e = f16x3_partial_launch(x_hi, x_lo, w_hi, w_lo, w_exp, kF16x3ActExp, M, N, Kp, want, part, nullptr, s);
  if (e == cudaSuccess)
    e = sgemm_reduce_store_launch(part, f16x3_effective_splits(Kp, want), M, N, bias, y, 0, nullptr, nullptr, s);
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "fp32 gemm");
}

int dit_attention_block_rows(void) { return attention_item_rows(); }

size_t dit_attention_workspace_bytes(int n_docs, int n_tokens) {
  if (n_docs < 1 || n_tokens < 1) return 0;
  return align_up(sizeof(StatusWords)) + align_up((size_t)attention_max_items(n_docs, n_tokens) * sizeof(int2));
}

dit_status dit_op_attention(const void* q, const void* k, const void* vt, int n_pad, const int32_t* cu_seqlens,
                            int n_docs, int n_tokens, int n_heads, int head_dim, void* o, void* workspace, int elem,
                            void* stream) {
  if (!q || !k || !vt || !o || !cu_seqlens || !workspace || n_docs < 1 || n_tokens < 1 || n_heads < 1 ||
      n_pad < n_tokens || n_pad % 8 || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) ||
      (elem != DIT_ELEM_BF16 && elem != DIT_ELEM_F16))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad attention arguments");
  if (head_dim != 128 && head_dim != 64) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "attention needs head_dim 64 or 128");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "attention operands must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StatusWords* sw = static_cast<StatusWords*>(workspace);
  int2* items = at<int2>(workspace, align_up(sizeof(StatusWords)));
  const int max_items = attention_max_items(n_docs, n_tokens);
  cudaError_t e = cudaMemsetAsync(sw, 0, sizeof(StatusWords), s);
  if (e == cudaSuccess)
    e = attention_schedule_launch(cu_seqlens, n_docs, n_tokens, nullptr, nullptr, 0, items, &sw->count, max_items,
                                  &sw->layout_code, &sw->bits, s);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "attention schedule");
  AttnArgs aa;
  aa.n_tokens = n_tokens; aa.n_heads = n_heads; aa.head_dim = head_dim; aa.n_pad = n_pad; aa.n_docs = n_docs;
  aa.cu = cu_seqlens; aa.items = items; aa.count = &sw->count; aa.max_items = max_items;
  aa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)head_dim));
  aa.status = &sw->bits;
  aa.f16 = elem;
  e = attention_launch(q, k, vt, o, aa, s);
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "attention");
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Attention without caller-provided scratch
//
// Some callers cannot call cudaMalloc: a plugin that runs inside another framework's executor and is
// handed no allocator, or a latency-critical serving thread for which cudaMalloc's implicit device
// synchronisation is not acceptable.  dit_op_attention needs a small scratch buffer (three status
// words and the (document, q-tile) list); this variant keeps that scratch in a fixed array in the
// library's own device memory instead, so it allocates nothing.  Every GPU that loads the library
// holds the array until the process exits.
// ------------------------------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxItems = DIT_ATTENTION_NOALLOC_MAX_TILES;  // (document, 128-row q-tile) work items
constexpr size_t kNoAllocStatusBytes = 256;                        // StatusWords, padded to the array's alignment
constexpr int kNoAllocCacheSlots = 64;
static_assert(sizeof(StatusWords) <= kNoAllocStatusBytes, "status words must fit their slot of the array");
static_assert(kNoAllocStatusBytes % alignof(int2) == 0, "the tile list must stay aligned");

static __device__ __align__(256) unsigned char g_attention_scratch[kNoAllocStatusBytes + kNoAllocMaxItems * 8];

// The array's device address is a property of the CUDA context that loaded the library's module:
// a cudaDeviceReset (which ends the primary context) or a caller-made context gives another one.
// Addresses are therefore cached per context, keyed by the driver's unique context id, which is never
// reused within a process.  Without that id (an older driver) the address is looked up on every call.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct NoAllocSlot {
  unsigned long long ctx_id;
  void* ptr;
};

std::mutex g_noalloc_mutex;
NoAllocSlot g_noalloc_cache[kNoAllocCacheSlots] = {};
int g_noalloc_next = 0;

template <typename F>
F driver_fn(const char* name) {
  cudaDriverEntryPointQueryResult q;
  void* p = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}

// Unique id of the calling thread's current context, or 0 when there is none or the driver cannot
// say.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_attention_scratch in the current context.  The host-side symbol is only a
// stand-in for the array, so its device address is looked up (cudaGetSymbolAddress, with the
// context current) the first time a context uses it and cached for that context.
cudaError_t noalloc_scratch(void** out) {
  unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (id)
    for (const NoAllocSlot& sl : g_noalloc_cache)
      if (sl.ctx_id == id) {
        *out = sl.ptr;
        return cudaSuccess;
      }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress((void**)&p, g_attention_scratch);
  if (e != cudaSuccess) return e;
  if (!id) id = current_context_id();  // the lookup above may have made the primary context current
  if (id) {
    g_noalloc_cache[g_noalloc_next] = NoAllocSlot{id, p};
    g_noalloc_next = (g_noalloc_next + 1) % kNoAllocCacheSlots;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" dit_status dit_op_attention_noalloc(const void* q, const void* k, const void* vt, int n_pad,
                                               const int32_t* cu_seqlens, int n_docs, int n_tokens, int n_heads,
                                               int head_dim, void* o, int elem, void* stream) {
  if (!q || !k || !vt || !o || !cu_seqlens || n_docs < 1 || n_tokens < 1 || n_heads < 1 || n_pad < n_tokens ||
      n_pad % 8 || (elem != DIT_ELEM_BF16 && elem != DIT_ELEM_F16))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "bad attention arguments");
  if (head_dim != 128 && head_dim != 64) return set_err(nullptr, DIT_ERR_UNSUPPORTED, "attention needs head_dim 64 or 128");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o))
    return set_err(nullptr, DIT_ERR_INVALID_ARG, "attention operands must be 16-byte aligned");
  const int max_items = attention_max_items(n_docs, n_tokens);
  if (max_items > kNoAllocMaxItems)
    return set_err(nullptr, DIT_ERR_CAPACITY,
                   "dit_op_attention_noalloc: ceil(n_tokens / 128) + n_docs = %d work items exceeds its fixed "
                   "scratch of %d; use dit_op_attention with a workspace",
                   max_items, kNoAllocMaxItems);
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "cudaGetSymbolAddress(attention scratch)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StatusWords* sw = static_cast<StatusWords*>(scratch);
  int2* items = reinterpret_cast<int2*>(static_cast<char*>(scratch) + kNoAllocStatusBytes);
  // The array keeps the previous call's contents: the status bits are OR-ed into, so they start at
  // zero; the count, the layout code and the tile list are rewritten by the schedule kernel.
  e = cudaMemsetAsync(sw, 0, sizeof(StatusWords), s);
  if (e == cudaSuccess)
    e = attention_schedule_launch(cu_seqlens, n_docs, n_tokens, nullptr, nullptr, 0, items, &sw->count, max_items,
                                  &sw->layout_code, &sw->bits, s);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "attention schedule");
  AttnArgs aa;
  aa.n_tokens = n_tokens; aa.n_heads = n_heads; aa.head_dim = head_dim; aa.n_pad = n_pad; aa.n_docs = n_docs;
  aa.cu = cu_seqlens; aa.items = items; aa.count = &sw->count; aa.max_items = max_items;
  aa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)head_dim));
  aa.status = &sw->bits;
  aa.f16 = elem;
  e = attention_launch(q, k, vt, o, aa, s);
  return e == cudaSuccess ? DIT_OK : cuda_err(nullptr, e, "attention");
}

extern "C" dit_status dit_op_attention_noalloc_status(int* layout_code, void* stream) {
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "cudaGetSymbolAddress(attention scratch)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StatusWords sw;
  e = cudaMemcpyAsync(&sw, scratch, sizeof(sw), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(nullptr, e, "reading the attention scratch's status words");
  if (layout_code) *layout_code = sw.layout_code;
  if (sw.bits & kDevTimeout) return set_err(nullptr, DIT_ERR_DEVICE_TIMEOUT, "attention: a bounded wait ran out");
  if (sw.bits & kDevLayout)
    return set_err(nullptr, DIT_ERR_LAYOUT, "attention: cu_seqlens rejected (layout code %d)", sw.layout_code);
  if (sw.bits & kDevCapacity) return set_err(nullptr, DIT_ERR_CAPACITY, "attention: tile list overflow");
  return DIT_OK;
}
