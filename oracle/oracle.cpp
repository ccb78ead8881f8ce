// CPU oracle for the packed-varlen joint video+audio DiT forward and its Euler loop.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct statement of what the
// GPU library computes.  Only the test suite, the package smoke check and the bench's CPU-baseline
// leg may load it; the library itself never does.  It shares no code, header, table or helper with
// the CUDA path.  Every sum accumulates in double, every op is a naive loop in the order its
// definition states, and inputs (bf16-valued or fp32 weights, fp32 tokens) are widened to double.
// The Euler step alone is fp32, because the page fixes it as an exact, bit-reproducible step.
//
// Sources (page title, then the section):
//   [H3]  "feat(minimax-h3): port the MiniMax-H3 omni-modal video+audio DiT"
//   [M3]  "feat(MODEL-MUSIC-MUSIC3): the 2.4B fp32 DiT onto the device, staged once"
//   [BF]  "feat(minimax-h3): stream the ORIGINAL bf16 DiT to the device, one tensor at a time"
//
// Readings where the pages are silent are marked READING and are listed in the design notes.
// Functions whose values no page or closed form pins are marked "parity unpinned".
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

typedef struct {
  int n_blocks, hidden, n_heads, head_dim, ffn_hidden;
  int norm;  // 0 = RMSNorm, 1 = LayerNorm
  double norm_eps;
  int adaln;  // 1 = modality-indexed AdaLN with gated residuals; 0 = plain residual adds
  int n_mod, t_dim;
  int rope_axes;
  int rope_dims[3];  // per-axis rotary widths in dims (pairs = dims / 2)
  int rotary_dim;    // sum of rope_dims, <= head_dim
  double rope_base;
  int io_channels;   // > 0: 1x1 pre/post convolutions io_channels <-> hidden
  // The video-VAE ViT3D decoder block ([H3] "Update: video-VAE decoder block ported"):
  int qk_norm;          // 1: per-head RMS norm of q and k, no affine, before RoPE
  int qkv_interleaved;  // 1: the fused qkv rows per head, [q_h | k_h | v_h] (else [q_all | k_all | v_all])
  int final_norm;       // without AdaLN: 0 the blocks' norm, 1 RMSNorm, 2 LayerNorm
} orc_config;

typedef struct {
  const float *w_qkv, *b_qkv, *w_o, *b_o, *w_in, *b_in, *w_down, *b_down;
  const float *w_ada, *b_ada;
  const float *ln1_g, *ln1_b, *ln2_g, *ln2_b;  // norm gains / shifts (either norm; NULL = none)
  const float *res1, *res2;                   // per-channel residual scales (NULL = 1)
} orc_block;

typedef struct {
  const orc_block* blocks;
  const float *w_ada_final, *b_ada_final;
  const float *lnf_g, *lnf_b;
  const float *w_pre, *b_pre, *w_post, *b_post;
} orc_weights;

static int g_threads = 1;

void orc_set_threads(int n) { g_threads = n > 0 ? n : 1; }

int orc_get_threads(void) { return g_threads; }

// ---------------------------------------------------------------------------------------------
// Packed layout.  [H3] "Correctness gates": the packed layout carries ids, tags, masks,
// cu_seqlens and doc ids, gated exact.  Contract checked here: cu[0] = 0, strictly increasing,
// cu[D] = N, doc_ids[i] = j exactly when cu[j] <= i < cu[j+1], every tag < n_mod.
// Returns 0 when valid, else a positive code naming the first broken rule.
// ---------------------------------------------------------------------------------------------
int orc_check_layout(const int32_t* cu, int n_docs, const int32_t* doc_ids, const uint8_t* tags, int n_tokens,
                     int n_mod) {
  if (n_docs < 1) return 1;
  if (cu[0] != 0) return 2;
  for (int j = 0; j < n_docs; ++j)
    if (cu[j + 1] <= cu[j]) return 3;
  if (cu[n_docs] != n_tokens) return 4;
  for (int j = 0; j < n_docs; ++j)
    for (int i = cu[j]; i < cu[j + 1]; ++i)
      if (doc_ids[i] != j) return 5;
  for (int i = 0; i < n_tokens; ++i)
    if ((int)tags[i] >= n_mod) return 6;
  return 0;
}

// Number of 128-row query tiles the varlen attention visits: sum over documents of
// ceil(len / 128).  Every (document, row) pair falls in exactly one tile.
int orc_count_q_tiles(const int32_t* cu, int n_docs, int tile) {
  int n = 0;
  for (int j = 0; j < n_docs; ++j) n += (cu[j + 1] - cu[j] + tile - 1) / tile;
  return n;
}

// ---------------------------------------------------------------------------------------------
// fp64 position grid.  [H3] "Correctness gates": numpy.linspace(endpoint=False) evaluates
// i*step + start, and that arithmetic order is what makes the grid bit-exact.
// step = (stop - start) / n.
// ---------------------------------------------------------------------------------------------
void orc_linspace(double start, double stop, int n, double* out) {
  double step = (stop - start) / (double)n;
  for (int i = 0; i < n; ++i) out[i] = (double)i * step + start;
}

// ---------------------------------------------------------------------------------------------
// Span sums of the packed layouts.  [H3] "Correctness gates": the fp64 grid of the packed layouts
// is gated bit-exact, and upstream keeps two span sums apart on purpose, a numpy-pairwise one and a
// Python-sequential one, because the two differ in the last ulp from n = 16.  Both are written out
// here in their own arithmetic order (the pages give the order, not the layout that uses them):
//   sequential: s = 0; s = s + x[i] for i = 0, 1, ..., n - 1 (every add rounded in turn)
//   pairwise:   numpy's summation of a contiguous float64 array: fewer than 8 terms are summed left
//               to right from 0; up to 128 terms go into 8 running partial sums (term i into sum
//               i mod 8, over the largest multiple of 8), which are combined as a balanced tree
//               ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)) before the leftover terms are
//               added left to right; above 128 terms the array is cut after m terms, m = n / 2
//               rounded down to a multiple of 8, and the two parts' sums are added.
// ---------------------------------------------------------------------------------------------
double orc_span_sum_sequential(const double* x, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s = s + x[i];
  return s;
}

double orc_span_sum_pairwise(const double* x, int n) {
  if (n < 8) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s = s + x[i];
    return s;
  }
  if (n <= 128) {
    double p[8];
    for (int j = 0; j < 8; ++j) p[j] = x[j];
    const int full = n - n % 8;
    for (int i = 8; i < full; i += 8)
      for (int j = 0; j < 8; ++j) p[j] = p[j] + x[i + j];
    double s = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
    for (int i = full; i < n; ++i) s = s + x[i];
    return s;
  }
  int m = n / 2;
  m -= m % 8;
  return orc_span_sum_pairwise(x, m) + orc_span_sum_pairwise(x + m, n - m);
}

// ---------------------------------------------------------------------------------------------
// Timestep embedding.  READING (pages silent on the formula): the usual DiT sinusoid,
// half = t_dim/2, f_k = exp(-ln(10000) * k / half), e = [cos(1000 t f_k) | sin(1000 t f_k)].
// The ungated SiLU of [H3] "The device-resident forward (W2b)" is applied by the caller.
// Pinned to that reading by closed forms and invariants: t = 0, the quarter and half turn of the
// first pair at t = pi / 2000 and pi / 1000, the unit circle, and the geometric fall of the angles.
// ---------------------------------------------------------------------------------------------
void orc_timestep_embedding(double t, int t_dim, double* out) {
  int half = t_dim / 2;
  for (int k = 0; k < half; ++k) {
    double f = exp(-log(10000.0) * (double)k / (double)half);
    double a = 1000.0 * t * f;
    out[k] = cos(a);
    out[half + k] = sin(a);
  }
}

static inline double silu(double v) { return v / (1.0 + exp(-v)); }

// ---------------------------------------------------------------------------------------------
// Modality-indexed AdaLN conditioning.  [H3] "The device-resident forward (W2b)": an ungated
// SiLU on the conditioning path and two indexed AdaLN modulates.  Per block l and modality m:
//   mod[l][m][:] = W_ada[l][m*6d : (m+1)*6d, :] . silu(e) + b_ada[...]
// split into six d-wide chunks in the order shift1, scale1, gate1, shift2, scale2, gate2 (READING:
// the DiT convention).  The final layer uses [n_mod][2d] = (shift_f, scale_f).
// ---------------------------------------------------------------------------------------------
// With one timestep per modality (the per-modality sigma schedules of [H3] "Milestone: the whole
// t2va path composes end to end": video shift 12, audio 3), the rows of modality m are computed
// from the embedding of t_mod[m].
void orc_adaln_mod(const orc_config* c, const orc_weights* w, const double* t_mod, double* mod, double* mod_final) {
  int d = c->hidden, td = c->t_dim;
  std::vector<double> se((size_t)c->n_mod * td);
  for (int m = 0; m < c->n_mod; ++m) {
    std::vector<double> e(td);
    orc_timestep_embedding(t_mod[m], td, e.data());
    for (int k = 0; k < td; ++k) se[(size_t)m * td + k] = silu(e[k]);
  }
  int rows = c->n_mod * 6 * d;
  for (int l = 0; l < c->n_blocks; ++l) {
    const orc_block* b = &w->blocks[l];
    for (int r = 0; r < rows; ++r) {
      const double* sm = &se[(size_t)(r / (6 * d)) * td];
      double s = 0.0;
      for (int k = 0; k < td; ++k) s += (double)b->w_ada[(size_t)r * td + k] * sm[k];
      if (b->b_ada) s += (double)b->b_ada[r];
      mod[(size_t)l * rows + r] = s;
    }
  }
  int rf = c->n_mod * 2 * d;
  for (int r = 0; r < rf; ++r) {
    const double* sm = &se[(size_t)(r / (2 * d)) * td];
    double s = 0.0;
    for (int k = 0; k < td; ++k) s += (double)w->w_ada_final[(size_t)r * td + k] * sm[k];
    if (w->b_ada_final) s += (double)w->b_ada_final[r];
    mod_final[r] = s;
  }
}

void orc_adaln(const orc_config* c, const orc_weights* w, double t, double* mod, double* mod_final) {
  std::vector<double> tm((size_t)c->n_mod, t);
  orc_adaln_mod(c, w, tm.data(), mod, mod_final);
}

// ---------------------------------------------------------------------------------------------
// Rectified-flow time shift.  [H3] "Milestone: the whole t2va path composes end to end": sigma
// schedules with video shift 12 and audio 3.  READING (the pages name the shift, not its formula):
// the usual rectified-flow shift of a sigma in [0, 1],
//   shift(sigma, s) = s * sigma / (1 + (s - 1) * sigma),
// evaluated in double on the fp32 base sigma and rounded to fp32 by the caller.
// ---------------------------------------------------------------------------------------------
double orc_time_shift(double sigma, double s) { return s * sigma / (1.0 + (s - 1.0) * sigma); }

// ---------------------------------------------------------------------------------------------
// RoPE angles.  [H3] "The device-resident forward (W2b)": plain NeoX rotate_half whose angles come
// from three axes of the fp64 position grid, fed through a per-row cos/sin cache.  [BF] "What this
// enables": rope.inv_freq is a stored tensor (READING: fp32).
//   inv_a[k] = base^(-2k / dim_a), k < dim_a/2, computed in double and rounded to fp32.
//   The per-row angle vector concatenates the axis blocks (t, h, w); theta_j = pos[axis(j)] * inv[j]
//   in double.  cos/sin are returned in double.
// ---------------------------------------------------------------------------------------------
void orc_rope_inv_freq(const orc_config* c, float* inv) {
  int j = 0;
  for (int a = 0; a < c->rope_axes; ++a) {
    int da = c->rope_dims[a];
    for (int k = 0; k < da / 2; ++k) inv[j++] = (float)pow(c->rope_base, -2.0 * (double)k / (double)da);
  }
}

void orc_rope_cos_sin(const orc_config* c, const double* pos, int n_tokens, double* cos_out, double* sin_out) {
  int half = c->rotary_dim / 2;
  std::vector<float> inv(half);
  std::vector<int> axis(half);
  orc_rope_inv_freq(c, inv.data());
  int j = 0;
  for (int a = 0; a < c->rope_axes; ++a)
    for (int k = 0; k < c->rope_dims[a] / 2; ++k) axis[j++] = a;
  for (int r = 0; r < n_tokens; ++r)
    for (int q = 0; q < half; ++q) {
      double th = pos[(size_t)r * 3 + axis[q]] * (double)inv[q];
      cos_out[(size_t)r * half + q] = cos(th);
      sin_out[(size_t)r * half + q] = sin(th);
    }
}

// NeoX rotate_half over the first R = rotary_dim dims of every head, in place; dims >= R pass
// through ([M3] "What moved": ApplyPartialRotary).  For j < R/2 the pair is (x_j, x_{j+R/2}):
//   x'_j       = x_j cos - x_{j+R/2} sin
//   x'_{j+R/2} = x_{j+R/2} cos + x_j sin
void orc_rope_apply(double* x, int n_tokens, int n_heads, int head_dim, int rotary_dim, const double* cs,
                    const double* sn) {
  int half = rotary_dim / 2;
  for (int r = 0; r < n_tokens; ++r)
    for (int h = 0; h < n_heads; ++h) {
      double* v = x + ((size_t)r * n_heads + h) * head_dim;
      for (int j = 0; j < half; ++j) {
        double c0 = cs[(size_t)r * half + j], s0 = sn[(size_t)r * half + j];
        double a = v[j], b = v[j + half];
        v[j] = a * c0 - b * s0;
        v[j + half] = b * c0 + a * s0;
      }
    }
}

// ---------------------------------------------------------------------------------------------
// Norms.  [H3] "The device-resident forward (W2b)": RmsNorm (the CPU reference accumulates in
// double).  READING: no affine weight (the "bare norm" of the AdaLN invariant).
//   RMS(x) = x / sqrt(mean(x^2) + eps)
// [M3] "What moved": LayerNorm for the music DiT: (x - mean) / sqrt(var + eps) * g + b,
// var the biased (population) variance.
// ---------------------------------------------------------------------------------------------
void orc_rms_norm(const double* x, int n, int d, double eps, double* y) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int r = 0; r < n; ++r) {
    const double* xr = x + (size_t)r * d;
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; ++i) y[(size_t)r * d + i] = xr[i] * inv;
  }
}

void orc_layer_norm(const double* x, int n, int d, double eps, const float* g, const float* b, double* y) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int r = 0; r < n; ++r) {
    const double* xr = x + (size_t)r * d;
    double mu = 0.0;
    for (int i = 0; i < d; ++i) mu += xr[i];
    mu /= (double)d;
    double var = 0.0;
    for (int i = 0; i < d; ++i) var += (xr[i] - mu) * (xr[i] - mu);
    var /= (double)d;
    double inv = 1.0 / sqrt(var + eps);
    for (int i = 0; i < d; ++i) {
      double v = (xr[i] - mu) * inv;
      if (g) v *= (double)g[i];
      if (b) v += (double)b[i];
      y[(size_t)r * d + i] = v;
    }
  }
}

// The block norm: RMSNorm or LayerNorm of each row, then the per-channel gain and shift when
// present ([H3] "Update: video-VAE ViT3D decoder complete": rms_norm affine).
static void block_norm(int norm, const double* x, int n, int d, double eps, const float* g, const float* b,
                       double* y) {
  if (norm == 1) {
    orc_layer_norm(x, n, d, eps, g, b, y);
    return;
  }
  orc_rms_norm(x, n, d, eps, y);
  if (g || b)
    for (int r = 0; r < n; ++r)
      for (int i = 0; i < d; ++i) {
        double v = y[(size_t)r * d + i];
        if (g) v *= (double)g[i];
        if (b) v += (double)b[i];
        y[(size_t)r * d + i] = v;
      }
}

// Indexed AdaLN modulate: token r takes the row of its modality tag.
//   y = n * (1 + scale[tag]) + shift[tag]
// shift / scale point at [n_mod] rows of d values, ``stride`` doubles apart.
void orc_modulate(const double* nrm, int n, int d, const uint8_t* tags, const double* shift, const double* scale,
                  size_t stride, double* y) {
  for (int r = 0; r < n; ++r) {
    const double* sh = shift + (size_t)tags[r] * stride;
    const double* sc = scale + (size_t)tags[r] * stride;
    for (int i = 0; i < d; ++i) y[(size_t)r * d + i] = nrm[(size_t)r * d + i] * (1.0 + sc[i]) + sh[i];
  }
}

// ---------------------------------------------------------------------------------------------
// Linear map, MatmulBT: y[i][o] = sum_k x[i][k] * W[o][k] + b[o], W row-major [n_out, k]
// ([M3] "What moved": Linear -> vt::MatmulBT plus a rank-1 bias add).
// ---------------------------------------------------------------------------------------------
void orc_linear(const double* x, int m, int k, const float* W, const float* b, int n_out, double* y) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int i = 0; i < m; ++i) {
    const double* xi = x + (size_t)i * k;
    for (int o = 0; o < n_out; ++o) {
      const float* wo = W + (size_t)o * k;
      double s = 0.0;
      for (int q = 0; q < k; ++q) s += xi[q] * (double)wo[q];
      if (b) s += (double)b[o];
      y[(size_t)i * n_out + o] = s;
    }
  }
}

// 1x1 convolution written as the convolution itself, per document, channel-major:
//   y[co][t] = sum_ci W[co][ci] * x[ci][t] + b[co]
// [M3] "What moved" states that this equals MatmulBT on the frame-major transposed activation;
// the tests check that identity against orc_linear.
void orc_conv1x1(const double* x, int ci, int T, const float* W, const float* b, int co, double* y) {
  for (int o = 0; o < co; ++o)
    for (int t = 0; t < T; ++t) {
      double s = 0.0;
      for (int c = 0; c < ci; ++c) s += (double)W[(size_t)o * ci + c] * x[(size_t)c * T + t];
      if (b) s += (double)b[o];
      y[(size_t)o * T + t] = s;
    }
}

// ---------------------------------------------------------------------------------------------
// Varlen non-causal attention.  [H3] "Correctness gates": vt::DFlashBlockAttention(causal=false)
// over the packed sequence; [M3] "What moved": non-causal attention with no bias.  For each
// document [a, b) and head h, with q, k, v laid [N][H][Dh]:
//   s_ij = q_i . k_j / sqrt(Dh)   for i, j in [a, b)     (READING: the usual 1/sqrt(Dh) scale)
//   p_i  = softmax_j(s_i)         (max-subtracted, double)
//   o_i  = sum_j p_ij v_j
// No mask other than the document block.
// ---------------------------------------------------------------------------------------------
static void attend_row(const double* q, const double* k, const double* v, int H, int Dh, int a, int b, int i,
                       int h, double* o, std::vector<double>& s) {
  int hd = H * Dh;
  double scale = 1.0 / sqrt((double)Dh);
  const double* qi = q + (size_t)i * hd + (size_t)h * Dh;
  double mx = -INFINITY;
  for (int j = a; j < b; ++j) {
    const double* kj = k + (size_t)j * hd + (size_t)h * Dh;
    double acc = 0.0;
    for (int e = 0; e < Dh; ++e) acc += qi[e] * kj[e];
    s[j - a] = acc * scale;
    if (s[j - a] > mx) mx = s[j - a];
  }
  double den = 0.0;
  for (int j = a; j < b; ++j) {
    s[j - a] = exp(s[j - a] - mx);
    den += s[j - a];
  }
  for (int e = 0; e < Dh; ++e) {
    double acc = 0.0;
    for (int j = a; j < b; ++j) acc += s[j - a] * v[(size_t)j * hd + (size_t)h * Dh + e];
    o[e] = acc / den;
  }
}

void orc_attention(const double* q, const double* k, const double* v, int n_tokens, int H, int Dh,
                   const int32_t* cu, int n_docs, double* o) {
  (void)n_tokens;
  for (int dj = 0; dj < n_docs; ++dj) {
    int a = cu[dj], b = cu[dj + 1];
#pragma omp parallel num_threads(g_threads)
    {
      std::vector<double> s(b - a);
#pragma omp for schedule(dynamic, 4)
      for (int idx = 0; idx < (b - a) * H; ++idx) {
        int i = a + idx / H, h = idx % H;
        attend_row(q, k, v, H, Dh, a, b, i, h, o + (size_t)i * H * Dh + (size_t)h * Dh, s);
      }
    }
  }
}

// The same attention for a list of query rows only (out[r] for rows[r], all heads).
void orc_attention_rows(const double* q, const double* k, const double* v, int n_tokens, int H, int Dh,
                        const int32_t* cu, int n_docs, const int32_t* rows, int n_rows, double* o) {
  (void)n_tokens;
#pragma omp parallel num_threads(g_threads)
  {
    std::vector<double> s;
#pragma omp for schedule(dynamic, 1)
    for (int idx = 0; idx < n_rows * H; ++idx) {
      int r = idx / H, h = idx % H, i = rows[r];
      int dj = 0;
      while (!(cu[dj] <= i && i < cu[dj + 1])) ++dj;
      s.resize(cu[dj + 1] - cu[dj]);
      attend_row(q, k, v, H, Dh, cu[dj], cu[dj + 1], i, h, o + (size_t)r * H * Dh + (size_t)h * Dh, s);
    }
  }
  (void)n_docs;
}

// ---------------------------------------------------------------------------------------------
// Gated FFN.  [M3] "What moved" and "Correctness": the FFN computes value * silu(gate) with the
// value in the first half of the merged up projection and the gate in the second half.
//   uv = [u | g] (2F wide);  h = u * silu(g)
// ---------------------------------------------------------------------------------------------
void orc_swiglu(const double* uv, int n, int F, double* hout) {
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < F; ++i) {
      double u = uv[(size_t)r * 2 * F + i], g = uv[(size_t)r * 2 * F + F + i];
      hout[(size_t)r * F + i] = u * silu(g);
    }
}

// ---------------------------------------------------------------------------------------------
// One Euler-ancestral (eta = 0) step of the rectified flow, in fp32 and in exactly this order
// ([H3] "Correctness gates": the euler-ancestral eta0 scheduler and rf_v_to_x0, gated exact):
//   x0 = x - sigma * v
//   x  <- x0 + sigma_next * (x - x0) / sigma      (left to right: (sigma_next * (x - x0)) / sigma)
// Built with -ffp-contract=off so that no product is fused into an add.
// ---------------------------------------------------------------------------------------------
void orc_euler_step(float* x, const float* v, int64_t n, float sigma, float sigma_next) {
  for (int64_t i = 0; i < n; ++i) {
    float sv = sigma * v[i];
    float x0 = x[i] - sv;
    float dx = x[i] - x0;
    float num = sigma_next * dx;
    float q = num / sigma;
    x[i] = x0 + q;
  }
}

// The same step with the sigma pair of each token's modality: row r of x [n_tokens][d] uses
// (sigma[tags[r]], sigma_next[tags[r]]).
void orc_euler_step_tagged(float* x, const float* v, int n_tokens, int d, const uint8_t* tags, const float* sigma,
                           const float* sigma_next) {
  for (int r = 0; r < n_tokens; ++r)
    orc_euler_step(x + (size_t)r * d, v + (size_t)r * d, d, sigma[tags[r]], sigma_next[tags[r]]);
}

// ---------------------------------------------------------------------------------------------
// Latent <-> token packing.  [H3] "Correctness gates": patchify / unpatchify / audio pack / unpack
// are gated exact with a round-trip identity; [H3] "Milestone: the whole t2va path composes end to
// end": unpatchify and audio unpack follow the denoise loop.  [H3] "Encoder complete": a patch
// embedding whose Conv3d has kernel == stride is a plain linear over the flattened patch.
// READING (the pages give neither the order nor the patch): a latent [C][T*pt][H*ph][W*pw] becomes
// T*H*W tokens in (t, h, w) order, w fastest (the packed layout's order); token features are the
// patch flattened as a Conv3d weight [d][C][pt][ph][pw] flattens, (c, a, b, e) with e fastest.
// Audio pack is the same map on a [C][T] latent with H = W = 1 and a 1x1x1 patch: [T][C].
// Pure index permutations; values are copied, never computed.
// ---------------------------------------------------------------------------------------------
void orc_patchify(const float* lat, int C, int T, int H, int W, int pt, int ph, int pw, float* tok) {
  const int P = C * pt * ph * pw;
  const size_t Tf = (size_t)T * pt, Hf = (size_t)H * ph, Wf = (size_t)W * pw;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int w = 0; w < W; ++w) {
        float* row = tok + ((size_t)(t * H + h) * W + w) * P;
        int f = 0;
        for (int c = 0; c < C; ++c)
          for (int a = 0; a < pt; ++a)
            for (int b = 0; b < ph; ++b)
              for (int e = 0; e < pw; ++e)
                row[f++] = lat[(((size_t)c * Tf + (size_t)t * pt + a) * Hf + (size_t)h * ph + b) * Wf +
                               (size_t)w * pw + e];
      }
}

void orc_unpatchify(const float* tok, int C, int T, int H, int W, int pt, int ph, int pw, float* lat) {
  const int P = C * pt * ph * pw;
  const size_t Tf = (size_t)T * pt, Hf = (size_t)H * ph, Wf = (size_t)W * pw;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int w = 0; w < W; ++w) {
        const float* row = tok + ((size_t)(t * H + h) * W + w) * P;
        int f = 0;
        for (int c = 0; c < C; ++c)
          for (int a = 0; a < pt; ++a)
            for (int b = 0; b < ph; ++b)
              for (int e = 0; e < pw; ++e)
                lat[(((size_t)c * Tf + (size_t)t * pt + a) * Hf + (size_t)h * ph + b) * Wf + (size_t)w * pw + e] =
                    row[f++];
      }
}

// ---------------------------------------------------------------------------------------------
// RotaryEmbeddingND positions of the video-VAE decoder.  [H3] "Update: video-VAE ViT3D decoder
// complete": each axis id i of n becomes (i + 0.5) / n mapped into [-1, 1), scaled by 2 pi; the
// per-axis frequency blocks are concatenated and tiled twice (the NeoX rotate_half layout of
// orc_rope_apply).  pos [T*H*W][3] for a T x H x W grid, w fastest, in double:
//   pos_a(i) = (2 * ((i + 0.5) / n_a) - 1) * (2 pi)
// READING: the frequencies are rope_theta^(-2k / dim_a) per axis, as for the DiT's axes.
// ---------------------------------------------------------------------------------------------
void orc_vit_positions(int T, int H, int W, double* pos) {
  const double two_pi = 2.0 * 3.14159265358979323846;
  const int n[3] = {T, H, W};
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int w = 0; w < W; ++w) {
        const int id[3] = {t, h, w};
        double* p = pos + ((size_t)(t * H + h) * W + w) * 3;
        for (int a = 0; a < 3; ++a) p[a] = (2.0 * ((id[a] + 0.5) / (double)n[a]) - 1.0) * two_pi;
      }
}

// ---------------------------------------------------------------------------------------------
// NVFP4 weights.  [H3] "What this push adds" (the NVFP4 checkpoint): each quantized projection
// carries a U8 weight packing two FP4 values per byte (logical [N][K] stored [N][K/2]), an
// F8_E4M3 scale per group of 16 along K ([N][K/16]) and an F32 global scale.
// READINGS: the logical weight is fp4 * e4m3 scale * global (the global scale multiplies); the
// element with the even K index sits in the low nibble.  FP4 is E2M1 (1 sign, 2 exponent bits
// with bias 1, 1 mantissa bit; exponent 0 is subnormal, no inf/NaN); E4M3 is the "fn" form (bias
// 7, exponent 0 subnormal, S.1111.111 NaN, no inf).  Both decoded from those definitions.
// ---------------------------------------------------------------------------------------------
double orc_e2m1_decode(uint8_t code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

double orc_e4m3_decode(uint8_t code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// y [M][N] = x [M][K] W^T + b with W[n][k] = e2m1(q[n][k/2] nibble) * e4m3(s[n][k/16]) * g, in double.
void orc_nvfp4_linear(const double* x, int M, int K, const uint8_t* q, const uint8_t* sc, float g, const float* b,
                      int N, double* y) {
  std::vector<double> W((size_t)N * K);
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      const uint8_t byte = q[(size_t)n * (K / 2) + k / 2];
      const uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      W[(size_t)n * K + k] = orc_e2m1_decode(code) * orc_e4m3_decode(sc[(size_t)n * (K / 16) + k / 16]) * (double)g;
    }
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int i = 0; i < M; ++i)
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += x[(size_t)i * K + k] * W[(size_t)n * K + k];
      if (b) acc += (double)b[n];
      y[(size_t)i * N + n] = acc;
    }
}

// ---------------------------------------------------------------------------------------------
// One transformer block, in place on the fp64 residual x [N][d].  [H3] "The device-resident
// forward (W2b)" lists the ops; with AdaLN on:
//   y  = RMS(x) * (1 + scale1[tag]) + shift1[tag]
//   [q | k | v] = y W_qkv^T + b_qkv          (fused order [q_all | k_all | v_all], heads contiguous)
//   q, k <- NeoX rotate_half with the per-row cos/sin
//   o  = varlen attention(q, k, v)
//   x += gate1[tag] * (o W_o^T + b_o)
//   y2 = RMS(x) * (1 + scale2[tag]) + shift2[tag]
//   h  = u * silu(g),  [u | g] = y2 W_in^T + b_in
//   x += gate2[tag] * (h W_down^T + b_down)
// With AdaLN off (the music DiT, [M3] "What moved"): LayerNorm with (g, b) in place of the
// modulated RMSNorm and plain residual adds in place of the gated ones.
// mod points at this block's [n_mod][6d] row block (NULL when AdaLN is off).
// ---------------------------------------------------------------------------------------------
void orc_block_forward(const orc_config* c, const orc_block* w, const double* mod, double* x, int n,
                       const int32_t* cu, int n_docs, const uint8_t* tags, const double* cs, const double* sn) {
  int d = c->hidden, F = c->ffn_hidden, H = c->n_heads, Dh = c->head_dim;
  size_t md = (size_t)6 * d;
  std::vector<double> nrm((size_t)n * d), y((size_t)n * d), qkv((size_t)n * 3 * d);
  std::vector<double> q((size_t)n * d), k((size_t)n * d), v((size_t)n * d), o((size_t)n * d), t((size_t)n * d);
  block_norm(c->norm, x, n, d, c->norm_eps, w->ln1_g, w->ln1_b, nrm.data());
  if (c->adaln)
    orc_modulate(nrm.data(), n, d, tags, mod + 0 * d, mod + 1 * d, md, y.data());
  else
    y = nrm;
  orc_linear(y.data(), n, d, w->w_qkv, w->b_qkv, 3 * d, qkv.data());
  for (int r = 0; r < n; ++r)
    for (int h = 0; h < H; ++h)
      for (int j = 0; j < Dh; ++j) {
        const size_t o = (size_t)r * d + (size_t)h * Dh + j, row = (size_t)r * 3 * d;
        if (c->qkv_interleaved) {  // the ViT's qkv.view(S, H, 3 Dh).chunk(3): [q_h | k_h | v_h] per head
          q[o] = qkv[row + (size_t)h * 3 * Dh + j];
          k[o] = qkv[row + (size_t)h * 3 * Dh + Dh + j];
          v[o] = qkv[row + (size_t)h * 3 * Dh + 2 * Dh + j];
        } else {
          q[o] = qkv[row + (size_t)h * Dh + j];
          k[o] = qkv[row + d + (size_t)h * Dh + j];
          v[o] = qkv[row + 2 * d + (size_t)h * Dh + j];
        }
      }
  if (c->qk_norm)  // per-head RMS norm of q and k over Dh, no affine ([H3] "Update: video-VAE decoder block ported")
    for (std::vector<double>* m : {&q, &k})
      for (int r = 0; r < n; ++r)
        for (int h = 0; h < H; ++h) {
          double* p = m->data() + (size_t)r * d + (size_t)h * Dh;
          double ss = 0.0;
          for (int j = 0; j < Dh; ++j) ss += p[j] * p[j];
          const double inv = 1.0 / sqrt(ss / (double)Dh + c->norm_eps);
          for (int j = 0; j < Dh; ++j) p[j] *= inv;
        }
  orc_rope_apply(q.data(), n, H, Dh, c->rotary_dim, cs, sn);
  orc_rope_apply(k.data(), n, H, Dh, c->rotary_dim, cs, sn);
  orc_attention(q.data(), k.data(), v.data(), n, H, Dh, cu, n_docs, o.data());
  orc_linear(o.data(), n, d, w->w_o, w->b_o, d, t.data());
  for (int r = 0; r < n; ++r) {
    const double* g1 = c->adaln ? mod + (size_t)tags[r] * md + 2 * d : nullptr;
    for (int i = 0; i < d; ++i)
      x[(size_t)r * d + i] += (g1 ? g1[i] : (w->res1 ? (double)w->res1[i] : 1.0)) * t[(size_t)r * d + i];
  }
  block_norm(c->norm, x, n, d, c->norm_eps, w->ln2_g, w->ln2_b, nrm.data());
  if (c->adaln)
    orc_modulate(nrm.data(), n, d, tags, mod + 3 * d, mod + 4 * d, md, y.data());
  else
    y = nrm;
  std::vector<double> uv((size_t)n * 2 * F), hh((size_t)n * F);
  orc_linear(y.data(), n, d, w->w_in, w->b_in, 2 * F, uv.data());
  orc_swiglu(uv.data(), n, F, hh.data());
  orc_linear(hh.data(), n, F, w->w_down, w->b_down, d, t.data());
  for (int r = 0; r < n; ++r) {
    const double* g2 = c->adaln ? mod + (size_t)tags[r] * md + 5 * d : nullptr;
    for (int i = 0; i < d; ++i)
      x[(size_t)r * d + i] += (g2 ? g2[i] : (w->res2 ? (double)w->res2[i] : 1.0)) * t[(size_t)r * d + i];
  }
}

// ---------------------------------------------------------------------------------------------
// Whole forward.  x_in: token-major [N][d] fp32, or, when io_channels > 0, channel-major per
// document ([io][len_j] blocks back to back).  out has the same layout and size as x_in.
// Final layer (READING: the configs give no latent widths, so the patch embedding and output heads
// are not part of this forward): with AdaLN, out = RMS(x) * (1 + scale_f[tag]) + shift_f[tag];
// without it, out = LN_f(x), then the 1x1 post-convolution back to io channels.
// dumps (may be NULL) receives the residual after each block, [L][N][d].
// Returns the layout check's code (0 when valid).
// ---------------------------------------------------------------------------------------------
static void forward_core(const orc_config* c, const orc_weights* w, std::vector<double>& x, int n, const int32_t* cu,
                         int n_docs, const uint8_t* tags, const double* pos, const double* t_mod, double* out,
                         double* dumps);

int orc_forward_mod(const orc_config* c, const orc_weights* w, const float* x_in, int n, const int32_t* cu,
                    int n_docs, const int32_t* doc_ids, const uint8_t* tags, const double* pos, const double* t_mod,
                    double* out, double* dumps) {
  int rc = orc_check_layout(cu, n_docs, doc_ids, tags, n, c->adaln ? c->n_mod : 1);
  if (rc) return rc;
  int d = c->hidden;
  std::vector<double> x((size_t)n * d);
  if (c->io_channels > 0) {
    int ci = c->io_channels;
    for (int j = 0; j < n_docs; ++j) {
      int a = cu[j], len = cu[j + 1] - cu[j];
      std::vector<double> xin((size_t)ci * len), yd((size_t)d * len);
      for (size_t e = 0; e < xin.size(); ++e) xin[e] = (double)x_in[(size_t)ci * a + e];
      orc_conv1x1(xin.data(), ci, len, w->w_pre, w->b_pre, d, yd.data());
      for (int s = 0; s < len; ++s)
        for (int o = 0; o < d; ++o) x[(size_t)(a + s) * d + o] = yd[(size_t)o * len + s];
    }
  } else {
    for (size_t e = 0; e < x.size(); ++e) x[e] = (double)x_in[e];
  }
  forward_core(c, w, x, n, cu, n_docs, tags, pos, t_mod, out, dumps);
  return 0;
}

// The forward from the residual x [N][d] (already embedded) to the final layer's output.
static void forward_core(const orc_config* c, const orc_weights* w, std::vector<double>& x, int n, const int32_t* cu,
                         int n_docs, const uint8_t* tags, const double* pos, const double* t_mod, double* out,
                         double* dumps) {
  int d = c->hidden, half = c->rotary_dim / 2;
  std::vector<double> cs((size_t)n * half), sn((size_t)n * half);
  orc_rope_cos_sin(c, pos, n, cs.data(), sn.data());
  std::vector<double> mod, modf;
  if (c->adaln) {
    mod.resize((size_t)c->n_blocks * c->n_mod * 6 * d);
    modf.resize((size_t)c->n_mod * 2 * d);
    orc_adaln_mod(c, w, t_mod, mod.data(), modf.data());
  }
  for (int l = 0; l < c->n_blocks; ++l) {
    const double* ml = c->adaln ? mod.data() + (size_t)l * c->n_mod * 6 * d : nullptr;
    orc_block_forward(c, &w->blocks[l], ml, x.data(), n, cu, n_docs, tags, cs.data(), sn.data());
    if (dumps) memcpy(dumps + (size_t)l * n * d, x.data(), sizeof(double) * (size_t)n * d);
  }
  std::vector<double> nrm((size_t)n * d);
  if (c->adaln) {
    orc_rms_norm(x.data(), n, d, c->norm_eps, nrm.data());
    orc_modulate(nrm.data(), n, d, tags, modf.data(), modf.data() + d, (size_t)2 * d, out);
  } else {
    const int fnorm = c->final_norm == 0 ? c->norm : c->final_norm - 1;  // 0 RMS, 1 LN
    block_norm(fnorm, x.data(), n, d, c->norm_eps, w->lnf_g, w->lnf_b, nrm.data());
    if (c->io_channels > 0) {
      int co = c->io_channels;
      for (int j = 0; j < n_docs; ++j) {
        int a = cu[j], len = cu[j + 1] - cu[j];
        std::vector<double> xd((size_t)d * len), yd((size_t)co * len);
        for (int s = 0; s < len; ++s)
          for (int o = 0; o < d; ++o) xd[(size_t)o * len + s] = nrm[(size_t)(a + s) * d + o];
        orc_conv1x1(xd.data(), d, len, w->w_post, w->b_post, co, yd.data());
        memcpy(out + (size_t)co * a, yd.data(), sizeof(double) * yd.size());
      }
    } else {
      memcpy(out, nrm.data(), sizeof(double) * nrm.size());
    }
  }
}

int orc_forward(const orc_config* c, const orc_weights* w, const float* x_in, int n, const int32_t* cu, int n_docs,
                const int32_t* doc_ids, const uint8_t* tags, const double* pos, double t, double* out,
                double* dumps) {
  std::vector<double> tm((size_t)(c->n_mod > 0 ? c->n_mod : 1), t);
  return orc_forward_mod(c, w, x_in, n, cu, n_docs, doc_ids, tags, pos, tm.data(), out, dumps);
}

// ---------------------------------------------------------------------------------------------
// The forward between latent tokens.  [H3] "What this push adds": both patch projections and both
// output heads stay fp32 islands around the bf16 block stream.  For each modality m the rows of
// the packed sequence with tag m, in increasing order, are the rows of z[m] [rows_m][width[m]]:
//   x[row]  = z[m][r] W_patch[m]^T + b_patch[m]          (W_patch[m] [d][width[m]])
//   out     = the forward of x (blocks and the final layer)
//   v[m][r] = out[row] W_head[m]^T + b_head[m]           (W_head[m] [width[m]][d])
// everything in double.  n_rows[m] must equal the number of tokens tagged m (else code 8).
// ---------------------------------------------------------------------------------------------
int orc_forward_latent(const orc_config* c, const orc_weights* w, int n_mod, const float* const* z,
                       const int* n_rows, const int* width, const float* const* w_patch, const float* const* b_patch,
                       const float* const* w_head, const float* const* b_head, int n, const int32_t* cu, int n_docs,
                       const int32_t* doc_ids, const uint8_t* tags, const double* pos, const double* t_mod,
                       double* const* v_out, double* dumps) {
  int rc = orc_check_layout(cu, n_docs, doc_ids, tags, n, n_mod);
  if (rc) return rc;
  const int d = c->hidden;
  std::vector<std::vector<int>> rows((size_t)n_mod);
  for (int i = 0; i < n; ++i) rows[tags[i]].push_back(i);
  for (int m = 0; m < n_mod; ++m)
    if ((int)rows[m].size() != n_rows[m]) return 8;
  std::vector<double> x((size_t)n * d);
  for (int m = 0; m < n_mod; ++m) {
    const int M = n_rows[m], K = width[m];
    if (M == 0) continue;
    std::vector<double> zm((size_t)M * K), xm((size_t)M * d);
    for (size_t e = 0; e < zm.size(); ++e) zm[e] = (double)z[m][e];
    orc_linear(zm.data(), M, K, w_patch[m], b_patch[m], d, xm.data());
    for (int r = 0; r < M; ++r) memcpy(&x[(size_t)rows[m][r] * d], &xm[(size_t)r * d], sizeof(double) * d);
  }
  std::vector<double> out((size_t)n * d);
  forward_core(c, w, x, n, cu, n_docs, tags, pos, t_mod, out.data(), dumps);
  for (int m = 0; m < n_mod; ++m) {
    const int M = n_rows[m];
    if (M == 0) continue;
    std::vector<double> om((size_t)M * d);
    for (int r = 0; r < M; ++r) memcpy(&om[(size_t)r * d], &out[(size_t)rows[m][r] * d], sizeof(double) * d);
    orc_linear(om.data(), M, d, w_head[m], b_head[m], width[m], v_out[m]);
  }
  return 0;
}

}  // extern "C"
