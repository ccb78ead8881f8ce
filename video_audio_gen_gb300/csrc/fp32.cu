// The fp32 forward path: the music DiT shape of [M3] "What moved" (fp32 stays fp32: every weight and
// activation is fp32; LayerNorm, partial rotary, non-causal attention with no bias,
// value * silu(gate), 1x1 pre/post convolutions as MatmulBT on the frame-major activation).
// A single TF32 product would round operands to 10 mantissa bits, far above the 1e-5 tolerance;
// three of them on split operands (3xTF32) keep fp32-level accuracy on the tensor cores:
//   tf32_split_kernel       x -> tf32(x), tf32(x - tf32(x)) (the latent islands' operands)
//   f16_split_kernel        x -> f16 hi and lo parts of x * 2^e (the forward's operands: weights once
//                           at bind with a per-tensor e, activations per GEMM with a fixed e)
//   x3_partial_kernel       three products per fp32 product on the tcgen05 tensor cores, kind::tf32
//                           or kind::f16, 12-MMA accumulation chunks summed in fp32; split-K, each
//                           split writes its partial sums to a [S][M][N] buffer
//   sgemm_reduce_*          sums the S partials in a fixed order and applies the epilogue (bias,
//                           residual add, NeoX RoPE + q/k/v split, value * silu(gate))
//   attention_f32_kernel    exact fp32 online softmax with expf; keys and values staged in shared memory
//   io_transpose_kernel     channel-major [io, len] per document <-> frame-major [N, io]
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

#include <math.h>

namespace dit {

namespace {

__device__ __forceinline__ float sum_parts(const float* __restrict__ part, int S, size_t MN, size_t idx) {
  float v = 0.f;
  for (int s = 0; s < S; ++s) v += part[(size_t)s * MN + idx];
  return v;
}

// Sum of the S partials of the four consecutive elements at idx (a multiple of 4), in split order.
__device__ __forceinline__ float4 sum_parts4(const float* __restrict__ part, int S, size_t MN, size_t idx) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < S; ++s) {
    const float4 p = __ldcs(reinterpret_cast<const float4*>(part + (size_t)s * MN + idx));
    v.x += p.x;
    v.y += p.y;
    v.z += p.z;
    v.w += p.w;
  }
  return v;
}

// The reductions run on a 2-D grid: x = 4-column groups of a row (256 threads, 1024 columns per
// block), y = rows (grid-stride), so no index needs a 64-bit division.  N is a multiple of 4.
// out = sum + bias (add = 0: store into out [M, N]; add = 1: out[M, N] += sum + bias).  With `lo`
// the residual is a compensated pair (out = high part, lo = low part): the add is an exact TwoSum
// whose rounding error goes into lo, so the residual stream keeps about twice fp32's precision.
__global__ void sgemm_reduce_store_kernel(const float* __restrict__ part, int S, int M, int N,
                                          const float* __restrict__ bias, float* __restrict__ out, int add,
                                          float* __restrict__ lo, const int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t MN = (size_t)M * N;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (c >= N) return;
  const float4 b4 = bias ? *reinterpret_cast<const float4*>(bias + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = blockIdx.y; r < M; r += gridDim.y) {
    const size_t i = (size_t)r * N + c;
    const float4 p = sum_parts4(part, S, MN, i);
    const float v[4] = {p.x + b4.x, p.y + b4.y, p.z + b4.z, p.w + b4.w};
    float4* o4 = reinterpret_cast<float4*>(out + i);
    if (!add) {
      *o4 = make_float4(v[0], v[1], v[2], v[3]);
      if (lo) *reinterpret_cast<float4*>(lo + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (lo) {
      const float4 a4 = *o4, l4 = *reinterpret_cast<const float4*>(lo + i);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w}, l[4] = {l4.x, l4.y, l4.z, l4.w};
      float so[4], lo_[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float s = __fadd_rn(a[e], v[e]);
        const float bb = __fsub_rn(s, a[e]);
        const float err = __fadd_rn(__fsub_rn(a[e], __fsub_rn(s, bb)), __fsub_rn(v[e], bb));
        so[e] = s;
        lo_[e] = __fadd_rn(l[e], err);
      }
      *o4 = make_float4(so[0], so[1], so[2], so[3]);
      *reinterpret_cast<float4*>(lo + i) = make_float4(lo_[0], lo_[1], lo_[2], lo_[3]);
    } else {
      const float4 a4 = *o4;
      *o4 = make_float4(a4.x + v[0], a4.y + v[1], a4.z + v[2], a4.w + v[3]);
    }
  }
}

// The split reduction of an fp32 GEMM whose output is added into the residual stream, fused with the
// LayerNorm (or RMSNorm) that reads that stream next: one CTA per row (grid-stride), 256 threads of
// VPT float4 each (d = 1024 * VPT).
//   resid (+)= sum of the S partials + bias       (add = 0: resid = ..., resid_lo = 0; add = 1: the
//                                                  compensated TwoSum add of sgemm_reduce_store_kernel)
//   y = norm(resid + resid_lo) * g + b             (out_kind 1: fp32 [M][d]; 3: the next 3xF16
//                                                  GEMM's token-tiled split operand)
// The norm is the one of norm_mod_persistent_kernel on the compensated input, without modulation.
template <int VPT>
__global__ void __launch_bounds__(256) sgemm_reduce_resid_norm_kernel(
    const float* __restrict__ part, int S, int M, int d, const float* __restrict__ bias, float* __restrict__ resid,
    float* __restrict__ resid_lo, int add, int norm, float eps, const float* __restrict__ g,
    const float* __restrict__ b, void* y, int out_kind, int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  __shared__ float red[2][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t MN = (size_t)M * d;
  int parity = 0;
  auto block_sum = [&](float s) -> float {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) red[parity][warp] = s;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[parity][w];
    parity ^= 1;
    return t;
  };
  const int nt = x3_token_tile(M), mt = (M + nt - 1) / nt;
  bool over = false;
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    float4 cur[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = (i * 256 + threadIdx.x) * 4;
      const size_t at = (size_t)row * d + c;
      const float4 p = sum_parts4(part, S, MN, at);
      const float4 b4 = bias ? *reinterpret_cast<const float4*>(bias + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float v[4] = {p.x + b4.x, p.y + b4.y, p.z + b4.z, p.w + b4.w};
      float hi[4], lo[4];
      if (!add) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hi[e] = v[e];
          lo[e] = 0.f;
        }
      } else {
        const float4 a4 = *reinterpret_cast<const float4*>(resid + at);
        const float4 l4 = *reinterpret_cast<const float4*>(resid_lo + at);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w}, lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float s = __fadd_rn(av[e], v[e]);
          const float bb = __fsub_rn(s, av[e]);
          const float err = __fadd_rn(__fsub_rn(av[e], __fsub_rn(s, bb)), __fsub_rn(v[e], bb));
          hi[e] = s;
          lo[e] = __fadd_rn(lv[e], err);
        }
      }
      *reinterpret_cast<float4*>(resid + at) = make_float4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<float4*>(resid_lo + at) = make_float4(lo[0], lo[1], lo[2], lo[3]);
      cur[i] = make_float4(hi[0] + lo[0], hi[1] + lo[1], hi[2] + lo[2], hi[3] + lo[3]);
    }
    float mean = 0.f;
    if (norm == 1) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < VPT; ++i) s += (cur[i].x + cur[i].y) + (cur[i].z + cur[i].w);
      mean = block_sum(s) / (float)d;
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const float a0 = cur[i].x - mean, a1 = cur[i].y - mean, a2 = cur[i].z - mean, a3 = cur[i].w - mean;
      ss += a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
    }
    const float inv = 1.0f / sqrtf(block_sum(ss) / (float)d + eps);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = (i * 256 + threadIdx.x) * 4;
      float o[4] = {(cur[i].x - mean) * inv, (cur[i].y - mean) * inv, (cur[i].z - mean) * inv,
                    (cur[i].w - mean) * inv};
      if (g) {
        const float4 gg = *reinterpret_cast<const float4*>(g + c);
        o[0] *= gg.x; o[1] *= gg.y; o[2] *= gg.z; o[3] *= gg.w;
      }
      if (b) {
        const float4 bb = *reinterpret_cast<const float4*>(b + c);
        o[0] += bb.x; o[1] += bb.y; o[2] += bb.z; o[3] += bb.w;
      }
      if (out_kind == 3) {
        const size_t xi = x3_xs_index(row, c, nt, mt);
        uint16_t* xs = static_cast<uint16_t*>(y);
        over |= store_f16_split4(o, kF16x3ActExp, xs + xi, xs + xi + (size_t)nt * 32);
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)row * d + c) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  if (over && status) atomicOr(status, kDevRange);
}

// [q | k | v] = sum + bias, NeoX rotate_half over the first R = 2 half dims of each q/k head, stored
// fp32 [M, d] each.  A 4-column group never straddles a head, a segment or the rotary boundary
// (d, Dh and half are multiples of 4).
__global__ void sgemm_reduce_qkv_kernel(const float* __restrict__ part, int S, int M, int d, int Dh, int half,
                                        const float* __restrict__ bias, const float* __restrict__ cs,
                                        const float* __restrict__ sn, float* __restrict__ q, float* __restrict__ k,
                                        float* __restrict__ v, const int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const int N = 3 * d;
  const size_t MN = (size_t)M * N;
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (c0 >= N) return;
  const int seg = c0 / d, cc = c0 - seg * d;
  const int jd = cc % Dh;  // dim within the head
  const bool rot = seg < 2 && jd < 2 * half;
  const int j = jd < half ? jd : jd - half;
  const int pc = jd < half ? c0 + half : c0 - half;  // partner columns
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 b4 = bias ? *reinterpret_cast<const float4*>(bias + c0) : zero;
  const float4 pb4 = bias && rot ? *reinterpret_cast<const float4*>(bias + pc) : zero;
  float* dst = seg == 0 ? q : (seg == 1 ? k : v);
  for (int r = blockIdx.y; r < M; r += gridDim.y) {
    float4 x = sum_parts4(part, S, MN, (size_t)r * N + c0);
    x = make_float4(x.x + b4.x, x.y + b4.y, x.z + b4.z, x.w + b4.w);
    if (rot) {
      float4 y = sum_parts4(part, S, MN, (size_t)r * N + pc);
      y = make_float4(y.x + pb4.x, y.y + pb4.y, y.z + pb4.z, y.w + pb4.w);
      const float4 co = *reinterpret_cast<const float4*>(cs + (size_t)r * half + j);
      const float4 si = *reinterpret_cast<const float4*>(sn + (size_t)r * half + j);
      if (jd < half)
        x = make_float4(x.x * co.x - y.x * si.x, x.y * co.y - y.y * si.y, x.z * co.z - y.z * si.z,
                        x.w * co.w - y.w * si.w);
      else
        x = make_float4(x.x * co.x + y.x * si.x, x.y * co.y + y.y * si.y, x.z * co.z + y.z * si.z,
                        x.w * co.w + y.w * si.w);
    }
    *reinterpret_cast<float4*>(dst + (size_t)r * d + cc) = x;
  }
}

// h[r, f] = (u + b_u) * silu(g + b_g): value columns [0, F), gate columns [F, 2F).  With h_split the
// result goes out as the 3xF16 GEMM's f16 (hi, lo) operand, four features per thread (F % 4 == 0).
__global__ void sgemm_reduce_swiglu_kernel(const float* __restrict__ part, int S, int M, int F,
                                           const float* __restrict__ bias, float* __restrict__ h,
                                           uint16_t* __restrict__ h_split, int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t MN = (size_t)M * 2 * F;
  const int f0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (f0 >= F) return;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 bu = bias ? *reinterpret_cast<const float4*>(bias + f0) : zero;
  const float4 bg = bias ? *reinterpret_cast<const float4*>(bias + F + f0) : zero;
  bool over = false;
  const int nt = x3_token_tile(M), mt = (M + nt - 1) / nt;
  for (int r = blockIdx.y; r < M; r += gridDim.y) {
    const float4 u4 = sum_parts4(part, S, MN, (size_t)r * 2 * F + f0);
    const float4 g4 = sum_parts4(part, S, MN, (size_t)r * 2 * F + F + f0);
    const float u[4] = {u4.x + bu.x, u4.y + bu.y, u4.z + bu.z, u4.w + bu.w};
    const float g[4] = {g4.x + bg.x, g4.y + bg.y, g4.z + bg.z, g4.w + bg.w};
    float hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) hv[e] = u[e] * (g[e] / (1.0f + expf(-g[e])));
    if (h_split) {
      const size_t xi = x3_xs_index(r, f0, nt, mt);
      over |= store_f16_split4(hv, kF16x3ActExp, h_split + xi, h_split + xi + (size_t)nt * 32);
    } else {
      *reinterpret_cast<float4*>(h + (size_t)r * F + f0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    }
  }
  if (over && status) atomicOr(status, kDevRange);
}

// Exact fp32 softmax attention over the document of each row.  One CTA per (document, 128-row
// q-tile, head, 16-row block), 4 warps of 4 query rows each.  The document's keys and values pass
// through shared memory 32 at a time (lane j scores key j of the chunk for all 4 rows of its warp);
// every row keeps an exact fp32 online softmax (running max m, sum l, accumulator o, each chunk
// rescaled by exp(m_old - m_new)):
//     o_i = sum_j exp(s_ij - m_i) v_j / sum_j exp(s_ij - m_i),   s_ij = q_i . k_j / sqrt(Dh)
// Lane l accumulates output dims [l * DH / 32, (l + 1) * DH / 32).  The next chunk's keys and values
// are loaded into registers while the current one is scored.
constexpr int AF_KC = 32;      // keys per chunk
constexpr int AF_ROWS = 4;     // query rows per warp
constexpr int AF_WARPS = 4;
constexpr int AF_CTA_ROWS = AF_ROWS * AF_WARPS;  // 16
constexpr int AF_BLOCKS = 128 / AF_CTA_ROWS;     // CTAs per 128-row item of the schedule

template <int DH>
__host__ __device__ constexpr int af_kstride() {
  return DH + 4;  // float4 rows; lanes 8 apart fall in one 128-byte phase, conflict-free
}

template <int DH>
constexpr int af_smem_bytes() {
  return (AF_KC * af_kstride<DH>() + AF_KC * DH + AF_WARPS * AF_ROWS * DH) * 4;
}

template <int DH>
__global__ void __launch_bounds__(AF_WARPS * 32) attention_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v, const int32_t* __restrict__ cu,
    const int2* __restrict__ items, const int* __restrict__ count, int n_tokens, int H, float scale,
    float* __restrict__ o, uint16_t* __restrict__ o_split, int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  constexpr int PL = DH / 32;
  constexpr int KS = af_kstride<DH>();
  constexpr int D4 = DH / 4;
  constexpr int LD = AF_KC * D4 / (AF_WARPS * 32);  // float4 of K (and of V) per thread per chunk
  static_assert(AF_KC * D4 % (AF_WARPS * 32) == 0, "chunk load must divide evenly");
  extern __shared__ float4 af_smem4[];
  float* sk = reinterpret_cast<float*>(af_smem4);  // [KC][KS]
  float* sv = sk + AF_KC * KS;                     // [KC][DH]
  float* sq = sv + AF_KC * DH;                     // [warps][rows][DH]
  const int blk = blockIdx.x % AF_BLOCKS, item_idx = blockIdx.x / AF_BLOCKS, h = blockIdx.y;
  if (item_idx >= *count) return;
  const int2 it = items[item_idx];
  const int a = cu[it.x], b = cu[it.x + 1];
  const int d = H * DH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = it.y + blk * AF_CTA_ROWS + warp * AF_ROWS;  // this warp's first row
  if (it.y + blk * AF_CTA_ROWS >= b) return;                  // the whole CTA is past the document's end
  float* myq = sq + warp * AF_ROWS * DH;
#pragma unroll
  for (int t = lane; t < AF_ROWS * D4; t += 32) {
    const int i = t / D4, e4 = t - i * D4;
    const int r = r0 + i;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < b) x = *reinterpret_cast<const float4*>(q + (size_t)r * d + h * DH + e4 * 4);
    *reinterpret_cast<float4*>(myq + i * DH + e4 * 4) = x;
  }
  float4 nk4[LD], nv4[LD];
  auto fetch = [&](int c0) {
#pragma unroll
    for (int u = 0; u < LD; ++u) {
      const int t = threadIdx.x + u * AF_WARPS * 32;
      const int j = t / D4, e4 = t - j * D4;
      nk4[u] = nv4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 + j < b) {
        const size_t at = (size_t)(c0 + j) * d + h * DH + e4 * 4;
        nk4[u] = *reinterpret_cast<const float4*>(k + at);
        nv4[u] = *reinterpret_cast<const float4*>(v + at);
      }
    }
  };
  float m[AF_ROWS], l[AF_ROWS], acc[AF_ROWS][PL];
#pragma unroll
  for (int i = 0; i < AF_ROWS; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[i][e] = 0.f;
  }
  fetch(a);
  for (int c0 = a; c0 < b; c0 += AF_KC) {
    const int nk = b - c0 < AF_KC ? b - c0 : AF_KC;
    __syncthreads();  // the previous chunk is no longer read
#pragma unroll
    for (int u = 0; u < LD; ++u) {
      const int t = threadIdx.x + u * AF_WARPS * 32;
      const int j = t / D4, e4 = t - j * D4;
      *reinterpret_cast<float4*>(sk + j * KS + e4 * 4) = nk4[u];
      *reinterpret_cast<float4*>(sv + j * DH + e4 * 4) = nv4[u];
    }
    __syncthreads();
    if (c0 + AF_KC < b) fetch(c0 + AF_KC);
    // four partial sums per row (4-dim groups e4 mod 4) quarter the dependent FMA chains
    float s[AF_ROWS], sp[4][AF_ROWS];
#pragma unroll
    for (int i = 0; i < AF_ROWS; ++i) sp[0][i] = sp[1][i] = sp[2][i] = sp[3][i] = 0.f;
    const float4* kj = reinterpret_cast<const float4*>(sk + lane * KS);
#pragma unroll 2
    for (int e4 = 0; e4 < D4; e4 += 4) {
      float4 kv[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) kv[g] = kj[e4 + g];
#pragma unroll
      for (int i = 0; i < AF_ROWS; ++i) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 qv = reinterpret_cast<const float4*>(myq + i * DH)[e4 + g];
          sp[g][i] = fmaf(qv.x, kv[g].x, sp[g][i]);
          sp[g][i] = fmaf(qv.y, kv[g].y, sp[g][i]);
          sp[g][i] = fmaf(qv.z, kv[g].z, sp[g][i]);
          sp[g][i] = fmaf(qv.w, kv[g].w, sp[g][i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < AF_ROWS; ++i) s[i] = (sp[0][i] + sp[1][i]) + (sp[2][i] + sp[3][i]);
    float p[AF_ROWS];
#pragma unroll
    for (int i = 0; i < AF_ROWS; ++i) {
      const float si = lane < nk ? s[i] * scale : -INFINITY;
      float cm = si;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      const float mn = fmaxf(m[i], cm);
      const float alpha = expf(m[i] - mn);  // 0 on the first chunk (m = -inf)
      p[i] = lane < nk ? expf(si - mn) : 0.f;
      float ps = p[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[i] = l[i] * alpha + ps;
#pragma unroll
      for (int e = 0; e < PL; ++e) acc[i][e] *= alpha;
      m[i] = mn;
    }
#pragma unroll 4
    for (int j = 0; j < nk; ++j) {
      float vv[PL];
      if constexpr (PL == 4) {
        const float4 x = reinterpret_cast<const float4*>(sv + j * DH)[lane];
        vv[0] = x.x; vv[1] = x.y; vv[2] = x.z; vv[3] = x.w;
      } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) vv[e] = sv[j * DH + lane * PL + e];
      }
#pragma unroll
      for (int i = 0; i < AF_ROWS; ++i) {
        const float pj = __shfl_sync(0xffffffffu, p[i], j);
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[i][e] = fmaf(pj, vv[e], acc[i][e]);
      }
    }
  }
  bool over = false;
  const int xnt = x3_token_tile(n_tokens), xmt = (n_tokens + xnt - 1) / xnt;
#pragma unroll
  for (int i = 0; i < AF_ROWS; ++i) {
    const int r = r0 + i;
    if (r >= b) continue;
    const float inv = 1.0f / l[i];
    float ov[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) ov[e] = acc[i][e] * inv;
    const size_t at = (size_t)r * d + h * DH + lane * PL;
    if (o_split) {
      if constexpr (PL % 4 == 0) {
#pragma unroll
        for (int e = 0; e < PL; e += 4) {
          const float v4[4] = {ov[e], ov[e + 1], ov[e + 2], ov[e + 3]};
          const size_t xi = x3_xs_index(r, h * DH + lane * PL + e, xnt, xmt);
          over |= store_f16_split4(v4, kF16x3ActExp, o_split + xi, o_split + xi + (size_t)xnt * 32);
        }
      } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) {
          const float x = ldexpf(ov[e], kF16x3ActExp);
          over |= fabsf(x) > kF16Max;
          const __half hh = __float2half_rn(x);
          const size_t xi = x3_xs_index(r, h * DH + lane * PL + e, xnt, xmt);
          o_split[xi] = __half_as_ushort(hh);
          o_split[xi + (size_t)xnt * 32] = __half_as_ushort(__float2half_rn(__fsub_rn(x, __half2float(hh))));
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < PL; ++e) o[at + e] = ov[e];
    }
  }
  if (over && status) atomicOr(status, kDevRange);
}

// to_frames = 1: channel-major per document (document j is [io, len_j] at offset io * cu[j]) ->
// frame-major [N, io].  to_frames = 0: the reverse.
__global__ void io_transpose_kernel(const float* __restrict__ src, float* __restrict__ dst, const int32_t* __restrict__ cu,
                                    const int32_t* __restrict__ doc_ids, int n, int io, int to_frames,
                                    const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t total = (size_t)n * io;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / io), c = (int)(e - (size_t)t * io);  // frame t, channel c
    const int j = doc_ids[t];
    const int a = cu[j], len = cu[j + 1] - a;
    const size_t cm = (size_t)io * a + (size_t)c * len + (t - a);
    if (to_frames)
      dst[e] = src[cm];
    else
      dst[cm] = src[e];
  }
}

// ------------------------------------------------------------------------------------------
// Three-product partial GEMM on the tcgen05 tensor cores.  Every fp32 operand x is split into a high
// and a low part of a narrower type T, x ~ x_hi + x_lo, and
//     a . b  ~=  a_hi b_hi + a_hi b_lo + a_lo b_hi
// drops only a_lo b_lo and the rounding of the low parts, about 2^-21 of |a b| per product when T
// has an 11-bit significand.  Two types serve:
//   tf32 (kind::tf32, 32 K per 128-byte row): x_hi = tf32(x), x_lo = tf32(x - x_hi)
//   f16  (kind::f16,  32 K per 64-byte row):  x_hi = f16(x 2^e), x_lo = f16(x 2^e - x_hi), with e
//        chosen so that both parts stay in f16's normal range (per weight tensor from its largest
//        magnitude; a fixed e for activations); the sums are scaled back by 2^-(e_w + e_x), exactly.
//        kind::f16 runs at twice the tf32 rate and its two parts take 4 bytes per weight, so the
//        weight stream is half of tf32's.
// The tensor core's fp32 accumulation of these products is biased (measured on GB300: the error
// of a TMEM accumulation grows linearly with its depth, about 2e-5 relative at K = 2048), so the
// MMAs accumulate only one stage (32 K: 2 f16 or 4 tf32 K-steps x 3 products), in turn into as many
// TMEM accumulators as fit (2 to 4), and the epilogue adds each
// chunk into fp32 running sums in registers (round to nearest).  The roles are transposed so that the
// small token count sits on the MMA's N side: one CTA owns 128 output features (M = 128 rows of W) x
// NT tokens (N = NT <= 192, all the tokens of a music forward in one tile) x one K split, and writes
// part[split][token][feature] for the fixed-order reductions.  At these token counts the weights stream from HBM at about
// one byte per two tensor-core FLOPs, so the loads need depth: the stage ring is as deep as shared
// memory allows (f16: five 38 KB stages of 64-byte rows at NT = 176; tf32: two of 128-byte rows).
//   warp 0     producer: W_hi, W_lo [128 x R] and X_hi, X_lo [NT x R] per stage (R row bytes)
//   warp 1     TMEM allocator + MMA issuer of the even chunks: the chunk's cross products, then its
//              hi x hi products
//   warp 10    MMA issuer of the odd chunks (one thread alone left the tensor core idle while it
//              waited on its barriers)
//   warps 2-9  epilogue: TMEM lane = feature, column = token; two warps per lane quarter split the
//              token columns; running sums in registers, coalesced stores along features
constexpr int T3_ROWS = kTf32x3N;                 // output features per CTA (MMA M)
constexpr int T3_MAX_STAGES = 8;
constexpr int T3_MAX_ACC = 4;                     // TMEM accumulator buffers at most
constexpr int T3_THREADS = 352;                   // producer, MMA, 8 epilogue warps, second MMA issuer
constexpr int T3_MAX_UNITS = 6;                   // 16-column units per epilogue warp (NT <= 192)
constexpr int T3_SMEM_MAX = 232448;               // opt-in dynamic shared memory per CTA
constexpr int X3_F16_BK = 32;                     // K per stage, f16
constexpr int X3_TF32_BK = kTf32x3K;              // K per stage, tf32 (32)

// Stage geometry per operand type: one swizzled row of K per operand row and stage.
template <bool F16>
struct X3Geom {
  static constexpr int ROW_BYTES = F16 ? 64 : 128;  // SWIZZLE_64B rows of 32 f16, SWIZZLE_128B of 32 tf32
  static constexpr int BK = F16 ? X3_F16_BK : X3_TF32_BK;
  static constexpr int KSTEPS = ROW_BYTES / 32;     // 32 bytes of K per MMA: 16 f16 or 8 tf32
  static constexpr int W_BYTES = T3_ROWS * ROW_BYTES;
  static constexpr int CHUNK = 1;                    // stages per TMEM accumulation chunk
};

struct T3Args {
  int M, N, K, k_split, nt, stages;
  int w_tiled;  // f16: W in pre-swizzled 128 x 32 tiles (hi then lo), one 16 KB bulk copy per stage
  int x_tiled;  // f16: X in the token-tiled layout (hi then lo per tile), one bulk copy per stage
  const uint16_t* w_hi;
  const uint16_t* x_hi;
  float* part;
  int* status;
  const int* w_exp;  // f16: the weight's scale exponent (device); the sums are scaled by 2^-(w_exp + x_exp)
  int x_exp;
};

template <bool F16>
__global__ void __launch_bounds__(T3_THREADS, 1)
    x3_partial_kernel(const __grid_constant__ CUtensorMap tmWhi, const __grid_constant__ CUtensorMap tmWlo,
                      const __grid_constant__ CUtensorMap tmXhi, const __grid_constant__ CUtensorMap tmXlo,
                      const T3Args a) {
  pdl_wait();
  pdl_trigger();
  using G = X3Geom<F16>;
  constexpr int T3_BK = G::BK;  // K elements per stage
  constexpr int T3_CHUNK = G::CHUNK;
  constexpr int T3_W_BYTES = G::W_BYTES;
  if (a.status && (*reinterpret_cast<const volatile int*>(a.status) & kDevLayout)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nt = a.nt;
  const int acc_cols = (nt + 31) & ~31;  // TMEM columns per accumulator buffer
  // as many accumulator buffers as the 512 TMEM columns hold (2 at NT = 176, 4 at NT <= 128): the
  // MMAs of a chunk wait only for the drain of the chunk n_acc before it
  const int n_acc = 512 / acc_cols < T3_MAX_ACC ? 512 / acc_cols : T3_MAX_ACC;
  const int T3_STAGES = a.stages;
  const int x_bytes = nt * G::ROW_BYTES;
  const int stage_bytes = 2 * T3_W_BYTES + 2 * x_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T3_STAGES * stage_bytes);
  uint64_t* empty = full + T3_MAX_STAGES;
  uint64_t* chunk_full = empty + T3_MAX_STAGES;       // [NB] an accumulator holds a finished chunk
  uint64_t* chunk_empty = chunk_full + T3_MAX_ACC;    // [NB] the epilogue has added it to its sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(chunk_empty + T3_MAX_ACC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * T3_ROWS, m0 = blockIdx.y * nt, split = blockIdx.z;
  const int kb = split * a.k_split;
  const int ke = min(a.K, kb + a.k_split);
  const int n_kb = ke > kb ? (ke - kb) / T3_BK : 0;
  const int n_chunks = (n_kb + T3_CHUNK - 1) / T3_CHUNK;

  if (threadIdx.x == 0) {
    for (int st = 0; st < T3_STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int b = 0; b < T3_MAX_ACC; ++b) {
      mbar_init(&chunk_full[b], 1);
      mbar_init(&chunk_empty[b], 8);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto produce = [&]() {
    // the weights are read once per forward: evict them first, so that the activations and the
    // split partials (read by the next kernel) stay in L2
    const uint64_t w_policy = l2_policy_evict_first();
    // CTAs side by side start at different K blocks of their range, so that they do not all ask L2
    // for the same activation rows at the same time (the chunk sums are independent of order)
    const int rot = n_kb > 0 ? (int)((long long)blockIdx.x * n_kb / gridDim.x) : 0;
    int i = 0;
    for (; i < n_kb; ++i) {
      const int st = i % T3_STAGES;
      if (!mbar_wait(&empty[st], ((i / T3_STAGES) & 1) ^ 1, abort_flag, a.status)) break;
      uint8_t* base = smem + st * stage_bytes;
      const int j = i + rot < n_kb ? i + rot : i + rot - n_kb;
      const int k0 = kb + j * T3_BK;
      mbar_arrive_expect_tx(&full[st], stage_bytes);
      if (a.w_tiled) {
        const size_t t = ((size_t)blockIdx.x * (a.K / T3_BK) + k0 / T3_BK) * (2 * T3_ROWS * T3_BK);
        bulk_load_hint(base, a.w_hi + t, 2 * T3_W_BYTES, &full[st], w_policy);
      } else {
        tma_load_2d(base, &tmWhi, &full[st], k0, n0);
        tma_load_2d(base + T3_W_BYTES, &tmWlo, &full[st], k0, n0);
      }
      if (a.x_tiled) {
        const size_t t = ((size_t)(k0 / T3_BK) * gridDim.y + blockIdx.y) * (size_t)(2 * nt * T3_BK);
        bulk_load(base + 2 * T3_W_BYTES, a.x_hi + t, 2 * x_bytes, &full[st]);
      } else {
        tma_load_2d(base + 2 * T3_W_BYTES, &tmXhi, &full[st], k0, m0);
        tma_load_2d(base + 2 * T3_W_BYTES + x_bytes, &tmXlo, &full[st], k0, m0);
      }
    }
    // Every copy issued must land before the CTA exits: wait for the stages still in flight.
    for (int j = i - T3_STAGES < 0 ? 0 : i - T3_STAGES; j < i; ++j)
      mbar_wait(&full[j % T3_STAGES], (j / T3_STAGES) & 1, abort_flag, nullptr);
  };
  if (warp == 0) {
    if (lane == 0) produce();
  } else if (warp == 1 || warp == T3_THREADS / 32 - 1) {
    // Two MMA issuers take alternate chunks (each into its own accumulator buffers), so that one
    // issues while the other waits on its barriers: a single issuing thread left the tensor core
    // idle for most of each chunk.
    if (lane == 0) {
      const uint32_t idesc = F16 ? idesc_f16_f32(T3_ROWS, nt) : idesc_tf32_f32(T3_ROWS, nt);
      // 32 bytes per instruction: K = 8 tf32 or 16 f16
      auto mma = [&](uint32_t acc, uint32_t w, uint32_t x, uint32_t accumulate) {
        if (F16)
          umma_bf16(acc, sdesc_sw64(w), sdesc_sw64(x), idesc, accumulate);
        else
          umma_tf32(acc, sdesc_sw128(w), sdesc_sw128(x), idesc, accumulate);
      };
      bool ok = true;
      for (int c = warp == 1 ? 0 : 1; c < n_chunks && ok; c += 2) {
        const int cb = c % n_acc;
        const int i0 = c * T3_CHUNK, i1 = min(n_kb, i0 + T3_CHUNK);
        if (!mbar_wait(&chunk_empty[cb], ((c / n_acc) & 1) ^ 1, abort_flag, a.status)) break;
        const uint32_t acc = tmem + cb * acc_cols;
        // Stage by stage: its small cross terms, then its hi x hi products, then the stage goes back
        // to the producer as soon as its MMAs complete (a chunk never holds more than the stage it is
        // working on).
        for (int i = i0; i < i1 && ok; ++i) {
          ok = mbar_wait(&full[i % T3_STAGES], (i / T3_STAGES) & 1, abort_flag, a.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t whi = smem_u32(smem + (i % T3_STAGES) * stage_bytes);
          const uint32_t xhi = whi + 2 * T3_W_BYTES;
#pragma unroll
          for (int ks = 0; ks < G::KSTEPS; ++ks) {
            const uint32_t off = ks * 32;
            mma(acc, whi + off, xhi + x_bytes + off, (i == i0 && ks == 0) ? 0u : 1u);
            mma(acc, whi + T3_W_BYTES + off, xhi + off, 1);
          }
#pragma unroll
          for (int ks = 0; ks < G::KSTEPS; ++ks) {
            const uint32_t off = ks * 32;
            mma(acc, whi + off, xhi + off, 1);
          }
          umma_commit(&empty[i % T3_STAGES]);
        }
        if (!ok) break;
        umma_commit(&chunk_full[cb]);
      }
    }
  } else {
    // epilogue: lane quarter = warp % 4 (TMEM access rule), column half = (warp - 2) / 4 (split at an
    // even unit so that every 32-column load starts on a multiple of 32 columns)
    const int quarter = warp & 3;
    const int units = nt / 16;
    const int half_u = ((units + 1) / 2 + 1) & ~1;
    const int u0 = (warp - 2) >> 2 ? half_u : 0;
    const int u1 = (warp - 2) >> 2 ? units : (half_u < units ? half_u : units);
    const int nu = u1 > u0 ? u1 - u0 : 0;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float run[T3_MAX_UNITS * 16];
#pragma unroll
    for (int i = 0; i < T3_MAX_UNITS * 16; ++i) run[i] = 0.f;
    bool ok = true;
    for (int c = 0; c < n_chunks; ++c) {
      const int cb = c % n_acc;
      if (!mbar_wait(&chunk_full[cb], (c / n_acc) & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // 32 columns per load; the accumulator is handed back as soon as the warp's last load has
      // landed, before the adds of that batch
#define T3_RELEASE()                                 \
  do {                                               \
    tc_fence_before();                               \
    __syncwarp();                                    \
    if (lane == 0) mbar_arrive(&chunk_empty[cb]);   \
  } while (0)
      if (nu == 0) T3_RELEASE();
      const uint32_t col0 = tmem + lane_off + cb * acc_cols + u0 * 16;
#pragma unroll
      for (int p = 0; p < T3_MAX_UNITS / 2; ++p) {
        const int u = 2 * p;
        if (u + 1 < nu) {
          uint32_t v[32];
          tmem_ld32(col0 + u * 16, v);
          tmem_ld_wait_regs(v);
          if (u + 2 >= nu) T3_RELEASE();
#pragma unroll
          for (int j = 0; j < 32; ++j) run[u * 16 + j] = __fadd_rn(run[u * 16 + j], __uint_as_float(v[j]));
        } else if (u < nu) {
          uint32_t v[16];
          tmem_ld16(col0 + u * 16, v);
          tmem_ld_wait_regs(v);
          T3_RELEASE();
#pragma unroll
          for (int j = 0; j < 16; ++j) run[u * 16 + j] = __fadd_rn(run[u * 16 + j], __uint_as_float(v[j]));
        }
      }
#undef T3_RELEASE
    }
    if (ok) {
      // f16: undo the operands' power-of-two scales (exact)
      const float osc = (F16 && a.w_exp) ? ldexpf(1.f, -(*a.w_exp + a.x_exp)) : 1.f;
      float* dst = a.part + (size_t)split * a.M * a.N + n0 + quarter * 32 + lane;
#pragma unroll
      for (int u = 0; u < T3_MAX_UNITS; ++u) {
        if (u0 + u < u1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + (u0 + u) * 16 + j;
            if (m < a.M) dst[(size_t)m * a.N] = run[u * 16 + j] * osc;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// x -> (tf32(x), tf32(x - tf32(x))), round to nearest (ties away from zero)
__global__ void tf32_split_kernel(const float* __restrict__ x, size_t n, float* __restrict__ hi, float* __restrict__ lo) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = x[i];
    uint32_t h, l;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(v));
    const float r = __fsub_rn(v, __uint_as_float(h));
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(r));
    hi[i] = __uint_as_float(h);
    lo[i] = __uint_as_float(l);
  }
}

// Row-gathered, column-padded split: row r of the [M][Kp] outputs is x row (rows ? rows[r] : r)
// of stride ldx, columns K..Kp-1 zero (the GEMM's K is a multiple of its 32-deep chunk).
__global__ void tf32_split_rows_kernel(const float* __restrict__ x, long long ldx, int K, const int* __restrict__ rows,
                                       int M, int Kp, float* __restrict__ hi, float* __restrict__ lo,
                                       const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t n = (size_t)M * Kp;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / Kp), k = (int)(i - (size_t)r * Kp);
    float v = 0.f;
    if (k < K) v = x[(size_t)(rows ? rows[r] : r) * ldx + k];
    uint32_t h, l;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(v));
    const float rr = __fsub_rn(v, __uint_as_float(h));
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(rr));
    hi[i] = __uint_as_float(h);
    lo[i] = __uint_as_float(l);
  }
}

// Largest magnitude of x, as the bits of a non-negative float (they order like the values).
__global__ void absmax_kernel(const float* __restrict__ x, size_t n, unsigned int* __restrict__ out) {
  unsigned int m = 0;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = max(m, __float_as_uint(fabsf(x[i])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

// The scale exponent e of a weight tensor from its largest magnitude: max * 2^e in [2^14, 2^15), so
// the high parts stay below f16's largest finite value (65504) and the low parts of all but the
// smallest weights stay normal.  e = 0 for an all-zero tensor.
__device__ __forceinline__ int weight_exp(unsigned int max_bits) {
  if (max_bits == 0 || max_bits >= 0x7F800000u) return 0;
  const int ex = (int)(max_bits >> 23) - 127;  // floor(log2(max)) for a normal max
  const int e = 14 - ex;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// x [M][K] (row stride ldx) -> hi, lo [M][Kp] f16 bits of x * 2^e, zero-padded for k >= K:
//   hi = f16(x 2^e), lo = f16(x 2^e - hi)     (round to nearest even)
// With `tiled` the outputs are laid out as the 3xF16 GEMM's weight tiles, [M / 128][Kp / 32][128][32],
// each tile already in the shared-memory image of the 64-byte swizzle (16-byte chunk c of row r at
// c ^ ((r >> 1) & 3)): every stage of the GEMM then reads one contiguous 8 KB block per part with a
// plain bulk copy (M % 128 == 0, Kp % 32 == 0).
// e is the weight exponent of *max_bits when given (and then written to *e_out by block 0), else
// e_fixed.  A magnitude of x 2^e beyond 65504 sets kDevRange in *status.
__global__ void f16_split_kernel(const float* __restrict__ x, long long ldx, int K, int M, int Kp,
                                 const unsigned int* __restrict__ max_bits, int e_fixed, int* __restrict__ e_out,
                                 uint16_t* __restrict__ hi, uint16_t* __restrict__ lo, int layout, int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const int e = max_bits ? weight_exp(*max_bits) : e_fixed;
  if (e_out && blockIdx.x == 0 && threadIdx.x == 0) *e_out = e;
  const int tok_nt = x3_token_tile(M), tok_mt = (M + tok_nt - 1) / tok_nt;
  const size_t n = (size_t)M * Kp;
  bool over = false;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / Kp), k = (int)(i - (size_t)r * Kp);
    const float v = k < K ? ldexpf(x[(size_t)r * ldx + k], e) : 0.f;
    over |= fabsf(v) > kF16Max;
    const __half h = __float2half_rn(v);
    const __half l = __float2half_rn(__fsub_rn(v, __half2float(h)));
    size_t o = i;
    if (layout == kSplitWeightTiles) {
      const int rr = r % T3_ROWS, kk = k % X3_F16_BK;
      o = ((size_t)(r / T3_ROWS) * (Kp / X3_F16_BK) + k / X3_F16_BK) * (2 * T3_ROWS * X3_F16_BK) + rr * X3_F16_BK +
          ((((kk >> 3) ^ (rr >> 1)) & 3) << 3) + (kk & 7);
    } else if (layout == kSplitTokenTiles) {
      o = x3_xs_index(r, k, tok_nt, tok_mt);
    }
    hi[o] = __half_as_ushort(h);
    if (layout == kSplitTokenTiles)
      hi[o + (size_t)tok_nt * 32] = __half_as_ushort(l);
    else
      lo[o] = __half_as_ushort(l);
  }
  if (over && status) atomicOr(status, kDevRange);
}

// out[(rows ? rows[r] : r) * ld_out + n] = sum over S partials [S][M][Np] + bias[n], n < n_out:
// the row-scattered, column-trimmed store of a GEMM whose N was padded to Np.
__global__ void sgemm_reduce_rows_kernel(const float* __restrict__ part, int S, int M, int Np, int n_out,
                                         const float* __restrict__ bias, const int* __restrict__ rows,
                                         float* __restrict__ out, long long ld_out, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t MNp = (size_t)M * Np;
  const size_t n = (size_t)M * n_out;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / n_out), c = (int)(i - (size_t)r * n_out);
    const float v = sum_parts(part, S, MNp, (size_t)r * Np + c) + (bias ? bias[c] : 0.f);
    out[(size_t)(rows ? rows[r] : r) * ld_out + c] = v;
  }
}

int ew_grid(size_t work) {
  size_t g = (work + 255) / 256;
  const size_t cap = (size_t)num_sms() * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

// Tokens per CTA (the MMA's N).
int tf32x3_token_tile(int M) { return x3_token_tile(M); }

static int x3_effective_splits(int K, int S, int bk) {
  int ks = (K + S - 1) / S;
  ks = (ks + bk - 1) / bk * bk;
  return (K + ks - 1) / ks;
}

// The K split count: the most CTAs (one per SM, each with a deep stage ring) that still run as one
// wave; 1 when the output tiles alone fill the SMs.
static int x3_splits(int M, int N, int K, int bk) {
  const int tiles = (N / T3_ROWS) * ((M + tf32x3_token_tile(M) - 1) / tf32x3_token_tile(M));
  int max_s = K / bk > 0 ? K / bk : 1;
  if (max_s > kSgemmMaxSplits) max_s = kSgemmMaxSplits;
  int best = 1;
  for (int S = 2; S <= max_s; ++S)
    if (tiles * x3_effective_splits(K, S, bk) <= num_sms()) best = S;
  return best;
}

int tf32x3_splits(int M, int N, int K) { return x3_splits(M, N, K, X3_TF32_BK); }
int tf32x3_effective_splits(int K, int S) { return x3_effective_splits(K, S, X3_TF32_BK); }
int f16x3_splits(int M, int N, int K) { return x3_splits(M, N, K, X3_F16_BK); }
int f16x3_effective_splits(int K, int S) { return x3_effective_splits(K, S, X3_F16_BK); }

template <bool F16>
static cudaError_t x3_partial_launch(const void* x_hi, const void* x_lo, const void* w_hi, const void* w_lo,
                                     const int* w_exp, int x_exp, int M, int N, int K, int S, float* part,
                                     const int* status, cudaStream_t s, int w_tiled, int x_tiled) {
  constexpr int BK = F16 ? X3_F16_BK : X3_TF32_BK;
  if (M <= 0) return cudaSuccess;
  if (N % T3_ROWS || K % BK) return cudaErrorInvalidValue;
  const int nt = tf32x3_token_tile(M);
  int ks = (K + S - 1) / S;
  ks = (ks + BK - 1) / BK * BK;
  const int S_eff = (K + ks - 1) / ks;
  // the tiled layouts are loaded with plain bulk copies: their tensor maps are never read, so they
  // are left zeroed instead of encoded (the encoding is most of this launch's host time)
  CUtensorMap whi = {}, wlo = {}, xhi = {}, xlo = {};
  bool ok = true;
  if (F16) {
    if (!w_tiled)
      ok = make_tmap_bf16_2d(&whi, w_hi, K, N, (uint64_t)K * 2, BK, T3_ROWS, CU_TENSOR_MAP_SWIZZLE_64B) &&
           make_tmap_bf16_2d(&wlo, w_lo, K, N, (uint64_t)K * 2, BK, T3_ROWS, CU_TENSOR_MAP_SWIZZLE_64B);
    if (ok && !x_tiled)
      ok = make_tmap_bf16_2d(&xhi, x_hi, K, M, (uint64_t)K * 2, BK, nt, CU_TENSOR_MAP_SWIZZLE_64B) &&
           make_tmap_bf16_2d(&xlo, x_lo, K, M, (uint64_t)K * 2, BK, nt, CU_TENSOR_MAP_SWIZZLE_64B);
  } else
    ok = make_tmap_f32_2d(&whi, w_hi, K, N, (uint64_t)K * 4, T3_ROWS) &&
         make_tmap_f32_2d(&wlo, w_lo, K, N, (uint64_t)K * 4, T3_ROWS) &&
         make_tmap_f32_2d(&xhi, x_hi, K, M, (uint64_t)K * 4, nt) &&
         make_tmap_f32_2d(&xlo, x_lo, K, M, (uint64_t)K * 4, nt);
  if (!ok) return cudaErrorInvalidValue;
  // as many stages as fit: 1024 bytes of alignment slack and 256 of barriers besides the ring
  const int stage_bytes = 2 * X3Geom<F16>::W_BYTES + 2 * nt * X3Geom<F16>::ROW_BYTES;
  int stages = (T3_SMEM_MAX - 1024 - 256) / stage_bytes;
  if (stages > T3_MAX_STAGES) stages = T3_MAX_STAGES;
  if (stages < 2) return cudaErrorInvalidValue;
  const int smem = stages * stage_bytes + 1024 + 256;
  static unsigned long long smem_set = 0;  // opted in to the largest size once per device
  cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(x3_partial_kernel<F16>), T3_SMEM_MAX, &smem_set);
  if (e != cudaSuccess) return e;
  T3Args a{M, N, K, ks, nt, stages, F16 && w_tiled, F16 && x_tiled, static_cast<const uint16_t*>(w_hi),
           static_cast<const uint16_t*>(x_hi), part, const_cast<int*>(status), w_exp, x_exp};
  dim3 grid(N / T3_ROWS, (M + nt - 1) / nt, S_eff);
  e = launch_pdl(x3_partial_kernel<F16>, grid, dim3(T3_THREADS), smem, s, whi, wlo, xhi, xlo, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t tf32x3_partial_launch(const float* x_hi, const float* x_lo, const float* w_hi, const float* w_lo, int M,
                                  int N, int K, int S, float* part, const int* status, cudaStream_t s) {
  return x3_partial_launch<false>(x_hi, x_lo, w_hi, w_lo, nullptr, 0, M, N, K, S, part, status, s, 0, 0);
}

cudaError_t f16x3_partial_launch(const uint16_t* x_hi, const uint16_t* x_lo, const uint16_t* w_hi,
                                 const uint16_t* w_lo, const int* w_exp, int x_exp, int M, int N, int K, int S,
                                 float* part, const int* status, cudaStream_t s, int w_tiled, int x_tiled) {
  return x3_partial_launch<true>(x_hi, x_lo, w_hi, w_lo, w_exp, x_exp, M, N, K, S, part, status, s, w_tiled,
                                 x_tiled);
}

cudaError_t absmax_launch(const float* x, size_t n, unsigned int* out, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess || n == 0) return e;
  absmax_kernel<<<ew_grid(n), 256, 0, s>>>(x, n, out);
  return cudaGetLastError();
}

cudaError_t f16_split_launch(const float* x, long long ldx, int K, int M, int Kp, const unsigned int* max_bits,
                             int e_fixed, int* e_out, uint16_t* hi, uint16_t* lo, int* status, cudaStream_t s,
                             int layout) {
  if (M <= 0) return cudaSuccess;
  if (K < 1 || Kp < K || ldx < K) return cudaErrorInvalidValue;
  if (layout == kSplitWeightTiles && (M % T3_ROWS || Kp % X3_F16_BK)) return cudaErrorInvalidValue;
  if (layout == kSplitTokenTiles && Kp % X3_F16_BK) return cudaErrorInvalidValue;
  f16_split_kernel<<<ew_grid((size_t)M * Kp), 256, 0, s>>>(x, ldx, K, M, Kp, max_bits, e_fixed, e_out, hi, lo, layout,
                                                             status);
  return cudaGetLastError();
}

cudaError_t tf32_split_launch(const float* x, size_t n, float* hi, float* lo, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  tf32_split_kernel<<<ew_grid(n), 256, 0, s>>>(x, n, hi, lo);
  return cudaGetLastError();
}

cudaError_t tf32_split_rows_launch(const float* x, long long ldx, int K, const int* rows, int M, int Kp, float* hi,
                                   float* lo, const int* status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (K < 1 || Kp < K || ldx < K) return cudaErrorInvalidValue;
  tf32_split_rows_kernel<<<ew_grid((size_t)M * Kp), 256, 0, s>>>(x, ldx, K, rows, M, Kp, hi, lo, status);
  return cudaGetLastError();
}

cudaError_t sgemm_reduce_rows_launch(const float* part, int S, int M, int Np, int n_out, const float* bias,
                                     const int* rows, float* out, long long ld_out, const int* status,
                                     cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (n_out < 1 || n_out > Np || ld_out < n_out) return cudaErrorInvalidValue;
  sgemm_reduce_rows_kernel<<<ew_grid((size_t)M * n_out), 256, 0, s>>>(part, S, M, Np, n_out, bias, rows, out, ld_out,
                                                                      status);
  return cudaGetLastError();
}

// 2-D grid of the reductions: 1024 columns per 256-thread block, rows up to 65535 per launch row
static dim3 reduce_grid(int M, int cols) { return dim3((cols + 1023) / 1024, M < 65535 ? M : 65535); }

cudaError_t sgemm_reduce_store_launch(const float* part, int S, int M, int N, const float* bias, float* out, int add,
                                      float* lo, const int* status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (N % 4) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(sgemm_reduce_store_kernel, reduce_grid(M, N), dim3(256), 0, s, part, S, M, N, bias, out,
                             add, lo, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t sgemm_reduce_resid_norm_launch(const float* part, int S, int M, int d, const float* bias, float* resid,
                                           float* resid_lo, int add, int norm, float eps, const float* g,
                                           const float* b, void* y, int out_kind, int* status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (!reduce_norm_fusable(d) || (out_kind != 1 && out_kind != 3) || !resid_lo) return cudaErrorInvalidValue;
  const int blocks = M < num_sms() * 8 ? M : num_sms() * 8;
  cudaError_t e = cudaErrorInvalidValue;
  switch (d / 1024) {
#define DIT_RN(k)                                                                                                   \
  case k:                                                                                                           \
    e = launch_pdl(sgemm_reduce_resid_norm_kernel<k>, dim3(blocks), dim3(256), 0, s, part, S, M, d, bias, resid,   \
                   resid_lo, add, norm, eps, g, b, y, out_kind, status);                                            \
    break;
    DIT_RN(1) DIT_RN(2) DIT_RN(3) DIT_RN(4) DIT_RN(5) DIT_RN(6) DIT_RN(7) DIT_RN(8)
#undef DIT_RN
    default: break;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool reduce_norm_fusable(int d) { return d > 0 && d % 1024 == 0 && d <= 8192; }

cudaError_t sgemm_reduce_qkv_launch(const float* part, int S, int M, int d, int Dh, int half, const float* bias,
                                    const float* cs, const float* sn, float* q, float* k, float* v, const int* status,
                                    cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (d % 4 || Dh % 4 || half % 4) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(sgemm_reduce_qkv_kernel, reduce_grid(M, 3 * d), dim3(256), 0, s, part, S, M, d, Dh, half,
                             bias, cs, sn, q, k, v, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t sgemm_reduce_swiglu_launch(const float* part, int S, int M, int F, const float* bias, float* h,
                                       uint16_t* h_split, int* status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (F % 4) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(sgemm_reduce_swiglu_kernel, reduce_grid(M, F), dim3(256), 0, s, part, S, M, F, bias, h,
                             h_split, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t attention_f32_launch(const float* q, const float* k, const float* v, const int32_t* cu, const int2* items,
                                 const int* count, int max_items, int n_tokens, int H, int Dh, float* o,
                                 uint16_t* o_split, int* status, cudaStream_t s) {
  if (max_items <= 0) return cudaSuccess;
  const dim3 grid(max_items * AF_BLOCKS, H);
  const float scale = (float)(1.0 / sqrt((double)Dh));
  if (Dh == 128) {
    static unsigned long long set = 0;
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(attention_f32_kernel<128>), af_smem_bytes<128>(), &set);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attention_f32_kernel<128>, grid, dim3(AF_WARPS * 32), af_smem_bytes<128>(), s, q, k, v, cu, items,
                   count, n_tokens, H, scale, o, o_split, status);
    if (e != cudaSuccess) return e;
  } else if (Dh == 64) {
    static unsigned long long set = 0;
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(attention_f32_kernel<64>), af_smem_bytes<64>(), &set);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attention_f32_kernel<64>, grid, dim3(AF_WARPS * 32), af_smem_bytes<64>(), s, q, k, v, cu, items,
                   count, n_tokens, H, scale, o, o_split, status);
    if (e != cudaSuccess) return e;
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t io_transpose_launch(const float* src, float* dst, const int32_t* cu, const int32_t* doc_ids, int n, int io,
                                int to_frames, const int* status, cudaStream_t s) {
  io_transpose_kernel<<<ew_grid((size_t)n * io), 256, 0, s>>>(src, dst, cu, doc_ids, n, io, to_frames, status);
  return cudaGetLastError();
}

}  // namespace dit
