// The fp32 forward path: the music DiT shape of [M3] "What moved" (fp32 stays fp32: every weight and
// activation is fp32; LayerNorm, partial rotary, non-causal attention with no bias,
// value * silu(gate), 1x1 pre/post convolutions as MatmulBT on the frame-major activation).
// TF32 tensor cores would round operands to 10 mantissa bits, far above the 1e-5 tolerance, so the
// contractions run on the fp32 FMA pipes:
//   sgemm_partial_kernel   register-blocked 64x128x16 tiles, split-K; each split writes its partial
//                          sums (accumulated in 64-deep chunks) to a [S][M][N] buffer
//   sgemm_reduce_*         sums the S partials in a fixed order and applies the epilogue (bias,
//                          residual add, NeoX RoPE + q/k/v split, value * silu(gate))
//   attention_f32_kernel   one warp per (query row, head), exact fp32 online softmax with expf
//   io_transpose_kernel    channel-major [io, len] per document <-> frame-major [N, io]
#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace dit {

namespace {

constexpr int SBM = 64, SBN = 128, SBK = 16;
constexpr int SCHUNK = 64;  // k-depth of one partial-sum chunk

__global__ void __launch_bounds__(256) sgemm_partial_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                            int M, int N, int K, int k_split,
                                                            float* __restrict__ part, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  __shared__ __align__(16) float As[SBK][SBM + 4];
  __shared__ __align__(16) float Bs[SBK][SBN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.x * SBN, m0 = blockIdx.y * SBM, s = blockIdx.z;
  const int kb = s * k_split, ke = min(K, kb + k_split);
  float acc[4][8], chk[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = chk[i][j] = 0.f;
  // load mapping: A row (tid / 4), k quad (tid % 4); B rows (tid / 4) and (tid / 4 + 64)
  const int lr = tid >> 2, lq = (tid & 3) * 4;
  const int am = m0 + lr;
  float4 ra, rb0, rb1;
  auto gload = [&](int k0) {
    ra = am < M ? *reinterpret_cast<const float4*>(A + (size_t)am * K + k0 + lq) : make_float4(0.f, 0.f, 0.f, 0.f);
    rb0 = *reinterpret_cast<const float4*>(B + (size_t)(n0 + lr) * K + k0 + lq);
    rb1 = *reinterpret_cast<const float4*>(B + (size_t)(n0 + lr + 64) * K + k0 + lq);
  };
  if (kb < ke) gload(kb);
  for (int k0 = kb; k0 < ke; k0 += SBK) {
    __syncthreads();
    As[lq + 0][lr] = ra.x; As[lq + 1][lr] = ra.y; As[lq + 2][lr] = ra.z; As[lq + 3][lr] = ra.w;
    Bs[lq + 0][lr] = rb0.x; Bs[lq + 1][lr] = rb0.y; Bs[lq + 2][lr] = rb0.z; Bs[lq + 3][lr] = rb0.w;
    Bs[lq + 0][lr + 64] = rb1.x; Bs[lq + 1][lr + 64] = rb1.y; Bs[lq + 2][lr + 64] = rb1.z; Bs[lq + 3][lr + 64] = rb1.w;
    __syncthreads();
    if (k0 + SBK < ke) gload(k0 + SBK);  // prefetch the next tile while this one is consumed
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) chk[i][j] = fmaf(av[i], bv[j], chk[i][j]);
    }
    if (((k0 - kb + SBK) % SCHUNK) == 0 || k0 + SBK >= ke) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[i][j] += chk[i][j];
          chk[i][j] = 0.f;
        }
    }
  }
  float* out = part + (size_t)s * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    *reinterpret_cast<float4*>(out + (size_t)m * N + n0 + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(out + (size_t)m * N + n0 + 64 + tx * 4) =
        make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

__device__ __forceinline__ float sum_parts(const float* __restrict__ part, int S, size_t MN, size_t idx) {
  float v = 0.f;
  for (int s = 0; s < S; ++s) v += part[(size_t)s * MN + idx];
  return v;
}

// out = sum + bias (add = 0: store into out [M, N]; add = 1: out[M, N] += sum + bias).  With `lo`
// the residual is a compensated pair (out = high part, lo = low part): the add is an exact TwoSum
// whose rounding error goes into lo, so the residual stream keeps about twice fp32's precision.
__global__ void sgemm_reduce_store_kernel(const float* __restrict__ part, int S, int M, int N,
                                          const float* __restrict__ bias, float* __restrict__ out, int add,
                                          float* __restrict__ lo, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t MN = (size_t)M * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < MN; i += (size_t)gridDim.x * blockDim.x) {
    const float v = sum_parts(part, S, MN, i) + (bias ? bias[i % N] : 0.f);
    if (!add) {
      out[i] = v;
      if (lo) lo[i] = 0.f;
    } else if (lo) {
      const float a = out[i];
      const float s = __fadd_rn(a, v);
      const float bb = __fsub_rn(s, a);
      const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(v, bb));
      out[i] = s;
      lo[i] = __fadd_rn(lo[i], err);
    } else {
      out[i] = out[i] + v;
    }
  }
}

// [q | k | v] = sum + bias, NeoX rotate_half over the first R dims of each q/k head, stored fp32
// [M, d] each.
__global__ void sgemm_reduce_qkv_kernel(const float* __restrict__ part, int S, int M, int d, int Dh, int half,
                                        const float* __restrict__ bias, const float* __restrict__ cs,
                                        const float* __restrict__ sn, float* __restrict__ q, float* __restrict__ k,
                                        float* __restrict__ v, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const int N = 3 * d;
  const size_t MN = (size_t)M * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < MN; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / N), c = (int)(i - (size_t)r * N);
    const int seg = c / d, cc = c - seg * d;
    const float x = sum_parts(part, S, MN, i) + (bias ? bias[c] : 0.f);
    if (seg == 2) {
      v[(size_t)r * d + cc] = x;
      continue;
    }
    const int jd = cc % Dh;  // dim within the head
    float o = x;
    if (jd < 2 * half) {
      const int j = jd < half ? jd : jd - half;
      const int pc = jd < half ? c + half : c - half;  // partner column
      const float y = sum_parts(part, S, MN, (size_t)r * N + pc) + (bias ? bias[pc] : 0.f);
      const float co = cs[(size_t)r * half + j], si = sn[(size_t)r * half + j];
      o = jd < half ? x * co - y * si : x * co + y * si;
    }
    (seg == 0 ? q : k)[(size_t)r * d + cc] = o;
  }
}

// h[r, f] = (u + b_u) * silu(g + b_g): value columns [0, F), gate columns [F, 2F)
__global__ void sgemm_reduce_swiglu_kernel(const float* __restrict__ part, int S, int M, int F,
                                           const float* __restrict__ bias, float* __restrict__ h, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const size_t MN = (size_t)M * 2 * F;
  const size_t total = (size_t)M * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / F), f = (int)(i - (size_t)r * F);
    const float u = sum_parts(part, S, MN, (size_t)r * 2 * F + f) + (bias ? bias[f] : 0.f);
    const float g = sum_parts(part, S, MN, (size_t)r * 2 * F + F + f) + (bias ? bias[F + f] : 0.f);
    h[i] = u * (g / (1.0f + expf(-g)));
  }
}

// Exact fp32 softmax attention over the document of each row.  One warp per (row, head); lanes
// hold DH/32 dims of q, o; running max / sum (online softmax) in registers.
template <int DH>
__global__ void __launch_bounds__(256) attention_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                            const float* __restrict__ v, const int32_t* __restrict__ cu,
                                                            const int32_t* __restrict__ doc_ids, int n, int H,
                                                            float scale, float* __restrict__ o, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  constexpr int PL = DH / 32;
  const int lane = threadIdx.x & 31;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= n * H) return;
  const int i = w / H, h = w - i * H;
  const int d = H * DH;
  const int doc = doc_ids[i];
  const int a = cu[doc], b = cu[doc + 1];
  float qv[PL], ov[PL];
#pragma unroll
  for (int e = 0; e < PL; ++e) {
    qv[e] = q[(size_t)i * d + h * DH + lane * PL + e];
    ov[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = a; j < b; ++j) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) s = fmaf(qv[e], k[(size_t)j * d + h * DH + lane * PL + e], s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);  // 0 for the first key
    const float p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < PL; ++e) ov[e] = fmaf(p, v[(size_t)j * d + h * DH + lane * PL + e], ov[e] * corr);
    m = mn;
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int e = 0; e < PL; ++e) o[(size_t)i * d + h * DH + lane * PL + e] = ov[e] * inv;
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

int ew_grid(size_t work) {
  size_t g = (work + 255) / 256;
  const size_t cap = (size_t)num_sms() * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

int sgemm_splits(int M, int N, int K) {
  const int tiles = (N / SBN) * ((M + SBM - 1) / SBM);
  const int target = 4 * num_sms();  // about two resident CTAs per SM, twice over
  int S = (target + tiles - 1) / tiles;
  const int max_s = K / SCHUNK > 0 ? K / SCHUNK : 1;
  if (S > max_s) S = max_s;
  if (S > kSgemmMaxSplits) S = kSgemmMaxSplits;
  return S < 1 ? 1 : S;
}

cudaError_t sgemm_partial_launch(const float* A, const float* B, int M, int N, int K, int S, float* part,
                                 const int* status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  int ks = (K + S - 1) / S;
  ks = (ks + SCHUNK - 1) / SCHUNK * SCHUNK;  // split boundaries on chunk boundaries
  const int S_eff = (K + ks - 1) / ks;
  dim3 grid(N / SBN, (M + SBM - 1) / SBM, S_eff);
  sgemm_partial_kernel<<<grid, 256, 0, s>>>(A, B, M, N, K, ks, part, status);
  return cudaGetLastError();
}

int sgemm_effective_splits(int K, int S) {
  int ks = (K + S - 1) / S;
  ks = (ks + SCHUNK - 1) / SCHUNK * SCHUNK;
  return (K + ks - 1) / ks;
}

cudaError_t sgemm_reduce_store_launch(const float* part, int S, int M, int N, const float* bias, float* out, int add,
                                      float* lo, const int* status, cudaStream_t s) {
  sgemm_reduce_store_kernel<<<ew_grid((size_t)M * N), 256, 0, s>>>(part, S, M, N, bias, out, add, lo, status);
  return cudaGetLastError();
}

cudaError_t sgemm_reduce_qkv_launch(const float* part, int S, int M, int d, int Dh, int half, const float* bias,
                                    const float* cs, const float* sn, float* q, float* k, float* v, const int* status,
                                    cudaStream_t s) {
  sgemm_reduce_qkv_kernel<<<ew_grid((size_t)M * 3 * d), 256, 0, s>>>(part, S, M, d, Dh, half, bias, cs, sn, q, k, v,
                                                                      status);
  return cudaGetLastError();
}

cudaError_t sgemm_reduce_swiglu_launch(const float* part, int S, int M, int F, const float* bias, float* h,
                                       const int* status, cudaStream_t s) {
  sgemm_reduce_swiglu_kernel<<<ew_grid((size_t)M * F), 256, 0, s>>>(part, S, M, F, bias, h, status);
  return cudaGetLastError();
}

cudaError_t attention_f32_launch(const float* q, const float* k, const float* v, const int32_t* cu,
                                 const int32_t* doc_ids, int n, int H, int Dh, float* o, const int* status,
                                 cudaStream_t s) {
  const long long warps = (long long)n * H;
  const int blocks = (int)((warps * 32 + 255) / 256);
  const float scale = (float)(1.0 / sqrt((double)Dh));
  if (Dh == 128)
    attention_f32_kernel<128><<<blocks, 256, 0, s>>>(q, k, v, cu, doc_ids, n, H, scale, o, status);
  else if (Dh == 64)
    attention_f32_kernel<64><<<blocks, 256, 0, s>>>(q, k, v, cu, doc_ids, n, H, scale, o, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t io_transpose_launch(const float* src, float* dst, const int32_t* cu, const int32_t* doc_ids, int n, int io,
                                int to_frames, const int* status, cudaStream_t s) {
  io_transpose_kernel<<<ew_grid((size_t)n * io), 256, 0, s>>>(src, dst, cu, doc_ids, n, io, to_frames, status);
  return cudaGetLastError();
}

}  // namespace dit
