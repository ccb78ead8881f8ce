// Bandwidth-bound kernels of the forward: fused norm + indexed AdaLN modulate, the per-row RoPE
// cos/sin cache, the AdaLN conditioning GEMV, the Euler step, and bind-time repacks.
#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace dit {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------------------------
// Norm + indexed AdaLN modulate.  [H3] "The device-resident forward (W2b)": RmsNorm followed by
// an indexed AdaLN modulate (shift/scale chosen per token by its modality tag).  One warp per row;
// the row stays in registers between the statistics pass and the output pass; fp32 statistics.
//   RMS:   n = x / sqrt(mean(x^2) + eps)
//   LN:    n = (x - mean) / sqrt(mean((x - mean)^2) + eps) * g + b
//   out    y = n * (1 + scale[tag]) + shift[tag]       (no modulation when shift == nullptr)
// ---------------------------------------------------------------------------------------------
template <int NV>
__global__ void __launch_bounds__(256) norm_mod_kernel(const float* __restrict__ x, const float* __restrict__ x_lo,
                                                       int n, int d, int norm, float eps,
                                                       const float* __restrict__ g, const float* __restrict__ b,
                                                       const uint8_t* __restrict__ tags,
                                                       const float* __restrict__ shift,
                                                       const float* __restrict__ scale, long long stride, void* y,
                                                       int out_kind, int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n) return;
  const float* xr = x + (size_t)row * d;
  float4 v[NV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    v[i] = *reinterpret_cast<const float4*>(xr + (i * 32 + lane) * 4);
    if (x_lo) {
      const float4 e = *reinterpret_cast<const float4*>(x_lo + (size_t)row * d + (i * 32 + lane) * 4);
      v[i].x += e.x; v[i].y += e.y; v[i].z += e.z; v[i].w += e.w;
    }
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
  float mean = 0.f, inv;
  if (norm == 0) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    ss = warp_sum(ss);
    inv = 1.0f / sqrtf(ss / (float)d + eps);
  } else {
    mean = warp_sum(s) / (float)d;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float a0 = v[i].x - mean, a1 = v[i].y - mean, a2 = v[i].z - mean, a3 = v[i].w - mean;
      ss += a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
    }
    ss = warp_sum(ss);
    inv = 1.0f / sqrtf(ss / (float)d + eps);
  }
  const float* sh = shift ? shift + (size_t)tags[row] * stride : nullptr;
  const float* sc = scale ? scale + (size_t)tags[row] * stride : nullptr;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = (i * 32 + lane) * 4;
    float o[4] = {(v[i].x - mean) * inv, (v[i].y - mean) * inv, (v[i].z - mean) * inv, (v[i].w - mean) * inv};
    {  // gain and shift of either norm (NULL = none)
      if (g) {
        const float4 gg = *reinterpret_cast<const float4*>(g + c);
        o[0] *= gg.x; o[1] *= gg.y; o[2] *= gg.z; o[3] *= gg.w;
      }
      if (b) {
        const float4 bb = *reinterpret_cast<const float4*>(b + c);
        o[0] += bb.x; o[1] += bb.y; o[2] += bb.z; o[3] += bb.w;
      }
    }
    if (sh) {
      const float4 a = *reinterpret_cast<const float4*>(sh + c);
      const float4 m = *reinterpret_cast<const float4*>(sc + c);
      o[0] = o[0] * (1.f + m.x) + a.x;
      o[1] = o[1] * (1.f + m.y) + a.y;
      o[2] = o[2] * (1.f + m.z) + a.z;
      o[3] = o[3] * (1.f + m.w) + a.w;
    }
    if (out_kind == 0 || out_kind == 2) {
      const bool f = out_kind == 2;
      if (f && status && fmaxf(fmaxf(fabsf(o[0]), fabsf(o[1])), fmaxf(fabsf(o[2]), fabsf(o[3]))) > kF16Max)
        atomicOr(status, kDevRange);
      uint2 pk = make_uint2(pack16(f, o[0], o[1]), pack16(f, o[2], o[3]));
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + (size_t)row * d + c) = pk;
    } else if (out_kind == 3) {
      const int nt = x3_token_tile(n);
      const size_t xi = x3_xs_index(row, c, nt, (n + nt - 1) / nt);
      uint16_t* xs = static_cast<uint16_t*>(y);
      if (store_f16_split4(o, kF16x3ActExp, xs + xi, xs + xi + (size_t)nt * 32) && status) atomicOr(status, kDevRange);
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)row * d + c) = make_float4(o[0], o[1], o[2], o[3]);
    }
  }
}

// The same norm + modulate for widths d = 1024 * VPT: a persistent grid of 256-thread blocks, each
// thread owning VPT float4 of a row, walks the rows with a stride of gridDim.x and prefetches the
// next row into registers before reducing the current one, so every block keeps a row's loads in
// flight while it computes (the kernel is HBM-bound: 4 bytes in, 2 or 4 out per element).
template <int VPT, bool LO>
__global__ void __launch_bounds__(256) norm_mod_persistent_kernel(
    const float* __restrict__ x, const float* __restrict__ x_lo, int n, int d, int norm, float eps, const float* __restrict__ g,
    const float* __restrict__ b, const uint8_t* __restrict__ tags, const float* __restrict__ shift,
    const float* __restrict__ scale, long long stride, void* y, int out_kind, int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  __shared__ float red[2][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int row = blockIdx.x;
  float4 cur[VPT], nxt[VPT];
  auto load = [&](int r, float4 (&v)[VPT]) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      v[i] = *reinterpret_cast<const float4*>(x + (size_t)r * d + (i * 256 + threadIdx.x) * 4);
      if (LO) {  // compensated residual: high + low part
        const float4 e = *reinterpret_cast<const float4*>(x_lo + (size_t)r * d + (i * 256 + threadIdx.x) * 4);
        v[i].x += e.x; v[i].y += e.y; v[i].z += e.z; v[i].w += e.w;
      }
    }
  };
  if (row < n) load(row, cur);
  int parity = 0;
  // block sum through one of two shared slots (alternating, so one barrier per reduction suffices)
  auto block_sum = [&](float s) -> float {
    s = warp_sum(s);
    if (lane == 0) red[parity][warp] = s;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[parity][w];
    parity ^= 1;
    return t;
  };
  for (; row < n; row += gridDim.x) {
    const int nrow = row + gridDim.x;
    if (nrow < n) load(nrow, nxt);
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
    const float* sh = shift ? shift + (size_t)tags[row] * stride : nullptr;
    const float* sc = scale ? scale + (size_t)tags[row] * stride : nullptr;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = (i * 256 + threadIdx.x) * 4;
      float o[4] = {(cur[i].x - mean) * inv, (cur[i].y - mean) * inv, (cur[i].z - mean) * inv,
                    (cur[i].w - mean) * inv};
      {  // gain and shift of either norm (NULL = none)
        if (g) {
          const float4 gg = *reinterpret_cast<const float4*>(g + c);
          o[0] *= gg.x; o[1] *= gg.y; o[2] *= gg.z; o[3] *= gg.w;
        }
        if (b) {
          const float4 bb = *reinterpret_cast<const float4*>(b + c);
          o[0] += bb.x; o[1] += bb.y; o[2] += bb.z; o[3] += bb.w;
        }
      }
      if (sh) {
        const float4 a = *reinterpret_cast<const float4*>(sh + c);
        const float4 m = *reinterpret_cast<const float4*>(sc + c);
        o[0] = o[0] * (1.f + m.x) + a.x;
        o[1] = o[1] * (1.f + m.y) + a.y;
        o[2] = o[2] * (1.f + m.z) + a.z;
        o[3] = o[3] * (1.f + m.w) + a.w;
      }
      if (out_kind == 0 || out_kind == 2) {
        const bool f = out_kind == 2;
        if (f && status && fmaxf(fmaxf(fabsf(o[0]), fabsf(o[1])), fmaxf(fabsf(o[2]), fabsf(o[3]))) > kF16Max)
          atomicOr(status, kDevRange);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + (size_t)row * d + c) =
            make_uint2(pack16(f, o[0], o[1]), pack16(f, o[2], o[3]));
      } else if (out_kind == 3) {
        const int nt = x3_token_tile(n);
        const size_t xi = x3_xs_index(row, c, nt, (n + nt - 1) / nt);
        uint16_t* xs = static_cast<uint16_t*>(y);
        if (store_f16_split4(o, kF16x3ActExp, xs + xi, xs + xi + (size_t)nt * 32) && status)
          atomicOr(status, kDevRange);
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)row * d + c) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) cur[i] = nxt[i];
  }
}

// ---------------------------------------------------------------------------------------------
// RoPE cos/sin cache.  [BF] "What this enables": BuildRopeCosSin runs before any kernel with a
// stored inv_freq; [H3] "The device-resident forward (W2b)": a per-row cos/sin cache whose angles
// come from three axes of the fp64 position grid.  theta = pos[row][axis(j)] * (double)inv[j]
// in fp64; cos and sin in fp64, rounded to fp32.
// ---------------------------------------------------------------------------------------------
struct RopeTable {
  float inv[128];
  unsigned char axis[128];
};

__global__ void rope_cache_kernel(const double* __restrict__ pos, int n, int half, const RopeTable tab,
                                  float* __restrict__ cs, float* __restrict__ sn, const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  const long long total = (long long)n * half;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(i / half), j = (int)(i - (long long)row * half);
    const double th = pos[(size_t)row * 3 + tab.axis[j]] * (double)tab.inv[j];
    double s, c;
    sincos(th, &s, &c);
    cs[i] = (float)c;
    sn[i] = (float)s;
  }
}

// ---------------------------------------------------------------------------------------------
// AdaLN conditioning.  e = [cos(1000 t f_k) | sin(1000 t f_k)], f_k = exp(-ln(1e4) k / half)
// (fp64), silu(e) in fp64 -> fp32 ([H3] "The device-resident forward (W2b)": the ungated SiLU;
// the time embedder is an fp32 island per [H3] "Update: quantized arms land").  Then
// mod[r] = W[r] . silu(e) + b[r], one warp per row, fp32 accumulation.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) adaln_kernel(const __nv_bfloat16* __restrict__ w, const float* __restrict__ b,
                                                    int rows, int t_dim, const AdaTimesteps ts, float* __restrict__ mod,
                                                    const int* status) {
  if (status && (*reinterpret_cast<const volatile int*>(status) & kDevLayout)) return;
  extern __shared__ float se[];  // [n_t][t_dim]: silu(embedding) of each timestep
  const int half = t_dim / 2;
  for (int e = threadIdx.x; e < ts.n_t * half; e += blockDim.x) {
    const int m = e / half, k = e - m * half;
    const double f = exp(-log(10000.0) * (double)k / (double)half);
    const double a = 1000.0 * (double)ts.t[m] * f;
    const double ec = cos(a), es = sin(a);
    se[m * t_dim + k] = (float)(ec / (1.0 + exp(-ec)));
    se[m * t_dim + half + k] = (float)(es / (1.0 + exp(-es)));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const __nv_bfloat16* wr = w + (size_t)r * t_dim;
    // the modality of row r: blocks' rows are [n_mod][6d] per block, the final rows [n_mod][2d]
    int m = 0;
    if (ts.n_t > 1) {
      m = r < ts.block_rows ? (r % ts.mod_block) / ts.six_d : (r - ts.block_rows) / ts.two_d;
      m = m < ts.n_t ? m : ts.n_t - 1;
    }
    const float* sm = se + m * t_dim;
    float acc = 0.f;
    for (int k0 = lane * 8; k0 < t_dim; k0 += 256) {
      const uint4 raw = *reinterpret_cast<const uint4*>(wr + k0);
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(p[q]);
        acc = fmaf(f.x, sm[k0 + 2 * q], acc);
        acc = fmaf(f.y, sm[k0 + 2 * q + 1], acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) mod[r] = acc + (b ? b[r] : 0.f);
  }
}

// ---------------------------------------------------------------------------------------------
// Euler-ancestral (eta = 0) step of the rectified flow, fp32, exactly this sequence of IEEE
// round-to-nearest operations with no contraction ([H3] "Correctness gates": euler-ancestral
// eta0 scheduler + rf_v_to_x0, gated exact):
//   x0 = x - sigma * v;  x <- x0 + (sigma_next * (x - x0)) / sigma
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float euler_one(float x, float v, float s, float sn) {
  const float x0 = __fsub_rn(x, __fmul_rn(s, v));
  const float q = __fdiv_rn(__fmul_rn(sn, __fsub_rn(x, x0)), s);
  return __fadd_rn(x0, q);
}

__global__ void euler_kernel(float* __restrict__ x, const float* __restrict__ v, long long n, float s, float sn) {
  const long long n4 = n / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = reinterpret_cast<float4*>(x)[i];
    const float4 b = reinterpret_cast<const float4*>(v)[i];
    a.x = euler_one(a.x, b.x, s, sn);
    a.y = euler_one(a.y, b.y, s, sn);
    a.z = euler_one(a.z, b.z, s, sn);
    a.w = euler_one(a.w, b.w, s, sn);
    reinterpret_cast<float4*>(x)[i] = a;
  }
  for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
    x[i] = euler_one(x[i], v[i], s, sn);
}

__global__ void euler_kernel_scalar(float* __restrict__ x, const float* __restrict__ v, long long n, float s, float sn) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
    x[i] = euler_one(x[i], v[i], s, sn);
}

// Euler step with each row's modality sigma pair: row r of x [n_tokens, d] uses
// (sigma[tags[r]], sigma_next[tags[r]]); the same fp32 operations as euler_one.
__global__ void euler_tagged_kernel(float* __restrict__ x, const float* __restrict__ v, int n_tokens, int d,
                                    const uint8_t* __restrict__ tags, const ModalSigmas sg) {
  const long long n = (long long)n_tokens * d;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
    const int m = tags[i / d];
    if (m < sg.n) x[i] = euler_one(x[i], v[i], sg.sigma[m], sg.sigma_next[m]);
  }
}

// ---------------------------------------------------------------------------------------------
// Bind-time repacks
// ---------------------------------------------------------------------------------------------
// Packed row p of the FFN up projection: group g = p / 256, w = p % 256; value rows first.
__global__ void pack_ffn_in_kernel(const __nv_bfloat16* __restrict__ src, const float* __restrict__ b_src, int F, int d,
                                   __nv_bfloat16* __restrict__ dst, float* __restrict__ b_dst) {
  const int p = blockIdx.x;
  const int g = p >> 8, w = p & 255;
  const int s = w < 128 ? 128 * g + w : F + 128 * g + (w - 128);
  if (src) {  // NULL: the biases alone (the weight is bound in another form)
    const uint4* in = reinterpret_cast<const uint4*>(src + (size_t)s * d);
    uint4* out = reinterpret_cast<uint4*>(dst + (size_t)p * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) out[i] = in[i];
  }
  if (threadIdx.x == 0) b_dst[p] = b_src ? b_src[s] : 0.f;
}

// bf16 -> f16 in place or into another buffer; a value beyond f16's finite range sets kDevRange.
__global__ void bf16_to_f16_kernel(const uint16_t* src, uint16_t* dst, long long n, int* flag) {
  bool over = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = __bfloat162float(__ushort_as_bfloat16(src[i]));
    over |= fabsf(v) > kF16Max;
    dst[i] = __half_as_ushort(__float2half_rn(v));
  }
  if (over) atomicOr(flag, kDevRange);
}

__global__ void to_f32_kernel(const void* __restrict__ src, int is_bf16, long long n, float* __restrict__ dst) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dst[i] = is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(src)[i]) : static_cast<const float*>(src)[i];
}

// Failure-path self-test: wait on an mbarrier that nothing ever arrives at, through the same bounded
// wait every pipelined kernel uses, with a short limit.  The wait must run out, record kDevTimeout
// in the status word and return, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  mbar_fence_init();
  mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}

template <int NV>
cudaError_t norm_launch_t(const float* x, const float* x_lo, int n, int d, int norm, float eps, const float* g,
                          const float* b,
                          const uint8_t* tags, const float* shift, const float* scale, long long stride, void* y,
                          int out_kind, int* status, cudaStream_t s) {
  const int rows_per_block = 8;
  cudaError_t e = launch_pdl(norm_mod_kernel<NV>, dim3((n + rows_per_block - 1) / rows_per_block),
                             dim3(32 * rows_per_block), 0, s, x, x_lo, n, d, norm, eps, g, b, tags, shift, scale,
                             stride, y, out_kind, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 8;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

cudaError_t norm_modulate_launch(const float* x, const float* x_lo, int n, int d, int norm, float eps, const float* ln_g,
                                 const float* ln_b, const uint8_t* tags, const float* shift, const float* scale,
                                 long long mod_stride, void* y, int out_kind, int* status, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (d % 1024 == 0 && d <= 8192) {
    switch (d / 1024) {
#define DIT_VPT(k)                                                                                              \
  case k: {                                                                                                     \
    static int per_sm = 0;                                                                                      \
    if (!per_sm &&                                                                                              \
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_mod_persistent_kernel<k, false>, 256, 0) != \
            cudaSuccess)                                                                                        \
      per_sm = 4;                                                                                               \
    int blocks = num_sms() * (per_sm > 0 ? per_sm : 1);                                                         \
    if (blocks > n) blocks = n;                                                                                 \
    cudaError_t e = x_lo ? launch_pdl(norm_mod_persistent_kernel<k, true>, dim3(blocks), dim3(256), 0, s, x, x_lo, n, \
                                      d, norm, eps, ln_g, ln_b, tags, shift, scale, mod_stride, y, out_kind, status) \
                         : launch_pdl(norm_mod_persistent_kernel<k, false>, dim3(blocks), dim3(256), 0, s, x, x_lo,  \
                                      n, d, norm, eps, ln_g, ln_b, tags, shift, scale, mod_stride, y, out_kind,     \
                                      status);                                                                   \
    return e != cudaSuccess ? e : cudaGetLastError();                                                           \
  }
      DIT_VPT(1) DIT_VPT(2) DIT_VPT(3) DIT_VPT(4) DIT_VPT(5) DIT_VPT(6) DIT_VPT(7) DIT_VPT(8)
#undef DIT_VPT
      default: break;
    }
  }
  switch (d / 128) {
#define DIT_NV(k) \
  case k: return norm_launch_t<k>(x, x_lo, n, d, norm, eps, ln_g, ln_b, tags, shift, scale, mod_stride, y, out_kind, status, s);
    DIT_NV(1) DIT_NV(2) DIT_NV(3) DIT_NV(4) DIT_NV(5) DIT_NV(6) DIT_NV(8) DIT_NV(10) DIT_NV(12) DIT_NV(16)
    DIT_NV(20) DIT_NV(24) DIT_NV(32) DIT_NV(40) DIT_NV(48) DIT_NV(64)
#undef DIT_NV
    default: return cudaErrorInvalidValue;
  }
}

bool norm_width_supported(int d) {
  if (d <= 0 || d % 128) return false;
  switch (d / 128) {
    case 1: case 2: case 3: case 4: case 5: case 6: case 8: case 10: case 12: case 16: case 20: case 24:
    case 32: case 40: case 48: case 64: return true;
    default: return false;
  }
}

cudaError_t rope_cache_launch(const double* pos, int n, int n_axes, const int* dims, double base, float* cos_out,
                              float* sin_out, const int* status, cudaStream_t s) {
  RopeTable tab;
  int half = 0;
  for (int a = 0; a < n_axes; ++a)
    for (int k = 0; k < dims[a] / 2; ++k) {
      if (half >= 128) return cudaErrorInvalidValue;
      tab.inv[half] = (float)pow(base, -2.0 * (double)k / (double)dims[a]);
      tab.axis[half] = (unsigned char)a;
      ++half;
    }
  if (n <= 0 || half == 0) return cudaSuccess;
  rope_cache_kernel<<<grid_for((long long)n * half, 256), 256, 0, s>>>(pos, n, half, tab, cos_out, sin_out, status);
  return cudaGetLastError();
}

cudaError_t adaln_launch(const void* w, const float* b, int rows, int t_dim, const AdaTimesteps& ts, float* mod,
                         const int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (ts.n_t < 1 || ts.n_t > kMaxModalTimesteps) return cudaErrorInvalidValue;
  if ((size_t)ts.n_t * t_dim * sizeof(float) > 48 * 1024) return cudaErrorInvalidValue;  // static smem budget
  const int warps_per_block = 8;
  int blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  adaln_kernel<<<blocks, 32 * warps_per_block, ts.n_t * t_dim * sizeof(float), s>>>(
      static_cast<const __nv_bfloat16*>(w), b, rows, t_dim, ts, mod, status);
  return cudaGetLastError();
}

cudaError_t euler_launch(float* x, const float* v, long long n, float sigma, float sigma_next, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
  if (aligned)
    euler_kernel<<<grid_for(n / 4 + 1, 256), 256, 0, s>>>(x, v, n, sigma, sigma_next);
  else
    euler_kernel_scalar<<<grid_for(n, 256), 256, 0, s>>>(x, v, n, sigma, sigma_next);
  return cudaGetLastError();
}

cudaError_t euler_tagged_launch(float* x, const float* v, int n_tokens, int d, const uint8_t* tags,
                                const ModalSigmas& sg, cudaStream_t s) {
  const long long n = (long long)n_tokens * d;
  if (n <= 0) return cudaSuccess;
  euler_tagged_kernel<<<grid_for(n, 256), 256, 0, s>>>(x, v, n_tokens, d, tags, sg);
  return cudaGetLastError();
}

// Row r of the [q_all | k_all | v_all] order, r = s * H * Dh + h * Dh + j (s = 0 q, 1 k, 2 v), is
// row h * 3 Dh + s * Dh + j of the per-head interleaved [q_h | k_h | v_h] order; rows of row_bytes.
__global__ void qkv_deinterleave_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int H, int Dh,
                                        int row_bytes) {
  const int r = blockIdx.x;
  const int HD = H * Dh;
  const int sgm = r / HD, h = (r - sgm * HD) / Dh, j = r - sgm * HD - h * Dh;
  const size_t from = ((size_t)h * 3 * Dh + (size_t)sgm * Dh + j) * row_bytes;
  const size_t to = (size_t)r * row_bytes;
  for (int b = threadIdx.x; b < row_bytes; b += blockDim.x) dst[to + b] = src[from + b];
}

cudaError_t qkv_deinterleave_launch(const void* src, void* dst, int H, int Dh, int row_bytes, cudaStream_t s) {
  if (H < 1 || Dh < 1 || row_bytes < 1) return cudaErrorInvalidValue;
  qkv_deinterleave_kernel<<<3 * H * Dh, 128, 0, s>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), H, Dh,
                                                     row_bytes);
  return cudaGetLastError();
}

cudaError_t pack_ffn_in_launch(const void* w_in, const float* b_in, int F, int d, void* w_packed, float* b_packed,
                               cudaStream_t s) {
  pack_ffn_in_kernel<<<2 * F, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(w_in), b_in, F, d,
                                           static_cast<__nv_bfloat16*>(w_packed), b_packed);
  return cudaGetLastError();
}

cudaError_t to_f32_launch(const void* src, int src_is_bf16, long long n, float* dst, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  to_f32_kernel<<<grid_for(n, 256), 256, 0, s>>>(src, src_is_bf16, n, dst);
  return cudaGetLastError();
}

cudaError_t bf16_to_f16_launch(const void* src, void* dst, long long n, int* flag, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  bf16_to_f16_kernel<<<grid_for(n, 256), 256, 0, s>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst),
                                                      n, flag);
  return cudaGetLastError();
}

cudaError_t wait_timeout_selftest_launch(int* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace dit
