// Latent <-> token packing and the row maps of the per-modality fp32 islands.
//
// [H3] "Correctness gates": patchify / unpatchify / audio pack / unpack are exact maps with a
// round-trip identity.  A latent [C][T*pt][H*ph][W*pw] becomes T*H*W tokens in (t, h, w) order,
// w fastest (the packed layout's order); the C*pt*ph*pw features of a token are its patch in
// (c, a, b, e) order, e fastest, the order a Conv3d weight [d][C][pt][ph][pw] flattens in, so the
// patch projection is a plain linear over the token ([H3] "Encoder complete": kernel == stride).
// Audio pack is the same map on a [C][T] latent with H = W = 1 and a 1x1x1 patch.
//
//   patch_kernel<false>   latent -> tokens   } one CTA per (t, h, run of w): the patch rows of the
//   patch_kernel<true>    tokens -> latent   } run are contiguous on both sides, so the CTA stages
//                                              them through shared memory and both the latent rows
//                                              and the token rows move as coalesced streams
//   row_map_kernel        rows of each modality in increasing packed order, from the tags
#include "common.cuh"
#include "kernels.h"

namespace dit {

namespace {

constexpr int kPatchThreads = 256;
constexpr int kPatchSmemFloats = 12 * 1024;  // 48 KB of static shared memory per CTA

// Shared tile [Wc][P + 1] (the +1 keeps the column writes of the latent side off one bank).
// Latent side: for each (c, a, b) the run of Wc patches is one contiguous segment of Wc * pw
// floats of latent row (c, t*pt + a, h*ph + b).  Token side: tokens (t, h, w0 .. w0+Wc) are
// Wc consecutive rows of P floats.
template <bool kInverse>
__global__ void __launch_bounds__(kPatchThreads) patch_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                             int C, int T, int H, int W, int pt, int ph, int pw,
                                                             int Wc) {
  __shared__ float tile[kPatchSmemFloats];
  const int runs_per_row = (W + Wc - 1) / Wc;
  const int th = blockIdx.x / runs_per_row;
  const int w0 = (blockIdx.x - th * runs_per_row) * Wc;
  const int t = th / H, h = th - t * H;
  const int wn = min(Wc, W - w0);
  const int P = C * pt * ph * pw;
  const int ld = P + 1;
  const size_t Hf = (size_t)H * ph, Wf = (size_t)W * pw, Tf = (size_t)T * pt;
  const int seg = wn * pw;              // floats of one latent segment
  const int n_seg = C * pt * ph;        // segments of the run, one per (c, a, b)
  const size_t tok0 = ((size_t)t * H + h) * W + w0;
  // latent segment q = (c * pt + a) * ph + b starts at lat[c][t*pt + a][h*ph + b][w0*pw]
  auto seg_base = [&](int q) -> size_t {
    const int b = q % ph, ca = q / ph;
    const int a = ca % pt, c = ca / pt;
    return (((size_t)c * Tf + (size_t)t * pt + a) * Hf + (size_t)h * ph + b) * Wf + (size_t)w0 * pw;
  };
  if (!kInverse) {
    for (int i = threadIdx.x; i < n_seg * seg; i += blockDim.x) {
      const int q = i / seg, j = i - q * seg;
      const int wi = j / pw, e = j - wi * pw;
      tile[wi * ld + q * pw + e] = src[seg_base(q) + j];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < wn * P; i += blockDim.x) {
      const int wi = i / P, f = i - wi * P;
      dst[(tok0 + wi) * P + f] = tile[wi * ld + f];
    }
  } else {
    for (int i = threadIdx.x; i < wn * P; i += blockDim.x) {
      const int wi = i / P, f = i - wi * P;
      tile[wi * ld + f] = src[(tok0 + wi) * P + f];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_seg * seg; i += blockDim.x) {
      const int q = i / seg, j = i - q * seg;
      const int wi = j / pw, e = j - wi * pw;
      dst[seg_base(q) + j] = tile[wi * ld + q * pw + e];
    }
  }
}

// One CTA of 1024 threads walks the tags in chunks of 1024.  Per chunk and modality a warp ballot
// gives each token its rank inside its warp and an exclusive scan over the 32 warp counts gives the
// warp's rank inside the chunk; running counts carry across chunks.  rows[off[m] + k] = the k-th
// token tagged m.  A final count that disagrees with the caller's count[m] marks the layout invalid
// (code 8); no row at or past the caller's count is ever written.
__global__ void __launch_bounds__(1024) row_map_kernel(const uint8_t* __restrict__ tags, int n, const ModalRows mr,
                                                       int* __restrict__ rows, int* layout_code, int* status) {
  if (*reinterpret_cast<const volatile int*>(status) & kDevLayout) return;
  __shared__ int warp_cnt[kMaxModalTimesteps][32];
  __shared__ int warp_pre[kMaxModalTimesteps][32];
  __shared__ int chunk_tot[kMaxModalTimesteps];
  __shared__ int base[kMaxModalTimesteps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  if (threadIdx.x < kMaxModalTimesteps) base[threadIdx.x] = 0;
  __syncthreads();
  for (int c0 = 0; c0 < n; c0 += 1024) {
    const int i = c0 + threadIdx.x;
    const int tag = i < n ? (int)tags[i] : -1;
    for (int m = 0; m < mr.n; ++m) {
      const unsigned bal = __ballot_sync(0xffffffffu, tag == m);
      if (lane == 0) warp_cnt[m][warp] = __popc(bal);
    }
    __syncthreads();
    if (warp < mr.n) {  // warp m scans modality m's 32 warp counts
      const int v = warp_cnt[warp][lane];
      int incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      warp_pre[warp][lane] = incl - v;
      if (lane == 31) chunk_tot[warp] = incl;
    }
    __syncthreads();
    for (int m = 0; m < mr.n; ++m) {
      const unsigned bal = __ballot_sync(0xffffffffu, tag == m);
      if (tag == m) {
        const int k = base[m] + warp_pre[m][warp] + __popc(bal & lt_mask);
        if (k < mr.count[m]) rows[mr.off[m] + k] = i;
      }
    }
    __syncthreads();
    if (threadIdx.x < mr.n) base[threadIdx.x] += chunk_tot[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x < mr.n && base[threadIdx.x] != mr.count[threadIdx.x]) {
    atomicOr(status, kDevLayout);
    *layout_code = 8;
  }
}

}  // namespace

cudaError_t patch_launch(const float* src, float* dst, int C, int T, int H, int W, int pt, int ph, int pw,
                         int inverse, cudaStream_t s) {
  if (C < 1 || T < 1 || H < 1 || W < 1 || pt < 1 || ph < 1 || pw < 1) return cudaErrorInvalidValue;
  const long long P = (long long)C * pt * ph * pw;
  if (P + 1 > kPatchSmemFloats) return cudaErrorInvalidValue;
  int Wc = (int)(kPatchSmemFloats / (P + 1));
  if (Wc > W) Wc = W;
  const long long blocks = (long long)T * H * ((W + Wc - 1) / Wc);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (inverse)
    patch_kernel<true><<<(unsigned)blocks, kPatchThreads, 0, s>>>(src, dst, C, T, H, W, pt, ph, pw, Wc);
  else
    patch_kernel<false><<<(unsigned)blocks, kPatchThreads, 0, s>>>(src, dst, C, T, H, W, pt, ph, pw, Wc);
  return cudaGetLastError();
}

cudaError_t row_map_launch(const uint8_t* tags, int n, const ModalRows& mr, int* rows, int* layout_code, int* status,
                           cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (mr.n < 1 || mr.n > kMaxModalTimesteps) return cudaErrorInvalidValue;
  row_map_kernel<<<1, 1024, 0, s>>>(tags, n, mr, rows, layout_code, status);
  return cudaGetLastError();
}

}  // namespace dit
