// tcgen05 GEMM engine: D[M, N] = A[M, K] . B[N, K]^T, bf16 operands, fp32 accumulation in TMEM,
// with the DiT's epilogues fused in.  Every linear map of the forward runs here: the fused QKV
// projection (bias + NeoX RoPE + q/k/v split), the attention output projection and the FFN down
// projection (bias + modality-gated residual add into the fp32 stream), and the FFN up projection
// (bias + value * silu(gate)).  [M3] "What moved": every Linear is a MatmulBT with a rank-1 bias
// add; [H3] "The device-resident forward (W2b)": QkvSplit, RopeFromCache, SiluAndMul and the
// indexed AdaLN gated add, here folded into the GEMM epilogue instead of separate passes.
//
// Design (one CTA per SM, persistent over output tiles):
//   tile 128 x 256, K step 64, 4-stage TMA -> shared-memory ring (128-byte swizzle)
//   warp 0   TMA producer (one elected lane)
//   warp 1   TMEM allocator + UMMA issuer (one lane): tcgen05.mma M=128 N=256 K=16
//   warps 2-5 epilogue: each warp reads its 32 TMEM lanes (= 32 tile rows) with tcgen05.ld,
//            one thread per output row
//   the 512 TMEM columns hold two 128x256 fp32 accumulators, so the epilogue of tile i overlaps
//   the main loop of tile i+1.
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace dit {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int GEMM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr int SMEM_BYTES_RESID = SMEM_BYTES + BM * 64 * 4;  // + the residual epilogue's staging tile
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct TileCoord {
  int mb, nb;
};

// Raster: N-blocks in groups of `gn`; within a group the N-block index runs fastest, so the
// group's slice of B stays in L2 while consecutive M-blocks stream through.
__device__ __forceinline__ TileCoord tile_coord(int tile, int n_m, int n_n, int gn) {
  int full_groups = n_n / gn;
  int per_group = n_m * gn;
  int g = tile / per_group;
  int width = gn;
  int r = tile - g * per_group;
  if (g >= full_groups) {
    width = n_n - full_groups * gn;
    r = tile - full_groups * per_group;
    g = full_groups;
  }
  TileCoord c;
  c.mb = r / width;
  c.nb = g * gn + (r - c.mb * width);
  return c;
}

__device__ __forceinline__ void load_bias4(const float* b, int col, float (&o)[4]) {
  if (b) {
    float4 v = *reinterpret_cast<const float4*>(b + col);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else {
    o[0] = o[1] = o[2] = o[3] = 0.f;
  }
}

// ---------------------------------------------------------------------------------------------
// epilogues: the calling thread owns tile row `row` (global), TMEM address `t` = its lane, the
// accumulator's column 0.  n0 = first global output column of the tile.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void epi_store(const GemmArgs& a, uint32_t t, int row, int n0) {
  const bool live = row < a.M;
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    uint32_t r[32];
    tmem_ld32_sync(t + c, r);
    if (!live) continue;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float b[4];
      load_bias4(a.bias, n0 + c + i, b);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[i + j] = __uint_as_float(r[i + j]) + b[j];
    }
    if (a.out_kind == 0) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (size_t)row * a.N + n0 + c;
#pragma unroll
      for (int i = 0; i < 32; i += 8)
        st_global_v4(o + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                     pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
    } else {
      float* o = static_cast<float*>(a.out) + (size_t)row * a.N + n0 + c;
#pragma unroll
      for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* o, const float (&v)[16]) {
  st_global_v4(o, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  st_global_v4(o + 8, pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
               pack_bf16x2(v[14], v[15]));
}

// Fused QKV epilogue.  Columns [0, d) are q, [d, 2d) k, [2d, 3d) v ([q_all | k_all | v_all]);
// d % 256 == 0, so a tile never straddles two of them, and a tile holds 256 / Dh whole heads.
// q and k get NeoX rotate_half on the first R = 2 * rot_half dims of each head: for j < R/2,
//   out_j = a_j cos_j - a_{j+R/2} sin_j,   out_{j+R/2} = a_{j+R/2} cos_j + a_j sin_j,
// with a = acc + bias and cos/sin the row's cache entries.
__device__ __forceinline__ void epi_qkv(const GemmArgs& a, uint32_t t, int row, int n0) {
  const bool live = row < a.M;
  const int seg = n0 / a.d;
  const int col0 = n0 - seg * a.d;
  if (seg == 2) {
    // v is stored transposed; its padding columns [M, n_pad) are written as zeros so that the
    // attention's masked key/value tiles never multiply uninitialised memory (0 * NaN = NaN).
    __nv_bfloat16* vt = static_cast<__nv_bfloat16*>(a.vt);
    const bool pad = !live && row < a.n_pad;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      tmem_ld32_sync(t + c, r);
      if (!live && !pad) continue;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float b[4];
        load_bias4(a.bias, n0 + c + i, b);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          vt[(size_t)(col0 + c + i + j) * a.n_pad + row] =
              __float2bfloat16_rn(live ? __uint_as_float(r[i + j]) + b[j] : 0.f);
      }
    }
    return;
  }
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(seg == 0 ? a.q : a.k) + (size_t)row * a.d + col0;
  const int Dh = a.head_dim, half = a.rot_half;
  const float* cs = a.cos_cache + (size_t)row * half;
  const float* sn = a.sin_cache + (size_t)row * half;
#pragma unroll 1
  for (int hb = 0; hb < BN; hb += Dh) {
#pragma unroll 1
    for (int c = 0; c < half; c += 16) {
      uint32_t r1[16], r2[16];
      tmem_ld16(t + hb + c, r1);
      tmem_ld16(t + hb + half + c, r2);
      tmem_ld_wait_regs(r1);
      tmem_ld_wait_regs(r2);
      if (!live) continue;
      float o1[16], o2[16];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        float b1[4], b2[4];
        load_bias4(a.bias, n0 + hb + c + i, b1);
        load_bias4(a.bias, n0 + hb + half + c + i, b2);
        float4 cv = *reinterpret_cast<const float4*>(cs + c + i);
        float4 sv = *reinterpret_cast<const float4*>(sn + c + i);
        float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x1 = __uint_as_float(r1[i + j]) + b1[j];
          float x2 = __uint_as_float(r2[i + j]) + b2[j];
          o1[i + j] = x1 * cc[j] - x2 * ss[j];
          o2[i + j] = x2 * cc[j] + x1 * ss[j];
        }
      }
      store_bf16x16(dst + hb + c, o1);
      store_bf16x16(dst + hb + half + c, o2);
    }
#pragma unroll 1
    for (int c = 2 * half; c < Dh; c += 16) {  // partial rotary: dims >= R pass through
      uint32_t r1[16];
      tmem_ld16(t + hb + c, r1);
      tmem_ld_wait_regs(r1);
      if (!live) continue;
      float o1[16];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        float b1[4];
        load_bias4(a.bias, n0 + hb + c + i, b1);
#pragma unroll
        for (int j = 0; j < 4; ++j) o1[i + j] = __uint_as_float(r1[i + j]) + b1[j];
      }
      store_bf16x16(dst + hb + c, o1);
    }
  }
}

// x[row, n0 + c] += gate[tag[row]][n0 + c] * (acc + bias)     (gate == nullptr: plain add)
//
// The residual stream is fp32 in HBM, so this epilogue is a read-modify-write of a 128 x 256 fp32
// tile.  TMEM hands each thread one row, which would make every global access a 32-row scatter;
// instead the tile goes through shared memory 64 columns at a time:
//   phase A  each thread moves its row's 64 accumulator columns TMEM -> registers -> shared memory
//            (16-byte chunks XOR-swizzled by row so a warp's stores spread over all banks)
//   phase B  each warp walks 32 rows; per row its 32 lanes own 2 adjacent columns, so the loads and
//            stores of x (and of the gate and bias) are 256 contiguous bytes per row.
constexpr int RES_COLS = 64;
constexpr int RES_BATCH = 32;  // rows whose loads a warp has in flight at once

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void epi_resid(const GemmArgs& a, uint32_t t, int tile_row0, int quarter, int ew, int n0,
                                          float* stage, uint64_t* tempty_bar) {
  const int lane = threadIdx.x & 31;
  const int r_own = quarter * 32 + lane;  // the tile row whose TMEM lane this thread reads
  const uint32_t st_row = smem_u32(stage) + r_own * (RES_COLS * 4);
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += RES_COLS) {
    // phase A: TMEM -> shared memory (swizzled)
#pragma unroll
    for (int h = 0; h < RES_COLS; h += 32) {
      uint32_t r[32];
      tmem_ld32_sync(t + c0 + h, r);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int chunk = (h >> 2) + q;  // 16-byte chunk index within the 256-byte row
        st_shared_v4(st_row + ((chunk ^ (r_own & 7)) << 4), r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
      }
    }
    if (c0 + RES_COLS == BN) {
      // every accumulator column of this tile is out of TMEM: hand the buffer back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);
    }
    epi_bar();
    // phase B: coalesced read-modify-write of 32 rows x 64 columns per warp
    const int col = n0 + c0 + 2 * lane;
    float2 bb = make_float2(0.f, 0.f);
    if (a.bias) bb = *reinterpret_cast<const float2*>(a.bias + col);
    const int chunk = lane >> 1, half8 = (lane & 1) * 8;
#pragma unroll 1
    for (int rr0 = 0; rr0 < 32; rr0 += RES_BATCH) {
      float2 acc[RES_BATCH], xv[RES_BATCH], gv[RES_BATCH];
      int rows[RES_BATCH];
#pragma unroll
      for (int u = 0; u < RES_BATCH; ++u) {
        const int rt = ew * 32 + rr0 + u;
        rows[u] = tile_row0 + rt;
        const uint32_t sa = smem_u32(stage) + rt * (RES_COLS * 4) + ((chunk ^ (rt & 7)) << 4) + half8;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(acc[u].x), "=f"(acc[u].y) : "r"(sa));
        if (rows[u] < a.M) {
          xv[u] = *reinterpret_cast<const float2*>(a.x + (size_t)rows[u] * a.N + col);
          gv[u] = a.gate ? *reinterpret_cast<const float2*>(a.gate + (size_t)a.tags[rows[u]] * a.gate_stride + col)
                         : make_float2(1.f, 1.f);
        }
      }
#pragma unroll
      for (int u = 0; u < RES_BATCH; ++u) {
        if (rows[u] < a.M) {
          float2 o;
          o.x = xv[u].x + gv[u].x * (acc[u].x + bb.x);
          o.y = xv[u].y + gv[u].y * (acc[u].y + bb.y);
          *reinterpret_cast<float2*>(a.x + (size_t)rows[u] * a.N + col) = o;
        }
      }
    }
    epi_bar();  // the staging buffer is reused by the next column block
  }
}

// Tile columns [0, 128) hold value features f0 .. f0+127 and [128, 256) their gates
// (the interleaved packing of the FFN up projection); h[row, f0 + j] = u_j * silu(g_j).
__device__ __forceinline__ void epi_swiglu(const GemmArgs& a, uint32_t t, int row, int n0) {
  const bool live = row < a.M;
  const int F = a.N / 2;
  const int f0 = n0 / 2;
  __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(a.out) + (size_t)row * F + f0;
#pragma unroll 1
  for (int c = 0; c < BN / 2; c += 16) {
    uint32_t ru[16], rg[16];
    tmem_ld16(t + c, ru);
    tmem_ld16(t + BN / 2 + c, rg);
    tmem_ld_wait_regs(ru);
    tmem_ld_wait_regs(rg);
    if (!live) continue;
    float h[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      float bu[4], bg[4];
      load_bias4(a.bias, n0 + c + i, bu);
      load_bias4(a.bias, n0 + BN / 2 + c + i, bg);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float u = __uint_as_float(ru[i + j]) + bu[j];
        float g = __uint_as_float(rg[i + j]) + bg[j];
        h[i + j] = u * silu_f(g);
      }
    }
    store_bf16x16(hrow + c, h);
  }
}

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* res_stage = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);  // residual epilogue only

  if (args.status && (*reinterpret_cast<volatile int*>(args.status) & kDevLayout)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (args.M + BM - 1) / BM, n_n = args.N / BN, k_blocks = args.K / BK;
  const int tiles = n_m * n_n;
  const int gn = args.group_n > 0 ? args.group_n : n_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        TileCoord tc = tile_coord(tile, n_m, n_n, gn);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) goto producer_done;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, tc.mb * BM);
          tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, tc.nb * BN);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: wait until the MMAs consumed every stage we filled, so no TMA write into this
      // CTA's shared memory is still in flight when the CTA exits.
      for (int s = 0; s < STAGES; ++s) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), IDESC, (kb | k) != 0);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    const int quarter = warp & 3;  // TMEM lanes [32 * quarter, +32) belong to this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      TileCoord tc = tile_coord(tile, n_m, n_n, gn);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, args.status)) break;
      tc_fence_after();
      const int row = tc.mb * BM + quarter * 32 + lane;
      const uint32_t t = tmem + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int n0 = tc.nb * BN;
      if (EPI == kEpiGatedResid) {
        epi_resid(args, t, tc.mb * BM, quarter, warp - 2, n0, res_stage, &tempty[acc]);
      } else {
        if (EPI == kEpiStore) epi_store(args, t, row, n0);
        if (EPI == kEpiQkvRope) epi_qkv(args, t, row, n0);
        if (EPI == kEpiSwiglu) epi_swiglu(args, t, row, n0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int EPI>
cudaError_t launch_t(const void* A, const void* B, const GemmArgs& args, cudaStream_t stream) {
  constexpr int smem = EPI == kEpiGatedResid ? SMEM_BYTES_RESID : SMEM_BYTES;
  static unsigned long long smem_set = 0;
  cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(gemm_kernel<EPI>), smem, &smem_set);
  if (e != cudaSuccess) return e;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, A, args.K, args.M, (uint64_t)args.K * 2, BK, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tb, B, args.K, args.N, (uint64_t)args.K * 2, BK, BN)) return cudaErrorInvalidValue;
  const int tiles = ((args.M + BM - 1) / BM) * (args.N / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  gemm_kernel<EPI><<<grid, GEMM_THREADS, smem, stream>>>(ta, tb, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_launch(int epilogue, const void* A, const void* B, const GemmArgs& args_in, cudaStream_t stream) {
  GemmArgs args = args_in;
  if (args.M <= 0) return cudaSuccess;
  if (args.group_n <= 0) {
    // Keep a group's slice of B within ~48 MB of L2.
    long long per_nb = (long long)BN * args.K * 2;
    int g = (int)((48ll << 20) / (per_nb > 0 ? per_nb : 1));
    args.group_n = g < 1 ? 1 : g;
  }
  switch (epilogue) {
    case kEpiStore: return launch_t<kEpiStore>(A, B, args, stream);
    case kEpiQkvRope: return launch_t<kEpiQkvRope>(A, B, args, stream);
    case kEpiGatedResid: return launch_t<kEpiGatedResid>(A, B, args, stream);
    case kEpiSwiglu: return launch_t<kEpiSwiglu>(A, B, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dit
