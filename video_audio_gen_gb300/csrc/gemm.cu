// tcgen05 GEMM engine: D[M, N] = A[M, K] . B[N, K]^T, bf16 operands, fp32 accumulation in TMEM,
// with the DiT's epilogues fused in.  Every linear map of the forward runs here: the fused QKV
// projection (bias + NeoX RoPE + q/k/v split), the attention output projection and the FFN down
// projection (bias + modality-gated residual add into the fp32 stream), and the FFN up projection
// (bias + value * silu(gate)).  [M3] "What moved": every Linear is a MatmulBT with a rank-1 bias
// add; [H3] "The device-resident forward (W2b)": QkvSplit, RopeFromCache, SiluAndMul and the
// indexed AdaLN gated add, here folded into the GEMM epilogue instead of separate passes.
//
// Design for bf16 / f16 weights (gemm_pair_kernel: CTA pairs, one CTA per SM, persistent over
// 256 x 256 output tiles):
//   K step 64, a 6-stage TMA -> shared-memory ring (128-byte swizzle) per CTA holding its own 128
//   rows of A and its half (128 rows) of the B tile
//   warp 0   TMA producer (one lane per CTA)
//   warp 1   TMEM allocator (both CTAs) + UMMA issuer (the first CTA, elect.sync): tcgen05.mma
//            cta_group::2 M=256 N=256 K=16, each CTA's TMEM taking its own 128 rows
//   warps 2-9 epilogue: each warp reads its 32 TMEM lanes (= 32 tile rows) with tcgen05.ld,
//            one thread per output row; warps 2-5 take the tile's columns [0, 128) and warps 6-9
//            [128, 256), so two warps share each lane quarter (a warp may only read the quarter
//            warp % 4) and a tile's epilogue runs in half the time of one warp per quarter
//   the 512 TMEM columns hold two 128x256 fp32 accumulators, so the epilogue of tile i overlaps
//   the main loop of tile i+1.
// gemm_kernel (one CTA of 128 x 256 tiles, 4 stages of 48 KB) runs the NVFP4 mode below.
//
// NVFP4 weights ([H3] "What this push adds": U8 codes two per byte, an E4M3 scale per 16 along K,
// an F32 global scale).  Every E2M1 x E4M3 product is exact in f16, and E2M1 -> f16 is one
// conversion per pair, so this mode runs the same kind::f16 MMA with f16 operands:
//   4 stages (3 with the residual epilogue's staging tile) of {A f16 tile (TMA), the dequantised
//   B tile}, and a 2-slot ring of packed weight tiles (one 9 KB bulk copy each of a bind-time
//   tile-contiguous repack), released by the converters once expanded
//   warps 6-13 converters: wait for a packed tile, expand 256 rows x 64 codes with their scales
//            into the stage's 128-byte-swizzled f16 B tile (the layout a TMA load would have
//            written), fence the writes to the async proxy, release the packed slot and arrive on
//            the stage's full barrier, which therefore completes when A has landed AND B is
//            expanded: the MMA thread waits once per K-block, as in the bf16 mode (every wait in
//            the issuing thread idles the pipe)
//   the epilogues take acc * global scale in place of acc.
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace dit {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each on half of the tile's columns
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
// NVFP4 mode
constexpr int Q_STAGES = 4, Q_STAGES_RESID = 3;  // A + dequantised B stages
constexpr int Q_RAW_SLOTS = 2;                   // packed weight tiles in flight
constexpr int Q_RAW_BYTES = kNvfp4TileBytes;     // 256 rows x 32 bytes of codes, then 256 x 4 scales
constexpr int Q_CODE_BYTES = BN * BK / 2;
constexpr int Q_CONV_WARPS = 8;                  // one weight row per converter thread
constexpr int Q_EPI_WARPS = 4;                   // one per lane quarter, all 256 columns
constexpr int Q_BASE_THREADS = 64 + 32 * Q_EPI_WARPS;
constexpr int Q_THREADS = Q_BASE_THREADS + 32 * Q_CONV_WARPS;
constexpr int Q_SMEM_BYTES = Q_STAGES * STAGE_BYTES + Q_RAW_SLOTS * Q_RAW_BYTES + 1024 + 256;
constexpr int Q_SMEM_BYTES_RESID = Q_STAGES_RESID * STAGE_BYTES + Q_RAW_SLOTS * Q_RAW_BYTES + 1024 + 256 + BM * 64 * 4;
constexpr uint32_t IDESC_F16 = idesc_f16_f32(BM, BN);
static_assert(Q_RAW_BYTES == BN * BK / 2 + BN * BK / 16, "packed tile size");
static_assert(Q_SMEM_BYTES <= 227 * 1024 && Q_SMEM_BYTES_RESID <= 227 * 1024, "NVFP4 stages exceed shared memory");

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
// accumulator's column 0.  n0 = first global output column of the tile.  The tile's columns are
// split into NG groups (NG warps per lane quarter); the caller's warp handles group `grp`.
// ---------------------------------------------------------------------------------------------
template <int NG>
__device__ __forceinline__ void epi_store(const GemmArgs& a, uint32_t t, int row, int n0, int grp) {
  const bool live = row < a.M;
  constexpr int GC = BN / NG;
#pragma unroll 1
  for (int c = grp * GC; c < (grp + 1) * GC; c += 32) {
    uint32_t r[32];
    tmem_ld32_sync(t + c, r);
    if (!live) continue;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float b[4];
      load_bias4(a.bias, n0 + c + i, b);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[i + j] = __uint_as_float(r[i + j]) * a.w_scale + b[j];
    }
    if (a.out_kind == 0) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (size_t)row * a.N + n0 + c;
#pragma unroll
      for (int i = 0; i < 32; i += 8)
        st_global_v4(o + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                     pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
    } else if (a.out_kind == 2) {
      __half* o = static_cast<__half*>(a.out) + (size_t)row * a.N + n0 + c;
#pragma unroll
      for (int i = 0; i < 32; i += 8)
        st_global_v4(o + i, pack_f16x2(v[i], v[i + 1]), pack_f16x2(v[i + 2], v[i + 3]),
                     pack_f16x2(v[i + 4], v[i + 5]), pack_f16x2(v[i + 6], v[i + 7]));
    } else {
      float* o = static_cast<float*>(a.out) + (size_t)row * a.N + n0 + c;
#pragma unroll
      for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
}

// The epilogues' 16-bit outputs (q, k, h) are read by the next kernel, not by this GEMM: they are
// stored evict-first so that they do not push the weight panels out of L2.
__device__ __forceinline__ void store_f16x16(__half* o, const float (&v)[16]) {
  st_global_v4_stream(o, pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                      pack_f16x2(v[6], v[7]));
  st_global_v4_stream(o + 8, pack_f16x2(v[8], v[9]), pack_f16x2(v[10], v[11]), pack_f16x2(v[12], v[13]),
               pack_f16x2(v[14], v[15]));
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* o, const float (&v)[16]) {
  st_global_v4_stream(o, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
  st_global_v4_stream(o + 8, pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
               pack_bf16x2(v[14], v[15]));
}

// NeoX rotate_half on W-column chunks of one head: columns [c, c + W) and [c + half, ...), each value
// x = (acc + bias) * rn; out_j = x_j cos_j - x_{j+half} sin_j, out_{j+half} = x_{j+half} cos_j + x_j sin_j.
template <int W>
__device__ __forceinline__ void rope_chunk(const GemmArgs& a, uint32_t t, int hb, int c, int half, float rn, bool live,
                                           const float* cs, const float* sn, uint16_t* dst, int n0) {
  uint32_t r1[W], r2[W];
  if constexpr (W == 16) {
    tmem_ld16(t + hb + c, *reinterpret_cast<uint32_t(*)[16]>(r1));
    tmem_ld16(t + hb + half + c, *reinterpret_cast<uint32_t(*)[16]>(r2));
    tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[16]>(r1));
    tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[16]>(r2));
  } else {
    tmem_ld8(t + hb + c, *reinterpret_cast<uint32_t(*)[8]>(r1));
    tmem_ld8(t + hb + half + c, *reinterpret_cast<uint32_t(*)[8]>(r2));
    tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[8]>(r1));
    tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[8]>(r2));
  }
  if (!live) return;
  float o1[W], o2[W];
#pragma unroll
  for (int i = 0; i < W; i += 4) {
    float b1[4], b2[4];
    load_bias4(a.bias, n0 + hb + c + i, b1);
    load_bias4(a.bias, n0 + hb + half + c + i, b2);
    float4 cv = *reinterpret_cast<const float4*>(cs + c + i);
    float4 sv = *reinterpret_cast<const float4*>(sn + c + i);
    float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float x1 = (__uint_as_float(r1[i + j]) * a.w_scale + b1[j]) * rn;
      float x2 = (__uint_as_float(r2[i + j]) * a.w_scale + b2[j]) * rn;
      o1[i + j] = x1 * cc[j] - x2 * ss[j];
      o2[i + j] = x2 * cc[j] + x1 * ss[j];
    }
  }
  const bool f = a.f16;
#pragma unroll
  for (int i = 0; i < W; i += 8) {
    st_global_v4_stream(dst + hb + c + i, pack16(f, o1[i], o1[i + 1]), pack16(f, o1[i + 2], o1[i + 3]),
                 pack16(f, o1[i + 4], o1[i + 5]), pack16(f, o1[i + 6], o1[i + 7]));
    st_global_v4_stream(dst + hb + half + c + i, pack16(f, o2[i], o2[i + 1]), pack16(f, o2[i + 2], o2[i + 3]),
                 pack16(f, o2[i + 4], o2[i + 5]), pack16(f, o2[i + 6], o2[i + 7]));
  }
}

// Fused QKV epilogue.  Columns [0, d) are q, [d, 2d) k, [2d, 3d) v ([q_all | k_all | v_all]);
// d % 256 == 0, so a tile never straddles two of them, and a tile holds 256 / Dh whole heads.
// q and k get NeoX rotate_half on the first R = 2 * rot_half dims of each head: for j < R/2,
//   out_j = a_j cos_j - a_{j+R/2} sin_j,   out_{j+R/2} = a_{j+R/2} cos_j + a_j sin_j,
// with a = acc + bias and cos/sin the row's cache entries.  With qk_norm, a is first divided by the
// head's RMS, sqrt(mean(a^2) + eps) ([H3] "Update: video-VAE decoder block ported": per-head RMS
// q/k norm without affine).
// A head is never split between column groups: with Dh wider than a group, group 0 takes them all.
template <int NG>
__device__ __forceinline__ void epi_qkv(const GemmArgs& a, uint32_t t, int row, int n0, int grp) {
  const bool live = row < a.M;
  const int seg = n0 / a.d;
  const int col0 = n0 - seg * a.d;
  constexpr int GC = BN / NG;
  if (seg == 2) {
    // v is stored transposed; its padding columns [M, n_pad) are written as zeros so that the
    // attention's masked key/value tiles never multiply uninitialised memory (0 * NaN = NaN).
    uint16_t* vt = static_cast<uint16_t*>(a.vt);
    const bool pad = !live && row < a.n_pad;
    const bool f = a.f16;
#pragma unroll 1
    for (int c = grp * GC; c < (grp + 1) * GC; c += 32) {
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
              to16(f, live ? __uint_as_float(r[i + j]) * a.w_scale + b[j] : 0.f);
      }
    }
    return;
  }
  uint16_t* dst = static_cast<uint16_t*>(seg == 0 ? a.q : a.k) + (size_t)row * a.d + col0;
  const int Dh = a.head_dim, half = a.rot_half;
  const float* cs = a.cos_cache + (size_t)row * half;
  const float* sn = a.sin_cache + (size_t)row * half;
  const int h_lo = Dh <= GC ? grp * GC : (grp == 0 ? 0 : BN);
  const int h_hi = Dh <= GC ? h_lo + GC : BN;
#pragma unroll 1
  for (int hb = h_lo; hb < h_hi; hb += Dh) {
    // qk_norm: x / sqrt(mean over the head of x^2 + eps), x = acc + bias, before the rotation
    float rn = 1.f;
    if (a.qk_norm) {
      float ss = 0.f;
#pragma unroll 1
      for (int c = 0; c < Dh; c += 16) {
        uint32_t r1[16];
        tmem_ld16(t + hb + c, r1);
        tmem_ld_wait_regs(r1);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          float b1[4];
          load_bias4(a.bias, n0 + hb + c + i, b1);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float x = __uint_as_float(r1[i + j]) * a.w_scale + b1[j];
            ss += x * x;
          }
        }
      }
      rn = 1.f / sqrtf(ss / (float)Dh + a.qk_eps);
    }
    if (half % 16 == 0) {
#pragma unroll 1
      for (int c = 0; c < half; c += 16) rope_chunk<16>(a, t, hb, c, half, rn, live, cs, sn, dst, n0);
    } else {  // a rotary half of 8 (mod 16) columns, e.g. 24 of a 64-wide head
#pragma unroll 1
      for (int c = 0; c < half; c += 8) rope_chunk<8>(a, t, hb, c, half, rn, live, cs, sn, dst, n0);
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
        for (int j = 0; j < 4; ++j) o1[i + j] = (__uint_as_float(r1[i + j]) * a.w_scale + b1[j]) * rn;
      }
      if (a.f16)
        store_f16x16(reinterpret_cast<__half*>(dst + hb + c), o1);
      else
        store_bf16x16(reinterpret_cast<__nv_bfloat16*>(dst + hb + c), o1);
    }
  }
}

// x[row, n0 + c] += gate[tag[row]][n0 + c] * (acc + bias)     (gate == nullptr: plain add)
//
// The residual stream is fp32 in HBM, so this epilogue is a read-modify-write of a 128 x 256 fp32
// tile.  TMEM hands each thread one row, which would make every global access a 32-row scatter;
// instead each column group's part of the tile goes through shared memory RC = 64 / NG columns at
// a time (the staging area is 128 x 64 floats whichever NG):
//   phase A  each thread moves its row's RC accumulator columns TMEM -> registers -> shared memory
//            (16-byte chunks XOR-swizzled by row so a warp's stores spread over all banks)
//   phase B  each warp walks 32 rows; RC / 2 lanes share a row, two adjacent columns each, so the
//            loads and stores of x (and of the gate and bias) are RC * 4 contiguous bytes per row.
// The NG groups run on their own named barriers (ids 1 .. NG), so they overlap one another.
constexpr int RES_STAGE_FLOATS = BM * 64;
constexpr int RES_BATCH = 32;  // rows whose loads a warp has in flight at once (4 in the NVFP4 mode,
                               // whose 448-thread launch leaves fewer registers per thread)

__device__ __forceinline__ void epi_bar(int grp) { asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory"); }

// Where an epilogue warp hands an accumulator buffer back: a local mbarrier, or (CTA pairs) the
// pair's first CTA's barrier at a shared::cluster address.
struct TRelease {
  uint64_t* local;
  uint32_t cluster;  // non-zero: arrive at this shared::cluster address instead
  __device__ __forceinline__ void arrive() const {
    if (cluster)
      mbar_arrive_cluster(cluster);
    else
      mbar_arrive(local);
  }
};

template <int RB, int NG>
__device__ __forceinline__ void epi_resid(const GemmArgs& a, uint32_t t, int tile_row0, int quarter, int ew, int grp,
                                          int n0, float* stage_all, TRelease rel) {
  constexpr int RC = 64 / NG;          // columns per pass
  constexpr int GC = BN / NG;          // columns of this group
  constexpr int LPR = RC / 2;          // lanes per row in phase B
  constexpr int RPI = 32 / LPR;        // rows per warp-wide access
  static_assert(RB % RPI == 0 && 32 % RB == 0, "row batch");
  const int lane = threadIdx.x & 31;
  float* stage = stage_all + grp * (RES_STAGE_FLOATS / NG);
  const int r_own = quarter * 32 + lane;  // the tile row whose TMEM lane this thread reads
  const uint32_t st_row = smem_u32(stage) + r_own * (RC * 4);
  const int sub = lane / LPR, lc = lane % LPR;
  const int chunk = lc >> 1, half8 = (lc & 1) * 8;
#pragma unroll 1
  for (int c0 = grp * GC; c0 < (grp + 1) * GC; c0 += RC) {
    // phase A: TMEM -> shared memory (swizzled)
#pragma unroll
    for (int h = 0; h < RC; h += 32) {
      uint32_t r[32];
      tmem_ld32_sync(t + c0 + h, r);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int ch = (h >> 2) + q;  // 16-byte chunk index within the row
        st_shared_v4(st_row + ((ch ^ (r_own & 7)) << 4), r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
      }
    }
    if (c0 + RC == (grp + 1) * GC) {
      // every accumulator column of this group is out of TMEM: this warp's part of the buffer is
      // handed back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) rel.arrive();
    }
    epi_bar(grp);
    // phase B: coalesced read-modify-write of 32 rows x RC columns per warp
    const int col = n0 + c0 + 2 * lc;
    float2 bb = make_float2(0.f, 0.f);
    if (a.bias) bb = *reinterpret_cast<const float2*>(a.bias + col);
#pragma unroll 1
    for (int rr0 = 0; rr0 < 32; rr0 += RB) {
      constexpr int U = RB / RPI;
      float2 acc[U], xv[U], gv[U];
      int rows[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rt = ew * 32 + rr0 + u * RPI + sub;
        rows[u] = tile_row0 + rt;
        const uint32_t sa = smem_u32(stage) + rt * (RC * 4) + ((chunk ^ (rt & 7)) << 4) + half8;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(acc[u].x), "=f"(acc[u].y) : "r"(sa));
        if (rows[u] < a.M) {
          xv[u] = *reinterpret_cast<const float2*>(a.x + (size_t)rows[u] * a.N + col);
          gv[u] = a.gate ? *reinterpret_cast<const float2*>(a.gate + (size_t)a.tags[rows[u]] * a.gate_stride + col)
                         : make_float2(1.f, 1.f);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (rows[u] < a.M) {
          float2 o;
          o.x = xv[u].x + gv[u].x * (acc[u].x * a.w_scale + bb.x);
          o.y = xv[u].y + gv[u].y * (acc[u].y * a.w_scale + bb.y);
          *reinterpret_cast<float2*>(a.x + (size_t)rows[u] * a.N + col) = o;
        }
      }
    }
    epi_bar(grp);  // the staging buffer is reused by the next column block
  }
}

// Tile columns [0, 128) hold value features f0 .. f0+127 and [128, 256) their gates
// (the interleaved packing of the FFN up projection); h[row, f0 + j] = u_j * silu(g_j).
template <int NG>
__device__ __forceinline__ void epi_swiglu(const GemmArgs& a, uint32_t t, int row, int n0, int grp) {
  const bool live = row < a.M;
  const int F = a.N / 2;
  const int f0 = n0 / 2;
  __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(a.out) + (size_t)row * F + f0;
  __half* hrow16 = static_cast<__half*>(a.out) + (size_t)row * F + f0;  // out_kind 2
  bool over = false;  // an f16 value beyond the finite range
  constexpr int GF = BN / 2 / NG;  // value/gate pairs per group
#pragma unroll 1
  for (int c = grp * GF; c < (grp + 1) * GF; c += 16) {
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
        float u = __uint_as_float(ru[i + j]) * a.w_scale + bu[j];
        float g = __uint_as_float(rg[i + j]) * a.w_scale + bg[j];
        h[i + j] = u * silu_f(g);
      }
    }
    if (a.out_kind == 2) {
#pragma unroll
      for (int i = 0; i < 16; ++i) over |= fabsf(h[i]) > kF16Max;
      store_f16x16(hrow16 + c, h);
    } else {
      store_bf16x16(hrow + c, h);
    }
  }
  if (over && a.status) atomicOr(a.status, kDevRange);
}

// NVFP4 converter: expand row r of a stage's packed weight tile (256 rows x 64
// E2M1 codes, even k in the low nibble, and 4 E4M3 scales per row, one per 16 codes) into f16 in
// the layout a 128-byte-swizzled TMA load of a [256 x 64] f16 box writes: row r at r * 128 bytes,
// its 16-byte chunk c at position c ^ (r & 7).  code * scale is exact in f16.
__device__ __forceinline__ void nvfp4_expand_row(uint32_t raw, uint32_t dst, int r) {
  {
    uint32_t w[8], sc;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(raw + r * 32));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(raw + r * 32 + 16));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(raw + Q_CODE_BYTES + r * 4));
    uint32_t s01, s23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s01) : "h"(static_cast<uint16_t>(sc & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s23) : "h"(static_cast<uint16_t>(sc >> 16)));
    uint32_t sg[4];  // each group's scale in both halves
    asm("prmt.b32 %0, %1, %1, 0x1010;" : "=r"(sg[0]) : "r"(s01));
    asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(sg[1]) : "r"(s01));
    asm("prmt.b32 %0, %1, %1, 0x1010;" : "=r"(sg[2]) : "r"(s23));
    asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(sg[3]) : "r"(s23));
    const uint32_t row = dst + r * 128;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 2; ++q)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
            "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
            "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(h[4 * q]), "=r"(h[4 * q + 1]), "=r"(h[4 * q + 2]), "=r"(h[4 * q + 3])
            : "r"(w[2 * g + q]));
#pragma unroll
      for (int j = 0; j < 8; ++j) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[j]) : "r"(sg[g]));
      st_shared_v4(row + (((2 * g) ^ (r & 7)) << 4), h[0], h[1], h[2], h[3]);
      st_shared_v4(row + (((2 * g + 1) ^ (r & 7)) << 4), h[4], h[5], h[6], h[7]);
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(Q_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const GemmArgs args) {
  constexpr int NST = EPI == kEpiGatedResid ? Q_STAGES_RESID : Q_STAGES;
  constexpr int RING_BYTES = NST * STAGE_BYTES + Q_RAW_SLOTS * Q_RAW_BYTES;
  const uint32_t ID = IDESC_F16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + NST * A_BYTES;
  uint8_t* sQ = sB + NST * B_BYTES;  // the packed weight tiles (Q_RAW_SLOTS)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  uint64_t* empty = full + NST;
  uint64_t* rawfull = empty + NST;             // a packed tile has landed
  uint64_t* rawempty = rawfull + Q_RAW_SLOTS;  // the converters are done with a slot
  uint64_t* tfull = rawempty + Q_RAW_SLOTS;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;  // unwind: the MMAs issued before an abort have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* res_stage = reinterpret_cast<float*>(smem + RING_BYTES + 256);  // residual epilogue only

  if (args.status && (*reinterpret_cast<volatile int*>(args.status) & kDevLayout)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (args.M + BM - 1) / BM, n_n = args.N / BN, k_blocks = args.K / BK;
  const int tiles = n_m * n_n;
  const int gn = args.group_n > 0 ? args.group_n : n_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1 + Q_CONV_WARPS);  // the producer, and one arrival per converter warp
      mbar_init(&empty[s], 1);
    }
    for (int q = 0; q < Q_RAW_SLOTS; ++q) {
      mbar_init(&rawfull[q], 1);
      mbar_init(&rawempty[q], Q_CONV_WARPS);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], Q_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmA);
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, rslot = 0, issued = 0, raw_issued = 0;
      uint32_t phase = 0, rphase = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        TileCoord tc = tile_coord(tile, n_m, n_n, gn);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) goto producer_done;
          // the packed slot is free once the converters expanded its previous tile; the stage's B
          // tile is free because empty[stage] fired before this copy is issued
          if (!mbar_wait(&rawempty[rslot], rphase ^ 1, abort_flag, args.status)) goto producer_done;
          mbar_arrive_expect_tx(&rawfull[rslot], Q_RAW_BYTES);
          bulk_load(sQ + rslot * Q_RAW_BYTES, args.b_packed + ((size_t)tc.nb * k_blocks + kb) * Q_RAW_BYTES,
                    Q_RAW_BYTES, &rawfull[rslot]);
          ++raw_issued;
          if (++rslot == Q_RAW_SLOTS) {
            rslot = 0;
            rphase ^= 1;
          }
          mbar_arrive_expect_tx(&full[stage], A_BYTES);
          tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, tc.mb * BM);
          ++issued;
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: wait until the MMAs consumed every stage we filled, so no TMA write into this
      // CTA's shared memory is still in flight when the CTA exits.
      for (int s = 0; s < NST; ++s) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) goto producer_done;
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
      goto producer_exit;
    producer_done:
      // Unwind: the copies of the last fills of each stage (and packed slot) may still be in
      // flight; each is the latest phase of its barrier, so its landing completes that phase.
      // (full[] also waits for the converters, and may run out its bound when they aborted.)
      for (int j = issued - NST < 0 ? 0 : issued - NST; j < issued; ++j)
        mbar_wait_landed(&full[j % NST], (uint32_t)(j / NST) & 1u);
      for (int j = raw_issued - Q_RAW_SLOTS < 0 ? 0 : raw_issued - Q_RAW_SLOTS; j < raw_issued; ++j)
        mbar_wait_landed(&rawfull[j % Q_RAW_SLOTS], (uint32_t)(j / Q_RAW_SLOTS) & 1u);
    producer_exit:;
    }
  } else if (warp == 1) {
    // The MMA warp runs converged: every lane waits and computes the descriptors, elect.sync picks
    // the issuing lane (a branch taken by one lane issues markedly slower).
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA)), b_desc0 = sdesc_sw128(smem_u32(sB));
    bool unwound = false;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, args.status))) {
        unwound = true;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      bool ok = true;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, args.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // a descriptor's start field is the address / 16: offsets are added to it
        const uint64_t ad = a_desc0 + (uint64_t)((stage * A_BYTES) >> 4);
        const uint64_t bd = b_desc0 + (uint64_t)((stage * B_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) umma_bf16_elect(d_tmem, ad + 2 * k, bd + 2 * k, ID, (kb | k) != 0);
        umma_commit_elect(&empty[stage]);
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        unwound = true;
        break;
      }
      umma_commit_elect(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (unwound) {
      // the MMAs already issued still write TMEM and read shared memory: let them finish before
      // the CTA frees either
      umma_commit_elect(mma_done);
      mbar_wait_landed(mma_done, 0);
    }
  } else if (warp >= 6) {
    // converters: one pass over the same (tile, k-block) sequence as the producer
    // The stage's B tile is free: the packed tile of this fill was copied only after the MMA's
    // commit for the previous fill of the stage (the producer waits on empty[stage] first).
    const int ct = threadIdx.x - Q_BASE_THREADS;
    int stage = 0, rslot = 0;
    uint32_t phase = 0, rphase = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(&rawfull[rslot], rphase, abort_flag, args.status)) goto convert_done;
        nvfp4_expand_row(smem_u32(sQ + rslot * Q_RAW_BYTES), smem_u32(sB + stage * B_BYTES), ct);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rawempty[rslot]);
          mbar_arrive(&full[stage]);
        }
        if (++rslot == Q_RAW_SLOTS) {
          rslot = 0;
          rphase ^= 1;
        }
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  convert_done:;
  } else {
    const int quarter = warp & 3;  // TMEM lanes [32 * quarter, +32) belong to this warp
    constexpr int NG = Q_EPI_WARPS / 4;
    const int grp = (warp - 2) >> 2, ew = (warp - 2) & 3;
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
        epi_resid<4, NG>(args, t, tc.mb * BM, quarter, ew, grp, n0, res_stage, TRelease{&tempty[acc], 0u});
      } else {
        if (EPI == kEpiStore) epi_store<NG>(args, t, row, n0, grp);
        if (EPI == kEpiQkvRope) epi_qkv<NG>(args, t, row, n0, grp);
        if (EPI == kEpiSwiglu) epi_swiglu<NG>(args, t, row, n0, grp);
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


// ---------------------------------------------------------------------------------------------
// CTA pairs (clusters of 2) on tcgen05 cta_group::2: one MMA instruction covers a 256 x 256 x 16
// block, each CTA holding 128 rows of A and 128 rows (one half) of B, and each CTA's TMEM the
// accumulator of its own 128 rows.  A CTA's stage is then 32 KB instead of 48 for the same MMA work
// per SM, so six stages fit where four did, and the loads run 1.5x further ahead of the MMAs: a
// per-stage clock trace of the single-CTA kernel showed about 40 % of its K-blocks waiting beyond
// the 512 cycles of MMA work for their stage.  Each CTA also fetches half the B bytes per tile.
//   warp 0     TMA producer (both CTAs): this CTA's A tile and B half into its own stage; the bytes
//              of both CTAs complete on the first CTA's barrier (a forward of "stage landed" from
//              the second CTA by a remote mbarrier arrive, in series with every K-block, measured
//              2.5x slower)
//   warp 1     TMEM allocator (both CTAs).  First CTA: MMA issuer, waits for the pair's stage,
//              issues the pair MMAs, commits to both CTAs' barriers
//   warps 2-9  epilogue (both CTAs), each on its own TMEM; the buffers are released to the first
//              CTA's MMA warp (16 arrivals: 8 warps in each CTA)
constexpr int P_STAGES = 6;
constexpr int PB_BYTES = (BN / 2) * BK * 2;   // one CTA's half of the B tile
constexpr int P_STAGE_BYTES = A_BYTES + PB_BYTES;
constexpr int P_SMEM_BYTES = P_STAGES * P_STAGE_BYTES + 1024 + 256;
constexpr int P_SMEM_BYTES_RESID = P_SMEM_BYTES + BM * 64 * 4;
static_assert(P_SMEM_BYTES_RESID <= 227 * 1024, "pair stages exceed shared memory");

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args) {
  constexpr int NST = P_STAGES;
  const uint32_t ID = args.f16 ? idesc_f16_f32(2 * BM, BN) : idesc_bf16_f32(2 * BM, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + NST * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * P_STAGE_BYTES);  // [NST] first CTA: both stages landed
  uint64_t* empty = full + NST;       // [NST] the pair MMAs are done with the stage (both CTAs)
  uint64_t* tfull = empty + NST;      // [2] accumulator ready (both CTAs)
  uint64_t* tempty = tfull + 2;       // [2] first CTA: both CTAs' epilogues are done with it
  uint64_t* mma_done = tempty + 2;    // first CTA, unwind: the pair MMAs issued before an abort are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* res_stage = reinterpret_cast<float*>(smem + NST * P_STAGE_BYTES + 256);  // residual epilogue only

  if (args.status && (*reinterpret_cast<volatile int*>(args.status) & kDevLayout)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int n_m = (args.M + BM - 1) / BM, n_n = args.N / BN, k_blocks = args.K / BK;
  const int n_mp = (n_m + 1) / 2;  // row-block pairs; rank r takes row block 2 p + r
  const int tiles = n_mp * n_n;
  const int gn = args.group_n > 0 ? args.group_n : n_n;
  const int t0 = (int)(blockIdx.x >> 1), tstep = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 2 * EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t b_policy = l2_policy_evict_last();
      const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int tile = t0; tile < tiles; tile += tstep) {
        const TileCoord tc = tile_coord(tile, n_mp, n_n, gn);
        const int mb = 2 * tc.mb + (int)rank;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) goto producer_done;
          // both CTAs' bytes complete on the first CTA's barrier, which expects them all; its
          // pending arrival keeps the phase open however the two CTAs' copies interleave
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
          const uint32_t bar = leader_full + (uint32_t)stage * 8u;
          tma_load_2d_pair(sA + stage * A_BYTES, &tmA, bar, kb * BK, mb * BM);
          tma_load_2d_pair_hint(sB + stage * PB_BYTES, &tmB, bar, kb * BK, tc.nb * BN + (int)rank * (BN / 2),
                                b_policy);
          ++issued;
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every stage this CTA filled has been consumed, so no copy is in flight at exit.
      for (int s = 0; s < NST; ++s) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) goto producer_done;
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
      goto producer_exit;
    producer_done:
      // Unwind: the last fill of each stage may still be in flight.  Its bytes complete on the
      // first CTA's barrier, where the first CTA can wait for them; the second CTA cannot, and
      // waits out the same bound instead.
      if (rank == 0) {
        for (int j = issued - NST < 0 ? 0 : issued - NST; j < issued; ++j)
          mbar_wait_landed(&full[j % NST], (uint32_t)(j / NST) & 1u);
      } else if (issued > 0) {
        landed_grace();
      }
    producer_exit:;
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // the first CTA: the pair's MMA warp, converged, elect.sync picks the issuing lane
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA)), b_desc0 = sdesc_sw128(smem_u32(sB));
      bool unwound = false;
      for (int tile = t0; tile < tiles; tile += tstep) {
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, args.status))) {
          unwound = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, args.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + (uint64_t)((stage * A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)((stage * PB_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) umma_pair_elect(d_tmem, ad + 2 * k, bd + 2 * k, ID, (kb | k) != 0);
          umma_commit_pair_elect(&empty[stage]);  // the stage is free in both CTAs
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) {
          unwound = true;
          break;
        }
        umma_commit_pair_elect(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (unwound) {
        // the pair MMAs already issued still write both CTAs' TMEM: let them finish before either
        // CTA frees it (the final cluster barrier holds the second CTA until this returns)
        umma_commit_pair_elect(mma_done, 1);
        mbar_wait_landed(mma_done, 0);
      }
    }
  } else {
    const int quarter = warp & 3;  // TMEM lanes [32 * quarter, +32) belong to this warp
    constexpr int NG = EPI_WARPS / 4;
    const int grp = (warp - 2) >> 2, ew = (warp - 2) & 3;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = t0; tile < tiles; tile += tstep) {
      const TileCoord tc = tile_coord(tile, n_mp, n_n, gn);
      const int mb = 2 * tc.mb + (int)rank;
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, args.status)) break;
      tc_fence_after();
      const int row = mb * BM + quarter * 32 + lane;
      const uint32_t t = tmem + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int n0 = tc.nb * BN;
      const TRelease rel{&tempty[acc], leader_tempty + (uint32_t)acc * 8u};
      if (EPI == kEpiGatedResid) {
        epi_resid<RES_BATCH, NG>(args, t, mb * BM, quarter, ew, grp, n0, res_stage, rel);
      } else {
        if (EPI == kEpiStore) epi_store<NG>(args, t, row, n0, grp);
        if (EPI == kEpiQkvRope) epi_qkv<NG>(args, t, row, n0, grp);
        if (EPI == kEpiSwiglu) epi_swiglu<NG>(args, t, row, n0, grp);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) rel.arrive();
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA frees TMEM or leaves while the pair's MMAs or arrivals may still reach it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// The bf16 / f16 modes run on CTA pairs, the NVFP4 mode on single CTAs.
template <int EPI, bool BQ>
cudaError_t launch_t(const void* A, const void* B, const GemmArgs& args, cudaStream_t stream) {
  CUtensorMap ta, tb;
  // The NVFP4 mode's A is f16: the map only moves 2-byte elements, so the bf16 map serves it.
  if (!make_tmap_bf16_2d(&ta, A, args.K, args.M, (uint64_t)args.K * 2, BK, BM)) return cudaErrorInvalidValue;
  const int n_m = (args.M + BM - 1) / BM, n_n = args.N / BN;
  if constexpr (BQ) {
    constexpr int smem = EPI == kEpiGatedResid ? Q_SMEM_BYTES_RESID : Q_SMEM_BYTES;
    static unsigned long long smem_set = 0;
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(gemm_kernel<EPI>), smem, &smem_set);
    if (e != cudaSuccess) return e;
    const int tiles = n_m * n_n;
    const int grid = tiles < num_sms() ? tiles : num_sms();
    gemm_kernel<EPI><<<grid, Q_THREADS, smem, stream>>>(ta, args);
    return cudaGetLastError();
  } else {
    constexpr int smem = EPI == kEpiGatedResid ? P_SMEM_BYTES_RESID : P_SMEM_BYTES;
    static unsigned long long smem_set = 0;
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(gemm_pair_kernel<EPI>), smem, &smem_set);
    if (e != cudaSuccess) return e;
    // each CTA of a pair loads one half (128 rows) of the B tile
    if (!make_tmap_bf16_2d(&tb, B, args.K, args.N, (uint64_t)args.K * 2, BK, BN / 2)) return cudaErrorInvalidValue;
    const int pair_tiles = ((n_m + 1) / 2) * n_n;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // The persistent grid holds only the pairs that can be resident at once (a second wave would
    // double the launch): all 76 on a 152-SM part, fewer if another kernel holds SMs.
    static int resident = 0;
    if (resident == 0) {
      cfg.gridDim = dim3(num_sms());
      e = cudaOccupancyMaxActiveClusters(&resident, gemm_pair_kernel<EPI>, &cfg);
      if (e != cudaSuccess) return e;
      if (resident < 1) return cudaErrorLaunchOutOfResources;
    }
    const int pairs = pair_tiles < resident ? pair_tiles : resident;
    cfg.gridDim = dim3(2 * pairs);
    e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<EPI>, ta, tb, args);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
}

// ffn_F > 0: the weight is an FFN up projection [2F, K] whose rows are interleaved in 128-feature
// groups as they are packed (packed row p of group p / 256 takes value row 128 (p / 256) + p % 256 for
// p % 256 < 128, else gate row F + 128 (p / 256) + p % 256 - 128), the layout the SiLU-gate epilogue
// reads.
__global__ void nvfp4_pack_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sc, int N, int K,
                                  int ffn_F, uint8_t* __restrict__ packed) {
  const int kbs = K / BK;
  const size_t total = (size_t)(N / BN) * kbs * Q_RAW_BYTES;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / Q_RAW_BYTES;
    const int o = (int)(i - t * Q_RAW_BYTES);
    const int nb = (int)(t / kbs), kb = (int)(t - (size_t)nb * kbs);
    uint8_t v;
    auto src_row = [&](int p) {
      if (!ffn_F) return p;
      const int g = p >> 8, w = p & 255;
      return w < 128 ? 128 * g + w : ffn_F + 128 * g + (w - 128);
    };
    if (o < Q_CODE_BYTES) {
      const int r = o / (BK / 2), j = o - r * (BK / 2);
      v = q[(size_t)src_row(nb * BN + r) * (K / 2) + kb * (BK / 2) + j];
    } else {
      const int o2 = o - Q_CODE_BYTES;
      const int r = o2 / (BK / 16), j = o2 - r * (BK / 16);
      v = sc[(size_t)src_row(nb * BN + r) * (K / 16) + kb * (BK / 16) + j];
    }
    packed[i] = v;
  }
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
    case kEpiStore: return launch_t<kEpiStore, false>(A, B, args, stream);
    case kEpiQkvRope: return launch_t<kEpiQkvRope, false>(A, B, args, stream);
    case kEpiGatedResid: return launch_t<kEpiGatedResid, false>(A, B, args, stream);
    case kEpiSwiglu: return launch_t<kEpiSwiglu, false>(A, B, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_nvfp4_launch(int epilogue, const void* A, const GemmArgs& args_in, cudaStream_t stream) {
  GemmArgs args = args_in;
  if (args.M <= 0) return cudaSuccess;
  if (!args.b_packed || (reinterpret_cast<uintptr_t>(args.b_packed) & 15) || args.N % BN || args.K % BK)
    return cudaErrorInvalidValue;
  if (args.group_n <= 0) {
    long long per_nb = (long long)BN * args.K * 9 / 16;  // codes + scales of one N-block
    int g = (int)((48ll << 20) / (per_nb > 0 ? per_nb : 1));
    args.group_n = g < 1 ? 1 : g;
  }
  switch (epilogue) {
    case kEpiStore: return launch_t<kEpiStore, true>(A, nullptr, args, stream);
    case kEpiQkvRope: return launch_t<kEpiQkvRope, true>(A, nullptr, args, stream);
    case kEpiGatedResid: return launch_t<kEpiGatedResid, true>(A, nullptr, args, stream);
    case kEpiSwiglu: return launch_t<kEpiSwiglu, true>(A, nullptr, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t nvfp4_pack_launch(const uint8_t* q, const uint8_t* s, int N, int K, uint8_t* packed, cudaStream_t st,
                              int ffn_F) {
  if (N % BN || K % BK || N <= 0 || K <= 0 || (ffn_F && (N != 2 * ffn_F || ffn_F % 128))) return cudaErrorInvalidValue;
  const size_t total = (size_t)(N / BN) * (K / BK) * Q_RAW_BYTES;
  size_t g = (total + 255) / 256;
  const size_t cap = (size_t)num_sms() * 16;
  nvfp4_pack_kernel<<<(unsigned)(g < cap ? g : cap), 256, 0, st>>>(q, s, N, K, ffn_F, packed);
  return cudaGetLastError();
}

}  // namespace dit
