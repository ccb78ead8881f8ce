// Varlen, bidirectional (non-causal) flash attention over a packed sequence on the tcgen05 tensor
// cores.  [H3] "Correctness gates": attention reuses DFlashBlockAttention(causal=false) for packed
// varlen; [M3] "What moved": non-causal attention with no bias.  For document [a, b) and head h:
//     o_i = sum_j softmax_j(q_i . k_j / sqrt(Dh)) v_j,   i, j in [a, b)
// The block-diagonal structure comes from cu_seqlens alone: no mask tensor exists.
//
// One CTA = one (document, 128-row q-tile, head).  Key/value tiles are 128 tokens wide and start
// at multiples of 128 in the packed sequence (so the TMA x coordinate of the transposed V is
// 16-byte aligned); columns outside the document are masked to -inf in S and zeroed in V^T.
//   warp 0     TMA producer: Q once, then K and V^T tiles through a 3-stage and a 2-stage ring
//   warp 1     TMEM allocator + S issuer: S(j) = Q K(j)^T into S buffer j % S_BUFS, issued as soon
//              as K(j) has landed and the softmax has read that buffer's previous scores
//   warps 10, 11  PV issuers, one per O half: O_h += P(j) V(j) once P(j) is in TMEM and V(j) has
//              landed (one barrier counts both); key columns [0, 64) accumulate into O_0 (warp 10),
//              [64, 128) into O_1 (warp 11).
//              On a document's boundary tiles the warp first zeroes the V^T columns outside the
//              document, so that a non-finite value in a neighbouring document cannot reach this
//              one through 0 * inf (their softmax weights are exactly 0 already)
//   warps 2-9  softmax, two warps per query row: warp half h owns key columns [64h, 64h + 64) of
//              every tile and keeps its own running max m_h, sum l_h and accumulator O_h, exactly as
//              two independent passes over disjoint key subsets would; the halves exchange nothing
//              per tile and are merged once at the end:
//                  o = (2^(m_0-m) O_0 + 2^(m_1-m) O_1) / (2^(m_0-m) l_0 + 2^(m_1-m) l_1),  m = max(m_0, m_1)
// Three issuing warps, each running converged and issuing through elect.sync: with S and PV on
// separate threads, S(j + 1) runs while the softmax works on tile j, and PV(j) while it works on
// j + 1.
// TMEM: S_BUFS S buffers of 128 columns (two at head_dim 64, one at 128), O_0 and O_1 (Dh columns
// each), and two P buffers of 64 columns: P(j) (16-bit pairs, the type of the PV operands) goes to
// buffer j % 2 and the PV MMA reads it as its TMEM operand.  A P buffer is rewritten only after the
// PV of two tiles back is complete.
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace dit {

namespace {

constexpr int TQ = 128, TK = 128;
constexpr int ATOM = 128 * 64 * 2;         // 128 rows x 64 16-bit columns, 128-byte swizzled (16 KB)
constexpr int KV_STAGES = 2;               // V^T ring
constexpr int K_STAGES = 3;                // K ring: K(j + 1) is wanted a tile before V(j + 1)
constexpr int ATT_THREADS = 384;           // producer, S issuer, 8 softmax warps, two PV issuers
constexpr int SOFTMAX_THREADS = 256;
constexpr int PV_WARP = 10;                // PV issuers: warp 10 for O_0, warp 11 for O_1
static_assert(KV_STAGES == 2, "V(j) lands on the barrier of P buffer j % 2");

// Shared-memory plan for head dim HD (64 or 128):
//   Q  [128 q, HD]   HD/64 atoms of 16 KB          K  [128 kv, HD]  HD/64 atoms of 16 KB
//   Vt [HD, 128 kv]  2 atoms (kv halves) of HD * 128 bytes each
template <int HD>
struct AttPlan {
  static constexpr int Q_BYTES = 128 * HD * 2;
  static constexpr int K_BYTES = 128 * HD * 2;
  static constexpr int V_ATOM = HD * 128;
  static constexpr int V_BYTES = 2 * V_ATOM;
  static constexpr int SMEM = Q_BYTES + K_STAGES * K_BYTES + KV_STAGES * V_BYTES + 1024 + 256;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, TK);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(128, HD);
  // S buffers in TMEM: two where they fit beside O_0, O_1 and the two P buffers (head_dim 64), else
  // one (S(j + 1) then waits for the softmax to have read S(j), and runs under its exponentials)
  static constexpr int S_BUFS = HD == 64 ? 2 : 1;
  static_assert(S_BUFS * TK + 2 * HD + 2 * 64 <= 512, "TMEM plan");
};

__device__ __forceinline__ bool wait_noabort(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 255u) == 255u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Zero the columns of a landed V^T tile (two 64-column atoms of HD rows, 128-byte swizzled) whose
// key index lies outside [lo, hi): one 16-byte chunk (8 keys of one row) per step, by the 32 lanes of
// one warp.  Chunks wholly inside the document are left alone.
template <int HD>
__device__ __forceinline__ void zero_v_outside(uint8_t* sv_tile, int lo, int hi, int lane, int atom) {
  const uint32_t base = smem_u32(sv_tile);
  for (int idx = lane; idx < HD * 8; idx += 32) {
    const int row = idx >> 3, chunk = atom * 8 + (idx & 7);  // chunk: keys [8 chunk, 8 chunk + 8)
    const int k0 = chunk * 8;
    if (k0 >= lo && k0 + 8 <= hi) continue;
    const uint32_t addr = base + (chunk >> 3) * (HD * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
    uint4 v = ld_shared_v4(addr);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = k0 + 2 * e;
      const uint32_t keep_lo = (k >= lo && k < hi) ? 0x0000FFFFu : 0u;
      const uint32_t keep_hi = (k + 1 >= lo && k + 1 < hi) ? 0xFFFF0000u : 0u;
      w[e] &= keep_lo | keep_hi;
    }
    st_shared_v4(addr, w[0], w[1], w[2], w[3]);
  }
}

// F16: the 16-bit operand type (q, k, V^T, P and o) is f16, else bf16.  A template parameter, so that
// the softmax's conversions are one instruction per pair with no select.
template <int HD, bool F16>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, uint16_t* __restrict__ O, const AttnArgs args) {
  if (args.status && (*reinterpret_cast<volatile int*>(args.status) & kDevLayout)) return;
  const int count = *args.count;
  const int head = blockIdx.x / args.max_items;
  const int item_idx = blockIdx.x - head * args.max_items;
  if (item_idx >= count || head >= args.n_heads) return;
  const int2 item = args.items[item_idx];
  const int doc = item.x, q0 = item.y;
  const int ds = args.cu[doc], de = args.cu[doc + 1];
  const int kv_base = (ds / TK) * TK;
  const int n_kv = (de - kv_base + TK - 1) / TK;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Plan = AttPlan<HD>;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + Plan::Q_BYTES;                    // [stage]
  uint8_t* sV = sK + K_STAGES * Plan::K_BYTES;         // [stage]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + KV_STAGES * Plan::V_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                         // [stage]  K tile landed
  uint64_t* k_empty = k_full + K_STAGES;               // [stage]  S MMA done with the K tile
  uint64_t* v_empty = k_empty + K_STAGES;              // [stage]  PV MMA done with the V^T tile
  uint64_t* s_full = v_empty + KV_STAGES;              // [S_BUFS] S(j) in TMEM buffer j % S_BUFS (two
                                                       //   buffers: and P(j - 2) V(j - 2) done)
  uint64_t* s_free = s_full + Plan::S_BUFS;            // [S_BUFS] the softmax has loaded S(j)
  uint64_t* p_full = s_free + Plan::S_BUFS;            // [2]  P(j) in TMEM buffer j % 2 and V(j) landed
  uint64_t* o_done = p_full + 2;                       // [2]  O += P(j) V(j) complete
  uint64_t* s_drain = o_done + 2;                      // every S MMA complete
  uint64_t* o_drain = s_drain + 1;                     // every PV MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < K_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(&v_empty[s], 2);                         // both PV issuers
    }
    for (int b = 0; b < Plan::S_BUFS; ++b) {
      mbar_init(&s_full[b], Plan::S_BUFS == 2 ? 3 : 1);  // two buffers: + both PV commits of tile j - 2
      mbar_init(&s_free[b], SOFTMAX_THREADS / 32);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&p_full[s], SOFTMAX_THREADS / 32 + 1);   // softmax warps + the V^T load
      mbar_init(&o_done[s], 2);                          // both PV issuers
    }
    mbar_init(s_drain, 1);
    mbar_init(o_drain, 2);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S_BUFS S buffers of 128 columns, O_0 and O_1 (HD each), then P buffers 0 and 1 of 64
  // columns each (16-bit pairs), which the P.V MMA reads as its TMEM operand.
  constexpr int SB = Plan::S_BUFS;
  const uint32_t t_s = tmem;
  const uint32_t t_o = tmem + SB * TK;
  const uint32_t t_p = t_o + 2 * HD;

  if (warp == 0) {
    if (lane == 0) {
      const int hx = head * HD;
      mbar_arrive_expect_tx(q_full, Plan::Q_BYTES);
#pragma unroll
      for (int a = 0; a < HD / 64; ++a) tma_load_2d(sQ + a * ATOM, &tmQ, q_full, hx + 64 * a, q0);
      // K(j) waits for S(j - K_STAGES), V(j) for P(j - KV_STAGES) V(j - KV_STAGES).  The two rings
      // are polled side by side, so that a K stage still in use never holds back a free V stage or
      // the other way round.
      auto load_k = [&](int j) {
        const int st = j % K_STAGES;
        mbar_arrive_expect_tx(&k_full[st], Plan::K_BYTES);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          tma_load_2d(sK + st * Plan::K_BYTES + a * ATOM, &tmK, &k_full[st], hx + 64 * a, kv_base + j * TK);
      };
      auto load_v = [&](int j) {
        const int st = j % KV_STAGES;
        const int kv0 = kv_base + j * TK;
        // V(j) completes on the barrier that also counts the softmax warps' P(j) (stage = j % 2)
        mbar_arrive_expect_tx(&p_full[st], Plan::V_BYTES);
        tma_load_2d(sV + st * Plan::V_BYTES, &tmV, &p_full[st], kv0, hx);
        tma_load_2d(sV + st * Plan::V_BYTES + Plan::V_ATOM, &tmV, &p_full[st], kv0 + 64, hx);
      };
      int nk = 0, nv = 0;
      uint64_t t_last = globaltimer_ns();
      for (uint32_t spin = 0; nk < n_kv || nv < n_kv; ++spin) {
        bool moved = false;
        if (nk < n_kv && mbar_test_wait(&k_empty[nk % K_STAGES], ((nk / K_STAGES) & 1) ^ 1)) {
          load_k(nk++);
          moved = true;
        }
        if (nv < n_kv && mbar_test_wait(&v_empty[nv % KV_STAGES], ((nv / KV_STAGES) & 1) ^ 1)) {
          load_v(nv++);
          moved = true;
        }
        if (moved) {
          spin = 0;
        } else if ((spin & 255u) == 255u) {
          if (*abort_flag) break;
          const uint64_t now = globaltimer_ns();
          if (spin == 255u) t_last = now;  // the first idle check after progress starts the clock
          if (now - t_last > kWaitLimitNs) {
            *abort_flag = 1;
            if (args.status) atomicOr(args.status, kDevTimeout);
            break;
          }
        }
      }
      // Every copy this CTA issued must land before the CTA may exit.
      wait_noabort(q_full, 0);
      for (int j = nk - K_STAGES < 0 ? 0 : nk - K_STAGES; j < nk; ++j)
        wait_noabort(&k_full[j % K_STAGES], (j / K_STAGES) & 1);
      for (int j = nv - KV_STAGES < 0 ? 0 : nv - KV_STAGES; j < nv; ++j)
        wait_noabort(&p_full[j % KV_STAGES], (j / KV_STAGES) & 1);
    }
  } else if (warp == 1) {
    // S(j) into buffer j % SB once K(j) has landed and the softmax has read S(j - SB) from it.  The
    // warp runs converged and elect.sync picks the issuing lane.
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, args.status));
    tc_fence_after();
    const uint64_t q_desc = sdesc_sw128(smem_u32(sQ));
    constexpr uint32_t id_s = F16 ? idesc_f16_f32(128, TK) : Plan::IDESC_S;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int st = j % K_STAGES, sb = j % SB;
      if (j >= SB) ok = __all_sync(0xffffffffu, mbar_wait(&s_free[sb], (j / SB - 1) & 1, abort_flag, args.status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&k_full[st], (j / K_STAGES) & 1, abort_flag, args.status));
      if (!ok) break;
      tc_fence_after();
      const uint64_t k_desc = sdesc_sw128(smem_u32(sK + st * Plan::K_BYTES));
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const uint64_t off = (uint64_t)(((ks >> 2) * ATOM + (ks & 3) * 32) >> 4);
        umma_bf16_elect(t_s + sb * TK, q_desc + off, k_desc + off, id_s, ks != 0);
      }
      umma_commit_elect(&s_full[sb]);
      umma_commit_elect(&k_empty[st]);
    }
    // No MMA may still read shared memory or write TMEM when the CTA tears down.
    umma_commit_elect(s_drain);
    wait_noabort(s_drain, 0);
  } else if (warp == PV_WARP || warp == PV_WARP + 1) {
    // Two PV issuers, one per O half (key columns [64 hv, 64 hv + 64) -> O_hv), issuing side by
    // side.
    const int hv = warp - PV_WARP;
    // With two S buffers, "S(j) ready" also counts both PV commits of tile j - 2 (so one wait tells
    // the softmax that P buffer j % 2 is free); tiles 0 and 1 get those arrivals now.
    if (SB == 2 && lane == 0) {
      mbar_arrive(&s_full[0]);
      mbar_arrive(&s_full[1]);
    }
    for (int j = 0; j < n_kv; ++j) {
      const int pb = j & 1, st = j % KV_STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(&p_full[pb], (j >> 1) & 1, abort_flag, args.status))) break;
      const int c0 = kv_base + j * TK;
      const int lo = ds > c0 ? ds - c0 : 0;
      const int hi = de - c0 < TK ? de - c0 : TK;
      if (lo > 0 || hi < TK) {
        // a boundary tile: every lane sees the landed V^T tile through the barrier (its phase cannot
        // move on before this tile's PV is committed), zeroes its share of the outside columns of
        // this issuer's V^T half and makes the stores visible to the tensor core's operand reads
        wait_noabort(&p_full[pb], (j >> 1) & 1);
        zero_v_outside<HD>(sV + st * Plan::V_BYTES, lo, hi, lane, hv);
        fence_proxy_async_smem();
      }
      __syncwarp();
      tc_fence_after();
      {
        // the whole warp computes the descriptors; elect.sync picks the issuing lane
        constexpr uint32_t id_o = F16 ? idesc_f16_f32(128, HD) : Plan::IDESC_O;
        const uint64_t v_desc = sdesc_sw128(smem_u32(sV + st * Plan::V_BYTES));
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int ks = hv * 4 + kq;  // keys [16 ks, 16 ks + 16): 8 TMEM columns of P, V^T atom hv
          const uint64_t v_off = (uint64_t)((hv * Plan::V_ATOM + kq * 32) >> 4);
          umma_bf16_ts_elect(t_o + hv * HD, t_p + pb * 64 + ks * 8, v_desc + v_off, id_o, (j | kq) != 0);
        }
        umma_commit_elect(&o_done[pb]);
        umma_commit_elect(&v_empty[st]);
        if (SB == 2) umma_commit_elect(&s_full[pb]);  // an arrival of "S(j + 2) ready"
      }
      __syncwarp();
    }
    umma_commit_elect(o_drain);
    wait_noabort(o_drain, 0);
  } else {
    // ---------------- softmax warps ----------------
    // Two warps per row: TMEM lane quarter = warp % 4 (the rows a warp may access), key-column half
    // = (warp - 2) / 4.  O_h accumulates in TMEM through the MMA; the running max m_h is only raised
    // (and O_h, l_h rescaled by exp2(m_old - m_new)) when the half-row max grows by more than 2^8,
    // so most tiles never touch O_h.  Between raises p = exp2(s * scale - m_h) stays below 2^8.
    constexpr int HC = TK / 2;                   // key columns per half
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;           // tile row owned by this thread
    const int row = q0 + r;                      // packed-sequence row
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_oh = t_o + half * HD + lane_off;
    const float sc = args.scale_log2;
    constexpr bool f16 = F16;                    // P and o as f16 (else bf16)
    constexpr float kRescaleThreshold = 8.0f;    // log2 units
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    bool s_seen = false;  // "S(j) ready" already observed by the probe at the end of tile j - 1

    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;  // P buffer
      if (!s_seen && !mbar_wait(&s_full[j % SB], (j / SB) & 1, abort_flag, args.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int c0 = kv_base + j * TK + half * HC;
      const int lo = ds > c0 ? ds - c0 : 0;
      const int hi = de - c0 < HC ? de - c0 : HC;
      const bool interior = (lo == 0) && (hi == HC);
      const uint32_t ts = t_s + (j % SB) * TK + half * HC + lane_off;
      uint32_t sv[HC];
#pragma unroll
      for (int c = 0; c < HC; c += 32) tmem_ld32(ts + c, *reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
#pragma unroll
      for (int c = 0; c < HC; c += 32) tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
      // the scores are in registers: the S issuer may overwrite this buffer with S(j + SB)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[j % SB]);
      // one buffer: probe now whether P(j - 2) V(j - 2) is complete (it nearly always is), so that
      // the probe's latency hides under the exponentials
      const bool p_buf_free = SB == 2 || j < 2 || mbar_test_wait(&o_done[sb], ((j - 2) >> 1) & 1);
      if (!interior) {
#pragma unroll
        for (int i = 0; i < HC; ++i)
          if (i < lo || i >= hi) sv[i] = __float_as_uint(-INFINITY);
      }
      // half-row max: four independent chains of three-input max
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int i = 0; i < HC; i += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sv[i + 4]), __uint_as_float(sv[i + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sv[i + 6]), __uint_as_float(sv[i + 7]));
      }
      const float m_cand = fmaxf(fmax3(mx0, mx1, mx2), mx3) * sc;
      // true on the first tile with a key of the document in this half (m = -inf until then)
      const bool raise = m_cand > m + kRescaleThreshold;
      if (__any_sync(0xffffffffu, raise)) {
        const float m_new = raise ? m_cand : m;
        const float alpha = raise ? fast_exp2(m - m_new) : 1.f;  // exp2(-inf) = 0 before the first key
        if (j > 0) {
          // O_h holds this half's sum over tiles < j relative to m: wait for the last PV, rescale
          if (!mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1  // a rare path: kept out of line so the tile loop stays small
          for (int c = 0; c < HD; c += 32) {
            uint32_t ov[32];
            tmem_ld32_sync(t_oh + c, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(t_oh + c, ov);
            tmem_st_wait();
          }
        }
        l *= alpha;
        m = m_new;
      }
      // A half that has seen no key of the document yet has m = -inf and only masked scores:
      // p = exp2(-inf - 0) = 0 keeps O_h and l_h at zero.
      const float mu = m == -INFINITY ? 0.f : m;
      // p = exp2(s * scale - m) -> 16-bit pairs, this half's 32 columns of TMEM P buffer j % 2
      uint32_t pk[HC / 2];
      // paired fp32 arithmetic (one f32x2 FMA / add per two scores); four partial row sums
      const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-mu, -mu);
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < HC; c += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 x = ffma2(make_float2(__uint_as_float(sv[c + 2 * u]), __uint_as_float(sv[c + 2 * u + 1])), sc2, nm2);
          const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          rs[u] = fadd2(rs[u], e);
          pk[c / 2 + u] = pack16(f16, e.x, e.y);
        }
      }
      l += (rs[0].x + rs[0].y + rs[1].x + rs[1].y) + (rs[2].x + rs[2].y + rs[3].x + rs[3].y);
      // P buffer j % 2 is free once O += P(j - 2) V(j - 2) is complete (with two S buffers "S(j)
      // ready" said so already; with one, the S barrier cannot count it: a PV commit of the next
      // tile could then complete it before S(j) lands)
      if (!p_buf_free && !mbar_wait(&o_done[sb], ((j - 2) >> 1) & 1, abort_flag, args.status)) {
        ok = false;
        break;
      }
      // this half's 64 keys are columns [32 half, 32 half + 32) of TMEM P buffer j % 2
      tmem_st32(t_p + sb * 64 + lane_off + 32 * half, pk);
      // probe "S(j + 1) ready" now, so that the probe's latency overlaps the P store
      s_seen = j + 1 < n_kv && mbar_test_wait(&s_full[(j + 1) % SB], ((j + 1) / SB) & 1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok && n_kv > 0) {
      const int jl = n_kv - 1;
      ok = mbar_wait(&o_done[jl & 1], (jl >> 1) & 1, abort_flag, args.status);
      tc_fence_after();
    }
    // Merge the halves.  Once the last PV is done no MMA reads shared memory and every K tile has
    // landed, so K stage 0 holds the exchange of (m_h, l_h).  Every softmax warp reaches the barrier
    // (all waits above are bounded).
    float* xch = reinterpret_cast<float*>(sK);   // [2 halves][m | l][128 rows]
    xch[half * 256 + r] = m;
    xch[half * 256 + 128 + r] = l;
    asm volatile("bar.sync 1, %0;" ::"n"(SOFTMAX_THREADS) : "memory");
    if (ok) {
      const float m0 = xch[r], l0 = xch[128 + r], m1 = xch[256 + r], l1 = xch[384 + r];
      const float mm = fmaxf(m0, m1);
      const float a0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mm);
      const float a1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mm);
      const float inv = 1.f / (a0 * l0 + a1 * l1);
      const float w0 = a0 * inv, w1 = a1 * inv;
      // this warp writes output columns [half * HD / 2, half * HD / 2 + HD / 2)
      uint16_t* orow = O + (size_t)row * (args.n_heads * HD) + head * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t o0[32], o1[32];
        tmem_ld32(t_o + lane_off + half * (HD / 2) + c, o0);
        tmem_ld32(t_o + HD + lane_off + half * (HD / 2) + c, o1);
        tmem_ld_wait_regs(o0);
        tmem_ld_wait_regs(o1);
        if (row < de) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __uint_as_float(o0[i + u]) * w0 + __uint_as_float(o1[i + u]) * w1;
            st_global_v4(orow + c + i, pack16(f16, v[0], v[1]), pack16(f16, v[2], v[3]), pack16(f16, v[4], v[5]),
                         pack16(f16, v[6], v[7]));
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

constexpr int ITEM_ROWS = TQ;  // query rows per scheduled work item

// Validate the packed layout and emit the (document, q-tile) list, longest documents first.
// Codes follow the layout contract: 1 no documents, 2 cu[0] != 0, 3 not strictly increasing,
// 4 cu[D] != N, 5 a doc id disagrees with cu_seqlens, 6 a tag >= n_mod, 7 list overflow.
__global__ void schedule_kernel(const int32_t* cu, int n_docs, int n_tokens, const int32_t* doc_ids,
                                const uint8_t* tags, int n_mod, int2* items, int* count, int max_items,
                                int* layout_code, int* status) {
  __shared__ int code;
  if (threadIdx.x == 0) {
    code = 0;
    if (n_docs < 1) code = 1;
    else if (cu[0] != 0) code = 2;
    else {
      for (int j = 0; j < n_docs && !code; ++j)
        if (cu[j + 1] <= cu[j]) code = 3;
      if (!code && cu[n_docs] != n_tokens) code = 4;
    }
  }
  __syncthreads();
  if (code == 0 && doc_ids) {
    for (int i = threadIdx.x; i < n_tokens; i += blockDim.x) {
      const int j = doc_ids[i];
      if (j < 0 || j >= n_docs || i < cu[j] || i >= cu[j + 1]) atomicCAS(&code, 0, 5);
    }
  }
  __syncthreads();
  if (code == 0 && tags) {
    for (int i = threadIdx.x; i < n_tokens; i += blockDim.x)
      if ((int)tags[i] >= n_mod) atomicCAS(&code, 0, 6);
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  int n = 0;
  if (code == 0) {
    // selection by length, longest first (n_docs is small; ties keep packing order)
    int prev_len = 0x7fffffff, prev_idx = -1;
    for (int k = 0; k < n_docs && !code; ++k) {
      int best = -1, best_len = -1;
      for (int j = 0; j < n_docs; ++j) {
        const int len = cu[j + 1] - cu[j];
        const bool after_prev = len < prev_len || (len == prev_len && j > prev_idx);
        if (after_prev && len > best_len) {
          best = j;
          best_len = len;
        }
      }
      prev_len = best_len;
      prev_idx = best;
      for (int q = cu[best]; q < cu[best + 1]; q += ITEM_ROWS) {
        if (n >= max_items) {
          code = 7;
          break;
        }
        items[n++] = make_int2(best, q);
      }
    }
  }
  if (code) {
    n = 0;
    atomicOr(status, code == 7 ? kDevCapacity : kDevLayout);
  }
  *count = n;
  if (layout_code) *layout_code = code;
}

int attention_max_items_impl(int n_docs, int n_tokens) { return (n_tokens + ITEM_ROWS - 1) / ITEM_ROWS + n_docs; }

template <int HD, bool F16>
cudaError_t attention_launch_t(const void* q, const void* k, const void* vt, void* o, const AttnArgs& args,
                               cudaStream_t stream);

}  // namespace

int attention_max_items(int n_docs, int n_tokens) { return attention_max_items_impl(n_docs, n_tokens); }

int attention_item_rows() { return ITEM_ROWS; }

cudaError_t attention_schedule_launch(const int32_t* cu, int n_docs, int n_tokens, const int32_t* doc_ids,
                                      const uint8_t* tags, int n_mod, int2* items, int* count, int max_items,
                                      int* layout_code, int* status, cudaStream_t stream) {
  schedule_kernel<<<1, 256, 0, stream>>>(cu, n_docs, n_tokens, doc_ids, tags, n_mod, items, count, max_items,
                                         layout_code, status);
  return cudaGetLastError();
}

namespace {

template <int HD, bool F16>
cudaError_t attention_launch_t(const void* q, const void* k, const void* vt, void* o, const AttnArgs& args,
                               cudaStream_t stream) {
  static unsigned long long smem_set = 0;
  cudaError_t e =
      opt_in_smem(reinterpret_cast<const void*>(attention_kernel<HD, F16>), AttPlan<HD>::SMEM, &smem_set);
  if (e != cudaSuccess) return e;
  const int d = args.n_heads * HD;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_2d(&tq, q, d, args.n_tokens, (uint64_t)d * 2, 64, TQ)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tk, k, d, args.n_tokens, (uint64_t)d * 2, 64, TK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tv, vt, args.n_pad, d, (uint64_t)args.n_pad * 2, 64, HD)) return cudaErrorInvalidValue;
  const int grid = args.max_items * args.n_heads;
  if (grid <= 0) return cudaSuccess;
  attention_kernel<HD, F16><<<grid, ATT_THREADS, AttPlan<HD>::SMEM, stream>>>(tq, tk, tv, static_cast<uint16_t*>(o),
                                                                               args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attention_launch(const void* q, const void* k, const void* vt, void* o, const AttnArgs& args,
                             cudaStream_t stream) {
  if (args.head_dim == 128)
    return args.f16 ? attention_launch_t<128, true>(q, k, vt, o, args, stream)
                    : attention_launch_t<128, false>(q, k, vt, o, args, stream);
  if (args.head_dim == 64)
    return args.f16 ? attention_launch_t<64, true>(q, k, vt, o, args, stream)
                    : attention_launch_t<64, false>(q, k, vt, o, args, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dit
