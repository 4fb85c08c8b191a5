// fwd_fp8.cu -- exact attention forward with e4m3 (fp8) Q, K and V for sm_103a:
// the same online-softmax algorithm as fwd.cu with both products on the fp8
// tensor core (tcgen05.mma kind::f8f6f4, twice the bf16 rate).
//
// What it computes: O = softmax(scale * (sq Q8)(sk K8)^T) (sv V8) and the
// natural-log LSE per row, where Q8, K8, V8 hold e4m3 codes and sq, sk, sv are
// per-tensor dequantisation factors ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness": the abstract's exact
// attention tiled between HBM and on-chip memory; its related-papers entry for
// FlashAttention-3: FP8 attention on H100 near 1.2 PFLOP/s).
//
// Differences from fwd.cu, all forced by or chosen for 8-bit operands:
//   - every operand is K-major (128-byte rows = 128 e4m3 values): Q and K as
//     stored, V as V^T (head-dim rows, keys contiguous), written to a
//     workspace by a transpose kernel first;
//   - P goes back to tensor memory as e4m3 (four per 32-bit column) over the
//     first 32 columns of S_t, and PV takes it from there (the TS form): of
//     the two products only S reads both operands from shared memory, and
//     nothing writes P to shared memory.  As in fwd.cu, S_t of the next key
//     tile is issued right behind the PV_t that reads those columns;
//   - P is taken against the running max minus 7 and the max moves as soon as
//     it grows by more than 1 (log2 units), so P <= 2^8 fits e4m3 (largest
//     finite 448) and weights down to 2^-16 of the row max stay representable;
//   - O is normalised by the fp32 row sum of the unrounded weights.  Rounding
//     a weight to e4m3 errs by at most 2^-4 of it when it is normal (>= 2^-6)
//     and by 2^-10 below; a weight under 2^-13 of the row max is below 2^-6
//     (P of the row max >= 2^6), so |O - O_exact| <= max |v| (2^-4 +
//     2^-17 n_small / sum_j w_j), w_j = weights relative to the row max and
//     n_small the visible keys with w_j < 2^-13.
//
// Warp roles and tensor memory as in fwd.cu: warp 0 TMA producer, warp 1 MMA
// issuer, warps 4-7 / 8-11 softmax of query tiles 0 / 1; TMEM S_0, S_1, O_0,
// O_1 (512 columns).
#include "internal.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

namespace {

constexpr float FP8_THRESHOLD = 1.0f;  // move the reference max when a row's max exceeds it by more
constexpr float FP8_P_OFFSET = 7.0f;   // P = 2^(x - m + 7) <= 2^(1 + 7)

struct Fp8Cfg {
  static constexpr int D = 128;
  static constexpr int NS = 6;                                // K / V^T ring depth
  static constexpr uint32_t TILE_BYTES = 128 * 128;           // 128 rows x 128 bytes
  static constexpr uint32_t OFF_K = 2 * TILE_BYTES;           // after Q_0, Q_1
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;  // V^T tiles: 128 head-dim rows x 128 keys
  static constexpr uint32_t SMEM_BYTES = OFF_V + NS * TILE_BYTES + 1024;
  static constexpr uint32_t TMEM_O = 256;
  static constexpr int THREADS = 384;
  static constexpr uint32_t REGS_CTRL = 56, REGS_SOFTMAX = 224;
};

__global__ void __launch_bounds__(Fp8Cfg::THREADS, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tvt, const FwdParams p, float v_descale) {
  using C = Fp8Cfg;
  constexpr int NS = C::NS;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[1 + 4 * NS + 7];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar_q = smem_u32(&bars[0]);
  auto bar_k = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto bar_v = [&](int s) { return smem_u32(&bars[1 + NS + s]); };
  auto bar_kfree = [&](int s) { return smem_u32(&bars[1 + 2 * NS + s]); };  // K slot read by both S MMAs
  auto bar_vfree = [&](int s) { return smem_u32(&bars[1 + 3 * NS + s]); };  // V^T slot read by both PV MMAs
  auto bar_s = [&](int t) { return smem_u32(&bars[1 + 4 * NS + t]); };       // S_t in TMEM
  auto bar_p = [&](int t) { return smem_u32(&bars[1 + 4 * NS + 2 + t]); };   // P_t in TMEM
  auto bar_o = [&](int t) { return smem_u32(&bars[1 + 4 * NS + 4 + t]); };   // PV_t done
  const uint32_t bar_done = smem_u32(&bars[1 + 4 * NS + 6]);

  const Unit u = fwd_unit(blockIdx.x, p.B, p.Hq, p.Hkv, p.Nq, p.Nk, p.nqc, p.head_group, p.mask_kind,
                          p.causal_in_blocks, p.block_mask, p.nkb, p.window, p.q_offset, p.kv_offset);
  WaitCtx wc{p.wait_limit_ns, p.status, &abort_flag};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_v(s), 1);
      mbar_init(bar_kfree(s), 1);
      mbar_init(bar_vfree(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), 128);
      mbar_init(bar_o(t), 1);
    }
    mbar_init(bar_done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tvt);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp < 4) {
   reg_dealloc<C::REGS_CTRL>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    // one 16 KB box per tile (128 rows x 128 bytes); Q tiles on lanes 0-1,
    // each ring slot's K and V^T on lanes 0 and 1
    if (lane == 0) mbar_arrive_expect_tx(bar_q, 2 * C::TILE_BYTES);
    __syncwarp();
    if (lane < 2) tma_load_3d(s_base + lane * C::TILE_BYTES, &tq, 0, u.row0 + lane * TILE, u.bh, bar_q);
    int n = 0;
    bool ok = true;
    for (int kt = u.kt_begin; kt < u.kt_end && ok; ++kt) {
      if (!unit_uses(u, kt)) continue;
      const int s = n % NS;
      const uint32_t fph = ((n / NS) - 1) & 1;
      if (n >= NS) ok = wait_bar(bar_kfree(s), fph, wc) && wait_bar(bar_vfree(s), fph, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_k(s), C::TILE_BYTES);
        mbar_arrive_expect_tx(bar_v(s), C::TILE_BYTES);
      }
      __syncwarp();
      if (lane == 0) tma_load_3d(s_base + C::OFF_K + s * C::TILE_BYTES, &tk, 0, kt * TILE, u.kvh, bar_k(s));
      if (lane == 1) tma_load_3d(s_base + C::OFF_V + s * C::TILE_BYTES, &tvt, kt * TILE, 0, u.kvh, bar_v(s));
      ++n;
    }
    if ((!ok || abort_flag) && lane == 0) {
      // drain: every issued copy must land before the CTA's shared memory is released
      wait_bar(bar_q, 0, wc, false);
      for (int j = n - NS < 0 ? 0 : n - NS; j < n; ++j) {
        wait_bar(bar_k(j % NS), (j / NS) & 1, wc, false);
        wait_bar(bar_v(j % NS), (j / NS) & 1, wc, false);
      }
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Order per key tile n: PV_0(n), S_0(n+1), PV_1(n), S_1(n+1).  S_t(n+1)
    // overwrites the columns P_t(n) occupies; it is issued right after the
    // PV_t(n) that reads them (tcgen05.mma from one thread execute in issue
    // order), so each softmax has the other tile's PV and S of cover.  Each
    // product is four MMAs of K = 32; a k-step adds 32 bytes (2 in the
    // descriptor's 16-byte units) inside the 128-byte swizzled rows, or 8
    // tensor-memory columns of P.
    // The loop keeps ring counters only, with the descriptors' upper words
    // fixed and the lower words built once; the whole warp runs it and
    // elect.sync picks the issuing lane (always the same one while the warp
    // is converged).
    {
      // every lane waits, so the warp leaves a wait together
      auto wt = [&](uint32_t bar, uint32_t par) { return __all_sync(0xffffffffu, wait_bar(bar, par, wc)); };
      constexpr uint32_t ID = idesc_e4m3(128, 128);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      const uint32_t HI = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t d_q = (uint32_t)sdesc_sw128(s_base, 16, 1024);
      const uint32_t d_k = (uint32_t)sdesc_sw128(s_base + C::OFF_K, 16, 1024);
      const uint32_t d_v = (uint32_t)sdesc_sw128(s_base + C::OFF_V, 16, 1024);
      auto desc = [&](uint32_t lo) { return ((uint64_t)HI << 32) | lo; };
      auto next_kt = [&](int from) {
        int k = from;
        while (k < u.kt_end && !unit_uses(u, k)) ++k;
        return k;
      };
      auto issue_s = [&](int t, int slot) {   // S_t = Q_t K^T
        const uint32_t kd = d_k + (uint32_t)slot * TILE16, qd = d_q + (uint32_t)t * TILE16;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_ss_f8_e(tmem + t * 128, desc(qd + kk * 2), desc(kd + kk * 2), ID, kk > 0);
        mma_commit_e(bar_s(t));
      };
      auto issue_pv = [&](int t, int slot, bool acc) {   // O_t += P_t (V^T)^T, P_t from tensor memory
        const uint32_t vd = d_v + (uint32_t)slot * TILE16;
#pragma unroll
        for (int kk = 0; kk < TILE / 32; ++kk)
          mma_ts_f8_e(tmem + C::TMEM_O + t * D, tmem + t * 128 + kk * 8, desc(vd + kk * 2), ID, acc || kk > 0);
        mma_commit_e(bar_o(t));
      };
      int cp0 = 0, cp1 = 0;   // PV MMAs issued per query tile
      bool ok = wt(bar_q, 0);
      int kt = next_kt(u.kt_begin);
      uint32_t use = kt < u.kt_end ? unit_uses(u, kt) : 0u;
      if (ok && use) {
        ok = wt(bar_k(0), 0);
        if (ok) {
          tc_fence_after();
          if (use & 1u) issue_s(0, 0);
          if (use & 2u) issue_s(1, 0);
          mma_commit_e(bar_kfree(0));
        }
      }
      int s = 0;
      uint32_t ph = 0;   // ring slot of key tile n and the parity of its fill
      while (ok && use) {
        const int sn = (s + 1 == NS) ? 0 : s + 1;
        const uint32_t phn = (s + 1 == NS) ? ph ^ 1u : ph;
        const int ktn = next_kt(kt + 1);
        const uint32_t usen = ktn < u.kt_end ? unit_uses(u, ktn) : 0u;
        bool kwaited = false;
        if (!(ok = wt(bar_v(s), ph))) break;
        if (use & 1u) {
          if (!(ok = wt(bar_p(0), (uint32_t)cp0 & 1u))) break;
          tc_fence_after();
          issue_pv(0, s, cp0 > 0);
          ++cp0;
        }
        if (usen & 1u) {
          if (!(ok = wt(bar_k(sn), phn))) break;
          tc_fence_after();
          kwaited = true;
          issue_s(0, sn);
        }
        if (use & 2u) {
          if (!(ok = wt(bar_p(1), (uint32_t)cp1 & 1u))) break;
          tc_fence_after();
          issue_pv(1, s, cp1 > 0);
          ++cp1;
        }
        mma_commit_e(bar_vfree(s));   // both P.V products of this key tile issued
        if (usen & 2u) {
          if (!kwaited && !(ok = wt(bar_k(sn), phn))) break;
          tc_fence_after();
          issue_s(1, sn);
        }
        if (usen) mma_commit_e(bar_kfree(sn));
        kt = ktn;
        use = usen;
        s = sn;
        ph = phn;
      }
      // every commit above lands before the CTA leaves
      mma_commit_e(bar_done);
      wait_bar(bar_done, 0, wc, false);
    }
   }
  } else {
    reg_alloc<C::REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                  // row inside the tile == TMEM lane
    const int qrow = u.row0 + t * TILE + r;        // local query row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
    const float c = p.scale_log2;                  // scale * log2(e) * dequantisation of Q and K
    const bool causal = mask_is_causal(p.mask_kind, p.causal_in_blocks);
    const int64_t row_first_pos = p.q_offset + u.row0 + t * TILE;
    const int64_t qpos = p.q_offset + qrow;
    float m = -INFINITY, l = 0.f;
    int it = 0;
    bool ok = true;
    for (int kt = u.kt_begin; kt < u.kt_end; ++kt) {
      if (!(unit_uses(u, kt) & (1u << t))) continue;
      ok = wait_bar(bar_s(t), it & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // element mask as in fwd.cu: column j is visible iff lo <= j < lim
      const int64_t key0 = p.kv_offset + (int64_t)kt * TILE;
      const bool tail = (kt == u.nkt - 1) && (u.nk % TILE) != 0;
      const bool diag = causal && (key0 + TILE - 1 > row_first_pos);
      const bool wedge = p.mask_kind == MASK_SLIDING_WINDOW && key0 + p.window <= row_first_pos + TILE - 1;
      const bool edge = tail || diag || wedge;
      int lo = 0, lim = 128;
      if (edge) {
        int64_t l64 = u.nk - (int64_t)kt * TILE;
        if (causal) {
          const int64_t lc = qpos - key0 + 1;
          l64 = lc < l64 ? lc : l64;
        }
        lim = (int)(l64 < 0 ? 0 : (l64 > 128 ? 128 : l64));
        if (wedge) {
          const int64_t f64 = qpos - p.window + 1 - key0;
          lo = (int)(f64 < 0 ? 0 : (f64 > 128 ? 128 : f64));
        }
      }
      // the whole score row into registers (P_t then goes over its first 32
      // columns)
      float s[128];
      {
        uint32_t rr[128];
        tmem_ld128(tS, rr);
#pragma unroll
        for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(rr[j]);
      }
      if (edge) {
#pragma unroll
        for (int j = 0; j < 128; ++j) s[j] = (j >= lo && j < lim) ? s[j] : -INFINITY;
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 128; j += 8) {
        mx0 = max3(mx0, s[j], s[j + 1]);
        mx1 = max3(mx1, s[j + 2], s[j + 3]);
        mx2 = max3(mx2, s[j + 4], s[j + 5]);
        mx3 = max3(mx3, s[j + 6], s[j + 7]);
      }
      mx0 = max3(mx0, mx1, fmaxf(mx2, mx3));
      const float m_new = fmaxf(m, mx0 * c);
      float alpha = 1.f;
      bool rescale = false;
      if (__any_sync(0xffffffffu, it == 0 || m_new > m + FP8_THRESHOLD)) {
        // the reference max moves: O_t (if any) is rescaled by 2^(m_old - m_new)
        if (it > 0) {
          alpha = (m_new == -INFINITY) ? 1.f : ex2(m - m_new);
          rescale = true;
        }
        m = m_new;
      }
      // p = 2^(s c - m + 7) <= 2^8, two lanes per packed FMA, and the exact fp32 sum
      const float mb = ((m == -INFINITY) ? 0.f : m) - FP8_P_OFFSET;
      float la[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 128; j += 2) {
        float x0, x1;
        fma2(x0, x1, s[j], s[j + 1], c, c, -mb, -mb);
        s[j] = ex2(x0);
        s[j + 1] = ex2(x1);
        const int a = (j >> 1) & 3;
        add2(la[2 * a], la[2 * a + 1], la[2 * a], la[2 * a + 1], s[j], s[j + 1]);
      }
      // P as e4m3 into the first 32 columns of S_t: column j holds keys
      // 4j..4j+3, the first in the lowest byte
      {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = pack_e4m3x4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
        tmem_st32(tS, pk);
      }
      // O_t must hold the previous PV before a rescale (PV_t of this key tile
      // follows it on the tensor core, so nothing else has to wait)
      if (rescale) {
        ok = wait_bar(bar_o(t), (it - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      if (rescale) {
#pragma unroll
        for (int h64 = 0; h64 < D / 64; ++h64) {
          uint32_t rr[64];
          tmem_ld64(tO + h64 * 64, rr);
#pragma unroll
          for (int j = 0; j < 64; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
          tmem_st64(tO + h64 * 64, rr);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_p(t));
      ++it;
      l = l * alpha + (((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7])));
    }
    // ---------------------------------------------------------- epilogue
    if (ok && !abort_flag) {
      const bool have = it > 0;
      if (have) {
        ok = wait_bar(bar_o(t), (it - 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        const bool valid_row = qrow < p.Nq;
        const float inv_l = (l > 0.f) ? v_descale / l : 0.f;
        const size_t o_off = (size_t)((int64_t)u.bh * p.o_hs + (int64_t)qrow * p.o_rs);
#pragma unroll
        for (int h64 = 0; h64 < D / 64; ++h64) {
          uint32_t rr[64];
          if (have) {
            tmem_ld64(tO + h64 * 64, rr);
          } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) rr[j] = 0u;
          }
          if (valid_row) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o_off + h64 * 64);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4 v4;
              v4.x = pack_bf16(__uint_as_float(rr[8 * j + 0]) * inv_l, __uint_as_float(rr[8 * j + 1]) * inv_l);
              v4.y = pack_bf16(__uint_as_float(rr[8 * j + 2]) * inv_l, __uint_as_float(rr[8 * j + 3]) * inv_l);
              v4.z = pack_bf16(__uint_as_float(rr[8 * j + 4]) * inv_l, __uint_as_float(rr[8 * j + 5]) * inv_l);
              v4.w = pack_bf16(__uint_as_float(rr[8 * j + 6]) * inv_l, __uint_as_float(rr[8 * j + 7]) * inv_l);
              dst[j] = v4;
            }
          }
        }
        if (valid_row && p.lse != nullptr)
          p.lse[(int64_t)u.bh * p.l_hs + (int64_t)qrow * p.l_rs] =
              (l > 0.f) ? (m - FP8_P_OFFSET + __log2f(l)) * 0.69314718055994531f : -INFINITY;
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

// V [heads][N][128] e4m3 -> V^T [heads][128][Np] e4m3 with keys past N zeroed,
// one 128-key tile per CTA through shared memory (rows padded to 132 bytes so
// the column reads spread over the banks).
__global__ void __launch_bounds__(256) transpose_v_fp8_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                              int N, int Np) {
  __shared__ __align__(16) uint8_t tile[128][132];
  const int head = blockIdx.y, k0 = blockIdx.x * 128;
  const uint8_t* src = v + ((size_t)head * N + k0) * 128;
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {   // 16-byte chunks of 128 key rows
    const int kr = i >> 3, c = i & 7;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + kr < N) x = *reinterpret_cast<const uint4*>(src + (size_t)kr * 128 + c * 16);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&tile[kr][c * 16]);
    dst[0] = x.x; dst[1] = x.y; dst[2] = x.z; dst[3] = x.w;
  }
  __syncthreads();
  uint8_t* out = vt + (size_t)head * 128 * Np + k0;
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {   // 16-byte chunks of 128 head-dim rows
    const int dr = i >> 3, c = i & 7;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = c * 16 + q * 4;
      w[q] = (uint32_t)tile[k][dr] | ((uint32_t)tile[k + 1][dr] << 8) | ((uint32_t)tile[k + 2][dr] << 16) |
             ((uint32_t)tile[k + 3][dr] << 24);
    }
    *reinterpret_cast<uint4*>(out + (size_t)dr * Np + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_transpose_v_fp8(const void* v, void* vt, int heads, int N, int Np, cudaStream_t s) {
  transpose_v_fp8_kernel<<<dim3((unsigned)(Np / 128), (unsigned)heads), 256, 0, s>>>(
      static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, Np);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const FwdParams& p,
                           float v_descale, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(p.B * p.Hq) * (unsigned)p.nqc;
  fwd_fp8_kernel<<<grid, Fp8Cfg::THREADS, Fp8Cfg::SMEM_BYTES, s>>>(tq, tk, tvt, p, v_descale);
  return cudaGetLastError();
}

}  // namespace attn
