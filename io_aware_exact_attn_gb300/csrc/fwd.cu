// fwd.cu -- exact attention forward for sm_103a: TMA-fed tcgen05 MMAs with the
// score and output accumulators in tensor memory, online softmax in base 2,
// deferred normalisation and one saved log-sum-exp per row.
//
// What it computes: O = softmax(scale * Q K^T) V over the visible keys and
// LSE = ln sum_j exp(scale * q.k_j)  ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", abstract: tiling between
// HBM and on-chip memory so S and P never reach HBM; "FlashAttention-2"
// reviews, first review questions: the online-softmax recurrences with
// diag(l)^-1 applied once at the end; second review items 1-2: deferred
// rescaling, one LSE per row saved for the backward pass).
//
// One CTA = one work unit = 256 query rows (two 128-row tiles, t = 0, 1) of
// one (batch, query head); launched heaviest-first (see schedule.h).
// Warp roles (12 warps, three warpgroups):
//   warp 0      TMA producer: Q0/Q1 once, then K_j and V_j into NS-deep rings;
//               one lane per 16 KB box, K slots released after the S MMAs
//   warp 1      MMA issuer (the whole warp runs the loop, one elected lane
//               issues): S_t = Q_t K_j^T, then O_t += P_t V_j
//               with P_t read from tensor memory; owns the TMEM allocation
//   warps 2-3   idle (they complete the control warpgroup)
//   warps 4-7   softmax for tile 0 (warp w owns TMEM lanes 32*(w%4)..+31)
//   warps 8-11  softmax for tile 1
// The control warpgroup gives registers back (56 per thread) so that the two
// softmax warpgroups can hold a full 128-column score row each (224 per
// thread): 128*56 + 256*224 = 384*168, the block's launch allotment.
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [256+d, 256+2d).  P_t (bf16 pairs) overwrites the first 64 columns of S_t.
// The tensor core order is PV_0(n), S_0(n+1), PV_1(n), S_1(n+1): S_t of the
// next key tile follows the PV_t that reads P_t out of the same columns.
//
// Online softmax per row, in units of log2: x = s * scale * log2(e),
// m = reference max, p = 2^(x - m), l = sum p.  The weights of a tile are
// first taken against the current m; only when they sum past 2^8 (which any
// weight above 2^8 would cause) is the tile's row max found and m moved to it,
// so p <= 256 always and the max costs nothing in the usual case.  When m
// moves, O_t is rescaled in tensor memory by 2^(m_old - m_new).  This keeps
// the result exact: O and l always share the same reference max and the final
// O / l cancels it.
#include "internal.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

namespace {

// the reference max moves once a tile's weights (relative to it) sum past
// 2^8, which any single weight above 2^8 implies
constexpr float RESCALE_LIMIT = 256.0f;

template <int D>
struct FwdCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;          // K/V ring depth
  static constexpr int NBOX = D / 64;                     // 64-column TMA boxes per row
  static constexpr uint32_t BOX_BYTES = 128 * 128;        // 128 rows x 128 bytes
  static constexpr uint32_t TILE_BYTES = NBOX * BOX_BYTES;
  static constexpr uint32_t OFF_K = 2 * TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;
  // d = 64: the P.V product also sums the rounded weights.  Its B operand is
  // V followed by a 64-column block of ones (N = 80: 64 columns of V, then 16
  // of ones), so column 64 of O_t accumulates the sum of the bf16 weights,
  // rescaled with O.  At d = 128 tensor memory has no room for those columns
  // and the softmax sums the weights itself.
  static constexpr bool ROWSUM_MMA = (D == 64);
  static constexpr uint32_t OFF_ONES = OFF_V + NS * TILE_BYTES;   // 128 rows x 128 bytes of bf16 1.0
  static constexpr uint32_t SMEM_TILES = OFF_ONES + (ROWSUM_MMA ? BOX_BYTES : 0u);
  static constexpr uint32_t SMEM_BYTES = SMEM_TILES + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_O = 256;
  static constexpr uint32_t O_STRIDE = ROWSUM_MMA ? 128 : D;     // TMEM columns between O_0 and O_1
  static constexpr int PV_N = ROWSUM_MMA ? D + 16 : D;
  static constexpr int THREADS = 384;
  static constexpr uint32_t REGS_CTRL = 56, REGS_SOFTMAX = 224;
};

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::NS;
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
  auto bar_vfree = [&](int s) { return smem_u32(&bars[1 + 3 * NS + s]); };  // V slot read by both PV MMAs
  auto bar_s = [&](int t) { return smem_u32(&bars[1 + 4 * NS + t]); };
  auto bar_p = [&](int t) { return smem_u32(&bars[1 + 4 * NS + 2 + t]); };
  auto bar_o = [&](int t) { return smem_u32(&bars[1 + 4 * NS + 4 + t]); };
  const uint32_t bar_done = smem_u32(&bars[1 + 4 * NS + 6]);

  Unit u;   // warp-uniform: every warp works it out for itself
  if (p.n_splits > 0)
    u = decode_unit(blockIdx.x, p.B, p.Hq, p.Hkv, p.dec_nq, p.Nk, p.seq_lens, p.n_splits, p.split_tiles,
                    p.dec_interleave != 0);
  else if (p.cu_seqlens != nullptr)
    u = varlen_unit(blockIdx.x, p.B, p.Hq, p.Hkv, D, p.cu_seqlens, p.total, p.Nq, p.mask_kind, p.window);
  else
    u = fwd_unit(blockIdx.x, p.B, p.Hq, p.Hkv, p.Nq, p.Nk, p.nqc, p.head_group, p.mask_kind, p.causal_in_blocks,
                 p.block_mask, p.nkb, p.window, p.q_offset, p.kv_offset);
  if (u.bad && threadIdx.x == 0) atomicOr(p.status, ATTN_DEV_BOUNDS);
  if (u.empty) return;   // a chunk past the end of its sequence (or of a malformed one): nothing set up yet
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
    prefetch_tmap(&tv);
  }
  if constexpr (C::ROWSUM_MMA) {
    // the block of ones the P.V product reads after V; the tensor core reads it
    // through the async proxy
    uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::OFF_ONES);
    for (int i = threadIdx.x; i < (int)(C::BOX_BYTES / 4); i += C::THREADS) ones[i] = 0x3F803F80u;
    fence_proxy_async_smem();
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
    // Each box of a tile is issued by its own lane: TMA copies issued by one
    // thread are processed one after another, so spreading them over lanes is
    // what lets several 16 KB boxes stream into the SM at the same time.
    // decoding with alternating tiles: both query tiles read the rows of tile 0
    const int q_tiles = u.alternate ? 1 : 2;
    if (lane == 0) mbar_arrive_expect_tx(bar_q, q_tiles * C::TILE_BYTES);
    __syncwarp();
    if (lane < q_tiles * C::NBOX) {
      const int t = lane / C::NBOX, bx = lane % C::NBOX;
      tma_load_3d(s_base + t * C::TILE_BYTES + bx * C::BOX_BYTES, &tq, bx * 64, (int)(u.seq0 + u.row0 + t * TILE), u.bh,
                  bar_q);
    }
    if (p.tile_counts != nullptr && lane == 0) {   // the unit's identity in the debug record
      int32_t* rec = p.tile_counts + (size_t)DEBUG_FIELDS * blockIdx.x;
      rec[0] = u.bh;
      rec[1] = u.row0;
      rec[2] = u.split;
      rec[3] = (int32_t)u.seq0;
      rec[5] = 0;   // not recorded by the forward kernel
    }
    int n = 0;
    bool ok = true;
    for (int kt = u.kt_begin; kt < u.kt_end && ok; ++kt) {
      if (!unit_uses(u, kt)) continue;
      const int s = n % NS;
      const uint32_t fph = ((n / NS) - 1) & 1;
      if (n >= NS) ok = wait_bar(bar_kfree(s), fph, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (lane == 0) mbar_arrive_expect_tx(bar_k(s), C::TILE_BYTES);
      __syncwarp();
      if (lane < C::NBOX)
        tma_load_3d(s_base + C::OFF_K + s * C::TILE_BYTES + lane * C::BOX_BYTES, &tk, lane * 64,
                    (int)(u.seq0 + kt * TILE), u.kvh,
                    bar_k(s));
      if (n >= NS) ok = wait_bar(bar_vfree(s), fph, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (lane == 0) mbar_arrive_expect_tx(bar_v(s), C::TILE_BYTES);
      __syncwarp();
      if (lane >= C::NBOX && lane < 2 * C::NBOX)
        tma_load_3d(s_base + C::OFF_V + s * C::TILE_BYTES + (lane - C::NBOX) * C::BOX_BYTES, &tv,
                    (lane - C::NBOX) * 64, (int)(u.seq0 + kt * TILE), u.kvh, bar_v(s));
      ++n;
    }
    if (p.tile_counts != nullptr && lane == 0) p.tile_counts[(size_t)DEBUG_FIELDS * blockIdx.x + 4] = n;   // key tiles loaded
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
    // PV_t(n) that reads them, and tcgen05.mma from one thread execute in
    // issue order.  Each softmax thus has two MMAs of cover (PV of the other
    // tile and its S) before its own PV is needed.
    // tcgen05.mma issue stalls once a few MMAs are queued, so the issuer is
    // held for most of each group and anything it does between groups idles
    // the tensor pipe: it keeps ring counters only, and descriptors are built
    // once (a k-step adds a compile-time offset to the start-address field;
    // shared-memory addresses stay below 256 KB, so the 14-bit field never
    // carries).  The whole warp runs the loop converged and elect.sync picks
    // the issuing lane for each MMA and commit (the lowest active lane, so
    // always the same thread, as in-order execution and commit tracking
    // need): the same loop run by one lane of a diverged warp issued about
    // one MMA per 90-110 cycles here, slower than the pipe's 64.
    {
      // every lane waits, so the warp leaves a wait together
      auto wt = [&](uint32_t bar, uint32_t par) { return __all_sync(0xffffffffu, wait_bar(bar, par, wc)); };
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint32_t id_pv = idesc_bf16(128, C::PV_N, false, true);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      const uint32_t hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t d_q = (uint32_t)sdesc_sw128(s_base, 16, 1024);
      const uint32_t d_k = (uint32_t)sdesc_sw128(s_base + C::OFF_K, 16, 1024);
      // MN-major V: at d = 128 the leading offset is the distance between its two
      // 64-column boxes; with the row-sum columns (d = 64) it is the distance
      // from the slot to the block of ones, which shrinks by a tile per slot
      const uint32_t d_vmn = (uint32_t)sdesc_sw128(s_base + C::OFF_V, C::ROWSUM_MMA ? C::OFF_ONES - C::OFF_V : C::BOX_BYTES, 1024);
      constexpr uint32_t V_SLOT_STEP = C::ROWSUM_MMA ? (C::TILE_BYTES >> 4) - ((C::TILE_BYTES >> 4) << 16) : (C::TILE_BYTES >> 4);
      auto desc = [&](uint32_t lo) { return ((uint64_t)hi << 32) | lo; };
      auto kstep = [](int kk) { return (uint32_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4); };
      auto next_kt = [&](int from) {
        int k = from;
        while (k < u.kt_end && !unit_uses(u, k)) ++k;
        return k;
      };
      const uint32_t q_step = u.alternate ? 0u : TILE16;   // alternating decode: one Q tile for both
      auto issue_s = [&](int t, int slot) {
        const uint32_t kd = d_k + (uint32_t)slot * TILE16;
        const uint32_t qd = d_q + (uint32_t)t * q_step;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_e(tmem + t * 128, desc(qd + kstep(kk)), desc(kd + kstep(kk)), id_s, kk > 0);
        mma_commit_e(bar_s(t));
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint32_t vd = d_vmn + (uint32_t)slot * V_SLOT_STEP;
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          mma_ts_e(tmem + C::TMEM_O + t * C::O_STRIDE, tmem + t * 128 + kk * 8, desc(vd + (uint32_t)kk * (2048 >> 4)), id_pv,
                 (acc || kk > 0));
        mma_commit_e(bar_o(t));
      };
      int it0 = 0, it1 = 0;   // PV MMAs issued per tile
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
          if (!(ok = wt(bar_p(0), (uint32_t)it0 & 1u))) break;
          tc_fence_after();
          issue_pv(0, s, it0 > 0);
          ++it0;
        }
        if (usen & 1u) {
          if (!(ok = wt(bar_k(sn), phn))) break;
          tc_fence_after();
          kwaited = true;
          issue_s(0, sn);
        }
        if (use & 2u) {
          if (!(ok = wt(bar_p(1), (uint32_t)it1 & 1u))) break;
          tc_fence_after();
          issue_pv(1, s, it1 > 0);
          ++it1;
        }
        mma_commit_e(bar_vfree(s));   // both PV MMAs of this key tile issued
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
    const int trow0 = u.row0 + (u.alternate ? 0 : t * TILE);   // first local row of the tile
    const int qrow = trow0 + r;                    // local query row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::TMEM_O + t * C::O_STRIDE;
    const float c = p.scale_log2;
    const bool causal = mask_is_causal(p.mask_kind, p.causal_in_blocks);
    // positions: row i of the call sits at q_offset + i; when decoding, row r
    // is query r % dec_nq of its head, at u.pos0 + r % dec_nq
    const bool decoding = p.n_splits > 0;
    const int64_t row_first_pos = decoding ? u.pos0 : p.q_offset + trow0;  // earliest row of the tile
    const int64_t qpos = decoding ? u.pos0 + qrow % p.dec_nq : p.q_offset + qrow;
    float m = -INFINITY, l = 0.f, lr = 0.f;
    int it = 0;
    bool ok = true;
    for (int kt = u.kt_begin; kt < u.kt_end; ++kt) {
      if (!(unit_uses(u, kt) & (1u << t))) continue;
      ok = wait_bar(bar_s(t), it & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // element mask on the ragged last key tile, on causal diagonal tiles
      // and on tiles crossing the lower edge of a sliding window: column j is
      // visible iff lo <= j < lim
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
          const int64_t f64 = qpos - p.window + 1 - key0;   // first key in the row's window
          lo = (int)(f64 < 0 ? 0 : (f64 > 128 ? 128 : f64));
        }
      }
      auto load_scores = [&](float (&sc)[128]) {
        uint32_t rr[128];
        tmem_ld128(tS, rr);   // the whole score row in one round trip
#pragma unroll
        for (int j = 0; j < 128; ++j) sc[j] = __uint_as_float(rr[j]);
        if (edge) {
#pragma unroll
          for (int j = 0; j < 128; ++j) sc[j] = (j >= lo && j < lim) ? sc[j] : -INFINITY;
        }
      };
      // p = 2^(s*c - mb), two lanes per packed FMA; in place
      auto exponentials = [&](float (&sc)[128], float mb) {
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
          float x0, x1;
          fma2(x0, x1, sc[j], sc[j + 1], c, c, -mb, -mb);
          sc[j] = ex2(x0);
          sc[j + 1] = ex2(x1);
        }
      };
      // l sums the fp32 weights (for the log-sum-exp); lr, below, sums the
      // bf16-rounded weights P.V sees, so O / lr cancels the rounding of a
      // dominant weight
      uint32_t pk[64];
      auto pack_sum = [&](const float (&sc)[128]) {
        float la[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // four independent packed chains
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          // bf16, rounded to nearest; O is normalised by the sum of these same
          // weights, so a dominant weight's rounding cancels
          pk[j] = pack_bf16(sc[2 * j], sc[2 * j + 1]);
          const int a = 2 * (j & 3);
          add2(la[a], la[a + 1], la[a], la[a + 1], sc[2 * j], sc[2 * j + 1]);
        }
        return ((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7]));
      };
      // Exponentials against the current reference max first.  Every weight
      // stays within 2^THRESHOLD unless the row's sum of them exceeds that, so
      // in the usual case the tile's row max is never needed; otherwise (and
      // for a row's first visible tile) the max is found from the scores
      // still in TMEM, the reference moves to it, and the weights are redone.
      float s[128];
      float lt = 0.f;
      load_scores(s);
      if (it > 0) {   // a tile's first key tile always needs its row max: no speculative pass
        exponentials(s, (m == -INFINITY) ? 0.f : m);
        lt = pack_sum(s);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (__any_sync(0xffffffffu, m == -INFINITY || !(lt <= RESCALE_LIMIT))) {
        if (it > 0) load_scores(s);
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
        // O_t (if any) is rescaled by 2^(m_old - m_new) below
        if (it > 0) {
          alpha = (m_new == -INFINITY) ? 1.f : ex2(m - m_new);
          rescale = true;
        }
        m = m_new;
        exponentials(s, (m == -INFINITY) ? 0.f : m);
        lt = pack_sum(s);
      }
      tmem_st64(tS, pk);    // P_t (bf16 pairs) over the first 64 columns of S_t
      if (rescale) {
        // PV_t of the previous key tile must have landed in O_t first
        ok = wait_bar(bar_o(t), (it - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int h64 = 0; h64 < D / 64; ++h64) {
          uint32_t rr[64];
          tmem_ld64(tO + h64 * 64, rr);
#pragma unroll
          for (int j = 0; j < 64; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
          tmem_st64(tO + h64 * 64, rr);
        }
        if constexpr (C::ROWSUM_MMA) {   // the row-sum columns scale with O
          uint32_t rr[16];
          tmem_ld16(tO + D, rr);
#pragma unroll
          for (int j = 0; j < 16; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
          tmem_st16(tO + D, rr);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_p(t));
      ++it;
      l = l * alpha + lt;
      if constexpr (!C::ROWSUM_MMA) {
        // rounded-weight sum after P has been handed to the tensor core
        float ra[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int a = 2 * (j & 3);
          add_bf16x2_to_f32(ra[a], ra[a + 1], pk[j]);
        }
        const float r0 = (ra[0] + ra[1]) + (ra[2] + ra[3]), r1 = (ra[4] + ra[5]) + (ra[6] + ra[7]);
        lr = lr * alpha + (r0 + r1);
      }

    }
    if (p.tile_counts != nullptr && r == 0) p.tile_counts[(size_t)DEBUG_FIELDS * blockIdx.x + 6 + t] = it;
    // ---------------------------------------------------------- epilogue
    if (ok && !abort_flag) {
      const bool have = it > 0;
      if (have) {
        ok = wait_bar(bar_o(t), (it - 1) & 1, wc);
      } else {   // no key tile: the bf16 rows below are staged where the Q copy may still be landing
        ok = wait_bar(bar_q, 0, wc);
      }
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const bool valid_row = qrow < u.nq;
        if constexpr (C::ROWSUM_MMA) {   // the sum of the rounded weights, from the P.V product
          uint32_t rr[16];
          if (have) tmem_ld16(tO + D, rr);
          lr = have ? __uint_as_float(rr[0]) : 0.f;
        }
        const float inv_l = (lr > 0.f) ? 1.f / lr : 0.f;
        const int64_t grow = u.seq0 + qrow;   // row within the head (token index when batches are ragged)
        // alternating decode: tile t's partial is split 2 * split + t
        const int64_t split_off = (int64_t)(u.alternate ? 2 * u.split + t : u.split) * p.split_rows;
        const size_t o_off = (size_t)(split_off * D + (int64_t)u.bh * p.o_hs + grow * p.o_rs);
        const size_t l_off = (size_t)(split_off + (int64_t)u.bh * p.l_hs + grow * p.l_rs);
        uint32_t ob[OUT_F32 ? 1 : D / 2];   // the bf16 row (OUT_F32 writes fp32 rows directly)
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
            if constexpr (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + o_off + h64 * 64);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                dst[j] = make_float4(__uint_as_float(rr[4 * j]) * inv_l, __uint_as_float(rr[4 * j + 1]) * inv_l,
                                     __uint_as_float(rr[4 * j + 2]) * inv_l,
                                     __uint_as_float(rr[4 * j + 3]) * inv_l);
            }
          }
          if constexpr (!OUT_F32) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              ob[h64 * 32 + j] = pack_bf16(__uint_as_float(rr[2 * j]) * inv_l, __uint_as_float(rr[2 * j + 1]) * inv_l);
          }
        }
        if constexpr (!OUT_F32) {
          // bf16 rows staged through a Q tile, so each store covers whole
          // rows.  Tile t stages in Q_t: no MMA reads it once this tile's last
          // P.V has completed.  Alternating decode loads Q_0 alone and both
          // tiles' S read it, so an S of tile 1 may still be reading Q_0 when
          // tile 0 ends: there tile 0 stages in the unused Q_1 and tile 1, whose
          // last P.V follows every other MMA of the unit, in Q_0.
          const int wrow = trow0 + wq * 32;   // this warp's first local row
          const int region = u.alternate ? 1 - t : t;
          char* base = reinterpret_cast<char*>(static_cast<__nv_bfloat16*>(p.o) +
                                               (size_t)(split_off * D + (int64_t)u.bh * p.o_hs +
                                                        (u.seq0 + wrow) * p.o_rs));
          warp_store_rows<D / 8>(s_base + (uint32_t)(region * 4 + wq) * (32u * D * 2), ob, base,
                                 (size_t)p.o_rs * sizeof(__nv_bfloat16), u.nq - wrow);
        }
        if (valid_row && p.lse != nullptr)
          p.lse[l_off] = (l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
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

template <int D, bool F32>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t s) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = fwd_grid(p);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, cudaStream_t s) {
  if (d == 128) return out_f32 ? launch_fwd_t<128, true>(tq, tk, tv, p, s) : launch_fwd_t<128, false>(tq, tk, tv, p, s);
  return out_f32 ? launch_fwd_t<64, true>(tq, tk, tv, p, s) : launch_fwd_t<64, false>(tq, tk, tv, p, s);
}

}  // namespace attn
