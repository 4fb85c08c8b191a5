// bwd.cu -- exact attention backward for sm_103a.  The N x N probabilities are
// never stored: every kernel recomputes P = 2^(S * scale * log2(e) - lse2) from
// the saved log-sum-exp ("DISTFLASHATTN" reviews, first review point 3: the
// backward pass needs no stored attention matrix; "FlashAttention-2" reviews,
// second review items 2-3: the saved log-sum-exp, and the backward pass
// restructured around the query-derivative update).
//
// Gradient of the loss <O, dO> (D_i = sum_k dO_ik O_ik, written by the
// preprocessing kernel in merge.cu):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q.
// Two kernels, both TMA-fed with tcgen05 accumulators in tensor memory:
//   dkdv_kernel  a run of 128-key tiles of (batch, kv head) per CTA; loops
//                over the query tiles that see each key tile, for every query
//                head of the GQA group, so dK and dV need no atomics.  Per
//                query tile: S^T - lse2/c = K Q^T and dP^T - D = V dO^T
//                (tensor cores; the per-query statistics enter through one
//                extra K = 16 step of each product), P^T and dS^T
//                (elementwise warpgroups, written back to tensor memory as
//                bf16), dV += P^T dO, dK += dS^T Q (A operand from tensor
//                memory).
//   dq_kernel    one CTA per 128-row query tile of one (batch, query head);
//                loops over the key tiles it sees: S = Q K^T, dP = dO V^T,
//                dS = P * (dP - D), dQ += dS K, dQ accumulated in fp32 in
//                tensor memory and scaled / rounded once at the end.
// Warp roles (12 warps): warp 0 TMA producer (the dQ kernel's second
// producer is warp 2), warp 1 MMA issuer (one elected lane, owns the TMEM
// allocation), warps 4-11 elementwise work in two warpgroups that split the
// 128 columns of every tile row between them (warp w owns TMEM lanes
// 32*(w%4)..+31; one thread per row and half); warps 1-3 of the dK/dV kernel
// first decode the run's units.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

namespace {

template <int D>
struct BwdCfg {
  static constexpr int NBOX = D / 64;
  static constexpr uint32_t BOX_BYTES = 128 * 128;
  static constexpr uint32_t TILE_BYTES = NBOX * BOX_BYTES;
  // dK/dV rings: {Q_i, statistics block of tile i} QS deep, dO_i OS deep.
  // dO_i is last read by dV_i, Q_i by dK_i a product later, and S^T_{i+1}
  // (which needs Q_{i+1}) is issued right after dV_i, so the Q slots are the
  // ones that must be refilled well ahead
  static constexpr int QS = (D == 128) ? 3 : 4;
  static constexpr int OS = (D == 128) ? 1 : 2;
  // both kernels: 12 warps; the control warpgroup gives registers back to the
  // two elementwise warpgroups: 128*112 + 256*176 = 59392 <= 384*168 (launch
  // allotment).  The dK/dV control warps walk a run of units over two rings
  // with three kinds of operand descriptors: ptxas reports spills for them up
  // to 104, none at 112; the elementwise warps need no more than 176
  static constexpr int SPLIT_THREADS = 384;
  static constexpr uint32_t REGS_CTRL = 112, REGS_ELEM = 176;
};

// The sliding window includes the causal rule.
__device__ __forceinline__ bool causal_of(const BwdParams& p) {
  return p.mask_kind == MASK_CAUSAL || p.mask_kind == MASK_SLIDING_WINDOW ||
         (p.mask_kind == MASK_BLOCK_SPARSE && p.causal_in_blocks);
}

// Width of the sliding window, or a bound no position difference reaches.
__device__ __forceinline__ int window_of(const BwdParams& p) {
  return p.mask_kind == MASK_SLIDING_WINDOW ? p.window : 0x7fffffff;
}

// Positions from the first key of key tile kt to the first query of query
// tile qt: query row r of qt and key column c of kt are base + r - c apart
// (delta = q_offset - kv_offset, 0 unless the call is one chunk pair).
__device__ __forceinline__ int tile_base(const BwdParams& p, int qt, int kt) { return p.delta + (qt - kt) * TILE; }

// Query tile qt sees key tile kt: some query of qt lies 0..window-1 positions
// after some key of kt (the largest distance in the pair is base + 127, the
// smallest base - 127), and the block mask keeps the pair.
__device__ __forceinline__ bool tile_pair_visible(const BwdParams& p, int qt, int kt) {
  const int base = tile_base(p, qt, kt);
  if (causal_of(p) && base + (TILE - 1) < 0) return false;
  if (base - (TILE - 1) >= window_of(p)) return false;
  if (p.mask_kind == MASK_BLOCK_SPARSE && p.block_mask[(size_t)qt * p.nkb + kt] == 0) return false;
  return true;
}

// Ragged batches: the sequence b owning backward unit `cta` when every
// sequence owns heads * (its 128-row tiles) consecutive units, in index order
// (pcu: the tile-padded row offsets of the preprocess pass, so a malformed
// sequence owns none), and the unit's index j inside it.  False past the last.
__device__ __forceinline__ bool ragged_tile_unit(const int* pcu, int B, int heads, int64_t cta, int* b, int* nt,
                                                 int64_t* j) {
  if (cta >= (int64_t)heads * (pcu[B] / TILE)) return false;
  int lo = 0, hi = B;   // the largest b with heads * pcu[b] / 128 <= cta
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)heads * (pcu[mid] / TILE) <= cta) lo = mid;
    else hi = mid;
  }
  *b = lo;
  *nt = (pcu[lo + 1] - pcu[lo]) / TILE;
  *j = cta - (int64_t)heads * (pcu[lo] / TILE);
  return true;
}

// Causal masks: the first query tile with a query at or after the first key
// of key tile kt (base + 127 >= 0).
__device__ __forceinline__ int first_query_tile(const BwdParams& p, int kt) {
  const int y = kt * TILE - p.delta - (TILE - 1);
  return y <= 0 ? 0 : (y + TILE - 1) / TILE;
}

// Causal masks: one past the last key tile with a key at or before the last
// query of query tile qt, capped at nkt.
__device__ __forceinline__ int key_tile_end(const BwdParams& p, int qt, int nkt) {
  const int z = p.delta + qt * TILE + (TILE - 1);
  return z < 0 ? 0 : min(nkt, z / TILE + 1);
}

// TMEM column of the bf16 A operand for MMA k-step kk (16 rows of K each) when
// the operand is written in two halves: k-steps 0-3 at columns [0, 32) and
// 4-7 at [64, 96) relative to the region start.
__host__ __device__ constexpr uint32_t half_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

// =========================================================================
// dK / dV
// Tensor memory: S^T [0,128) (P^T bf16 overwrites [0,64)), dP^T [128,256)
// (dS^T bf16 overwrites [128,192)), dV [256,256+d), dK [256+d,256+2d).
// Shared memory: K, V (resident per unit), a ring of {Q_i, the statistics
// operand of query tile i} and one of dO_i, the two constant A operands of
// the statistics steps, and 1 KB per elementwise warp to stage the
// epilogue's rows.
// Each S^T and dP^T product has one more K = 16 step whose B operand is the
// query tile's block of the statistics operand (the preprocessing kernel
// writes it: -lse2 and -D as bf16 triples) and whose A operand is constant:
// the bf16 split of 1/c (c = scale * log2 e) under the lse2 columns for S^T,
// ones under the D columns for dP^T.  So the accumulators already hold
// S^T - lse2/c and dP^T - D, and the elementwise phases read no per-column
// values from shared memory: such loads wait behind the tensor core's operand
// reads while a product with both operands in shared memory runs (measured on
// GB300: the two phases took 2.2 times as long under such products when each
// lane loaded its columns' lse2 and D, and no longer without those loads).
// Order on the tensor core: S^T_0, dP^T_0, then dV_i, S^T_{i+1}, dK_i,
// dP^T_{i+1} per query tile i (see the MMA issuer).
//
// A CTA takes a run of kv_run consecutive units of the launch order (similar
// costs; the hardware still balances the CTAs).  The ring, the barriers and
// tensor memory carry on from one unit to the next, so the next unit's K/V
// load (as soon as its predecessor's last S^T and dP^T products are done) and
// first two products overlap the current unit's last tile and epilogue; the
// next unit's first dV product waits until the epilogue has read the
// accumulators.
// =========================================================================

// One work unit of the dK/dV kernel: a 128-key tile of one (batch, kv head).
struct KvUnit {
  int kt, bkv, b, hkv, tok0, n_seq, nqt, qt_first, kv_head;
  int ntile;                 // (query head, query tile) pairs it visits
  int64_t lrow_b, lrow_hs;   // rows of its lse2 / D entries: sequence start, distance between query heads
};
constexpr int MAX_KV_RUN = 8;   // units per CTA at most

// Unit u of the launch order (heaviest first inside each head group); false
// when it does nothing (past the last unit, or past the end of a shorter
// ragged sequence).  Every role of a CTA walks the same units.  Called by a
// whole warp (the visible query tiles are counted 32 at a time).
template <int D>
__device__ __forceinline__ bool kv_unit(const BwdParams& p, int64_t u, KvUnit& x) {
  const bool ragged = p.cu_seqlens != nullptr;
  if (ragged) {   // sequence by sequence; inside one, kv-head groups sized for L2, key tiles ascending
    int sb = 0, nt = 0;
    int64_t j = 0;
    if (!ragged_tile_unit(p.pcu, p.B, p.Hkv, u, &sb, &nt, &j)) return false;
    if (!seq_range_ok(p.cu_seqlens, sb, p.total, p.Nq)) return false;   // never: such a sequence owns no tile
    const int len = p.cu_seqlens[sb + 1] - p.cu_seqlens[sb];
    int hk = 0;
    grouped_unit(j, p.Hkv, nt, q_stream_group(1, p.Hq, p.Hkv, len, D), &hk, &x.kt);
    x.bkv = sb * p.Hkv + hk;
  } else {
    const int nkt_all = (p.Nk + TILE - 1) / TILE;
    if (u >= (int64_t)p.B * p.Hkv * nkt_all) return false;
    grouped_unit(u, p.B * p.Hkv, nkt_all, p.kv_group, &x.bkv, &x.kt);  // key tiles ascending: heaviest first
  }
  x.b = x.bkv / p.Hkv;
  x.hkv = x.bkv % p.Hkv;
  x.tok0 = ragged ? p.cu_seqlens[x.b] : 0;    // packed tensors hold fewer than 2^31 tokens
  x.n_seq = ragged ? p.cu_seqlens[x.b + 1] - x.tok0 : p.Nk;
  if (x.kt * TILE >= x.n_seq) return false;
  const int nq_seq = ragged ? x.n_seq : p.Nq;
  x.lrow_hs = ragged ? (int64_t)p.pcu[p.B] : (int64_t)p.Np;
  x.lrow_b = ragged ? (int64_t)p.pcu[x.b] : (int64_t)x.b * p.Hq * p.Np;
  x.kv_head = ragged ? x.hkv : x.bkv;   // head coordinate in the K / V maps
  x.nqt = (nq_seq + TILE - 1) / TILE;
  x.qt_first = causal_of(p) ? first_query_tile(p, x.kt) : 0;
  const int lane = threadIdx.x & 31;
  int nvis = 0;
  for (int q0 = x.qt_first; q0 < x.nqt; q0 += 32) {
    const int qt = q0 + lane;
    nvis += __popc(__ballot_sync(0xffffffffu, qt < x.nqt && tile_pair_visible(p, qt, x.kt)));
  }
  x.ntile = nvis * (p.Hq / p.Hkv);
  return true;
}

template <int D, bool F32>
__global__ void __launch_bounds__(BwdCfg<D>::SPLIT_THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int QS = C::QS, OS = C::OS;
  constexpr uint32_t OFF_V = C::TILE_BYTES;
  constexpr uint32_t OFF_QR = 2 * C::TILE_BYTES;                             // Q ring
  constexpr uint32_t QSTAGE = C::TILE_BYTES + (uint32_t)QX_TILE_BYTES;        // Q, statistics block
  constexpr uint32_t OFF_OR = OFF_QR + QS * QSTAGE;                          // dO ring
  constexpr uint32_t OFF_CONST = OFF_OR + OS * C::TILE_BYTES;   // constant A operands: K side, V side
  constexpr uint32_t OFF_EPI = OFF_CONST + 2 * (uint32_t)QX_TILE_BYTES;   // 8 x 1 KB epilogue staging
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[1 + 2 * QS + 2 * OS + 10];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ KvUnit units[MAX_KV_RUN];   // this CTA's units, decoded once
  __shared__ int unit_ok[MAX_KV_RUN];    // 0: the unit does nothing

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar_kv = smem_u32(&bars[0]);
  auto bar_q = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto bar_qfree = [&](int s) { return smem_u32(&bars[1 + QS + s]); };
  auto bar_o = [&](int s) { return smem_u32(&bars[1 + 2 * QS + s]); };
  auto bar_ofree = [&](int s) { return smem_u32(&bars[1 + 2 * QS + OS + s]); };
  constexpr int B0 = 1 + 2 * QS + 2 * OS;
  const uint32_t bar_s = smem_u32(&bars[B0 + 0]);
  const uint32_t bar_dp = smem_u32(&bars[B0 + 1]);
  const uint32_t bar_p = smem_u32(&bars[B0 + 2]);    // P^T of the second 32 columns of each half written
  const uint32_t bar_pa = smem_u32(&bars[B0 + 9]);   // P^T of the first 32 columns of each half written
  const uint32_t bar_ds = smem_u32(&bars[B0 + 3]);
  const uint32_t bar_dv = smem_u32(&bars[B0 + 4]);
  const uint32_t bar_dk = smem_u32(&bars[B0 + 5]);
  const uint32_t bar_done = smem_u32(&bars[B0 + 6]);
  const uint32_t bar_kvfree = smem_u32(&bars[B0 + 7]);   // a unit's K and V are read by no further MMA
  const uint32_t bar_accfree = smem_u32(&bars[B0 + 8]);  // a unit's dV, dK have been read out

  const int64_t u_begin = (int64_t)blockIdx.x * p.kv_run;
  const int run = (int)min((int64_t)p.kv_run, p.kv_units - u_begin);   // units of this CTA: u_begin + j
  const int g = p.Hq / p.Hkv;
  WaitCtx wc{p.wait_limit_ns, p.status, &abort_flag};

  if (warp >= 1 && warp < 4) {   // warps 1-3 decode the run's units, one warp per unit
    for (int j = warp - 1; j < run; j += 3) {
      KvUnit x;
      const bool ok = kv_unit<D>(p, u_begin + j, x);
      if (lane == 0) {
        unit_ok[j] = ok ? 1 : 0;
        if (ok) units[j] = x;
      }
    }
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(bar_q(s), 1);
      mbar_init(bar_qfree(s), 1);
    }
    for (int s = 0; s < OS; ++s) {
      mbar_init(bar_o(s), 1);
      mbar_init(bar_ofree(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 256);
    mbar_init(bar_pa, 256);
    mbar_init(bar_ds, 256);
    mbar_init(bar_dv, 1);
    mbar_init(bar_dk, 1);
    mbar_init(bar_done, 1);
    mbar_init(bar_kvfree, 1);
    mbar_init(bar_accfree, 256);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tdo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp >= 4) {   // the constant A operands of the statistics steps, one row per thread
    const int t = threadIdx.x - 128, row = t & (TILE - 1);
    float ah = 0.f, am = 0.f, al = 0.f;
    const float a = 1.f / p.scale_log2;
    ah = __bfloat162float(__float2bfloat16_rn(a));
    am = __bfloat162float(__float2bfloat16_rn(a - ah));
    al = __bfloat162float(__float2bfloat16_rn(a - ah - am));
    uint8_t* dst = smem + OFF_CONST + (t >= TILE ? QX_TILE_BYTES : 0) + row * 16;
    const uint32_t one2 = pack_bf16(1.f, 1.f);
    if (t < TILE) {   // S^T: (ah + am + al) times each of the three lse2 terms
      *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16(ah, ah), pack_bf16(ah, am), pack_bf16(am, am),
                                                  pack_bf16(al, al));
      *reinterpret_cast<uint4*>(dst + QX_TILE_BYTES / 2) = make_uint4(pack_bf16(al, 0.f), 0u, 0u, 0u);
    } else {          // dP^T: ones under the three D terms
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dst + QX_TILE_BYTES / 2) = make_uint4(pack_bf16(0.f, 1.f), one2, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp < 4) {
   reg_dealloc<C::REGS_CTRL>();
   if (warp == 0) {
    // ---------------------------------------------------------- producer
    // one lane per TMA copy (copies issued by one thread are serialised)
    int n = 0;    // query tiles whose Q (with its statistics block) was loaded, over all units
    int no = 0;   // query tiles whose dO was loaded
    int uc = 0;   // units whose K and V were loaded
    bool ok = true;
    for (int ju = 0; ju < run && ok; ++ju) {
      if (!unit_ok[ju]) continue;
      const KvUnit x = units[ju];   // in registers: asm with memory clobbers would force reloads
      const int64_t u = u_begin + ju;
      // K, V go into the same slots as the previous unit's: wait until its
      // last S^T and dP^T products have read them
      if (uc > 0) ok = wait_bar(bar_kvfree, (uint32_t)(uc - 1) & 1u, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (lane == 0) mbar_arrive_expect_tx(bar_kv, 2 * C::TILE_BYTES);
      __syncwarp();
      const int krow = x.tok0 + x.kt * TILE;
      if (lane < C::NBOX) tma_load_3d(s_base + lane * C::BOX_BYTES, &tk, lane * 64, krow, x.kv_head, bar_kv);
      else if (lane < 2 * C::NBOX)
        tma_load_3d(s_base + OFF_V + (lane - C::NBOX) * C::BOX_BYTES, &tv, (lane - C::NBOX) * 64, krow, x.kv_head,
                    bar_kv);
      ++uc;
      int nu = 0;   // stages of this unit
      for (int h = 0; h < g && ok; ++h) {
        const int hq = x.hkv * g + h;                 // query head within the batch
        const int q_head = p.cu_seqlens != nullptr ? hq : x.b * p.Hq + hq;
        for (int qt = x.qt_first; qt < x.nqt && ok; ++qt) {
          if (!tile_pair_visible(p, qt, x.kt)) continue;
          const size_t roff = (size_t)(x.lrow_b + hq * x.lrow_hs) + (size_t)qt * TILE;
          const int qrow0 = x.tok0 + qt * TILE;
          const int s = n % QS;
          if (n >= QS) ok = wait_bar(bar_qfree(s), ((n / QS) - 1) & 1, wc);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          const uint32_t st = s_base + OFF_QR + s * QSTAGE;
          if (lane == 0) mbar_arrive_expect_tx(bar_q(s), C::TILE_BYTES + (uint32_t)QX_TILE_BYTES);
          __syncwarp();
          if (lane < C::NBOX)
            tma_load_3d(st + lane * C::BOX_BYTES, &tq, lane * 64, qrow0, q_head, bar_q(s));
          else if (lane == C::NBOX)
            bulk_load(st + C::TILE_BYTES, p.qx + roff * QX_ROW_BYTES, (uint32_t)QX_TILE_BYTES, bar_q(s));
          ++n;
          const int so = no % OS;
          if (no >= OS) ok = wait_bar(bar_ofree(so), ((no / OS) - 1) & 1, wc);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          const uint32_t sto = s_base + OFF_OR + so * C::TILE_BYTES;
          if (lane == 0) mbar_arrive_expect_tx(bar_o(so), C::TILE_BYTES);
          __syncwarp();
          if (lane > C::NBOX && lane <= 2 * C::NBOX)   // other lanes than the Q copies'
            tma_load_3d(sto + (lane - C::NBOX - 1) * C::BOX_BYTES, &tdo, (lane - C::NBOX - 1) * 64, qrow0, q_head,
                        bar_o(so));
          ++no;
          ++nu;
        }
      }
      if (p.dkdv_counts != nullptr && lane == 0) {   // the unit's identity and stages in its debug record
        int32_t* rec = p.dkdv_counts + (size_t)DEBUG_FIELDS * u;
        rec[0] = x.bkv;
        rec[1] = x.kt;
        rec[2] = 0;
        rec[3] = x.tok0;
        rec[4] = nu;
      }
    }
    if ((!ok || abort_flag) && lane == 0) {   // drain the copies still in flight
      if (uc > 0) wait_bar(bar_kv, (uint32_t)(uc - 1) & 1u, wc, false);
      for (int j = n - QS < 0 ? 0 : n - QS; j < n; ++j) wait_bar(bar_q(j % QS), (j / QS) & 1, wc, false);
      for (int j = no - OS < 0 ? 0 : no - OS; j < no; ++j) wait_bar(bar_o(j % OS), (j / OS) & 1, wc, false);
    }
   } else if (warp == 1) {
    {
      // every lane waits, so the warp leaves a wait together
      auto wt = [&](uint32_t bar, uint32_t par) { return __all_sync(0xffffffffu, wait_bar(bar, par, wc)); };
      // ---------------------------------------------------------- MMA issuer
      // Order: S^T_0, dP^T_0, then per query tile i: dV_i, S^T_{i+1}, dK_i,
      // dP^T_{i+1}.  S^T_{i+1} overwrites the P^T_i columns dV_i reads and
      // dP^T_{i+1} the dS^T_i columns dK_i reads; each is issued right after
      // that reader (tcgen05.mma from one thread execute in issue order).
      // Each elementwise phase has two MMAs of cover.  The next unit's S^T_0
      // and dP^T_0 follow the last dK the same way.
      // tcgen05.mma issue stalls once a few MMAs are queued, so the issuer
      // is held for most of each group and anything it does between groups
      // idles the tensor pipe: it keeps ring counters only, and descriptors
      // are built once (a k-step adds a compile-time offset to the
      // start-address field; shared-memory addresses stay below 256 KB, so
      // the 14-bit field never carries).  The whole warp runs the loop and
      // elect.sync picks the issuing lane (always the same one while the warp
      // is converged), which feeds the pipe faster than a one-lane loop.
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint32_t id_acc = idesc_bf16(128, D, false, true);
      constexpr uint32_t QSTAGE16 = QSTAGE >> 4, TILE16 = C::TILE_BYTES >> 4;
      const uint32_t hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t d_k = (uint32_t)sdesc_sw128(s_base, 16, 1024);
      const uint32_t d_v = (uint32_t)sdesc_sw128(s_base + OFF_V, 16, 1024);
      const uint32_t d_q = (uint32_t)sdesc_sw128(s_base + OFF_QR, 16, 1024);               // K-major
      const uint32_t d_o = (uint32_t)sdesc_sw128(s_base + OFF_OR, 16, 1024);
      const uint32_t d_q_mn = (uint32_t)sdesc_sw128(s_base + OFF_QR, C::BOX_BYTES, 1024);  // MN-major
      const uint32_t d_o_mn = (uint32_t)sdesc_sw128(s_base + OFF_OR, C::BOX_BYTES, 1024);
      auto desc = [&](uint32_t lo) { return ((uint64_t)hi << 32) | lo; };
      // the statistics steps: plain K-major operands, two 2 KB planes
      const uint32_t hi_x = (uint32_t)(sdesc_plain(0, QX_TILE_BYTES / 2, 128) >> 32);
      const uint32_t d_ck = (uint32_t)sdesc_plain(s_base + OFF_CONST, QX_TILE_BYTES / 2, 128);
      const uint32_t d_cv = (uint32_t)sdesc_plain(s_base + OFF_CONST + QX_TILE_BYTES, QX_TILE_BYTES / 2, 128);
      const uint32_t d_qx = (uint32_t)sdesc_plain(s_base + OFF_QR + C::TILE_BYTES, QX_TILE_BYTES / 2, 128);
      auto desc_x = [&](uint32_t lo) { return ((uint64_t)hi_x << 32) | lo; };
      auto kstep = [](int kk) { return (uint32_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4); };
      auto issue_st = [&](int qslot) {   // S^T = K Q^T
        const uint32_t qd = d_q + (uint32_t)qslot * QSTAGE16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss_e(tmem + 0, desc(d_k + kstep(kk)), desc(qd + kstep(kk)), id_s, kk > 0);
        mma_ss_e(tmem + 0, desc_x(d_ck), desc_x(d_qx + (uint32_t)qslot * QSTAGE16), id_s, 1u);   // - lse2 / c
        mma_commit_e(bar_s);
      };
      auto issue_dpt = [&](int oslot, int qslot) {  // dP^T = V dO^T
        const uint32_t dd = d_o + (uint32_t)oslot * TILE16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_e(tmem + 128, desc(d_v + kstep(kk)), desc(dd + kstep(kk)), id_s, kk > 0);
        mma_ss_e(tmem + 128, desc_x(d_cv), desc_x(d_qx + (uint32_t)qslot * QSTAGE16), id_s, 1u);   // - D
        mma_commit_e(bar_dp);
      };
      // ring slots of the next query tile and the parities of their fills
      int s = 0, so = 0;
      uint32_t spar = 0, sopar = 0;
      int itot = 0;        // query tiles whose dV and dK products were issued, over all units
      int uc = 0;          // units started
      bool ok = true;
      for (int ju = 0; ju < run && ok; ++ju) {
        if (!unit_ok[ju]) continue;
        const int ntile = units[ju].ntile;   // (query head, query tile) pairs, in the producer's order
        if (!(ok = wt(bar_kv, (uint32_t)uc & 1u))) break;
        if (ntile > 0) {
          if (!(ok = wt(bar_q(s), spar))) break;
          tc_fence_after();
          issue_st(s);
          if (!(ok = wt(bar_o(so), sopar))) break;
          tc_fence_after();
          issue_dpt(so, s);
        }
        if (ntile <= 1) mma_commit_e(bar_kvfree);   // no later S^T or dP^T reads this unit's K and V
        int i = 0;   // after the loop: query tiles of this unit whose dV and dK products were issued
        for (; i < ntile; ++i) {
          const bool more = i + 1 < ntile;
          const int sn = (s + 1 == QS) ? 0 : s + 1;
          const uint32_t snpar = (s + 1 == QS) ? spar ^ 1u : spar;
          const int son = (so + 1 == OS) ? 0 : so + 1;
          const uint32_t sonpar = (so + 1 == OS) ? sopar ^ 1u : sopar;
          const uint32_t par = (uint32_t)itot & 1u;
          const uint32_t mq = d_q_mn + (uint32_t)s * QSTAGE16, mo = d_o_mn + (uint32_t)so * TILE16;
          // dV += P^T dO   (dO as an MN-major operand: N = d, K = query rows),
          // in the order phase A hands P^T over: first the k-steps of the
          // first 32 query columns of each half (0, 1, 4, 5), while the
          // elementwise warps still compute the rest, then 2, 3, 6, 7.  The
          // first dV of a unit overwrites the accumulator the previous unit's
          // epilogue reads
          if (!(ok = wt(bar_pa, par))) break;
          if (i == 0 && uc > 0 && !(ok = wt(bar_accfree, (uint32_t)(uc - 1) & 1u))) break;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = (q & 1) + 4 * (q >> 1);
            mma_ts_e(tmem + 256, tmem + half_col(kk), desc(mo + (uint32_t)kk * (2048 >> 4)), id_acc, (i > 0 || q > 0));
          }
          if (!(ok = wt(bar_p, par))) break;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 2 + (q & 1) + 4 * (q >> 1);
            mma_ts_e(tmem + 256, tmem + half_col(kk), desc(mo + (uint32_t)kk * (2048 >> 4)), id_acc, 1u);
          }
          mma_commit_e(bar_dv);
          mma_commit_e(bar_ofree(so));   // dP^T_i and dV_i have read dO_i
          if (more) {
            if (!(ok = wt(bar_q(sn), snpar))) break;
            tc_fence_after();
            issue_st(sn);
          }
          // dK += dS^T Q
          if (!(ok = wt(bar_ds, par))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < TILE / 16; ++kk)
            mma_ts_e(tmem + 256 + D, tmem + 128 + half_col(kk), desc(mq + (uint32_t)kk * (2048 >> 4)), id_acc,
                     (i > 0 || kk > 0));
          mma_commit_e(bar_dk);
          mma_commit_e(bar_qfree(s));
          if (more) {
            if (!(ok = wt(bar_o(son), sonpar))) break;
            tc_fence_after();
            issue_dpt(son, sn);
            if (i + 2 == ntile) mma_commit_e(bar_kvfree);   // the unit's last S^T and dP^T are issued
          }
          s = sn;
          spar = snpar;
          so = son;
          sopar = sonpar;
          ++itot;
        }
        if (p.dkdv_counts != nullptr && lane == 0) p.dkdv_counts[(size_t)DEBUG_FIELDS * (u_begin + ju) + 5] = i;
        ++uc;
      }
      mma_commit_e(bar_done);
      wait_bar(bar_done, 0, wc, false);
    }
   }
  } else {
    reg_alloc<C::REGS_ELEM>();
    // ------------------------------------------------------------ elementwise
    // warpgroup hf (0: warps 4-7, 1: warps 8-11) owns query columns
    // [64*hf, 64*hf + 64) of every row; its bf16 results go over the first 32
    // of those columns, which only it has read
    const int hf = (warp - 4) >> 2;
    const int cb = 64 * hf;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                   // key row inside the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t stage = s_base + OFF_EPI + (uint32_t)(warp - 4) * 1024u;
    const float c = p.scale_log2;
    const bool causal = causal_of(p);
    const bool ragged = p.cu_seqlens != nullptr;
    int i = 0;   // query tiles processed, over all units
    bool ok = true;
    for (int ju = 0; ju < run && ok; ++ju) {
      if (!unit_ok[ju]) continue;
      const KvUnit x = units[ju];   // in registers: asm with memory clobbers would force reloads
      const int64_t u = u_begin + ju;
      const int kt = x.kt;
      const int i0 = i;
      for (int h = 0; h < g && ok; ++h) {
        for (int qt = x.qt_first; qt < x.nqt; ++qt) {
          if (!tile_pair_visible(p, qt, kt)) continue;
          ok = wait_bar(bar_s, i & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          // key r sees query column j iff 0 <= base + j - r < window: j >= lo
          // where the causal edge crosses the tile, j < hi where the window's
          // edge does
          const int base = tile_base(p, qt, kt);
          const bool cedge = causal && base < TILE - 1;
          const bool wedge = base + (TILE - 1) >= window_of(p);
          const int hi = wedge ? window_of(p) + r - base : TILE;
          // phase A: P^T = 2^((S^T - lse2/c) c) for this warpgroup's 64 query columns,
          // kept in fp32 for phase B and rounded to bf16 pairs for dV = P^T dO,
          // in two passes of 32 columns, each handed to the tensor core as
          // soon as it is written (its pairs go over the first 16 of the
          // columns it has read).  Masked tiles (the diagonal, a window's
          // edge) take their own copy of the loop so that the others carry no
          // mask arithmetic at all.
          float pf[64];
          const int lo = cedge ? r - base : 0;        // visible query columns: lo <= j < hi
          auto phase_a = [&](auto masked, auto pass) {
            constexpr int G = decltype(pass)::value;
            uint32_t sr[32];
            tmem_ld32(tmem + lane_off + cb + 32 * G, sr);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const int col = cb + 32 * G + 4 * j4;
              float x0, x1, x2, x3;
              mul2(x0, x1, __uint_as_float(sr[4 * j4 + 0]), __uint_as_float(sr[4 * j4 + 1]), c, c);
              mul2(x2, x3, __uint_as_float(sr[4 * j4 + 2]), __uint_as_float(sr[4 * j4 + 3]), c, c);
              float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
              if constexpr (decltype(masked)::value) {
                p0 = (col + 0 >= lo && col + 0 < hi) ? p0 : 0.f;
                p1 = (col + 1 >= lo && col + 1 < hi) ? p1 : 0.f;
                p2 = (col + 2 >= lo && col + 2 < hi) ? p2 : 0.f;
                p3 = (col + 3 >= lo && col + 3 < hi) ? p3 : 0.f;
              }
              pf[32 * G + 4 * j4 + 0] = p0;
              pf[32 * G + 4 * j4 + 1] = p1;
              pf[32 * G + 4 * j4 + 2] = p2;
              pf[32 * G + 4 * j4 + 3] = p3;
            }
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(pf[32 * G + 2 * j], pf[32 * G + 2 * j + 1]);
            tmem_st16(tmem + lane_off + cb + 16 * G, pk);
            tc_fence_before();
            mbar_arrive(G == 0 ? bar_pa : bar_p);
          };
          if (cedge || wedge) {
            phase_a(std::true_type{}, std::integral_constant<int, 0>{});
            phase_a(std::true_type{}, std::integral_constant<int, 1>{});
          } else {
            phase_a(std::false_type{}, std::integral_constant<int, 0>{});
            phase_a(std::false_type{}, std::integral_constant<int, 1>{});
          }
          ok = wait_bar(bar_dp, i & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          // phase B: dS^T = P^T * (dP^T - D) for the same 64 columns (the
          // accumulator holds dP^T - D); the bf16 pairs go over the first 32
          // dP^T columns of the half
          {
            uint32_t dr[64];
            tmem_ld64(tmem + lane_off + 128 + cb, dr);
            uint32_t ds[32];
#pragma unroll
            for (int j4 = 0; j4 < 16; ++j4) {
              float d0, d1, d2, d3;
              mul2(d0, d1, pf[4 * j4 + 0], pf[4 * j4 + 1], __uint_as_float(dr[4 * j4 + 0]), __uint_as_float(dr[4 * j4 + 1]));
              mul2(d2, d3, pf[4 * j4 + 2], pf[4 * j4 + 3], __uint_as_float(dr[4 * j4 + 2]), __uint_as_float(dr[4 * j4 + 3]));
              ds[2 * j4] = pack_bf16(d0, d1);
              ds[2 * j4 + 1] = pack_bf16(d2, d3);
            }
            tmem_st32(tmem + lane_off + 128 + cb, ds);
          }
          tc_fence_before();
          mbar_arrive(bar_ds);
          ++i;
        }
      }
      const int nt = i - i0;   // query tiles of this unit
      if (p.dkdv_counts != nullptr && r == 0) p.dkdv_counts[(size_t)DEBUG_FIELDS * u + 6 + hf] = nt;
      if (!ok || abort_flag) break;
      // ---------------------------------------------------------- epilogue
      // warpgroup 0 writes dV, warpgroup 1 writes scale * dK, each row
      // through this warp's 1 KB of staging so that every store instruction
      // covers 32-byte pieces of 16 rows
      if (nt > 0) {
        ok = wait_bar(bar_dv, (uint32_t)(i - 1) & 1u, wc) && wait_bar(bar_dk, (uint32_t)(i - 1) & 1u, wc);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
      }
      const float mul = hf == 0 ? 1.f : p.scale;
      const int wkey0 = kt * TILE + wq * 32;   // this warp's first key
      const uint32_t acc = tmem + lane_off + 256 + hf * D;
      if constexpr (F32) {
        // float32 rows, 16 columns at a time (two 32-byte pieces); added
        // (p.accumulate) or stored.  With no visible query tile an add has
        // nothing to contribute and a store writes zeros.
        char* base = reinterpret_cast<char*>(static_cast<float*>(hf == 0 ? p.dv : p.dk) +
                                             ((size_t)x.bkv * p.dkv_hs + wkey0) * D);
        if (nt > 0 || !p.accumulate) {
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {
            uint32_t rv[16];
            if (nt > 0) {
              tmem_ld16(acc + q * 16, rv);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) rv[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) rv[j] = __float_as_uint(__uint_as_float(rv[j]) * mul);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              if (p.accumulate)
                warp_store_rows<2, true>(stage, rv + 8 * hh, base + q * 64 + hh * 32, (size_t)D * 4, x.n_seq - wkey0);
              else
                warp_store_rows<2>(stage, rv + 8 * hh, base + q * 64 + hh * 32, (size_t)D * 4, x.n_seq - wkey0);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar_accfree);   // the accumulators have been read
      } else {
        // read all of the row's accumulator columns first (the next unit's
        // first dV product waits for them), then store 32 bytes of each row
        // per round from registers
        uint32_t w[D / 2];
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t rv[32];
          if (nt > 0) {
            tmem_ld32(acc + q4 * 32, rv);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) rv[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[q4 * 16 + j] = pack_bf16(__uint_as_float(rv[2 * j]) * mul, __uint_as_float(rv[2 * j + 1]) * mul);
        }
        tc_fence_before();
        mbar_arrive(bar_accfree);   // the accumulators have been read
        const size_t orow0 = ragged ? (size_t)(x.tok0 + wkey0) * p.Hkv + x.hkv : (size_t)x.bkv * p.dkv_hs + wkey0;
        char* base = reinterpret_cast<char*>(static_cast<__nv_bfloat16*>(hf == 0 ? p.dv : p.dk) + orow0 * D);
        const size_t stride = (ragged ? (size_t)p.Hkv : (size_t)1) * D * sizeof(__nv_bfloat16);
#pragma unroll
        for (int q = 0; q < D / 16; ++q) warp_store_rows<2>(stage, w + 8 * q, base + q * 32, stride, x.n_seq - wkey0);
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

// =========================================================================
// dQ
// Tensor memory: S [0,128), dP [128,256), dQ [256,256+d), two bf16 dS buffers
// [384,448) and [448,512): dS_j goes to buffer j % 2, so writing dS_{j+1} does
// not wait for dQ_j (the MMA issuer queues dQ_j behind S_{j+1} and dP_{j+1}).
// Shared memory: Q, dO (resident), a KS-deep ring of K_j and a VS-deep ring of
// V_j.  K_j is read by S_j and dQ_j, V_j only by dP_j, so the V slots come
// free much earlier and the K ring is the deeper one.
// Tensor-core order: S_0, dP_0, then per key tile j: S_{j+1} (as soon as S_j
// has been read out of TMEM), dP_{j+1} (as soon as dP_j has been read), dQ_j
// (once dS_j is written to its buffer).
// =========================================================================
template <int D>
struct DqCfg {
  static constexpr int KS = (D == 128) ? 3 : 6;
  static constexpr int VS = (D == 128) ? 2 : 4;
  static constexpr uint32_t TILE_BYTES = BwdCfg<D>::TILE_BYTES;
  static constexpr uint32_t OFF_DO = TILE_BYTES;
  static constexpr uint32_t OFF_K = 2 * TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KS * TILE_BYTES;
  static constexpr uint32_t SMEM = OFF_V + VS * TILE_BYTES + 1024;
  // two producers and the ragged-batch bookkeeping need more than 56 registers
  // in the control warps: 128*72 + 256*216 <= 384*168
  static constexpr uint32_t REGS_CTRL = 72, REGS_ELEM = 216;
};

template <int D, bool F32>
__global__ void __launch_bounds__(BwdCfg<D>::SPLIT_THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
              const BwdParams p) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  constexpr int KS = Q::KS, VS = Q::VS;
  static_assert(KS >= 2 && VS >= 2, "the issuer's ring counters start at slot 1");
  constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256, T_DS = 384;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[1 + 2 * KS + 2 * VS + 9];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar_qdo = smem_u32(&bars[0]);
  auto bar_k = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto bar_kfree = [&](int s) { return smem_u32(&bars[1 + KS + s]); };
  auto bar_v = [&](int s) { return smem_u32(&bars[1 + 2 * KS + s]); };
  auto bar_vfree = [&](int s) { return smem_u32(&bars[1 + 2 * KS + VS + s]); };
  const uint32_t bar_s = smem_u32(&bars[1 + 2 * KS + 2 * VS + 0]);
  const uint32_t bar_dp = smem_u32(&bars[1 + 2 * KS + 2 * VS + 1]);
  const uint32_t bar_sfree = smem_u32(&bars[1 + 2 * KS + 2 * VS + 2]);
  const uint32_t bar_done = smem_u32(&bars[1 + 2 * KS + 2 * VS + 3]);
  const uint32_t bar_dpread = smem_u32(&bars[1 + 2 * KS + 2 * VS + 4]);
  // per dS buffer: dS_j written (256 arrivals), dQ_j done (its buffer is free)
  auto bar_ds = [&](int j) { return smem_u32(&bars[1 + 2 * KS + 2 * VS + 5 + (j & 1)]); };
  auto bar_dq = [&](int j) { return smem_u32(&bars[1 + 2 * KS + 2 * VS + 7 + (j & 1)]); };

  const bool ragged = p.cu_seqlens != nullptr;
  int bh = 0, qt = 0;
  if (ragged) {   // sequence by sequence; inside one, head groups sized for L2, latest query tiles first
    int sb = 0, nt = 0;
    int64_t j = 0;
    if (!ragged_tile_unit(p.pcu, p.B, p.Hq, blockIdx.x, &sb, &nt, &j)) return;
    const int len = p.cu_seqlens[sb + 1] - p.cu_seqlens[sb];
    int h = 0, qpos = 0;
    grouped_unit(j, p.Hq, nt, kv_stream_group(1, p.Hq, p.Hkv, len, D), &h, &qpos);
    bh = sb * p.Hq + h;
    qt = nt - 1 - qpos;
  } else {
    const int nqt_all = (p.Nq + TILE - 1) / TILE;
    int qpos = 0;
    grouped_unit(blockIdx.x, p.B * p.Hq, nqt_all, p.q_group, &bh, &qpos);
    qt = nqt_all - 1 - qpos;  // latest query tile first: heaviest under a causal mask
  }
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  if (ragged && !seq_range_ok(p.cu_seqlens, b, p.total, p.Nq)) {   // malformed: skipped and reported
    if (threadIdx.x == 0) atomicOr(p.status, ATTN_DEV_BOUNDS);
    return;
  }
  const int tok0 = ragged ? p.cu_seqlens[b] : 0;    // packed tensors hold fewer than 2^31 tokens
  const int n_seq = ragged ? p.cu_seqlens[b + 1] - tok0 : p.Nq;   // query rows of the unit's sequence
  const int nk_seq = ragged ? n_seq : p.Nk;                       // and its keys
  if (qt * TILE >= n_seq) return;   // past the end of a shorter sequence; nothing is set up yet
  const int q_head = ragged ? h : bh, kv_head = ragged ? h / (p.Hq / p.Hkv) : bkv;   // heads in the maps
  const int nkt = (nk_seq + TILE - 1) / TILE;
  const int kt_end = causal_of(p) ? key_tile_end(p, qt, nkt) : nkt;
  WaitCtx wc{p.wait_limit_ns, p.status, &abort_flag};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_qdo, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_kfree(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar_v(s), 1);
      mbar_init(bar_vfree(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_sfree, 256);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_ds(t), 256);
      mbar_init(bar_dq(t), 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_dpread, 256);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tdo);
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
   reg_dealloc<Q::REGS_CTRL>();
   if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------- producers
    // warp 0 streams K (and loads Q, dO once), warp 2 streams V: a K slot is
    // only free once dQ_j has run, a V slot once dP_j has, so the V stream
    // must not wait behind the K stream.  One lane per TMA copy (copies
    // issued by one thread are serialised).
    const bool is_k = warp == 0;
    if (is_k) {
      if (lane == 0) mbar_arrive_expect_tx(bar_qdo, 2 * C::TILE_BYTES);
      __syncwarp();
      const int qrow0 = tok0 + qt * TILE;
      if (lane < C::NBOX) tma_load_3d(s_base + lane * C::BOX_BYTES, &tq, lane * 64, qrow0, q_head, bar_qdo);
      else if (lane < 2 * C::NBOX)
        tma_load_3d(s_base + Q::OFF_DO + (lane - C::NBOX) * C::BOX_BYTES, &tdo, (lane - C::NBOX) * 64, qrow0, q_head,
                    bar_qdo);
    }
    const int depth = is_k ? KS : VS;
    const uint32_t ring = s_base + (is_k ? Q::OFF_K : Q::OFF_V);
    const CUtensorMap* map = is_k ? &tk : &tv;
    auto full = [&](int sl) { return is_k ? bar_k(sl) : bar_v(sl); };
    auto freed = [&](int sl) { return is_k ? bar_kfree(sl) : bar_vfree(sl); };
    int n = 0;
    bool ok = true;
    for (int kt = 0; kt < kt_end && ok; ++kt) {
      if (!tile_pair_visible(p, qt, kt)) continue;
      const int sl = n % depth;
      if (n >= depth) ok = wait_bar(freed(sl), ((n / depth) - 1) & 1, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (lane == 0) mbar_arrive_expect_tx(full(sl), C::TILE_BYTES);
      __syncwarp();
      if (lane < C::NBOX)
        tma_load_3d(ring + sl * C::TILE_BYTES + lane * C::BOX_BYTES, map, lane * 64, tok0 + kt * TILE, kv_head,
                    full(sl));
      ++n;
    }
    if (is_k && p.dq_counts != nullptr && lane == 0) p.dq_counts[(size_t)DEBUG_FIELDS * blockIdx.x + 4] = n;   // key tiles loaded
    if ((!ok || abort_flag) && lane == 0) {
      if (is_k) wait_bar(bar_qdo, 0, wc, false);
      for (int j = n - depth < 0 ? 0 : n - depth; j < n; ++j) wait_bar(full(j % depth), (j / depth) & 1, wc, false);
    }
   } else if (warp == 1) {
    {
      // every lane waits, so the warp leaves a wait together
      auto wt = [&](uint32_t bar, uint32_t par) { return __all_sync(0xffffffffu, wait_bar(bar, par, wc)); };
      // ---------------------------------------------------------- MMA issuer
      // tcgen05.mma issue stalls once a few MMAs are queued, so the issuer
      // is held for most of each 8-MMA group; whatever it does between groups
      // leaves the tensor pipe idle.  The loop therefore keeps no more than
      // ring counters: descriptors are built once and each k-step adds a
      // compile-time offset to the start-address field (shared-memory
      // addresses stay below 256 KB, so the 14-bit field never carries).
      // The whole warp runs the loop and elect.sync picks the issuing lane
      // (always the same one while the warp is converged).
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint32_t id_dq = idesc_bf16(128, D, false, true);
      // the upper descriptor word (stride offset, version, swizzle) is the
      // same for every operand here; only the lower word moves
      constexpr uint32_t SLOT = C::TILE_BYTES >> 4;
      const uint32_t hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t d_q = (uint32_t)sdesc_sw128(s_base, 16, 1024);
      const uint32_t d_do = (uint32_t)sdesc_sw128(s_base + Q::OFF_DO, 16, 1024);
      const uint32_t d_k = (uint32_t)sdesc_sw128(s_base + Q::OFF_K, 16, 1024);               // K-major (S)
      const uint32_t d_kmn = (uint32_t)sdesc_sw128(s_base + Q::OFF_K, C::BOX_BYTES, 1024);   // MN-major (dQ)
      const uint32_t d_v = (uint32_t)sdesc_sw128(s_base + Q::OFF_V, 16, 1024);
      auto desc = [&](uint32_t lo) { return ((uint64_t)hi << 32) | lo; };
      auto kstep = [](int kk) { return (uint32_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4); };
      auto issue_s = [&](int slot) {   // S = Q K^T
        const uint32_t kd = d_k + (uint32_t)slot * SLOT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss_e(tmem + T_S, desc(d_q + kstep(kk)), desc(kd + kstep(kk)), id_s, kk > 0);
        mma_commit_e(bar_s);
      };
      auto issue_dp = [&](int slot) {  // dP = dO V^T; the V slot is free once it completes
        const uint32_t vd = d_v + (uint32_t)slot * SLOT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_e(tmem + T_DP, desc(d_do + kstep(kk)), desc(vd + kstep(kk)), id_s, kk > 0);
        mma_commit_e(bar_dp);
        mma_commit_e(bar_vfree(slot));
      };
      int nvis = 0;
      for (int kt = 0; kt < kt_end; ++kt) nvis += tile_pair_visible(p, qt, kt) ? 1 : 0;
      // ring positions: K_{j+1} / V_{j+1} (next S / dP) and K_j (dQ)
      int ks = 0, kpar = 0, vs = 0, vpar = 0, kq = 0;
      bool ok = wt(bar_qdo, 0);
      if (ok && nvis > 0) {
        ok = wt(bar_k(0), 0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          ok = wt(bar_v(0), 0);
        }
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
        ks = vs = 1;
      }
      int j = 0;   // after the loop: key tiles whose dQ product was issued
      for (; ok && j < nvis; ++j) {
        const uint32_t par = (uint32_t)j & 1u;
        if (j + 1 < nvis) {
          // S_{j+1} once S_j has been read out of TMEM
          if (!(ok = wt(bar_k(ks), kpar) && wt(bar_sfree, par))) break;
          tc_fence_after();
          issue_s(ks);
          if (++ks == KS) { ks = 0; kpar ^= 1; }
          // dP_{j+1} as soon as dP_j has been read out of TMEM
          if (!(ok = wt(bar_v(vs), vpar) && wt(bar_dpread, par))) break;
          tc_fence_after();
          issue_dp(vs);
          if (++vs == VS) { vs = 0; vpar ^= 1; }
        }
        // dQ_j += dS_j K_j   (K_j as an MN-major operand: N = d, K = keys)
        if (!(ok = wt(bar_ds(j), ((uint32_t)j >> 1) & 1u))) break;
        tc_fence_after();
        const uint32_t kd = d_kmn + (uint32_t)kq * SLOT;
        const uint32_t ds = tmem + T_DS + (par << 6);
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          mma_ts_e(tmem + T_DQ, ds + kk * 8, desc(kd + (uint32_t)kk * (2048 >> 4)), id_dq, (j > 0 || kk > 0));
        mma_commit_e(bar_dq(j));
        mma_commit_e(bar_kfree(kq));
        if (++kq == KS) kq = 0;
      }
      if (p.dq_counts != nullptr && lane == 0) p.dq_counts[(size_t)DEBUG_FIELDS * blockIdx.x + 5] = j;
      mma_commit_e(bar_done);
      wait_bar(bar_done, 0, wc, false);
    }
   }
  } else {
    reg_alloc<Q::REGS_ELEM>();
    // ------------------------------------------------------------ elementwise
    // warpgroup hf (0: warps 4-7, 1: warps 8-11) owns key columns
    // [64*hf, 64*hf + 64) of every query row
    const int hf = (warp - 4) >> 2;
    const int cb = 64 * hf;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                   // query row inside the tile
    const int qrow = qt * TILE + r;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    const bool causal = causal_of(p);
    const size_t prow = ragged ? (size_t)h * p.pcu[p.B] + p.pcu[b] + qrow : (size_t)bh * p.Np + qrow;
    const float l2 = p.lse2[prow];
    const float dr = p.dsum[prow];
    int j = 0;
    bool ok = true;
    for (int kt = 0; kt < kt_end; ++kt) {
      if (!tile_pair_visible(p, qt, kt)) continue;
      ok = wait_bar(bar_s, j & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // key column col is visible iff the key exists, key <= query (causal:
      // base + r - col >= 0) and query - key < window: lo <= col < lim
      const int wnd = window_of(p);
      const int base = tile_base(p, qt, kt);
      const bool cedge = causal && base < TILE - 1;
      const bool wedge = base + (TILE - 1) >= wnd;
      const bool edge = (kt == nkt - 1 && (nk_seq % TILE) != 0) || cedge || wedge;
      int lim = nk_seq - kt * TILE;
      if (cedge) lim = min(lim, base + r + 1);
      const int lo = wedge ? base + r - wnd + 1 : 0;
      float pr[64];
      {
        uint32_t sr[64];
        tmem_ld64(tmem + lane_off + T_S + cb, sr);
        // S has been read: the next S MMA may overwrite it while P is computed
        tc_fence_before();
        mbar_arrive(bar_sfree);
#pragma unroll
        for (int col = 0; col < 64; col += 2) {
          float x0, x1;
          fma2(x0, x1, __uint_as_float(sr[col]), __uint_as_float(sr[col + 1]), c, c, -l2, -l2);
          pr[col] = ex2(x0);
          pr[col + 1] = ex2(x1);
        }
        if (edge) {
#pragma unroll
          for (int col = 0; col < 64; ++col) pr[col] = (cb + col >= lo && cb + col < lim) ? pr[col] : 0.f;
        }
      }
      // dS_j reuses the buffer of dS_{j-2}: dQ_{j-2} must have read it
      ok = wait_bar(bar_dp, j & 1, wc) && (j < 2 || wait_bar(bar_dq(j), ((j >> 1) - 1) & 1, wc));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t dpr[64];
        tmem_ld64(tmem + lane_off + T_DP + cb, dpr);
        // dP has been read: the next dP MMA may overwrite it while dS is computed
        tc_fence_before();
        mbar_arrive(bar_dpread);
        uint32_t pk[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          // dS = P * (dP - D) = P*dP + (-P*D)
          float a0, a1, d0, d1;
          fma2(a0, a1, pr[2 * jj], pr[2 * jj + 1], -dr, -dr, 0.f, 0.f);
          fma2(d0, d1, pr[2 * jj], pr[2 * jj + 1], __uint_as_float(dpr[2 * jj]), __uint_as_float(dpr[2 * jj + 1]), a0,
               a1);
          pk[jj] = pack_bf16(d0, d1);
        }
        // key columns [64 hf, 64 hf + 64) packed into columns [32 hf, 32 hf + 32) of the buffer
        tmem_st32(tmem + lane_off + T_DS + (j & 1) * 64 + hf * 32, pk);
      }
      tc_fence_before();
      mbar_arrive(bar_ds(j));
      ++j;
    }
    if (p.dq_counts != nullptr && r == 0) {
      int32_t* rec = p.dq_counts + (size_t)DEBUG_FIELDS * blockIdx.x;
      rec[6 + hf] = j;
      if (hf == 0) {   // the unit's identity
        rec[0] = bh;
        rec[1] = qt;
        rec[2] = 0;
        rec[3] = tok0;
      }
    }
    if (ok && !abort_flag) {
      // dQ MMAs complete in issue order: the last one covers them all.  With
      // no key tile the Q and dO copies were still issued, and their memory
      // stages the rows below: wait until they have landed
      if (j > 0) ok = __all_sync(0xffffffffu, wait_bar(bar_dq(j - 1), ((j - 1) >> 1) & 1, wc));
      else ok = __all_sync(0xffffffffu, wait_bar(bar_qdo, 0, wc));
      if (ok) {
        tc_fence_after();
        // each warpgroup writes its half of the dQ rows (D / 2 columns, scaled
        // and rounded to bf16).  At d = 128 the rows are staged through shared
        // memory that no MMA or copy uses any more (the Q tile's), so that the
        // stores cover whole rows (measured 1 % faster there; at d = 64 the
        // direct stores were faster)
        if constexpr (F32) {
          // float32 rows, 32 columns at a time through this warp's 4 KB of
          // staging (the Q and dO tiles' memory); added or stored
          const int wrow0 = qt * TILE + wq * 32;
          float* base = static_cast<float*>(p.dq) + ((size_t)bh * p.dq_hs + wrow0) * D + hf * (D / 2);
          const uint32_t stage = s_base + (uint32_t)(warp - 4) * (32u * 32u * 4u);
          if (j > 0 || !p.accumulate) {
#pragma unroll
            for (int q4 = 0; q4 < D / 64; ++q4) {
              uint32_t rq[32];
              if (j > 0) {
                tmem_ld32(tmem + lane_off + T_DQ + hf * (D / 2) + q4 * 32, rq);
              } else {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) rq[jj] = 0u;
              }
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) rq[jj] = __float_as_uint(__uint_as_float(rq[jj]) * p.scale);
              char* dst = reinterpret_cast<char*>(base + q4 * 32);
              if (p.accumulate) warp_store_rows<8, true>(stage, rq, dst, (size_t)D * 4, n_seq - wrow0);
              else warp_store_rows<8>(stage, rq, dst, (size_t)D * 4, n_seq - wrow0);
            }
          }
        } else {
        uint32_t w[D / 4];
#pragma unroll
        for (int q4 = 0; q4 < D / 64; ++q4) {
          uint32_t rq[32];
          if (j > 0) {
            tmem_ld32(tmem + lane_off + T_DQ + hf * (D / 2) + q4 * 32, rq);
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) rq[jj] = 0u;
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            w[q4 * 16 + jj] = pack_bf16(__uint_as_float(rq[2 * jj]) * p.scale, __uint_as_float(rq[2 * jj + 1]) * p.scale);
        }
        const size_t stride = (ragged ? (size_t)p.Hq : (size_t)1) * D * sizeof(__nv_bfloat16);
        if constexpr (D == 128) {
          const int wrow0 = qt * TILE + wq * 32;   // this warp's first query row
          const size_t qo0 = ragged ? (size_t)(tok0 + wrow0) * p.Hq + h : (size_t)bh * p.dq_hs + wrow0;
          char* base = reinterpret_cast<char*>(static_cast<__nv_bfloat16*>(p.dq) + qo0 * D + hf * (D / 2));
          warp_store_rows<D / 16>(s_base + (uint32_t)(warp - 4) * (32u * D), w, base, stride, n_seq - wrow0);
        } else if (qrow < n_seq) {
          const size_t qo = ragged ? (size_t)(tok0 + qrow) * p.Hq + h : (size_t)bh * p.dq_hs + qrow;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + qo * D + hf * (D / 2));
#pragma unroll
          for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
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

template <int D>
constexpr uint32_t dkdv_smem() {   // K, V, the ring, the constant operands, 8 x 1 KB of epilogue staging, alignment
  return 2 * BwdCfg<D>::TILE_BYTES + BwdCfg<D>::QS * (BwdCfg<D>::TILE_BYTES + (uint32_t)QX_TILE_BYTES) +
         BwdCfg<D>::OS * BwdCfg<D>::TILE_BYTES + 2 * (uint32_t)QX_TILE_BYTES + 8 * 1024 + 1024;
}
template <int D, bool F32>
cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, cudaStream_t s) {
  constexpr uint32_t smem = dkdv_smem<D>();
  static_assert(smem <= 232448 - 256, "dK/dV shared memory");
  cudaError_t e = cudaFuncSetAttribute(dkdv_kernel<D, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = dkdv_grid(p);
  dkdv_kernel<D, F32><<<grid, BwdCfg<D>::SPLIT_THREADS, smem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

template <int D, bool F32>
cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const BwdParams& p, cudaStream_t s) {
  constexpr uint32_t smem = DqCfg<D>::SMEM;
  static_assert(smem <= 232448 - 256, "dQ shared memory");
  static_assert(8 * 32 * 32 * 4 <= 2 * BwdCfg<D>::TILE_BYTES, "f32 epilogue staging fits in the Q and dO tiles");
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = dq_grid(p);
  dq_kernel<D, F32><<<grid, BwdCfg<D>::SPLIT_THREADS, smem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, cudaStream_t s) {
  if (d == 128)
    return out_f32 ? launch_dkdv_t<128, true>(tq, tk, tv, tdo, p, s) : launch_dkdv_t<128, false>(tq, tk, tv, tdo, p, s);
  return out_f32 ? launch_dkdv_t<64, true>(tq, tk, tv, tdo, p, s) : launch_dkdv_t<64, false>(tq, tk, tv, tdo, p, s);
}

cudaError_t launch_bwd_dq(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, cudaStream_t s) {
  if (d == 128)
    return out_f32 ? launch_dq_t<128, true>(tq, tk, tv, tdo, p, s) : launch_dq_t<128, false>(tq, tk, tv, tdo, p, s);
  return out_f32 ? launch_dq_t<64, true>(tq, tk, tv, tdo, p, s) : launch_dq_t<64, false>(tq, tk, tv, tdo, p, s);
}

}  // namespace attn
