// schedule.h -- work-unit bookkeeping shared by the kernels (device) and by
// attn_build_schedule (host), so the exported schedule is the one the kernels
// follow.
//
// A forward work unit is 256 query rows (two 128-row tiles) of one
// (batch, query head).  Units are taken heaviest first: unit i covers query
// chunk nqc-1 - i/(B*Hq) of head i%(B*Hq).  Under a causal mask later chunks
// see more key tiles, so this is a longest-processing-time-first list that the
// hardware block scheduler hands greedily to free SMs ("DISTFLASHATTN"
// reviews, first review point 1: with causal masking, careless placement of
// the chunks leaves processors idle; "FlashAttention-2" reviews, fourth
// review: fully masked blocks are skipped).
#pragma once

#include <stdint.h>

#include "internal.h"

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

struct Unit {
  int bh, kvh;
  int row0;         // first local query row of the unit
  int nkt;          // key tiles in the call
  int lim[2];       // per query tile t: key tiles [0, lim[t]) may be visible
  int kt_end;       // max(lim)
  const uint8_t* mrow[2];  // block-sparse mask row per tile, or null
};

// Key tiles [0, n) hold a key visible to local query row `last_row` under the
// causal rule kv_offset + j <= q_offset + i.
ATTN_HD int causal_tiles(int64_t last_row, int64_t q_off, int64_t kv_off, int nkt) {
  const int64_t last_pos = q_off + last_row;
  if (last_pos < kv_off) return 0;
  const int64_t n = (last_pos - kv_off) / TILE + 1;
  return n < nkt ? (int)n : nkt;
}

ATTN_HD bool mask_is_causal(int kind, int causal_in_blocks) {
  return kind == MASK_CAUSAL || (kind == MASK_BLOCK_SPARSE && causal_in_blocks);
}

// `block_mask` may be a host or a device pointer, matching the caller.
ATTN_HD Unit fwd_unit(int64_t i, int B, int Hq, int Hkv, int Nq, int Nk, int nqc, int mask_kind,
                      int causal_in_blocks, const uint8_t* block_mask, int nkb, int64_t q_off,
                      int64_t kv_off) {
  Unit u;
  const int64_t BH = (int64_t)B * Hq;
  const int qc = nqc - 1 - (int)(i / BH);
  u.bh = (int)(i % BH);
  const int b = u.bh / Hq, h = u.bh % Hq;
  u.kvh = b * Hkv + h / (Hq / Hkv);
  u.row0 = qc * UNIT_ROWS;
  u.nkt = (Nk + TILE - 1) / TILE;
  const bool causal = mask_is_causal(mask_kind, causal_in_blocks);
  u.kt_end = 0;
  for (int t = 0; t < 2; ++t) {
    const int r0 = u.row0 + t * TILE;
    int lim = 0;
    if (r0 < Nq) {
      const int rl = (Nq < r0 + TILE ? Nq : r0 + TILE) - 1;
      lim = causal ? causal_tiles(rl, q_off, kv_off, u.nkt) : u.nkt;
    }
    u.lim[t] = lim;
    u.kt_end = u.kt_end > lim ? u.kt_end : lim;
    u.mrow[t] = (mask_kind == MASK_BLOCK_SPARSE && r0 < Nq) ? block_mask + (int64_t)(r0 / TILE) * nkb : nullptr;
  }
  return u;
}

// Bit t set: query tile t of the unit sees key tile kt.
ATTN_HD uint32_t unit_uses(const Unit& u, int kt) {
  uint32_t m = 0;
  if (kt < u.lim[0] && (u.mrow[0] == nullptr || u.mrow[0][kt] != 0)) m |= 1u;
  if (kt < u.lim[1] && (u.mrow[1] == nullptr || u.mrow[1][kt] != 0)) m |= 2u;
  return m;
}

}  // namespace attn
