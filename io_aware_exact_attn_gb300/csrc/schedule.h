// schedule.h -- work-unit bookkeeping shared by the kernels (device) and by
// attn_build_schedule (host), so the exported schedule is the one the kernels
// follow.
//
// A forward work unit is 256 query rows (two 128-row tiles) of one
// (batch, query head).  Within each head-group (see grouped_unit) units are
// taken heaviest first: the latest query chunk of every head of the group,
// then the next latest, and so on.  Under a causal mask later chunks see more
// key tiles, so this is a longest-processing-time-first list that the hardware
// block scheduler hands greedily to free SMs ("DISTFLASHATTN" reviews, first
// review point 1: with causal masking, careless placement of the chunks leaves
// processors idle; "FlashAttention-2" reviews, fourth review: fully masked
// blocks are skipped).
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
  int nk;           // keys the unit's rows may see (Nk, or a cached sequence's length)
  int nkt;          // ceil(nk / 128)
  int split;        // decoding: which split of the key range (0 otherwise)
  int64_t pos0;     // decoding: position of query 0 (nk - dec_nq)
  int nq;           // query rows of the unit's sequence (rows at or past it are not written)
  int64_t seq0;     // variable-length batches: first token of the sequence (0 otherwise)
  bool empty;       // variable-length batches: no rows of this sequence in the unit
  bool bad;         // a device-side index (cu_seqlens, seq_lens) was out of range
  bool alternate;   // decoding: both query tiles hold the same rows, tile t takes
                    // the key tiles kt of its range with kt % 2 == t
  int lo[2], lim[2];  // per query tile t: key tiles [lo[t], lim[t]) may be visible
  int kt_begin, kt_end;  // min(lo), max(lim) over the unit's tiles
  const uint8_t* mrow[2];  // block-sparse mask row per tile, or null
};

// Sequence b of a packed batch is usable iff 0 <= cu[b] <= cu[b+1] <= total and
// it holds at most max_len tokens.  The kernels treat any other sequence as
// empty (so no index derived from it is ever used) and report a bounds error.
ATTN_HD bool seq_range_ok(const int* cu, int b, int64_t total, int max_len) {
  const int a = cu[b], e = cu[b + 1];
  return a >= 0 && e >= a && (int64_t)e <= total && e - a <= max_len;
}

// Key tiles [0, n) hold a key visible to local query row `last_row` under the
// causal rule kv_offset + j <= q_offset + i.
ATTN_HD int causal_tiles(int64_t last_row, int64_t q_off, int64_t kv_off, int nkt) {
  const int64_t last_pos = q_off + last_row;
  if (last_pos < kv_off) return 0;
  const int64_t n = (last_pos - kv_off) / TILE + 1;
  return n < nkt ? (int)n : nkt;
}

// First key tile holding a key inside the window of local query row
// `first_row`: the window of a row reaches back window - 1 positions, so the
// earliest key any row of a tile starting at first_row sees is
// q_offset + first_row - window + 1 (global position).
ATTN_HD int window_first_tile(int64_t first_row, int64_t q_off, int64_t kv_off, int window) {
  const int64_t first_key = q_off + first_row - window + 1 - kv_off;
  return first_key <= 0 ? 0 : (int)(first_key / TILE);
}

// The sliding window includes the causal rule.
ATTN_HD bool mask_is_causal(int kind, int causal_in_blocks) {
  return kind == MASK_CAUSAL || kind == MASK_SLIDING_WINDOW || (kind == MASK_BLOCK_SPARSE && causal_in_blocks);
}

// Work units are taken head-group by head-group so that the operand a group
// streams (K/V for the forward and dQ kernels, Q/dO for dK/dV) stays resident
// in L2 while every unit of the group re-reads it: groups hold as many heads as
// fit in L2_GROUP_BYTES of streamed bf16 operands.
constexpr int64_t L2_GROUP_BYTES = 64ll << 20;

ATTN_HD int clamp_group(int64_t g, int heads) {
  return (int)(g < 1 ? 1 : (g > heads ? heads : g));
}

// Query heads per group for kernels that stream one kv head's K and V
// (forward, dQ): the g query heads of a GQA group share them.
ATTN_HD int kv_stream_group(int B, int Hq, int Hkv, int Nk, int d) {
  const int64_t kv_bytes = 4ll * Nk * d;  // K + V of one kv head, bf16
  return clamp_group((int64_t)(Hq / Hkv) * (L2_GROUP_BYTES / kv_bytes), B * Hq);
}

// Kv heads per group for the dK/dV kernel, which streams Q and dO of the g
// query heads of each kv head.
ATTN_HD int q_stream_group(int B, int Hq, int Hkv, int Nq, int d) {
  const int64_t q_bytes = 4ll * Nq * d * (Hq / Hkv);
  return clamp_group(L2_GROUP_BYTES / q_bytes, B * Hkv);
}

// Unit i of `heads` x `per_head` units in grouped order: head-groups of
// `group` heads (the last may be smaller), inside a group position-major with
// the heads inner.  Returns the head and the position (0 = first taken).
ATTN_HD void grouped_unit(int64_t i, int heads, int per_head, int group, int* head, int* pos) {
  const int64_t full = heads / group;
  const int64_t per_full = (int64_t)group * per_head;
  int64_t grp, j, gs;
  if (i < full * per_full) {
    grp = i / per_full;
    j = i % per_full;
    gs = group;
  } else {
    grp = full;
    j = i - full * per_full;
    gs = heads - full * group;
  }
  *pos = (int)(j / gs);
  *head = (int)(grp * group + j % gs);
}

// `block_mask` may be a host or a device pointer, matching the caller.
ATTN_HD Unit fwd_unit(int64_t i, int B, int Hq, int Hkv, int Nq, int Nk, int nqc, int head_group, int mask_kind,
                      int causal_in_blocks, const uint8_t* block_mask, int nkb, int window, int64_t q_off,
                      int64_t kv_off) {
  Unit u;
  int pos = 0;
  grouped_unit(i, B * Hq, nqc, head_group, &u.bh, &pos);
  const int qc = nqc - 1 - pos;   // heaviest (latest) query chunk first
  const int b = u.bh / Hq, h = u.bh % Hq;
  u.kvh = b * Hkv + h / (Hq / Hkv);
  u.row0 = qc * UNIT_ROWS;
  u.nk = Nk;
  u.nkt = (Nk + TILE - 1) / TILE;
  u.split = 0;
  u.pos0 = 0;
  u.nq = Nq;
  u.seq0 = 0;
  u.empty = false;
  u.bad = false;
  u.alternate = false;
  const bool causal = mask_is_causal(mask_kind, causal_in_blocks);
  u.kt_begin = u.nkt;
  u.kt_end = 0;
  for (int t = 0; t < 2; ++t) {
    const int r0 = u.row0 + t * TILE;
    int lo = 0, lim = 0;
    if (r0 < Nq) {
      const int rl = (Nq < r0 + TILE ? Nq : r0 + TILE) - 1;
      lim = causal ? causal_tiles(rl, q_off, kv_off, u.nkt) : u.nkt;
      if (mask_kind == MASK_SLIDING_WINDOW) lo = window_first_tile(r0, q_off, kv_off, window);
      if (lo > lim) lo = lim;
    }
    u.lo[t] = lo;
    u.lim[t] = lim;
    if (lo < lim) {
      u.kt_begin = u.kt_begin < lo ? u.kt_begin : lo;
      u.kt_end = u.kt_end > lim ? u.kt_end : lim;
    }
    u.mrow[t] = (mask_kind == MASK_BLOCK_SPARSE && r0 < Nq) ? block_mask + (int64_t)(r0 / TILE) * nkb : nullptr;
  }
  if (u.kt_begin > u.kt_end) u.kt_begin = u.kt_end;
  return u;
}

// Split-KV decoding unit i of B * Hkv * n_splits: splits of one kv head are
// adjacent.  The rows are the g = Hq/Hkv heads x nq positions of kv head
// (b, hk), packed in q's own order (head-major), so row r is query position
// r % nq of head hk * g + r / nq.  Key tiles [split * split_tiles, ...) of the
// sequence's len = seq_lens[b] cached keys; a split past the end is empty.
ATTN_HD Unit decode_unit(int64_t i, int B, int Hq, int Hkv, int nq, int Nk, const int* seq_lens, int n_splits,
                         int split_tiles, bool alternate) {
  Unit u;
  u.split = (int)(i % n_splits);
  const int bkv = (int)(i / n_splits);
  const int b = bkv / Hkv;
  u.bh = bkv;
  u.kvh = bkv;
  u.row0 = 0;
  int len = seq_lens != nullptr ? seq_lens[b] : Nk;
  u.bad = len < 0 || len > Nk;   // reported, and clamped into the cache
  len = len < 0 ? 0 : (len > Nk ? Nk : len);
  u.nk = len;
  u.nkt = (len + TILE - 1) / TILE;
  u.pos0 = (int64_t)len - nq;
  const int rows = (Hq / Hkv) * nq;
  u.nq = rows;
  u.seq0 = 0;
  u.empty = false;
  u.alternate = alternate;
  int lo = u.split * split_tiles, lim = lo + split_tiles;
  if (lim > u.nkt) lim = u.nkt;
  if (lo > lim) lo = lim;
  u.kt_begin = lo;
  u.kt_end = lim;
  for (int t = 0; t < 2; ++t) {
    const bool has_rows = alternate || t * TILE < rows;
    u.lo[t] = has_rows ? lo : 0;
    u.lim[t] = has_rows ? lim : 0;
    u.mrow[t] = nullptr;
  }
  return u;
}

// Work units of a ragged batch, in the launch order of every ragged kernel:
// sequence by sequence (index order; a malformed sequence has none), and
// inside a sequence grouped by heads like the dense kernels (grouped_unit,
// groups sized for L2 from the sequence's own length, heaviest tiles first,
// heads inner), so concurrent CTAs share one group's streamed operand in L2.
// Launches cover at most heads * (ceil(total / rows) + B) units (each
// sequence wastes less than one unit per head), capped by the padded count.
ATTN_HD int64_t ragged_units_bound(int B, int heads, int64_t total, int max_len, int rows) {
  const int64_t padded = (int64_t)B * ((max_len + rows - 1) / rows);
  const int64_t tight = (total + rows - 1) / rows + B;
  return (int64_t)heads * (padded < tight ? padded : tight);
}

#if defined(__CUDACC__)
// The sequence that owns ragged unit `cta` when sequence b owns
// heads * ceil(len_b / rows) consecutive units: one warp (all 32 lanes, same
// arguments) scans cu_seqlens.  Returns false past the last unit; *any_bad
// tells whether some sequence was malformed (every call scans them all).
__device__ __forceinline__ bool ragged_locate(const int* cu, int B, int64_t total, int max_len, int heads, int rows,
                                              int64_t cta, int* seq, int64_t* first, bool* any_bad) {
  const int lane = threadIdx.x & 31;
  int64_t carry = 0, f = 0;
  int found = -1;
  bool bad = false;
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    int64_t n = 0;
    if (b < B) {
      if (seq_range_ok(cu, b, total, max_len)) n = (int64_t)heads * ((cu[b + 1] - cu[b] + rows - 1) / rows);
      else bad = true;
    }
    int64_t x = n;   // inclusive scan over the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    const int64_t excl = carry + x - n;
    const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && cta >= excl && cta < excl + n);
    if (hit != 0u && found < 0) {
      const int src = __ffs(hit) - 1;
      found = __shfl_sync(0xffffffffu, b, src);
      f = __shfl_sync(0xffffffffu, excl, src);
    }
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  *any_bad = __any_sync(0xffffffffu, bad) != 0;
  *seq = found;
  *first = f;
  return found >= 0;
}

// Forward unit `cta` of a ragged batch (256-row chunks; see ragged_locate).
// Called by whole warps.  Inside its sequence a unit is an ordinary forward
// unit (local positions, the same masks); bad reports a malformed sequence
// seen by CTA 0's scan.
__device__ __forceinline__ Unit varlen_unit(int64_t cta, int B, int Hq, int Hkv, int d, const int* cu_seqlens,
                                            int64_t total, int max_len, int mask_kind, int window) {
  int b = 0;
  int64_t first = 0;
  bool any_bad = false;
  const bool ok = ragged_locate(cu_seqlens, B, total, max_len, Hq, UNIT_ROWS, cta, &b, &first, &any_bad);
  Unit u;
  u.bad = any_bad && cta == 0;
  if (!ok) {
    u.empty = true;
    return u;
  }
  const int64_t seq0 = cu_seqlens[b];
  const int len = (int)(cu_seqlens[b + 1] - seq0);
  const int nqc = (len + UNIT_ROWS - 1) / UNIT_ROWS;
  int h = 0, pos = 0;
  grouped_unit(cta - first, Hq, nqc, kv_stream_group(1, Hq, Hkv, len, d), &h, &pos);
  const bool bad = u.bad;
  u = fwd_unit(pos, 1, 1, 1, len, len, nqc, 1, mask_kind, 0, nullptr, 0, window, 0, 0);
  u.bh = h;
  u.kvh = h / (Hq / Hkv);
  u.seq0 = seq0;
  u.bad = bad;
  return u;
}
#endif

// Bit t set: query tile t of the unit sees key tile kt.
ATTN_HD uint32_t unit_uses(const Unit& u, int kt) {
  if (u.alternate) return (kt >= u.lo[0] && kt < u.lim[0]) ? (1u << (kt & 1)) : 0u;
  uint32_t m = 0;
  if (kt >= u.lo[0] && kt < u.lim[0] && (u.mrow[0] == nullptr || u.mrow[0][kt] != 0)) m |= 1u;
  if (kt >= u.lo[1] && kt < u.lim[1] && (u.mrow[1] == nullptr || u.mrow[1][kt] != 0)) m |= 2u;
  return m;
}

}  // namespace attn
