// internal.h -- parameter blocks and launcher entry points shared between the
// C-ABI front end (api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

constexpr int TILE = 128;       // query-tile rows, key-tile rows, block-mask granularity

// Bits of the device status word (attn_get_status maps them to error codes).
constexpr unsigned int ATTN_DEV_TIMEOUT = 1u;   // a bounded wait ran out
constexpr unsigned int ATTN_DEV_BOUNDS = 2u;    // a device-side index array (cu_seqlens, seq_lens) was out of range
constexpr int UNIT_ROWS = 256;  // query rows per forward work unit (two query tiles)

enum MaskKind : int { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_BLOCK_SPARSE = 2, MASK_SLIDING_WINDOW = 3 };

// Everything a forward launch needs besides the three TMA descriptors.
struct FwdParams {
  void* o;                  // bf16 or f32 output rows, row stride d
  float* lse;               // may be null
  int B, Hq, Hkv, Nq, Nk;
  int nqc;                  // number of 256-row query chunks
  int head_group;           // heads per L2 group (schedule.h)
  float scale_log2;         // scale * log2(e)
  int mask_kind;
  int causal_in_blocks;
  const uint8_t* block_mask;  // [ceil(Nq/128)][ceil(Nk/128)]
  int nkb;                    // ceil(Nk/128)
  int window;                 // sliding window width (MASK_SLIDING_WINDOW)
  int64_t q_offset, kv_offset;
  // split-KV decoding (n_splits > 0): a unit is one (b * Hkv + kv head, split);
  // its query rows are the Hq/Hkv heads x dec_nq positions of that kv head
  // (contiguous in q), and it covers split_tiles key tiles of the cache
  const int* seq_lens;        // device [B] keys per sequence, or null (Nk each)
  int n_splits;
  int split_tiles;
  int dec_nq;                 // query positions per head
  int64_t split_rows;         // output rows between consecutive splits' partials
  int dec_interleave;         // the unit's rows fit one tile: both query tiles take
                              // them, tile t the key tiles kt with kt % 2 == t, and
                              // writes partial 2 * split + t
  // variable-length batches (cu_seqlens != null): q, k, v, o are token-major
  // [total, heads, d]; sequence b holds tokens [cu_seqlens[b], cu_seqlens[b+1])
  const int* cu_seqlens;      // device [B + 1]
  int varlen_nqc;             // 256-row chunks of the longest sequence
  int64_t total;              // tokens in the packed tensors
  // output element strides: O[head h, row r] at h * o_hs + r * o_rs (plus the
  // split offset when decoding), LSE at h * l_hs + r * l_rs
  int64_t o_hs, o_rs, l_hs, l_rs;
  unsigned int* status;
  int64_t wait_limit_ns;
  int32_t* tile_counts;       // per-CTA debug record (DEBUG_FIELDS int32 each), or null
};

// The backward statistics of a call (in its workspace, or the static
// scratch), for `rows` padded query rows: D, then LSE * log2(e) (float32, one
// per row, each array rounded up to 256 bytes), then the dK/dV kernel's
// per-row statistics operand: QX_ROW_BYTES per row in blocks of 128 rows
// (QX_TILE_BYTES, written by the preprocessing kernel, which describes it).
constexpr size_t QX_ROW_BYTES = 32;
constexpr size_t QX_TILE_BYTES = QX_ROW_BYTES * TILE;
struct StatsLayout {
  size_t lse2_off, qx_off, bytes;   // byte offsets from the start, total size
};
constexpr StatsLayout stats_layout(int64_t rows) {
  const size_t arr = ((size_t)rows * sizeof(float) + 255) & ~(size_t)255;
  const size_t qx = ((size_t)rows + TILE - 1) / TILE * QX_TILE_BYTES;
  return {arr, 2 * arr, 2 * arr + ((qx + 255) & ~(size_t)255)};
}

// Backward parameter block (kernels 2 and 3 of attn_bwd and attn_partial_bwd).
struct BwdParams {
  const float* lse2;        // LSE * log2(e), [B*Hq][Np], +inf on padding rows
  const float* dsum;        // D = rowsum(dO*O), [B*Hq][Np], 0 on padding rows
  const uint8_t* qx;        // the statistics operand, QX_ROW_BYTES per lse2 row
  int Np;                   // Nq rounded up to a multiple of 128
  void* dq;                 // bf16 (or f32) [B,Hq,*,d], heads dq_hs rows apart
  void* dk;                 // bf16 (or f32) [B,Hkv,*,d], heads dkv_hs rows apart
  void* dv;                 // likewise
  int B, Hq, Hkv;
  int Nq, Nk;               // query rows and keys per head (both the longest
                            // sequence for ragged batches)
  int delta;                // q_offset - kv_offset: query i and key j are
                            // delta + i - j positions apart
  int64_t dq_hs, dkv_hs;    // rows between heads of dq and of dk / dv
  int accumulate;           // f32 outputs: add into them instead of storing
  float scale;
  float scale_log2;
  int mask_kind;
  int causal_in_blocks;
  const uint8_t* block_mask;
  int nkb;
  int window;               // sliding window width (MASK_SLIDING_WINDOW)
  // variable-length batches (cu_seqlens != null): tensors are token-major
  // [total, heads, d], sequence b holds tokens [cu_seqlens[b], cu_seqlens[b+1])
  // and N is the longest sequence; lse2 / dsum rows of query head h and
  // sequence b start at h * pcu[B] + pcu[b] (sequences padded to whole tiles)
  const int* cu_seqlens;
  const int* pcu;
  int64_t total;            // tokens in the packed tensors
  int kv_group;             // kv heads per L2 group of the dK/dV kernel
  int q_group;              // query heads per L2 group of the dQ kernel
  int64_t kv_units;         // dK/dV work units in launch order (dkdv_units)
  int kv_run;               // consecutive dK/dV units per CTA
  unsigned int* status;
  int64_t wait_limit_ns;
  int32_t* dkdv_counts;     // per-CTA debug records of the two kernels, or null
  int32_t* dq_counts;
};

// Debug record: DEBUG_FIELDS int32 per work unit (the forward and dQ kernels:
// per CTA, [DEBUG_FIELDS * blockIdx.x]; the dK/dV kernel: per unit of its
// launch order) of the launch's record array; the fields of each kernel are
// listed with attn_debug_set_tile_counts in attn.h.
constexpr int DEBUG_FIELDS = 8;

// Grid sizes (one CTA per work unit), shared by the launchers and by the
// front end's check of the debug record's capacity.
// Ragged batches launch at most heads * (ceil(total / rows) + B) units
// (ragged_units_bound in schedule.h, repeated here for the host).
inline unsigned ragged_grid(int B, int heads, int64_t total, int max_len, int rows) {
  const int64_t padded = (int64_t)B * ((max_len + rows - 1) / rows);
  const int64_t tight = (total + rows - 1) / rows + B;
  return (unsigned)((int64_t)heads * (padded < tight ? padded : tight));
}
inline unsigned fwd_grid(const FwdParams& p) {
  return p.n_splits > 0           ? (unsigned)(p.B * p.Hkv) * (unsigned)p.n_splits
         : p.cu_seqlens != nullptr ? ragged_grid(p.B, p.Hq, p.total, p.Nq, UNIT_ROWS)
                                   : (unsigned)(p.B * p.Hq) * (unsigned)p.nqc;
}
inline unsigned dkdv_units(const BwdParams& p) {
  return p.cu_seqlens != nullptr ? ragged_grid(p.B, p.Hkv, p.total, p.Nk, TILE)
                                 : (unsigned)(p.B * p.Hkv) * (unsigned)((p.Nk + TILE - 1) / TILE);
}
// The dK/dV kernel gives each CTA a run of kv_run consecutive units.
inline unsigned dkdv_grid(const BwdParams& p) {
  return (unsigned)((p.kv_units + p.kv_run - 1) / p.kv_run);
}
inline unsigned dq_grid(const BwdParams& p) {
  return p.cu_seqlens != nullptr ? ragged_grid(p.B, p.Hq, p.total, p.Nq, TILE)
                                 : (unsigned)(p.B * p.Hq) * (unsigned)((p.Nq + TILE - 1) / TILE);
}

struct TensorMaps {
  CUtensorMap a, b, c, d;
};

// Encode a bf16 [heads][rows][d] tensor as a 3-D TMA descriptor with
// 128-byte swizzle and a 64 x 128 (columns x rows) box.
int encode_rows_map(CUtensorMap* map, const void* base, int d, int rows, int heads,
                    int64_t head_stride_rows);

cudaError_t launch_fwd(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, cudaStream_t s);

// e4m3 forward (d = 128): Q, K as [heads][rows][128] and V^T as
// [heads][128][Np] byte maps with a 128 x 128 box and 128-byte swizzle.
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const FwdParams& p,
                           float v_descale, cudaStream_t s);
cudaError_t launch_transpose_v_fp8(const void* v, void* vt, int heads, int N, int Np, cudaStream_t s);

cudaError_t launch_merge(const float* const* o_parts, const float* const* lse_parts, int n_parts,
                         void* o_out, bool out_f32, float* lse_out, int rows_per_head, int heads,
                         int d, int64_t out_head_stride, cudaStream_t s);

// Rows of head h of o / dout start at h * in_hs (in rows of d), of lse at h * in_hs.
cudaError_t launch_bwd_preprocess(const void* o, const void* dout, const float* lse, float* dsum, float* lse2,
                                  uint8_t* qx, int64_t heads, int N, int Np, int64_t in_hs, int d, cudaStream_t s);
// Malformed sequences (seq_range_ok in schedule.h) count as empty and set
// the bounds bit of *status.
cudaError_t launch_varlen_pad(const int* cu_seqlens, int B, int64_t total, int max_len, int* pcu,
                              unsigned int* status, cudaStream_t s);
cudaError_t launch_bwd_preprocess_varlen(const void* o, const void* dout, const float* lse, float* dsum, float* lse2,
                                         uint8_t* qx, int heads, int64_t total, const int* cu_seqlens, const int* pcu, int B,
                                         int max_len, int64_t padded_rows_bound, int d, cudaStream_t s);

// out_f32: dq / dk / dv are float32 (stored, or added with p.accumulate).
cudaError_t launch_bwd_dkdv(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                            cudaStream_t s);

cudaError_t launch_bwd_dq(int d, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                          cudaStream_t s);

cudaError_t launch_wait_selftest(unsigned int* status, int64_t limit_ns, cudaStream_t s);

}  // namespace attn
