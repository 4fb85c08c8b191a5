// merge.cu -- the streaming (HBM-bound) kernels:
//   * log-sum-exp merge of partial attention results over disjoint key sets
//     (BurstAttention author responses: local attention results combined
//     across devices with online-softmax statistics; "DISTFLASHATTN" reviews:
//     attention computed chunk by chunk);
//   * the backward preprocessing D_i = sum_k dO_ik * O_ik;
//   * the bounded-wait self-test kernel.
// Neither streaming kernel touches the tensor cores: each row is read with
// 16-byte, fully coalesced, streaming (evict-first) loads and written once.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

namespace {

constexpr int MAX_PARTS = 64;

struct MergeArgs {
  const float* o[MAX_PARTS];
  const float* lse[MAX_PARTS];
};

// One group of d/4 lanes per row; each lane owns 4 consecutive columns.
// out = sum_c w_c O_c / sum_c w_c with w_c = exp(LSE_c - max_c LSE_c).
template <int D, bool F32>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeArgs a, int n_parts,
                                                    void* __restrict__ o_out, float* __restrict__ lse_out,
                                                    int64_t rows, int rows_per_head, int64_t out_head_stride) {
  constexpr int LPR = D / 4;                 // lanes per row
  constexpr int RPW = 32 / LPR;              // rows per warp
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, col = (lane % LPR) * 4;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t wrow = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; wrow * RPW < rows;
       wrow += warps_total) {
    const int64_t row = wrow * RPW + sub;
    if (row >= rows) continue;
    float mx = -INFINITY;
    for (int c = 0; c < n_parts; ++c) mx = fmaxf(mx, __ldg(a.lse[c] + row));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
      int c = 0;
      for (; c + 4 <= n_parts; c += 4) {
        float4 v[4];
        float w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[j] = __ldcs(reinterpret_cast<const float4*>(a.o[c + j] + row * D + col));
          w[j] = __expf(__ldg(a.lse[c + j] + row) - mx);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc.x = fmaf(w[j], v[j].x, acc.x);
          acc.y = fmaf(w[j], v[j].y, acc.y);
          acc.z = fmaf(w[j], v[j].z, acc.z);
          acc.w = fmaf(w[j], v[j].w, acc.w);
          wsum += w[j];
        }
      }
      for (; c < n_parts; ++c) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(a.o[c] + row * D + col));
        const float w = __expf(__ldg(a.lse[c] + row) - mx);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
        wsum += w;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t head = row / rows_per_head, r = row % rows_per_head;
    const int64_t orow = head * out_head_stride + r;
    if constexpr (F32) {
      __stcs(reinterpret_cast<float4*>(static_cast<float*>(o_out) + orow * D + col),
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    } else {
      uint2 pk;
      pk.x = pack_bf16(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16(acc.z * inv, acc.w * inv);
      __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + orow * D + col), pk);
    }
    if (lse_out != nullptr && (lane % LPR) == 0)
      lse_out[orow] = (wsum > 0.f) ? mx + __logf(wsum) : -INFINITY;
  }
}

// Ragged backward passes pad every sequence to whole 128-row tiles in the
// D / lse2 arrays: pcu[b] = sum over b' < b of len(b') rounded up to a tile,
// pcu[B] their total.  A malformed sequence (seq_range_ok) counts as empty, so
// pcu[B] never exceeds total + 127 B (the workspace's size), and is reported.
// One warp, 32 sequences per step.
__global__ void __launch_bounds__(32) varlen_pad_kernel(const int* __restrict__ cu, int B, int64_t total,
                                                        int max_len, int* __restrict__ pcu,
                                                        unsigned int* __restrict__ status) {
  const int lane = threadIdx.x;
  int carry = 0;
  for (int base = 0; base <= B; base += 32) {
    const int b = base + lane;
    int v = 0;
    if (b < B) {
      if (seq_range_ok(cu, b, total, max_len)) {
        const int len = cu[b + 1] - cu[b];
        v = len > 0 ? (len + TILE - 1) / TILE * TILE : 0;
      } else {
        atomicOr(status, ATTN_DEV_BOUNDS);
      }
    }
    int x = v;   // inclusive scan over the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (b <= B) pcu[b] = carry + x - v;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
}

// D_i = sum_k dO_ik * O_ik and lse2_i = LSE_i * log2(e) for the backward
// kernels; groups of d/8 lanes per row, 8 bf16 per lane.  Both outputs are
// [heads][Np] with Np = N rounded up to a whole tile; rows past N (and rows
// whose LSE is -inf, i.e. that saw no key) get D = 0 and lse2 = +inf, which
// makes every recomputed probability of such a row exactly 0.
//
// qx: the same two statistics as one 16-element bf16 row per query row i,
// the B operand of one extra K = 16 step of the dK/dV kernel's S^T and dP^T
// products.  With l = -lse2_i (-2^100 in place of -inf) and e = -D_i, each
// split into three bf16 terms whose sum is the float32 value to about 2^-24
// relative (x = x_h + x_m + x_l, each term the rounding of what the earlier
// ones leave), the row is
//   [l_h l_m l_l  l_h l_m l_l  l_h l_m l_l  e_h e_m e_l  0 0 0 0].
// Against the kernel's constant A rows (the split of 1/c, c = scale*log2 e,
// under the first nine columns; ones under the next three) the extra step
// adds l / c to S^T and -D to dP^T, so the kernel's elementwise phases need
// no per-column loads.  Layout: blocks of 128 rows (tile t of the padded
// rows at t * QX_TILE_BYTES), each two planes of 2 KB (columns 0-7, then
// 8-15), 16 bytes per row: the K-major core-matrix layout without swizzle.  Head h's rows
// of O, dO and LSE start in_hs rows apart (a chunk of a longer sequence when
// in_hs > N).  Ragged
// batches (RAGGED): O, dO token-major [total][heads][d], LSE [heads][total],
// outputs [heads][pcu[B]] with sequence b's rows from pcu[b] (see above).
// x as three bf16 values (returned as the floats they hold) whose sum is x to
// about 2^-24 relative: each is x minus the earlier ones, rounded to bf16
// (the differences are exact in float32).
__device__ __forceinline__ void split3_bf16(float x, float* h, float* m, float* l) {
  *h = __bfloat162float(__float2bfloat16_rn(x));
  *m = __bfloat162float(__float2bfloat16_rn(x - *h));
  *l = __bfloat162float(__float2bfloat16_rn(x - *h - *m));
}

template <int D, bool RAGGED>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         const float* __restrict__ lse,
                                                         float* __restrict__ dsum, float* __restrict__ lse2,
                                                         uint8_t* __restrict__ qx, int64_t heads, int N, int Np, int64_t in_hs,
                                                         const int* __restrict__ cu,
                                                         const int* __restrict__ pcu, int B, int64_t total,
                                                         int max_len) {
  constexpr int LPR = D / 8;
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, col = (lane % LPR) * 8;
  const int64_t per_head = RAGGED ? (int64_t)pcu[B] : (int64_t)Np;   // padded rows per head
  const int64_t rows = heads * per_head;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t wrow = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; wrow * RPW < rows;
       wrow += warps_total) {
    const int64_t prow = wrow * RPW + sub;        // padded row index
    const int64_t head = prow / per_head;
    const int64_t pr = prow - head * per_head;
    bool valid;
    int64_t row, lrow;                            // row of O / dO (in d-element units), index of LSE
    if constexpr (RAGGED) {
      int lo = 0, hi = B;                         // the sequence: largest b with pcu[b] <= pr
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pcu[mid] <= pr) lo = mid;
        else hi = mid;
      }
      const int64_t i = pr - pcu[lo];
      valid = prow < rows && seq_range_ok(cu, lo, total, max_len) && i < (int64_t)(cu[lo + 1] - cu[lo]);
      const int64_t t = cu[lo] + i;               // token
      row = t * heads + head;
      lrow = head * total + t;
    } else {
      valid = prow < rows && pr < N;
      row = head * in_hs + pr;                    // dense row index
      lrow = row;
    }
    float acc = 0.f;
    if (valid) {
      const uint4 a = __ldcs(reinterpret_cast<const uint4*>(o + row * D + col));
      const uint4 b = __ldcs(reinterpret_cast<const uint4*>(dout + row * D + col));
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fa = __bfloat1622float2(pa[j]);
        const float2 fb = __bfloat1622float2(pb[j]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (prow < rows && (lane % LPR) == 0) {
      float l2 = INFINITY;
      if (valid) {
        const float L = lse[lrow];
        l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
      }
      dsum[prow] = valid ? acc : 0.f;
      lse2[prow] = l2;
      float lh, lm, ll, eh, em, el;
      split3_bf16(l2 == INFINITY ? -0x1p100f : -l2, &lh, &lm, &ll);
      split3_bf16(valid ? -acc : 0.f, &eh, &em, &el);
      uint8_t* row = qx + (size_t)(prow / TILE) * QX_TILE_BYTES + (size_t)(prow % TILE) * 16;
      *reinterpret_cast<uint4*>(row) = make_uint4(pack_bf16(lh, lm), pack_bf16(ll, lh), pack_bf16(lm, ll),
                                                  pack_bf16(lh, lm));
      *reinterpret_cast<uint4*>(row + QX_TILE_BYTES / 2) = make_uint4(pack_bf16(ll, eh), pack_bf16(em, el), 0u, 0u);
    }
  }
}

// Waits, with the given limit, on a barrier that nothing ever signals.
__global__ void wait_selftest_kernel(unsigned int* status, int64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtx w{limit_ns, status, &abort_flag};
    wait_bar(smem_u32(&bar), 0, w);
  }
}

int grid_for(int64_t warps_needed) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (warps_needed + 7) / 8;       // 8 warps per 256-thread block
  const int64_t cap = (int64_t)sms * 8;              // 8 resident blocks per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_merge(const float* const* o_parts, const float* const* lse_parts, int n_parts,
                         void* o_out, bool out_f32, float* lse_out, int rows_per_head, int heads, int d,
                         int64_t out_head_stride, cudaStream_t s) {
  MergeArgs a;
  for (int c = 0; c < MAX_PARTS; ++c) {
    a.o[c] = c < n_parts ? o_parts[c] : nullptr;
    a.lse[c] = c < n_parts ? lse_parts[c] : nullptr;
  }
  const int64_t rows = (int64_t)rows_per_head * heads;
  const int rpw = 32 / (d / 4);
  const int grid = grid_for((rows + rpw - 1) / rpw);
  if (d == 128) {
    if (out_f32) merge_kernel<128, true><<<grid, 256, 0, s>>>(a, n_parts, o_out, lse_out, rows, rows_per_head, out_head_stride);
    else merge_kernel<128, false><<<grid, 256, 0, s>>>(a, n_parts, o_out, lse_out, rows, rows_per_head, out_head_stride);
  } else {
    if (out_f32) merge_kernel<64, true><<<grid, 256, 0, s>>>(a, n_parts, o_out, lse_out, rows, rows_per_head, out_head_stride);
    else merge_kernel<64, false><<<grid, 256, 0, s>>>(a, n_parts, o_out, lse_out, rows, rows_per_head, out_head_stride);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, const float* lse, float* dsum, float* lse2,
                                  uint8_t* qx, int64_t heads, int N, int Np, int64_t in_hs, int d, cudaStream_t s) {
  const int rpw = 32 / (d / 8);
  const int grid = grid_for((heads * Np + rpw - 1) / rpw);
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  if (d == 128)
    preprocess_kernel<128, false><<<grid, 256, 0, s>>>(po, pd, lse, dsum, lse2, qx, heads, N, Np, in_hs, nullptr, nullptr,
                                                       0, 0, 0);
  else
    preprocess_kernel<64, false><<<grid, 256, 0, s>>>(po, pd, lse, dsum, lse2, qx, heads, N, Np, in_hs, nullptr, nullptr,
                                                      0, 0, 0);
  return cudaGetLastError();
}

cudaError_t launch_varlen_pad(const int* cu_seqlens, int B, int64_t total, int max_len, int* pcu,
                              unsigned int* status, cudaStream_t s) {
  varlen_pad_kernel<<<1, 32, 0, s>>>(cu_seqlens, B, total, max_len, pcu, status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess_varlen(const void* o, const void* dout, const float* lse, float* dsum, float* lse2,
                                         uint8_t* qx, int heads, int64_t total, const int* cu_seqlens, const int* pcu, int B,
                                         int max_len, int64_t padded_rows_bound, int d, cudaStream_t s) {
  const int rpw = 32 / (d / 8);
  const int grid = grid_for((heads * padded_rows_bound + rpw - 1) / rpw);
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  if (d == 128)
    preprocess_kernel<128, true><<<grid, 256, 0, s>>>(po, pd, lse, dsum, lse2, qx, heads, 0, 0, 0, cu_seqlens, pcu, B,
                                                      total, max_len);
  else
    preprocess_kernel<64, true><<<grid, 256, 0, s>>>(po, pd, lse, dsum, lse2, qx, heads, 0, 0, 0, cu_seqlens, pcu, B,
                                                     total, max_len);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned int* status, int64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
