// api.cu -- the C ABI (include/attn.h): argument validation, TMA descriptor
// encoding, launches, the per-device status word, and the host-only schedule
// builders.  Every compute step runs in the kernels of fwd.cu, bwd.cu and
// merge.cu; nothing here computes attention.  The library allocates no device
// memory: the status word and the scratch of attn_bwd_static_scratch are
// static device variables of this file.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "attn.h"
#include "internal.h"
#include "schedule.h"

using namespace attn;

namespace {

thread_local std::string g_msg;
std::mutex g_mu;
int64_t g_wait_limit_ns = 2000000000ll;
int32_t* g_debug_counts = nullptr;   // attn_debug_set_tile_counts
int64_t g_debug_capacity = 0;

constexpr int MAX_DEVICES = 64;
unsigned int* g_status[MAX_DEVICES] = {};   // device address of g_status_word, per device
int g_dev_ok[MAX_DEVICES] = {};  // 0 unknown, 1 ok, -1 unsupported

// The device status word every kernel reports to (ATTN_DEV_TIMEOUT when a
// bounded wait runs out) and attn_get_status reads and clears: a static
// device variable, so no call allocates for it.  Host code passes kernels its
// device address (looked up per device), never the host-side name.
__device__ unsigned int g_status_word;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Current device, checked to be sm_103; the device address of its status word
// looked up on first use (make a device's first call before any stream capture).
int device_ready(unsigned int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= MAX_DEVICES) return fail(ATTN_ERR_NO_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] < 0) return fail(ATTN_ERR_NO_DEVICE, "device %d is not sm_103 (GB300)", dev);
  if (g_status[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    g_status[dev] = static_cast<unsigned int*>(p);
  }
  *status = g_status[dev];
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(ATTN_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
  return ATTN_OK;
}

int check_dims(int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must be positive (B=%d Hq=%d Hkv=%d Nq=%d Nk=%d)", B, Hq, Hkv, Nq, Nk);
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d not supported (64 or 128)", d);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if ((int64_t)B * Hq > (int64_t)1 << 30 || (int64_t)Nq * d > (int64_t)1 << 40)
    return fail(ATTN_ERR_INVALID_ARG, "problem too large");
  return ATTN_OK;
}

struct MaskArgs {
  int kind = MASK_NONE;
  int causal_in_blocks = 0;
  const uint8_t* block_mask = nullptr;
  int window = 0;
};

int read_mask(const attn_mask_t* m, MaskArgs* out) {
  *out = MaskArgs();
  if (m == nullptr) return ATTN_OK;
  if (m->kind != ATTN_MASK_NONE && m->kind != ATTN_MASK_CAUSAL && m->kind != ATTN_MASK_BLOCK_SPARSE &&
      m->kind != ATTN_MASK_SLIDING_WINDOW)
    return fail(ATTN_ERR_INVALID_ARG, "unknown mask kind %d", (int)m->kind);
  out->kind = m->kind;
  out->causal_in_blocks = m->causal_in_blocks ? 1 : 0;
  if (m->kind == ATTN_MASK_BLOCK_SPARSE) {
    if (m->block_mask == nullptr) return fail(ATTN_ERR_INVALID_ARG, "block-sparse mask without block_mask");
    out->block_mask = m->block_mask;
  }
  if (m->kind == ATTN_MASK_SLIDING_WINDOW) {
    if (m->window < 1) return fail(ATTN_ERR_INVALID_ARG, "sliding window %d < 1", (int)m->window);
    out->window = m->window;
  }
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---- launch tracing: event pairs recorded on the launching stream
struct TraceEntry {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
int g_trace_cap = 0;
int64_t g_trace_count = 0;
std::vector<TraceEntry> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch; a no-op unless tracing is enabled.
struct TraceScope {
  int slot = -1;
  cudaStream_t s;
  TraceScope(int kernel, cudaStream_t stream) : s(stream) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace_on) return;
    ++g_trace_count;
    if ((int)g_trace.size() >= g_trace_cap) return;
    TraceEntry t{kernel, take_event(), take_event()};
    if (t.start == nullptr || t.stop == nullptr) return;
    cudaEventRecord(t.start, s);
    g_trace.push_back(t);
    slot = (int)g_trace.size() - 1;
  }
  ~TraceScope() {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (slot < (int)g_trace.size()) cudaEventRecord(g_trace[slot].stop, s);
  }
};

}  // namespace

namespace attn {

int encode_rows_map(CUtensorMap* map, const void* base, int d, int rows, int heads, int64_t head_stride_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)head_stride_rows * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

// Token-major [total][heads][d] bf16 as the same 3-D view (columns, rows =
// tokens, heads): consecutive tokens of one head are heads*d elements apart.
int encode_tokens_map(CUtensorMap* map, const void* base, int d, int64_t total, int heads) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)total, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)heads * d * 2, (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled (token-major) failed (%d)", (int)r);
  return ATTN_OK;
}

}  // namespace attn

// ====================================================================== C ABI

extern "C" {

int attn_version(void) { return 1; }

const char* attn_last_error_message(void) { return g_msg.c_str(); }

const char* attn_status_string(int s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
    case ATTN_ERR_WORKSPACE: return "workspace too small";
    case ATTN_ERR_NO_DEVICE: return "no usable sm_103 device";
    case ATTN_ERR_DEVICE_BOUNDS: return "a device-side index array was out of range";
    default: return "unknown status";
  }
}

void attn_set_wait_limit_ns(int64_t limit_ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_wait_limit_ns = limit_ns > 0 ? limit_ns : 2000000000ll;
}

static int64_t wait_limit() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_wait_limit_ns;
}

int attn_debug_set_tile_counts(int32_t* counts, int64_t capacity) {
  if (counts != nullptr && capacity < 0) return fail(ATTN_ERR_INVALID_ARG, "negative debug record capacity");
  if (reinterpret_cast<uintptr_t>(counts) & 3u) return fail(ATTN_ERR_MISALIGNED, "debug records not 4-byte aligned");
  std::lock_guard<std::mutex> lk(g_mu);
  g_debug_counts = counts;
  g_debug_capacity = counts != nullptr ? capacity : 0;
  return ATTN_OK;
}

// Work units of the dK/dV kernel and how many consecutive ones each CTA takes
// (at most 8): the per-CTA setup and epilogue are paid once per run and
// overlap the neighbouring units' work, while the hardware still balances the
// CTAs.  Runs grow (up to 4) while they leave twelve waves of CTAs (one CTA
// per SM), and
// light units (few query tiles each: a unit costs about the fixed part of
// 16 tiles' work) get runs of about 16 tiles even with fewer waves.  Long
// runs of equal-cost units fill the last wave badly, so nothing else lengthens
// them.  (Measured on GB300: a causal 2x32x8192 head set and the BERT-shaped
// shape gain from runs; a random 1/8 block mask, whose units all cost the
// same, does best with single units.)
static void set_kv_run(BwdParams* p) {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 148;
  }
  const int64_t n_sm = (dev >= 0 && dev < 64) ? sms[dev] : 148;
  p->kv_units = dkdv_units(*p);
  // query tiles a unit visits, expected: the query heads of its group times
  // the query tiles its key tile sees (half of them under a causal mask, the
  // window's share under a sliding window; all of them otherwise, a block
  // mask's density being unknown on the host)
  const int64_t nqt = (p->Nq + TILE - 1) / TILE;
  int64_t seen = nqt;
  if (p->mask_kind == MASK_CAUSAL || (p->mask_kind == MASK_BLOCK_SPARSE && p->causal_in_blocks)) seen = (nqt + 1) / 2;
  if (p->mask_kind == MASK_SLIDING_WINDOW) seen = std::min<int64_t>(nqt, p->window / TILE + 1);
  const int64_t tiles = std::max<int64_t>(1, seen * (p->Hq / p->Hkv));
  const int64_t by_waves = std::min<int64_t>(4, p->kv_units / (12 * n_sm));
  const int64_t by_weight = 16 / tiles;
  const int64_t run = std::max(by_waves, by_weight);
  p->kv_run = (int)(run < 1 ? 1 : (run > 8 ? 8 : run));   // at most the kernel's table of 8 units
}

// The debug record array for a launch of `ctas` CTAs (after `skip` records
// of an earlier kernel of the same call), or null when recording is off.
static int debug_records(int64_t skip, int64_t ctas, int32_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  *out = nullptr;
  if (g_debug_counts == nullptr) return ATTN_OK;
  if ((skip + ctas) * DEBUG_FIELDS > g_debug_capacity)
    return fail(ATTN_ERR_INVALID_ARG, "debug record array holds %lld int32, the launch needs %lld",
                (long long)g_debug_capacity, (long long)((skip + ctas) * DEBUG_FIELDS));
  *out = g_debug_counts + skip * DEBUG_FIELDS;
  return ATTN_OK;
}

static int fwd_common(const void* q, const void* k, const void* v, void* o, bool out_f32, float* lse, int B,
                      int Hq, int Hkv, int Nq, int Nk, int d, float scale, const attn_mask_t* mask,
                      int64_t q_off, int64_t kv_off, int64_t q_hs, int64_t kv_hs, void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")))
    return rc;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(ATTN_ERR_MISALIGNED, "lse not 4-byte aligned");
  if ((rc = check_dims(B, Hq, Hkv, Nq, Nk, d, scale))) return rc;
  if (q_hs < Nq || kv_hs < Nk) return fail(ATTN_ERR_INVALID_ARG, "head stride smaller than the rows per head");
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = encode_rows_map(&tq, q, d, Nq, B * Hq, q_hs)) || (rc = encode_rows_map(&tk, k, d, Nk, B * Hkv, kv_hs)) ||
      (rc = encode_rows_map(&tv, v, d, Nk, B * Hkv, kv_hs)))
    return rc;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.o_hs = (int64_t)Nq * d;
  p.o_rs = d;
  p.l_hs = Nq;
  p.l_rs = 1;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nk = Nk;
  p.nqc = (int)cdiv(Nq, UNIT_ROWS);
  p.head_group = kv_stream_group(B, Hq, Hkv, Nk, d);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.causal_in_blocks = m.causal_in_blocks;
  p.block_mask = m.block_mask;
  p.window = m.window;
  p.nkb = (int)cdiv(Nk, TILE);
  p.q_offset = q_off;
  p.kv_offset = kv_off;
  p.dec_nq = 1;
  p.status = status;
  p.wait_limit_ns = wait_limit();
  if ((rc = debug_records(0, fwd_grid(p), &p.tile_counts))) return rc;
  cudaError_t e;
  {
    TraceScope ts(out_f32 ? ATTN_KERNEL_PARTIAL_FWD : ATTN_KERNEL_FWD, static_cast<cudaStream_t>(stream));
    e = launch_fwd(d, out_f32, tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
             float scale, const attn_mask_t* mask, void* stream) {
  return fwd_common(q, k, v, o, false, lse, B, Hq, Hkv, N, N, d, scale, mask, 0, 0, N, N, stream);
}

int attn_partial_fwd(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int Hq,
                     int Hkv, int Nq, int Nk, int d, float scale, const attn_mask_t* mask, int64_t q_offset,
                     int64_t kv_offset, int64_t q_head_stride, int64_t kv_head_stride, void* stream) {
  if (lse_part == nullptr) return fail(ATTN_ERR_INVALID_ARG, "lse_part is NULL");
  return fwd_common(q, k, v, o_part, true, lse_part, B, Hq, Hkv, Nq, Nk, d, scale, mask, q_offset, kv_offset,
                    q_head_stride > 0 ? q_head_stride : Nq, kv_head_stride > 0 ? kv_head_stride : Nk, stream);
}

int attn_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens, int B,
                    int max_len, int64_t total, int Hq, int Hkv, int d, float scale, const attn_mask_t* mask,
                    void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) || (rc = check_ptr(o, "o")))
    return rc;
  if (cu_seqlens == nullptr) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(ATTN_ERR_MISALIGNED, "cu_seqlens not 4-byte aligned");
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(ATTN_ERR_MISALIGNED, "lse not 4-byte aligned");
  if (total < 1 || total > ((int64_t)1 << 31) - 1) return fail(ATTN_ERR_INVALID_ARG, "total=%lld", (long long)total);
  if (max_len < 1) return fail(ATTN_ERR_INVALID_ARG, "max_len=%d", max_len);
  if ((rc = check_dims(B, Hq, Hkv, max_len, max_len, d, scale))) return rc;
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  if (m.kind == MASK_BLOCK_SPARSE) return fail(ATTN_ERR_UNSUPPORTED, "block-sparse masks are not built for ragged batches");
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = encode_tokens_map(&tq, q, d, total, Hq)) || (rc = encode_tokens_map(&tk, k, d, total, Hkv)) ||
      (rc = encode_tokens_map(&tv, v, d, total, Hkv)))
    return rc;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.o_hs = d;
  p.o_rs = (int64_t)Hq * d;
  p.l_hs = total;
  p.l_rs = 1;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = max_len; p.Nk = max_len;
  p.nqc = (int)cdiv(max_len, UNIT_ROWS);
  p.head_group = 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.window = m.window;
  p.nkb = (int)cdiv(max_len, TILE);
  p.dec_nq = 1;
  p.cu_seqlens = cu_seqlens;
  p.varlen_nqc = p.nqc;
  p.total = total;
  p.status = status;
  p.wait_limit_ns = wait_limit();
  if ((rc = debug_records(0, fwd_grid(p), &p.tile_counts))) return rc;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_VARLEN_FWD, static_cast<cudaStream_t>(stream));
    e = launch_fwd(d, false, tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "variable-length forward launch");
  return ATTN_OK;
}

size_t attn_fwd_fp8_workspace_bytes(int B, int Hkv, int N, int d) {
  if (B < 1 || Hkv < 1 || N < 1 || d < 1) return 0;
  return (size_t)B * Hkv * d * (size_t)(cdiv(N, TILE) * TILE);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, float q_descale, float k_descale, float v_descale,
                 void* o, float* lse, int B, int Hq, int Hkv, int N, int d, float scale, const attn_mask_t* mask,
                 void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_ptr(q8, "q8")) || (rc = check_ptr(k8, "k8")) || (rc = check_ptr(v8, "v8")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(workspace, "workspace")))
    return rc;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(ATTN_ERR_MISALIGNED, "lse not 4-byte aligned");
  if ((rc = check_dims(B, Hq, Hkv, N, N, d, scale))) return rc;
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the e4m3 forward is built for d = 128 only (d=%d)", d);
  for (float f : {q_descale, k_descale, v_descale})
    if (!(f > 0.f) || !std::isfinite(f)) return fail(ATTN_ERR_INVALID_ARG, "descale factors must be finite and > 0");
  if (workspace_bytes < attn_fwd_fp8_workspace_bytes(B, Hkv, N, d))
    return fail(ATTN_ERR_WORKSPACE, "workspace %zu < %zu bytes", workspace_bytes,
                attn_fwd_fp8_workspace_bytes(B, Hkv, N, d));
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  auto fn = encode_fn();
  if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int Np = (int)(cdiv(N, TILE) * TILE);
  // byte maps, 128 x 128 boxes (128 e4m3 values = one 128-byte swizzle row)
  auto encode = [&](CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t heads) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(cols * rows)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled (e4m3) failed (%d)", (int)r);
    return (int)ATTN_OK;
  };
  CUtensorMap tq, tk, tvt;
  if ((rc = encode(&tq, q8, d, N, (int64_t)B * Hq)) || (rc = encode(&tk, k8, d, N, (int64_t)B * Hkv)) ||
      (rc = encode(&tvt, workspace, Np, d, (int64_t)B * Hkv)))
    return rc;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.o_hs = (int64_t)N * d;
  p.o_rs = d;
  p.l_hs = N;
  p.l_rs = 1;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = N; p.Nk = N;
  p.nqc = (int)cdiv(N, UNIT_ROWS);
  p.head_group = kv_stream_group(B, Hq, Hkv, N, d / 2);   // K + V are half the bf16 bytes
  p.scale_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.causal_in_blocks = m.causal_in_blocks;
  p.block_mask = m.block_mask;
  p.window = m.window;
  p.nkb = (int)cdiv(N, TILE);
  p.dec_nq = 1;
  p.status = status;
  p.wait_limit_ns = wait_limit();
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_FP8_TRANSPOSE_V, st);
    e = launch_transpose_v_fp8(v8, workspace, B * Hkv, N, Np, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 V transpose launch");
  {
    TraceScope ts(ATTN_KERNEL_FP8_FWD, st);
    e = launch_fwd_fp8(tq, tk, tvt, p, v_descale, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 forward launch");
  return ATTN_OK;
}

int attn_decode_splits(int B, int Hkv, int Nk) {
  if (B < 1 || Hkv < 1 || Nk < 1) return 1;
  // about six waves of CTAs on 148 SMs (measured on B=8, Hkv=8, Nk=32768:
  // 5 splits 3.9 TB/s, 8: 4.5, 16: 4.7, 32: 4.1), at least one key tile each
  const int64_t want = cdiv(6 * 148, (int64_t)B * Hkv);
  const int64_t tiles = cdiv(Nk, TILE);
  int64_t n = want < tiles ? want : tiles;
  if (n > 64) n = 64;
  return n < 1 ? 1 : (int)n;
}

// Decoding units whose g * Nq rows fit one 128-row tile give the second query
// tile (otherwise idle) the same rows and every other key tile of the split;
// each tile writes its own partial, so a split leaves two (within the
// merge's 64 parts).
static int decode_parts(int Hq, int Hkv, int Nq, int n_splits) {
  const bool alternate = Hkv > 0 && (Hq / Hkv) * Nq <= TILE && 2 * n_splits <= 64;
  return alternate ? 2 * n_splits : n_splits;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int n_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  const int ns = n_splits > 0 ? n_splits : attn_decode_splits(B, Hkv, Nk);
  const size_t rows = (size_t)B * Hq * Nq;
  const size_t per = ((rows * (size_t)d * 4 + 255) & ~(size_t)255) + ((rows * 4 + 255) & ~(size_t)255);
  return per * (size_t)decode_parts(Hq, Hkv, Nq, ns);
}

int attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens, void* o,
                    float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal, int n_splits,
                    void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k_cache, "k_cache")) || (rc = check_ptr(v_cache, "v_cache")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(workspace, "workspace")))
    return rc;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(ATTN_ERR_MISALIGNED, "lse not 4-byte aligned");
  if (seq_lens != nullptr && (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(ATTN_ERR_MISALIGNED, "seq_lens not 4-byte aligned");
  if ((rc = check_dims(B, Hq, Hkv, Nq, Nk, d, scale))) return rc;
  const int rows = (Hq / Hkv) * Nq;
  if (rows > UNIT_ROWS) return fail(ATTN_ERR_INVALID_ARG, "(Hq/Hkv)*Nq = %d exceeds %d rows", rows, UNIT_ROWS);
  if (Nq > Nk) return fail(ATTN_ERR_INVALID_ARG, "Nq=%d exceeds the cache length Nk=%d", Nq, Nk);
  if (n_splits < 0 || n_splits > 64) return fail(ATTN_ERR_INVALID_ARG, "n_splits=%d outside [0, 64]", n_splits);
  const int ns = n_splits > 0 ? n_splits : attn_decode_splits(B, Hkv, Nk);
  const int parts = decode_parts(Hq, Hkv, Nq, ns);
  if (workspace_bytes < attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, ns))
    return fail(ATTN_ERR_WORKSPACE, "decode workspace of %zu bytes is too small", workspace_bytes);
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv;
  // q viewed as [B*Hkv][g*Nq rows][d]: the g heads of a kv head are adjacent
  if ((rc = encode_rows_map(&tq, q, d, rows, B * Hkv, rows)) ||
      (rc = encode_rows_map(&tk, k_cache, d, Nk, B * Hkv, Nk)) || (rc = encode_rows_map(&tv, v_cache, d, Nk, B * Hkv, Nk)))
    return rc;
  // the split partials lie one after another, each laid out like o_part /
  // lse_part of attn_partial_fwd: all O blocks first, then all LSE blocks
  const int64_t total_rows = (int64_t)B * Hq * Nq;
  const size_t o_bytes = ((size_t)total_rows * d * 4 + 255) & ~(size_t)255;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_l = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes * parts);
  FwdParams p{};
  p.o = ws_o;
  p.lse = ws_l;
  p.o_hs = (int64_t)rows * d;
  p.o_rs = d;
  p.l_hs = rows;
  p.l_rs = 1;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = rows; p.Nk = Nk;
  p.nqc = 1;
  p.head_group = 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = causal ? MASK_CAUSAL : MASK_NONE;
  p.nkb = (int)cdiv(Nk, TILE);
  p.seq_lens = seq_lens;
  p.n_splits = ns;
  p.split_tiles = (int)cdiv(cdiv(Nk, TILE), ns);
  p.dec_nq = Nq;
  p.split_rows = total_rows;
  p.dec_interleave = parts > ns ? 1 : 0;
  p.status = status;
  p.wait_limit_ns = wait_limit();
  if ((rc = debug_records(0, fwd_grid(p), &p.tile_counts))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_DECODE, s);
    e = launch_fwd(d, true, tq, tk, tv, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  const float* op[64];
  const float* lp[64];
  for (int c = 0; c < parts; ++c) {
    op[c] = ws_o + (size_t)c * total_rows * d;
    lp[c] = ws_l + (size_t)c * total_rows;
  }
  {
    TraceScope ts(ATTN_KERNEL_MERGE, s);
    e = launch_merge(op, lp, parts, o, false, lse, Nq, B * Hq, d, Nq, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode merge launch");
  return ATTN_OK;
}

int attn_merge_lse(const float* const* o_parts, const float* const* lse_parts, int n_parts, void* o_out,
                   int out_dtype, float* lse_out, int B, int Hq, int Nq, int d, int64_t out_head_stride,
                   void* stream) {
  if (o_parts == nullptr || lse_parts == nullptr) return fail(ATTN_ERR_INVALID_ARG, "part arrays are NULL");
  if (n_parts < 1 || n_parts > 64) return fail(ATTN_ERR_INVALID_ARG, "n_parts=%d outside [1, 64]", n_parts);
  int rc;
  for (int c = 0; c < n_parts; ++c) {
    if ((rc = check_ptr(o_parts[c], "o_parts[c]"))) return rc;
    if (lse_parts[c] == nullptr) return fail(ATTN_ERR_INVALID_ARG, "lse_parts[%d] is NULL", c);
  }
  if ((rc = check_ptr(o_out, "o_out"))) return rc;
  if (out_dtype != ATTN_DTYPE_BF16 && out_dtype != ATTN_DTYPE_F32)
    return fail(ATTN_ERR_INVALID_ARG, "out_dtype=%d", out_dtype);
  if ((rc = check_dims(B, Hq, Hq, Nq, Nq, d, 1.f))) return rc;
  const int64_t hs = out_head_stride > 0 ? out_head_stride : Nq;
  if (hs < Nq) return fail(ATTN_ERR_INVALID_ARG, "out_head_stride smaller than Nq");
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_MERGE, static_cast<cudaStream_t>(stream));
    e = launch_merge(o_parts, lse_parts, n_parts, o_out, out_dtype == ATTN_DTYPE_F32, lse_out, Nq, B * Hq, d, hs,
                     static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  (void)Hkv;
  (void)d;
  if (B < 1 || Hq < 1 || N < 1) return 0;
  // D, LSE*log2(e) and the dK/dV statistics operand per query row, rows
  // padded to whole tiles
  return stats_layout((int64_t)B * Hq * cdiv(N, TILE) * TILE).bytes;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
             float scale, const attn_mask_t* mask, void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")) || (rc = check_ptr(dout, "dout")) ||
      (rc = check_ptr(dq, "dq")) || (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")) ||
      (rc = check_ptr(workspace, "workspace")))
    return rc;
  if ((rc = check_dims(B, Hq, Hkv, N, N, d, scale))) return rc;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Hkv, N, d))
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace_bytes,
                attn_bwd_workspace_bytes(B, Hq, Hkv, N, d));
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = encode_rows_map(&tq, q, d, N, B * Hq, N)) || (rc = encode_rows_map(&tk, k, d, N, B * Hkv, N)) ||
      (rc = encode_rows_map(&tv, v, d, N, B * Hkv, N)) || (rc = encode_rows_map(&tdo, dout, d, N, B * Hq, N)))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Np = (int)(cdiv(N, TILE) * TILE);
  const StatsLayout sl = stats_layout((int64_t)B * Hq * Np);
  float* dsum = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + sl.lse2_off);
  uint8_t* qx = static_cast<uint8_t*>(workspace) + sl.qx_off;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_BWD_PREPROCESS, s);
    e = launch_bwd_preprocess(o, dout, lse, dsum, lse2, qx, (int64_t)B * Hq, N, Np, N, d, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  BwdParams p{};
  p.lse2 = lse2;
  p.dsum = dsum;
  p.qx = qx;
  p.Np = Np;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = N; p.Nk = N;
  p.dq_hs = N; p.dkv_hs = N;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.causal_in_blocks = m.causal_in_blocks;
  p.block_mask = m.block_mask;
  p.window = m.window;
  p.nkb = (int)cdiv(N, TILE);
  p.kv_group = q_stream_group(B, Hq, Hkv, N, d);
  p.q_group = kv_stream_group(B, Hq, Hkv, N, d);
  p.status = status;
  p.wait_limit_ns = wait_limit();
  set_kv_run(&p);
  if ((rc = debug_records(0, p.kv_units, &p.dkdv_counts)) ||
      (rc = debug_records(p.kv_units, dq_grid(p), &p.dq_counts)))
    return rc;
  {
    TraceScope ts(ATTN_KERNEL_BWD_DKDV, s);
    e = launch_bwd_dkdv(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
  {
    TraceScope ts(ATTN_KERNEL_BWD_DQ, s);
    e = launch_bwd_dq(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward dQ launch");
  return ATTN_OK;
}

int attn_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int Hq, int Nq, int d,
                        int64_t head_stride, void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_ptr(o, "o")) || (rc = check_ptr(dout, "dout")) || (rc = check_ptr(workspace, "workspace")))
    return rc;
  if (lse == nullptr) return fail(ATTN_ERR_INVALID_ARG, "lse is NULL");
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return fail(ATTN_ERR_MISALIGNED, "lse not 4-byte aligned");
  if ((rc = check_dims(B, Hq, Hq, Nq, Nq, d, 1.f))) return rc;
  const int64_t hs = head_stride > 0 ? head_stride : Nq;
  if (hs < Nq) return fail(ATTN_ERR_INVALID_ARG, "head_stride %lld smaller than Nq=%d", (long long)hs, Nq);
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Hq, Nq, d))
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace_bytes,
                attn_bwd_workspace_bytes(B, Hq, Hq, Nq, d));
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Np = (int)(cdiv(Nq, TILE) * TILE);
  const StatsLayout sl = stats_layout((int64_t)B * Hq * Np);
  float* dsum = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + sl.lse2_off);
  uint8_t* qx = static_cast<uint8_t*>(workspace) + sl.qx_off;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_BWD_PREPROCESS, s);
    e = launch_bwd_preprocess(o, dout, lse, dsum, lse2, qx, (int64_t)B * Hq, Nq, Np, hs, d, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  return ATTN_OK;
}

int attn_partial_bwd(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                     size_t workspace_bytes, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                     int d, float scale, const attn_mask_t* mask, int64_t q_offset, int64_t kv_offset,
                     int64_t q_head_stride, int64_t kv_head_stride, int accumulate, void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(dout, "dout")) || (rc = check_ptr(workspace, "workspace")) || (rc = check_ptr(dq, "dq")) ||
      (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")))
    return rc;
  if ((rc = check_dims(B, Hq, Hkv, Nq, Nk, d, scale))) return rc;
  const int64_t qhs = q_head_stride > 0 ? q_head_stride : Nq;
  const int64_t khs = kv_head_stride > 0 ? kv_head_stride : Nk;
  if (qhs < Nq || khs < Nk) return fail(ATTN_ERR_INVALID_ARG, "head stride smaller than the rows per head");
  // the kernels compare position differences in 32-bit integers
  const int64_t delta = q_offset - kv_offset;
  if (q_offset < 0 || kv_offset < 0 || delta > ((int64_t)1 << 30) || delta < -((int64_t)1 << 30) ||
      (int64_t)Nq + Nk > ((int64_t)1 << 30))
    return fail(ATTN_ERR_INVALID_ARG, "offsets must be >= 0, |q_offset - kv_offset| <= 2^30 and Nq + Nk <= 2^30");
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Hkv, Nq, d))
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace_bytes,
                attn_bwd_workspace_bytes(B, Hq, Hkv, Nq, d));
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = encode_rows_map(&tq, q, d, Nq, B * Hq, qhs)) || (rc = encode_rows_map(&tk, k, d, Nk, B * Hkv, khs)) ||
      (rc = encode_rows_map(&tv, v, d, Nk, B * Hkv, khs)) || (rc = encode_rows_map(&tdo, dout, d, Nq, B * Hq, qhs)))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Np = (int)(cdiv(Nq, TILE) * TILE);
  const StatsLayout sl = stats_layout((int64_t)B * Hq * Np);
  BwdParams p{};
  p.dsum = static_cast<const float*>(workspace);
  p.lse2 = reinterpret_cast<const float*>(static_cast<const char*>(workspace) + sl.lse2_off);
  p.qx = static_cast<const uint8_t*>(workspace) + sl.qx_off;
  p.Np = Np;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nk = Nk;
  p.delta = (int)delta;
  p.dq_hs = qhs; p.dkv_hs = khs;
  p.accumulate = accumulate ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.causal_in_blocks = m.causal_in_blocks;
  p.block_mask = m.block_mask;
  p.window = m.window;
  p.nkb = (int)cdiv(Nk, TILE);
  p.kv_group = q_stream_group(B, Hq, Hkv, Nq, d);
  p.q_group = kv_stream_group(B, Hq, Hkv, Nk, d);
  p.status = status;
  p.wait_limit_ns = wait_limit();
  set_kv_run(&p);
  if ((rc = debug_records(0, p.kv_units, &p.dkdv_counts)) ||
      (rc = debug_records(p.kv_units, dq_grid(p), &p.dq_counts)))
    return rc;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_BWD_DKDV, s);
    e = launch_bwd_dkdv(d, true, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "partial backward dK/dV launch");
  {
    TraceScope ts(ATTN_KERNEL_BWD_DQ, s);
    e = launch_bwd_dq(d, true, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "partial backward dQ launch");
  return ATTN_OK;
}

size_t attn_varlen_bwd_workspace_bytes(int B, int64_t total, int Hq) {
  if (B < 1 || total < 1 || Hq < 1) return 0;
  const size_t pcu = ((size_t)(B + 1) * sizeof(int) + 255) & ~(size_t)255;
  // each sequence padded to whole tiles: at most total + 127 B rows per head
  return pcu + stats_layout((int64_t)Hq * (total + (int64_t)(TILE - 1) * B)).bytes;
}

int attn_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int B, int max_len, int64_t total, int Hq,
                    int Hkv, int d, float scale, const attn_mask_t* mask, void* workspace, size_t workspace_bytes,
                    void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")) || (rc = check_ptr(dout, "dout")) ||
      (rc = check_ptr(dq, "dq")) || (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")) ||
      (rc = check_ptr(workspace, "workspace")))
    return rc;
  if (cu_seqlens == nullptr) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(ATTN_ERR_MISALIGNED, "cu_seqlens not 4-byte aligned");
  if (total < 1 || total > ((int64_t)1 << 31) - 1) return fail(ATTN_ERR_INVALID_ARG, "total=%lld", (long long)total);
  if (max_len < 1) return fail(ATTN_ERR_INVALID_ARG, "max_len=%d", max_len);
  if ((rc = check_dims(B, Hq, Hkv, max_len, max_len, d, scale))) return rc;
  if (workspace_bytes < attn_varlen_bwd_workspace_bytes(B, total, Hq))
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace_bytes,
                attn_varlen_bwd_workspace_bytes(B, total, Hq));
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  if (m.kind == MASK_BLOCK_SPARSE) return fail(ATTN_ERR_UNSUPPORTED, "block-sparse masks are not built for ragged batches");
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = encode_tokens_map(&tq, q, d, total, Hq)) || (rc = encode_tokens_map(&tk, k, d, total, Hkv)) ||
      (rc = encode_tokens_map(&tv, v, d, total, Hkv)) || (rc = encode_tokens_map(&tdo, dout, d, total, Hq)))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* pcu = static_cast<int*>(workspace);
  const size_t pcu_bytes = ((size_t)(B + 1) * sizeof(int) + 255) & ~(size_t)255;
  const int64_t bound = total + (int64_t)(TILE - 1) * B;   // padded rows per head, at most
  char* stats = static_cast<char*>(workspace) + pcu_bytes;
  const StatsLayout sl = stats_layout((int64_t)Hq * bound);
  float* dsum = reinterpret_cast<float*>(stats);
  float* lse2 = reinterpret_cast<float*>(stats + sl.lse2_off);
  uint8_t* qx = reinterpret_cast<uint8_t*>(stats + sl.qx_off);
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_BWD_PREPROCESS, s);
    e = launch_varlen_pad(cu_seqlens, B, total, max_len, pcu, status, s);
    if (e == cudaSuccess)
      e = launch_bwd_preprocess_varlen(o, dout, lse, dsum, lse2, qx, Hq, total, cu_seqlens, pcu, B, max_len, bound, d,
                                       s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "ragged backward preprocess launch");
  BwdParams p{};
  p.lse2 = lse2;
  p.dsum = dsum;
  p.qx = qx;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = max_len; p.Nk = max_len;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.window = m.window;
  p.nkb = (int)cdiv(max_len, TILE);
  p.cu_seqlens = cu_seqlens;
  p.pcu = pcu;
  p.total = total;
  p.kv_group = 1;
  p.q_group = 1;
  p.status = status;
  p.wait_limit_ns = wait_limit();
  set_kv_run(&p);
  if ((rc = debug_records(0, p.kv_units, &p.dkdv_counts)) ||
      (rc = debug_records(p.kv_units, dq_grid(p), &p.dq_counts)))
    return rc;
  {
    TraceScope ts(ATTN_KERNEL_BWD_DKDV, s);
    e = launch_bwd_dkdv(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "ragged backward dK/dV launch");
  {
    TraceScope ts(ATTN_KERNEL_BWD_DQ, s);
    e = launch_bwd_dq(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "ragged backward dQ launch");
  return ATTN_OK;
}

int attn_build_schedule(int mask_kind, int causal_in_blocks, const uint8_t* host_block_mask, int window, int B, int Hq,
                        int Hkv,
                        int Nq, int Nk, int d, int64_t q_offset, int64_t kv_offset, int32_t* out, size_t cap,
                        size_t* n_out) {
  if (n_out == nullptr) return fail(ATTN_ERR_INVALID_ARG, "n_out is NULL");
  *n_out = 0;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1) return fail(ATTN_ERR_INVALID_ARG, "sizes must be positive");
  if (Hq % Hkv) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (mask_kind < 0 || mask_kind > 3) return fail(ATTN_ERR_INVALID_ARG, "unknown mask kind %d", mask_kind);
  if (mask_kind == ATTN_MASK_BLOCK_SPARSE && host_block_mask == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "block-sparse schedule needs host_block_mask");
  if (mask_kind == ATTN_MASK_SLIDING_WINDOW && window < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sliding window %d < 1", window);
  const int nqc = (int)cdiv(Nq, UNIT_ROWS);
  const int nkb = (int)cdiv(Nk, TILE);
  const int64_t units = (int64_t)B * Hq * nqc;
  const int group = kv_stream_group(B, Hq, Hkv, Nk, d);
  *n_out = (size_t)units;
  if (out == nullptr || cap < (size_t)units * 3) return fail(ATTN_ERR_INVALID_ARG, "output capacity too small");
  for (int64_t i = 0; i < units; ++i) {
    const Unit u = fwd_unit(i, B, Hq, Hkv, Nq, Nk, nqc, group, mask_kind, causal_in_blocks, host_block_mask, nkb,
                            window, q_offset, kv_offset);
    int cnt = 0;
    for (int kt = u.kt_begin; kt < u.kt_end; ++kt) cnt += unit_uses(u, kt) ? 1 : 0;
    out[3 * i + 0] = u.bh;
    out[3 * i + 1] = u.row0 / UNIT_ROWS;
    out[3 * i + 2] = cnt;
  }
  return ATTN_OK;
}

int attn_build_chunk_schedule(int n_chunks, int n_lanes, int32_t* pairs_out, size_t cap, size_t* n_out) {
  if (n_out == nullptr) return fail(ATTN_ERR_INVALID_ARG, "n_out is NULL");
  *n_out = 0;
  if (n_chunks < 1 || n_chunks > 4096) return fail(ATTN_ERR_INVALID_ARG, "n_chunks=%d", n_chunks);
  const int lanes = n_lanes > 0 ? n_lanes : n_chunks;
  struct Pair { int qc, kc, cost; };
  std::vector<Pair> pairs;
  for (int qc = 0; qc < n_chunks; ++qc)
    for (int kc = 0; kc <= qc; ++kc) pairs.push_back({qc, kc, qc == kc ? 1 : 2});
  *n_out = pairs.size();
  if (pairs_out == nullptr || cap < 2 * pairs.size()) return fail(ATTN_ERR_INVALID_ARG, "output capacity too small");
  std::stable_sort(pairs.begin(), pairs.end(), [](const Pair& a, const Pair& b) {
    if (a.cost != b.cost) return a.cost > b.cost;
    if (a.qc != b.qc) return a.qc > b.qc;
    return a.kc < b.kc;
  });
  std::vector<int64_t> load(lanes, 0);
  std::vector<std::vector<Pair>> per(lanes);
  for (const Pair& p : pairs) {
    int best = 0;
    for (int l = 1; l < lanes; ++l)
      if (load[l] < load[best]) best = l;
    load[best] += p.cost;
    per[best].push_back(p);
  }
  size_t depth = 0, n = 0;
  for (auto& v : per) depth = std::max(depth, v.size());
  for (size_t pos = 0; pos < depth; ++pos)
    for (int l = 0; l < lanes; ++l)
      if (pos < per[l].size()) {
        pairs_out[2 * n] = per[l][pos].qc;
        pairs_out[2 * n + 1] = per[l][pos].kc;
        ++n;
      }
  return ATTN_OK;
}

int attn_get_status(void* stream) {
  unsigned int* status = nullptr;
  int rc = device_ready(&status);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int h = 0;
  e = cudaMemcpy(&h, status, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (h != 0) {
    e = cudaMemset(status, 0, sizeof h);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (h & ATTN_DEV_BOUNDS)
      return fail(ATTN_ERR_DEVICE_BOUNDS, "a device-side index array was out of range; the affected sequences were "
                                          "skipped (status 0x%x)", h);
    return fail(ATTN_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (status 0x%x)", h);
  }
  return ATTN_OK;
}

int attn_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  unsigned int* status = nullptr;
  int rc = device_ready(&status);
  if (rc) return rc;
  if (limit_ns <= 0 || limit_ns > 10000000000ll) return fail(ATTN_ERR_INVALID_ARG, "limit_ns outside (0, 1e10]");
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_SELFTEST, static_cast<cudaStream_t>(stream));
    e = launch_wait_selftest(status, limit_ns, static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ATTN_OK;
}

int attn_trace_enable(int capacity) {
  if (capacity < 1 || capacity > (1 << 20)) return fail(ATTN_ERR_INVALID_ARG, "trace capacity %d", capacity);
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& t : g_trace) {
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_trace.clear();
  g_trace.reserve(capacity);
  g_trace_cap = capacity;
  g_trace_count = 0;
  g_trace_on = true;
  return ATTN_OK;
}

int attn_trace_disable(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  return ATTN_OK;
}

int attn_trace_read(attn_trace_record_t* out, int cap, int* n_out) {
  if (n_out == nullptr) return fail(ATTN_ERR_INVALID_ARG, "n_out is NULL");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  *n_out = (int)g_trace_count;
  int rc = ATTN_OK;
  for (size_t i = 0; i < g_trace.size(); ++i) {
    TraceEntry& t = g_trace[i];
    cudaError_t e = cudaEventSynchronize(t.stop);
    float ms = -1.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
    if (e != cudaSuccess) rc = cuda_fail(e, "reading a trace event");
    if (out != nullptr && (int)i < cap) {
      out[i].kernel = t.kernel;
      out[i].ms = ms;
    }
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_trace.clear();
  g_trace_count = 0;
  return rc;
}

}  // extern "C"

// ============================================================ static scratch
// attn_bwd_static_scratch: attn_bwd without a caller workspace and without any
// device allocation, for callers that cannot call cudaMalloc.  The scratch is a
// file-scope static device array; host code never passes the array's name to a
// kernel (in host code that name is only a host-side stand-in) but its device
// address, looked up once per device with cudaGetSymbolAddress.
namespace {

static_assert(stats_layout(ATTN_STATIC_SCRATCH_ROWS).bytes <= ATTN_STATIC_SCRATCH_BYTES,
              "the static scratch holds the statistics of ATTN_STATIC_SCRATCH_ROWS query rows");
static __device__ __align__(256) float g_static_scratch[ATTN_STATIC_SCRATCH_BYTES / sizeof(float)];

float* g_static_dev[MAX_DEVICES] = {};
std::mutex g_static_mu;

// Device address of the static scratch on the current device (device_ready
// has checked the device and looked up its status word).
int static_scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= MAX_DEVICES) return fail(ATTN_ERR_NO_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_dev[dev] == nullptr) {
    void* ps = nullptr;
    e = cudaGetSymbolAddress(&ps, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_dev[dev] = static_cast<float*>(ps);
  }
  *out = g_static_dev[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                       int Hq, int Hkv, int N, int d, float scale, const attn_mask_t* mask,
                                       void* stream) {
  int rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")) || (rc = check_ptr(dout, "dout")) ||
      (rc = check_ptr(dq, "dq")) || (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")))
    return rc;
  if ((rc = check_dims(B, Hq, Hkv, N, N, d, scale))) return rc;
  const int64_t Np = cdiv(N, TILE) * TILE;
  const int64_t rows = (int64_t)B * Hq * Np;
  if (rows > ATTN_STATIC_SCRATCH_ROWS)
    return fail(ATTN_ERR_WORKSPACE,
                "B*Hq*ceil(N/128)*128 = %lld query rows exceed the static scratch limit of %lld rows",
                (long long)rows, (long long)ATTN_STATIC_SCRATCH_ROWS);
  static_assert(ATTN_STATIC_SCRATCH_ROWS % TILE == 0, "whole tiles");
  MaskArgs m;
  if ((rc = read_mask(mask, &m))) return rc;
  unsigned int* status = nullptr;
  if ((rc = device_ready(&status))) return rc;
  float* scratch = nullptr;
  if ((rc = static_scratch_for_current_device(&scratch))) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = encode_rows_map(&tq, q, d, N, B * Hq, N)) || (rc = encode_rows_map(&tk, k, d, N, B * Hkv, N)) ||
      (rc = encode_rows_map(&tv, v, d, N, B * Hkv, N)) || (rc = encode_rows_map(&tdo, dout, d, N, B * Hq, N)))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const StatsLayout sl = stats_layout(rows);
  float* dsum = scratch;
  float* lse2 = reinterpret_cast<float*>(reinterpret_cast<char*>(scratch) + sl.lse2_off);
  uint8_t* qx = reinterpret_cast<uint8_t*>(scratch) + sl.qx_off;
  cudaError_t e;
  {
    TraceScope ts(ATTN_KERNEL_BWD_PREPROCESS, s);
    e = launch_bwd_preprocess(o, dout, lse, dsum, lse2, qx, (int64_t)B * Hq, N, (int)Np, N, d, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  BwdParams p{};
  p.lse2 = lse2;
  p.dsum = dsum;
  p.qx = qx;
  p.Np = (int)Np;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = N; p.Nk = N;
  p.dq_hs = N; p.dkv_hs = N;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = m.kind;
  p.causal_in_blocks = m.causal_in_blocks;
  p.block_mask = m.block_mask;
  p.window = m.window;
  p.nkb = (int)cdiv(N, TILE);
  p.kv_group = q_stream_group(B, Hq, Hkv, N, d);
  p.q_group = kv_stream_group(B, Hq, Hkv, N, d);
  p.status = status;
  p.wait_limit_ns = wait_limit();
  set_kv_run(&p);
  if ((rc = debug_records(0, p.kv_units, &p.dkdv_counts)) ||
      (rc = debug_records(p.kv_units, dq_grid(p), &p.dq_counts)))
    return rc;
  {
    TraceScope ts(ATTN_KERNEL_BWD_DKDV, s);
    e = launch_bwd_dkdv(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
  {
    TraceScope ts(ATTN_KERNEL_BWD_DQ, s);
    e = launch_bwd_dq(d, false, tq, tk, tv, tdo, p, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward dQ launch");
  return ATTN_OK;
}
