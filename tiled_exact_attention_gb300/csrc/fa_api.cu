// Host side of the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, the split-count heuristic, launches and status codes.
// No allocation happens here: every buffer, including the split-KV workspace,
// belongs to the caller.
#include <array>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// One status word per device: kernels record the first wait that ran out.
__device__ int g_fa_status;

// Split-KV scratch for callers that cannot allocate device memory
// (fa_fwd_splitkv_noalloc).  Every device that loads this library holds it
// until the process exits.  Host code must not use the symbol's address
// directly (it is a host-side stand-in): the device address comes from
// cudaGetSymbolAddress, once per device.
static_assert(FA_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) uint8_t g_splitkv_scratch[FA_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 128;

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int* status = nullptr;
  int sms = 0;
};

bool device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& di = cache[dev];
  if (di.status == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    di.status = static_cast<int*>(p);
    di.sms = sms;
  }
  *out = di;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool strides_ok(const int64_t s[3]) {
  for (int i = 0; i < 3; ++i) {
    if (s[i] <= 0 || (s[i] % 8) != 0) return false;
    if (s[i] * 2 >= (static_cast<int64_t>(1) << 40)) return false;
  }
  return true;
}

// softcap: 0 (off) or a finite positive cap
bool softcap_ok(float c) { return c == 0.f || (c > 0.f && std::isfinite(c)); }

// Softcap constants for a kernel whose score x relates to the scaled score s by
// s = s_per_x * x: tanh(s / c) = 1 - 2 / (2^(k x) + 1) with k = 2 log2(e) s_per_x / c,
// and the capped score in log2 units is b tanh(s / c) with b = c log2(e).  c = 0: off.
void softcap_consts(float c, double s_per_x, float* k, float* b) {
  constexpr double kLog2eD = 1.4426950408889634;
  if (!(c > 0.f)) {
    *k = 0.f;
    *b = 0.f;
    return;
  }
  *k = static_cast<float>(2.0 * kLog2eD * s_per_x / static_cast<double>(c));
  *b = static_cast<float>(static_cast<double>(c) * kLog2eD);
}

fa_status validate(const fa_fwd_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->sq < 0 || a->skv < 0 || a->hq < 1 || a->hkv < 1) return FA_ERR_INVALID_ARG;
  if (a->hq % a->hkv != 0) return FA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return FA_ERR_INVALID_ARG;
  if (a->local != 0 && a->local != 1) return FA_ERR_INVALID_ARG;
  if (a->local && (a->window_left < -1 || a->window_right < -1)) return FA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return FA_ERR_INVALID_ARG;
  if (!softcap_ok(a->softcap)) return FA_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128 && a->d != 256) return FA_ERR_UNSUPPORTED;
  if (a->sq > (1 << 30) || a->skv > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (a->sq == 0) return FA_OK;
  if (a->q == nullptr || a->o == nullptr || a->lse == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4)) return FA_ERR_INVALID_ARG;
  if (!strides_ok(a->q_strides) || !strides_ok(a->o_strides)) return FA_ERR_INVALID_ARG;
  if (a->skv > 0) {
    if (a->k == nullptr || a->v == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(a->k, 16) || !aligned(a->v, 16)) return FA_ERR_INVALID_ARG;
    if (!strides_ok(a->k_strides) || !strides_ok(a->v_strides)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

// 4-D tiled map over [b][s][h][d] storage: dims (d, h, s, b), box (inner, 1, rows, 1).
bool encode_map(CUtensorMap* m, const void* ptr, fa_dtype dt, int d, int h, int s, int b, const int64_t st[3],
                int box_inner, int box_rows, bool swizzle128) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                        static_cast<cuuint64_t>(s > 0 ? s : 1), static_cast<cuuint64_t>(b)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                           static_cast<cuuint64_t>(st[0]) * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = dt == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(m, t, 4, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// General 4-D map over one-byte elements: dims innermost first, strides in bytes
// of dims 1..3, the given box, 128-byte swizzle.
// Box rows of box_in[0] bytes: the 128-byte swizzle, or the 64-byte one for 64-byte
// rows; swizzle = false: plain row-major boxes (the CUDA-core decode reads them so).
bool encode_map_u8(CUtensorMap* m, const void* ptr, const uint64_t dims_in[4], const int64_t strides_b[3],
                   const uint32_t box_in[4], bool swizzle = true) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4];
  for (int i = 0; i < 4; ++i) dims[i] = static_cast<cuuint64_t>(dims_in[i] > 0 ? dims_in[i] : 1);
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(strides_b[0]), static_cast<cuuint64_t>(strides_b[1]),
                           static_cast<cuuint64_t>(strides_b[2])};
  cuuint32_t box[4] = {box_in[0], box_in[1], box_in[2], box_in[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = !swizzle          ? CU_TENSOR_MAP_SWIZZLE_NONE
                                : box_in[0] == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The mask as the kernels use it: row i sees key j < skv only if
// j <= i + off (when causal) and j >= i + left_off (when local).  An edge that
// hides nothing is dropped; offsets are clamped to where every row sees nothing,
// so they fit in an int.
struct MaskPlan {
  int causal;
  int off;
  int local;
  int left_off;
};

MaskPlan plan_mask(const fa_fwd_args* a) {
  MaskPlan c{0, 0, 0, 0};
  constexpr int64_t kBig = static_cast<int64_t>(1) << 40;  // beyond any row or key index
  const int64_t sq = a->sq, skv = a->skv;
  int64_t base = a->q_pos_offset == FA_OFFSET_BOTTOM_RIGHT ? skv - sq : a->q_pos_offset;
  base = base < -kBig ? -kBig : (base > kBig ? kBig : base);
  const bool right_win = a->local && a->window_right >= 0;
  if (a->causal || right_win) {
    int64_t off = kBig;
    if (a->causal) off = base;
    if (right_win) {
      const int64_t w = a->window_right > kBig ? kBig : a->window_right;
      off = off < base + w ? off : base + w;
    }
    if (off < skv - 1) {  // otherwise row 0 already sees every key
      c.causal = 1;
      c.off = static_cast<int>(off < -sq - 1 ? -sq - 1 : off);  // below: every row sees nothing
    }
  }
  if (a->local && a->window_left >= 0) {
    const int64_t w = a->window_left > kBig ? kBig : a->window_left;
    const int64_t lo = base - w;
    if (lo + sq - 1 > 0) {  // otherwise even the last row's edge is at or before key 0
      c.local = 1;
      c.left_off = static_cast<int>(lo > skv ? skv : lo);  // above: every row sees nothing
    }
  }
  return c;
}

// One query row (sq == 1) with many query heads per KV head and no sliding
// window: Q is viewed as g rows of hkv heads, so the g query heads sharing a KV
// head become the rows of one tensor-core tile of the prefill kernel ("ai-reference-
// codex: forward CUDA kernel", 7.4; "flash attention V2 code walkthrough", the
// ngroups > 1 launch).  Smaller groups stay on the CUDA-core decode kernel: a
// 128-row tile would be mostly padding, while that kernel's arithmetic per KV
// byte grows only with g.
constexpr int kHeadRowsMinG = 8;
bool use_head_rows(const fa_fwd_args* a) {
  return a->sq == 1 && a->hq / a->hkv >= kHeadRowsMinG && !plan_mask(a).local;
}

bool use_decode_kernel(const fa_fwd_args* a) {
  return a->sq == 1 && !use_head_rows(a) && decode_supported(a->d, a->hq / a->hkv);
}

// Keys a decode row can see (sq == 1): kv_start <= j < kv_limit.
int decode_kv_limit(const fa_fwd_args* a) {
  const MaskPlan c = plan_mask(a);
  if (!c.causal) return a->skv;
  const int64_t lim = static_cast<int64_t>(c.off) + 1;
  return static_cast<int>(lim < 0 ? 0 : (lim > a->skv ? a->skv : lim));
}

int decode_kv_start(const fa_fwd_args* a) {
  const MaskPlan c = plan_mask(a);
  if (!c.local) return 0;
  const int lim = decode_kv_limit(a);
  return c.left_off < 0 ? 0 : (c.left_off > lim ? lim : c.left_off);
}

struct SplitShape {
  int64_t units;
  int64_t slots;
  int64_t nblk;
};

// Key blocks a split range is cut from, per path (host-only: no device query).
int64_t split_blocks(const fa_fwd_args* a) {
  if (use_head_rows(a)) return ceil_div64(decode_kv_limit(a), prefill_block_n(a->d));
  if (use_decode_kernel(a))
    return ceil_div64(decode_kv_limit(a), decode_block_n(a->d)) - decode_kv_start(a) / decode_block_n(a->d);
  return ceil_div64(a->skv, prefill_block_n(a->d));
}

bool split_shape(const fa_fwd_args* a, const DeviceInfo& di, SplitShape* s) {
  s->nblk = split_blocks(a);
  if (use_head_rows(a)) {
    const int g = a->hq / a->hkv;
    const int64_t n_mcta = ceil_div64(ceil_div64(g, 128), prefill_q_tiles(a->d));
    s->units = static_cast<int64_t>(a->b) * a->hkv * n_mcta;
    s->slots = di.sms;
  } else if (use_decode_kernel(a)) {
    const int g = a->hq / a->hkv;
    s->units = static_cast<int64_t>(a->b) * a->hkv * (g / decode_heads_per_cta(g));
    s->slots = static_cast<int64_t>(di.sms) * decode_ctas_per_sm(a->d, a->dtype);
  } else {
    const int nq = prefill_q_tiles(a->d);
    const int64_t n_mcta = ceil_div64(ceil_div64(a->sq, 128), nq);
    s->units = static_cast<int64_t>(a->b) * a->hq * n_mcta;
    s->slots = di.sms;
  }
  return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of g_splitkv_scratch on the current device, resolved on the
// first call for that device (with the device current) and cached.
bool noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr) return false;
    cache[dev] = p;
  }
  *out = cache[dev];
  return true;
}

// Merge counters of the fused split-KV decode: one int per (batch, query-head
// group), at most one per (batch, query head).
size_t counters_bytes(int b, int hq) { return align256(static_cast<size_t>(b) * hq * sizeof(int)); }

size_t workspace_bytes_for(const fa_fwd_args* a, int ns) {
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq * a->sq;
  return align256(rows * a->d * sizeof(float)) + align256(rows * sizeof(float)) + counters_bytes(a->b, a->hq);
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

bool strides_pos(const int64_t* s, int n) {
  for (int i = 0; i < n; ++i)
    if (s[i] <= 0) return false;
  return true;
}

fa_status validate_kvcache(const fa_kvcache_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->hq < 1 || a->hkv < 1 || a->hq % a->hkv != 0) return FA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return FA_ERR_INVALID_ARG;
  if (!softcap_ok(a->softcap)) return FA_ERR_INVALID_ARG;
  if ((a->local != 0 && a->local != 1) || (a->local && a->window_left < -1)) return FA_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128 && a->d != 256) return FA_ERR_UNSUPPORTED;
  if (a->max_seqlen_k < 0 || a->max_seqlen_k > (1 << 30) || a->num_pages < 1) return FA_ERR_INVALID_ARG;
  if (a->q == nullptr || a->k == nullptr || a->v == nullptr || a->o == nullptr || a->lse == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(a->q, 2) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 2) || !aligned(a->lse, 4))
    return FA_ERR_INVALID_ARG;
  if (!strides_pos(a->q_strides, 2) || !strides_pos(a->o_strides, 2)) return FA_ERR_INVALID_ARG;
  if (a->page_size > 0) {
    if (a->page_size % 64 != 0) return FA_ERR_UNSUPPORTED;
    if (a->block_table == nullptr || a->seqlens_k == nullptr || a->block_table_stride < 1) return FA_ERR_INVALID_ARG;
    if (!aligned(a->block_table, 4) || !aligned(a->seqlens_k, 4)) return FA_ERR_INVALID_ARG;
    if (!strides_ok(a->k_strides) || !strides_ok(a->v_strides)) return FA_ERR_INVALID_ARG;
  } else if (a->page_size == 0) {
    if (a->cu_seqlens_k == nullptr || !aligned(a->cu_seqlens_k, 4)) return FA_ERR_INVALID_ARG;
    for (int i = 1; i < 3; ++i)
      if (a->k_strides[i] <= 0 || a->k_strides[i] % 8 != 0 || a->v_strides[i] <= 0 || a->v_strides[i] % 8 != 0)
        return FA_ERR_INVALID_ARG;
  } else {
    return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

bool strides2_ok(const int64_t s[2]) {
  for (int i = 0; i < 2; ++i) {
    if (s[i] <= 0 || (s[i] % 8) != 0) return false;
    if (s[i] * 2 >= (static_cast<int64_t>(1) << 40)) return false;
  }
  return true;
}

fa_status validate_varlen(const fa_varlen_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->hq < 1 || a->hkv < 1 || a->hq % a->hkv != 0) return FA_ERR_INVALID_ARG;
  if (a->total_q < 0 || a->total_k < 0 || a->max_seqlen_q < 0) return FA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return FA_ERR_INVALID_ARG;
  if (a->local != 0 && a->local != 1) return FA_ERR_INVALID_ARG;
  if (a->local && (a->window_left < -1 || a->window_right < -1)) return FA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return FA_ERR_INVALID_ARG;
  if (!softcap_ok(a->softcap)) return FA_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128 && a->d != 256) return FA_ERR_UNSUPPORTED;
  if (a->total_q > (1 << 30) || a->total_k > (1 << 30) || a->max_seqlen_q > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (a->total_q == 0 || a->max_seqlen_q == 0) return FA_OK;
  if (a->q == nullptr || a->o == nullptr || a->lse == nullptr || a->cu_seqlens_q == nullptr ||
      a->cu_seqlens_k == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4) || !aligned(a->cu_seqlens_q, 4) ||
      !aligned(a->cu_seqlens_k, 4))
    return FA_ERR_INVALID_ARG;
  if (!strides2_ok(a->q_strides) || !strides2_ok(a->o_strides)) return FA_ERR_INVALID_ARG;
  if (a->total_k > 0) {
    if (a->k == nullptr || a->v == nullptr || !aligned(a->k, 16) || !aligned(a->v, 16)) return FA_ERR_INVALID_ARG;
    if (!strides2_ok(a->k_strides) || !strides2_ok(a->v_strides)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

// The KV-cache decode with g >= 8 query heads per KV head and no window runs
// as the heads-as-rows tile of the prefill kernel, as fa_fwd_splitkv does.
bool kvcache_head_rows(const fa_kvcache_args* a) {
  return a->hq / a->hkv >= kHeadRowsMinG && !(a->local && a->window_left >= 0);
}

int kvcache_splits(const fa_kvcache_args* a, int32_t requested, const DeviceInfo& di) {
  const int g = a->hq / a->hkv;
  int64_t units, slots, nblk;
  if (kvcache_head_rows(a)) {
    units = static_cast<int64_t>(a->b) * a->hkv * ceil_div64(ceil_div64(g, 128), prefill_q_tiles(a->d));
    slots = di.sms;
    nblk = ceil_div64(a->max_seqlen_k, prefill_block_n(a->d));
  } else {
    units = static_cast<int64_t>(a->b) * a->hkv * (g / decode_heads_per_cta(g));
    slots = static_cast<int64_t>(di.sms) * decode_ctas_per_sm(a->d, a->dtype);
    int64_t keys = a->max_seqlen_k;
    if (a->local && a->window_left >= 0 && a->window_left + 1 < keys) keys = a->window_left + 1 + decode_block_n(a->d);
    nblk = ceil_div64(keys, decode_block_n(a->d));
  }
  int ns = requested > 0 ? requested : fa_num_splits_heuristic(units, slots, nblk, kMaxSplits);
  const int64_t cap = nblk > 0 ? nblk : 1;
  if (ns > cap) ns = static_cast<int>(cap);
  return ns < 1 ? 1 : ns;
}

// A split count capped at the key blocks there are (a split with no block is
// useless) and at kMaxSplits * 8.
int cap_splits(const fa_fwd_args* a, int64_t ns) {
  const int64_t nblk = split_blocks(a);
  const int64_t cap = nblk > 0 ? nblk : 1;
  if (ns > cap) ns = cap;
  if (ns > kMaxSplits * 8) ns = kMaxSplits * 8;
  return ns < 1 ? 1 : static_cast<int>(ns);
}

int resolve_splits(const fa_fwd_args* a, int32_t requested, const DeviceInfo& di) {
  if (requested > 0) return cap_splits(a, requested);
  SplitShape s{};
  split_shape(a, di, &s);
  return cap_splits(a, fa_num_splits_heuristic(s.units, s.slots, s.nblk, kMaxSplits));
}

}  // namespace
}  // namespace fa

using namespace fa;

// KV-cache decode with the heads as rows: Q [b][hq][d] viewed as [b][g][hkv][d]
// (as in fa_fwd_splitkv), the cache read through the prefill kernel's paged or
// packed K/V loads, split partials merged by the combine kernel.
static fa_status kvcache_head_rows_run(const fa_kvcache_args* a, int ns, float* o_part, float* lse_part,
                                       const DeviceInfo& di, int32_t* splits_used, void* stream) {
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const int g = a->hq / a->hkv;
  const int bn = prefill_block_n(a->d);
  const bool paged = a->page_size > 0;
  const int64_t q_view[3] = {a->q_strides[0], a->q_strides[1], static_cast<int64_t>(g) * a->q_strides[1]};
  if (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hkv, g, a->b, q_view, 64, 128, true)) return FA_ERR_INVALID_ARG;
  // 4-D views (d, hkv, rows, outer): paged rows = page_size, outer = pages; packed rows = total_k, outer = 1
  const int64_t k_st[3] = {paged ? a->k_strides[0] : a->k_strides[1] * (a->num_pages > 0 ? a->num_pages : 1),
                           a->k_strides[1], a->k_strides[2]};
  const int64_t v_st[3] = {paged ? a->v_strides[0] : a->v_strides[1] * (a->num_pages > 0 ? a->num_pages : 1),
                           a->v_strides[1], a->v_strides[2]};
  const int rows_dim = paged ? a->page_size : a->num_pages;
  const int outer_dim = paged ? a->num_pages : 1;
  const int box_rows = (!paged || a->page_size % bn == 0) ? bn : 64;
  if (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, rows_dim, outer_dim, k_st, 64, box_rows, true) ||
      !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, rows_dim, outer_dim, v_st, 64, box_rows, true))
    return FA_ERR_INVALID_ARG;
  p.lse = lse_part;  // partials [ns][b][hkv][g] = [ns][b][hq]
  p.o_part = o_part;
  p.b = a->b;
  p.sq = g;
  p.skv = a->max_seqlen_k;
  p.hq = a->hkv;
  p.hkv = a->hkv;
  p.g = 1;
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
  p.n_mtiles = static_cast<int>(ceil_div64(g, 128));
  p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
  p.num_splits = ns;
  p.blocks_per_split = 1;  // set per sequence in the kernel
  p.max_ctas = di.sms;
  p.status = di.status;
  p.cu_k = paged ? nullptr : a->cu_seqlens_k;
  p.total_k = a->num_pages;
  p.kv_mode = paged ? kKvPaged : kKvPacked;
  p.block_table = a->block_table;
  p.bt_stride = a->block_table_stride;
  p.page_size = a->page_size;
  p.box_rows = box_rows;
  p.seqlens = a->seqlens_k;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_prefill(p, a->d, a->dtype, st) != cudaSuccess) return FA_ERR_CUDA;
  if (splits_used) *splits_used = ns;
  const int64_t o_st[3] = {a->o_strides[0], a->o_strides[1], a->o_strides[1]};  // (one row: its stride is unused)
  return fa_splitkv_combine(o_part, lse_part, ns, a->b, a->hq, 1, a->d, a->dtype, a->o, o_st, a->lse, stream);
}

extern "C" {

int32_t fa_version(void) { return 3; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape or head dimension";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more split-KV scratch than the built-in buffer holds";
    case FA_ERR_DEVICE_ARG: return "an argument read on the device (sequence offsets) failed its check";
    default: return "unknown status";
  }
}

int32_t fa_num_splits_heuristic(int64_t units, int64_t slots, int64_t num_kv_blocks, int32_t max_splits) {
  if (units <= 0 || slots <= 0) return 1;
  int64_t smax = max_splits < num_kv_blocks ? max_splits : num_kv_blocks;
  if (smax < 1) smax = 1;
  auto eff = [&](int64_t s) {
    const double w = static_cast<double>(units * s) / static_cast<double>(slots);
    return w / std::ceil(w);
  };
  double best = 0.0;
  for (int64_t s = 1; s <= smax; ++s) best = eff(s) > best ? eff(s) : best;
  for (int64_t s = 1; s <= smax; ++s)
    if (eff(s) >= 0.85 * best) return static_cast<int32_t>(s);
  return 1;
}

fa_status fa_fwd(const fa_fwd_args* a, void* stream) {
  const fa_status v = validate(a);
  if (v != FA_OK || a->sq == 0) return v;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const int bn = prefill_block_n(a->d);
  if (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hq, a->sq, a->b, a->q_strides, 64, 128, true))
    return FA_ERR_INVALID_ARG;
  if (a->skv > 0 &&
      (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->skv, a->b, a->k_strides, 64, bn, true) ||
       !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->skv, a->b, a->v_strides, 64, bn, true)))
    return FA_ERR_INVALID_ARG;
  const MaskPlan c = plan_mask(a);
  p.o = a->o;
  p.lse = a->lse;
  p.o_part = nullptr;
  p.o_stride_b = a->o_strides[0];
  p.o_stride_row = a->o_strides[1];
  p.o_stride_h = a->o_strides[2];
  p.o_vec32 = aligned(a->o, 32) && a->o_strides[0] % 16 == 0 && a->o_strides[1] % 16 == 0 &&
              a->o_strides[2] % 16 == 0;
  p.o_tma = encode_map(&p.tm_o, a->o, a->dtype, a->d, a->hq, a->sq, a->b, a->o_strides, 64, 32, true) ? 1 : 0;
  p.b = a->b;
  p.sq = a->sq;
  p.skv = a->skv;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.causal = c.causal;
  p.off = c.off;
  p.local = c.local;
  p.left_off = c.left_off;
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
  p.n_mtiles = static_cast<int>(ceil_div64(a->sq, 128));
  p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
  p.num_splits = 1;
  p.blocks_per_split = static_cast<int>(ceil_div64(a->skv, bn));
  p.max_ctas = di.sms;
  p.status = di.status;
  return from_cuda(launch_prefill(p, a->d, a->dtype, static_cast<cudaStream_t>(stream)));
}

int32_t fa_splitkv_default_splits(const fa_fwd_args* a) {
  if (validate(a) != FA_OK) return 0;
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  return resolve_splits(a, 0, di);
}

size_t fa_splitkv_workspace_size(const fa_fwd_args* a, int32_t num_splits) {
  if (validate(a) != FA_OK || num_splits < 0) return 0;
  // the split count fa_fwd_splitkv will use: a request capped at the key blocks
  // there are (no device needed), or the heuristic's
  if (num_splits > 0) return workspace_bytes_for(a, cap_splits(a, num_splits));
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  return workspace_bytes_for(a, resolve_splits(a, 0, di));
}

fa_status fa_splitkv_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t b, int32_t hq,
                             int32_t sq, int32_t d, fa_dtype dtype, void* o, const int64_t o_strides[3],
                             float* lse, void* stream) {
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (num_splits < 1 || b < 1 || hq < 1 || sq < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (sq == 0) return FA_OK;
  if (o_part == nullptr || lse_part == nullptr || o == nullptr || o_strides == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(o_part, 4) || !aligned(lse_part, 4) || !aligned(o, 2) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (o_strides[i] <= 0) return FA_ERR_INVALID_ARG;
  CombineParams p;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.o = o;
  p.o_stride_b = o_strides[0];
  p.o_stride_row = o_strides[1];
  p.o_stride_h = o_strides[2];
  p.lse = lse;
  p.num_splits = num_splits;
  p.b = b;
  p.hq = hq;
  p.sq = sq;
  p.d = d;
  return from_cuda(launch_combine(p, dtype, static_cast<cudaStream_t>(stream)));
}

fa_status fa_fwd_splitkv(const fa_fwd_args* a, int32_t num_splits, void* workspace, size_t workspace_bytes,
                         int32_t* splits_used, void* stream) {
  const fa_status v = validate(a);
  if (v != FA_OK) return v;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  if (a->sq == 0) {
    if (splits_used) *splits_used = 0;
    return FA_OK;
  }
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  const int ns = resolve_splits(a, num_splits, di);
  const size_t need = workspace_bytes_for(a, ns);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
  float* o_part = static_cast<float*>(workspace);
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq * a->sq;
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * a->d * sizeof(float)));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  cudaError_t e;
  if (use_head_rows(a)) {
    // Q viewed as [b][g rows][hkv heads][d]: row r of head kvh is query head kvh * g + r,
    // and every row sees the same keys j < kv_limit (no per-row mask)
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    const int g = a->hq / a->hkv;
    const int bn = prefill_block_n(a->d);
    const int64_t q_view[3] = {a->q_strides[0], a->q_strides[2], static_cast<int64_t>(g) * a->q_strides[2]};
    if (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hkv, g, a->b, q_view, 64, 128, true)) return FA_ERR_INVALID_ARG;
    if (a->skv > 0 &&
        (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->skv, a->b, a->k_strides, 64, bn, true) ||
         !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->skv, a->b, a->v_strides, 64, bn, true)))
      return FA_ERR_INVALID_ARG;
    const int lim = decode_kv_limit(a);
    if (ns == 1) {
      // one split: the kernel writes O and LSE itself, through the same view of O
      // (LSE [b][hkv][g] is [b][hq][1])
      p.o = a->o;
      p.lse = a->lse;
      p.o_stride_b = a->o_strides[0];
      p.o_stride_row = a->o_strides[2];
      p.o_stride_h = static_cast<int64_t>(g) * a->o_strides[2];
      p.o_vec32 = aligned(a->o, 32) && a->o_strides[0] % 16 == 0 && a->o_strides[2] % 16 == 0;
    } else {
      p.lse = lse_part;  // partials [ns][b][hkv][g] = [ns][b][hq]: the layout the combine reads
      p.o_part = o_part;
    }
    p.b = a->b;
    p.sq = g;
    p.skv = lim;
    p.hq = a->hkv;
    p.hkv = a->hkv;
    p.g = 1;
    p.scale_log2 = scale_log2;
    softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
    p.n_mtiles = static_cast<int>(ceil_div64(g, 128));
    p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
    p.num_splits = ns;
    const int64_t nblk = ceil_div64(lim, bn);
    p.blocks_per_split = static_cast<int>(ceil_div64(nblk > 0 ? nblk : 1, ns));
    p.max_ctas = di.sms;
    p.status = di.status;
    e = launch_prefill(p, a->d, a->dtype, st);
    if (ns == 1) {
      if (e != cudaSuccess) return FA_ERR_CUDA;
      if (splits_used) *splits_used = 1;
      return FA_OK;
    }
  } else if (use_decode_kernel(a)) {
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    const int bn = decode_block_n(a->d);
    if (a->skv > 0 &&
        (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->skv, a->b, a->k_strides, a->d, bn, false) ||
         !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->skv, a->b, a->v_strides, a->d, bn, false)))
      return FA_ERR_INVALID_ARG;
    p.q = a->q;
    p.q_stride_b = a->q_strides[0];
    p.q_stride_h = a->q_strides[2];
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.b = a->b;
    p.skv = a->skv;
    p.hq = a->hq;
    p.hkv = a->hkv;
    p.g = a->hq / a->hkv;
    p.kv_limit = decode_kv_limit(a);
    p.kv_start = decode_kv_start(a);
    p.window_left = -1;
    p.nblk = static_cast<int>(ceil_div64(p.kv_limit, bn));
    p.num_splits = ns;
    const int span = p.nblk - p.kv_start / bn;
    p.blocks_per_split = static_cast<int>(ceil_div64(span > 0 ? span : 1, ns));
    p.scale_log2 = scale_log2;
    softcap_consts(a->softcap, 1.0 / 1.4426950408889634, &p.sc_k, &p.sc_b);  // (scores arrive times scale log2 e)
    p.status = di.status;
    p.box_rows = bn;
    p.counters = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(lse_part) + align256(rows * sizeof(float)));
    p.o = a->o;
    p.o_stride_b = a->o_strides[0];
    p.o_stride_h = a->o_strides[2];
    p.lse = a->lse;
    e = cudaMemsetAsync(p.counters, 0, counters_bytes(a->b, a->hq), st);
    if (e == cudaSuccess) e = launch_decode(p, a->d, a->dtype, st);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (splits_used) *splits_used = ns;
    return FA_OK;  // the decode kernel merges the splits itself
  } else if (ns == 1) {
    // one split is the plain forward (the kernel writes O and LSE itself)
    if (splits_used) *splits_used = 1;
    return fa_fwd(a, stream);
  } else {
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    const int bn = prefill_block_n(a->d);
    if (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hq, a->sq, a->b, a->q_strides, 64, 128, true))
      return FA_ERR_INVALID_ARG;
    if (a->skv > 0 &&
        (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->skv, a->b, a->k_strides, 64, bn, true) ||
         !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->skv, a->b, a->v_strides, 64, bn, true)))
      return FA_ERR_INVALID_ARG;
    const MaskPlan c = plan_mask(a);
    p.o = nullptr;
    p.lse = lse_part;
    p.o_part = o_part;
    p.b = a->b;
    p.sq = a->sq;
    p.skv = a->skv;
    p.hq = a->hq;
    p.hkv = a->hkv;
    p.g = a->hq / a->hkv;
    p.causal = c.causal;
    p.off = c.off;
    p.local = c.local;
    p.left_off = c.left_off;
    p.scale_log2 = scale_log2;
    softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
    p.n_mtiles = static_cast<int>(ceil_div64(a->sq, 128));
    p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
    p.num_splits = ns;
    const int64_t nblk = ceil_div64(a->skv, bn);
    p.blocks_per_split = static_cast<int>(ceil_div64(nblk > 0 ? nblk : 1, ns));
    p.max_ctas = di.sms;
    p.status = di.status;
    e = launch_prefill(p, a->d, a->dtype, st);
  }
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (splits_used) *splits_used = ns;
  return fa_splitkv_combine(o_part, lse_part, ns, a->b, a->hq, a->sq, a->d, a->dtype, a->o, a->o_strides, a->lse,
                            stream);
}

fa_status fa_fwd_splitkv_noalloc(const fa_fwd_args* a, int32_t num_splits, int32_t* splits_used, void* stream) {
  const fa_status v = validate(a);
  if (v != FA_OK) return v;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  if (a->sq == 0) {
    if (splits_used) *splits_used = 0;
    return FA_OK;
  }
  // the same split count and workspace layout fa_fwd_splitkv would use
  const size_t need = fa_splitkv_workspace_size(a, num_splits);
  if (need == 0) return FA_ERR_CUDA;
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (!noalloc_scratch(&scratch)) return FA_ERR_CUDA;
  return fa_fwd_splitkv(a, num_splits, scratch, FA_NOALLOC_SCRATCH_BYTES, splits_used, stream);
}

fa_status fa_fwd_kvcache(const fa_kvcache_args* a, int32_t num_splits, void* workspace, size_t workspace_bytes,
                         int32_t* splits_used, void* stream) {
  const fa_status v = validate_kvcache(a);
  if (v != FA_OK) return v;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  const int ns = kvcache_splits(a, num_splits, di);
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq;
  const size_t need = align256(rows * a->d * sizeof(float)) + align256(rows * sizeof(float)) + counters_bytes(a->b, a->hq);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * a->d * sizeof(float)));
  if (kvcache_head_rows(a)) return kvcache_head_rows_run(a, ns, o_part, lse_part, di, splits_used, stream);
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  const int bn = decode_block_n(a->d);
  const bool paged = a->page_size > 0;
  // 4-D views (d, hkv, rows, outer): paged rows = page_size, outer = pages; packed rows = total_k, outer = 1
  const int64_t k_st[3] = {paged ? a->k_strides[0] : a->k_strides[1] * (a->num_pages > 0 ? a->num_pages : 1),
                           a->k_strides[1], a->k_strides[2]};
  const int64_t v_st[3] = {paged ? a->v_strides[0] : a->v_strides[1] * (a->num_pages > 0 ? a->num_pages : 1),
                           a->v_strides[1], a->v_strides[2]};
  const int rows_dim = paged ? a->page_size : a->num_pages;
  const int outer_dim = paged ? a->num_pages : 1;
  // a block of bn keys is loaded as boxes that never straddle a page
  const int box_rows = (!paged || a->page_size % bn == 0) ? bn : 64;
  if (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, rows_dim, outer_dim, k_st, a->d, box_rows, false) ||
      !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, rows_dim, outer_dim, v_st, a->d, box_rows, false))
    return FA_ERR_INVALID_ARG;
  p.q = a->q;
  p.q_stride_b = a->q_strides[0];
  p.q_stride_h = a->q_strides[1];
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.b = a->b;
  p.skv = a->max_seqlen_k;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.kv_limit = 0;
  p.kv_start = 0;
  p.window_left = a->local ? a->window_left : -1;
  p.nblk = static_cast<int>(ceil_div64(a->max_seqlen_k, bn));
  p.num_splits = ns;
  p.blocks_per_split = 1;  // set per sequence in the kernel
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  softcap_consts(a->softcap, 1.0 / 1.4426950408889634, &p.sc_k, &p.sc_b);  // (scores arrive times scale log2 e)
  p.status = di.status;
  p.kv_mode = paged ? kKvPaged : kKvPacked;
  p.block_table = a->block_table;
  p.bt_stride = a->block_table_stride;
  p.page_size = a->page_size;
  p.box_rows = box_rows;
  p.seqlens = a->seqlens_k;
  p.cu_seqlens = a->cu_seqlens_k;
  p.total_k = a->num_pages;
  p.counters = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(lse_part) + align256(rows * sizeof(float)));
  p.o = a->o;
  p.o_stride_b = a->o_strides[0];
  p.o_stride_h = a->o_strides[1];
  p.lse = a->lse;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.counters, 0, counters_bytes(a->b, a->hq), st) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_decode(p, a->d, a->dtype, st) != cudaSuccess) return FA_ERR_CUDA;
  if (splits_used) *splits_used = ns;
  return FA_OK;  // the decode kernel merges the splits itself
}

size_t fa_kvcache_workspace_size(const fa_kvcache_args* a, int32_t num_splits) {
  if (validate_kvcache(a) != FA_OK || num_splits < 0) return 0;
  DeviceInfo di;
  if (num_splits == 0 && !device_info(&di)) return 0;
  const int ns = num_splits > 0 ? num_splits : kvcache_splits(a, 0, di);
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq;
  return align256(rows * a->d * sizeof(float)) + align256(rows * sizeof(float)) + counters_bytes(a->b, a->hq);
}

fa_status fa_fwd_varlen(const fa_varlen_args* a, void* stream) {
  const fa_status v = validate_varlen(a);
  if (v != FA_OK || a->total_q == 0 || a->max_seqlen_q == 0) return v;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const int bn = prefill_block_n(a->d);
  // 4-D views (d, h, total, 1) of the packed tensors
  auto st3 = [](const int64_t s2[2], int64_t total) {
    return std::array<int64_t, 3>{s2[0] * (total > 0 ? total : 1), s2[0], s2[1]};
  };
  const auto qs = st3(a->q_strides, a->total_q);
  if (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hq, a->total_q, 1, qs.data(), 64, 128, true))
    return FA_ERR_INVALID_ARG;
  if (a->total_k > 0) {
    const auto ks = st3(a->k_strides, a->total_k), vs = st3(a->v_strides, a->total_k);
    if (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->total_k, 1, ks.data(), 64, bn, true) ||
        !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->total_k, 1, vs.data(), 64, bn, true))
      return FA_ERR_INVALID_ARG;
  }
  // Mask edges relative to each sequence's diagonal (the kernel adds skv - sq).
  constexpr int64_t kEdge = static_cast<int64_t>(1) << 30;
  p.causal = 0;
  p.off = 0;
  if (a->causal || (a->local && a->window_right >= 0)) {
    int64_t off = kEdge;
    if (a->causal) off = 0;
    if (a->local && a->window_right >= 0 && a->window_right < off) off = a->window_right;
    p.causal = 1;
    p.off = static_cast<int>(off);
  }
  if (a->local && a->window_left >= 0) {
    p.local = 1;
    p.left_off = static_cast<int>(-(a->window_left < kEdge ? a->window_left : kEdge));
  }
  p.o = a->o;
  p.lse = a->lse;
  p.o_stride_b = 0;
  p.o_stride_row = a->o_strides[0];
  p.o_stride_h = a->o_strides[1];
  p.o_vec32 = aligned(a->o, 32) && a->o_strides[0] % 16 == 0 && a->o_strides[1] % 16 == 0;
  {
    const auto os = st3(a->o_strides, a->total_q);
    p.o_tma = encode_map(&p.tm_o, a->o, a->dtype, a->d, a->hq, a->total_q, 1, os.data(), 64, 32, true) ? 1 : 0;
  }
  p.b = a->b;
  p.sq = a->max_seqlen_q;
  p.skv = 0;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
  p.n_mtiles = static_cast<int>(ceil_div64(a->max_seqlen_q, 128));
  p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
  p.num_splits = 1;
  p.blocks_per_split = 0;
  p.max_ctas = di.sms;
  p.status = di.status;
  p.cu_q = a->cu_seqlens_q;
  p.cu_k = a->cu_seqlens_k;
  p.total_q = a->total_q;
  p.total_k = a->total_k;
  return from_cuda(launch_prefill(p, a->d, a->dtype, static_cast<cudaStream_t>(stream)));
}

namespace {

// The forward description of a backward problem (validation and the mask plan are shared).
fa_fwd_args fwd_view(const fa_bwd_args* a) {
  fa_fwd_args f;
  std::memset(&f, 0, sizeof(f));
  f.dtype = a->dtype;
  f.b = a->b;
  f.sq = a->sq;
  f.skv = a->skv;
  f.hq = a->hq;
  f.hkv = a->hkv;
  f.d = a->d;
  f.q = a->q;
  f.k = a->k;
  f.v = a->v;
  f.o = const_cast<void*>(a->o);
  f.lse = const_cast<float*>(a->lse);
  for (int i = 0; i < 3; ++i) {
    f.q_strides[i] = a->q_strides[i];
    f.k_strides[i] = a->k_strides[i];
    f.v_strides[i] = a->v_strides[i];
    f.o_strides[i] = a->o_strides[i];
  }
  f.causal = a->causal;
  f.q_pos_offset = a->q_pos_offset;
  f.scale = a->scale;
  f.local = a->local;
  f.window_left = a->window_left;
  f.window_right = a->window_right;
  f.softcap = a->softcap;
  return f;
}

fa_status validate_bwd(const fa_bwd_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  const fa_fwd_args f = fwd_view(a);
  const fa_status v = validate(&f);
  if (v != FA_OK) return v;
  if (!bwd_supported(a->d)) return FA_ERR_UNSUPPORTED;
  if (a->sq == 0 && a->skv == 0) return FA_OK;
  if (a->sq > 0) {
    if (a->dout == nullptr || a->dq == nullptr || !aligned(a->dout, 16) || !aligned(a->dq, 16))
      return FA_ERR_INVALID_ARG;
    if (!strides_ok(a->do_strides) || !strides_ok(a->dq_strides)) return FA_ERR_INVALID_ARG;
  }
  if (a->skv > 0) {
    if (a->dk == nullptr || a->dv == nullptr || !aligned(a->dk, 16) || !aligned(a->dv, 16))
      return FA_ERR_INVALID_ARG;
    if (!strides_ok(a->dk_strides) || !strides_ok(a->dv_strides)) return FA_ERR_INVALID_ARG;
    if (a->sq == 0 && (a->k == nullptr || a->v == nullptr)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

size_t bwd_workspace_bytes(const fa_bwd_args* a) {
  const size_t rows = static_cast<size_t>(a->b) * a->hq * static_cast<size_t>(ceil_div64(a->sq, 128) * 128);
  return 2 * align256(rows * sizeof(float));
}

}  // namespace

size_t fa_bwd_workspace_size(const fa_bwd_args* a) {
  if (validate_bwd(a) != FA_OK) return 0;
  const size_t w = bwd_workspace_bytes(a);
  return w > 0 ? w : 256;
}

fa_status fa_bwd(const fa_bwd_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  const fa_status v = validate_bwd(a);
  if (v != FA_OK) return v;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a->sq == 0 && a->skv == 0) return FA_OK;  // (sq == 0 alone: the dK / dV kernel writes zeros)
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  const size_t need = bwd_workspace_bytes(a);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return FA_ERR_INVALID_ARG;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const fa_fwd_args f = fwd_view(a);
  if (a->sq > 0 &&
      (!encode_map(&p.tm_q, a->q, a->dtype, a->d, a->hq, a->sq, a->b, a->q_strides, 64, 128, true) ||
       !encode_map(&p.tm_do, a->dout, a->dtype, a->d, a->hq, a->sq, a->b, a->do_strides, 64, 128, true)))
    return FA_ERR_INVALID_ARG;
  if (a->skv > 0 &&
      (!encode_map(&p.tm_k, a->k, a->dtype, a->d, a->hkv, a->skv, a->b, a->k_strides, 64, 128, true) ||
       !encode_map(&p.tm_v, a->v, a->dtype, a->d, a->hkv, a->skv, a->b, a->v_strides, 64, 128, true)))
    return FA_ERR_INVALID_ARG;
  const MaskPlan c = plan_mask(&f);
  p.o = a->o;
  p.dout = a->dout;
  p.lse = a->lse;
  p.dq = a->dq;
  p.dk = a->dk;
  p.dv = a->dv;
  for (int i = 0; i < 3; ++i) {
    p.o_st[i] = a->o_strides[i];
    p.do_st[i] = a->do_strides[i];
    p.dq_st[i] = a->dq_strides[i];
    p.dk_st[i] = a->dk_strides[i];
    p.dv_st[i] = a->dv_strides[i];
  }
  p.b = a->b;
  p.sq = a->sq;
  p.skv = a->skv;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.n_mtiles = static_cast<int>(ceil_div64(a->sq, 128));
  p.n_ntiles = static_cast<int>(ceil_div64(a->skv, 128));
  p.sq_pad = p.n_mtiles * 128;
  {
    // dQ grid: as many (batch, query head) pairs per group as keep their K and V
    // within about 32 MiB (a quarter of L2), whole KV-head groups where possible
    const int64_t kv_bytes_per_kv_head = 2 * static_cast<int64_t>(a->skv) * a->d * 2;
    const int g = a->hq / a->hkv;
    int64_t heads = kv_bytes_per_kv_head > 0 ? (int64_t{32} << 20) / kv_bytes_per_kv_head * g : g;
    heads = heads < g ? g : heads - heads % g;
    const int64_t bh = static_cast<int64_t>(a->b) * a->hq;
    p.head_group = static_cast<int>(heads > bh ? bh : heads);
  }
  p.causal = c.causal;
  p.off = c.off;
  p.local = c.local;
  p.left_off = c.left_off;
  p.scale = a->scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  softcap_consts(a->softcap, a->scale, &p.sc_k, &p.sc_b);
  const size_t rows = static_cast<size_t>(a->b) * a->hq * p.sq_pad;
  p.dpre = static_cast<float*>(workspace);
  p.l2pre = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * sizeof(float)));
  p.status = di.status;
  return from_cuda(launch_bwd(p, a->d, a->dtype, st));
}

namespace {

bool strides16_ok(const int64_t s[3]) {
  for (int i = 0; i < 3; ++i) {
    if (s[i] <= 0 || (s[i] % 16) != 0) return false;
    if (s[i] >= (static_cast<int64_t>(1) << 40)) return false;
  }
  return true;
}

fa_status validate_quant(const fa_quant_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->s < 0 || a->h < 1) return FA_ERR_INVALID_ARG;
  if ((a->transpose != 0 && a->transpose != 1) || (a->per_head != 0 && a->per_head != 1)) return FA_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128 && a->d != 256) return FA_ERR_UNSUPPORTED;
  if (a->s > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (a->s == 0) return FA_OK;
  if (a->x == nullptr || a->out == nullptr || a->descale == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a->x, 16) || !aligned(a->out, 16) || !aligned(a->descale, 4)) return FA_ERR_INVALID_ARG;
  if (!strides_ok(a->x_strides) || !strides16_ok(a->out_strides)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status validate_e4m3(const fa_fwd_e4m3_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->sq < 0 || a->skv < 0 || a->hq < 1 || a->hkv < 1 || a->hq % a->hkv != 0)
    return FA_ERR_INVALID_ARG;
  if ((a->causal != 0 && a->causal != 1) || (a->local != 0 && a->local != 1)) return FA_ERR_INVALID_ARG;
  if (a->local && (a->window_left < -1 || a->window_right < -1)) return FA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return FA_ERR_INVALID_ARG;
  if (!prefill_e4m3_supported(a->d)) return FA_ERR_UNSUPPORTED;
  if (a->sq > (1 << 30) || a->skv > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (a->sq == 0) return FA_OK;
  if (a->q == nullptr || a->o == nullptr || a->lse == nullptr || a->q_descale == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4) || !aligned(a->q_descale, 4))
    return FA_ERR_INVALID_ARG;
  if (!strides16_ok(a->q_strides) || !strides_ok(a->o_strides)) return FA_ERR_INVALID_ARG;
  if (a->skv > 0) {
    if (a->k == nullptr || a->vt == nullptr || a->k_descale == nullptr || a->v_descale == nullptr)
      return FA_ERR_INVALID_ARG;
    if (!aligned(a->k, 16) || !aligned(a->vt, 16) || !aligned(a->k_descale, 4) || !aligned(a->v_descale, 4))
      return FA_ERR_INVALID_ARG;
    if (!strides16_ok(a->k_strides) || !strides16_ok(a->vt_strides)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

}  // namespace

fa_status fa_quantize_e4m3(const fa_quant_args* a, void* stream) {
  const fa_status v = validate_quant(a);
  if (v != FA_OK || a->s == 0) return v;
  QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.x = a->x;
  p.out = a->out;
  p.descale = a->descale;
  for (int i = 0; i < 3; ++i) {
    p.x_st[i] = a->x_strides[i];
    p.out_st[i] = a->out_strides[i];
  }
  p.b = a->b;
  p.s = a->s;
  p.h = a->h;
  p.d = a->d;
  p.nblk = static_cast<int>(ceil_div64(a->s, 128));
  p.transpose = a->transpose;
  p.per_head = a->per_head;
  return from_cuda(launch_quant_e4m3(p, a->dtype, static_cast<cudaStream_t>(stream)));
}

fa_status fa_fwd_e4m3(const fa_fwd_e4m3_args* a, void* stream) {
  const fa_status v = validate_e4m3(a);
  if (v != FA_OK || a->sq == 0) return v;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  {
    const uint64_t qd[4] = {static_cast<uint64_t>(a->d), static_cast<uint64_t>(a->hq), static_cast<uint64_t>(a->sq),
                            static_cast<uint64_t>(a->b)};
    const int64_t qs[3] = {a->q_strides[2], a->q_strides[1], a->q_strides[0]};
    // one 128-row tile in chunks of up to 128 bytes per row (64 for d = 64)
    const uint32_t box[4] = {static_cast<uint32_t>(a->d < 128 ? a->d : 128), 1, 128, 1};
    if (!encode_map_u8(&p.tm_q, a->q, qd, qs, box)) return FA_ERR_INVALID_ARG;
  }
  if (a->skv > 0) {
    const uint64_t kd[4] = {static_cast<uint64_t>(a->d), static_cast<uint64_t>(a->hkv), static_cast<uint64_t>(a->skv),
                            static_cast<uint64_t>(a->b)};
    const int64_t ks[3] = {a->k_strides[2], a->k_strides[1], a->k_strides[0]};
    // V transposed: dims (key, d-row, head, batch)
    const uint64_t vd[4] = {static_cast<uint64_t>(a->skv), static_cast<uint64_t>(a->d), static_cast<uint64_t>(a->hkv),
                            static_cast<uint64_t>(a->b)};
    const int64_t vs[3] = {a->vt_strides[2], a->vt_strides[1], a->vt_strides[0]};
    const uint32_t kbox[4] = {static_cast<uint32_t>(a->d < 128 ? a->d : 128), 1, 128, 1};
    const uint32_t vbox[4] = {128, static_cast<uint32_t>(a->d), 1, 1};  // 128 keys of every d-row
    if (!encode_map_u8(&p.tm_k, a->k, kd, ks, kbox) || !encode_map_u8(&p.tm_v, a->vt, vd, vs, vbox))
      return FA_ERR_INVALID_ARG;
  }
  fa_fwd_args f;
  std::memset(&f, 0, sizeof(f));
  f.sq = a->sq;
  f.skv = a->skv;
  f.causal = a->causal;
  f.q_pos_offset = a->q_pos_offset;
  f.local = a->local;
  f.window_left = a->window_left;
  f.window_right = a->window_right;
  const MaskPlan c = plan_mask(&f);
  p.o = a->o;
  p.lse = a->lse;
  p.o_stride_b = a->o_strides[0];
  p.o_stride_row = a->o_strides[1];
  p.o_stride_h = a->o_strides[2];
  p.o_vec32 = aligned(a->o, 32) && a->o_strides[0] % 16 == 0 && a->o_strides[1] % 16 == 0 &&
              a->o_strides[2] % 16 == 0;
  p.o_tma = encode_map(&p.tm_o, a->o, FA_BF16, a->d, a->hq, a->sq, a->b, a->o_strides, 64, 32, true) ? 1 : 0;
  p.b = a->b;
  p.sq = a->sq;
  p.skv = a->skv;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.causal = c.causal;
  p.off = c.off;
  p.local = c.local;
  p.left_off = c.left_off;
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  p.n_mtiles = static_cast<int>(ceil_div64(a->sq, 128));
  p.n_mcta = static_cast<int>(ceil_div64(p.n_mtiles, prefill_q_tiles(a->d)));
  p.num_splits = 1;
  p.blocks_per_split = static_cast<int>(ceil_div64(a->skv, 128));
  p.max_ctas = di.sms;
  p.status = di.status;
  p.q_descale = a->q_descale;
  p.k_descale = a->k_descale;
  p.v_descale = a->v_descale;
  p.n_kblocks = static_cast<int>(ceil_div64(a->skv, 128));
  return from_cuda(launch_prefill_e4m3(p, a->d, static_cast<cudaStream_t>(stream)));
}

namespace {

fa_status validate_splitkv_e4m3(const fa_splitkv_e4m3_args* a) {
  if (a == nullptr) return FA_ERR_INVALID_ARG;
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (a->b < 1 || a->skv < 0 || a->hq < 1 || a->hkv < 1 || a->hq % a->hkv != 0) return FA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return FA_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128) return FA_ERR_UNSUPPORTED;
  if (a->skv > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (a->q == nullptr || a->o == nullptr || a->lse == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4)) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < 2; ++i)
    if (a->q_strides[i] <= 0 || a->q_strides[i] % 8 != 0 || a->o_strides[i] <= 0 || a->o_strides[i] % 8 != 0)
      return FA_ERR_INVALID_ARG;
  if (a->skv > 0) {
    if (a->k == nullptr || a->v == nullptr || a->k_descale == nullptr || a->v_descale == nullptr)
      return FA_ERR_INVALID_ARG;
    if (!aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->k_descale, 4) || !aligned(a->v_descale, 4))
      return FA_ERR_INVALID_ARG;
    if (!strides16_ok(a->k_strides) || !strides16_ok(a->v_strides)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

// Split count of the e4m3 decode: the heuristic over its CTAs (a group of up to 4
// query heads of one KV head each) and resident slots, or the request, capped at
// the key blocks there are.
int splitkv_e4m3_splits(const fa_splitkv_e4m3_args* a, int32_t requested, const DeviceInfo* di) {
  const int bn = decode_e4m3_block_n();
  const int64_t nblk = ceil_div64(a->skv, bn);
  int64_t ns = requested;
  if (ns <= 0) {
    if (di == nullptr) return 1;
    const int g = a->hq / a->hkv;
    const int64_t units = static_cast<int64_t>(a->b) * a->hkv * (g / decode_heads_per_cta(g));
    ns = fa_num_splits_heuristic(units, di->sms, nblk, kMaxSplits);
  }
  const int64_t cap = nblk > 0 ? nblk : 1;
  if (ns > cap) ns = cap;
  if (ns > kMaxSplits * 8) ns = kMaxSplits * 8;
  return ns < 1 ? 1 : static_cast<int>(ns);
}

size_t splitkv_e4m3_ws_bytes(const fa_splitkv_e4m3_args* a, int ns) {
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq;
  return align256(rows * a->d * sizeof(float)) + align256(rows * sizeof(float)) + counters_bytes(a->b, a->hq);
}

}  // namespace

size_t fa_splitkv_e4m3_workspace_size(const fa_splitkv_e4m3_args* a, int32_t num_splits) {
  if (validate_splitkv_e4m3(a) != FA_OK || num_splits < 0) return 0;
  if (num_splits > 0) return splitkv_e4m3_ws_bytes(a, splitkv_e4m3_splits(a, num_splits, nullptr));
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  return splitkv_e4m3_ws_bytes(a, splitkv_e4m3_splits(a, 0, &di));
}

fa_status fa_fwd_splitkv_e4m3(const fa_splitkv_e4m3_args* a, int32_t num_splits, void* workspace,
                              size_t workspace_bytes, int32_t* splits_used, void* stream) {
  const fa_status v = validate_splitkv_e4m3(a);
  if (v != FA_OK) return v;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  const int ns = splitkv_e4m3_splits(a, num_splits, &di);
  const size_t need = splitkv_e4m3_ws_bytes(a, ns);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(ns) * a->b * a->hq;
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  const int bn = decode_e4m3_block_n();
  if (a->skv > 0) {
    // (d, hkv, rows, batch) views of K and V, one plain box of bn rows of d bytes
    const uint64_t dims[4] = {static_cast<uint64_t>(a->d), static_cast<uint64_t>(a->hkv),
                              static_cast<uint64_t>(a->skv), static_cast<uint64_t>(a->b)};
    const int64_t ks[3] = {a->k_strides[2], a->k_strides[1], a->k_strides[0]};
    const int64_t vs[3] = {a->v_strides[2], a->v_strides[1], a->v_strides[0]};
    const uint32_t box[4] = {static_cast<uint32_t>(a->d), 1, static_cast<uint32_t>(bn), 1};
    if (!encode_map_u8(&p.tm_k, a->k, dims, ks, box, false) || !encode_map_u8(&p.tm_v, a->v, dims, vs, box, false))
      return FA_ERR_INVALID_ARG;
  }
  p.q = a->q;
  p.q_stride_b = a->q_strides[0];
  p.q_stride_h = a->q_strides[1];
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * a->d * sizeof(float)));
  p.b = a->b;
  p.skv = a->skv;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.g = a->hq / a->hkv;
  p.kv_limit = a->skv;
  p.kv_start = 0;
  p.window_left = -1;
  p.nblk = static_cast<int>(ceil_div64(a->skv, bn));
  p.num_splits = ns;
  p.blocks_per_split = static_cast<int>(ceil_div64(p.nblk > 0 ? p.nblk : 1, ns));
  p.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
  p.status = di.status;
  p.kv_mode = kKvDense;
  p.box_rows = bn;
  p.counters = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(p.lse_part) + align256(rows * sizeof(float)));
  p.o = a->o;
  p.o_stride_b = a->o_strides[0];
  p.o_stride_h = a->o_strides[1];
  p.lse = a->lse;
  p.k_descale = a->k_descale;
  p.v_descale = a->v_descale;
  p.n_kblocks = p.nblk;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(p.counters, 0, counters_bytes(a->b, a->hq), st);
  if (e == cudaSuccess) e = launch_decode_e4m3(p, a->d, a->dtype, st);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (splits_used) *splits_used = ns;
  return FA_OK;
}

fa_status fa_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, di.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (code != 0) {
    const int zero = 0;
    if (cudaMemcpy(di.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return code == kErrDeviceArg ? FA_ERR_DEVICE_ARG : FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(void* stream) {
  DeviceInfo di;
  if (!device_info(&di)) return FA_ERR_CUDA;
  return from_cuda(launch_wait_selftest(di.status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
