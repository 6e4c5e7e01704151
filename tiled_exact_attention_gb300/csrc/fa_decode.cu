// Split-KV decode (one query row per head) and the LSE-weighted combine.
//
// Decode reads the whole KV cache once and does a few flops per byte, so it is
// bound by HBM bandwidth, not by the tensor cores: it runs on the CUDA cores.
// Following "ai-reference-codex: forward CUDA kernel", section 7:
//  * 7.4: the g = hq / hkv query heads that share one KV head are folded into
//    one CTA, so each K/V byte is read once for the whole group;
//  * 7.1-7.2: the KV range is cut into num_splits contiguous block ranges, one
//    CTA each, so that the grid fills the GPU;
//  * 7.3: each split writes its normalised partial output and its LSE (-inf for
//    a split with no visible key); the partials are merged with weights
//    e^(LSE_s - LSE).  Here the merge is fused into the split kernel: the last
//    CTA of a (batch, head group) to finish, found with one atomic counter per
//    group, merges all splits' partials (still in L2) into O and LSE, so no
//    second launch waits on the tail of the first.  fa_combine_kernel keeps the
//    same merge as a kernel of its own for the multi-row split path.
// K/V blocks stream through a shared-memory ring filled by TMA; eight compute
// warps each take 8 rows of every block and keep their own running (m, l, o)
// per head (packed f32x2 FMAs), merged across warps at the end of the split.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kDecWarps = 8;        // compute warps
constexpr int kDecSubRows = 64;     // rows of the smallest TMA box (a 64-key page)

// E8: e4m3 K and V (one byte per element), 128-key blocks so that each block has
// one K scale (the quantiser's 128-row blocks).
template <int D, bool E8 = false>
struct DecCfg {
  static constexpr int ELT = E8 ? 1 : 2;  // bytes per K / V element
  // keys per ring stage: the larger the TMA boxes, the closer the stream gets to
  // the copy bandwidth (128-key stages measured 10% faster than 64-key ones at
  // d = 128); d = 256 keeps 64 so that three stages still fit
  static constexpr int BN = (D == 256 && !E8) ? 64 : 128;
  static constexpr int STAGES = E8 ? ((D == 128) ? 6 : 12) : (D == 256) ? 3 : (D == 128) ? 3 : 6;
  static constexpr int ROWS_PER_WARP = BN / kDecWarps;
  static constexpr int KV_BYTES = BN * D * ELT;          // one K or V block
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  // two compute warpgroups + one control warpgroup (producer and three idle
  // warps) so that registers can move to the compute warps: launched at 168 per
  // thread, control drops to 40 and compute rises to 232 (256 * 232 + 128 * 40
  // = 384 * 168)
  static constexpr int THREADS = 32 * (kDecWarps + 4);
  static constexpr int PRODUCER_WARP = kDecWarps;
  static constexpr int REG_COMPUTE = 232;
  static constexpr int REG_CONTROL = 40;
};

template <int D, int G, bool E8 = false>
struct DecLane {
  static_assert(G == 1 || G == 2 || G == 4, "heads per CTA");
  static constexpr int DPL = 16;                  // head dims per lane
  static constexpr int ESEG = E8 ? 16 : 8;        // elements per 16-byte segment
  static constexpr int SEG = DPL / ESEG;          // 16-byte segments per lane
  static constexpr int LPR = D / DPL;             // lanes per key row
  static constexpr int RPP = 32 / LPR;            // key rows per pass
  static constexpr int PASSES = DecCfg<D, E8>::ROWS_PER_WARP / RPP;
  static_assert(LPR <= 32 && 32 % LPR == 0, "lane layout");
  static_assert(PASSES >= 1, "rows per warp");
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

// Sixteen e4m3 values (element 0 in the lowest byte) to fp32, exactly: each byte
// pair widens to an f16 pair (every e4m3 value is an f16 value), then to fp32.
__device__ __forceinline__ void unpack16_e4m3(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint16_t pr = static_cast<uint16_t>(w[i] >> (16 * j));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pr));
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      f[4 * i + 2 * j] = x.x;
      f[4 * i + 2 * j + 1] = x.y;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t idx) {
  const uint16_t u = static_cast<const uint16_t*>(base)[idx];
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  } else {
    return __half2float(__ushort_as_half(u));
  }
}

enum : int { kSiteDecEmpty = 16, kSiteDecFull, kSiteDecDrain };

template <int D, int G, bool BF16, bool SC, bool E8>
__device__ __forceinline__ void compute_split(const DecodeParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                              float* red, int* flags, int warp, int lane, int split, int bi, int kvh,
                                              int h_first, int blk_lo, int nb, int start, int limit);

// Dynamic shared memory: the K/V ring, its barriers, the cross-warp merge buffer
// [warps][G][D + 2] and two flag words (abort, merging CTA).
template <int D, int G, bool E8 = false>
constexpr int dec_smem_bytes() {
  return DecCfg<D, E8>::STAGES * DecCfg<D, E8>::STAGE_BYTES + 2 * DecCfg<D, E8>::STAGES * 8 +
         kDecWarps * G * (D + 2) * 4 + 16 + 128;
}

// SC: softcap, each score capped to c tanh(s / c) before the mask.
// Keys of sequence k of a KV cache (clamped at 0).
__device__ __forceinline__ int cache_seq_len(const DecodeParams& p, int k) {
  const int n = p.kv_mode == kKvPaged ? p.seqlens[k] : p.cu_seqlens[k + 1] - p.cu_seqlens[k];
  return n > 0 ? n : 0;
}

// CACHE: a paged or packed KV cache (p.kv_mode), a separate instantiation so that
// the dense kernel keeps its code.
template <int D, int G, bool BF16, bool SC, bool CACHE, bool E8 = false>
__global__ void __launch_bounds__(DecCfg<D, E8>::THREADS, 1) fa_decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecCfg<D, E8>;
  using L = DecLane<D, G, E8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  float* red = reinterpret_cast<float*>(empty + C::STAGES);  // [warps][G][D + 2]
  int* flags = reinterpret_cast<int*>(red + kDecWarps * G * (D + 2));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  int bi = blockIdx.z;
  if constexpr (CACHE) {
    // Sequences longest first: grid slice z takes the sequence of rank z by length
    // (ties in index order), so that the hardware starts the largest CTAs first
    // (each takes 1 / num_splits of its own sequence; measured +2.5% on 8 shuffled
    // paged sequences of 20k-47k keys).  Small batches only.
    if (p.b <= 64) {
      if (threadIdx.x < p.b) {
        const int t = threadIdx.x, lt = cache_seq_len(p, t);
        int rank = 0;
        for (int k = 0; k < p.b; ++k) {
          const int lk = cache_seq_len(p, k);
          rank += (lk > lt || (lk == lt && k < t)) ? 1 : 0;
        }
        if (rank == static_cast<int>(blockIdx.z)) flags[2] = t;
      }
      __syncthreads();
      bi = flags[2];
    }
  }
  const int groups = p.g / G;                    // CTAs per KV head
  const int kvh = blockIdx.y / groups;
  const int h_first = kvh * p.g + (blockIdx.y % groups) * G;  // first query head of this CTA
  // Keys of this sequence (start <= j < limit) and where its rows live
  // (contiguous, paged or packed).
  int limit = p.kv_limit, start = p.kv_start, nblk = p.nblk, bps = p.blocks_per_split, row_base = 0;
  if (p.kv_mode != kKvDense) {
    // The lengths live on the device, so they are checked here before anything
    // they address is read: a paged sequence may not outrun its block-table row,
    // a packed one must lie inside the packed rows.  A sequence that fails is not
    // read (its keys count as none) and FA_ERR_DEVICE_ARG is recorded.
    bool seq_ok;
    if (p.kv_mode == kKvPaged) {
      limit = p.seqlens[bi];
      seq_ok = static_cast<int64_t>(limit) <= p.bt_stride * p.page_size;
    } else {
      row_base = p.cu_seqlens[bi];
      const int end = p.cu_seqlens[bi + 1];
      seq_ok = row_base >= 0 && end >= row_base && end <= p.total_k;
      limit = end - row_base;
    }
    if (!seq_ok) {
      if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) record_error(p.status, kErrDeviceArg);
      limit = 0;
      row_base = 0;
    }
    limit = max(limit, 0);
    start = p.window_left >= 0 ? max(0, limit - 1 - p.window_left) : 0;
    nblk = (limit + C::BN - 1) / C::BN;
    // every sequence is cut into num_splits ranges of its own length (measured
    // better balanced than ranges of one size set by the longest sequence)
    bps = max(1, (nblk - start / C::BN + p.num_splits - 1) / p.num_splits);
  }
  // blocks before the sliding window's left edge are never read
  const int blk_lo = start / C::BN + split * bps;
  const int blk_hi = min(nblk, blk_lo + bps);
  const int nb = max(0, blk_hi - blk_lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    fence_mbar_init();
    flags[0] = 0;
    flags[1] = 0;
  }
  __syncthreads();

  if (warp >= C::PRODUCER_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_CONTROL));
    if (warp > C::PRODUCER_WARP) {  // idle warps of the control warpgroup
      __syncthreads();
      return;
    }
    if (lane == 0 && nb > 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      // A block is loaded as BN / box_rows boxes (two when 64-key pages hold a
      // 128-key block), none straddling a page.  Paged: the pages of the next
      // block are fetched one iteration ahead, so the table lookups overlap the
      // wait for a free slot; a box that starts past the sequence's end (its
      // rows are masked) reuses the block's first page, so the table is never
      // read beyond the sequence's own entries.
      constexpr int MAXSUB = C::BN / kDecSubRows;
      const int nsub = C::BN / p.box_rows;
      const int* bt_row = p.block_table + static_cast<int64_t>(bi) * p.bt_stride;
      int pg_next[MAXSUB];
#pragma unroll
      for (int j = 0; j < MAXSUB; ++j) {
        const int r = blk_lo * C::BN + j * p.box_rows;
        pg_next[j] = (p.kv_mode == kKvPaged && j < nsub && r < limit) ? bt_row[r / p.page_size] : -1;
      }
      for (int i = 0; i < nb; ++i) {
        const int slot = i % C::STAGES, use = i / C::STAGES;
        const int row = (blk_lo + i) * C::BN;
        int pg[MAXSUB];
#pragma unroll
        for (int j = 0; j < MAXSUB; ++j) {
          pg[j] = pg_next[j];
          const int r = row + C::BN + j * p.box_rows;
          if (p.kv_mode == kKvPaged && i + 1 < nb) pg_next[j] = (j < nsub && r < limit) ? bt_row[r / p.page_size] : -1;
        }
        if (use > 0 && !mbar_wait(&empty[slot], (use - 1) & 1, p.status, kSiteDecEmpty)) break;
        uint8_t* st = smem + slot * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[slot], C::STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < MAXSUB; ++j) {
          if (j < nsub) {
            // coordinates (row, outer) of this box in the K/V tensor view
            const int r = row + j * p.box_rows;
            int c_row = r, c_outer = bi;
            if (p.kv_mode == kKvPaged) {
              c_outer = pg[j] >= 0 ? pg[j] : pg[0];
              c_row = r % p.page_size;
            } else if (p.kv_mode == kKvPacked) {
              c_row = row_base + r;
              c_outer = 0;
            }
            const int off = j * p.box_rows * D * C::ELT;
            tma_load_4d_hint(st + off, &p.tm_k, &full[slot], 0, kvh, c_row, c_outer, pol);
            tma_load_4d_hint(st + C::KV_BYTES + off, &p.tm_v, &full[slot], 0, kvh, c_row, c_outer, pol);
          }
        }
        ++issued;
      }
      for (int i = max(0, issued - C::STAGES); i < issued; ++i)
        if (!mbar_wait(&full[i % C::STAGES], (i / C::STAGES) & 1, p.status, kSiteDecDrain, true)) break;
    }
    __syncwarp();
    __syncthreads();
  } else {
    // ------------------------------ compute warps ------------------------------
    // (each register budget covers only its own role's code)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_COMPUTE));
    compute_split<D, G, BF16, SC, E8>(p, smem, full, empty, red, flags, warp, lane, split, bi, kvh, h_first, blk_lo, nb,
                                  start, limit);
  }
}

// The merge of all splits of one (batch, head group), run by the CTA that
// finished last (its 256 compute threads): per head h, LSE = logsumexp_s LSE_s
// and weights w_s = e^(LSE_s - LSE) (0 for a split that saw no key) into
// shared memory, then O = sum_s w_s O_s per dim; a head whose splits all saw no
// key gets O = 0 and LSE = -inf.  The partials are read through L2 (__ldcg):
// other SMs wrote them.
template <int D, int G, bool BF16>
__device__ __forceinline__ void merge_splits(const DecodeParams& p, float* wts, int bi, int h_first) {
  constexpr float kLog2e = 1.4426950408889634f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ns = p.num_splits;
  const int64_t nrows = static_cast<int64_t>(p.b) * p.hq;  // partial rows per split (sq == 1)
  if (warp < G) {
    const int64_t row = static_cast<int64_t>(bi) * p.hq + h_first + warp;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, __ldcg(p.lse_part + s * nrows + row));
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    float lse = -INFINITY;
    if (M != -INFINITY) {
      float ssum = 0.f;
      for (int s = lane; s < ns; s += 32) ssum += ex2_approx((__ldcg(p.lse_part + s * nrows + row) - M) * kLog2e);
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, x);
      lse = M + lg2_approx(ssum) * kLn2;
    }
    for (int s = lane; s < ns; s += 32) {
      const float ls = __ldcg(p.lse_part + s * nrows + row);
      wts[warp * ns + s] = (ls == -INFINITY) ? 0.f : ex2_approx((ls - lse) * kLog2e);
    }
    if (lane == 0 && p.lse != nullptr) p.lse[row] = lse;
  }
  named_bar_sync(1, kDecWarps * 32);
  for (int idx = threadIdx.x; idx < G * D; idx += kDecWarps * 32) {
    const int h = idx / D, e = idx % D;
    const int64_t row = static_cast<int64_t>(bi) * p.hq + h_first + h;
    const float* op = p.o_part + row * D + e;
    float o = 0.f;
#pragma unroll 8
    for (int s = 0; s < ns; ++s) {
      const float w = wts[h * ns + s];
      if (w != 0.f) o = fmaf(w, __ldcg(op + s * nrows * D), o);
    }
    uint16_t* orow = static_cast<uint16_t*>(p.o) + bi * p.o_stride_b + (h_first + h) * p.o_stride_h;
    if constexpr (BF16) {
      orow[e] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
    } else {
      orow[e] = __half_as_ushort(__float2half_rn(o));
    }
  }
}

template <int D, int G, bool BF16, bool SC, bool E8>
__device__ __forceinline__ void compute_split(const DecodeParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                              float* red, int* flags, int warp, int lane, int split, int bi, int kvh,
                                              int h_first, int blk_lo, int nb, int start, int limit) {
  using C = DecCfg<D, E8>;
  using L = DecLane<D, G, E8>;
  constexpr int ELT = C::ELT;
  // e4m3: the K scales of this KV head's 128-key blocks (one block per stage) and
  // its V scale, applied to the partial output
  const float* kdsc = E8 ? p.k_descale + (static_cast<int64_t>(bi) * p.hkv + kvh) * p.n_kblocks : nullptr;
  const int c = lane % L::LPR;      // dim group of this lane
  const int rg = lane / L::LPR;     // row within a pass
  // dims owned: segment s covers [s * D / SEG + 8 c, + 8)
  float q[G][L::DPL];
  float acc[G][L::DPL];
  float m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int hq = h_first + h;
    const void* qrow = static_cast<const uint8_t*>(p.q) + 2 * (bi * p.q_stride_b + hq * p.q_stride_h);
#pragma unroll
    for (int s = 0; s < L::SEG; ++s)
#pragma unroll
      for (int e = 0; e < L::ESEG; ++e) {
        q[h][L::ESEG * s + e] = load_elem<BF16>(qrow, s * (D / L::SEG) + L::ESEG * c + e) * p.scale_log2;
        acc[h][L::ESEG * s + e] = 0.f;
      }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }

  bool ok = true;
  for (int i = 0; i < nb; ++i) {
    const int slot = i % C::STAGES;
    // warp-uniform outcome: the shuffles below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (i / C::STAGES) & 1, p.status, kSiteDecFull))) {
      ok = false;
      break;
    }
    const uint8_t* ks = smem + slot * C::STAGE_BYTES;
    const uint8_t* vs = ks + C::KV_BYTES;
    const int key0 = (blk_lo + i) * C::BN + warp * C::ROWS_PER_WARP;
    // the last block of a sequence may hold rows past its end (another sequence's
    // keys, or cache slots never written), the first one rows before the window:
    // their V rows are zeroed below
    const bool edge_block = (blk_lo + i + 1) * C::BN > limit || (blk_lo + i) * C::BN < start;
    if (edge_block) {
      // zero this warp's V rows outside [start, limit) in shared memory (the TMA
      // copy has landed: the full barrier was waited on), so the loop below stays as is
      uint8_t* vw = smem + slot * C::STAGE_BYTES + C::KV_BYTES;
#pragma unroll
      for (int ps = 0; ps < L::PASSES; ++ps) {
        const int kr = warp * C::ROWS_PER_WARP + ps * L::RPP + rg;
        const int key = key0 + ps * L::RPP + rg;
        if (key >= limit || key < start) {
#pragma unroll
          for (int sg = 0; sg < L::SEG; ++sg)
            *reinterpret_cast<uint4*>(vw + kr * (D * ELT) + ELT * (sg * (D / L::SEG) + L::ESEG * c)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
    }
    // scores (log2 domain, scale folded into q) for this lane's row in each pass
    const float kdb = E8 ? kdsc[blk_lo + i] : 1.f;  // (e4m3: this block's K scale)
    float sc[L::PASSES][G];
#pragma unroll
    for (int ps = 0; ps < L::PASSES; ++ps) {
      const int kr = warp * C::ROWS_PER_WARP + ps * L::RPP + rg;
      float kf[L::DPL];
#pragma unroll
      for (int s = 0; s < L::SEG; ++s) {
        const uint4 u = *reinterpret_cast<const uint4*>(ks + kr * (D * ELT) + ELT * (s * (D / L::SEG) + L::ESEG * c));
        if constexpr (E8)
          unpack16_e4m3(u, kf);
        else
          unpack8<BF16>(u, kf + 8 * s);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < L::DPL; e += 2)
          a2 = __ffma2_rn(make_float2(q[h][e], q[h][e + 1]), make_float2(kf[e], kf[e + 1]), a2);
        sc[ps][h] = a2.x + a2.y;
      }
#pragma unroll
      for (int x = 1; x < L::LPR; x <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) sc[ps][h] += __shfl_xor_sync(0xffffffffu, sc[ps][h], x);
      if constexpr (E8) {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[ps][h] *= kdb;
      }
      if constexpr (SC) {
        // capped scores (log2 units): c log2(e) tanh(s / c), before the mask
#pragma unroll
        for (int h = 0; h < G; ++h) sc[ps][h] = p.sc_b * tanh_from_exp2_arg(sc[ps][h] * p.sc_k);
      }
      const int key = key0 + ps * L::RPP + rg;
      if (key >= limit || key < start) {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[ps][h] = -INFINITY;
      }
    }
    // block max per head over this warp's rows
    float mn[G], alpha[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float bm = sc[0][h];
#pragma unroll
      for (int ps = 1; ps < L::PASSES; ++ps) bm = fmaxf(bm, sc[ps][h]);
#pragma unroll
      for (int x = L::LPR; x < 32; x <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, x));
      mn[h] = fmaxf(m[h], bm);
      const float mu = (mn[h] == -INFINITY) ? 0.f : mn[h];
      alpha[h] = ex2_approx(m[h] - mu);
      m[h] = mn[h];
      mn[h] = mu;
    }
    // probabilities, running sums, rescale and accumulate P V
    float ps_sum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      ps_sum[h] = 0.f;
#pragma unroll
      for (int e = 0; e < L::DPL; e += 2) {
        const float2 r = __fmul2_rn(make_float2(acc[h][e], acc[h][e + 1]), make_float2(alpha[h], alpha[h]));
        acc[h][e] = r.x;
        acc[h][e + 1] = r.y;
      }
    }
#pragma unroll
    for (int ps = 0; ps < L::PASSES; ++ps) {
      const int kr = warp * C::ROWS_PER_WARP + ps * L::RPP + rg;
      float vf[L::DPL];
#pragma unroll
      for (int s = 0; s < L::SEG; ++s) {
        const uint4 u = *reinterpret_cast<const uint4*>(vs + kr * (D * ELT) + ELT * (s * (D / L::SEG) + L::ESEG * c));
        if constexpr (E8)
          unpack16_e4m3(u, vf);
        else
          unpack8<BF16>(u, vf + 8 * s);
      }

#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = ex2_approx(sc[ps][h] - mn[h]);
        ps_sum[h] += pr;
#pragma unroll
        for (int e = 0; e < L::DPL; e += 2) {
          const float2 r = __ffma2_rn(make_float2(pr, pr), make_float2(vf[e], vf[e + 1]),
                                      make_float2(acc[h][e], acc[h][e + 1]));
          acc[h][e] = r.x;
          acc[h][e + 1] = r.y;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float sgl = ps_sum[h];
#pragma unroll
      for (int x = L::LPR; x < 32; x <<= 1) sgl += __shfl_xor_sync(0xffffffffu, sgl, x);
      l[h] = alpha[h] * l[h] + sgl;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ---- merge the lanes that handled different rows (same dims) ----
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < L::DPL; ++e)
#pragma unroll
      for (int x = L::LPR; x < 32; x <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], x);
  // ---- merge the four warps through shared memory ----
  float* my = red + warp * G * (D + 2);
  if (rg == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int s = 0; s < L::SEG; ++s)
#pragma unroll
        for (int e = 0; e < L::ESEG; ++e)
          my[h * (D + 2) + s * (D / L::SEG) + L::ESEG * c + e] = acc[h][L::ESEG * s + e];
      if (c == 0) {
        my[h * (D + 2) + D] = m[h];
        my[h * (D + 2) + D + 1] = l[h];
      }
    }
  }
  if (!ok) flags[0] = 1;  // a wait gave up: no partial is written and nothing merged
  // all compute threads (and the producer) meet here
  __syncthreads();
  if (flags[0] != 0) return;
  const int nthreads = kDecWarps * 32;
  for (int idx = threadIdx.x; idx < G * D; idx += nthreads) {
    const int h = idx / D, e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red[(w * G + h) * (D + 2) + D]);
    float Lsum = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = ex2_approx(red[(w * G + h) * (D + 2) + D] - M);
        Lsum += f * red[(w * G + h) * (D + 2) + D + 1];
        o += f * red[(w * G + h) * (D + 2) + e];
      }
    }
    const int hq = h_first + h;
    const int64_t prow = (static_cast<int64_t>(split) * p.b + bi) * p.hq + hq;  // sq == 1
    const float vsc = E8 ? p.v_descale[static_cast<int64_t>(bi) * p.hkv + kvh] : 1.f;
    p.o_part[prow * D + e] = Lsum > 0.f ? o / Lsum * vsc : 0.f;
    if (e == 0) p.lse_part[prow] = Lsum > 0.f ? (M + lg2_approx(Lsum)) * kLn2 : -INFINITY;
  }
  // ---- fused merge: the last CTA of this (batch, group) to count itself in ----
  __threadfence();  // this CTA's partials are visible device-wide before it counts itself
  named_bar_sync(1, kDecWarps * 32);
  const int64_t ctr = static_cast<int64_t>(bi) * gridDim.y + blockIdx.y;
  if (threadIdx.x == 0) flags[1] = atomicAdd(p.counters + ctr, 1) == p.num_splits - 1;
  named_bar_sync(1, kDecWarps * 32);
  if (flags[1] == 0) return;
  __threadfence();
  // the K/V ring is idle now (every block consumed, the producer drained): it
  // holds the merge weights
  merge_splits<D, G, BF16>(p, reinterpret_cast<float*>(smem), bi, h_first);
  if (threadIdx.x == 0) p.counters[ctr] = 0;
}

template <int D, int G, bool BF16>
cudaError_t launch_dec(const DecodeParams& p, cudaStream_t stream) {
  using C = DecCfg<D>;
  const bool sc = p.sc_b > 0.f;
  auto kern = sc ? fa_decode_kernel<D, G, BF16, true, false> : fa_decode_kernel<D, G, BF16, false, false>;
  if (p.kv_mode != kKvDense)
    kern = sc ? fa_decode_kernel<D, G, BF16, true, true> : fa_decode_kernel<D, G, BF16, false, true>;
  const int smem = dec_smem_bytes<D, G>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.hkv * (p.g / G), p.b);
  kern<<<grid, C::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int G, bool BF16>
cudaError_t launch_dec_e4m3(const DecodeParams& p, cudaStream_t stream) {
  using C = DecCfg<D, true>;
  auto kern = fa_decode_kernel<D, G, BF16, false, false, true>;
  const int smem = dec_smem_bytes<D, G, true>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.hkv * (p.g / G), p.b);
  kern<<<grid, C::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int G, bool BF16>
int dec_occupancy() {
  using C = DecCfg<D>;
  const int smem = dec_smem_bytes<D, G>();
  auto kern = fa_decode_kernel<D, G, BF16, false, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, smem) != cudaSuccess || n < 1) return 1;
  return n;
}

template <int D, bool BF16>
cudaError_t launch_dec_g(const DecodeParams& p, cudaStream_t stream) {
  switch (decode_heads_per_cta(p.g)) {
    case 1: return launch_dec<D, 1, BF16>(p, stream);
    case 2: return launch_dec<D, 2, BF16>(p, stream);
    default: return launch_dec<D, 4, BF16>(p, stream);
  }
}

// ------------------------------------------------------------------ combine
template <bool BF16>
__global__ void __launch_bounds__(256) fa_combine_kernel(const __grid_constant__ CombineParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nrows = static_cast<int64_t>(p.b) * p.hq * p.sq;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= nrows) return;
  const int i = static_cast<int>(row % p.sq);
  const int h = static_cast<int>((row / p.sq) % p.hq);
  const int bi = static_cast<int>(row / (static_cast<int64_t>(p.sq) * p.hq));
  constexpr float kLog2e = 1.4426950408889634f;
  // LSE_total = logsumexp over splits
  float M = -INFINITY;
  for (int s = lane; s < p.num_splits; s += 32) M = fmaxf(M, p.lse_part[s * nrows + row]);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
  uint16_t* orow = static_cast<uint16_t*>(p.o) + bi * p.o_stride_b + static_cast<int64_t>(i) * p.o_stride_row +
                   h * p.o_stride_h;
  if (M == -INFINITY) {
    for (int e = lane; e < p.d; e += 32) orow[e] = 0;
    if (lane == 0 && p.lse != nullptr) p.lse[row] = -INFINITY;
    return;
  }
  float ssum = 0.f;
  for (int s = lane; s < p.num_splits; s += 32) ssum += ex2_approx((p.lse_part[s * nrows + row] - M) * kLog2e);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, x);
  const float lse = M + lg2_approx(ssum) * kLn2;
  // O = sum_s e^(LSE_s - LSE) O_s; lanes own dims e = lane + 32 k (k < 8, d <= 256)
  float o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = 0.f;
  for (int s = 0; s < p.num_splits; ++s) {
    const float ls = p.lse_part[s * nrows + row];
    if (ls == -INFINITY) continue;
    const float w = ex2_approx((ls - lse) * kLog2e);
    const float* op = p.o_part + (s * nrows + row) * p.d;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = lane + 32 * k;
      if (e < p.d) o[k] = fmaf(w, op[e], o[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = lane + 32 * k;
    if (e < p.d) {
      if constexpr (BF16) {
        orow[e] = __bfloat16_as_ushort(__float2bfloat16_rn(o[k]));
      } else {
        orow[e] = __half_as_ushort(__float2half_rn(o[k]));
      }
    }
  }
  if (lane == 0 && p.lse != nullptr) p.lse[row] = lse;
}

// ------------------------------------------------------------------ self test
// A wait that nothing completes: it must give up after the limit, record the
// timeout in the status word and return.
__global__ void fa_wait_selftest_kernel(int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, 0x7f);
  __syncthreads();
}

}  // namespace

int decode_block_n(int d) {
  switch (d) {
    case 64: return DecCfg<64>::BN;
    case 128: return DecCfg<128>::BN;
    default: return DecCfg<256>::BN;
  }
}

int decode_heads_per_cta(int g) { return (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1; }

bool decode_supported(int d, int g) { return (d == 64 || d == 128 || d == 256) && g >= 1; }

// Resident decode CTAs per SM, from the occupancy query on the first call per
// (device, d, dtype) and cached: the split heuristic asks on every split-KV call.
int decode_ctas_per_sm(int d, int dtype) {
  constexpr int kDevs = 64;
  static std::atomic<int> cache[kDevs][3][2];  // 0 = not yet queried (static storage starts zeroed)
  const bool bf16 = dtype == 0;
  const int di = d == 64 ? 0 : d == 128 ? 1 : d == 256 ? 2 : -1;
  if (di < 0) return 1;
  int dev = -1;
  const bool cacheable = cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kDevs;
  if (cacheable) {
    const int n = cache[dev][di][bf16 ? 1 : 0].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 1;
  switch (d) {
    case 64: n = bf16 ? dec_occupancy<64, 4, true>() : dec_occupancy<64, 4, false>(); break;
    case 128: n = bf16 ? dec_occupancy<128, 4, true>() : dec_occupancy<128, 4, false>(); break;
    default: n = bf16 ? dec_occupancy<256, 4, true>() : dec_occupancy<256, 4, false>(); break;
  }
  if (cacheable) cache[dev][di][bf16 ? 1 : 0].store(n, std::memory_order_relaxed);
  return n;
}

template <int D, bool BF16>
cudaError_t launch_dec_e4m3_g(const DecodeParams& p, cudaStream_t stream) {
  switch (decode_heads_per_cta(p.g)) {
    case 1: return launch_dec_e4m3<D, 1, BF16>(p, stream);
    case 2: return launch_dec_e4m3<D, 2, BF16>(p, stream);
    default: return launch_dec_e4m3<D, 4, BF16>(p, stream);
  }
}

int decode_e4m3_block_n() { return DecCfg<128, true>::BN; }

cudaError_t launch_decode_e4m3(const DecodeParams& p, int d, int dtype, cudaStream_t stream) {
  const bool bf16 = dtype == 0;
  switch (d) {
    case 64: return bf16 ? launch_dec_e4m3_g<64, true>(p, stream) : launch_dec_e4m3_g<64, false>(p, stream);
    case 128: return bf16 ? launch_dec_e4m3_g<128, true>(p, stream) : launch_dec_e4m3_g<128, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeParams& p, int d, int dtype, cudaStream_t stream) {
  const bool bf16 = dtype == 0;
  switch (d) {
    case 64: return bf16 ? launch_dec_g<64, true>(p, stream) : launch_dec_g<64, false>(p, stream);
    case 128: return bf16 ? launch_dec_g<128, true>(p, stream) : launch_dec_g<128, false>(p, stream);
    case 256: return bf16 ? launch_dec_g<256, true>(p, stream) : launch_dec_g<256, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const CombineParams& p, int dtype, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.b) * p.hq * p.sq;
  if (nrows == 0) return cudaSuccess;
  const int64_t blocks = (nrows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (dtype == 0)
    fa_combine_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  else
    fa_combine_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, cudaStream_t stream) {
  fa_wait_selftest_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace fa
