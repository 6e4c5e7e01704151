// Backward pass in the recompute form of "hs-black: FlashAttention 1/2/3",
// sections "Backward: from the softmax derivative", "Training: recompute in
// backward" and "Backward: back to Q, K, V": the forward pass keeps only O and
// one L = m + log l per row; the backward pass recomputes S tile by tile,
// recovers P = exp(S - L), and forms
//   D = rowsum(dO * O), dP = dO V^T, dS = P (dP - D),
//   dV = P^T dO, dQ = dS K * scale, dK = dS^T Q * scale,
// with P and dS zero where the mask hides a key.  Two kernels:
//   * fa_bwd_dq_kernel: a CTA owns 128 query rows and streams the key blocks
//     they see (S = Q K^T, dP = dO V^T, dQ += dS K on tcgen05, one TMEM lane per
//     row for the elementwise work); its elementwise threads first form D and
//     L * log2(e) of their rows, which it also writes for the second kernel;
//   * fa_bwd_dkdv_kernel: a CTA owns 128 keys of one key/value head and streams
//     the query tiles that see them, over every query head of its group (S^T =
//     K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q, one TMEM lane per key),
//     so dK and dV are reduced in TMEM without atomics.
// Splitting dQ from dK / dV costs two extra products per block pair (S and dP
// are computed by both kernels) but needs no atomic accumulation and keeps every
// accumulator of a CTA in its 512 TMEM columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Wait sites of the backward kernels (recorded in the status word on timeout).
enum : int {
  kSiteBwdQFull = 32,
  kSiteBwdKvFull,
  kSiteBwdKvEmpty,
  kSiteBwdSFull,
  kSiteBwdDsFull,
  kSiteBwdDone,
  kSiteBwdDrain,
  kSiteBwdQdFull,
  kSiteBwdQdEmpty,
};

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;             // query rows per tile
  static constexpr int BN = 128;             // keys per block
  static constexpr int DC = D / 64;          // 64-column chunks (128-byte rows)
  static constexpr int TILE_BYTES = 128 * D * 2;
  // two elementwise warpgroups (each takes half of the columns of every block:
  // nothing in the backward elementwise pass reduces along a row) + producer + MMA + 2 idle
  static constexpr int THREADS = 384;
  static constexpr int EW_THREADS = 256;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  // register split: launched at 168 per thread (384 threads); the control warpgroup
  // drops to 72 and the elementwise warpgroups rise to 208: 256 * 208 + 128 * 72 <= 384 * 168
  static constexpr int REG_EW = 208;
  static constexpr int REG_CONTROL = 72;
  static_assert(EW_THREADS * REG_EW + 128 * REG_CONTROL <= THREADS * 168, "register split");
  static constexpr int TMEM_COLS = 512;
  // dQ kernel: Q and dO tiles, then a ring of K / V blocks
  static constexpr int DQ_STAGES = 5;
  static constexpr int DQ_RING_OFF = 2 * TILE_BYTES;
  static constexpr int DQ_BAR_OFF = DQ_RING_OFF + DQ_STAGES * TILE_BYTES;
  // (at least 117 KiB, so that one CTA, which holds all 512 TMEM columns, runs per SM)
  static constexpr int MIN_SMEM = 117 * 1024;
  static constexpr int DQ_SMEM_RAW = DQ_BAR_OFF + 8 * (2 * DQ_STAGES + 7) + 16 + 1024;
  static constexpr int DQ_SMEM = DQ_SMEM_RAW > MIN_SMEM ? DQ_SMEM_RAW : MIN_SMEM;
  // dK / dV kernel: K and V tiles, then stages of (Q tile, dO tile, L and D of their rows)
  static constexpr int KV_STAGES = 2;
  static constexpr int QD_STAGE_BYTES = 2 * TILE_BYTES + 1024;  // + 128 floats of L, 128 of D
  static constexpr int QD_OFF = 2 * TILE_BYTES;
  static constexpr int KV_BAR_OFF = QD_OFF + KV_STAGES * QD_STAGE_BYTES;
  static constexpr int KV_SMEM_RAW = KV_BAR_OFF + 8 * (2 * KV_STAGES + 8) + 16 + 1024;
  static constexpr int KV_SMEM = KV_SMEM_RAW > MIN_SMEM ? KV_SMEM_RAW : MIN_SMEM;
  static_assert(DQ_SMEM <= 227 * 1024 && KV_SMEM <= 227 * 1024, "shared memory budget");
  static_assert(QD_STAGE_BYTES % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  // TMEM: S (or S^T) at 0, dP (or dP^T) at 128, accumulators from 256; the dQ
  // kernel keeps a second S buffer at 384 (S of the next block while dQ reads dS)
  static constexpr int S_COL = 0, DP_COL = 128, ACC_COL = 256, S2_COL = 384;
  static_assert(ACC_COL + D <= S2_COL, "the dQ accumulator and the second S buffer must not overlap");
  static_assert(ACC_COL + 2 * D <= TMEM_COLS, "dK and dV accumulators must fit in TMEM");
};

// ------------------------------------------------------------------ row terms

// acc + sum of the 8 products of two rows' 16-bit values (widened exactly to fp32).
template <bool BF16>
__device__ __forceinline__ float dot8(const uint4 a, const uint4 b, float acc) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float a0, a1, b0, b1;
    if constexpr (BF16) {
      a0 = __uint_as_float(aw[e] << 16);
      a1 = __uint_as_float(aw[e] & 0xffff0000u);
      b0 = __uint_as_float(bw[e] << 16);
      b1 = __uint_as_float(bw[e] & 0xffff0000u);
    } else {
      const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
      const float2 bf = __half22float2(*reinterpret_cast<const __half2*>(&bw[e]));
      a0 = af.x;
      a1 = af.y;
      b0 = bf.x;
      b1 = bf.y;
    }
    acc = fmaf(a0, b0, acc);
    acc = fmaf(a1, b1, acc);
  }
  return acc;
}

// Store NC fp32 values (scaled by `mul`) from TMEM columns [tcol, tcol + NC) of
// this thread's lane to global memory as 16-bit values (when `valid`).
template <int NC, bool BF16>
__device__ __forceinline__ void store_acc_row(uint32_t tcol, float mul, uint16_t* dst, bool valid) {
#pragma unroll
  for (int c = 0; c < NC; c += 32) {
    uint32_t v[32];
    tmem_load_row<32>(tcol + c, v);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
      for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

// ------------------------------------------------------------------ dQ

// Key blocks [lo, hi) that some row of the 128-row tile starting at row0 sees.
__device__ __forceinline__ void key_block_range(const BwdParams& p, int row0, int* lo, int* hi) {
  const int nblk = (p.skv + 127) / 128;
  const int last_row = min(row0 + 128, p.sq) - 1;
  int h = nblk, l = 0;
  if (p.causal) h = min(h, floor_div(last_row + p.off, 128) + 1);
  if (p.local) l = max(l, floor_div(row0 + p.left_off, 128));
  if (h < l) h = l;
  *lo = l;
  *hi = h;
}

// SC: softcap; the score is capped to c tanh(s / c) and dS gains the factor 1 - tanh^2.
template <int D, bool BF16, bool SC>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, ST = C::DQ_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem + C::DQ_RING_OFF;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + C::DQ_BAR_OFF);  // Q and dO landed
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + ST;
  uint64_t* s_full = kv_empty + ST;   // S of a block is in TMEM, one barrier per S buffer
  uint64_t* dp_full = s_full + 2;     // dP of a block is in TMEM
  uint64_t* ds_half = dp_full + 1;    // dS of the first / second half of a block's keys is in TMEM
  uint64_t* dq_done = ds_half + 2;    // every dQ MMA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dq_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Longest row tiles first (causal: the last tiles see the most keys), within
  // groups of head_group consecutive (batch, query head) pairs taken one group
  // after the other: the CTAs in flight then read the K / V of a few heads only,
  // which stay in L2 (longest first over every head at once kept all of them in
  // flight and re-read K / V from DRAM); the hardware hands the next CTA to the
  // first SM that frees, so each group is balanced as the whole grid was.
  const int BH = p.b * p.hq;
  const int per_group = p.head_group * p.n_mtiles;
  const int g0 = static_cast<int>(blockIdx.x / per_group) * p.head_group;
  const int gsize = min(p.head_group, BH - g0);
  const int r_in = static_cast<int>(blockIdx.x % per_group);
  const int bh = g0 + r_in % gsize;
  const int m = p.n_mtiles - 1 - r_in / gsize;
  const int h = bh % p.hq, bi = bh / p.hq, kvh = h / p.g;
  const int row0 = m * BM;
  int n_lo, n_hi;
  key_block_range(p, row0, &n_lo, &n_hi);
  const int N = n_hi - n_lo;  // key blocks visited, from n_hi - 1 down

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(&ds_half[0], C::EW_THREADS);
    mbar_init(&ds_half[1], C::EW_THREADS);
    mbar_init(dq_done, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp >= 8) {
    // control warpgroup (producer, MMA issuer, two idle warps): registers move to the elementwise warps
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_CONTROL));
  if (warp == C::PRODUCER_WARP) {
    if (lane == 0 && N > 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::DC; ++c) {
        tma_load_4d(smem + c * (BM * 128), &p.tm_q, q_full, c * 64, h, row0, bi);
        tma_load_4d(smem + C::TILE_BYTES + c * (BM * 128), &p.tm_do, q_full, c * 64, h, row0, bi);
      }
      const uint64_t pol = l2_policy_evict_last();
      int issued = 0;
      // V_j, then K_j: V is released as soon as dP has read it, K only once dQ has
      // (it is read twice), so with V first each load reuses a slot freed earlier
      for (int L = 0; L < 2 * N; ++L) {
        const int slot = L % ST, use = L / ST;
        if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, p.status, kSiteBwdKvEmpty, false, 128)) break;
        const int n = n_hi - 1 - (L >> 1);
        mbar_arrive_expect_tx(&kv_full[slot], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::DC; ++c)
          tma_load_4d_hint(ring + slot * C::TILE_BYTES + c * (BN * 128), (L & 1) ? &p.tm_k : &p.tm_v,
                           &kv_full[slot], c * 64, kvh, n * BN, bi, pol);
        ++issued;
      }
      for (int L = max(0, issued - ST); L < issued; ++L)
        if (!mbar_wait(&kv_full[L % ST], (L / ST) & 1, p.status, kSiteBwdDrain, true)) break;
      mbar_wait(q_full, 0, p.status, kSiteBwdDrain, true);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && N > 0) {
      constexpr uint32_t kIdS = idesc_f16(BM, BN, BF16, false);
      constexpr uint32_t kIdQ = idesc_f16(BM, D, BF16, true);
      const uint32_t ring_s = smem_u32(ring);
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t do_desc = sdesc_sw128(smem_u32(smem + C::TILE_BYTES), 16, 1024);
      const uint64_t kk_desc = sdesc_sw128(ring_s, 16, 1024);        // a ring slot read K-major
      const uint64_t kmn_desc = sdesc_sw128(ring_s, BN * 128, 1024);  // a ring slot read MN-major
      // Software-pipelined over the key blocks: S of block it + 1 goes to the other
      // S buffer at the start of iteration it, and dP of block it + 1 as soon as the
      // elementwise warps are done with block it, so they form P of the next block
      // while the tensor pipe runs dQ of this one (in issue order).  Every barrier
      // is at most one phase ahead of its waiters: S of block it + 2 is issued only
      // after block it (the same S buffer and barrier) is done.
#define FA_SCOL(i) ((i) & 1 ? C::S2_COL : C::S_COL)
      bool ok = mbar_wait(q_full, 0, p.status, kSiteBwdQFull) &&
                mbar_wait(&kv_full[0], 0, p.status, kSiteBwdKvFull) && mbar_wait(&kv_full[1], 0, p.status, kSiteBwdKvFull);
      if (ok) {
        tc_fence_after();
        issue_s_tile<D, BN, BM, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + C::S_COL, q_desc, kk_desc, 0, 1);
        umma_commit(&s_full[0]);
        issue_s_tile<D, BN, BM, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + C::DP_COL, do_desc, kk_desc, 0, 0);
        umma_commit(dp_full);
        umma_commit(&kv_empty[0]);
      }
      for (int it = 0; ok && it < N; ++it) {
        const int Lk = 2 * it + 1, Lk1 = 2 * it + 3, Lv1 = 2 * it + 2;
        const bool more = it + 1 < N;
        // S of the next block into the other buffer (dQ of block it - 1 has read it: in order)
        if (more) {
          if (!mbar_wait(&kv_full[Lk1 % ST], (Lk1 / ST) & 1, p.status, kSiteBwdKvFull)) break;
          tc_fence_after();
          issue_s_tile<D, BN, BM, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + FA_SCOL(it + 1), q_desc, kk_desc, 0,
                                                                      Lk1 % ST);
          umma_commit(&s_full[(it + 1) & 1]);
        }
        // dQ += dS K by halves of the block's keys: dS of keys [32 c, 32 c + 32) is packed
        // at columns [32 c, 32 c + 16) of the block's S buffer; K is read MN-major
        if (!mbar_wait(&ds_half[0], it & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        const uint32_t sc = tbase + FA_SCOL(it);
        issue_pv_tile<D, BN, C::TILE_BYTES, kIdQ, 0, 2>(tbase + C::ACC_COL, sc, kmn_desc, Lk % ST, it > 0);
        issue_pv_tile<D, BN, C::TILE_BYTES, kIdQ, 2, 4>(tbase + C::ACC_COL, sc + 16, kmn_desc, Lk % ST, true);
        if (!mbar_wait(&ds_half[1], it & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        // the elementwise warps are done with block it (and have read its dP): the next block's dP
        if (more) {
          if (!mbar_wait(&kv_full[Lv1 % ST], (Lv1 / ST) & 1, p.status, kSiteBwdKvFull)) break;
          tc_fence_after();
          issue_s_tile<D, BN, BM, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + C::DP_COL, do_desc, kk_desc, 0,
                                                                      Lv1 % ST);
          umma_commit(dp_full);
          umma_commit(&kv_empty[Lv1 % ST]);
        }
        issue_pv_tile<D, BN, C::TILE_BYTES, kIdQ, 4, 6>(tbase + C::ACC_COL, sc + 32, kmn_desc, Lk % ST, true);
        issue_pv_tile<D, BN, C::TILE_BYTES, kIdQ, 6, 8>(tbase + C::ACC_COL, sc + 48, kmn_desc, Lk % ST, true);
        umma_commit(&kv_empty[Lk % ST]);
      }
#undef FA_SCOL
      umma_commit(dq_done);
      mbar_wait(dq_done, 0, p.status, kSiteBwdDrain, true);
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_EW));
    // ---------------- elementwise: one query row per thread, half of the keys per warpgroup ----------------
    const int eg = warp >> 2;  // keys [64 eg, 64 eg + 64) of every block
    const int r = 32 * (warp & 3) + lane;
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tP = tbase + lane_off + C::DP_COL;
    const int64_t prow = (static_cast<int64_t>(bi) * p.hq + h) * p.sq_pad + row;  // row < sq_pad
    // D = rowsum(dO * O) over the stored (rounded) O and L2 = LSE * log2(e) of this
    // row: O's row is loaded from global memory at once, dO's is read from the
    // tile the producer stages (from global memory too when no key block is
    // visited); both warpgroups form them and the first writes them for the
    // dK / dV kernel (which runs after this one).  Padding rows and rows that see
    // no key get L2 = +inf (every probability recovered from it is 0) and D = 0.
    bool ok = true;
    float l2 = INFINITY, dd = 0.f;
    {
      constexpr int NC = D / 8;
      const bool live = row < p.sq;
      uint4 ov[NC];
      float lse = -INFINITY;
      if (live) {
        lse = p.lse[(static_cast<int64_t>(bi) * p.hq + h) * p.sq + row];
        const uint4* o4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + bi * p.o_st[0] +
                                                         static_cast<int64_t>(row) * p.o_st[1] + h * p.o_st[2]);
#pragma unroll
        for (int c = 0; c < NC; ++c) ov[c] = o4[c];
      }
      if (N > 0) {
        ok = warp_wait(q_full, 0, p.status, kSiteBwdQFull);
        if (ok && live) {
          const uint8_t* dtile = smem + C::TILE_BYTES;  // 64-column chunks of 128-byte rows, 128-byte swizzle
#pragma unroll
          for (int c = 0; c < NC; ++c)
            dd = dot8<BF16>(ov[c],
                            *reinterpret_cast<const uint4*>(dtile + (c / 8) * (BM * 128) + r * 128 +
                                                            (((c % 8) ^ (r & 7)) << 4)),
                            dd);
        }
      } else if (live) {
        const uint4* g4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + bi * p.do_st[0] +
                                                         static_cast<int64_t>(row) * p.do_st[1] + h * p.do_st[2]);
#pragma unroll
        for (int c = 0; c < NC; ++c) dd = dot8<BF16>(ov[c], g4[c], dd);
      }
      if (live) l2 = lse > -INFINITY ? lse * kLog2e : INFINITY;
    }
    if (eg == 0) {
      p.dpre[prow] = dd;
      p.l2pre[prow] = l2;
    }
    const float sl2 = p.scale_log2;
    // keys lo_row <= j < lim_row are visible to this row
    const int lim_row = p.causal ? min(p.skv, max(row + p.off + 1, 0)) : p.skv;
    const int lo_row = p.local ? row + p.left_off : 0;
    for (int it = 0; ok && it < N; ++it) {
      const int n = n_hi - 1 - it;
      const uint32_t tSb = tbase + lane_off + ((it & 1) ? C::S2_COL : C::S_COL);  // this block's S buffer
      // ---- P = 2^(S scale log2 e - L2) as soon as S is in TMEM ----
      if (!warp_wait(&s_full[it & 1], (it >> 1) & 1, p.status, kSiteBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int lim = lim_row - n * BN, lo = lo_row - n * BN;
      // chunk of 32 keys: warpgroup eg takes chunk eg of each half; the half is
      // signalled once both warpgroups have packed their chunk; both chunks of this
      // warpgroup are loaded at once (the second load's latency hides behind the
      // first chunk's arithmetic)
      uint32_t sv2[2][32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) tmem_ld32_issue(tSb + hf * (BN / 2) + eg * 32, sv2[hf]);
      tmem_ld_wait();
      reg_fence<32>(sv2[0]);
      reg_fence<32>(sv2[1]);
      float pf[2][32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = hf * (BN / 2) + eg * 32;
        const bool edge = lim < c0 + 32 || lo > c0;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          // pairs of keys in packed f32x2 math; the mask only where an edge cuts the chunk
          float2 x, w = make_float2(1.f, 1.f);
          if constexpr (SC) {
            // capped score c log2(e) tanh(s / c); dS gains w = 1 - tanh^2
            const float t0 = tanh_from_exp2_arg(__uint_as_float(sv2[hf][i]) * p.sc_k);
            const float t1 = tanh_from_exp2_arg(__uint_as_float(sv2[hf][i + 1]) * p.sc_k);
            x = make_float2(fmaf(p.sc_b, t0, -l2), fmaf(p.sc_b, t1, -l2));
            w = make_float2(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
          } else {
            x = __ffma2_rn(make_float2(__uint_as_float(sv2[hf][i]), __uint_as_float(sv2[hf][i + 1])),
                           make_float2(sl2, sl2), make_float2(-l2, -l2));
          }
          float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (edge) {
            const int c = c0 + i;
            if (c >= lim || c < lo) pr.x = 0.f;
            if (c + 1 >= lim || c + 1 < lo) pr.y = 0.f;
          }
          if constexpr (SC) pr = __fmul2_rn(pr, w);
          pf[hf][i] = pr.x;
          pf[hf][i + 1] = pr.y;
        }
      }
      // ---- dS = P (dP - D) once dP is in TMEM ----
      if (!warp_wait(dp_full, it & 1, p.status, kSiteBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pv2[2][32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) tmem_ld32_issue(tP + hf * (BN / 2) + eg * 32, pv2[hf]);
      tmem_ld_wait();
      reg_fence<32>(pv2[0]);
      reg_fence<32>(pv2[1]);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = hf * (BN / 2) + eg * 32;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 ds = __fmul2_rn(make_float2(pf[hf][i], pf[hf][i + 1]),
                                       __fadd2_rn(make_float2(__uint_as_float(pv2[hf][i]), __uint_as_float(pv2[hf][i + 1])),
                                                  make_float2(-dd, -dd)));
          pk[i / 2] = pack2<BF16>(ds.x, ds.y);
        }
        tmem_st16(tSb + c0, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_half[hf]);
      }
    }
    uint16_t* dst = static_cast<uint16_t*>(p.dq) + bi * p.dq_st[0] + static_cast<int64_t>(row) * p.dq_st[1] +
                    h * p.dq_st[2];
    // each warpgroup writes half of the row's d columns
    if (ok && N > 0 && warp_wait(dq_done, 0, p.status, kSiteBwdDone)) {
      tc_fence_after();
      store_acc_row<D / 2, BF16>(tbase + lane_off + C::ACC_COL + eg * (D / 2), p.scale, dst + eg * (D / 2),
                                 row < p.sq);
    } else if (ok && N == 0 && row < p.sq) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + eg * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 16; ++c) d4[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dK, dV

// Query tiles [lo, hi) with some row that sees a key of the block starting at key j0.
__device__ __forceinline__ void query_tile_range(const BwdParams& p, int j0, int* lo, int* hi) {
  const int j_last = min(j0 + 127, p.skv - 1);
  int l = 0, h = p.n_mtiles;
  if (p.causal) l = max(l, floor_div(j0 - p.off, 128));       // row i sees j0 only if i >= j0 - off
  if (p.local) h = min(h, floor_div(j_last - p.left_off, 128) + 1);  // ... j_last only if i <= j_last - left_off
  if (h < l) h = l;
  *lo = l;
  *hi = h;
}

template <int D, bool BF16, bool SC>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, ST = C::KV_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::KV_BAR_OFF);  // K and V landed
  uint64_t* qd_full = kv_full + 1;   // per stage: Q, dO, L2, D of a query tile landed
  uint64_t* qd_empty = qd_full + ST;
  uint64_t* s_full = qd_empty + ST;  // S^T in TMEM
  uint64_t* dp_full = s_full + 1;    // dP^T in TMEM
  uint64_t* p_half = dp_full + 1;    // P^T of the first / second half of a tile's rows in TMEM
  uint64_t* ds_half = p_half + 2;    // dS^T of the first / second half
  uint64_t* mma_done = ds_half + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  auto stage_ptr = [&](int s) { return smem + C::QD_OFF + s * C::QD_STAGE_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x % p.n_ntiles;
  const int bk = blockIdx.x / p.n_ntiles;
  const int kvh = bk % p.hkv, bi = bk / p.hkv;
  const int j0 = nb * BN;
  int m_lo, m_hi;
  query_tile_range(p, j0, &m_lo, &m_hi);
  const int nm = m_hi - m_lo;
  const int T = nm * p.g;  // query tiles visited: every head of the group, rows m_lo.. of each

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(&p_half[hf], C::EW_THREADS);
      mbar_init(&ds_half[hf], C::EW_THREADS);
    }
    mbar_init(mma_done, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp >= 8) {
    // control warpgroup (producer, MMA issuer, two idle warps): registers move to the elementwise warps
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_CONTROL));
  if (warp == C::PRODUCER_WARP) {
    if (lane == 0 && T > 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::DC; ++c) {
        tma_load_4d(smem + c * (BN * 128), &p.tm_k, kv_full, c * 64, kvh, j0, bi);
        tma_load_4d(smem + C::TILE_BYTES + c * (BN * 128), &p.tm_v, kv_full, c * 64, kvh, j0, bi);
      }
      int issued = 0;
      for (int ti = 0; ti < T; ++ti) {
        const int s = ti % ST, use = ti / ST;
        if (use > 0 && !mbar_wait(&qd_empty[s], (use - 1) & 1, p.status, kSiteBwdQdEmpty, false, 128)) break;
        const int h = kvh * p.g + ti / nm, m = m_lo + ti % nm;
        uint8_t* st = stage_ptr(s);
        mbar_arrive_expect_tx(&qd_full[s], 2 * C::TILE_BYTES + 1024);
#pragma unroll
        for (int c = 0; c < C::DC; ++c) {
          tma_load_4d(st + c * (BM * 128), &p.tm_q, &qd_full[s], c * 64, h, m * BM, bi);
          tma_load_4d(st + C::TILE_BYTES + c * (BM * 128), &p.tm_do, &qd_full[s], c * 64, h, m * BM, bi);
        }
        const int64_t prow = (static_cast<int64_t>(bi) * p.hq + h) * p.sq_pad + m * BM;
        bulk_load(st + 2 * C::TILE_BYTES, p.l2pre + prow, 512, &qd_full[s]);
        bulk_load(st + 2 * C::TILE_BYTES + 512, p.dpre + prow, 512, &qd_full[s]);
        ++issued;
      }
      for (int ti = max(0, issued - ST); ti < issued; ++ti)
        if (!mbar_wait(&qd_full[ti % ST], (ti / ST) & 1, p.status, kSiteBwdDrain, true)) break;
      mbar_wait(kv_full, 0, p.status, kSiteBwdDrain, true);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && T > 0) {
      constexpr uint32_t kIdS = idesc_f16(BN, BM, BF16, false);  // S^T: M = keys, N = query rows
      constexpr uint32_t kIdA = idesc_f16(BN, D, BF16, true);    // dV, dK: M = keys, N = d, B MN-major
      const uint32_t k_s = smem_u32(smem);  // K tile, then V tile (read K-major)
      // (descriptors are formed where they are used: fewer live registers in this warp)
#define FA_KDESC() sdesc_sw128(opaque_u32(k_s), 16, 1024)
#define FA_VDESC() sdesc_sw128(opaque_u32(k_s) + C::TILE_BYTES, 16, 1024)
      // Software-pipelined over the query tiles: the next tile's S^T is issued as
      // soon as dV has read this tile's P^T out of its columns, and its dP^T as soon
      // as dK has read dS^T, so the elementwise warps form P of tile ti + 1 while
      // the tensor pipe still runs dK of tile ti (the pipe executes in issue order).
      bool ok = mbar_wait(kv_full, 0, p.status, kSiteBwdKvFull) && mbar_wait(&qd_full[0], 0, p.status, kSiteBwdQdFull);
      if (ok) {
        tc_fence_after();
        const uint32_t st0 = smem_u32(stage_ptr(0));
        issue_s_tile<D, BM, BN, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + C::S_COL, FA_KDESC(), sdesc_sw128(st0, 16, 1024),
                                                                    0, 0);
        umma_commit(s_full);
        issue_s_tile<D, BM, BN, C::TILE_BYTES, C::TILE_BYTES, kIdS>(tbase + C::DP_COL, FA_VDESC(),
                                                                    sdesc_sw128(st0 + C::TILE_BYTES, 16, 1024), 0, 0);
        umma_commit(dp_full);
      }
      for (int ti = 0; ok && ti < T; ++ti) {
        const int s = ti % ST, s1 = (ti + 1) % ST;
        const bool more = ti + 1 < T;
        const uint32_t st = smem_u32(stage_ptr(s));
        const uint64_t qmn_desc = sdesc_sw128(st, BM * 128, 1024);                     // Q, MN-major
        const uint64_t domn_desc = sdesc_sw128(st + C::TILE_BYTES, BM * 128, 1024);  // dO, MN-major
        // dV += P^T dO, half a tile of query rows at a time (the first half's products
        // run while the second half is formed); P^T of rows [32 c, 32 c + 32) is packed
        // at columns [32 c, 32 c + 16) of the S^T region, dO is read MN-major
        if (!mbar_wait(&p_half[0], ti & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 0, 2>(tbase + C::ACC_COL, tbase + C::S_COL, domn_desc, 0, ti > 0);
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 2, 4>(tbase + C::ACC_COL, tbase + C::S_COL + 16, domn_desc, 0,
                                                        true);
        if (!mbar_wait(&p_half[1], ti & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 4, 6>(tbase + C::ACC_COL, tbase + C::S_COL + 32, domn_desc, 0,
                                                        true);
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 6, 8>(tbase + C::ACC_COL, tbase + C::S_COL + 48, domn_desc, 0,
                                                        true);
        // the next tile's S^T = K Q^T over the columns dV has just read: here if its
        // Q / dO stage has landed, else after dK (anywhere after dV keeps the order)
        bool s_issued = false;
        if (more && mbar_test(&qd_full[s1], ((ti + 1) / ST) & 1)) {
          tc_fence_after();
          issue_s_tile<D, BM, BN, C::TILE_BYTES, C::TILE_BYTES, kIdS>(
              tbase + C::S_COL, FA_KDESC(), sdesc_sw128(opaque_u32(smem_u32(stage_ptr(s1))), 16, 1024), 0, 0);
          umma_commit(s_full);
          s_issued = true;
        }
        // dK += dS^T Q, likewise by halves; Q read MN-major
        if (!mbar_wait(&ds_half[0], ti & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 0, 2>(tbase + C::ACC_COL + D, tbase + C::DP_COL, qmn_desc, 0,
                                                        ti > 0);
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 2, 4>(tbase + C::ACC_COL + D, tbase + C::DP_COL + 16, qmn_desc, 0,
                                                        true);
        if (!mbar_wait(&ds_half[1], ti & 1, p.status, kSiteBwdDsFull)) break;
        tc_fence_after();
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 4, 6>(tbase + C::ACC_COL + D, tbase + C::DP_COL + 32, qmn_desc, 0,
                                                        true);
        issue_pv_tile<D, BM, C::TILE_BYTES, kIdA, 6, 8>(tbase + C::ACC_COL + D, tbase + C::DP_COL + 48, qmn_desc, 0,
                                                        true);
        // the next tile's dP^T = V dO^T over the columns dK has just read
        if (more) {
          if (!s_issued) {
            if (!mbar_wait(&qd_full[s1], ((ti + 1) / ST) & 1, p.status, kSiteBwdQdFull)) break;
            tc_fence_after();
            issue_s_tile<D, BM, BN, C::TILE_BYTES, C::TILE_BYTES, kIdS>(
                tbase + C::S_COL, FA_KDESC(), sdesc_sw128(opaque_u32(smem_u32(stage_ptr(s1))), 16, 1024), 0, 0);
            umma_commit(s_full);
          }
          issue_s_tile<D, BM, BN, C::TILE_BYTES, C::TILE_BYTES, kIdS>(
              tbase + C::DP_COL, FA_VDESC(), sdesc_sw128(opaque_u32(smem_u32(stage_ptr(s1))) + C::TILE_BYTES, 16, 1024),
              0, 0);
          umma_commit(dp_full);
        }
        umma_commit(&qd_empty[s]);
      }
#undef FA_KDESC
#undef FA_VDESC
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, p.status, kSiteBwdDrain, true);
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_EW));
    // ---------------- elementwise: one key per thread, query rows along the columns ----------------
    const int eg = warp >> 2;  // query rows [64 eg, 64 eg + 64) of every tile (the columns)
    const int r = 32 * (warp & 3) + lane;
    const int j = j0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tbase + lane_off + C::S_COL;
    const uint32_t tP = tbase + lane_off + C::DP_COL;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int ti = 0; ti < T; ++ti) {
      const int s = ti % ST;
      const int m = m_lo + ti % nm;
      // ---- P^T = 2^(S^T scale log2 e - L2) as soon as S^T is in TMEM ----
      // (the L2 and D vectors were written by the copy engine: observe their arrival)
      if (!warp_wait(&qd_full[s], (ti / ST) & 1, p.status, kSiteBwdQdFull) ||
          !warp_wait(s_full, ti & 1, p.status, kSiteBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* l2v = reinterpret_cast<const float*>(stage_ptr(s) + 2 * C::TILE_BYTES);
      const float* dv = l2v + 128;
      // row i (column c) sees this key iff c >= cmin and c <= cmax (relative to the tile)
      const int i0 = m * BM;
      int cmin = 0, cmax = BM - 1;
      if (j >= p.skv) cmin = BM;  // a key past the end: nothing
      if (p.causal) cmin = max(cmin, j - p.off - i0);        // j <= i + off
      if (p.local) cmax = min(cmax, j - p.left_off - i0);    // j >= i + left_off
      // both chunks of this warpgroup (one per half) are loaded at once, so the
      // second load's latency hides behind the first chunk's arithmetic
      uint32_t sv[2][32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) tmem_ld32_issue(tS + hf * (BM / 2) + eg * 32, sv[hf]);
      tmem_ld_wait();
      reg_fence<32>(sv[0]);
      reg_fence<32>(sv[1]);
      float pf[2][32];  // P in fp32 (times 1 - tanh^2 under softcap), kept for dS
      const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = hf * (BM / 2) + eg * 32;  // warpgroup eg takes chunk eg of each half
        // the mask only where an edge cuts this chunk; pairs of columns in packed f32x2 math
        const bool edge = cmin > c0 || cmax < c0 + 31;
        uint32_t pp[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          // L2 of four query rows at once (the same address in every lane)
          const float4 l4 = *reinterpret_cast<const float4*>(l2v + c0 + i);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float2 nl = e == 0 ? make_float2(-l4.x, -l4.y) : make_float2(-l4.z, -l4.w);
            float2 x, w = make_float2(1.f, 1.f);
            if constexpr (SC) {
              // capped score c log2(e) tanh(s / c); dS gains w = 1 - tanh^2
              const float t0 = tanh_from_exp2_arg(__uint_as_float(sv[hf][i + e]) * p.sc_k);
              const float t1 = tanh_from_exp2_arg(__uint_as_float(sv[hf][i + e + 1]) * p.sc_k);
              x = make_float2(fmaf(p.sc_b, t0, nl.x), fmaf(p.sc_b, t1, nl.y));
              w = make_float2(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
            } else {
              x = __ffma2_rn(make_float2(__uint_as_float(sv[hf][i + e]), __uint_as_float(sv[hf][i + e + 1])), sl2v,
                             nl);
            }
            float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (edge) {
              const int c = c0 + i + e;
              if (c < cmin || c > cmax) pr.x = 0.f;
              if (c + 1 < cmin || c + 1 > cmax) pr.y = 0.f;
            }
            pp[(i + e) / 2] = pack2<BF16>(pr.x, pr.y);
            if constexpr (SC) pr = __fmul2_rn(pr, w);  // (P itself goes to dV; P w to dS)
            pf[hf][i + e] = pr.x;
            pf[hf][i + e + 1] = pr.y;
          }
        }
        tmem_st16(tS + c0, pp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_half[hf]);
      }
      // ---- dS^T = P^T (dP^T - D) once dP^T is in TMEM ----
      if (!warp_wait(dp_full, ti & 1, p.status, kSiteBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pv[2][32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) tmem_ld32_issue(tP + hf * (BM / 2) + eg * 32, pv[hf]);
      tmem_ld_wait();
      reg_fence<32>(pv[0]);
      reg_fence<32>(pv[1]);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = hf * (BM / 2) + eg * 32;
        uint32_t pd[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dv + c0 + i);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float2 nd = e == 0 ? make_float2(-d4.x, -d4.y) : make_float2(-d4.z, -d4.w);
            const float2 dpd = __fadd2_rn(make_float2(__uint_as_float(pv[hf][i + e]), __uint_as_float(pv[hf][i + e + 1])), nd);
            const float2 ds = __fmul2_rn(make_float2(pf[hf][i + e], pf[hf][i + e + 1]), dpd);
            pd[(i + e) / 2] = pack2<BF16>(ds.x, ds.y);
          }
        }
        tmem_st16(tP + c0, pd);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_half[hf]);
      }
    }
    const bool valid = j < p.skv;
    uint16_t* dvr = static_cast<uint16_t*>(p.dv) + bi * p.dv_st[0] + static_cast<int64_t>(j) * p.dv_st[1] +
                    kvh * p.dv_st[2];
    uint16_t* dkr = static_cast<uint16_t*>(p.dk) + bi * p.dk_st[0] + static_cast<int64_t>(j) * p.dk_st[1] +
                    kvh * p.dk_st[2];
    if (ok && T > 0 && warp_wait(mma_done, 0, p.status, kSiteBwdDone)) {
      tc_fence_after();
      // the first warpgroup writes dV, the second dK
      if (eg == 0)
        store_acc_row<D, BF16>(tbase + lane_off + C::ACC_COL, 1.f, dvr, valid);
      else
        store_acc_row<D, BF16>(tbase + lane_off + C::ACC_COL + D, p.scale, dkr, valid);
    } else if (ok && T == 0 && valid) {
      // no query row sees these keys: zero gradients
      uint4* z = reinterpret_cast<uint4*>(eg == 0 ? dvr : dkr);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  {
    auto kern = p.sc_b > 0.f ? fa_bwd_dq_kernel<D, BF16, true> : fa_bwd_dq_kernel<D, BF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DQ_SMEM);
    if (e != cudaSuccess) return e;
    const int64_t grid = static_cast<int64_t>(p.n_mtiles) * p.b * p.hq;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (grid > 0) kern<<<static_cast<unsigned>(grid), C::THREADS, C::DQ_SMEM, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = p.sc_b > 0.f ? fa_bwd_dkdv_kernel<D, BF16, true> : fa_bwd_dkdv_kernel<D, BF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM);
    if (e != cudaSuccess) return e;
    const int64_t grid = static_cast<int64_t>(p.n_ntiles) * p.b * p.hkv;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (grid > 0) kern<<<static_cast<unsigned>(grid), C::THREADS, C::KV_SMEM, stream>>>(p);
    return cudaGetLastError();
  }
}

}  // namespace

bool bwd_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_bwd(const BwdParams& p, int d, int dtype, cudaStream_t stream) {
  const bool bf16 = dtype == 0;
  switch (d) {
    case 64:
      return bf16 ? launch_bwd_t<64, true>(p, stream) : launch_bwd_t<64, false>(p, stream);
    case 128:
      return bf16 ? launch_bwd_t<128, true>(p, stream) : launch_bwd_t<128, false>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
