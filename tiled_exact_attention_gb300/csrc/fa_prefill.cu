// Prefill forward kernel: O = softmax(Q K^T * scale + mask) V and LSE per row,
// computed tile by tile with the online softmax so that no score matrix ever
// reaches global memory.
//
// Work decomposition (after "ai-reference-codex: forward CUDA kernel", sections
// 2-6, and "hs-black: FlashAttention 1/2/3", sections FlashAttention-2/-3):
// one CTA owns NQ (1 or 2) Q tiles of 128 rows of one (batch, head) and streams
// the K/V blocks the tiles can see through a shared-memory ring; each K/V block
// is read once per CTA.  Roles are specialised by warp:
//   * softmax warpgroups (one per Q tile, one TMEM lane = one query row per
//     thread): read S from TMEM, mask (diagonal / tail blocks only), update the
//     running max m and sum l, write P (bf16/fp16) back into the S columns,
//     rescale the O accumulator, and finally normalise O and write O and LSE;
//   * a TMA producer warp: Q tiles once, then K_j, V_j in consumption order;
//   * an MMA warp: S_t = Q_t K_j^T (both operands in shared memory) and
//     O_t += P_t V_j (P from TMEM, V from shared memory) with tcgen05, fp32
//     accumulators in TMEM.
// KV blocks are visited from the highest to the lowest index, so the blocks that
// need the elementwise causal / tail mask come first; blocks past the causal
// diagonal, or wholly outside the sliding window, are never visited (the
// n_block_min / n_block_max rule of "flash attention V2 code walkthrough",
// section 2, per Q tile).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold (log2 units)

template <int D>
struct Cfg {
  static constexpr int BM = 128;                     // rows per Q tile (= TMEM lanes)
  static constexpr int NQ = (D <= 128) ? 2 : 1;      // Q tiles per CTA
  static constexpr int BN = (D <= 128) ? 128 : 64;   // keys per K/V block
  static constexpr int STAGES = (D == 64) ? 8 : 4;   // K/V ring slots
  static constexpr int DC = D / 64;                  // 64-column (128-byte) chunks
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  // softmax warpgroups + one control warpgroup (producer, MMA issuer, two idle
  // warps) so that register budgets can be moved between whole warpgroups
  static constexpr int NUM_WARPS = 4 * NQ + 4;
  static constexpr int THREADS = 32 * NUM_WARPS;
  static constexpr int PRODUCER_WARP = 4 * NQ;
  static constexpr int MMA_WARP = 4 * NQ + 1;
  static constexpr int TMEM_COLS = 512;
  static constexpr int O_COL0 = 256;
  static constexpr int RING_OFF = NQ * Q_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * KV_BYTES;
  static constexpr int NUM_BARS = 4 * NQ + 2 * STAGES;
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * NUM_BARS + 16 + 1024;
  // Register split (NQ == 2): launched at 168 per thread (384 threads), the
  // control warpgroup drops to 72 and the two softmax warpgroups rise to 216:
  // 2 * 128 * 216 + 128 * 72 = 384 * 168.
  static constexpr int REG_SOFTMAX = 216;
  static constexpr int REG_CONTROL = 72;
  static_assert(NQ == 1 || 2 * 128 * REG_SOFTMAX + 128 * REG_CONTROL <= THREADS * 168, "register split");
  static_assert(NQ * BN <= 256, "S buffers must fit below the O columns");
  static_assert(O_COL0 + NQ * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static __device__ __forceinline__ int s_col(int t) { return t * 128; }
  static __device__ __forceinline__ int o_col(int t) { return O_COL0 + t * D; }
};

// Wait sites (recorded in the status word on timeout).
enum : int { kSiteKvEmpty = 1, kSiteQFull, kSiteKvFull, kSitePFull, kSiteSFull, kSiteOFull, kSiteDrain };

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// A bounded wait whose outcome is the same on every lane of the warp, so that the
// warp stays converged for the warp-collective TMEM instructions that follow.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status, int site) {
  const bool ok = mbar_wait(bar, parity, status, site);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Load N consecutive fp32 columns of this thread's TMEM lane (N multiple of 32).
template <int N>
__device__ __forceinline__ void tmem_load_row(uint32_t taddr, uint32_t* r) {
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t* x = r + 32 * c;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
          "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]),
          "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]),
          "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]),
          "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
        : "r"(taddr + 32 * c)
        : "memory");
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  reg_fence<N>(r);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// S_t = Q_t K^T over the head dimension: D / 16 MMAs of K = 16, both operands
// K-major with 128-byte swizzle (64-column chunks of 128-byte rows).
template <int D, int BN, int BM, int Q_BYTES, int KV_BYTES, uint32_t ID>
__device__ __forceinline__ void issue_s_tile(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc, int t, int slot) {
  const uint64_t qd = q_desc + static_cast<uint32_t>((t * Q_BYTES) >> 4);
  const uint64_t kd = k_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t offa = static_cast<uint32_t>(((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4);
    const uint32_t offb = static_cast<uint32_t>(((k >> 2) * (BN * 128) + (k & 3) * 32) >> 4);
    umma_ss(d_tmem, qd + offa, kd + offb, ID, k > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t[:, 16 k0 : 16 k1] V[16 k0 : 16 k1, :]: P from TMEM (two 16-bit
// values per column), V MN-major with 128-byte swizzle (64-column atoms BN * 128
// bytes apart, 8-row groups 1024 bytes apart).
template <int D, int BN, int KV_BYTES, uint32_t ID, int K0, int K1>
__device__ __forceinline__ void issue_pv_tile(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, int slot, bool acc) {
  const uint64_t vd = v_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
#pragma unroll
  for (int k = K0; k < K1; ++k) {
    umma_ts(o_tmem, p_tmem + k * 8, vd + static_cast<uint32_t>((k * 2048) >> 4), ID, (acc || k > 0) ? 1u : 0u);
  }
}

// VARLEN: packed variable-length sequences (p.cu_q / p.cu_k); a separate
// instantiation so that the dense kernel keeps its sizes in the constant bank.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1) fa_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<D>;
  constexpr int BM = C::BM, BN = C::BN, NQ = C::NQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + NQ;
  uint64_t* kv_empty = kv_full + C::STAGES;
  uint64_t* s_full = kv_empty + C::STAGES;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_full = p_full + NQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + NQ);
  uint8_t* ring = smem + C::RING_OFF;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which tiles this CTA owns ----
  // Longest causal row-groups first over the whole grid (longest-processing-time
  // order balances the SMs best; grouping CTAs by head measured slower).
  int idx = blockIdx.x;
  const int split = idx % p.num_splits;
  idx /= p.num_splits;
  const int bh = idx % (p.b * p.hq);
  const int m_cta = p.n_mcta - 1 - idx / (p.b * p.hq);
  const int h = bh % p.hq, bi = bh / p.hq;
  const int kvh = h / p.g;

  // ---- the sequence: one batch entry, or one packed variable-length sequence ----
  // Packed: sequence bi owns Q rows [cu_q[bi], cu_q[bi + 1]) and K/V rows
  // [cu_k[bi], cu_k[bi + 1]); its mask edges sit on its own bottom-right
  // diagonal (the host passes them relative to that diagonal).
  int sq = p.sq, skv = p.skv, off = p.off, left_off = p.left_off;
  int q_base = 0, k_base = 0, tb = bi;  // row offsets and batch coordinate in the tensor maps
  if constexpr (VARLEN) {
    q_base = p.cu_q[bi];
    sq = p.cu_q[bi + 1] - q_base;
    k_base = p.cu_k[bi];
    skv = p.cu_k[bi + 1] - k_base;
    tb = 0;
    const bool ok_seq = q_base >= 0 && sq >= 0 && q_base <= p.total_q - sq && k_base >= 0 && skv >= 0 &&
                        k_base <= p.total_k - skv && sq <= p.n_mtiles * BM;
    if (!ok_seq) {
      // nothing of this CTA has started: no copy, barrier or TMEM to release
      if (threadIdx.x == 0) record_error(p.status, kErrDeviceArg);
      return;
    }
    if ((m_cta * NQ) * BM >= sq) return;  // no row of this sequence here
    const int64_t diag = static_cast<int64_t>(skv) - sq;
    const int64_t o64 = diag + p.off, l64 = diag + p.left_off;
    off = static_cast<int>(o64 < -sq - 1 ? -sq - 1 : (o64 > skv ? skv : o64));
    left_off = static_cast<int>(l64 < -sq ? -sq : (l64 > skv ? skv : l64));
  }

  const int nblk_total = (skv + BN - 1) / BN;
  int n_lo = 0, n_cap = nblk_total;
  if (p.num_splits > 1) {
    n_lo = split * p.blocks_per_split;
    n_cap = min(nblk_total, n_lo + p.blocks_per_split);
    if (n_lo > n_cap) n_lo = n_cap;
  }
  // Tile t visits the blocks [n_lo_t[t], n_hi[t]) (empty when equal); the CTA
  // streams the union [n_lo_min, n_hi_max), which is contiguous because the
  // tiles are adjacent row ranges.
  int n_hi[NQ], n_lo_t[NQ];
  int n_hi_max = n_lo, n_lo_min = n_cap;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int row0 = (m_cta * NQ + t) * BM;
    int lo = n_lo, hi = n_lo;
    if (row0 < sq) {
      const int last_row = min(row0 + BM, sq) - 1;
      hi = n_cap;
      if (p.causal) hi = min(hi, floor_div(last_row + off, BN) + 1);
      if (p.local) lo = max(lo, floor_div(row0 + left_off, BN));
      if (hi <= lo) hi = lo = n_lo;
    }
    n_hi[t] = hi;
    n_lo_t[t] = lo;
    if (hi > lo) {
      n_hi_max = max(n_hi_max, hi);
      n_lo_min = min(n_lo_min, lo);
    }
  }
  if (n_lo_min > n_hi_max) n_lo_min = n_hi_max;
  const int N = n_hi_max - n_lo_min;  // KV blocks visited by the CTA

  // ---- setup ----
  if (threadIdx.x == 0) {
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], BM);
      mbar_init(&o_full[t], 1);
    }
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) {
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

  if (warp >= 4 * NQ) {
    // Control warpgroup: each register budget covers only its own role's code.
    if constexpr (NQ == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_CONTROL));
  if (warp == C::PRODUCER_WARP) {
    // =========================== TMA producer ===========================
    if (lane == 0 && N > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t pol_kv = l2_policy_evict_last();
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (n_hi[t] > n_lo_t[t]) {
          mbar_arrive_expect_tx(&q_full[t], C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < C::DC; ++c)
            tma_load_4d(smem + t * C::Q_BYTES + c * (BM * 128), &p.tm_q, &q_full[t], c * 64, h,
                        q_base + (m_cta * NQ + t) * BM, tb);
        }
      }
      int issued = 0;
      for (int L = 0; L < 2 * N; ++L) {
        const int slot = L % C::STAGES, use = L / C::STAGES;
        if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, p.status, kSiteKvEmpty)) break;
        const int n = n_hi_max - 1 - (L >> 1);
        const CUtensorMap* map = (L & 1) ? &p.tm_v : &p.tm_k;
        mbar_arrive_expect_tx(&kv_full[slot], C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::DC; ++c)
          tma_load_4d_hint(ring + slot * C::KV_BYTES + c * (BN * 128), map, &kv_full[slot], c * 64, kvh,
                           k_base + n * BN, tb, pol_kv);
        ++issued;
      }
      // No copy may still be in flight when the CTA leaves: wait for the last ones.
      for (int L = max(0, issued - C::STAGES); L < issued; ++L)
        if (!mbar_wait(&kv_full[L % C::STAGES], (L / C::STAGES) & 1, p.status, kSiteDrain, true)) break;
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (n_hi[t] > n_lo_t[t]) mbar_wait(&q_full[t], 0, p.status, kSiteDrain, true);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // =========================== MMA issuer ===========================
    if (lane == 0 && N > 0) {
      constexpr uint32_t kIdS = idesc_f16(BM, BN, BF16, false);
      constexpr uint32_t kIdO = idesc_f16(BM, D, BF16, true);
      // Descriptors are built once; per slot, tile and K step only the start
      // address field (low bits, address >> 4) moves, by compile-time amounts.
      const uint32_t ring_s = smem_u32(ring);
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem), 16, 1024);  // Q tile 0, K step 0
      const uint64_t k_desc = sdesc_sw128(ring_s, 16, 1024);          // slot 0 read as K (K-major)
      const uint64_t v_desc = sdesc_sw128(ring_s, BN * 128, 1024);    // slot 0 read as V (MN-major)
      auto active = [&](int t, int it) {
        const int n = n_hi_max - 1 - it;
        return n < n_hi[t] && n >= n_lo_t[t];
      };
      bool ok = true;
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (ok && n_hi[t] > n_lo_t[t]) ok = mbar_wait(&q_full[t], 0, p.status, kSiteQFull);
      int pv_count[NQ];
#pragma unroll
      for (int t = 0; t < NQ; ++t) pv_count[t] = 0;
      if (ok && (ok = mbar_wait(&kv_full[0], 0, p.status, kSiteKvFull))) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (active(t, 0)) {
            issue_s_tile<D, BN, BM, C::Q_BYTES, C::KV_BYTES, kIdS>(tbase + Cfg<D>::s_col(t), q_desc, k_desc, t, 0);
            umma_commit(&s_full[t]);
          }
        umma_commit(&kv_empty[0]);
      }
      for (int it = 0; ok && it < N; ++it) {
        const int Lv = 2 * it + 1, Lk = 2 * it + 2;
        const bool has_next = it + 1 < N;
        if (!mbar_wait(&kv_full[Lv % C::STAGES], (Lv / C::STAGES) & 1, p.status, kSiteKvFull)) break;
        tc_fence_after();
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (active(t, it)) {
            // first half of P: start PV while the softmax finishes the second half
            if (!mbar_wait(&p_full[t], pv_count[t] & 1, p.status, kSitePFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv_tile<D, BN, C::KV_BYTES, kIdO, 0, BN / 16>(tbase + Cfg<D>::o_col(t),
                                                               tbase + Cfg<D>::s_col(t), v_desc,
                                                               Lv % C::STAGES, pv_count[t] > 0);
            umma_commit(&o_full[t]);
            ++pv_count[t];
          }
          if (has_next && active(t, it + 1)) {
            if (!k_ready) {
              if (!mbar_wait(&kv_full[Lk % C::STAGES], (Lk / C::STAGES) & 1, p.status, kSiteKvFull)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_ready = true;
            }
            issue_s_tile<D, BN, BM, C::Q_BYTES, C::KV_BYTES, kIdS>(tbase + Cfg<D>::s_col(t), q_desc, k_desc, t,
                                                                   Lk % C::STAGES);
            umma_commit(&s_full[t]);
          }
        }
        if (!ok) break;
        umma_commit(&kv_empty[Lv % C::STAGES]);
        if (has_next) umma_commit(&kv_empty[Lk % C::STAGES]);
      }
    }
    __syncwarp();
  }
  } else {
    if constexpr (NQ == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    // =========================== softmax warpgroups ===========================
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = 32 * wq + lane;
    const int row0 = (m_cta * NQ + t) * BM;
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tS = tbase + lane_off + Cfg<D>::s_col(t);
    const uint32_t tO = tbase + lane_off + Cfg<D>::o_col(t);
    const float sl2 = p.scale_log2;
    // keys lo_row <= j < lim_row are visible to this row (the causal / window
    // edges folded with the tail)
    const int lim_row = p.causal ? min(skv, max(row + off + 1, 0)) : skv;
    const int lo_row = p.local ? row + left_off : 0;
    // (selects, not a runtime index: the arrays stay in registers)
    const int it0 = n_hi_max - (t == 0 ? n_hi[0] : n_hi[NQ - 1]);
    const int it_end = n_hi_max - (t == 0 ? n_lo_t[0] : n_lo_t[NQ - 1]);
    float m_run = -INFINITY, l_run = 0.f;
    int k = 0;
    bool ok = true;
    for (int it = it0; it < it_end; ++it) {
      const int n = n_hi_max - 1 - it;
      if (!warp_wait(&s_full[t], k & 1, p.status, kSiteSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (k > 0) {
        // S_k complete implies PV_{k-1} complete; observe that phase of o_full so
        // the final wait below is never more than one phase behind.
        if (!warp_wait(&o_full[t], (k - 1) & 1, p.status, kSiteOFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      uint32_t sr[BN];
      tmem_load_row<BN>(tS, sr);
      float* s = reinterpret_cast<float*>(sr);
      const bool masked = (n + 1) * BN > skv || (p.causal && (n + 1) * BN - 1 > row0 + off);
      if (masked) {
        const int lim = lim_row - n * BN;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      if (p.local && n * BN < row0 + BM - 1 + left_off) {
        const int lo = lo_row - n * BN;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c < lo) s[c] = -INFINITY;
      }
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmax3(s[2 * i], s[2 * i + 1], s[8 + i]);
#pragma unroll
      for (int c = 12; c < BN; c += 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (c + 2 * i + 1 < BN) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
        }
      }
      const float bmax = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      // The reference max moves only when the block max exceeds it by more than
      // 2^kRescaleLog2 (exact: l and o share the reference, so O = o / l is
      // unchanged); probabilities stay below 2^kRescaleLog2.
      const float bm2 = bmax * sl2;
      const bool grow = bm2 > m_run + kRescaleLog2;
      const float m_new = grow ? bm2 : m_run;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = grow ? ex2_approx(m_run - m_use) : 1.f;
      if (k > 0 && __any_sync(0xffffffffu, grow)) {
        // O_t already holds the previous blocks' product (see the o_full wait).
        // 32 columns at a time: the 128 scores are still live in registers.
        constexpr int CH = 32;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += CH) {
          uint32_t o[CH];
          tmem_load_row<CH>(tO + c0, o);
#pragma unroll
          for (int i = 0; i < CH; i += 2) {
            const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                        make_float2(alpha, alpha));
            o[i] = __float_as_uint(r.x);
            o[i + 1] = __float_as_uint(r.y);
          }
#pragma unroll
          for (int c = 0; c < CH; c += 32) tmem_st32(tO + c0 + c, *reinterpret_cast<const uint32_t(*)[32]>(o + c));
        }
      }
      // P = 2^(s * scale * log2 e - m), written over the first half of the S
      // columns as packed 16-bit pairs; the MMA warp is signalled once per block
      // (a second, earlier signal for half of P measured slower).
      const float2 sl2v = make_float2(sl2, sl2);
      const float2 negm = make_float2(-m_use, -m_use);
      float2 sum2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sum2[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[BN / 4];
#pragma unroll
        for (int c = 0; c < BN / 2; c += 2) {
          const int cc = half * (BN / 2) + c;
          const float2 x = __ffma2_rn(make_float2(s[cc], s[cc + 1]), sl2v, negm);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          sum2[(c >> 1) & 3] = __fadd2_rn(sum2[(c >> 1) & 3], e);
          pk[c >> 1] = pack2<BF16>(e.x, e.y);
        }
#pragma unroll
        for (int c = 0; c < BN / 4; c += 16)
          tmem_st16(tS + half * (BN / 4) + c, *reinterpret_cast<const uint32_t(*)[16]>(pk + c));
        if (half == 1) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full[t]);
        }
      }
      const float2 s01 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      l_run = alpha * l_run + (s01.x + s01.y);
      m_run = m_new;
      ++k;
    }

    // ---------------- epilogue ----------------
    const bool split_mode = p.num_splits > 1;
    // LSE [b][hq][sq], or [hq][total_q] for packed sequences
    const int64_t lse_idx = VARLEN ? static_cast<int64_t>(h) * p.total_q + q_base + row
                                   : (static_cast<int64_t>(bi) * p.hq + h) * sq + row;
    uint16_t* o_row = static_cast<uint16_t*>(p.o) + bi * p.o_stride_b +
                      static_cast<int64_t>(q_base + row) * p.o_stride_row + h * p.o_stride_h;
    if (ok && k == 0) {
      // This tile sees no key (in this split): O = 0, LSE = -inf.
      if (row < sq) {
        if (split_mode) {
          const int64_t prow = ((static_cast<int64_t>(split) * p.b + bi) * p.hq + h) * sq + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse[prow] = -INFINITY;
        } else {
          uint4* dst = reinterpret_cast<uint4*>(o_row);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[lse_idx] = -INFINITY;
        }
      }
    } else if (ok) {
      if (warp_wait(&o_full[t], (k - 1) & 1, p.status, kSiteOFull)) {
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse = l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
        if (split_mode) {
          // The TMEM loads are warp-collective: every lane executes them and only
          // the global stores depend on whether the row exists.
          const bool valid = row < sq;
          const int64_t prow = ((static_cast<int64_t>(split) * p.b + bi) * p.hq + h) * sq + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_load_row<32>(tO + c, o);
            if (valid) {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                dst[(c + i) / 4] = make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                               __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
            }
          }
          if (valid) p.lse[prow] = lse;
        } else if (VARLEN && row0 + BM > sq) {
          // The last tile of a packed sequence: a 128-row TMA store would also write
          // the next sequence's rows, so each thread stores its own row.
          const bool valid = row < sq;
          uint4* dst = reinterpret_cast<uint4*>(o_row);
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_load_row<32>(tO + c, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            if (valid) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[c / 8 + q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
          }
          if (valid) p.lse[lse_idx] = lse;
        } else {
          // Stage O (normalised, rounded) through the Q tile's shared memory in the
          // same 128-byte-swizzled layout the TMA store reads.
          uint8_t* stage = smem + t * C::Q_BYTES;
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_load_row<32>(tO + c, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            const int cc = c >> 6;               // 64-column chunk
            const int piece0 = (c & 63) >> 3;   // first 16-byte piece within the 128-byte row
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int piece = piece0 + q4;
              uint4* dst = reinterpret_cast<uint4*>(stage + cc * (BM * 128) + r * 128 + ((piece ^ (r & 7)) << 4));
              *dst = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + t, BM);
          if (r == 0) {
#pragma unroll
            for (int cc = 0; cc < C::DC; ++cc)
              tma_store_4d(&p.tm_o, stage + cc * (BM * 128), cc * 64, h, q_base + row0, tb);
            bulk_commit_group();
            bulk_wait_group_read0();
          }
          if (row < sq) p.lse[lse_idx] = lse;
        }
      }
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
cudaError_t launch_t(const PrefillParams& p, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = p.cu_q != nullptr ? fa_prefill_kernel<D, BF16, true> : fa_prefill_kernel<D, BF16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_mcta) * p.b * p.hq * p.num_splits;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int prefill_block_n(int d) { return d <= 128 ? 128 : 64; }
int prefill_q_tiles(int d) { return d <= 128 ? 2 : 1; }

cudaError_t launch_prefill(const PrefillParams& p, int d, int dtype, cudaStream_t stream) {
  const bool bf16 = dtype == 0;
  switch (d) {
    case 64:
      return bf16 ? launch_t<64, true>(p, stream) : launch_t<64, false>(p, stream);
    case 128:
      return bf16 ? launch_t<128, true>(p, stream) : launch_t<128, false>(p, stream);
    case 256:
      return bf16 ? launch_t<256, true>(p, stream) : launch_t<256, false>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
