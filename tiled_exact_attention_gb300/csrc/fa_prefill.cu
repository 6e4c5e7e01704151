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
//     running max m and sum l, write P (bf16/fp16, or e4m3) back into TMEM (over
//     the S columns, or for d = 256 into columns of its own), rescale the O
//     accumulator, and finally normalise O and write O (through shared-memory
//     slices and TMA stores for d <= 128) and LSE;
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
#include "tc_common.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold (log2 units)

// E8: e4m3 Q, K, V (one byte per element) and e4m3 P.
template <int D, bool E8 = false>
struct Cfg {
  static constexpr int ELT = E8 ? 1 : 2;             // bytes per input element
  static constexpr int BM = 128;                     // rows per Q tile (= TMEM lanes)
  static constexpr int NQ = (D <= 128) ? 2 : 1;      // Q tiles per CTA
  // keys per K/V block (e4m3: 128, so that a row of the transposed V tile is 128 bytes)
  static constexpr int BN = (D <= 128 || E8) ? 128 : 64;
  static constexpr int STAGES = E8 ? (D == 256 ? 4 : 8) : (D == 64 ? 8 : 4);  // K/V ring slots
  // d = 256 (one row tile per CTA: every tile re-reads its head's K/V, mostly from
  // DRAM) also prefetches each K/V block into L2 two blocks ahead of its load:
  // measured +3.8% there, -3% on the causal d = 128 prefill
  static constexpr int KV_PREFETCH = (D == 256 && !E8) ? 2 : 0;
  // Q and K rows are staged in swizzle chunks of CHUNK_BYTES: 128-byte rows with the
  // 128-byte swizzle, or (e4m3, d = 64) one 64-byte chunk with the 64-byte swizzle
  static constexpr int ROW_BYTES = D * ELT;
  static constexpr int CHUNK_BYTES = ROW_BYTES < 128 ? ROW_BYTES : 128;
  static constexpr bool SW64 = CHUNK_BYTES == 64;
  static constexpr int DC = ROW_BYTES / CHUNK_BYTES;     // chunks per row
  static constexpr int CHUNK_ELEMS = CHUNK_BYTES / ELT;  // elements per chunk
  static constexpr int Q_BYTES = BM * D * ELT;
  static constexpr int KV_BYTES = BN * D * ELT;
  // softmax warpgroups + one control warpgroup (producer, MMA issuer, two idle
  // warps) so that register budgets can be moved between whole warpgroups
  static constexpr int NUM_WARPS = 4 * NQ + 4;
  static constexpr int THREADS = 32 * NUM_WARPS;
  static constexpr int PRODUCER_WARP = 4 * NQ;
  static constexpr int MMA_WARP = 4 * NQ + 1;
  static constexpr int TMEM_COLS = 512;
  static constexpr int O_COL0 = 256;
  static constexpr int RING_OFF = NQ * Q_BYTES;
  // O staging of the TMA-store epilogue (d <= 128; for d = 256 it measured 1.6%
  // slower than row-by-row stores): per softmax warp 32 rows x 64 columns of
  // 16-bit O (4 KB, 128-byte swizzle, 1024-byte aligned)
  static constexpr bool TMA_O = D <= 128;
  static constexpr int STG_OFF = RING_OFF + STAGES * KV_BYTES;
  static constexpr int STG_WARP = 32 * 128;
  static constexpr int BAR_OFF = STG_OFF + (TMA_O ? 4 * NQ * STG_WARP : 0);
  static constexpr int NUM_BARS = 3 + 7 * NQ + 2 * STAGES;
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
  // d = 256: P in TMEM columns of its own (S 64 + O 256 leave 192 free), so that
  // the next block's S is computed while the softmax still works on this one
  // (measured +17%).  d = 128 has no free columns (S 2 x 128 + O 2 x 128), and for
  // d = 64, where 128 are free, the same measured 3-8% slower: there P
  // overwrites S and the next S waits for the PV that reads it.
  static constexpr bool P_SEP = D == 256;
  static __device__ __forceinline__ int p_col(int t) { return P_SEP ? 128 : t * 128; }
  static __device__ __forceinline__ int o_col(int t) { return O_COL0 + t * D; }
};

// Wait sites (recorded in the status word on timeout).
enum : int {
  kSiteKvEmpty = 1,
  kSiteQFull,
  kSiteKvFull,
  kSitePFull,
  kSiteSFull,
  kSiteOFull,
  kSiteDrain,
  kSiteQEmpty,
  kSiteOEmpty,
  kSiteSFree,
  kSitePFree
};

// One work item: NQ Q tiles of one (split, batch or packed sequence, head) and
// the key-block ranges they visit.  Every role derives the same plan from the
// item index, so the roles need no channel to agree on it.
template <int NQ>
struct ItemPlan {
  int bi, h, kvh, m_cta, split;
  int sq, skv, off, left_off;  // the sequence's sizes and mask edges
  int q_base, k_base, tb;      // packed row offsets; batch coordinate of the Q map
  int tbk;                     // batch coordinate of the K/V maps (a KV cache's pages: per block)
  int n_hi[NQ], n_lo_t[NQ];    // tile t visits key blocks [n_lo_t[t], n_hi[t])
  int n_hi_max;                // the CTA streams blocks n_hi_max - 1 down to n_hi_max - N
  int N;
  bool valid;                  // false: packed offsets out of range (nothing is touched)
};

// E8 selects the 8-bit configuration, whose key blocks are 128 keys at every d
// (the 16-bit d = 256 configuration uses 64): the plan counts blocks of the
// kernel's own size.
template <int D, bool VARLEN, bool CACHE, bool E8 = false>
__device__ __forceinline__ ItemPlan<Cfg<D, E8>::NQ> plan_item(const PrefillParams& p, int item) {
  using C = Cfg<D, E8>;
  constexpr int BM = C::BM, BN = C::BN, NQ = C::NQ;
  ItemPlan<NQ> w;
  // Items are numbered longest causal row-group first (longest-processing-time
  // order balances the SMs best; grouping work by head measured slower).
  int idx = item;
  w.split = idx % p.num_splits;
  idx /= p.num_splits;
  const int bh = idx % (p.b * p.hq);
  w.m_cta = p.n_mcta - 1 - idx / (p.b * p.hq);
  w.h = bh % p.hq;
  w.bi = bh / p.hq;
  w.kvh = w.h / p.g;
  w.sq = p.sq;
  w.skv = p.skv;
  w.off = p.off;
  w.left_off = p.left_off;
  w.q_base = 0;
  w.k_base = 0;
  w.tb = w.bi;
  w.tbk = w.bi;
  w.valid = true;
  if constexpr (CACHE) {
    // KV cache: dense Q; the sequence's own keys, paged or packed (clamped
    // lengths; a page or row outside the cache reads as zeros, never faults)
    // The lengths live on the device and are checked before anything they
    // address is read: a paged sequence may not outrun its block-table row, a
    // packed one must lie inside the packed rows (else the item is skipped and
    // FA_ERR_DEVICE_ARG recorded).
    w.tbk = 0;
    if (p.kv_mode == kKvPaged) {
      const int len = p.seqlens[w.bi];
      w.valid = static_cast<int64_t>(len) <= static_cast<int64_t>(p.bt_stride) * p.page_size;
      w.skv = w.valid ? max(len, 0) : 0;
    } else {
      const int beg = p.cu_k[w.bi], end = p.cu_k[w.bi + 1];
      w.valid = beg >= 0 && end >= beg && end <= p.total_k;
      w.k_base = w.valid ? beg : 0;
      w.skv = w.valid ? end - beg : 0;
    }
  } else if constexpr (VARLEN) {
    // Packed: sequence bi owns Q rows [cu_q[bi], cu_q[bi + 1]) and K/V rows
    // [cu_k[bi], cu_k[bi + 1]); its mask edges sit on its own bottom-right
    // diagonal (the host passes them relative to that diagonal).
    w.q_base = p.cu_q[w.bi];
    w.sq = p.cu_q[w.bi + 1] - w.q_base;
    w.k_base = p.cu_k[w.bi];
    w.skv = p.cu_k[w.bi + 1] - w.k_base;
    w.tb = 0;
    w.tbk = 0;
    w.valid = w.q_base >= 0 && w.sq >= 0 && w.q_base <= p.total_q - w.sq && w.k_base >= 0 && w.skv >= 0 &&
              w.k_base <= p.total_k - w.skv && w.sq <= p.n_mtiles * BM;
    if (!w.valid) {
      w.sq = 0;
      w.skv = 0;
    }
    const int64_t diag = static_cast<int64_t>(w.skv) - w.sq;
    const int64_t o64 = diag + p.off, l64 = diag + p.left_off;
    w.off = static_cast<int>(o64 < -w.sq - 1 ? -w.sq - 1 : (o64 > w.skv ? w.skv : o64));
    w.left_off = static_cast<int>(l64 < -w.sq ? -w.sq : (l64 > w.skv ? w.skv : l64));
  }
  const int nblk_total = (w.skv + BN - 1) / BN;
  int n_lo = 0, n_cap = nblk_total;
  if (p.num_splits > 1) {
    // (a KV cache cuts every sequence into num_splits ranges of its own length)
    const int bps =
        CACHE ? max(1, (nblk_total + p.num_splits - 1) / p.num_splits) : p.blocks_per_split;
    n_lo = w.split * bps;
    n_cap = min(nblk_total, n_lo + bps);
    if (n_lo > n_cap) n_lo = n_cap;
  }
  // The union of the tiles' ranges is contiguous: the tiles are adjacent rows.
  int n_hi_max = n_lo, n_lo_min = n_cap;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int row0 = (w.m_cta * NQ + t) * BM;
    int lo = n_lo, hi = n_lo;
    if (row0 < w.sq) {
      const int last_row = min(row0 + BM, w.sq) - 1;
      hi = n_cap;
      if (p.causal) hi = min(hi, floor_div(last_row + w.off, BN) + 1);
      if (p.local) lo = max(lo, floor_div(row0 + w.left_off, BN));
      if (hi <= lo) hi = lo = n_lo;
    }
    w.n_hi[t] = hi;
    w.n_lo_t[t] = lo;
    if (hi > lo) {
      n_hi_max = max(n_hi_max, hi);
      n_lo_min = min(n_lo_min, lo);
    }
  }
  if (n_lo_min > n_hi_max) n_lo_min = n_hi_max;
  w.n_hi_max = n_hi_max;
  w.N = n_hi_max - n_lo_min;
  return w;
}

// The S and PV products in the 16-bit or the e4m3 form.
// (W: issued by the whole MMA warp, one elected lane issuing; see umma_ss)
template <int D, int BN, int BM, int Q_BYTES, int KV_BYTES, uint32_t ID, bool E8, bool W>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc, int t, int slot) {
  if constexpr (E8)
    issue_s_tile_e4m3<D, BN, BM, Q_BYTES, KV_BYTES, ID, W, (D < 128 ? D : 128)>(d_tmem, q_desc, k_desc, t, slot);
  else
    issue_s_tile<D, BN, BM, Q_BYTES, KV_BYTES, ID, W>(d_tmem, q_desc, k_desc, t, slot);
}

template <int D, int BN, int KV_BYTES, uint32_t ID, bool E8, bool W>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, int slot, bool acc) {
  if constexpr (E8)
    issue_pv_tile_e4m3<D, BN, KV_BYTES, ID, W>(o_tmem, p_tmem, v_desc, slot, acc);
  else
    issue_pv_tile<D, BN, KV_BYTES, ID, 0, BN / 16, W>(o_tmem, p_tmem, v_desc, slot, acc);
}

// A wait of the MMA issuer: warp-uniform when the whole warp issues (W), else
// the issuing thread's own.
template <bool W>
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, int* status, int site) {
  if constexpr (W)
    return warp_wait(bar, parity, status, site);
  else
    return mbar_wait(bar, parity, status, site);
}

// The j-th item of this CTA: a boustrophedon over the item list (CTA c takes c,
// 2G - 1 - c, 2G + c, ...), so that with items in decreasing size every CTA gets
// one large and one small item from each pair of rounds.
__device__ __forceinline__ int item_of(int j) {
  const int G = gridDim.x, c = blockIdx.x;
  return (j & 1) ? (j + 1) * G - 1 - c : j * G + c;
}

// VARLEN: packed variable-length sequences (p.cu_q / p.cu_k); a separate
// instantiation so that the dense kernel keeps its sizes in the constant bank.
// CACHE (with VARLEN): a KV cache read with dense Q (p.kv_mode), again a
// separate instantiation so that the packed-sequence kernel keeps its code.
//
// Persistent: one CTA per SM walks its items; the producer loads the next
// item's Q as soon as the last S MMA of the current item has read Q, and the MMA
// warp starts the next item's S MMAs while the softmax warps write the current
// item's output (its PV MMAs wait only until the previous O has been read out).
// SC: softcap, each score capped to c tanh(s / c) before the mask (a separate
// instantiation: two more special-function operations per score).
template <int D, bool BF16, bool VARLEN, bool E8 = false, bool SC = false, bool CACHE = false>
__global__ void __launch_bounds__(Cfg<D, E8>::THREADS, 1) fa_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<D, E8>;
  constexpr int BM = C::BM, BN = C::BN, NQ = C::NQ;
  // P released in two halves of the block's keys (the first half's PV runs while
  // the second is formed): measured faster for d = 64 (+6%), d = 256 (+5%) and
  // softcap (+2%), slower for d = 128 (-3%, long GQA -7%)
  constexpr bool HALF_P = !E8 && (D != 128 || SC);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 1;
  uint64_t* kv_full = q_empty + 1;
  uint64_t* kv_empty = kv_full + C::STAGES;
  uint64_t* s_full = kv_empty + C::STAGES;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_full = p_full + NQ;
  uint64_t* o_empty = o_full + NQ;
  uint64_t* mma_done = o_empty + NQ;
  uint64_t* p_half = mma_done + 1;  // P of the block's first half of keys written
  uint64_t* s_free = p_half + NQ;   // (P_SEP) the softmax has loaded S: the next S may overwrite it
  uint64_t* p_free = s_free + NQ;   // (P_SEP) a block's PV has completed: P may be rewritten, O rescaled
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_free + NQ);
  uint8_t* ring = smem + C::RING_OFF;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total_items = p.n_mcta * p.b * p.hq * p.num_splits;

  // ---- setup ----
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(mma_done, 1);
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], BM);
      mbar_init(&p_half[t], BM);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], BM);
      mbar_init(&s_free[t], BM);
      mbar_init(&p_free[t], 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      if (p.skv > 0 || p.total_k > 0) {  // the K/V maps exist
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
      }
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t gL = 0;       // K/V block loads issued by this CTA
      uint32_t q_loads = 0;  // Q loads issued by this CTA
      bool ok = true;
      for (int j = 0; ok; ++j) {
        const int item = item_of(j);
        if (item >= total_items) break;
        const ItemPlan<NQ> w = plan_item<D, VARLEN, CACHE, E8>(p, item);
        if (w.N == 0) continue;
        // Q buffer free: the previous item's S MMAs have completed
        if (q_loads > 0 && !mbar_wait(q_empty, (q_loads - 1) & 1, p.status, kSiteQEmpty)) break;
        uint32_t q_bytes = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (w.n_hi[t] > w.n_lo_t[t]) q_bytes += C::Q_BYTES;
        mbar_arrive_expect_tx(q_full, q_bytes);
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (w.n_hi[t] > w.n_lo_t[t]) {
#pragma unroll
            for (int c = 0; c < C::DC; ++c)
              tma_load_4d(smem + t * C::Q_BYTES + c * (BM * C::CHUNK_BYTES), &p.tm_q, q_full, c * C::CHUNK_ELEMS, w.h,
                          w.q_base + (w.m_cta * NQ + t) * BM, w.tb);
          }
        }
        ++q_loads;
        {
          // warm L2 with the next item's Q; its load is issued only when this
          // item's last S MMA has read the Q buffer
          const int nxt = item_of(j + 1);
          if (nxt < total_items) {
            const int idx = nxt / p.num_splits;
            const int bh = idx % (p.b * p.hq);
            const int m_cta = p.n_mcta - 1 - idx / (p.b * p.hq);
            const int bi = bh / p.hq, h = bh % p.hq;
            int base = 0, rows = p.sq, tb = bi;
            if constexpr (VARLEN && !CACHE) {  // (offsets are range-checked when the item itself is planned)
              base = p.cu_q[bi];
              rows = min(p.cu_q[bi + 1] - base, p.n_mtiles * BM);
              tb = 0;
            }
#pragma unroll
            for (int t = 0; t < NQ; ++t)
              if ((m_cta * NQ + t) * BM < rows) {
#pragma unroll
                for (int c = 0; c < C::DC; ++c)
                  tma_prefetch_l2_4d(&p.tm_q, c * C::CHUNK_ELEMS, h, base + (m_cta * NQ + t) * BM, tb);
              }
          }
        }
        for (int L = 0; L < 2 * w.N; ++L, ++gL) {
          const uint32_t slot = gL % C::STAGES, use = gL / C::STAGES;
          // (the producer runs ahead of its consumers: it backs off while it waits)
          if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, p.status, kSiteKvEmpty, false, 128)) {
            ok = false;
            break;
          }
          const int n = w.n_hi_max - 1 - (L >> 1);
          mbar_arrive_expect_tx(&kv_full[slot], C::KV_BYTES);
          if (E8 && (L & 1)) {
            // V transposed ([d rows][keys]): one box of D rows x BN keys
            tma_load_4d_hint(ring + slot * C::KV_BYTES, &p.tm_v, &kv_full[slot], w.k_base + n * BN, 0, w.kvh, w.tbk,
                             pol_kv);
          } else if (CACHE && p.kv_mode == kKvPaged) {
            // paged cache: box_rows keys per box (BN, or 64 when a page holds no
            // whole block), each from its page; a box past the sequence's end
            // (rows masked) reuses the block's first page
            const CUtensorMap* map = (L & 1) ? &p.tm_v : &p.tm_k;
            const int* bt_row = p.block_table + static_cast<int64_t>(w.bi) * p.bt_stride;
            const int r0 = n * BN;
            const int pg0 = bt_row[r0 / p.page_size];
            for (int sb = 0; sb * p.box_rows < BN; ++sb) {
              const int r = r0 + sb * p.box_rows;
              const int pg = (sb == 0 || r >= w.skv) ? pg0 : bt_row[r / p.page_size];
#pragma unroll
              for (int c = 0; c < C::DC; ++c)
                tma_load_4d_hint(ring + slot * C::KV_BYTES + c * (BN * 128) + sb * p.box_rows * 128, map,
                                 &kv_full[slot], c * C::CHUNK_ELEMS, w.kvh, r % p.page_size, pg, pol_kv);
            }
          } else {
            const CUtensorMap* map = (L & 1) ? &p.tm_v : &p.tm_k;
#pragma unroll
            for (int c = 0; c < C::DC; ++c)
              tma_load_4d_hint(ring + slot * C::KV_BYTES + c * (BN * C::CHUNK_BYTES), map, &kv_full[slot], c * C::CHUNK_ELEMS,
                               w.kvh, w.k_base + n * BN, w.tbk, pol_kv);
            if constexpr (C::KV_PREFETCH > 0) {
              // warm L2 with the same tensor's block KV_PREFETCH blocks further on
              const int npf = n - C::KV_PREFETCH;
              if (npf >= w.n_hi_max - w.N) {
#pragma unroll
                for (int c = 0; c < C::DC; ++c)
                  tma_prefetch_l2_4d(map, c * C::CHUNK_ELEMS, w.kvh, w.k_base + npf * BN, w.tbk);
              }
            }
          }
        }
      }
      // No copy may still be in flight when the CTA leaves: wait for the last ones.
      for (uint32_t L = gL > C::STAGES ? gL - C::STAGES : 0; L < gL; ++L)
        if (!mbar_wait(&kv_full[L % C::STAGES], (L / C::STAGES) & 1, p.status, kSiteDrain, true)) break;
      if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, p.status, kSiteDrain, true);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // =========================== MMA issuer ===========================
    // The whole warp runs the issue loop, converged, and one elected lane issues:
    // the issuer then runs ahead of the tensor pipe (measured +3.5% on the causal
    // prefill, +4% on long GQA).  Softcap and e4m3, whose softmax sets the pace,
    // measured faster with lane 0 alone issuing (703 vs 671 TFLOP/s with softcap).
    constexpr bool WI = !SC && !E8;
    if (WI || lane == 0) {
      constexpr uint32_t kIdS = E8 ? idesc_e4m3(BM, BN) : idesc_f16(BM, BN, BF16, false);
      constexpr uint32_t kIdO = E8 ? idesc_e4m3(BM, D) : idesc_f16(BM, D, BF16, true);
      // Descriptors are built once; per slot, tile and K step only the start
      // address field (low bits, address >> 4) moves, by compile-time amounts.
      const uint32_t ring_s = smem_u32(ring);
      // Q tile 0 and slot 0 read as K (K-major), K step 0
      const uint64_t q_desc = C::SW64 ? sdesc_sw64(smem_u32(smem), 16, 512) : sdesc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t k_desc = C::SW64 ? sdesc_sw64(ring_s, 16, 512) : sdesc_sw128(ring_s, 16, 1024);
      // slot 0 read as V: MN-major (16-bit), or K-major V^T (e4m3)
      const uint64_t v_desc = E8 ? sdesc_sw128(ring_s, 16, 1024) : sdesc_sw128(ring_s, BN * 128, 1024);
      uint32_t gL = 0, q_uses = 0;
      constexpr bool PS = C::P_SEP;
      uint32_t pv_cnt[NQ], o_uses[NQ], s_iss[NQ];  // s_iss: S tiles issued per Q tile (P_SEP)
#pragma unroll
      for (int t = 0; t < NQ; ++t) pv_cnt[t] = o_uses[t] = s_iss[t] = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        const int item = item_of(j);
        if (item >= total_items) break;
        int N, it_b[NQ], it_e[NQ];  // tile t is active in iterations [it_b[t], it_e[t])
        {
          const ItemPlan<NQ> w = plan_item<D, VARLEN, CACHE, E8>(p, item);
          N = w.N;
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            it_b[t] = w.n_hi_max - w.n_hi[t];
            it_e[t] = w.n_hi_max - w.n_lo_t[t];
          }
        }
        if (N == 0) continue;
#define FA_ACTIVE(t, it) ((it) >= it_b[t] && (it) < it_e[t])
        if (!issuer_wait<WI>(q_full, q_uses & 1, p.status, kSiteQFull)) break;
        ++q_uses;
        if (!issuer_wait<WI>(&kv_full[gL % C::STAGES], (gL / C::STAGES) & 1, p.status, kSiteKvFull)) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (FA_ACTIVE(t, 0)) {
            if constexpr (PS) {  // the S buffer is free once the softmax has loaded the previous S
              if (s_iss[t] > 0 && !issuer_wait<WI>(&s_free[t], (s_iss[t] - 1) & 1, p.status, kSiteSFree)) {
                ok = false;
                break;
              }
              tc_fence_after();
              ++s_iss[t];
            }
            issue_s<D, BN, BM, C::Q_BYTES, C::KV_BYTES, kIdS, E8, WI>(tbase + C::s_col(t), q_desc, k_desc, t,
                                                                   gL % C::STAGES);
            umma_commit<WI>(&s_full[t]);
          }
        if (!ok) break;
        if (N == 1) umma_commit<WI>(q_empty);  // the item's last S has been issued
        umma_commit<WI>(&kv_empty[gL % C::STAGES]);
        for (int it = 0; it < N; ++it) {
          const uint32_t Lv = gL + 2 * it + 1, Lk = gL + 2 * it + 2;
          const bool has_next = it + 1 < N;
          bool k_ready = false;
          if (!issuer_wait<WI>(&kv_full[Lv % C::STAGES], (Lv / C::STAGES) & 1, p.status, kSiteKvFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (PS && has_next && FA_ACTIVE(t, it + 1)) {
              // the tile's next S first: it waits only until the softmax has loaded
              // the current S, and runs while the softmax forms P
              if (!k_ready) {
                if (!issuer_wait<WI>(&kv_full[Lk % C::STAGES], (Lk / C::STAGES) & 1, p.status, kSiteKvFull)) {
                  ok = false;
                  break;
                }
                k_ready = true;
              }
              if (s_iss[t] > 0 && !issuer_wait<WI>(&s_free[t], (s_iss[t] - 1) & 1, p.status, kSiteSFree)) {
                ok = false;
                break;
              }
              tc_fence_after();
              ++s_iss[t];
              issue_s<D, BN, BM, C::Q_BYTES, C::KV_BYTES, kIdS, E8, WI>(tbase + C::s_col(t), q_desc, k_desc, t,
                                                                     Lk % C::STAGES);
              umma_commit<WI>(&s_full[t]);
            }
            if (FA_ACTIVE(t, it)) {
              if (!issuer_wait<WI>(HALF_P ? &p_half[t] : &p_full[t], pv_cnt[t] & 1, p.status, kSitePFull)) {
                ok = false;
                break;
              }
              // the first PV of an item overwrites O: the previous item's O must be read out
              const bool first = it == it_b[t];
              if (first && o_uses[t] > 0 && !issuer_wait<WI>(&o_empty[t], (o_uses[t] - 1) & 1, p.status, kSiteOEmpty)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if constexpr (!HALF_P) {
                issue_pv<D, BN, C::KV_BYTES, kIdO, E8, WI>(tbase + C::o_col(t), tbase + C::p_col(t), v_desc,
                                                           Lv % C::STAGES, !first);
              } else {
                // the block's first 64 keys as soon as their P is written, then the rest
                issue_pv_tile<D, BN, C::KV_BYTES, kIdO, 0, BN / 32, WI>(tbase + C::o_col(t), tbase + C::p_col(t),
                                                                       v_desc, Lv % C::STAGES, !first);
                if (!issuer_wait<WI>(&p_full[t], pv_cnt[t] & 1, p.status, kSitePFull)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_pv_tile<D, BN, C::KV_BYTES, kIdO, BN / 32, BN / 16, WI>(tbase + C::o_col(t), tbase + C::p_col(t),
                                                                             v_desc, Lv % C::STAGES, true);
              }
              if constexpr (PS) umma_commit<WI>(&p_free[t]);
              if (it + 1 == it_e[t]) umma_commit<WI>(&o_full[t]);  // the tile's last PV of the item
              ++pv_cnt[t];
            }
            if (!PS && has_next && FA_ACTIVE(t, it + 1)) {
              if (!k_ready) {
                if (!issuer_wait<WI>(&kv_full[Lk % C::STAGES], (Lk / C::STAGES) & 1, p.status, kSiteKvFull)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                k_ready = true;
              }
              issue_s<D, BN, BM, C::Q_BYTES, C::KV_BYTES, kIdS, E8, WI>(tbase + C::s_col(t), q_desc, k_desc, t,
                                                                     Lk % C::STAGES);
              umma_commit<WI>(&s_full[t]);
            }
          }
          if (!ok) break;
          if (it + 2 == N) umma_commit<WI>(q_empty);  // the item's last S has been issued
          umma_commit<WI>(&kv_empty[Lv % C::STAGES]);
          if (has_next) umma_commit<WI>(&kv_empty[Lk % C::STAGES]);
        }
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (it_e[t] > it_b[t]) ++o_uses[t];
#undef FA_ACTIVE
        gL += 2 * N;
      }
      // Every barrier arrive of the MMAs issued above has landed before the CTA
      // leaves (the commits complete in order).
      umma_commit<WI>(mma_done);
      mbar_wait(mma_done, 0, p.status, kSiteDrain, true);
    }
    __syncwarp();
  }
  } else {
    if constexpr (NQ == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    // =========================== softmax warpgroups ===========================
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = 32 * wq + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tS = tbase + lane_off + C::s_col(t);
    const uint32_t tP = tbase + lane_off + C::p_col(t);
    const uint32_t tO = tbase + lane_off + C::o_col(t);
    const float sl2 = p.scale_log2;
    const bool split_mode = p.o_part != nullptr;
    uint32_t gblk = 0;  // key blocks this tile has processed, over all items
    uint32_t oitems = 0;  // items whose O this tile has read out (o_full completes once per item)
    uint32_t g_loads = 0;  // K/V loads of the items before this one (the producer's count)
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int item = item_of(j);
      if (item >= total_items) break;
      int row0, n_top, it0, it_end, skv, off, left_off;
      float sl2q = sl2;        // e4m3: the tile's Q scale folded into the score scale
      const float* kd = nullptr;  // e4m3: the K scales of this head's key blocks
      {
        const ItemPlan<NQ> w = plan_item<D, VARLEN, CACHE, E8>(p, item);
        const uint32_t first_load = g_loads;
        if constexpr (CACHE) g_loads += 2 * w.N;
        if (VARLEN && !w.valid) {
          if (threadIdx.x == 0) record_error(p.status, kErrDeviceArg);
          continue;
        }
        row0 = (w.m_cta * NQ + t) * BM;
        if (row0 >= w.sq) continue;  // no row of this tile in the sequence
        if (CACHE && t == 0 && w.N > 0 && w.skv - (w.n_hi_max - 1) * BN < BN) {
          // KV cache: rows past a sequence's end may hold anything (NaN too) and
          // 0 * NaN is NaN in P V, so tile 0's threads zero the V rows of the
          // block that ends the sequence (the item's first) before its P is
          // released: generic stores, then the proxy fence that orders them
          // before the tensor core's reads; the slot is not refilled before that
          // PV has completed.
          const int v_zero = w.skv - (w.n_hi_max - 1) * BN;
          const uint32_t v_load = first_load + 1, slot = v_load % C::STAGES;
          if (!warp_wait(&kv_full[slot], (v_load / C::STAGES) & 1, p.status, kSiteKvFull)) {
            ok = false;
            break;
          }
          uint8_t* vs = ring + slot * C::KV_BYTES;
          const int units = (BN - v_zero) * C::DC * 8;  // 16-byte units
          for (int u = r; u < units; u += BM) {
            const int row = v_zero + u / (C::DC * 8), c = (u >> 3) % C::DC;
            *reinterpret_cast<uint4*>(vs + c * (BN * 128) + row * 128 + (u & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        if constexpr (E8) {  // (the tile exists: its scale index is below n_mtiles)
          sl2q = sl2 * p.q_descale[(static_cast<int64_t>(w.bi) * p.hq + w.h) * p.n_mtiles + w.m_cta * NQ + t];
          kd = p.k_descale + (static_cast<int64_t>(w.bi) * p.hkv + w.kvh) * p.n_kblocks;
        }
        n_top = w.n_hi_max - 1;
        // (selects, not a runtime index: the arrays stay in registers)
        it0 = w.n_hi_max - (t == 0 ? w.n_hi[0] : w.n_hi[NQ - 1]);
        it_end = w.n_hi_max - (t == 0 ? w.n_lo_t[0] : w.n_lo_t[NQ - 1]);
        // dense: the sizes stay constant-bank operands
        skv = VARLEN ? w.skv : p.skv;
        off = VARLEN ? w.off : p.off;
        left_off = VARLEN ? w.left_off : p.left_off;
      }
      const int row = row0 + r;
      // keys lo_row <= j < lim_row are visible to this row (the causal / window
      // edges folded with the tail)
      const int lim_row = p.causal ? min(skv, max(row + off + 1, 0)) : skv;
      const int lo_row = p.local ? row + left_off : 0;
      float m_run = -INFINITY, l_run = 0.f;
      int k = 0;
      for (int it = it0; it < it_end; ++it, ++gblk, ++k) {
        const int n = n_top - it;
        // score scale of this block (the K scale load overlaps the wait for S)
        float sl2b = sl2q;
        if constexpr (E8) sl2b = sl2q * kd[n];
        if (!warp_wait(&s_full[t], gblk & 1, p.status, kSiteSFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[BN];
        tmem_load_row<BN>(tS, sr);
        if constexpr (C::P_SEP) {  // the scores are in registers: the next S may overwrite them
          tc_fence_before();
          mbar_arrive(&s_free[t]);
        }
        float* s = reinterpret_cast<float*>(sr);
        // (P_SEP) P and O may be written once the previous block's PV has completed
        bool pv_done = !C::P_SEP || gblk == 0;
        if constexpr (SC) {
          // capped scores in log2 units, c log2(e) tanh(s / c), before the mask sets -inf
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = p.sc_b * tanh_from_exp2_arg(s[c] * p.sc_k);
        }
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
        const float bm2 = SC ? bmax : bmax * sl2b;  // (capped scores are already scaled, in log2 units)
        const bool grow = bm2 > m_run + kRescaleLog2;
        const float m_new = grow ? bm2 : m_run;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        float alpha = 1.f;  // (l_run is 0 before the first block: alpha is not needed there)
        if (k > 0 && __any_sync(0xffffffffu, grow)) {
          if (!pv_done) {
            if (!warp_wait(&p_free[t], (gblk - 1) & 1, p.status, kSitePFree)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv_done = true;
          }
          alpha = grow ? ex2_approx(m_run - m_use) : 1.f;
          // O_t holds the previous blocks' product: S_k complete implies PV_{k-1}
          // complete when P overwrites S (one issuing thread, in-order completion),
          // else the wait above.
          // 32 columns at a time: the 128 scores are still live in registers.
          constexpr int CH = 32;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += CH) {
            uint32_t o[CH];
            tmem_load_row<CH>(tO + c0, o);
#pragma unroll
            for (int i = 0; i < CH; i += 2) {
              const float2 r2 = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                           make_float2(alpha, alpha));
              o[i] = __float_as_uint(r2.x);
              o[i + 1] = __float_as_uint(r2.y);
            }
#pragma unroll
            for (int c = 0; c < CH; c += 32) tmem_st32(tO + c0 + c, *reinterpret_cast<const uint32_t(*)[32]>(o + c));
          }
        }
        // P = 2^(s * scale * log2 e - m), written over the first half of the S
        // columns as packed 16-bit pairs; the MMA warp is signalled once per block,
        // or once per half of the block's keys (HALF_P).
        const float2 sl2v = SC ? make_float2(1.f, 1.f) : make_float2(sl2b, sl2b);
        const float2 negm = make_float2(-m_use, -m_use);
        float2 sum2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sum2[i] = make_float2(0.f, 0.f);
        if constexpr (E8) {
          // e4m3 P, four per column (P <= 2^kRescaleLog2 = 256 < 448, the largest e4m3)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[BN / 8];
#pragma unroll
            for (int c = 0; c < BN / 2; c += 4) {
              const int cc = half * (BN / 2) + c;
              const float2 x0 = __ffma2_rn(make_float2(s[cc], s[cc + 1]), sl2v, negm);
              const float2 x1 = __ffma2_rn(make_float2(s[cc + 2], s[cc + 3]), sl2v, negm);
              const float2 e0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
              const float2 e1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
              sum2[(c >> 2) & 3] = __fadd2_rn(sum2[(c >> 2) & 3], __fadd2_rn(e0, e1));
              pk[c >> 2] = pack4_e4m3(e0.x, e0.y, e1.x, e1.y);
            }
            if (!pv_done) {
              if (!warp_wait(&p_free[t], (gblk - 1) & 1, p.status, kSitePFree)) break;
              tc_fence_after();
              pv_done = true;
            }
            tmem_st16(tP + half * (BN / 8), pk);
          }
          if (!pv_done) {
            ok = false;
            break;
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full[t]);
        } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[BN / 4];
#pragma unroll
          for (int c = 0; c < BN / 2; c += 2) {
            const int cc = half * (BN / 2) + c;
            const float2 x = __ffma2_rn(make_float2(s[cc], s[cc + 1]), sl2v, negm);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            pk[c >> 1] = pack2<BF16>(e.x, e.y);
            if constexpr (BF16) {
              sum2[(c >> 1) & 3] = __fadd2_rn(sum2[(c >> 1) & 3], e);
            } else {
              // fp16: l sums P as rounded for the P V product, so that O = o / l
              // weighs every key by exactly the factor its V row was multiplied
              // with (a dominant key's 2^-11 rounding would otherwise reach O in
              // full); LSE keeps that rounding, well inside its bound.  bf16 sums
              // the unrounded P: its 2^-9 rounding would reach LSE.
              add_packed_f16(sum2[(c >> 1) & 3], pk[c >> 1]);
            }
          }
          if (!pv_done) {
            if (!warp_wait(&p_free[t], (gblk - 1) & 1, p.status, kSitePFree)) break;
            tc_fence_after();
            pv_done = true;
          }
#pragma unroll
          for (int c = 0; c < BN / 4; c += 16)
            tmem_st16(tP + half * (BN / 4) + c, *reinterpret_cast<const uint32_t(*)[16]>(pk + c));
          if (HALF_P || half == 1) {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(half == 0 ? &p_half[t] : &p_full[t]);
          }
        }
        if (!pv_done) {
          ok = false;
          break;
        }
        }
        const float2 s01 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
        l_run = alpha * l_run + (s01.x + s01.y);
        m_run = m_new;
      }
      if (!ok) break;

      // ---------------- epilogue (overlaps the next item's first MMAs) ----------------
      const ItemPlan<NQ> w = plan_item<D, VARLEN, CACHE, E8>(p, item);  // recomputed: fewer registers in the loop
      const bool valid = row < w.sq;
      // LSE [b][hq][sq], or [hq][total_q] for packed sequences
      const int64_t lse_idx = VARLEN ? static_cast<int64_t>(w.h) * p.total_q + w.q_base + row
                                     : (static_cast<int64_t>(w.bi) * p.hq + w.h) * w.sq + row;
      const int64_t prow = ((static_cast<int64_t>(w.split) * p.b + w.bi) * p.hq + w.h) * w.sq + row;
      if (k == 0) {
        // This tile sees no key (in this split): O = 0, LSE = -inf.
        if (valid) {
          if (split_mode) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse[prow] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + w.bi * p.o_stride_b +
                                                  static_cast<int64_t>(w.q_base + row) * p.o_stride_row +
                                                  w.h * p.o_stride_h);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[lse_idx] = -INFINITY;
          }
        }
        continue;
      }
      if (!warp_wait(&o_full[t], oitems & 1, p.status, kSiteOFull)) {
        ok = false;
        break;
      }
      ++oitems;
      tc_fence_after();
      // (e4m3: the V scale of the head applies to the whole accumulator)
      const float vscale = E8 ? p.v_descale[static_cast<int64_t>(w.bi) * p.hkv + w.kvh] : 1.f;
      const float inv_l = l_run > 0.f ? vscale / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
      // O leaves TMEM 32 columns at a time (the loads are warp-collective: every
      // lane executes them; only the global stores depend on the row existing)
      // and goes straight to global memory; once the last columns are in
      // registers the accumulator is released to the next item's PV MMAs.
      if (split_mode) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_load_row<32>(tO + c, o);
          if (c + 32 == D) {
            tc_fence_before();
            mbar_arrive(&o_empty[t]);
          }
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              dst[(c + i) / 4] = make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                             __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
          }
        }
        if (valid) p.lse[prow] = lse;
      } else {
        // d <= 128 with a TMA-encodable O: O leaves TMEM 64 columns at a time,
        // normalised and rounded, into the warp's own staging slice (its 32 rows),
        // and one lane has the copy engine store the slice as whole 128-byte row
        // segments while the warp moves on to the next item (measured +2.8% on the
        // causal prefill against the row-by-row stores below, whose 32-row store
        // instructions drain slowly at every item boundary).  The slice is reused
        // once the previous store has read it; that wait overlaps the next
        // columns' TMEM load.  Rows past a dense sequence lie outside the map and
        // are not written; a packed sequence's last rows are followed by the next
        // sequence's, so a warp holding rows past its sequence's end stores row by row.
        if (C::TMA_O && p.o_tma && (!VARLEN || row0 + 32 * wq + 32 <= w.sq)) {
          const uint32_t stg = smem_u32(smem + C::STG_OFF + warp * C::STG_WARP);
#pragma unroll
          for (int cc = 0; cc < D; cc += 64) {
            uint32_t o[64], pk[32];
            tmem_load_row<64>(tO + cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            if (cc + 64 == D) {
              tc_fence_before();
              mbar_arrive(&o_empty[t]);  // the accumulator is free for the next item's PV MMAs
            }
            if (lane == 0) bulk_wait_group_read0();  // the slice's previous store has read it
            __syncwarp();
            // row = lane: its eight 16-byte units, unit i at position i ^ (row & 7)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(stg + lane * 128 + ((i ^ (lane & 7)) << 4), pk[4 * i], pk[4 * i + 1], pk[4 * i + 2],
                           pk[4 * i + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_4d(&p.tm_o, smem + C::STG_OFF + warp * C::STG_WARP, cc, w.h, w.q_base + row0 + 32 * wq, w.tb);
              bulk_commit_group();
            }
          }
          if (valid) p.lse[lse_idx] = lse;
          continue;
        }
        // Otherwise O leaves TMEM, normalised and rounded, HELD columns at a time
        // (all of it for d <= 128, so that the accumulator is released at once;
        // half for d = 256, register budget) and goes straight to global memory,
        // each thread its own row, in 32-byte stores where the layout allows
        // (16-byte ones otherwise).
        constexpr int HELD = D <= 128 ? D : D / 2;
        uint16_t* o_row = static_cast<uint16_t*>(p.o) + w.bi * p.o_stride_b +
                          static_cast<int64_t>(w.q_base + row) * p.o_stride_row + w.h * p.o_stride_h;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += HELD) {
          uint32_t pk[HELD / 2];
#pragma unroll
          for (int c = 0; c < HELD; c += 32) {
            uint32_t o[32];
            tmem_load_row<32>(tO + c0 + c, o);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[c / 2 + i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          }
          if (c0 + HELD == D) {
            tc_fence_before();
            mbar_arrive(&o_empty[t]);  // the accumulator is free for the next item's PV MMAs
          }
          if (valid) {
            if (p.o_vec32) {
#pragma unroll
              for (int i = 0; i < HELD / 16; ++i) st_global_v8(o_row + c0 + 16 * i, pk + 8 * i);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(o_row + c0);
#pragma unroll
              for (int i = 0; i < HELD / 8; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
        if (valid) p.lse[lse_idx] = lse;
      }
    }
  }

  // the O stores have read their staging slices before the CTA leaves
  if (C::TMA_O && warp < 4 * NQ && lane == 0) bulk_wait_group0();
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
  const bool sc = p.sc_b > 0.f;
  auto kern = sc ? fa_prefill_kernel<D, BF16, false, false, true> : fa_prefill_kernel<D, BF16, false>;
  if (p.kv_mode != kKvDense)
    kern = sc ? fa_prefill_kernel<D, BF16, true, false, true, true>
              : fa_prefill_kernel<D, BF16, true, false, false, true>;
  else if (p.cu_q != nullptr)
    kern = sc ? fa_prefill_kernel<D, BF16, true, false, true> : fa_prefill_kernel<D, BF16, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.n_mcta) * p.b * p.hq * p.num_splits;
  if (items <= 0) return cudaSuccess;
  if (items > 0x3fffffffLL) return cudaErrorInvalidConfiguration;
  // persistent: at most one CTA per SM, each walking its share of the items
  const long long grid = items < p.max_ctas ? items : p.max_ctas;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_e4m3_supported(int d) { return d == 64 || d == 128 || d == 256; }

template <int D>
cudaError_t launch_e4m3_t(const PrefillParams& p, cudaStream_t stream) {
  using C = Cfg<D, true>;
  auto kern = fa_prefill_kernel<D, true, false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.n_mcta) * p.b * p.hq;
  if (items <= 0) return cudaSuccess;
  if (items > 0x3fffffffLL) return cudaErrorInvalidConfiguration;
  const long long grid = items < p.max_ctas ? items : p.max_ctas;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_e4m3(const PrefillParams& p, int d, cudaStream_t stream) {
  if (p.cu_q != nullptr || p.num_splits != 1) return cudaErrorInvalidValue;
  switch (d) {
    case 64: return launch_e4m3_t<64>(p, stream);
    case 128: return launch_e4m3_t<128>(p, stream);
    case 256: return launch_e4m3_t<256>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

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
