// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Parameters of the prefill / split kernels (passed by value as a grid constant).
struct PrefillParams {
  CUtensorMap tm_q;  // Q  [b][sq][hq][d],  box {64, 1, 128, 1}
  CUtensorMap tm_k;  // K  [b][skv][hkv][d], box {64, 1, BN, 1}
  CUtensorMap tm_v;  // V  same as K
  // O [b][sq][hq][d] (or [total_q][hq][d] as (d, hq, total_q, 1)), box {64, 1, 32, 1},
  // 128-byte swizzle: each softmax warp stores its 32 rows from shared memory (valid
  // when o_tma != 0)
  CUtensorMap tm_o;
  void* o;           // O base (written row by row by the softmax threads when o_tma == 0)
  float* lse;        // LSE [b][hq][sq] (or LSE partials [ns][b][hq][sq] in split mode)
  float* o_part;     // split mode: normalised partial outputs [ns][b][hq][sq][d]
  int64_t o_stride_b, o_stride_row, o_stride_h;  // elements
  int o_vec32;         // O rows may be written with 32-byte stores (base and strides 32-byte aligned)
  int o_tma;           // tm_o maps O (16-bit outputs whose base and strides TMA accepts)
  int b, sq, skv, hq, hkv, g;
  int causal;          // right edge active: row i sees key j only if j <= i + off
  int off;
  int local;           // left edge active: row i sees key j only if j >= i + left_off
  int left_off;
  float scale_log2;    // scale * log2(e)
  int n_mtiles;        // ceil(sq / 128)
  int n_mcta;          // ceil(n_mtiles / NQ)
  int num_splits;      // 1 = plain forward
  int blocks_per_split;
  int max_ctas;        // grid bound of the persistent kernel (the SM count)
  int* status;
  // Packed variable-length sequences (null for the dense layout): Q/O rows of
  // sequence b are [cu_q[b], cu_q[b + 1]), K/V rows [cu_k[b], cu_k[b + 1]); the
  // tensor maps then cover [total][h][d] with one outer entry, sq is the longest
  // sequence, and off / left_off are relative to each sequence's diagonal.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  // e4m3 inputs (null descales otherwise): S = (Q8 K8^T) * q_descale[tile] *
  // k_descale[block] * scale, O = (P8 V8) * v_descale[head] / l; tm_v then maps
  // V transposed, [b][hkv][d][skv] with the key index innermost.
  const float* q_descale;  // [b][hq][n_mtiles]
  const float* k_descale;  // [b][hkv][n_kblocks]
  const float* v_descale;  // [b][hkv]
  int n_kblocks;
  // Softcap (sc_b > 0): the raw score x = q.k becomes, in log2 units,
  // sc_b * tanh(s / c) with tanh(s / c) = 1 - 2 / (2^(sc_k x) + 1); sc_b = c log2(e).
  float sc_k, sc_b;
  // KV cache (kv_mode = kKvPaged or kKvPacked; the packed-sequence kernels): Q
  // stays dense ([b][sq][hq][d] through tm_q, batch coordinate b); sequence b has
  // seqlens[b] keys in pages of block_table (tm_k / tm_v over [pages][page_size]
  // [hkv][d], boxes of box_rows keys that never straddle a page) or the keys
  // [cu_k[b], cu_k[b + 1]) (tm_k / tm_v over [total_k][hkv][d]); no mask edges,
  // split mode always, each sequence cut into num_splits ranges of its own length.
  int kv_mode;
  const int* block_table;
  int bt_stride, page_size, box_rows;
  const int* seqlens;
};

// Where the decode kernel finds a sequence's keys.
enum : int {
  kKvDense = 0,   // K/V [b][skv][hkv][d]; keys j < kv_limit visible
  kKvPaged = 1,   // K/V cache [num_pages][page_size][hkv][d] addressed through block_table; seqlens[b] keys
  kKvPacked = 2,  // K/V [total_k][hkv][d]; sequence b owns rows [cu_seqlens[b], cu_seqlens[b + 1])
};

// Parameters of the CUDA-core split-KV decode kernel (sq == 1).
struct DecodeParams {
  CUtensorMap tm_k;  // K [b][skv][hkv][d], box {d, 1, BN, 1}, no swizzle
  CUtensorMap tm_v;
  const void* q;     // Q [b][1][hq][d]
  int64_t q_stride_b, q_stride_h;
  float* o_part;     // [ns][b][hq][1][d]
  float* lse_part;   // [ns][b][hq][1]
  int b, skv, hq, hkv, g;
  int nblk;          // ceil(skv / BN)
  int blocks_per_split;
  int num_splits;
  int kv_limit;      // dense: keys j < kv_limit are visible (min(skv, off + 1) when causal)
  int kv_start;      // dense: keys j >= kv_start are visible (the sliding window's left edge)
  int window_left;   // paged / packed: keys j >= len - 1 - window_left are visible; -1 = all
  float scale_log2;
  int* status;
  int kv_mode;                  // kKvDense, kKvPaged or kKvPacked
  const int* block_table;       // paged: [b][bt_stride] page indices
  int64_t bt_stride;
  int page_size;                // paged: keys per page, a multiple of 64
  int box_rows;                 // rows per TMA box: the key block, or 64 when pages are smaller than it
  const int* seqlens;           // paged: [b] keys per sequence
  const int* cu_seqlens;        // packed: [b + 1] prefix sums of keys per sequence
  int total_k;                  // packed: rows of the packed K / V
  // Fused merge: the last split of a (batch, query-head group) to finish merges
  // all splits' partials into o / lse.  counters: one int per (batch, group),
  // zero at launch; the merging CTA puts its counter back to zero.
  int* counters;                // [b][hkv * g / heads_per_cta]
  void* o;                      // [b][1][hq][d] of the input type
  int64_t o_stride_b, o_stride_h;
  float* lse;                   // [b][hq], or null
  // Softcap (sc_b > 0): the score x (q.k * scale * log2 e) becomes sc_b * tanh(x / sc_b),
  // tanh through 2^(sc_k x) with sc_k = 2 / c; sc_b = c log2(e).
  float sc_k, sc_b;
  // e4m3 K / V: per-128-key-block K scales [b][hkv][n_kblocks], per-head V scales [b][hkv]
  const float* k_descale;
  const float* v_descale;
  int n_kblocks;
};

// Parameters of the backward kernels (recompute form: D and log2-scaled LSE per
// row are prepared once, then dQ and dK / dV are computed by two kernels).
struct BwdParams {
  CUtensorMap tm_q;   // Q  [b][sq][hq][d],   box {64, 1, 128, 1}, 128-byte swizzle
  CUtensorMap tm_do;  // dO like Q
  CUtensorMap tm_k;   // K  [b][skv][hkv][d], box {64, 1, 128, 1}
  CUtensorMap tm_v;   // V  like K
  const void* o;      // O (forward output), strides o_st (b, row, head) in elements
  const void* dout;   // dO, strides do_st
  const float* lse;   // [b][hq][sq]
  int64_t o_st[3], do_st[3];
  void* dq;           // outputs, strides (b, row, head) in elements
  void* dk;
  void* dv;
  int64_t dq_st[3], dk_st[3], dv_st[3];
  float* dpre;        // D  = rowsum(dO * O), [b][hq][sq_pad]; 0 on padding rows
  float* l2pre;       // LSE * log2(e), [b][hq][sq_pad]; +inf on padding rows and rows that see no key
  int b, sq, skv, hq, hkv, g, sq_pad;
  int causal, off;    // row i sees key j only if j <= i + off (when causal)
  int local, left_off;  // ... and only if j >= i + left_off (when local)
  float scale, scale_log2;
  int n_mtiles, n_ntiles;  // 128-row query tiles, 128-key blocks
  int* status;
  float sc_k, sc_b;     // softcap as in PrefillParams (sc_b = 0: off)
  int head_group;       // dQ grid: (batch, query head) pairs whose row tiles are interleaved, longest first
};

// e4m3 quantisation of one [b][s][h][d] tensor.
struct QuantParams {
  const void* x;      // bf16 / fp16, strides x_st (b, row, head) in elements
  int64_t x_st[3];
  void* out;          // e4m3; row-major: out_st = (b, row, head) bytes; transposed: (b, head, d-row) bytes
  int64_t out_st[3];
  float* descale;     // [b][h][nblk] (per 128-row block) or [b][h] (per head)
  int b, s, h, d, nblk;
  int transpose, per_head;
};

struct CombineParams {
  const float* o_part;   // [ns][b][hq][sq][d]
  const float* lse_part; // [ns][b][hq][sq]
  void* o;
  int64_t o_stride_b, o_stride_row, o_stride_h;
  float* lse;            // [b][hq][sq] (may be null)
  int num_splits, b, hq, sq, d;
};

// Launchers: return cudaSuccess or the launch error.  `dtype` 0 = bf16, 1 = fp16.
cudaError_t launch_prefill(const PrefillParams& p, int d, int dtype, cudaStream_t stream);
cudaError_t launch_prefill_e4m3(const PrefillParams& p, int d, cudaStream_t stream);  // bf16 output
bool prefill_e4m3_supported(int d);
cudaError_t launch_quant_e4m3(const QuantParams& p, int dtype, cudaStream_t stream);
int prefill_block_n(int d);   // keys per KV block of the prefill kernel
int prefill_q_tiles(int d);   // 128-row Q tiles per CTA

cudaError_t launch_decode(const DecodeParams& p, int d, int dtype, cudaStream_t stream);
cudaError_t launch_decode_e4m3(const DecodeParams& p, int d, int dtype, cudaStream_t stream);  // d in {64, 128}
int decode_e4m3_block_n();  // keys per block of the e4m3 decode (one K scale per block)
int decode_block_n(int d);
int decode_ctas_per_sm(int d, int dtype);
int decode_heads_per_cta(int g);  // query heads of one KV group handled by one CTA
bool decode_supported(int d, int g);

cudaError_t launch_combine(const CombineParams& p, int dtype, cudaStream_t stream);

cudaError_t launch_wait_selftest(int* status, cudaStream_t stream);

// Backward: preprocess, dQ and dK / dV kernels in sequence on `stream`.
cudaError_t launch_bwd(const BwdParams& p, int d, int dtype, cudaStream_t stream);
bool bwd_supported(int d);

}  // namespace fa
