/*
 * fa.h -- C ABI of the GB300 (sm_103a) tiled exact attention library (libfa.so).
 *
 * What is computed (the plain definition, "hs-black: FlashAttention 1/2/3",
 * section "Shapes"; LSE from "One row of runnable logic"):
 *
 *   for every batch b, query head h, query row i:
 *     kv_head  = h / (hq / hkv)                      (GQA mapping, "flash attention V2
 *                                                     code walkthrough", block_table / h_h_k_ratio)
 *     visible  = { j < skv : (!causal || j <= i + q_pos_offset)
 *                  && (!local || window_left < 0  || j >= i + q_pos_offset - window_left)
 *                  && (!local || window_right < 0 || j <= i + q_pos_offset + window_right) }
 *     s_j      = scale * <Q[b,i,h,:], K[b,j,kv_head,:]>
 *     O[b,i,h] = sum_j softmax(s)_j V[b,j,kv_head,:]   over visible j
 *     LSE[b,h,i] = log sum_j exp(s_j)                  over visible j
 *   A row with no visible key gets O = 0 and LSE = -inf.
 *
 * The causal rule is bottom-right aligned by default (q_pos_offset = skv - sq,
 * the mask pictures of "flash attention V2 code walkthrough", Is_causal); any
 * other offset gives the absolute query position used by a KV-cache decode
 * ("hs-black", section "Implementation: causal and tail blocks").  The sliding
 * window ("flash attention V2 code walkthrough", Is_local: query i attends to
 * keys [i + skv - sq - window_left, i + skv - sq + window_right], -1 leaving a
 * side open) is aligned on the same diagonal; causal is the window (-1, 0), and
 * causal together with a window keeps the keys both allow.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  Split-KV needs a caller-owned
 *     device workspace (see fa_splitkv_workspace_size).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on that stream; results are ready
 *     when the stream is synchronised.
 *   - Validation happens on the host before any launch; an invalid argument
 *     returns an error code and launches nothing.  No exception crosses the ABI.
 *   - Device-side waits are bounded (about two seconds each); a wait that runs
 *     out is recorded in a per-device status word that fa_sync_status reports.
 *   - Layouts: Q, O are [b, sq, hq, d] and K, V are [b, skv, hkv, d] with the
 *     head dimension contiguous and the other three strides given in elements
 *     (order: batch, row, head).  LSE is fp32 [b, hq, sq], contiguous.
 *   - Supported: d in {64, 128, 256}; bf16 or fp16 storage; fp32 accumulation.
 *     Base pointers 16-byte aligned; strides multiples of 8 elements.
 */
#ifndef TILED_EXACT_ATTENTION_FA_H
#define TILED_EXACT_ATTENTION_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, stride or alignment */
  FA_ERR_UNSUPPORTED = 2, /* a head dimension or shape outside the compiled set */
  FA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
  FA_ERR_TIMEOUT = 4,     /* a device-side wait gave up (reported by fa_sync_status) */
  FA_ERR_SCRATCH_LIMIT = 5, /* fa_fwd_splitkv_noalloc: the problem does not fit the built-in scratch */
  FA_ERR_DEVICE_ARG = 6     /* an argument read on the device (sequence offsets) failed its check
                               (reported by fa_sync_status) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/* q_pos_offset value meaning "bottom-right aligned": skv - sq. */
#define FA_OFFSET_BOTTOM_RIGHT INT64_MIN

typedef struct {
  fa_dtype dtype;     /* storage type of Q, K, V and O */
  int32_t b;          /* batch */
  int32_t sq;         /* query rows per sequence (>= 0) */
  int32_t skv;        /* key rows per sequence (>= 0) */
  int32_t hq;         /* query heads (>= 1) */
  int32_t hkv;        /* key/value heads, hq % hkv == 0 */
  int32_t d;          /* head dimension: 64, 128 or 256 */
  const void* q;      /* device, [b, sq, hq, d] */
  const void* k;      /* device, [b, skv, hkv, d] */
  const void* v;      /* device, [b, skv, hkv, d] */
  void* o;            /* device, [b, sq, hq, d], written */
  float* lse;         /* device, fp32 [b, hq, sq], written */
  int64_t q_strides[3]; /* (batch, row, head) strides of q, in elements */
  int64_t k_strides[3];
  int64_t v_strides[3];
  int64_t o_strides[3];
  int32_t causal;       /* 0 or 1 */
  int64_t q_pos_offset; /* causal: row i sees key j iff j <= i + q_pos_offset;
                           FA_OFFSET_BOTTOM_RIGHT = skv - sq.  Ignored when causal == 0 and local == 0. */
  float scale;          /* multiplies q.k before the mask and the max; finite, > 0 (e.g. 1/sqrt(d)) */
  int32_t local;        /* 0 or 1: apply the sliding window below (ABI version >= 2) */
  int64_t window_left;  /* local: row i sees keys j >= i + q_pos_offset - window_left; -1 = no left edge */
  int64_t window_right; /* local: row i sees keys j <= i + q_pos_offset + window_right; -1 = no right edge */
  float softcap;        /* 0 = off; c > 0: every scaled score s becomes c * tanh(s / c) before the mask and the
                           softmax (Is_softcap of "flash attention V2 code walkthrough"; ABI version >= 3) */
} fa_fwd_args;

/*
 * Prefill / general forward pass: O and LSE for every row.
 * Tiled exactly as "ai-reference-codex: forward CUDA kernel", sections 2-6: a
 * CTA owns Q row blocks, K/V blocks stream past, blocks beyond the causal
 * diagonal (or outside the sliding window: n_block_min / n_block_max of "flash
 * attention V2 code walkthrough", section 2) are skipped, the elementwise mask
 * runs only on the blocks an edge cuts, and the epilogue divides by l and
 * writes LSE = m + log l.
 * Returns FA_OK once the work is enqueued on `stream`.
 */
fa_status fa_fwd(const fa_fwd_args* args, void* stream);

/*
 * Split count for split-KV ("ai-reference-codex: forward CUDA kernel", 7.2):
 * with w(s) = units * s / slots and efficiency(s) = w / ceil(w), return the
 * smallest s in [1, min(max_splits, num_kv_blocks)] whose efficiency is at least
 * 85% of the best one.  units = independent CTAs before splitting, slots =
 * concurrently resident CTAs (SMs x CTAs per SM).  Pure host function.
 * Returns 1 for non-positive units or slots.
 */
int32_t fa_num_splits_heuristic(int64_t units, int64_t slots, int64_t num_kv_blocks, int32_t max_splits);

/*
 * The split count fa_fwd_splitkv would use for `args` with num_splits == 0 on
 * the current device (the heuristic above applied to this launch).  Returns
 * 0 and writes nothing if the arguments are invalid.
 */
int32_t fa_splitkv_default_splits(const fa_fwd_args* args);

/*
 * Workspace bytes fa_fwd_splitkv needs for `num_splits` splits (0 = the
 * default count): fp32 partial outputs [num_splits, b, hq, sq, d] followed
 * (256-byte aligned) by fp32 partial LSEs [num_splits, b, hq, sq] and
 * (256-byte aligned) b * hq int32 merge counters, which the call zeroes itself
 * on the stream before it uses them.  Returns 0 for invalid arguments.
 */
size_t fa_splitkv_workspace_size(const fa_fwd_args* args, int32_t num_splits);

/*
 * Split-KV forward ("ai-reference-codex: forward CUDA kernel", section 7; the
 * early-exit rule of "flash attention V2 code walkthrough",
 * compute_attn_1rowblock_splitkv): the key blocks are cut into num_splits
 * contiguous ranges of ceil(nblk / num_splits) blocks; split s writes its
 * normalised partial O_s and LSE_s into the workspace (0 and -inf for a split
 * with no visible key), then they are merged into args->o and args->lse as
 * fa_splitkv_combine does.  With one split the kernel writes O and LSE itself.
 * For sq == 1 the g = hq / hkv query heads sharing a KV head are folded
 * together (section 7.4): for g >= 8 without a sliding window they become the
 * rows of one tensor-core query tile (Q viewed as [b][g][hkv][d]; merged by
 * the combine kernel); otherwise up to four of them share a CUDA-core CTA and
 * the last split of each head group to finish merges the partials inside the
 * split kernel (one launch plus a small memset of the counters).
 * num_splits == 0 picks the count with the heuristic;
 * the count used is written to *splits_used (may be NULL).  The workspace is a
 * caller-owned device buffer of at least fa_splitkv_workspace_size bytes,
 * 256-byte aligned, needing no initialisation; two calls whose work overlaps on
 * the GPU (different streams) need different workspaces.  Same result as fa_fwd
 * up to rounding.
 */
fa_status fa_fwd_splitkv(const fa_fwd_args* args, int32_t num_splits, void* workspace, size_t workspace_bytes,
                         int32_t* splits_used, void* stream);

/*
 * LSE-weighted merge of split partials ("ai-reference-codex: forward CUDA
 * kernel", 7.3): per row, LSE = logsumexp_s LSE_s and O = sum_s
 * e^(LSE_s - LSE) O_s; if every LSE_s is -inf the row gets O = 0, LSE = -inf.
 *   o_part:   device fp32 [num_splits, b, hq, sq, d] (normalised partials)
 *   lse_part: device fp32 [num_splits, b, hq, sq]
 *   o:        device [b, sq, hq, d] of `dtype`, strides (batch, row, head) in elements
 *   lse:      device fp32 [b, hq, sq], or NULL to skip it
 * 1 <= num_splits; d in {64, 128, 256}.
 */
fa_status fa_splitkv_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t b,
                             int32_t hq, int32_t sq, int32_t d, fa_dtype dtype, void* o,
                             const int64_t o_strides[3], float* lse, void* stream);

/*
 * Decode against a KV cache: one new query row per sequence attending to all
 * keys of its own sequence, whose lengths differ.  The pages' KV-cache path
 * ("ai-reference-codex: forward CUDA kernel", section 8: flash_attn_with_kvcache
 * forces split-KV and supports a paged block table; "flash attention V2 code
 * walkthrough", Flash_fwd_params (cu_seqlens as prefix sums, block_table) and
 * "moving the kv cache": a cache of [num_blocks, block_size, heads, head_dim]
 * whose row for (sequence, position) is block_table[position / block_size] *
 * page_stride + (position % block_size) * row_stride + kv_head * head_stride).
 *
 * Two layouts of the keys/values:
 *   paged   (page_size > 0): k, v are [num_pages, page_size, hkv, d]; sequence
 *           b's position t lives in page block_table[b * block_table_stride +
 *           t / page_size] at row t % page_size; seqlens_k[b] keys per sequence.
 *           page_size must be a multiple of 64.
 *   packed  (page_size == 0): k, v are [total_k, hkv, d] with sequence b at rows
 *           [cu_seqlens_k[b], cu_seqlens_k[b + 1]); num_pages holds total_k.
 * The query of sequence b sees every one of its keys (it stands at position
 * len_b - 1), or with local = 1 only the last window_left + 1 of them (the
 * sliding window of fa_fwd_args, right edge at the query itself); a sequence
 * with no key gets O = 0, LSE = -inf.  Rows of the cache beyond a sequence's
 * length, or before its window, are never used, whatever they hold.
 */
typedef struct {
  fa_dtype dtype;
  int32_t b, hq, hkv, d;          /* hq % hkv == 0; d in {64, 128, 256} */
  const void* q;                  /* device, [b, hq, d] */
  int64_t q_strides[2];           /* (batch, head), in elements */
  const void* k;                  /* device, see above */
  const void* v;
  int64_t k_strides[3];           /* (page, row, head) in elements; packed: (unused, row, head) */
  int64_t v_strides[3];
  int32_t num_pages;              /* paged: pages in k / v; packed: total_k */
  int32_t page_size;              /* keys per page (multiple of 64), or 0 for the packed layout */
  const int32_t* block_table;     /* device, paged: [b, block_table_stride] page indices */
  int32_t block_table_stride;
  const int32_t* seqlens_k;       /* device, paged: [b] keys per sequence */
  const int32_t* cu_seqlens_k;    /* device, packed: [b + 1] prefix sums */
  int32_t max_seqlen_k;           /* host-side bound of the keys per sequence (used by the split heuristic only) */
  void* o;                        /* device, [b, hq, d] of dtype */
  int64_t o_strides[2];           /* (batch, head), in elements */
  float* lse;                     /* device, fp32 [b, hq] */
  float scale;
  int32_t local;                  /* 0 or 1 (ABI version >= 2) */
  int32_t window_left;            /* local: keys at positions >= len_b - 1 - window_left; -1 = all */
  float softcap;                  /* as in fa_fwd_args (ABI version >= 3) */
} fa_kvcache_args;

/* Workspace bytes fa_fwd_kvcache needs for num_splits splits (0 = its default); 0 if invalid. */
size_t fa_kvcache_workspace_size(const fa_kvcache_args* args, int32_t num_splits);

/*
 * Split-KV decode over a paged or packed KV cache (see fa_kvcache_args): the
 * same split kernel and LSE-weighted combine as fa_fwd_splitkv, with the key
 * blocks of each sequence addressed through its block table or its prefix sum
 * and cut into num_splits ranges of that sequence's own length (0 = the
 * split-count heuristic, applied with max_seqlen_k) and merged as for
 * fa_fwd_splitkv with sq == 1: with g = hq / hkv >= 8 query heads per KV head
 * and no window, the g heads are the rows of one tensor-core tile whose K/V
 * blocks are loaded page by page (the V rows of a sequence's last block that
 * lie past its end are zeroed in shared memory before they are multiplied, so
 * whatever the cache holds there never reaches O); otherwise the CUDA-core
 * kernel merges the splits itself.  The workspace is caller-owned device memory
 * of at least fa_kvcache_workspace_size bytes, 256-byte aligned, under the same
 * rules as fa_fwd_splitkv's.  The lengths live on the device, so the kernels
 * check them before reading anything they address: a paged sequence longer
 * than block_table_stride * page_size keys, or a packed sequence whose
 * [cu_seqlens_k[b], cu_seqlens_k[b + 1]) is not inside [0, num_pages), is not
 * read at all; FA_ERR_DEVICE_ARG is recorded for the next fa_sync_status and
 * that sequence's O and LSE are undefined (the other sequences are computed).
 */
fa_status fa_fwd_kvcache(const fa_kvcache_args* args, int32_t num_splits, void* workspace, size_t workspace_bytes,
                         int32_t* splits_used, void* stream);

/*
 * Forward pass over packed variable-length sequences ("flash attention V2 code
 * walkthrough", Flash_fwd_params: cu_seqlens_q / cu_seqlens_k are prefix sums of
 * the sequence lengths, e.g. [0, 248, 249, 250], and BlockInfo offsets each
 * sequence's rows by them).  Sequence s owns query rows [cu_seqlens_q[s],
 * cu_seqlens_q[s + 1]) of q / o and key rows [cu_seqlens_k[s], cu_seqlens_k[s + 1])
 * of k / v; each sequence is an independent attention problem with the
 * definition at the top of this file, its causal and window edges on its own
 * bottom-right diagonal (q_pos_offset = its skv - its sq).  Same kernel as fa_fwd.
 */
typedef struct {
  fa_dtype dtype;
  int32_t b;                      /* sequences (>= 1) */
  int32_t hq, hkv, d;             /* hq % hkv == 0; d in {64, 128, 256} */
  int32_t total_q, total_k;       /* rows of the packed tensors (>= 0) */
  int32_t max_seqlen_q;           /* host-side bound on every sequence's query rows (sizes the grid) */
  const void* q;                  /* device, [total_q, hq, d] */
  const void* k;                  /* device, [total_k, hkv, d] */
  const void* v;                  /* device, [total_k, hkv, d] */
  void* o;                        /* device, [total_q, hq, d], written */
  float* lse;                     /* device, fp32 [hq, total_q], written */
  int64_t q_strides[2];           /* (row, head) strides in elements, multiples of 8 */
  int64_t k_strides[2];
  int64_t v_strides[2];
  int64_t o_strides[2];
  const int32_t* cu_seqlens_q;    /* device, [b + 1], non-decreasing, cu[0] >= 0, cu[b] <= total_q */
  const int32_t* cu_seqlens_k;    /* device, [b + 1], likewise with total_k */
  int32_t causal;                 /* 0 or 1 */
  int32_t local;                  /* 0 or 1: sliding window (widths as in fa_fwd_args, -1 = open side) */
  int64_t window_left;
  int64_t window_right;
  float scale;                    /* finite, > 0 */
  float softcap;                  /* as in fa_fwd_args (ABI version >= 3) */
} fa_varlen_args;

/*
 * Enqueue the packed variable-length forward pass.  The host checks what it can
 * see; the prefix sums live on the device, so each CTA checks its sequence's
 * offsets against total_q / total_k and max_seqlen_q before touching memory, skips
 * the work if they are out of range and records FA_ERR_DEVICE_ARG for the next
 * fa_sync_status (outputs of the rejected sequences are then left unwritten).
 */
fa_status fa_fwd_varlen(const fa_varlen_args* args, void* stream);

/*
 * Backward pass ("hs-black: FlashAttention 1/2/3", sections "Backward: from the
 * softmax derivative", "Training: recompute in backward", "Backward: back to Q,
 * K, V"): given the forward inputs, its output O and per-row LSE, and the
 * upstream gradient dO, computes
 *   D = rowsum(dO * O),  P = exp(S - LSE) recomputed tile by tile,
 *   dV = P^T dO,  dS = P (dP - D) with dP = dO V^T,
 *   dQ = dS K * scale,  dK = dS^T Q * scale,
 * with the forward pass's mask (causal, window, tail); the query heads sharing
 * a key/value head add their contributions to its dK and dV.  Deterministic (no
 * atomics).  Supported: d in {64, 128}; bf16 or fp16; same layouts and stride
 * rules as fa_fwd_args.  A caller-owned device workspace of
 * fa_bwd_workspace_size bytes (256-byte aligned) holds D and LSE * log2(e) per
 * row, padded to 128 rows.
 */
typedef struct {
  fa_dtype dtype;
  int32_t b, sq, skv, hq, hkv, d;
  const void* q;        /* device, [b, sq, hq, d] */
  const void* k;        /* device, [b, skv, hkv, d] */
  const void* v;        /* device, [b, skv, hkv, d] */
  const void* o;        /* device, [b, sq, hq, d]: the forward output */
  const void* dout;     /* device, [b, sq, hq, d]: gradient of the loss with respect to O */
  const float* lse;     /* device, fp32 [b, hq, sq]: the forward LSE */
  void* dq;             /* device, [b, sq, hq, d], written */
  void* dk;             /* device, [b, skv, hkv, d], written */
  void* dv;             /* device, [b, skv, hkv, d], written */
  int64_t q_strides[3], k_strides[3], v_strides[3], o_strides[3], do_strides[3];  /* (batch, row, head) */
  int64_t dq_strides[3], dk_strides[3], dv_strides[3];
  int32_t causal;       /* as fa_fwd_args */
  int64_t q_pos_offset;
  float scale;
  int32_t local;
  int64_t window_left, window_right;
  float softcap;        /* as in fa_fwd_args; dS gains the cap's derivative 1 - tanh^2(s / c) (ABI version >= 3) */
} fa_bwd_args;

/* Workspace bytes fa_bwd needs (0 for invalid arguments). */
size_t fa_bwd_workspace_size(const fa_bwd_args* args);

/* Enqueue the backward pass on `stream`; FA_ERR_UNSUPPORTED for d = 256. */
fa_status fa_bwd(const fa_bwd_args* args, void* workspace, size_t workspace_bytes, void* stream);

/*
 * 8-bit forward path ("hs-black: FlashAttention 1/2/3", section "FlashAttention-3:
 * precision and hardware": FP8 as an extra speed path, a scale factor per block,
 * the scales carried into the computation, softmax statistics kept in fp32).
 *
 * fa_quantize_e4m3 turns one bf16 / fp16 tensor [b, s, h, d] (d in {64, 128, 256})
 * into e4m3 codes: descale = amax / 448 over each 128-row block of one (batch,
 * head) (per_head = 0; descale [b, h, ceil(s / 128)]) or over the whole (batch,
 * head) (per_head = 1; descale [b, h]); code = round-to-nearest-even e4m3 of
 * x * (1 / descale), saturating at +-448 (fp32 IEEE products, so the codes are
 * reproducible bit for bit).  An all-zero block gets descale 1.  Output
 * row-major [b, s, h, d] with out_strides (batch, row, head) in bytes, or
 * (transpose = 1) [b, h, d, s] with out_strides (batch, head, d-row) in bytes,
 * the row index contiguous; strides multiples of 16 bytes, base 16-byte aligned.
 */
typedef struct {
  fa_dtype dtype;              /* input storage type */
  int32_t b, s, h, d;
  const void* x;               /* device, [b, s, h, d] */
  int64_t x_strides[3];        /* (batch, row, head) in elements, multiples of 8 */
  void* out;                   /* device, e4m3 codes */
  int64_t out_strides[3];
  int32_t transpose;           /* 0 or 1 */
  int32_t per_head;            /* 0 or 1 */
  float* descale;              /* device, written */
} fa_quant_args;

fa_status fa_quantize_e4m3(const fa_quant_args* args, void* stream);

/*
 * Forward pass with e4m3 Q, K, V (d in {64, 128, 256}; FA_ERR_UNSUPPORTED otherwise): S = (Q8 K8^T) * q_descale[tile of
 * 128 rows] * k_descale[block of 128 keys] * scale, P = exp(S - m) rounded to e4m3
 * for the P V product (P <= 2^8 by the lazy-rescale rule, within e4m3's range),
 * row max and sum in fp32, O = (P8 V8) * v_descale[head] / l written as bf16,
 * LSE fp32.  Q, K as produced by fa_quantize_e4m3 with per-block scales; V
 * transposed ([b, hkv, d, skv]) with one scale per (batch, head), applied to the
 * whole accumulator since a per-block V scale folded into P could push P past 448.
 * Same mask, GQA and offset rules as fa_fwd; no split-KV or packed sequences.
 */
typedef struct {
  int32_t b, sq, skv, hq, hkv, d;
  const void* q;               /* device, e4m3 [b, sq, hq, d] */
  const void* k;               /* device, e4m3 [b, skv, hkv, d] */
  const void* vt;              /* device, e4m3 [b, hkv, d, skv] */
  const float* q_descale;      /* device, [b, hq, ceil(sq / 128)] */
  const float* k_descale;      /* device, [b, hkv, ceil(skv / 128)] */
  const float* v_descale;      /* device, [b, hkv] */
  void* o;                     /* device, bf16 [b, sq, hq, d], written */
  float* lse;                  /* device, fp32 [b, hq, sq], written */
  int64_t q_strides[3];        /* (batch, row, head) in bytes */
  int64_t k_strides[3];
  int64_t vt_strides[3];       /* (batch, head, d-row) in bytes */
  int64_t o_strides[3];        /* (batch, row, head) in elements */
  int32_t causal;
  int64_t q_pos_offset;
  float scale;
  int32_t local;
  int64_t window_left, window_right;
} fa_fwd_e4m3_args;

fa_status fa_fwd_e4m3(const fa_fwd_e4m3_args* args, void* stream);

/*
 * Split-KV decode over e4m3 keys and values ("hs-black: FlashAttention 1/2/3",
 * section "FlashAttention-3: precision and hardware": a scale per block, carried
 * into the computation; the split and its LSE-weighted merge of "ai-reference-codex:
 * forward CUDA kernel", section 7).  One query row per (batch, query head), in
 * bf16 / fp16, sees every one of the skv keys of its KV head (decode: the query
 * stands at position skv - 1).  K as produced by fa_quantize_e4m3 (one scale per
 * 128-key block), V by fa_quantize_e4m3 with per_head = 1 (not transposed):
 *   s_j = (q . K8_j) * k_descale[block of j] * scale,  p_j = exp(s_j - m),
 *   O = (sum_j p_j V8_j) * v_descale / sum_j p_j,  LSE = m + log sum_j p_j,
 * with the scores, the probabilities and every sum in fp32 (K and V are widened
 * exactly from e4m3; nothing is rounded to 8 bits on the way).  The key blocks
 * are cut into num_splits ranges (0 = the split-count heuristic); the last CTA of
 * each (batch, head group) merges the splits.  The workspace rules are those of
 * fa_fwd_splitkv.  d in {64, 128}.
 */
typedef struct {
  fa_dtype dtype;                 /* of q and o */
  int32_t b, skv, hq, hkv, d;     /* hq % hkv == 0; skv >= 0 */
  const void* q;                  /* device, [b, hq, d] of dtype */
  int64_t q_strides[2];           /* (batch, head), in elements, multiples of 8 */
  const void* k;                  /* device, e4m3 [b, skv, hkv, d] */
  const void* v;                  /* device, e4m3 [b, skv, hkv, d] */
  int64_t k_strides[3];           /* (batch, row, head), in bytes, multiples of 16 */
  int64_t v_strides[3];
  const float* k_descale;         /* device, [b, hkv, ceil(skv / 128)] */
  const float* v_descale;         /* device, [b, hkv] */
  void* o;                        /* device, [b, hq, d] of dtype, written */
  int64_t o_strides[2];           /* (batch, head), in elements */
  float* lse;                     /* device, fp32 [b, hq], written */
  float scale;                    /* finite, > 0 */
} fa_splitkv_e4m3_args;

/* Workspace bytes fa_fwd_splitkv_e4m3 needs for num_splits splits (0 = its default); 0 if invalid. */
size_t fa_splitkv_e4m3_workspace_size(const fa_splitkv_e4m3_args* args, int32_t num_splits);

fa_status fa_fwd_splitkv_e4m3(const fa_splitkv_e4m3_args* args, int32_t num_splits, void* workspace,
                              size_t workspace_bytes, int32_t* splits_used, void* stream);

/* Size of the built-in split-KV scratch used by fa_fwd_splitkv_noalloc (per device). */
#define FA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * fa_fwd_splitkv without a caller-supplied workspace (no counterpart in the
 * reference pages; an addition of this library).
 *
 * Some callers cannot allocate device memory for a workspace: a framework
 * whose memory manager owns the whole device and hands an operator only its
 * input and output buffers, a plugin interface that passes tensors but no
 * allocator, or a latency-critical path where cudaMalloc (and the device
 * synchronisation it may imply) is not acceptable.  This entry point runs
 * the same split-KV kernels and combine as fa_fwd_splitkv, with the split
 * partials kept in a fixed buffer compiled into the library: a file-scope
 * device array of FA_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU which loads
 * the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *   args, num_splits, splits_used, stream: as for fa_fwd_splitkv.
 *   Returns FA_ERR_SCRATCH_LIMIT, launching nothing, when the workspace the
 *   problem needs (fa_splitkv_workspace_size(args, num_splits)) exceeds
 *   FA_NOALLOC_SCRATCH_BYTES; use fa_fwd_splitkv with your own workspace then.
 *
 * The first call on a device looks up the buffer's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  All calls on a device share the one buffer: every call overwrites
 * the parts it uses before reading them, so nothing carries over between
 * calls, but calls whose work overlaps on the GPU (different streams, or
 * different host threads) race on the buffer and must be serialised by the
 * caller.
 */
fa_status fa_fwd_splitkv_noalloc(const fa_fwd_args* args, int32_t num_splits, int32_t* splits_used, void* stream);

/*
 * Synchronise `stream` and report device-side failures on the current device:
 * FA_ERR_TIMEOUT if any kernel of this library recorded a wait that ran out
 * since the last call, FA_ERR_DEVICE_ARG if a kernel rejected an argument it
 * read on the device (the first record wins; it is then cleared), FA_ERR_CUDA if
 * the synchronisation itself failed, FA_OK otherwise.
 */
fa_status fa_sync_status(void* stream);

/*
 * Self-test of the bounded-wait path: launches one tiny kernel that waits on
 * a barrier nothing completes.  The wait gives up after its limit (about two
 * seconds), records a timeout and returns, so that a following
 * fa_sync_status returns FA_ERR_TIMEOUT while the context stays usable.
 */
fa_status fa_selftest_wait_timeout(void* stream);

/* Static description of a status code. */
const char* fa_status_string(fa_status status);

/* ABI version of this header (incremented on incompatible changes). */
int32_t fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TILED_EXACT_ATTENTION_FA_H */
