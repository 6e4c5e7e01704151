// Helpers shared by the tensor-core kernels (forward and backward): warp-uniform
// bounded waits, TMEM row loads, 16-bit packing and the two tcgen05 MMA shapes
// the kernels issue.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace fa {

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// A bounded wait whose outcome is the same on every lane of the warp, so that the
// warp stays converged for the warp-collective TMEM instructions that follow.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status, int site,
                                          uint32_t sleep_ns = 0) {
  const bool ok = mbar_wait(bar, parity, status, site, false, sleep_ns);
  return __all_sync(0xffffffffu, ok);
}

// A value the optimiser may not hoist: expressions of it are formed where they
// are used instead of being held in registers across a loop.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t x) {
  asm volatile("" : "+r"(x));
  return x;
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

// Issue one 32-column TMEM load of this thread's lane without waiting for it
// (several loads can then share one tmem_ld_wait).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t* x) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
        "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]),
        "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
        "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

// a.x += lo, a.y += hi for a packed pair of fp16 values, each widened exactly to
// fp32 (mixed-precision add).
__device__ __forceinline__ void add_packed_f16(float2& a, uint32_t u) {
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(a.x), "+f"(a.y)
      : "r"(u));
}

// S_t = Q_t K^T over the head dimension: D / 16 MMAs of K = 16, both operands
// K-major with 128-byte swizzle (64-column chunks of 128-byte rows).
template <int D, int BN, int BM, int Q_BYTES, int KV_BYTES, uint32_t ID, bool W = false>
__device__ __forceinline__ void issue_s_tile(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc, int t, int slot) {
  uint64_t qd = q_desc + static_cast<uint32_t>((t * Q_BYTES) >> 4);
  uint64_t kd = k_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
  // opaque to the optimiser: the per-step descriptors are formed at issue time
  // instead of being hoisted (and held in registers) across the item loop
  asm volatile("" : "+l"(qd), "+l"(kd));
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t offa = static_cast<uint32_t>(((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4);
    const uint32_t offb = static_cast<uint32_t>(((k >> 2) * (BN * 128) + (k & 3) * 32) >> 4);
    umma_ss<W>(d_tmem, qd + offa, kd + offb, ID, k > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t[:, 16 k0 : 16 k1] V[16 k0 : 16 k1, :]: P from TMEM (two 16-bit
// values per column), V MN-major with 128-byte swizzle (64-column atoms BN * 128
// bytes apart, 8-row groups 1024 bytes apart).
template <int D, int BN, int KV_BYTES, uint32_t ID, int K0, int K1, bool W = false>
__device__ __forceinline__ void issue_pv_tile(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, int slot, bool acc) {
  uint64_t vd = v_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
  asm volatile("" : "+l"(vd));
#pragma unroll
  for (int k = K0; k < K1; ++k) {
    umma_ts<W>(o_tmem, p_tmem + k * 8, vd + static_cast<uint32_t>((k * 2048) >> 4), ID, (acc || k > 0) ? 1u : 0u);
  }
}


// 8-bit forms: S = Q K^T with e4m3 operands (D / 32 MMAs of K = 32, K-major rows
// staged in swizzle chunks of CB bytes: 128-byte chunks with the 128-byte swizzle,
// or for d = 64 one 64-byte chunk with the 64-byte swizzle; a K step of 32 elements
// advances the start address by 32 bytes inside the chunk) ...
template <int D, int BN, int BM, int Q_BYTES, int KV_BYTES, uint32_t ID, bool W = false, int CB = 128>
__device__ __forceinline__ void issue_s_tile_e4m3(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc, int q_slot,
                                                  int slot) {
  uint64_t qd = q_desc + static_cast<uint32_t>((q_slot * Q_BYTES) >> 4);
  uint64_t kd = k_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
  asm volatile("" : "+l"(qd), "+l"(kd));
  constexpr int SPC = CB / 32;  // K steps per chunk
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const uint32_t offa = static_cast<uint32_t>(((k / SPC) * (BM * CB) + (k % SPC) * 32) >> 4);
    const uint32_t offb = static_cast<uint32_t>(((k / SPC) * (BN * CB) + (k % SPC) * 32) >> 4);
    umma_ss_f8<W>(d_tmem, qd + offa, kd + offb, ID, k > 0 ? 1u : 0u);
  }
}

// ... and O (+)= P V with P e4m3 in TMEM (four per column, K = 32 per MMA = 8
// columns) and V stored transposed ([d rows][keys], K-major, one 128-byte chunk of
// BN = 128 keys per row).
template <int D, int BN, int KV_BYTES, uint32_t ID, bool W = false>
__device__ __forceinline__ void issue_pv_tile_e4m3(uint32_t o_tmem, uint32_t p_tmem, uint64_t vt_desc, int slot,
                                                   bool acc) {
  uint64_t vd = vt_desc + static_cast<uint32_t>((slot * KV_BYTES) >> 4);
  asm volatile("" : "+l"(vd));
#pragma unroll
  for (int k = 0; k < BN / 32; ++k) {
    const uint32_t off = static_cast<uint32_t>(((k >> 2) * (D * 128) + (k & 3) * 32) >> 4);
    umma_ts_f8<W>(o_tmem, p_tmem + k * 8, vd + off, ID, (acc || k > 0) ? 1u : 0u);
  }
}

}  // namespace fa
