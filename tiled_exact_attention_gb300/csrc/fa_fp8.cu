// e4m3 quantisation for the 8-bit forward path ("hs-black: FlashAttention 1/2/3",
// section "FlashAttention-3: precision and hardware": a scale factor per block
// so that a few large values do not crush the precision of the whole block, and
// the scales carried into the computation).
//
// Per tensor, bound by HBM:
//   * fa_amax_kernel (one CTA per 128-row block of one (batch, head)): the block's
//     largest |x|, max-reduced into its scale slot (one slot per block, or one per
//     (batch, head) shared by its blocks: an integer atomic max on the bits of a
//     non-negative float orders like the float);
//   * fa_quant_kernel: descale = amax / 448 (448 is the largest finite e4m3 value;
//     an all-zero block gets 1), code = round-to-nearest-even e4m3 of
//     x * (1 / descale), saturating, written row-major or transposed ([d][rows], for V);
//   * fa_descale_kernel: the slots turn from amax into descale.
// The products use IEEE round-to-nearest (division, reciprocal, multiplication
// written with the _rn intrinsics), so a CPU check reproduces every code bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kE4m3Max = 448.f;

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t u) {
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  } else {
    return __half2float(__ushort_as_half(u));
  }
}

__device__ __forceinline__ float descale_of(float amax) { return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f; }

__device__ __forceinline__ int64_t scale_slot(const QuantParams& p, int bh, int blk) {
  return p.per_head ? bh : static_cast<int64_t>(bh) * p.nblk + blk;
}

// One CTA of 256 threads per 128-row block of one (batch, head); the slots start at 0.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_amax_kernel(const __grid_constant__ QuantParams p) {
  __shared__ float red[8];
  const int blk = blockIdx.x % p.nblk;
  const int bh = blockIdx.x / p.nblk;
  const int h = bh % p.h, bi = bh / p.h;
  const int r0 = blk * 128;
  const int r1 = min(p.s, r0 + 128);
  const int vec = p.d / 8;  // 16-byte pieces per row
  float m = 0.f;
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(r1 - r0) * vec; i += 256) {
    const int row = r0 + static_cast<int>(i / vec), c = static_cast<int>(i % vec);
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + bi * p.x_st[0] +
                                                     static_cast<int64_t>(row) * p.x_st[1] + h * p.x_st[2] + c * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m = fmaxf(m, fabsf(to_f32<BF16>(static_cast<uint16_t>(w[e] & 0xffffu))));
      m = fmaxf(m, fabsf(to_f32<BF16>(static_cast<uint16_t>(w[e] >> 16))));
    }
  }
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, x));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
    atomicMax(reinterpret_cast<int*>(p.descale + scale_slot(p, bh, blk)), __float_as_int(a));
  }
}

// The slots hold amax; make them descales.
__global__ void __launch_bounds__(256) fa_descale_kernel(float* slots, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n; i += static_cast<int64_t>(gridDim.x) * 256)
    slots[i] = descale_of(slots[i]);
}

// One CTA of 256 threads per 128-row block of one (batch, head).
template <bool BF16, bool TRANSPOSE>
__global__ void __launch_bounds__(256) fa_quant_kernel(const __grid_constant__ QuantParams p) {
  __shared__ __align__(16) uint8_t tile[256 * 128 + 16];  // transposed: [d][128 rows], d <= 256
  const int blk = blockIdx.x % p.nblk;
  const int bh = blockIdx.x / p.nblk;
  const int h = bh % p.h, bi = bh / p.h;
  const int r0 = blk * 128;
  const int rows = min(128, p.s - r0);
  const float ds = descale_of(p.descale[scale_slot(p, bh, blk)]);  // (the slot holds amax until the end)
  const float inv = __frcp_rn(ds);
  const int vec = p.d / 8;
  for (int i = threadIdx.x; i < rows * vec; i += 256) {
    const int rr = i / vec, c = i % vec;
    const int row = r0 + rr;
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + bi * p.x_st[0] +
                                                     static_cast<int64_t>(row) * p.x_st[1] + h * p.x_st[2] + c * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __fmul_rn(to_f32<BF16>(static_cast<uint16_t>(w[e] & 0xffffu)), inv);
      f[2 * e + 1] = __fmul_rn(to_f32<BF16>(static_cast<uint16_t>(w[e] >> 16)), inv);
    }
    const uint32_t lo = pack4_e4m3(f[0], f[1], f[2], f[3]);
    const uint32_t hi = pack4_e4m3(f[4], f[5], f[6], f[7]);
    if constexpr (TRANSPOSE) {
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[(c * 8 + e) * 128 + rr] = static_cast<uint8_t>(((e < 4 ? lo : hi) >> (8 * (e & 3))) & 0xffu);
    } else {
      uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + bi * p.out_st[0] +
                                            static_cast<int64_t>(row) * p.out_st[1] + h * p.out_st[2] + c * 8);
      *dst = make_uint2(lo, hi);
    }
  }
  if constexpr (TRANSPOSE) {
    __syncthreads();
    // out [b][h][d][rows], the row index contiguous: 16-byte pieces of 16 rows
    const int pieces = (rows + 15) / 16;
    for (int i = threadIdx.x; i < p.d * pieces; i += 256) {
      const int dc = i / pieces, pc = i % pieces;
      uint8_t* dst = static_cast<uint8_t*>(p.out) + bi * p.out_st[0] + h * p.out_st[1] +
                     static_cast<int64_t>(dc) * p.out_st[2] + r0 + pc * 16;
      const uint8_t* src = tile + dc * 128 + pc * 16;
      if (pc * 16 + 16 <= rows) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      } else {
        for (int e = 0; pc * 16 + e < rows; ++e) dst[e] = src[e];
      }
    }
  }
}

template <bool BF16>
cudaError_t launch_quant_t(const QuantParams& p, cudaStream_t stream) {
  const int64_t nslots = static_cast<int64_t>(p.b) * p.h * (p.per_head ? 1 : p.nblk);
  const int64_t g = static_cast<int64_t>(p.b) * p.h * p.nblk;
  if (g <= 0) return cudaSuccess;
  if (g > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaMemsetAsync(p.descale, 0, static_cast<size_t>(nslots) * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  fa_amax_kernel<BF16><<<static_cast<unsigned>(g), 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.transpose)
    fa_quant_kernel<BF16, true><<<static_cast<unsigned>(g), 256, 0, stream>>>(p);
  else
    fa_quant_kernel<BF16, false><<<static_cast<unsigned>(g), 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t g3 = (nslots + 255) / 256;
  fa_descale_kernel<<<static_cast<unsigned>(g3 < 1024 ? g3 : 1024), 256, 0, stream>>>(p.descale, nslots);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_e4m3(const QuantParams& p, int dtype, cudaStream_t stream) {
  return dtype == 0 ? launch_quant_t<true>(p, stream) : launch_quant_t<false>(p, stream);
}

}  // namespace fa
