// quant.cuh -- per-tensor e4m3 quantisation of Q or K for the attention
// kernels, optionally after a Hadamard rotation of every head vector.
//
// "Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "How accurate is ZYFA's
// FP8 attention?": most of the FP8 error comes from quantising Q, K and V,
// and a Hadamard rotation of Q and K roughly halves it at a tiny cost.  A
// common orthogonal rotation leaves Q K^T unchanged, and spreads an outlier
// channel over the whole head vector, so one per-tensor scale fits all.
//
// Definition (all arithmetic fp32):
//   y = x, or the unnormalised Walsh-Hadamard transform of each head vector
//   in blocks of hb elements (hb = 128 for D = 128; three blocks of 64 for
//   D = 192): butterfly stages h = 1, 2, 4, ..., hb/2, each pair (i, i+h) with
//   i mod 2h < h becoming (y_i + y_{i+h}, y_i - y_{i+h}).
//   amax = max |y|; code = e4m3_rn_satfinite(y * (448 / amax));
//   descale = (amax / 448) * norm, norm = 1/sqrt(hb) (1 without rotation).
//
// Three launches, all HBM-bound: amax (atomic max into the descale word, the
// caller's output, so no scratch memory), quantisation (re-reads x) and a
// one-thread finalisation of the descale.  Four lanes per head vector, eight
// vectors per warp, in a grid-stride loop: lane j of a vector holds, of each
// block of hb elements, the hb/4 consecutive elements starting at j*hb/4.  The
// first log2(hb/4) butterfly stages run in registers, the last two exchange
// with lane j ^ 1 and j ^ 2 by shuffles (the lower element of a pair computes
// a + b, the upper a - b, exactly as above, each as one sign-selected fma).
// From the second stage on, elements 2k and 2k+1 of a segment always meet the
// same partner offset, so the stages run on packed f32x2 pairs: the same fp32
// operations, two per instruction.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa8 {

constexpr int kQuantThreads = 256;
constexpr int kQuantLanes = 4;                 // lanes per head vector
constexpr int kQuantVecPerWarp = 32 / kQuantLanes;

template <int D>
struct QuantLayout {
  static constexpr int kBlock = D == 192 ? 64 : D;  // Hadamard block
  static constexpr int kBlocks = D / kBlock;
  static constexpr int kSeg = kBlock / kQuantLanes;  // consecutive elements per lane and block
  static constexpr int kPerLane = kBlocks * kSeg;    // 32 (D = 128) or 48 (D = 192)
};

// Packed fp32 pairs (sm_100+): round-to-nearest a*b + c and a - b on both lanes.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Loads the lane's elements of vector v (zeros when v >= n_vec).
template <int D, bool F32>
__device__ __forceinline__ void quant_load(const void* x, int64_t v, int64_t n_vec, int j,
                                           float (&r)[QuantLayout<D>::kPerLane]) {
  using L = QuantLayout<D>;
  if (v >= n_vec) {
#pragma unroll
    for (int i = 0; i < L::kPerLane; ++i) r[i] = 0.0f;
    return;
  }
#pragma unroll
  for (int c = 0; c < L::kBlocks; ++c) {
    const int64_t e0 = v * D + c * L::kBlock + j * L::kSeg;  // first element
    if constexpr (F32) {
      const float4* src = reinterpret_cast<const float4*>(x) + e0 / 4;
#pragma unroll
      for (int t = 0; t < L::kSeg / 4; ++t) {
        const float4 w = src[t];
        r[c * L::kSeg + 4 * t] = w.x, r[c * L::kSeg + 4 * t + 1] = w.y;
        r[c * L::kSeg + 4 * t + 2] = w.z, r[c * L::kSeg + 4 * t + 3] = w.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x) + e0 / 8;
#pragma unroll
      for (int t = 0; t < L::kSeg / 8; ++t) {
        const uint4 w = src[t];
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          r[c * L::kSeg + 8 * t + 2 * u] = bf16_lo(q[u]);
          r[c * L::kSeg + 8 * t + 2 * u + 1] = bf16_hi(q[u]);
        }
      }
    }
  }
}

// One butterfly stage, for two packed elements, whose partner elements sit in
// lane (lane ^ m): the lower element of a pair (lane bit m clear) gets a + b,
// the upper a - b, both as fma(mine, +-1, other), which rounds exactly like
// the add or the subtraction.  `sg2` holds +1 twice in the lower lane and -1
// twice in the upper one.
__device__ __forceinline__ uint64_t xlane_butterfly2(uint64_t mine, uint64_t sg2, int m) {
  uint32_t lo, hi;
  f32x2_unpack(mine, lo, hi);
  const uint64_t other = f32x2_pack(__uint_as_float(__shfl_xor_sync(0xffffffffu, lo, m)),
                                    __uint_as_float(__shfl_xor_sync(0xffffffffu, hi, m)));
  return fma_f32x2(mine, sg2, other);
}

template <int D>
__device__ __forceinline__ void quant_rotate(float (&r)[QuantLayout<D>::kPerLane], int lane) {
  using L = QuantLayout<D>;
#pragma unroll
  for (int c = 0; c < L::kBlocks; ++c) {
    float* b = &r[c * L::kSeg];
    // stage h = 1 inside the lane's segment
#pragma unroll
    for (int i = 0; i < L::kSeg; i += 2) {
      const float a = b[i], e = b[i + 1];
      b[i] = a + e;
      b[i + 1] = a - e;
    }
    // stages h = 2 .. kSeg/2: elements 2k and 2k+1 have the same partner
    // offset, so each pair of pairs is one packed add and one packed
    // subtraction (the same fp32 operations, two at a time)
    uint64_t pk[L::kSeg / 2];
#pragma unroll
    for (int k = 0; k < L::kSeg / 2; ++k) pk[k] = f32x2_pack(b[2 * k], b[2 * k + 1]);
#pragma unroll
    for (int h2 = 1; h2 < L::kSeg / 2; h2 *= 2) {
#pragma unroll
      for (int k = 0; k < L::kSeg / 2; ++k)
        if ((k & h2) == 0) {
          const uint64_t a = pk[k], e = pk[k + h2];
          pk[k] = add_f32x2(a, e);
          pk[k + h2] = sub_f32x2(a, e);
        }
    }
    // stages h = kSeg, 2 kSeg: partner lane j ^ 1, j ^ 2 (vector-local lane j = lane & 3)
#pragma unroll
    for (int m = 1; m < kQuantLanes; m *= 2) {
      const float sg = (lane & m) ? -1.0f : 1.0f;
      const uint64_t sg2 = f32x2_pack(sg, sg);
#pragma unroll
      for (int k = 0; k < L::kSeg / 2; ++k) pk[k] = xlane_butterfly2(pk[k], sg2, m);
    }
#pragma unroll
    for (int k = 0; k < L::kSeg / 2; ++k) {
      uint32_t lo, hi;
      f32x2_unpack(pk[k], lo, hi);
      b[2 * k] = __uint_as_float(lo);
      b[2 * k + 1] = __uint_as_float(hi);
    }
  }
}

template <int D, bool F32>
__global__ void __launch_bounds__(kQuantThreads) quant_amax_kernel(const void* x, int64_t n_vec,
                                                                  int rotate, float* amax) {
  using L = QuantLayout<D>;
  const int lane = threadIdx.x & 31, j = lane & (kQuantLanes - 1);
  const int64_t g0 = ((int64_t)blockIdx.x * kQuantThreads + threadIdx.x) >> 5;  // warp
  const int64_t ng = ((int64_t)gridDim.x * kQuantThreads) >> 5;
  float m = 0.0f;
  for (int64_t g = g0; g * kQuantVecPerWarp < n_vec; g += ng) {
    const int64_t v = g * kQuantVecPerWarp + lane / kQuantLanes;
    float r[L::kPerLane];
    quant_load<D, F32>(x, v, n_vec, j, r);
    if (rotate) quant_rotate<D>(r, lane);
#pragma unroll
    for (int i = 0; i < L::kPerLane; ++i) m = fmaxf(m, fabsf(r[i]));
  }
  // non-negative floats order like their bit patterns
  const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if (lane == 0 && mb != 0) atomicMax(reinterpret_cast<unsigned int*>(amax), mb);
}

template <int D, bool F32>
__global__ void __launch_bounds__(kQuantThreads) quant_codes_kernel(const void* x, int64_t n_vec,
                                                                   int rotate, const float* amax,
                                                                   uint8_t* codes) {
  using L = QuantLayout<D>;
  const int lane = threadIdx.x & 31, j = lane & (kQuantLanes - 1);
  const int64_t g0 = ((int64_t)blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
  const int64_t ng = ((int64_t)gridDim.x * kQuantThreads) >> 5;
  const float a = *amax;
  const float sc = a > 0.0f ? 448.0f / a : 1.0f;
  const int64_t n_groups = (n_vec + kQuantVecPerWarp - 1) / kQuantVecPerWarp;
  for (int64_t i = g0; i < n_groups; i += ng) {
    // backwards: the amax pass swept forwards and has just left the end of x
    // in L2, so the first groups read here are L2 hits (each code depends
    // only on its vector and the amax, so the order changes no result)
    const int64_t g = n_groups - 1 - i;
    const int64_t v = g * kQuantVecPerWarp + lane / kQuantLanes;
    float r[L::kPerLane];
    quant_load<D, F32>(x, v, n_vec, j, r);
    if (rotate) quant_rotate<D>(r, lane);
    if (v >= n_vec) continue;
#pragma unroll
    for (int c = 0; c < L::kBlocks; ++c) {
      uint32_t w[L::kSeg / 4];
#pragma unroll
      for (int t = 0; t < L::kSeg / 4; ++t) {
        const float* e = &r[c * L::kSeg + 4 * t];
        w[t] = f32x2_to_e4m3x2(e[0] * sc, e[1] * sc) | (f32x2_to_e4m3x2(e[2] * sc, e[3] * sc) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(codes + v * D + c * L::kBlock + j * L::kSeg);
#pragma unroll
      for (int t = 0; t < L::kSeg / 16; ++t) dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
    }
  }
}

// descale = (amax / 448) * norm (1 * norm for an all-zero tensor).
__global__ void quant_finish_kernel(float* descale, float norm) {
  const float a = *descale;
  *descale = (a > 0.0f ? a / 448.0f : 1.0f) * norm;
}

}  // namespace fa8
