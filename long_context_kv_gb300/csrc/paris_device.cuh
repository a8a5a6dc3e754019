// Device helpers shared by the ParisKV kernels: input loads, the in-warp
// fast Walsh-Hadamard transform and warp/block scans.
#pragma once

#include "paris_internal.cuh"

namespace paris {

constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Four consecutive elements [i, i+4) of a float32 (dtype 0) or bf16 (dtype 1)
// array as float32.  Requires i % 4 == 0 and a 8/16-byte aligned base.
__device__ __forceinline__ void load4(const void* p, int dtype, int64_t i, float (&y)[4]) {
  if (dtype == 0) {
    float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    y[0] = v.x; y[1] = v.y; y[2] = v.z; y[3] = v.w;
  } else {
    uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i);
    y[0] = bf16_bits_to_float(v.x & 0xffffu);
    y[1] = bf16_bits_to_float(v.x >> 16);
    y[2] = bf16_bits_to_float(v.y & 0xffffu);
    y[3] = bf16_bits_to_float(v.y >> 16);
  }
}

__device__ __forceinline__ float load1(const void* p, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(p)[i];
  return bf16_bits_to_float(static_cast<const uint16_t*>(p)[i]);
}

// y_c <- D_c * y_c for the lane's coordinates c = 4*lane + i (exact negation).
__device__ __forceinline__ void apply_signs(float (&y)[4], const SignMask& sm, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = 4 * lane + i;
    if ((sm.w[c >> 5] >> (c & 31)) & 1u) y[i] = -y[i];
  }
}

// Unnormalised Walsh-Hadamard transform of a 128-vector held by one warp,
// lane l owning coordinates 4l..4l+3.  Stages run in the order h = 1, 2, 4,
// ..., 64; in stage h the pair (i, i + h) with i & h == 0 becomes
// (y_i + y_{i+h}, y_i - y_{i+h}), each rounded once (no contraction).
// Stages 1 and 2 stay in registers; stage h >= 4 exchanges with lane l ^ h/4.
__device__ __forceinline__ void fwht128_warp(float (&y)[4], int lane) {
  const float a0 = __fadd_rn(y[0], y[1]), a1 = __fsub_rn(y[0], y[1]);
  const float a2 = __fadd_rn(y[2], y[3]), a3 = __fsub_rn(y[2], y[3]);
  y[0] = __fadd_rn(a0, a2);
  y[2] = __fsub_rn(a0, a2);
  y[1] = __fadd_rn(a1, a3);
  y[3] = __fsub_rn(a1, a3);
#pragma unroll
  for (int dl = 1; dl < 32; dl <<= 1) {
    const bool upper = (lane & dl) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(kFull, y[i], dl);
      y[i] = upper ? __fsub_rn(p, y[i]) : __fadd_rn(y[i], p);
    }
  }
}

// Inclusive warp scan of unsigned values.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block scan of one unsigned value per thread; blockDim.x must be
// a multiple of 32 and at most 1024.  `tmp` holds 33 words of shared memory.
// Returns the exclusive prefix; *total receives the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* tmp, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint32_t inc = warp_incl_scan(v, lane);
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = lane < nw ? tmp[lane] : 0u;
    const uint32_t xi = warp_incl_scan(x, lane);
    if (lane < nw) tmp[lane] = xi - x;
    if (lane == 31) tmp[32] = xi;
  }
  __syncthreads();
  const uint32_t r = tmp[warp] + inc - v;
  *total = tmp[32];
  __syncthreads();
  return r;
}

}  // namespace paris
