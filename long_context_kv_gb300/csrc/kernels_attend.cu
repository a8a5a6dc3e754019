// Sparse decode attention of ParisKV over Sink U Local U Update Buffer U the
// retrieved top-k tokens, reading Retrieval-zone rows in place (HBM, or
// mapped pinned host memory through UVA).
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// attention over the top-k subset ("Problem definition"); system level,
// "Unified Virtual Addressing (UVA) offloading" and "Sliding-window update
// mechanism" (Sink and Local on the GPU, the history offloaded).
//
// Split-row flash decoding: block (split, sequence x query head) runs an
// online softmax over kAttnSplit rows of the head's row list (window rows
// first, then the retrieved rows) and writes (max, sum, o); a second kernel
// merges the splits.  Decode has one query row per head, so the work is a
// gather plus matrix-vector products: CUDA cores, not tensor cores.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kAttnThreads = 128;  // 4 warps
constexpr int kRowsPerIter = 8;

struct RowSrc {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
};

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
  return make_float4(bf16_bits_to_float(u.x & 0xffffu), bf16_bits_to_float(u.x >> 16),
                     bf16_bits_to_float(u.y & 0xffffu), bf16_bits_to_float(u.y >> 16));
}

__global__ void __launch_bounds__(kAttnThreads) k_attn_partial(const void* __restrict__ q, int dtype,
                                                              AttendArgs a, int64_t nsink, int64_t nwin,
                                                              float qscale) {
  __shared__ float s_m[4], s_l[4];
  __shared__ float s_o[4][kDim];
  const int split = blockIdx.x;
  const int sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t R = nwin + a.k_eff;
  const int64_t r0 = (int64_t)split * kAttnSplit;
  const int64_t r1 = min64(R, r0 + kAttnSplit);
  const int ring = a.s.local + a.s.ubuf;

  float qv[4];
  load4(q, dtype, (int64_t)sq * kDim + 4 * lane, qv);
#pragma unroll
  for (int i = 0; i < 4; ++i) qv[i] *= qscale;

  float m = -FLT_MAX, l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  const int32_t* tk = a.topk_idx + (int64_t)sq * a.k;
  const __nv_bfloat16* wk = a.kv.win_k + sh * a.kv.win * kDim;
  const __nv_bfloat16* wv = a.kv.win_v + sh * a.kv.win * kDim;
  const __nv_bfloat16* sk = a.kv.st_k + sh * a.kv.rcap * kDim;
  const __nv_bfloat16* sv = a.kv.st_v + sh * a.kv.rcap * kDim;

  // warp w takes rows r0 + w, r0 + w + 4, ... in groups of kRowsPerIter
  for (int64_t rb = r0 + warp; rb < r1; rb += 4 * kRowsPerIter) {
    int64_t off[kRowsPerIter];
    bool valid[kRowsPerIter];
    bool from_store[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int64_t r = rb + 4 * u;
      valid[u] = r < r1;
      from_store[u] = false;
      off[u] = 0;
      if (!valid[u]) continue;
      if (r < nsink) {
        off[u] = r * kDim;
      } else if (r < nwin) {
        const int64_t pos = a.s.sink + a.N + (r - nsink);
        off[u] = (a.s.sink + (pos - a.s.sink) % ring) * kDim;
      } else {
        const int64_t pos = tk[r - nwin];
        if (pos < 0) {
          valid[u] = false;
        } else if (pos < a.s.sink || pos >= a.s.sink + a.N) {
          valid[u] = false;
          if (lane == 0) atomicOr(a.status, kStatusBadIndex);
        } else {
          off[u] = (pos - a.s.sink) * kDim;
          from_store[u] = true;
        }
      }
    }
    float sc[kRowsPerIter];
    uint2 kr[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      kr[u] = make_uint2(0, 0);
      if (valid[u]) {
        const __nv_bfloat16* base = from_store[u] ? sk : wk;
        kr[u] = *reinterpret_cast<const uint2*>(base + off[u] + 4 * lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const float4 kf = bf16x4_to_float4(kr[u]);
      float d = qv[0] * kf.x + qv[1] * kf.y + qv[2] * kf.z + qv[3] * kf.w;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) d += __shfl_xor_sync(kFull, d, s);
      sc[u] = valid[u] ? d : -FLT_MAX;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) mn = fmaxf(mn, sc[u]);
    const float corr = exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] *= corr;
    m = mn;
    uint2 vr[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      vr[u] = make_uint2(0, 0);
      if (valid[u]) {
        const __nv_bfloat16* base = from_store[u] ? sv : wv;
        vr[u] = *reinterpret_cast<const uint2*>(base + off[u] + 4 * lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const float pr = valid[u] ? exp2f(sc[u] - m) : 0.f;
      const float4 vf = bf16x4_to_float4(vr[u]);
      l += pr;
      o[0] += pr * vf.x;
      o[1] += pr * vf.y;
      o[2] += pr * vf.z;
      o[3] += pr * vf.w;
    }
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s_o[warp][4 * lane + i] = o[i];
  __syncthreads();
  float* out = a.part + ((int64_t)sq * a.nsplit_max + split) * kPartStride;
  const float M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
  float f[4], L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    f[w] = s_l[w] > 0.f ? exp2f(s_m[w] - M) : 0.f;
    L += s_l[w] * f[w];
  }
  for (int d = threadIdx.x; d < kDim; d += blockDim.x)
    out[4 + d] = s_o[0][d] * f[0] + s_o[1][d] * f[1] + s_o[2][d] * f[2] + s_o[3][d] * f[3];
  if (threadIdx.x == 0) {
    out[0] = M;
    out[1] = L;
  }
}

__global__ void __launch_bounds__(kDim) k_attn_combine(int nsplit, int nsplit_max, const float* __restrict__ part,
                                                      __nv_bfloat16* __restrict__ out) {
  const int sq = blockIdx.x;
  const int d = threadIdx.x;
  const float* p = part + (int64_t)sq * nsplit_max * kPartStride;
  float M = -FLT_MAX;
  for (int s = 0; s < nsplit; ++s)
    if (p[s * kPartStride + 1] > 0.f) M = fmaxf(M, p[s * kPartStride]);
  float L = 0.f, o = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ls = p[s * kPartStride + 1];
    if (ls > 0.f) {
      const float f = exp2f(p[s * kPartStride] - M);
      L += ls * f;
      o += p[s * kPartStride + 4 + d] * f;
    }
  }
  out[(int64_t)sq * kDim + d] = __float2bfloat16_rn(L > 0.f ? o / L : 0.f);
}

}  // namespace

int attend_splits(const AttendArgs& a) {
  const int64_t nsink = min64(a.s.sink, a.T);
  const int64_t R = nsink + a.n_local_buf + a.k_eff;
  const int nsplit = (int)((R + kAttnSplit - 1) / kAttnSplit);
  return nsplit < 1 ? 1 : nsplit;
}

cudaError_t launch_attn_partial(const void* q, int dtype, const AttendArgs& a, int nsplit, cudaStream_t st) {
  if (nsplit > a.nsplit_max) return cudaErrorInvalidValue;
  const int64_t nsink = min64(a.s.sink, a.T);
  const int64_t nwin = nsink + a.n_local_buf;
  const float qscale = 1.4426950408889634f / sqrtf((float)kDim);
  k_attn_partial<<<dim3(nsplit, a.s.batch * a.s.hq), kAttnThreads, 0, st>>>(q, dtype, a, nsink, nwin, qscale);
  return cudaGetLastError();
}

cudaError_t launch_attn_combine(const AttendArgs& a, int nsplit, cudaStream_t st) {
  k_attn_combine<<<a.s.batch * a.s.hq, kDim, 0, st>>>(nsplit, a.nsplit_max, a.part, a.out);
  return cudaGetLastError();
}

}  // namespace paris
