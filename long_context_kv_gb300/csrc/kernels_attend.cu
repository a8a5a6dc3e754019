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
// first, then the retrieved rows) and writes (max, sum, o); the last split
// of a query head to finish merges all splits (atomic counter after a
// memory fence, no waiting).  Decode has one query row per head, so the work
// is a gather plus matrix-vector products: CUDA cores, not tensor cores.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kAttnThreads = 128;  // 4 warps x 32 rows
constexpr int kRowsPerIter = 8;
static_assert(kAttnThreads == kDim && kAttnThreads == kAttnSplit, "one thread per row and per output dimension");

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
  return make_float4(bf16_bits_to_float(u.x & 0xffffu), bf16_bits_to_float(u.x >> 16),
                     bf16_bits_to_float(u.y & 0xffffu), bf16_bits_to_float(u.y >> 16));
}

__global__ void __launch_bounds__(kAttnThreads) k_attend(const void* __restrict__ q, int dtype, AttendArgs a,
                                                        int64_t nsink, int64_t nwin, int nsplit, float qscale) {
  __shared__ const __nv_bfloat16* s_k[kAttnSplit];
  __shared__ const __nv_bfloat16* s_v[kAttnSplit];
  __shared__ float s_m[4], s_l[4];
  __shared__ float s_o[4][kDim];
  __shared__ int s_last;
  const int split = blockIdx.x;
  const int sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t R = nwin + a.k_eff;
  const int64_t r0 = (int64_t)split * kAttnSplit;
  const int ring = a.s.local + a.s.ubuf;

  // row addresses of the split (nullptr: no row)
  {
    const int64_t r = r0 + tid;
    const __nv_bfloat16 *kp = nullptr, *vp = nullptr;
    if (r < R) {
      if (r < nwin) {
        int64_t slot = r;
        if (r >= nsink) {
          const int64_t pos = a.s.sink + a.N + (r - nsink);
          slot = a.s.sink + (pos - a.s.sink) % ring;
        }
        kp = a.kv.win_k + (sh * a.kv.win + slot) * kDim;
        vp = a.kv.win_v + (sh * a.kv.win + slot) * kDim;
      } else {
        const int64_t pos = __ldg(a.topk_idx + (int64_t)sq * a.k + (r - nwin));
        if (pos >= a.s.sink && pos < a.s.sink + a.N) {
          kp = a.kv.st_k + (sh * a.kv.rcap + (pos - a.s.sink)) * kDim;
          vp = a.kv.st_v + (sh * a.kv.rcap + (pos - a.s.sink)) * kDim;
        } else if (pos >= 0) {
          atomicOr(a.status, kStatusBadIndex);
        }
      }
    }
    s_k[tid] = kp;
    s_v[tid] = vp;
  }
  float qv[4];
  load4(q, dtype, (int64_t)sq * kDim + 4 * lane, qv);
#pragma unroll
  for (int i = 0; i < 4; ++i) qv[i] *= qscale;
  __syncthreads();

  float m = -FLT_MAX, l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  // warp w takes rows 32w .. 32w + 31 of the split, kRowsPerIter at a time,
  // K and V of all of them in flight together
#pragma unroll 1
  for (int rb = 32 * warp; rb < 32 * warp + 32; rb += kRowsPerIter) {
    uint2 kr[kRowsPerIter], vr[kRowsPerIter];
    bool valid[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const __nv_bfloat16* kp = s_k[rb + u];
      const __nv_bfloat16* vp = s_v[rb + u];
      valid[u] = kp != nullptr;
      kr[u] = valid[u] ? *reinterpret_cast<const uint2*>(kp + 4 * lane) : make_uint2(0, 0);
      vr[u] = valid[u] ? *reinterpret_cast<const uint2*>(vp + 4 * lane) : make_uint2(0, 0);
    }
    float sc[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const float4 kf = bf16x4_to_float4(kr[u]);
      sc[u] = qv[0] * kf.x + qv[1] * kf.y + qv[2] * kf.z + qv[3] * kf.w;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) sc[u] += __shfl_xor_sync(kFull, sc[u], s);
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u)
      if (valid[u]) mn = fmaxf(mn, sc[u]);
    const float corr = exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] *= corr;
    m = mn;
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
  float* part = a.part + (int64_t)sq * a.nsplit_max * kPartStride;
  {
    const float M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
    float f[4], L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      f[w] = s_l[w] > 0.f ? exp2f(s_m[w] - M) : 0.f;
      L += s_l[w] * f[w];
    }
    float* out = part + (int64_t)split * kPartStride;
    const int d = tid;  // kAttnThreads == kDim
    out[4 + d] = s_o[0][d] * f[0] + s_o[1][d] * f[1] + s_o[2][d] * f[2] + s_o[3][d] * f[3];
    if (tid == 0) {
      out[0] = M;
      out[1] = L;
    }
  }
  // the last split of the query head merges all splits
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counter[sq], 1u) == (uint32_t)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int d = tid;
  float M = -FLT_MAX;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float mm[8], ll[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = s0 + u < nsplit;
      mm[u] = in ? __ldcg(part + (int64_t)(s0 + u) * kPartStride) : -FLT_MAX;
      ll[u] = in ? __ldcg(part + (int64_t)(s0 + u) * kPartStride + 1) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (ll[u] > 0.f) M = fmaxf(M, mm[u]);
  }
  float L = 0.f, acc = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float mm[8], ll[8], oo[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = s0 + u < nsplit;
      const float* p = part + (int64_t)(s0 + u) * kPartStride;
      mm[u] = in ? __ldcg(p) : 0.f;
      ll[u] = in ? __ldcg(p + 1) : 0.f;
      oo[u] = in ? __ldcg(p + 4 + d) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (ll[u] > 0.f) {
        const float f = exp2f(mm[u] - M);
        L += ll[u] * f;
        acc += oo[u] * f;
      }
    }
  }
  a.out[(int64_t)sq * kDim + d] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
  if (tid == 0) a.counter[sq] = 0;
}

}  // namespace

int attend_splits(const AttendArgs& a) {
  const int64_t nsink = min64(a.s.sink, a.T);
  const int64_t R = nsink + a.n_local_buf + a.k_eff;
  const int nsplit = (int)((R + kAttnSplit - 1) / kAttnSplit);
  return nsplit < 1 ? 1 : nsplit;
}

cudaError_t launch_attend(const void* q, int dtype, const AttendArgs& a, cudaStream_t st) {
  const int nsplit = attend_splits(a);
  if (nsplit > a.nsplit_max) return cudaErrorInvalidValue;
  const int64_t nsink = min64(a.s.sink, a.T);
  const int64_t nwin = nsink + a.n_local_buf;
  const float qscale = 1.4426950408889634f / sqrtf((float)kDim);
  k_attend<<<dim3(nsplit, a.s.batch * a.s.hq), kAttnThreads, 0, st>>>(q, dtype, a, nsink, nwin, nsplit, qscale);
  return cudaGetLastError();
}

}  // namespace paris
