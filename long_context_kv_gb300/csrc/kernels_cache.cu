// Cache-side kernels of ParisKV: K/V placement into the zones, key encoding
// (bucket ids, RSQ-IP codes, calibration w), the per-chunk inverted bucket
// index, and the decode-time append.
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// Methodology 1 ("Normalization and Rotation", "Analytic Centroids") and
// Methodology 2 ("Quantization", "Calibration": w_{i,b} precomputed at
// prefill); system level, "Sliding-window update mechanism".
#include "paris_device.cuh"

namespace paris {
namespace {

// One warp per key: keys at token positions [pos0, pos1) of every
// (sequence, KV head); input K is [batch][Hkv][T][d].
__global__ void __launch_bounds__(256) k_encode(const void* __restrict__ K, int dtype, int64_t T,
                                                int64_t pos0, int64_t pos1, Shape s, Tables t,
                                                SignMask sm, RsqParams rp) {
  const int lane = threadIdx.x & 31;
  const int64_t span = pos1 - pos0;
  const int64_t total = span * s.batch * s.hkv;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += nwarps) {
    const int64_t sh = w / span;  // seq * Hkv + kvh
    const int64_t pos = pos0 + (w - sh * span);
    float y[4];
    load4(K, dtype, (sh * T + pos) * kDim + 4 * lane, y);
    const int64_t row = sh * t.rcap + (pos - s.sink);
    encode_key_warp(y, lane, sm, rp, t.ids + row * kSub, t.rec + row * kRecBytes,
                    t.cent ? t.cent + (sh % s.hkv) * kTabPerHead : nullptr);
  }
}

__global__ void __launch_bounds__(256) k_place_kv(const void* __restrict__ K, const void* __restrict__ V,
                                                  int dtype, int64_t T, int64_t N, Shape s, KvStore kv) {
  const int64_t rows = T * s.batch * s.hkv;
  const int part = threadIdx.x & 15;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 4);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 4) + (threadIdx.x >> 4); r < rows; r += stride) {
    const int64_t sh = r / T, pos = r - sh * T;
    const uint4 kk = load8_as_bf16(K, dtype, r * kDim + 8 * part);
    const uint4 vv = load8_as_bf16(V, dtype, r * kDim + 8 * part);
    place_row(kk, vv, sh, pos, N, part, s, kv);
  }
}

// Decode append (standalone): one warp per (sequence, KV head).
__global__ void __launch_bounds__(256) k_append(const void* __restrict__ k, const void* __restrict__ v,
                                                int dtype, int64_t pos, Shape s, KvStore kv, Tables t,
                                                SignMask sm, RsqParams rp) {
  const int lane = threadIdx.x & 31;
  const int64_t sh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (sh >= (int64_t)s.batch * s.hkv) return;
  append_token_warp(k, v, dtype, pos, sh, lane, s, kv, t, sm, rp, t.cent);
}

// Inverted bucket index of one chunk of one (sequence, KV head): for every
// subspace b, the chunk-local key numbers grouped by bucket id (a counting
// sort; the order inside a bucket is not significant), with offsets
// off[b][id] .. off[b][id + 1].  The subspaces are independent, so each
// (chunk, sequence x KV head, subspace) is one block: it reads byte b of
// every key's ids once (kept in registers), counts the buckets, scans the
// counts and scatters the key numbers.
constexpr int kIndexThreads = 512;
constexpr int kIndexPer = kChunk / kIndexThreads;  // keys per thread
static_assert(kIndexPer % 4 == 0, "ids packed four to a word");

__global__ void __launch_bounds__(kIndexThreads) k_build_index(int64_t N, int chunk0, Shape s, Tables t) {
  __shared__ uint32_t cnt[kCentroids];
  const int c = chunk0 + blockIdx.x;
  const int64_t sh = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, N - base);
  const uint8_t* ids = t.ids + (sh * t.rcap + base) * kSub + b;
  uint32_t* off = t.off + ((sh * t.nchunk + c) * kSub + b) * kOffStride;
  uint16_t* ent = t.ent + ((sh * t.nchunk + c) * kSub + b) * (int64_t)kChunk;

  for (int i = tid; i < kCentroids; i += kIndexThreads) cnt[i] = 0;
  // key tid + kIndexThreads j; its id in byte j % 4 of word j / 4
  uint32_t packed[kIndexPer / 4];
#pragma unroll
  for (int j = 0; j < kIndexPer; ++j) {
    const int key = tid + kIndexThreads * j;
    const uint32_t id = key < len ? (uint32_t)__ldg(ids + (int64_t)key * kSub) : 0u;
    if ((j & 3) == 0) packed[j >> 2] = 0;
    packed[j >> 2] |= id << (8 * (j & 3));
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kIndexPer; ++j)
    if (tid + kIndexThreads * j < len) atomicAdd(&cnt[(packed[j >> 2] >> (8 * (j & 3))) & 0xffu], 1u);
  __syncthreads();
  // exclusive scan of the 256 counts: warp 0, 8 bins per lane
  if (warp == 0) {
    uint32_t vals[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      vals[i] = cnt[8 * lane + i];
      sum += vals[i];
    }
    uint32_t run = warp_incl_scan(sum, lane) - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      off[8 * lane + i] = run;
      cnt[8 * lane + i] = run;
      run += vals[i];
    }
    if (lane == 31) off[kCentroids] = run;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kIndexPer; ++j) {
    const int key = tid + kIndexThreads * j;
    if (key < len) {
      const uint32_t p = atomicAdd(&cnt[(packed[j >> 2] >> (8 * (j & 3))) & 0xffu], 1u);
      ent[p] = (uint16_t)key;
    }
  }
}

inline int grid_for(int64_t items, int per_block, int cap) {
  int64_t g = (items + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

}  // namespace

cudaError_t launch_place_kv(const void* K, const void* V, int dtype, int64_t T, int64_t N,
                            const Shape& s, const KvStore& kv, cudaStream_t st) {
  const int64_t rows = T * s.batch * s.hkv;
  if (rows == 0) return cudaSuccess;
  k_place_kv<<<grid_for(rows, 16, 152 * 16), 256, 0, st>>>(K, V, dtype, T, N, s, kv);
  return cudaGetLastError();
}

cudaError_t launch_encode(const void* K, int dtype, int64_t T, int64_t pos0, int64_t pos1,
                          const Shape& s, const Tables& t, const SignMask& sm, const RsqParams& rp,
                          cudaStream_t st) {
  const int64_t n = (pos1 - pos0) * s.batch * s.hkv;
  if (n <= 0) return cudaSuccess;
  k_encode<<<grid_for(n, 8, 152 * 32), 256, 0, st>>>(K, dtype, T, pos0, pos1, s, t, sm, rp);
  return cudaGetLastError();
}

cudaError_t launch_build_index(int64_t N, int chunk0, int chunk1, const Shape& s, const Tables& t,
                               cudaStream_t st) {
  if (chunk1 <= chunk0) return cudaSuccess;
  dim3 grid(chunk1 - chunk0, s.batch * s.hkv, kSub);
  k_build_index<<<grid, kIndexThreads, 0, st>>>(N, chunk0, s, t);
  return cudaGetLastError();
}

cudaError_t launch_append(const void* k, const void* v, int dtype, int64_t pos, const Shape& s,
                          const KvStore& kv, const Tables& t, const SignMask& sm,
                          const RsqParams& rp, cudaStream_t st) {
  const int n = s.batch * s.hkv;
  k_append<<<(n + 7) / 8, 256, 0, st>>>(k, v, dtype, pos, s, kv, t, sm, rp);
  return cudaGetLastError();
}

}  // namespace paris
