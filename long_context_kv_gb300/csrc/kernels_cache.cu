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

// Encode one key held by a warp (lane l owns coordinates 4l..4l+3 of the
// raw key).  Float32 order, every operation rounded once:
//   z = fwht(D * k);  id_b bit j = [z_{b,j} < 0];
//   n_b = sqrt(((0 + z_0 z_0) + z_1 z_1) + ... + z_7 z_7);
//   x_j = z_j / n_b;  sign s_j = [z_j < 0];  t_j = #{thr < |x_j|};
//   v_j = (-1)^s_j lev[t_j];  <v,x> = ((0 + v_0 x_0) + v_1 x_1) + ...;
//   w_b = n_b / (sqrt(d) * <v,x>), and w_b = 0, codes 0 where n_b = 0.
// Subspace b is lanes 2b (j = 0..3) and 2b+1 (j = 4..7); a sequential sum
// over j starts in the even lane and continues in the odd lane.
// Writes the 16 ids and the 128-byte record (16 code words, 16 w) of the key.
__device__ __forceinline__ void encode_key_warp(float (&y)[4], int lane, const SignMask& sm,
                                                const RsqParams& rp, uint8_t* ids_row,
                                                uint8_t* rec_row) {
  apply_signs(y, sm, lane);
  fwht128_warp(y, lane);
  const bool odd = (lane & 1) != 0;

  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) bits |= (y[i] < 0.f ? 1u : 0u) << i;
  const uint32_t obits = __shfl_xor_sync(kFull, bits, 1);
  const uint32_t id = odd ? (obits | (bits << 4)) : (bits | (obits << 4));

  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc = __fadd_rn(acc, __fmul_rn(y[i], y[i]));
  float acc2 = __shfl_xor_sync(kFull, acc, 1);
#pragma unroll
  for (int i = 0; i < 4; ++i) acc2 = __fadd_rn(acc2, __fmul_rn(y[i], y[i]));
  const float nsq = __shfl_sync(kFull, acc2, lane | 1);
  const float nb = __fsqrt_rn(nsq);
  const bool live = nb > 0.f;

  float x[4], v[4];
  uint32_t half = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = live ? __fdiv_rn(y[i], nb) : 0.f;
    const float ax = fabsf(x[i]);
    uint32_t t = 0;
#pragma unroll
    for (int r = 0; r < 7; ++r) t += (rp.thr[r] < ax) ? 1u : 0u;
    const uint32_t s = (live && y[i] < 0.f) ? 1u : 0u;
    const float l = rp.lev[t];
    v[i] = s ? -l : l;
    half |= ((s << 3) | t) << (4 * i);
  }
  float vx = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) vx = __fadd_rn(vx, __fmul_rn(v[i], x[i]));
  float vx2 = __shfl_xor_sync(kFull, vx, 1);
#pragma unroll
  for (int i = 0; i < 4; ++i) vx2 = __fadd_rn(vx2, __fmul_rn(v[i], x[i]));
  const float w = live ? __fdiv_rn(nb, __fmul_rn(rp.sqrtd, vx2)) : 0.f;  // valid in odd lanes

  // record word l: l < 16 the code word of subspace l, else w of subspace l - 16
  const uint32_t h_lo = __shfl_sync(kFull, half, (2 * lane) & 31);
  const uint32_t h_hi = __shfl_sync(kFull, half, (2 * lane + 1) & 31);
  const float w_src = __shfl_sync(kFull, w, (2 * (lane - 16) + 1) & 31);
  const uint32_t word = lane < 16 ? (h_lo | (h_hi << 16)) : __float_as_uint(w_src);
  reinterpret_cast<uint32_t*>(rec_row)[lane] = word;

  // ids word q (q < 4) holds the ids of subspaces 4q..4q+3, one byte each
  uint32_t idw = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t o = __shfl_sync(kFull, id, (2 * (4 * (lane & 3) + i)) & 31);
    idw |= (o & 0xffu) << (8 * i);
  }
  if (lane < 4) reinterpret_cast<uint32_t*>(ids_row)[lane] = idw;
}

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
    encode_key_warp(y, lane, sm, rp, t.ids + row * kSub, t.rec + row * kRecBytes);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Copy 8 consecutive elements (element offset e, multiple of 8) of a float32
// or bf16 row to bf16 destinations.
__device__ __forceinline__ uint4 load8_as_bf16(const void* p, int dtype, int64_t e) {
  if (dtype == 1) return *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + e);
  const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + e);
  const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + e + 4);
  return make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                    pack_bf16x2(b.z, b.w));
}

// Place K/V row `pos` of (sequence, KV head) `sh`: Sink slot if pos < S;
// otherwise the store row pos - S, and the Local/Buffer ring slot when the
// token is in Local or the Buffer (pos >= S + N).  16 threads per row.
__device__ __forceinline__ void place_row(uint4 kk, uint4 vv, int64_t sh, int64_t pos, int64_t N,
                                          int part, const Shape& s, const KvStore& kv) {
  const int ring = s.local + s.ubuf;
  if (pos < s.sink) {
    const int64_t o = (sh * kv.win + pos) * kDim + 8 * part;
    *reinterpret_cast<uint4*>(kv.win_k + o) = kk;
    *reinterpret_cast<uint4*>(kv.win_v + o) = vv;
    return;
  }
  const int64_t so = (sh * kv.rcap + (pos - s.sink)) * kDim + 8 * part;
  *reinterpret_cast<uint4*>(kv.st_k + so) = kk;
  *reinterpret_cast<uint4*>(kv.st_v + so) = vv;
  if (pos >= s.sink + N) {
    const int64_t slot = s.sink + (pos - s.sink) % ring;
    const int64_t o = (sh * kv.win + slot) * kDim + 8 * part;
    *reinterpret_cast<uint4*>(kv.win_k + o) = kk;
    *reinterpret_cast<uint4*>(kv.win_v + o) = vv;
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

// Decode append: one warp per (sequence, KV head).  Stores the token's K/V
// as bf16 and, outside the Sink, encodes its key at table row pos - S so the
// row is ready when the token is later evicted into the Retrieval zone.
__global__ void __launch_bounds__(256) k_append(const void* __restrict__ k, const void* __restrict__ v,
                                                int dtype, int64_t pos, Shape s, KvStore kv, Tables t,
                                                SignMask sm, RsqParams rp) {
  const int lane = threadIdx.x & 31;
  const int64_t sh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (sh >= (int64_t)s.batch * s.hkv) return;
  if (lane < 16) {
    const uint4 kk = load8_as_bf16(k, dtype, sh * kDim + 8 * lane);
    const uint4 vv = load8_as_bf16(v, dtype, sh * kDim + 8 * lane);
    // a new token is never in the Retrieval zone: with N = 0 every position
    // past the Sink also lands in its Local/Buffer ring slot
    place_row(kk, vv, sh, pos, /*N=*/0, lane, s, kv);
  }
  if (pos < s.sink) return;
  float y[4];
  load4(k, dtype, sh * kDim + 4 * lane, y);
  const int64_t row = sh * t.rcap + (pos - s.sink);
  encode_key_warp(y, lane, sm, rp, t.ids + row * kSub, t.rec + row * kRecBytes);
}

// Inverted bucket index of one chunk of one (sequence, KV head): for every
// subspace b, the chunk-local key numbers grouped by bucket id (a counting
// sort; the order inside a bucket is not significant), with offsets
// off[b][id] .. off[b][id + 1].  One block of 1024 threads per chunk.
__global__ void __launch_bounds__(1024) k_build_index(int64_t N, int chunk0, Shape s, Tables t) {
  __shared__ uint32_t cnt[kSub][kCentroids];
  const int c = chunk0 + blockIdx.x;
  const int64_t sh = blockIdx.y;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, N - base);
  const uint4* ids = reinterpret_cast<const uint4*>(t.ids + (sh * t.rcap + base) * kSub);
  uint32_t* off = t.off + ((sh * t.nchunk + c) * kSub) * kOffStride;
  uint16_t* ent = t.ent + ((sh * t.nchunk + c) * kSub) * (int64_t)kChunk;

  for (int i = threadIdx.x; i < kSub * kCentroids; i += blockDim.x) (&cnt[0][0])[i] = 0;
  __syncthreads();
  for (int key = threadIdx.x; key < len; key += blockDim.x) {
    const uint4 r = ids[key];
    const uint32_t wds[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int b = 0; b < kSub; ++b) atomicAdd(&cnt[b][(wds[b >> 2] >> (8 * (b & 3))) & 0xffu], 1u);
  }
  __syncthreads();
  // exclusive scan per subspace: warp b, 8 bins per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < kSub) {
    const int b = warp;
    uint32_t vals[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      vals[i] = cnt[b][8 * lane + i];
      sum += vals[i];
    }
    uint32_t run = warp_incl_scan(sum, lane) - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      off[b * kOffStride + 8 * lane + i] = run;
      cnt[b][8 * lane + i] = run;
      run += vals[i];
    }
    if (lane == 31) off[b * kOffStride + kCentroids] = run;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < len; key += blockDim.x) {
    const uint4 r = ids[key];
    const uint32_t wds[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int b = 0; b < kSub; ++b) {
      const uint32_t id = (wds[b >> 2] >> (8 * (b & 3))) & 0xffu;
      const uint32_t p = atomicAdd(&cnt[b][id], 1u);
      ent[(int64_t)b * kChunk + p] = (uint16_t)key;
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
  dim3 grid(chunk1 - chunk0, s.batch * s.hkv);
  k_build_index<<<grid, 1024, 0, st>>>(N, chunk0, s, t);
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
