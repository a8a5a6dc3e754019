// Device helpers shared by the ParisKV kernels: input loads, the in-warp
// fast Walsh-Hadamard transform and warp/block scans.
#pragma once

#include "paris_internal.cuh"

namespace paris {

constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Programmatic dependent launch.  pdl_wait(): wait until the preceding kernel
// of the stream has completed and its writes are visible (returns at once
// when the launch has no programmatic dependency).  pdl_trigger(): let the
// next kernel of the stream be scheduled; every kernel here triggers only
// after its own wait, so work a kernel does before its wait overlaps nothing
// but its immediate predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Phase trace: thread 0 of a chosen block stores the global nanosecond timer
// into trace[slot] (trace == nullptr: tracing off).
__device__ __forceinline__ void trace_mark(uint64_t* trace, int slot) {
  if (trace != nullptr && threadIdx.x == 0) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    trace[slot] = t;
  }
}

// Per-block trace: thread 0 of every block stores the timer into
// trace[kTraceSlots + ((kernel * kTraceBlocks + block) * 4 + phase)].
__device__ __forceinline__ void trace_block(uint64_t* trace, int kernel, int phase) {
  if (trace != nullptr && threadIdx.x == 0) {
    const int64_t blk = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
    if (blk < kTraceBlocks) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      trace[kTraceSlots + ((int64_t)kernel * kTraceBlocks + blk) * 4 + phase] = t;
    }
  }
}

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

__device__ __forceinline__ uint32_t shfl_xor_key(uint32_t x, int j) { return __shfl_xor_sync(kFull, x, j); }
__device__ __forceinline__ unsigned long long shfl_xor_key(unsigned long long x, int j) {
  return __shfl_xor_sync(kFull, x, j);
}

// One merge level k of Batcher's bitonic network on an aligned 64-element
// chunk held by a warp, two elements per lane (a = element ea = c + lane,
// b = element ea + 32): the distances min(k/2, 32) .. 1, ascending where
// bit k of the element index is 0.
template <typename T>
__device__ __forceinline__ void warp_merge_level(T& a, T& b, int ea, int lane, int k) {
  if (k >= 64) {  // distance 32: the pair (a, b), one direction for both
    const T lo = a < b ? a : b, hi = a < b ? b : a;
    const bool asc = (ea & k) == 0;
    a = asc ? lo : hi;
    b = asc ? hi : lo;
  }
  const bool asc_a = (ea & k) == 0, asc_b = ((ea + 32) & k) == 0;
#pragma unroll
  for (int j = 16; j >= 1; j >>= 1) {
    if (j < k) {
      const bool lower = (lane & j) == 0;
      const T pa = shfl_xor_key(a, j), pb = shfl_xor_key(b, j);
      a = ((lower == asc_a) == (pa < a)) ? pa : a;  // the smaller of the pair where lower == ascending
      b = ((lower == asc_b) == (pb < b)) ? pb : b;
    }
  }
}

// Sort s[0, n) ascending in shared memory (Batcher's bitonic network); n a
// power of two >= 64, keys distinct or not, every thread of the block calls
// it (blockDim.x a multiple of 32).  A merge of level k compares elements j
// apart for j = k/2 .. 1, ascending where bit k of the lower index is 0.
// Distances j >= 64 go through shared memory, one barrier each; j <= 32 run
// inside one warp on aligned 64-element chunks (warp_merge_level).  Starts
// and ends with a barrier.
template <typename T>
__device__ void block_sort_pow2(T* s, int n) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  for (int c = warp * 64; c < n; c += nw * 64) {  // levels 2 .. 64 inside each chunk
    T a = s[c + lane], b = s[c + 32 + lane];
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1) warp_merge_level(a, b, c + lane, lane, k);
    s[c + lane] = a;
    s[c + 32 + lane] = b;
  }
  __syncthreads();
  for (int k = 128; k <= n; k <<= 1) {
    for (int j = k >> 1; j >= 64; j >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
        const int lo = 2 * i - (i & (j - 1)), hi = lo + j;
        const T x = s[lo], y = s[hi];
        if ((y < x) == ((lo & k) == 0)) {
          s[lo] = y;
          s[hi] = x;
        }
      }
      __syncthreads();
    }
    for (int c = warp * 64; c < n; c += nw * 64) {
      T a = s[c + lane], b = s[c + 32 + lane];
      warp_merge_level(a, b, c + lane, lane, k);
      s[c + lane] = a;
      s[c + 32 + lane] = b;
    }
    __syncthreads();
  }
}

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
// Bucket id of subspace b = lane / 2 against a table of 256 learned
// centroids (tab: [16][256][8] of the key's KV head): the centroid c with
// the largest fp32 score ((0 + z_0 c_0) + z_1 c_1) + ... + z_7 c_7, the
// lowest id among equal scores.  Lanes 2b (ids 0..127) and 2b + 1 (ids
// 128..255) each scan half the table; all lanes return the id.
__device__ __forceinline__ uint32_t table_id_warp(const float (&y)[4], int lane, const float* __restrict__ tab) {
  const bool odd = (lane & 1) != 0;
  float z[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float o = __shfl_xor_sync(kFull, y[i], 1);
    z[i] = odd ? o : y[i];
    z[4 + i] = odd ? y[i] : o;
  }
  const float* row = tab + ((lane >> 1) * kCentroids + (odd ? kCentroids / 2 : 0)) * kM;
  float best = -INFINITY;
  uint32_t bid = odd ? kCentroids / 2 : 0;
  for (int c = 0; c < kCentroids / 2; ++c) {
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(row + c * kM));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(row + c * kM + 4));
    float sc = __fmul_rn(z[0], c0.x);
    sc = __fadd_rn(sc, __fmul_rn(z[1], c0.y));
    sc = __fadd_rn(sc, __fmul_rn(z[2], c0.z));
    sc = __fadd_rn(sc, __fmul_rn(z[3], c0.w));
    sc = __fadd_rn(sc, __fmul_rn(z[4], c1.x));
    sc = __fadd_rn(sc, __fmul_rn(z[5], c1.y));
    sc = __fadd_rn(sc, __fmul_rn(z[6], c1.z));
    sc = __fadd_rn(sc, __fmul_rn(z[7], c1.w));
    if (sc > best) {  // strict: among equal scores the lower id stays
      best = sc;
      bid = (odd ? kCentroids / 2 : 0) + c;
    }
  }
  const float ob = __shfl_xor_sync(kFull, best, 1);
  const uint32_t oid = __shfl_xor_sync(kFull, bid, 1);
  // the even lane holds the lower ids: it wins ties
  if (odd ? ob >= best : ob > best) return oid;
  return bid;
}

__device__ __forceinline__ void encode_key_warp(float (&y)[4], int lane, const SignMask& sm,
                                                const RsqParams& rp, uint8_t* ids_row,
                                                uint8_t* rec_row, const float* tab = nullptr) {
  apply_signs(y, sm, lane);
  fwht128_warp(y, lane);
  const bool odd = (lane & 1) != 0;

  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) bits |= (y[i] < 0.f ? 1u : 0u) << i;
  const uint32_t obits = __shfl_xor_sync(kFull, bits, 1);
  const uint32_t id = tab ? table_id_warp(y, lane, tab) : odd ? (obits | (bits << 4)) : (bits | (obits << 4));

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


// Append one token of (sequence, KV head) `sh` (one warp): store its K/V as
// bf16 (Sink slot, or store row + Local/Buffer ring slot) and, past the Sink,
// encode its key at table row pos - S.
__device__ __forceinline__ void append_token_warp(const void* k, const void* v, int dtype, int64_t pos,
                                                  int64_t sh, int lane, const Shape& s, const KvStore& kv,
                                                  const Tables& t, const SignMask& sm, const RsqParams& rp,
                                                  const float* cent) {
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
  encode_key_warp(y, lane, sm, rp, t.ids + row * kSub, t.rec + row * kRecBytes,
                  cent ? cent + (sh % s.hkv) * kTabPerHead : nullptr);
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key); -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (x == 0.f) x = 0.f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

}  // namespace paris
