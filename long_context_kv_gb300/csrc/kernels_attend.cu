// Sparse decode attention of ParisKV over Sink U Local U Update Buffer U the
// retrieved top-k tokens, reading Retrieval-zone rows in place (HBM, or
// mapped pinned host memory through UVA).
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// attention over the top-k subset ("Problem definition"); system level,
// "Unified Virtual Addressing (UVA) offloading" and "Sliding-window update
// mechanism" (Sink and Local on the GPU, the history offloaded).
//
// Split-row flash decoding: block (split, sequence x query head) stages the
// K and V rows of its kAttnSplit rows (window rows first, then the retrieved
// rows) in shared memory with asynchronous 16-byte copies, all in flight at
// once, then computes softmax(q K^T / sqrt(d)) V for them and writes
// (max, sum, o); the last split of a query head to finish merges the splits
// (atomic counter after a memory fence, no waiting), issuing its loads of
// the splits' partial outputs in batches rather than one after another.  Decode has one query
// row per head, so the work is a gather plus matrix-vector products: CUDA
// cores, not tensor cores.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kAttnThreads = 128;
// A staged K row is 256 B with its 16-byte pieces permuted by row (piece c
// of row r at c ^ (r & 7)): every 32-byte sector lands whole in an aligned
// 32-byte slot, so each copy instruction is served as whole-sector requests
// (a row stride padded to 272 B splits the sectors of every other row, which
// doubles the requests and cut reads of host-resident rows to about 60 % of
// the link's rate), and the 16-byte reads of the scores meet no bank conflict.
__device__ __forceinline__ int kpiece(int row, int c) { return row * kDim + 8 * (c ^ (row & 7)); }
static_assert(kAttnThreads == kDim && 2 * kAttnSplit == kAttnThreads, "one thread per output dimension, two per row");

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__global__ void __launch_bounds__(kAttnThreads) k_attend(const void* __restrict__ q, int dtype, AttendArgs a,
                                                        int64_t nsink, int64_t nwin, int nsplit, float qscale) {
  // The dynamic region follows the static arrays below; 128-byte alignment
  // keeps every staged row's 32-byte sectors on sector boundaries (at the
  // default 16-byte alignment it started 16 bytes off one, and every row read
  // from host memory cost twice its sectors).
  extern __shared__ __align__(128) uint16_t smem[];
  uint16_t* ks = smem;                      // [kAttnSplit][kDim], pieces permuted (kpiece)
  uint16_t* vs = smem + kAttnSplit * kDim;  // [kAttnSplit][kDim]
  __shared__ float qf[kDim];
  __shared__ float p[kAttnSplit];
  __shared__ float fs[kMaxSplits];
  __shared__ float red[8];
  __shared__ int s_last;
  __shared__ int64_t rsrc[kAttnSplit];  // element offset of each row (window rows flagged), -1: no row
  const int split = blockIdx.x;
  const int sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = tid >> 1, half = tid & 1;  // two threads per row, half a row each
  const int64_t R = nwin + a.k_eff;
  const int ring = a.s.local + a.s.ubuf;
  uint64_t* tr = (split == 0 && sq == 0) ? a.trace : nullptr;
  trace_mark(tr, kTrAttend0);
  trace_block(a.trace, kTkAttend, 0);

  // Everything is read after the wait: the preceding kernel may be a decode
  // step that writes its own token into a window slot, or the retrieval that
  // writes the top-k.  Thread r < kAttnSplit finds row r of the split; then
  // 16 consecutive threads copy one row's 16-byte pieces, so every copy
  // instruction covers whole rows (which keeps reads of host-resident rows
  // in whole sectors).
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkAttend, 1);
  constexpr int64_t kWin = int64_t(1) << 62;
  if (tid < kAttnSplit) {
    const int64_t r = (int64_t)split * kAttnSplit + tid;
    int64_t src = -1;
    if (r < nwin) {
      int64_t slot = r;
      if (r >= nsink) {
        const int64_t pos = a.s.sink + a.N + (r - nsink);
        slot = a.s.sink + (pos - a.s.sink) % ring;
      }
      src = kWin | ((sh * a.kv.win + slot) * kDim);
    } else if (r < R) {
      const int64_t pos = __ldcg(a.topk_idx + (int64_t)sq * a.k + (r - nwin));
      if (pos >= a.s.sink && pos < a.s.sink + a.N) src = (sh * a.kv.rcap + (pos - a.s.sink)) * kDim;
      else if (pos >= 0) atomicOr(a.status, kStatusBadIndex);
    }
    rsrc[tid] = src;
  }
  qf[tid] = load1(q, dtype, (int64_t)sq * kDim + tid) * qscale;
  __syncthreads();
#pragma unroll 4
  for (int i = tid; i < kAttnSplit * 16; i += kAttnThreads) {
    const int rw = i >> 4, pc = i & 15;
    const int64_t src = rsrc[rw];
    if (src >= 0) {
      const bool win = (src & kWin) != 0;
      const int64_t e = (src & (kWin - 1)) + 8 * pc;
      cp_async16(ks + kpiece(rw, pc), (win ? a.kv.win_k : a.kv.st_k) + e);
      cp_async16(vs + rw * kDim + 8 * pc, (win ? a.kv.win_v : a.kv.st_v) + e);
    } else {
      // no row: zeros, so the weighted V sum below reads finite values
      *reinterpret_cast<uint4*>(vs + rw * kDim + 8 * pc) = make_uint4(0, 0, 0, 0);
    }
  }
  const bool has_row = rsrc[row] >= 0;
  const int c0 = half * (kDim / 2);
  cp_async_wait_all();
  __syncthreads();
  trace_mark(tr, kTrAttend1);

  // score of the row (log2 domain): each thread half the dot product; the
  // second half takes its pieces starting four pieces on, so the two
  // threads of a row read different banks
  float s = -FLT_MAX;
  {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kDim / 16; ++j) {
      const int c = c0 / 8 + (j ^ (4 * half));
      const uint4 kv8 = *reinterpret_cast<const uint4*>(ks + kpiece(row, c));
      const uint32_t w[4] = {kv8.x, kv8.y, kv8.z, kv8.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc += qf[8 * c + 2 * i] * bf16_bits_to_float(w[i] & 0xffffu);
        acc += qf[8 * c + 2 * i + 1] * bf16_bits_to_float(w[i] >> 16);
      }
    }
    acc += __shfl_xor_sync(kFull, acc, 1);
    if (has_row) s = acc;
  }
  float mx = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float pr = has_row ? exp2f(s - M) : 0.f;
  if (half == 0) p[row] = pr;
  float l = half == 0 ? pr : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
  if (lane == 0) red[4 + warp] = l;
  __syncthreads();
  const float L = red[4] + red[5] + red[6] + red[7];
  // o[d] for d = tid over the split's rows
  const int nrows = (int)min64(kAttnSplit, R - (int64_t)split * kAttnSplit);
  float acc = 0.f;
  for (int rr = 0; rr < nrows; ++rr) acc += p[rr] * bf16_bits_to_float(vs[rr * kDim + tid]);
  float* part = a.part + (int64_t)sq * a.nsplit_max * kPartStride;
  float* out = part + (int64_t)split * kPartStride;
  out[4 + tid] = acc;
  if (tid == 0) {
    out[0] = M;
    out[1] = L;
  }

  trace_mark(tr, kTrAttend2);
  trace_block(a.trace, kTkAttend, 2);
  // the last split of the query head merges all splits
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counter[sq], 1u) == (uint32_t)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (sq == 0) trace_mark(a.trace, kTrAttend3);
  const int d = tid;
  // every thread's first batch of o loads goes out together with warp 0's
  // loads of the splits' (max, sum)
  constexpr int kBatch = 32;
  float oo[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) oo[u] = u < nsplit ? __ldcg(part + (int64_t)u * kPartStride + 4 + d) : 0.f;
  if (warp == 0) {
    float Mx = -FLT_MAX;
    for (int s0 = lane; s0 < nsplit; s0 += 32) {
      const float mm = __ldcg(part + (int64_t)s0 * kPartStride), ll = __ldcg(part + (int64_t)s0 * kPartStride + 1);
      if (ll > 0.f) Mx = fmaxf(Mx, mm);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(kFull, Mx, o));
    float Lt = 0.f;
    for (int s0 = lane; s0 < nsplit; s0 += 32) {
      const float mm = __ldcg(part + (int64_t)s0 * kPartStride), ll = __ldcg(part + (int64_t)s0 * kPartStride + 1);
      const float f = ll > 0.f ? exp2f(mm - Mx) : 0.f;
      fs[s0] = f;
      Lt += ll * f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lt += __shfl_xor_sync(kFull, Lt, o);
    if (lane == 0) red[0] = Lt;
  }
  __syncthreads();
  float ot = 0.f;
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    if (u < nsplit) ot += oo[u] * fs[u];
  for (int s0 = kBatch; s0 < nsplit; s0 += kBatch) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      oo[u] = s0 + u < nsplit ? __ldcg(part + (int64_t)(s0 + u) * kPartStride + 4 + d) : 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (s0 + u < nsplit) ot += oo[u] * fs[s0 + u];
  }
  const float Lt = red[0];
  a.out[(int64_t)sq * kDim + d] = __float2bfloat16_rn(Lt > 0.f ? ot / Lt : 0.f);
  if (tid == 0) a.counter[sq] = 0;
  if (sq == 0) trace_mark(a.trace, kTrAttend4);
  trace_block(a.trace, kTkAttend, 3);
}

constexpr size_t kAttendSmem = (size_t)kAttnSplit * 2 * kDim * sizeof(uint16_t);

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
  {
    const cudaError_t e = set_smem_limit((const void*)k_attend, (int)kAttendSmem, kSmemAttend);
    if (e != cudaSuccess) return e;
  }
  const int64_t nsink = min64(a.s.sink, a.T);
  const int64_t nwin = nsink + a.n_local_buf;
  const float qscale = 1.4426950408889634f / sqrtf((float)kDim);
  return launch_pdl(k_attend, dim3(nsplit, a.s.batch * a.s.hq), dim3(kAttnThreads), kAttendSmem, st, q, dtype, a,
                    nsink, nwin, nsplit, qscale);
}

}  // namespace paris
