// The decode-step path of ParisKV in one kernel: query preparation,
// collision votes, candidate selection, RSQ-IP rerank, top-k and (for a
// decode step) the sparse attention, for every (sequence, query head).
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// Methodology 2, "Coarse candidate generation (collision-based)", "Candidate
// reranking (RSQ-IP)" and "Estimation"; the attention over Sink, Local, the
// Update Buffer and the retrieved tokens ("Problem definition",
// "Sliding-window update mechanism").
//
// One thread-block cluster of CS <= 8 blocks per (sequence, query head);
// block r of the cluster owns a contiguous range of index chunks of the
// Retrieval zone, so block order is position order.  The steps that need
// the whole query head exchange small tables through distributed shared
// memory between cluster barriers (every block reaches every barrier):
//   1. each block: q~, ||q|| and the hot centroids (redundantly), the votes
//      of its chunks and their histogram;
//   2. barrier; every block sums the cluster's histograms, finds the vote
//      threshold and writes its candidates (positions ascending) at their
//      place in the query head's candidate list;
//   3. each block: estimates of its candidates;
//   4. top-k: four 8-bit radix passes over the estimates' order keys, one
//      barrier each; every block derives the same k-th key and, from every
//      block's counts, its own output offset;
//   5. barrier; the rows (window + top-k) are split evenly over the blocks;
//      each block stages its rows through a four-stage asynchronous-copy
//      pipeline with an online softmax; barrier; block 0 merges.
// A decode token appended in the same step is read from the caller's k/v
// where the attention needs it, and written to the cache by one block at
// the very end (nothing in this launch reads the slots it writes).
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kClusterMax = 8;
constexpr int kListCap = 2048;      // candidates per block kept in shared memory; the rest re-read from global
constexpr int kTile = 32;           // attention rows per pipeline stage
constexpr int kStages = 4;
constexpr int kKStride = kDim + 8;  // bf16 per staged row: 272 B keeps 16-byte reads conflict-free
constexpr int kSelCap = 16384;      // candidates whose keys block 0 stages for the top-k
constexpr int kSelBins = 2048;      // 11-bit radix digits
static_assert(kWarps == kSub, "warp b prepares subspace b");
static_assert(kTile * 16 == kThreads, "16 threads per staged row");

// byte offsets inside the phase-shared region
constexpr int kUKeys = 0;                                   // u32 [kSelCap]: top-k order keys (block 0)
constexpr int kUVotes = 0;                                  // u8 [kChunk]: votes of the block's last chunk
constexpr int kUOffs = kUVotes + kChunk;                    // u32 [kSub][kOffStride]
constexpr int kUSelHist = kUKeys + kSelCap * 4;             // u32 [kSelBins]
constexpr int kUListPos = kUSelHist + kSelBins * 4;         // i32 [kListCap]: the block's candidate slice
constexpr int kUListEst = kUListPos + kListCap * 4;         // f32 [kListCap]: its estimates
constexpr int kUVoteEnd = kUListEst + kListCap * 4;
constexpr int kUStageK = 0;                                 // bf16 [kStages][kTile][kKStride]
constexpr int kUStageV = kStages * kTile * kKStride * 2;
constexpr int kUAttnEnd = 2 * kStages * kTile * kKStride * 2;
constexpr int kUBytes = kUVoteEnd > kUAttnEnd ? kUVoteEnd : kUAttnEnd;
static_assert(kUOffs + kSub * kOffStride * 4 <= kUSelHist, "vote tables inside the key area");
static_assert(kUAttnEnd <= kUListPos, "attention stages below the candidate slice");

__host__ __device__ constexpr int hot_bytes(int nhot) { return (16 * nhot + 4 + 15) & ~15; }

struct DecodeArgs {
  Shape s;
  Tables t;
  KvStore kv;
  SignMask sm;
  RsqParams rp;
  int rho, flat, nbins, cpb, nchunk_active;
  int64_t N, C, k, k_eff, cmax;
  int64_t nsink, nwin;  // attention window rows
  const void* q;
  int qdtype;
  float qscale;
  const void* k_new;    // the step's own token (new_pos < 0: none)
  const void* v_new;
  int kvdtype;
  int64_t new_pos;
  float* qt;
  float* qnorm;
  uint32_t* hot;
  uint8_t* votes;
  int32_t* cand_idx;
  float* cand_est;
  uint32_t* status;
  uint64_t* trace;
  int32_t* topk_idx;
  float* topk_score;
  __nv_bfloat16* out;   // nullptr: no attention
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Cluster barrier: every thread of every block of the cluster arrives; the
// writes before it (shared and global) are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// 32-bit load from the same shared-memory variable of block `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_u32(const void* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// Estimate of one candidate from its 128-byte record, float32 in this order:
//   acc = 0; for b: dot = 0; for j: dot = dot + v_{b,j} q~_{b,j};
//   acc = acc + w_b dot;   est = ||q|| acc,
// v_{b,j} q~_{b,j} read from the table of the 16 possible products of each
// coordinate (sign bit x 8 levels), each rounded once.
__device__ __forceinline__ float estimate(const uint4 (&x)[8], const float* tq, float qn) {
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < kSub; ++b) {
    const uint4 cq = x[b >> 2];
    const uint32_t cw = (b & 3) == 0 ? cq.x : (b & 3) == 1 ? cq.y : (b & 3) == 2 ? cq.z : cq.w;
    const uint4 wq = x[4 + (b >> 2)];
    const float w = __uint_as_float((b & 3) == 0 ? wq.x : (b & 3) == 1 ? wq.y : (b & 3) == 2 ? wq.z : wq.w);
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kM; ++j) dot = __fadd_rn(dot, tq[(b * kM + j) * 16 + ((cw >> (4 * j)) & 15u)]);
    acc = __fadd_rn(acc, __fmul_rn(w, dot));
  }
  return __fmul_rn(qn, acc);
}

// Per byte of x: 0x80 where the byte equals the byte of c4 / exceeds it
// (unsigned), 0 elsewhere.
__device__ __forceinline__ uint32_t bytes_eq(uint32_t x, uint32_t c4) {
  const uint32_t y = x ^ c4;
  const uint32_t t = ((y & 0x7f7f7f7fu) + 0x7f7f7f7fu) | y;  // high bit set in every nonzero byte
  return ~t & 0x80808080u;
}
__device__ __forceinline__ uint32_t bytes_gt(uint32_t x, uint32_t c4) {
  // per byte (x | 0x80) - (c & 0x7f) never borrows; its high bit is [x_low7 >= c_low7]
  const uint32_t d = (x | 0x80808080u) - (c4 & 0x7f7f7f7fu);
  const uint32_t ge = ((x & ~c4) | (~(x ^ c4) & d)) & 0x80808080u;
  return ge & ~bytes_eq(x, c4);
}

// Block 0 of a query head's cluster: the k_eff-th largest order key over all
// C estimates (radix select, 11-bit digits below the bits all keys share),
// then, for every block's slice [C r / cs, C (r + 1) / cs), where its
// selected entries start in the output and how many of its keys equal to
// the k-th key it keeps (those equal keys go to the lowest positions, which
// are the lowest candidate indices).  Writes sel[r] = (offset, kept) and
// sel[kClusterMax][0] = the k-th key.  All threads of the block call it.
__device__ __noinline__ void select_kth(const int64_t C, const int64_t k_eff, const float* est, int cs,
                                        uint8_t* U, uint32_t* tmp, uint32_t (*sel)[2]) {
  __shared__ uint32_t s_digit, s_skip;
  __shared__ uint32_t cnt_gt[kClusterMax], cnt_eq[kClusterMax];
  __shared__ int64_t bounds[kClusterMax + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* keys = reinterpret_cast<uint32_t*>(U + kUKeys);
  uint32_t* hist = reinterpret_cast<uint32_t*>(U + kUSelHist);
  const bool staged = C <= kSelCap;
  auto key_at = [&](int64_t i) { return staged ? keys[i] : order_key(__ldcg(est + i)); };
  if (tid < kClusterMax) {
    cnt_gt[tid] = 0;
    cnt_eq[tid] = 0;
  }
  if (tid <= cs) bounds[tid] = C * tid / cs;
  // keys (8 loads in flight per thread), and the bits every key shares
  uint32_t kand = 0xffffffffu, kor = 0u;
  for (int64_t i0 = tid; i0 < C; i0 += 8 * kThreads) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = i0 + u * kThreads < C ? __ldcg(est + i0 + u * kThreads) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u * kThreads;
      if (i < C) {
        const uint32_t k = order_key(v[u]);
        if (staged) keys[i] = k;
        kand &= k;
        kor |= k;
      }
    }
  }
  kand = __reduce_and_sync(kFull, kand);
  kor = __reduce_or_sync(kFull, kor);
  if (lane == 0) {
    tmp[warp] = kand;
    tmp[16 + warp] = kor;
  }
  __syncthreads();
  kand = 0xffffffffu;
  kor = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    kand &= tmp[w];
    kor |= tmp[16 + w];
  }
  __syncthreads();
  const uint32_t diff = kand ^ kor;
  uint32_t prefix = kand, remaining = (uint32_t)k_eff;
  if (diff != 0) {
    const int top = 31 - __clz(diff);  // highest bit where keys differ
    uint32_t mask = top == 31 ? 0u : (0xffffffffu << (top + 1));
    prefix = kand & mask;
    for (int hi = top; hi >= 0;) {
      const int nb = min(11, hi + 1), lo = hi + 1 - nb;
      const uint32_t dmask = (1u << nb) - 1u;
      for (int i = tid; i < kSelBins; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < C; i += kThreads) {
        const uint32_t k = key_at(i);
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> lo) & dmask], 1u);
      }
      __syncthreads();
      // thread t owns digits kSelBins-1-4t .. kSelBins-4-4t, scanned from the top
      uint32_t c4[4], sum4 = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c4[u] = hist[kSelBins - 1 - 4 * tid - u];
        sum4 += c4[u];
      }
      uint32_t tot;
      const uint32_t exc = block_excl_scan(sum4, tmp, &tot);
      if (exc < remaining && exc + sum4 >= remaining) {
        uint32_t run = exc;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (run + c4[u] >= remaining) {
            s_digit = (uint32_t)(kSelBins - 1 - 4 * tid - u);
            s_skip = run;
            break;
          }
          run += c4[u];
        }
      }
      __syncthreads();
      prefix |= s_digit << lo;
      mask |= dmask << lo;
      remaining -= s_skip;
      hi = lo - 1;
      __syncthreads();
    }
  }
  // per slice: keys above / equal to the k-th key
  for (int64_t i0 = 0; i0 < C; i0 += kThreads) {
    const int64_t i = i0 + tid;
    int owner = 0;
    uint32_t g = 0, e = 0;
    if (i < C) {
#pragma unroll
      for (int q = 1; q < kClusterMax; ++q) owner += (q < cs && i >= bounds[q]) ? 1 : 0;
      const uint32_t k = key_at(i);
      g = k > prefix ? 1u : 0u;
      e = k == prefix ? 1u : 0u;
    }
    if (__all_sync(kFull, owner == __shfl_sync(kFull, owner, 0))) {
      const uint32_t gs = __reduce_add_sync(kFull, g), es = __reduce_add_sync(kFull, e);
      if (lane == 0) {
        if (gs) atomicAdd(&cnt_gt[owner], gs);
        if (es) atomicAdd(&cnt_eq[owner], es);
      }
    } else {
      if (g) atomicAdd(&cnt_gt[owner], 1u);
      if (e) atomicAdd(&cnt_eq[owner], 1u);
    }
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t rem = remaining, off = 0;
    for (int q = 0; q < cs; ++q) {
      const uint32_t et = min(cnt_eq[q], rem);
      rem -= et;
      sel[q][0] = off;
      sel[q][1] = et;
      off += cnt_gt[q] + et;
    }
    sel[kClusterMax][0] = prefix;
  }
}

__global__ void __launch_bounds__(kThreads, 2) k_decode(DecodeArgs a) {
  __shared__ float qs[kDim], zs[kDim], qts[kDim];
  __shared__ float tq[kDim * 16];
  __shared__ uint32_t hist[kMaxBins];                  // read by the cluster
  __shared__ __align__(16) float part[kPartStride];    // read by block 0
  __shared__ uint32_t tot[kMaxBins];
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t red[64];
  __shared__ uint32_t sel_info[kClusterMax + 1][2];      // block 0: per block (output offset, equal keys kept); k-th key
  __shared__ uint8_t rvalid[kStages][kTile];
  __shared__ float s_qn;
  __shared__ int s_T;
  __shared__ int64_t s_quota;
  extern __shared__ __align__(16) uint8_t dyn[];

  const int nhot = kSub * a.rho;
  uint32_t* hv = reinterpret_cast<uint32_t*>(dyn);  // hot entries: id | weight << 16 | subspace << 24
  uint32_t* hbeg = hv + nhot;
  uint32_t* hwt = hbeg + nhot;
  uint32_t* hpre = hwt + nhot;                       // nhot + 1
  uint8_t* U = dyn + hot_bytes(nhot);
  uint8_t* votes = U + kUVotes;
  uint32_t* offs = reinterpret_cast<uint32_t*>(U + kUOffs);
  int32_t* lpos = reinterpret_cast<int32_t*>(U + kUListPos);
  float* lest = reinterpret_cast<float*>(U + kUListEst);
  uint16_t* stK = reinterpret_cast<uint16_t*>(U + kUStageK);
  uint16_t* stV = reinterpret_cast<uint16_t*>(U + kUStageV);

  const int r = blockIdx.x, cs = gridDim.x, sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c_lo = min(r * a.cpb, a.nchunk_active), c_hi = min(c_lo + a.cpb, a.nchunk_active);
  uint64_t* tr = (r == 0 && sq == 0) ? a.trace : nullptr;
  trace_block(a.trace, kTkDecode0, 0);

  // ---- before the wait: cleared counters ---------------------------------
  for (int i = tid; i < kChunk / 16; i += kThreads) reinterpret_cast<uint4*>(votes)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kMaxBins; i += kThreads) hist[i] = 0;
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkDecode0, 1);
  trace_mark(tr, kTrDecode0);

  auto prefetch_offsets = [&](int c) {
    const uint32_t* og = a.t.off + ((sh * a.t.nchunk + c) * kSub) * kOffStride;
    for (int i = tid; i < kSub * kOffStride / 4; i += kThreads) cp_async16(offs + 4 * i, og + 4 * i);
  };
  if (c_lo < c_hi) prefetch_offsets(c_lo);

  // ---- 1. query preparation ------------------------------------------------
  //   ||q|| = sqrt(sequential sum over the d inputs of q_j q_j);
  //   z = fwht(D q); ||z|| likewise; q~ = z / ||z|| (0 if ||z|| = 0);
  //   score of centroid c in subspace b = sequential sum over j of +-z_{b,j}
  //   (minus where bit j of c is set); the top rho per subspace by
  //   (score desc, id asc) get weight rho - r (rank r) or 1 (flat).
  if (warp == 0) {
    float y[4];
    load4(a.q, a.qdtype, (int64_t)sq * kDim + 4 * lane, y);
#pragma unroll
    for (int i = 0; i < 4; ++i) qs[4 * lane + i] = y[i];
    apply_signs(y, a.sm, lane);
    fwht128_warp(y, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) zs[4 * lane + i] = y[i];
  }
  __syncthreads();
  if (warp == 0) {
    // the two sequential norm chains side by side in lanes 0 (q) and 1 (z)
    float acc = 0.f;
    if (lane < 2) {
      const float* src = lane == 0 ? qs : zs;
#pragma unroll
      for (int j0 = 0; j0 < kDim; j0 += 32) {
        float sqv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sqv[j] = __fmul_rn(src[j0 + j], src[j0 + j]);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc = __fadd_rn(acc, sqv[j]);
      }
    }
    const float nrm = __fsqrt_rn(acc);
    const float nq = __shfl_sync(kFull, nrm, 0), nz = __shfl_sync(kFull, nrm, 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * lane + i;
      const float v = nz > 0.f ? __fdiv_rn(zs[j], nz) : 0.f;
      qts[j] = v;
      if (r == 0) a.qt[(int64_t)sq * kDim + j] = v;
    }
    if (lane == 0) {
      s_qn = nq;
      if (r == 0) a.qnorm[sq] = nq;
    }
  }
  {
    const int b = warp;
    // the lane's centroids are lane + 32 i: bits 0-4 of the id are the lane's,
    // so the first five terms of the sequential sum are shared, then the
    // sums branch on bits 5, 6, 7 (the same additions in the same order)
    float zz[kM];
#pragma unroll
    for (int j = 0; j < kM; ++j) zz[j] = zs[b * kM + j];
    float acc5 = 0.f;
#pragma unroll
    for (int j = 0; j < 5; ++j) acc5 = __fadd_rn(acc5, ((lane >> j) & 1) ? -zz[j] : zz[j]);
    float a6[2], a7[4], a8[8];
#pragma unroll
    for (int t = 0; t < 2; ++t) a6[t] = __fadd_rn(acc5, (t & 1) ? -zz[5] : zz[5]);
#pragma unroll
    for (int t = 0; t < 4; ++t) a7[t] = __fadd_rn(a6[t & 1], (t & 2) ? -zz[6] : zz[6]);
#pragma unroll
    for (int t = 0; t < 8; ++t) a8[t] = __fadd_rn(a7[t & 3], (t & 4) ? -zz[7] : zz[7]);
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = order_key(a8[i]);  // never 0 for a finite score
    for (int rr = 0; rr < a.rho; ++rr) {
      uint32_t bk = 0;
      int bi = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (key[i] > bk) {  // strict: among equal keys the lowest id of the lane stays
          bk = key[i];
          bi = i;
        }
      const uint32_t wmax = __reduce_max_sync(kFull, bk);
      const uint32_t bid = __reduce_min_sync(kFull, bk == wmax && bk != 0 ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
      if ((int)(bid & 31) == lane) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i == (int)(bid >> 5)) key[i] = 0;
      }
      if (lane == 0) {
        const uint32_t e = bid | ((a.flat ? 1u : (uint32_t)(a.rho - rr)) << 16);
        hv[b * a.rho + rr] = e | ((uint32_t)b << 24);  // the subspace rides along in shared memory
        if (r == 0) a.hot[(int64_t)sq * nhot + b * a.rho + rr] = e;
      }
    }
  }
  __syncthreads();
  {
    // products of each coordinate of q~ with the 16 signed levels
#pragma unroll
    for (int u = 0; u < kDim * 16 / kThreads; ++u) {
      const int e = tid * (kDim * 16 / kThreads) + u;
      const int coord = e >> 4, nib = e & 15;
      const float l = a.rp.lev[nib & 7];
      tq[e] = __fmul_rn((nib & 8) ? -l : l, qts[coord]);
    }
  }
  trace_block(a.trace, kTkDecode0, 2);

  // ---- 1b. collision votes of the block's chunks ---------------------------
  // Each key of a chunk sits in exactly one bucket per subspace, so walking
  // the lists of the hot buckets and adding their weights gives every key
  // sum_b weight_b(id_{i,b}) (one byte per key, at most 255).
  uint32_t nz_mine = 0;
  int64_t own_len = 0;
  for (int c = c_lo; c < c_hi; ++c) {
    const int64_t base = (int64_t)c * kChunk;
    const int len = (int)min64(kChunk, a.N - base);
    own_len += len;
    cp_async_wait_all();
    __syncthreads();  // the chunk's offsets (and, first time, the hot list) are in place
    {
      constexpr int kHotPer = (kSub * kCentroids + kThreads - 1) / kThreads;
      const int per = (nhot + kThreads - 1) / kThreads;
      uint32_t lens[kHotPer];
      uint32_t my = 0;
#pragma unroll
      for (int i = 0; i < kHotPer; ++i) {
        const int e = tid * per + i;
        lens[i] = 0;
        if (i < per && e < nhot) {
          const uint32_t h = hv[e];
          const uint32_t b = h >> 24, id = h & 0xffu;
          const uint32_t beg = offs[b * kOffStride + id];
          lens[i] = offs[b * kOffStride + id + 1] - beg;
          hbeg[e] = b * kChunk + beg;
          hwt[e] = (h >> 16) & 0xffu;
        }
        my += lens[i];
      }
      uint32_t total;
      uint32_t run = block_excl_scan(my, tmp, &total);
#pragma unroll
      for (int i = 0; i < kHotPer; ++i) {
        const int e = tid * per + i;
        if (i < per && e < nhot) hpre[e] = run;
        run += lens[i];
      }
      if (tid == 0) hpre[nhot] = total;
    }
    __syncthreads();
    if (c == c_lo) trace_mark(tr, kTrDecodeFine + 0);
    if (c + 1 < c_hi) prefetch_offsets(c + 1);  // the offsets are not read again for this chunk
    const uint32_t total = hpre[nhot];
    const uint16_t* ent = a.t.ent + ((sh * a.t.nchunk + c) * kSub) * (int64_t)kChunk;
    // thread t takes kWalk consecutive list entries: one search, then linear
    // steps; all kWalk loads in flight together
    constexpr int kWalk = 8;
    for (uint32_t f0 = kWalk * tid; f0 < total; f0 += kWalk * kThreads) {
      int e = 0, hi = nhot - 1;  // last e with hpre[e] <= f0 (a non-empty list)
      while (e < hi) {
        const int mid = (e + hi + 1) >> 1;
        if (hpre[mid] <= f0) e = mid; else hi = mid - 1;
      }
      uint32_t key[kWalk], wt[kWalk];
#pragma unroll
      for (int u = 0; u < kWalk; ++u) {
        const uint32_t f = f0 + u;
        wt[u] = 0;
        key[u] = 0;
        if (f < total) {
          while (hpre[e + 1] <= f) ++e;
          key[u] = __ldg(ent + hbeg[e] + (f - hpre[e]));
          wt[u] = hwt[e];
        }
      }
#pragma unroll
      for (int u = 0; u < kWalk; ++u)
        if (wt[u]) atomicAdd(reinterpret_cast<uint32_t*>(votes) + (key[u] >> 2), wt[u] << ((key[u] & 3) * 8));
    }
    __syncthreads();
    if (c == c_lo) trace_mark(tr, kTrDecodeFine + 1);
    // histogram of the chunk's votes; votes out (and cleared for the next chunk)
    uint8_t* vout = a.votes + (int64_t)sq * a.t.nchunk * kChunk + base;
    const bool last = c + 1 == c_hi;
    uint32_t small = 0;
    for (int i = tid; i < kChunk / 16; i += kThreads) {
      uint4* vp = reinterpret_cast<uint4*>(votes) + i;
      const uint4 w4 = *vp;
      reinterpret_cast<uint4*>(vout)[i] = w4;
      if (!last) *vp = make_uint4(0, 0, 0, 0);
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint32_t v = (ws[k >> 2] >> (8 * (k & 3))) & 0xffu;
        const bool in = v != 0 && 16 * i + k < len;
        if (in && v <= 4) small += 1u << (8 * (v - 1));  // per-thread counts <= 32 fit a byte
        else if (in) atomicAdd(&hist[v], 1u);
        nz_mine += in ? 1u : 0u;
      }
    }
#pragma unroll
    for (int v = 1; v <= 4; ++v) {
      const uint32_t cnt = __reduce_add_sync(kFull, (small >> (8 * (v - 1))) & 0xffu);
      if (lane == 0 && cnt) atomicAdd(&hist[v], cnt);
    }
  }
  {
    uint32_t nz_all;
    block_excl_scan(nz_mine, tmp, &nz_all);
    if (tid == 0) hist[0] = (uint32_t)own_len - nz_all;
  }
  trace_block(a.trace, kTkDecode0, 3);
  trace_mark(tr, kTrDecode1);

  // ---- 2. candidates --------------------------------------------------------
  // The candidates are the first C keys by (votes desc, index asc): with T
  // the largest vote value whose suffix count reaches C, every key above T
  // and the lowest-index keys equal to T, up to C.
  cluster_sync();
  uint32_t bef = 0;
  if (tid < kMaxBins) {
    uint32_t v[kClusterMax];
#pragma unroll
    for (int q = 0; q < kClusterMax; ++q) v[q] = q < cs ? dsmem_u32(hist + tid, q) : 0u;
    uint32_t all = 0;
#pragma unroll
    for (int q = 0; q < kClusterMax; ++q) {
      all += v[q];
      bef += q < r ? v[q] : 0u;
    }
    tot[tid] = all;
  }
  __syncthreads();
  if (warp == 0) {
    // suffix sums from the top vote value down: lane l owns values 255-8l .. 248-8l
    uint32_t sum8 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum8 += tot[255 - 8 * lane - i];
    const uint32_t inc = warp_incl_scan(sum8, lane);
    const uint32_t exc = inc - sum8;
    const uint32_t C = (uint32_t)a.C;
    const int owner = __ffs(__ballot_sync(kFull, exc < C && inc >= C)) - 1;
    if (lane == (owner < 0 ? 0 : owner)) {
      uint32_t run = exc;
      int T = 255 - 8 * lane;
      for (int i = 0; i < 8; ++i) {
        const int s = 255 - 8 * lane - i;
        if (run + tot[s] >= C) {
          T = s;
          break;
        }
        run += tot[s];
      }
      s_T = owner < 0 ? 0 : T;
      s_quota = (int64_t)a.C - (owner < 0 ? 0 : run);
    }
  }
  __syncthreads();
  const int T = s_T;
  const int64_t quota = s_quota;
  int64_t sel_before, eq_allow;
  {
    uint32_t gtb = (tid < kMaxBins && tid > T) ? bef : 0u;
    uint32_t eqb = tid == T ? bef : 0u;
    gtb = __reduce_add_sync(kFull, gtb);
    eqb = __reduce_add_sync(kFull, eqb);
    if (lane == 0) {
      red[warp] = gtb;
      red[32 + warp] = eqb;
    }
    __syncthreads();
    gtb = 0;
    eqb = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      gtb += red[w];
      eqb += red[32 + w];
    }
    sel_before = gtb + min64(eqb, quota);
    eq_allow = max64(0, quota - (int64_t)eqb);
  }
  trace_mark(tr, kTrDecode2);

  // ordered compaction: thread t owns keys [32t, 32t + 32) of each chunk,
  // compared four at a time (bytes of a word)
  const int64_t cq = (int64_t)sq * a.cmax;
  {
    int64_t nsel = 0;
    const uint32_t T4 = (uint32_t)T * 0x01010101u;
    for (int c = c_lo; c < c_hi; ++c) {
      const int64_t base = (int64_t)c * kChunk;
      const int len = (int)min64(kChunk, a.N - base);
      constexpr int kPer = kChunk / kThreads;
      const int k0 = tid * kPer;
      uint32_t vw[kPer / 4];
      if (c + 1 == c_hi) {
        const uint4* vin = reinterpret_cast<const uint4*>(votes + k0);
#pragma unroll
        for (int i = 0; i < kPer / 16; ++i) {
          const uint4 x = vin[i];
          vw[4 * i] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
        }
      } else {
        const uint4* vin = reinterpret_cast<const uint4*>(a.votes + (int64_t)sq * a.t.nchunk * kChunk + base + k0);
#pragma unroll
        for (int i = 0; i < kPer / 16; ++i) {
          const uint4 x = __ldcg(vin + i);
          vw[4 * i] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
        }
      }
      // per byte: 0x80 where the vote is above T / equal to T (keys past len: neither)
      uint32_t gtm[kPer / 4], eqm[kPer / 4];
      uint32_t n_eq = 0, n_gt = 0;
#pragma unroll
      for (int w = 0; w < kPer / 4; ++w) {
        const int rest = len - (k0 + 4 * w);
        const uint32_t valid = rest >= 4 ? 0x80808080u : rest <= 0 ? 0u : (0x80808080u >> (8 * (4 - rest)));
        gtm[w] = bytes_gt(vw[w], T4) & valid;
        eqm[w] = bytes_eq(vw[w], T4) & valid;
        n_gt += __popc(gtm[w]);
        n_eq += __popc(eqm[w]);
      }
      uint32_t eq_tot;
      const uint32_t eq_rank0 = block_excl_scan(n_eq, tmp, &eq_tot);
      uint32_t eq_left = (uint32_t)max64(0, min64((int64_t)n_eq, eq_allow - (int64_t)eq_rank0));
      uint32_t csel;
      int64_t pos = nsel + block_excl_scan(n_gt + eq_left, tmp, &csel);
      int32_t* out = a.cand_idx + cq + sel_before;
#pragma unroll
      for (int w = 0; w < kPer / 4; ++w) {
        uint32_t e = eqm[w];
        // the lowest-position keys equal to T, up to this thread's share
        while (__popc(e) > (int)eq_left) e &= ~(0x80000000u >> __clz(e));
        eq_left -= __popc(e);
        uint32_t m = gtm[w] | e;
        while (m) {
          const int j = (31 - __clz(m & (0u - m))) >> 3;  // lowest flagged byte
          m &= m - 1;
          out[pos++] = (int32_t)(a.s.sink + base + k0 + 4 * w + j);
        }
      }
      eq_allow = max64(0, eq_allow - (int64_t)eq_tot);
      nsel += csel;
    }
  }
  trace_block(a.trace, kTkDecode1, 0);
  // every block's candidates are in the query head's list (ascending positions)
  cluster_sync();

  // ---- 3. estimates: block r takes the slice [C r / cs, C (r + 1) / cs) ------
  const int64_t s_lo = a.C * r / cs, s_hi = a.C * (r + 1) / cs;
  const uint32_t nown = (uint32_t)(s_hi - s_lo);
  {
    // two candidates per thread and round: the first one's record straight
    // into registers, the second one's by asynchronous copy into the
    // thread's own 128-byte slot (16-byte chunks swizzled against bank
    // conflicts), so both gathers are in flight together
    const uint8_t* rec = a.t.rec + sh * a.t.rcap * kRecBytes;
    const float qn = s_qn;
    uint4* slot = reinterpret_cast<uint4*>(U + kUKeys) + tid * 8;
    for (uint32_t i0 = 0; i0 < nown; i0 += 2 * kThreads) {
      const uint32_t ia = i0 + tid, ib = i0 + kThreads + tid;
      const int32_t pa = ia < nown ? __ldcg(a.cand_idx + cq + s_lo + ia) : -1;
      const int32_t pb = ib < nown ? __ldcg(a.cand_idx + cq + s_lo + ib) : -1;
      if (pb >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(rec + (int64_t)(pb - a.s.sink) * kRecBytes);
#pragma unroll
        for (int u = 0; u < 8; ++u) cp_async16(slot + (u ^ (tid & 7)), src + u);
      }
      cp_async_commit();
      if (pa >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(rec + (int64_t)(pa - a.s.sink) * kRecBytes);
        uint4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __ldg(src + u);
        const float e = estimate(x, tq, qn);
        a.cand_est[cq + s_lo + ia] = e;
        if (ia < kListCap) {
          lpos[ia] = pa;
          lest[ia] = e;
        }
      }
      cp_async_wait_all();  // this thread's own slot
      if (pb >= 0) {
        uint4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = slot[u ^ (tid & 7)];
        const float e = estimate(x, tq, qn);
        a.cand_est[cq + s_lo + ib] = e;
        if (ib < kListCap) {
          lpos[ib] = pb;
          lest[ib] = e;
        }
      }
    }
  }
  __syncthreads();
  trace_block(a.trace, kTkDecode1, 1);
  trace_mark(tr, kTrDecode3);

  // ---- 4. top-k ------------------------------------------------------------
  // The k_eff-th best candidate by (estimate desc, position asc): block 0
  // runs a radix select over the order keys of all C estimates, then tells
  // every block where its slice's selected entries go and how many of its
  // keys equal to the k-th key it keeps (the lowest positions first).
  const bool select_all = a.k_eff >= a.C;  // the same in every block
  uint32_t prefix = 0, my_eq_take = 0;
  int64_t out_off = s_lo;
  if (!select_all) {
    cluster_sync();  // every estimate is written
    if (r == 0) select_kth(a.C, a.k_eff, a.cand_est + cq, cs, U, tmp, sel_info);
    cluster_sync();
    prefix = dsmem_u32(&sel_info[kClusterMax][0], 0);
    out_off = dsmem_u32(&sel_info[r][0], 0);
    my_eq_take = dsmem_u32(&sel_info[r][1], 0);
  }
  trace_mark(tr, kTrDecodeFine + 20);
  {
    // ordered output: thread t owns entries [t * per, t * per + per) of the slice
    auto est_of = [&](uint32_t i) { return i < kListCap ? lest[i] : __ldcg(a.cand_est + cq + s_lo + i); };
    const uint32_t per = (nown + kThreads - 1) / kThreads;
    const uint32_t i0 = min(nown, tid * per), i1 = min(nown, i0 + per);
    uint32_t n_eq = 0, n_gt = 0;
    for (uint32_t i = i0; i < i1; ++i) {
      const uint32_t key = order_key(est_of(i));
      n_eq += key == prefix ? 1u : 0u;
      n_gt += key > prefix ? 1u : 0u;
    }
    uint32_t tot_eq;
    const uint32_t eq_rank0 = select_all ? 0u : block_excl_scan(n_eq, tmp, &tot_eq);
    const uint32_t eq_take = select_all ? 0u : (uint32_t)max64(0, min64(n_eq, (int64_t)my_eq_take - eq_rank0));
    const uint32_t cnt = select_all ? i1 - i0 : n_gt + eq_take;
    uint32_t tot_sel;
    uint32_t opos = block_excl_scan(cnt, tmp, &tot_sel);
    int32_t* oi = a.topk_idx + (int64_t)sq * a.k + out_off;
    float* os = a.topk_score ? a.topk_score + (int64_t)sq * a.k + out_off : nullptr;
    uint32_t eq_seen = 0;
    for (uint32_t i = i0; i < i1; ++i) {
      const float e = est_of(i);
      const uint32_t key = order_key(e);
      bool take = select_all || key > prefix;
      if (!select_all && key == prefix) {
        take = eq_seen < eq_take;
        ++eq_seen;
      }
      if (take) {
        if (out_off + opos < a.k_eff) {  // always, unless the counts above disagree
          oi[opos] = i < kListCap ? lpos[i] : __ldcg(a.cand_idx + cq + s_lo + i);
          if (os) os[opos] = e;
        }
        ++opos;
      }
    }
    if (r == 0) {
      for (int64_t i = a.k_eff + tid; i < a.k; i += kThreads) {
        a.topk_idx[(int64_t)sq * a.k + i] = -1;
        if (a.topk_score) a.topk_score[(int64_t)sq * a.k + i] = -INFINITY;
      }
    }
  }
  if (a.out != nullptr && tid < kDim) zs[tid] = qs[tid] * a.qscale;  // scaled q for the attention
  trace_block(a.trace, kTkDecode1, 2);
  trace_mark(tr, kTrDecode4);
  // the top-k of the whole cluster is written; no block reads another's
  // shared memory after this point until the attention merge
  cluster_sync();
  trace_block(a.trace, kTkDecode1, 3);

  // ---- 5. sparse attention ---------------------------------------------------
  if (a.out != nullptr) {
    const int64_t R = a.nwin + a.k_eff;
    const int64_t row_lo = R * r / cs, row_hi = R * (r + 1) / cs;
    const int ntiles = (int)((row_hi - row_lo + kTile - 1) / kTile);
    const int ring = a.s.local + a.s.ubuf;
    const int srow = tid >> 4, ch = tid & 15;  // staged row of the tile, 16-byte chunk of it
    // stage tile j into buffer j % kStages (one commit group per tile, empty past the end)
    // top-k positions of the block's retrieved rows, loaded once (all in flight)
    const int64_t ret0 = max64(row_lo, a.nwin);
    const int ntab = (int)min64(max64(0, row_hi - ret0), kListCap);
    int32_t* ptab = lpos;
    __syncthreads();  // the candidate slice in lpos is no longer read
    for (int t = tid; t < ntab; t += kThreads) ptab[t] = __ldcg(a.topk_idx + (int64_t)sq * a.k + (ret0 - a.nwin) + t);
    const uint32_t nmod = ring > 0 ? (uint32_t)(a.N % ring) : 0u;  // ring slot of the first Local token
    __syncthreads();
    auto stage = [&](int j) {
      const int buf = j % kStages;
      uint16_t* kd = stK + (buf * kTile + srow) * kKStride + 8 * ch;
      uint16_t* vd = stV + (buf * kTile + srow) * kKStride + 8 * ch;
      const int64_t row = row_lo + (int64_t)j * kTile + srow;
      bool have = false;
      if (j < ntiles && row < row_hi) {
        if (row < a.nwin) {
          int64_t slot = row, pos = row;
          if (row >= a.nsink) {
            uint32_t x = nmod + (uint32_t)(row - a.nsink);  // < 2 ring: the window holds at most ring tokens
            if (x >= (uint32_t)ring) x -= (uint32_t)ring;
            slot = a.s.sink + x;
            pos = a.s.sink + a.N + (row - a.nsink);
          }
          if (pos == a.new_pos) {
            // the step's own token: from the caller's k/v, converted as the append stores it
            *reinterpret_cast<uint4*>(kd) = load8_as_bf16(a.k_new, a.kvdtype, sh * kDim + 8 * ch);
            *reinterpret_cast<uint4*>(vd) = load8_as_bf16(a.v_new, a.kvdtype, sh * kDim + 8 * ch);
          } else {
            const int64_t e = (sh * a.kv.win + slot) * kDim + 8 * ch;
            cp_async16(kd, a.kv.win_k + e);
            cp_async16(vd, a.kv.win_v + e);
          }
          have = true;
        } else {
          const int64_t t = row - ret0;
          const int64_t pos = t < kListCap ? ptab[t] : __ldcg(a.topk_idx + (int64_t)sq * a.k + (row - a.nwin));
          if (pos >= a.s.sink && pos < a.s.sink + a.N) {
            const int64_t e = (sh * a.kv.rcap + (pos - a.s.sink)) * kDim + 8 * ch;
            cp_async16(kd, a.kv.st_k + e);
            cp_async16(vd, a.kv.st_v + e);
            have = true;
          } else if (pos >= 0 && ch == 0) {
            atomicOr(a.status, kStatusBadIndex);
          }
        }
      }
      if (!have) *reinterpret_cast<uint4*>(vd) = make_uint4(0, 0, 0, 0);  // finite zeros for the V sum
      if (ch == 0) rvalid[buf][srow] = have ? 1 : 0;
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kStages; ++j) stage(j);
    // Each warp keeps its own online softmax over rows 2w and 2w + 1 of
    // every tile: lanes 0-15 score row 2w and lanes 16-31 row 2w + 1
    // (8 dimensions each, q in registers); every lane accumulates output
    // dimensions 4 lane .. 4 lane + 3.  The warps merge once at the end.
    const int hrow = 2 * warp + (lane >> 4), sub = lane & 15;
    float qr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qr[i] = zs[8 * sub + i];
    float M = -FLT_MAX, l = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j % kStages;
      cp_async_wait_group<kStages - 1>();
      __syncthreads();
      const uint4 kv8 = *reinterpret_cast<const uint4*>(stK + (buf * kTile + hrow) * kKStride + 8 * sub);
      const uint32_t w[4] = {kv8.x, kv8.y, kv8.z, kv8.w};
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s += qr[2 * i] * bf16_bits_to_float(w[i] & 0xffffu);
        s += qr[2 * i + 1] * __uint_as_float(w[i] & 0xffff0000u);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
      const bool valid = rvalid[buf][hrow] != 0;
      if (!valid) s = -FLT_MAX;
      const float Mn = fmaxf(M, fmaxf(s, __shfl_xor_sync(kFull, s, 16)));
      const float sc = exp2f(M - Mn);
      const float pm = valid ? exp2f(s - Mn) : 0.f;
      const float p0 = __shfl_sync(kFull, pm, 0), p1 = __shfl_sync(kFull, pm, 16);
      l = l * sc + p0 + p1;
      const uint2 v0 = *reinterpret_cast<const uint2*>(stV + (buf * kTile + 2 * warp) * kKStride + 4 * lane);
      const uint2 v1 = *reinterpret_cast<const uint2*>(stV + (buf * kTile + 2 * warp + 1) * kKStride + 4 * lane);
      o4[0] = o4[0] * sc + p0 * bf16_bits_to_float(v0.x & 0xffffu) + p1 * bf16_bits_to_float(v1.x & 0xffffu);
      o4[1] = o4[1] * sc + p0 * __uint_as_float(v0.x & 0xffff0000u) + p1 * __uint_as_float(v1.x & 0xffff0000u);
      o4[2] = o4[2] * sc + p0 * bf16_bits_to_float(v0.y & 0xffffu) + p1 * bf16_bits_to_float(v1.y & 0xffffu);
      o4[3] = o4[3] * sc + p0 * __uint_as_float(v0.y & 0xffff0000u) + p1 * __uint_as_float(v1.y & 0xffff0000u);
      M = Mn;
      __syncthreads();  // buffer `buf` is free
      stage(j + kStages);
    }
    cp_async_wait_all();
    __syncthreads();
    trace_block(a.trace, kTkDecode2, 0);
    // merge the warps: wo[w][d], then per warp (max, sum)
    float* wo = reinterpret_cast<float*>(U);
    float* wml = wo + kWarps * kDim;
    *reinterpret_cast<float4*>(wo + warp * kDim + 4 * lane) = make_float4(o4[0], o4[1], o4[2], o4[3]);
    if (lane == 0) {
      wml[2 * warp] = M;
      wml[2 * warp + 1] = l;
    }
    __syncthreads();
    if (tid < kDim) {
      float Mb = -FLT_MAX;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2)
        if (wml[2 * w2 + 1] > 0.f) Mb = fmaxf(Mb, wml[2 * w2]);
      float ob = 0.f, lb = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        const float lw = wml[2 * w2 + 1];
        if (lw > 0.f) {
          const float f = exp2f(wml[2 * w2] - Mb);
          ob += wo[w2 * kDim + tid] * f;
          lb += lw * f;
        }
      }
      part[4 + tid] = ob;
      if (tid == 0) {
        part[0] = Mb;
        part[1] = lb;
      }
    }
    cluster_sync();
    trace_mark(tr, kTrDecode5);
    if (r == 0 && tid < kDim) {
      float mm[kClusterMax], ll[kClusterMax], oo[kClusterMax];
#pragma unroll
      for (int q = 0; q < kClusterMax; ++q) {
        mm[q] = q < cs ? __uint_as_float(dsmem_u32(part, q)) : 0.f;
        ll[q] = q < cs ? __uint_as_float(dsmem_u32(part + 1, q)) : 0.f;
        oo[q] = q < cs ? __uint_as_float(dsmem_u32(part + 4 + tid, q)) : 0.f;
      }
      float Mx = -FLT_MAX;
#pragma unroll
      for (int q = 0; q < kClusterMax; ++q)
        if (ll[q] > 0.f) Mx = fmaxf(Mx, mm[q]);
      float Lt = 0.f, ot = 0.f;
#pragma unroll
      for (int q = 0; q < kClusterMax; ++q) {
        if (ll[q] > 0.f) {
          const float f = exp2f(mm[q] - Mx);
          Lt += ll[q] * f;
          ot += oo[q] * f;
        }
      }
      a.out[(int64_t)sq * kDim + tid] = __float2bfloat16_rn(Lt > 0.f ? ot / Lt : 0.f);
    }
    // every block's shared memory stays until block 0 has read it
    cluster_sync();
    trace_block(a.trace, kTkDecode2, 1);
  }

  // ---- the step's own token into the cache ---------------------------------
  if (a.new_pos >= 0 && r == 0 && qh % a.s.g == 0 && warp == 0)
    append_token_warp(a.k_new, a.v_new, a.kvdtype, a.new_pos, sh, lane, a.s, a.kv, a.t, a.sm, a.rp);
  trace_mark(tr, kTrDecode6);
  trace_block(a.trace, kTkDecode2, 3);
}

// Empty Retrieval zone: no candidates, every top-k entry is (-1, -inf).
__global__ void k_fill_empty(int32_t* idx, float* score, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    idx[i] = -1;
    if (score) score[i] = -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fill_empty(int32_t* idx, float* score, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_fill_empty<<<(int)min64(1024, (n + 255) / 256), 256, 0, st>>>(idx, score, n);
  return cudaGetLastError();
}

int decode_cluster_size(int nchunk_active) { return nchunk_active < kClusterMax ? nchunk_active : kClusterMax; }

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t st) {
  const RetrieveArgs& ra = L.ra;
  DecodeArgs a;
  a.s = ra.s;
  a.t = ra.t;
  a.kv = L.kv;
  a.sm = ra.sm;
  a.rp = ra.rp;
  a.rho = ra.rho;
  a.flat = ra.flat;
  a.nbins = ra.nbins;
  a.nchunk_active = ra.nchunk_active;
  const int cs = decode_cluster_size(ra.nchunk_active);
  if (cs < 1) return cudaErrorInvalidValue;
  a.cpb = (ra.nchunk_active + cs - 1) / cs;
  a.N = ra.N;
  a.C = ra.C;
  a.k = ra.k;
  a.k_eff = ra.k_eff;
  a.cmax = ra.cmax;
  a.nsink = L.nsink;
  a.nwin = L.nwin;
  a.q = L.q;
  a.qdtype = L.qdtype;
  a.qscale = 1.4426950408889634f / sqrtf((float)kDim);
  a.k_new = L.k_new;
  a.v_new = L.v_new;
  a.kvdtype = L.kvdtype;
  a.new_pos = L.k_new ? L.new_pos : -1;
  a.qt = ra.qt;
  a.qnorm = ra.qnorm;
  a.hot = ra.hot;
  a.votes = ra.votes;
  a.cand_idx = ra.cand_idx;
  a.cand_est = ra.cand_est;
  a.status = L.status;
  a.trace = ra.trace;
  a.topk_idx = ra.topk_idx;
  a.topk_score = ra.topk_score;
  a.out = L.out;
  const size_t smem = (size_t)hot_bytes(kSub * ra.rho) + kUBytes;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               hot_bytes(kSub * kCentroids) + kUBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, ra.s.batch * ra.s.hq);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_decode, a);
}

}  // namespace paris
