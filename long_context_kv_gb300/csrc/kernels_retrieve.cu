// Retrieval kernels of ParisKV.
//
//   k_vote     query preparation + collision votes, one block per tile
//              (chunk of kChunk Retrieval-zone keys, sequence x query head);
//   k_compact  candidate selection (ordered compaction), same tiles;
//   k_rerank   RSQ-IP estimates of every candidate, blocks spread evenly over
//              the candidates of each query head; the last block of a query
//              head takes its top-k.
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// Methodology 2, "Coarse candidate generation (collision-based)" and
// "Candidate reranking (RSQ-IP)", "Estimation":
//   <k, q> ~ ||q||_2 sum_b w_{i,b} <v_{i,b}, q~_b>.
// The last-block reduction finds its block with an atomic counter after a
// memory fence; no block ever waits for another.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kVoteThreads = 512;
constexpr int kCompactThreads = 512;
constexpr int kRerankThreads = 256;
constexpr int kRerankPer = 2;                      // candidates per thread, loads in flight together
constexpr int kTopkThreads = 1024;
constexpr int kTopkRegs = 8;                       // candidates per thread the top-k holds in registers
constexpr int kTopkStage = 24576;                  // candidates the top-k stages in shared memory (192 KB)
constexpr int kHistRegs = 2;                       // histogram cells per thread held by k_compact

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ===========================================================================
// k_qprep
// ===========================================================================
//
// One block per (sequence, query head); warp w < 16 owns subspace w.
//   ||q|| = sqrt(sequential sum over the d inputs of q_j q_j);
//   z = fwht(D q); ||z|| likewise; q~ = z / ||z|| (0 if ||z|| = 0);
//   score of centroid c in subspace b = sequential sum over j of +-z_{b,j}
//   (minus where bit j of c is set); the top rho per subspace by
//   (score desc, id asc) get weight rho - r (rank r) or 1 (flat).
// Writes q~, ||q|| and the hot list (entry b * rho + r = id | weight << 16).
// Warps 16 and 17 run the two norm chains; in a decode step warp 18 of the
// first query head of each KV head appends the step's token.
constexpr int kQprepThreads = 19 * 32;

struct QprepArgs {
  SignMask sm;
  Shape s;
  int rho, flat;
  const void* q;
  int qdtype;
  float* qt;
  float* qnorm;
  uint32_t* hot;
  const void* k_new;  // fused append (nullptr: none)
  const void* v_new;
  int kvdtype;
  int64_t pos;
  KvStore kv;
  Tables t;
  RsqParams rp;
  uint64_t* trace;
};

__global__ void __launch_bounds__(kQprepThreads) k_qprep(QprepArgs a) {
  __shared__ float qs[kDim], zs[kDim];
  const int sq = blockIdx.x;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  trace_block(a.trace, kTkQprep, 0);
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkQprep, 1);
  uint64_t* tr = sq == 0 ? a.trace : nullptr;
  trace_mark(tr, kTrVote0);
  if (warp == 0) {
    float y[4];
    load4(a.q, a.qdtype, (int64_t)sq * kDim + 4 * lane, y);
#pragma unroll
    for (int i = 0; i < 4; ++i) qs[4 * lane + i] = y[i];
    apply_signs(y, a.sm, lane);
    fwht128_warp(y, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) zs[4 * lane + i] = y[i];
  } else if (warp == 18 && a.k_new != nullptr && qh % a.s.g == 0) {
    append_token_warp(a.k_new, a.v_new, a.kvdtype, a.pos, (int64_t)seq * a.s.hkv + kvh, lane, a.s, a.kv, a.t,
                      a.sm, a.rp);
  }
  __syncthreads();
  trace_mark(tr, kTrVote1);
  if (warp < kSub) {
    // scores of centroids lane + 32 i, as order keys
    const int b = warp;
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int cid = lane + 32 * i;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kM; ++j) {
        const float zz = zs[b * kM + j];
        acc = __fadd_rn(acc, ((cid >> j) & 1) ? -zz : zz);
      }
      key[i] = order_key(acc);  // never 0 for a finite score
    }
    uint32_t* hot = a.hot + (int64_t)sq * kSub * a.rho + b * a.rho;
    for (int r = 0; r < a.rho; ++r) {
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
      if (lane == 0) hot[r] = bid | ((a.flat ? 1u : (uint32_t)(a.rho - r)) << 16);
    }
  } else if (warp == 16 || warp == 17) {
    // sequential sums of squares (the products are formed ahead of the chain)
    const float* src = warp == 16 ? qs : zs;
    float acc = 0.f;
    if (lane == 0) {
#pragma unroll
      for (int j0 = 0; j0 < kDim; j0 += 32) {
        float sqv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sqv[j] = __fmul_rn(src[j0 + j], src[j0 + j]);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc = __fadd_rn(acc, sqv[j]);
      }
    }
    const float nrm = __shfl_sync(kFull, __fsqrt_rn(acc), 0);
    if (warp == 16) {
      if (lane == 0) a.qnorm[sq] = nrm;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 4 * lane + i;
        a.qt[(int64_t)sq * kDim + j] = nrm > 0.f ? __fdiv_rn(zs[j], nrm) : 0.f;
      }
    }
  }
  trace_mark(tr, kTrVote2);
  trace_block(a.trace, kTkQprep, 3);
}

// ===========================================================================
// k_vote
// ===========================================================================
//
// One block per tile (chunk of kChunk keys, sequence x query head).  Each key
// of the chunk sits in exactly one bucket per subspace, so walking the lists
// of the query's hot buckets and adding their weights gives every key
// sum_b weight_b(id_{i,b}) (one byte per key, at most 255).  The tile writes
// its votes and their histogram.
struct VoteArgs {
  Tables t;
  Shape s;
  int rho, nbins;
  int64_t N;
  const uint32_t* hot;
  uint8_t* votes;
  uint32_t* hist;
  uint64_t* trace;
};

__global__ void __launch_bounds__(kVoteThreads, 2) k_vote(VoteArgs a) {
  extern __shared__ __align__(16) uint32_t dyn[];
  const int nhot = kSub * a.rho;
  uint32_t* votes = dyn;                          // kChunk / 4 words
  uint32_t* offs = votes + kChunk / 4;            // [kSub][kOffStride]
  uint32_t* hbeg = offs + kSub * kOffStride;      // nhot
  uint32_t* hpre = hbeg + nhot;                   // nhot + 1
  uint32_t* hwt = hpre + nhot + 1;                // nhot
  __shared__ uint32_t hist[kMaxBins];
  __shared__ uint32_t tmp[33];

  const int c = blockIdx.x, sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, a.N - base);
  uint64_t* tr = (c == 0 && sq == 0) ? a.trace : nullptr;
  trace_block(a.trace, kTkVote, 0);

  // before the wait: the chunk's bucket offsets (written by the index build,
  // never by the query preparation) and cleared counters
  const uint32_t* off_g = a.t.off + ((sh * a.t.nchunk + c) * kSub) * kOffStride;
  for (int i = tid; i < kSub * kOffStride / 4; i += blockDim.x) cp_async16(offs + 4 * i, off_g + 4 * i);
  for (int i = tid; i < kChunk / 16; i += blockDim.x) reinterpret_cast<uint4*>(votes)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kMaxBins; i += blockDim.x) hist[i] = 0;
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkVote, 1);
  trace_mark(tr, kTrVote3);

  // hot buckets: list begin and length
  const uint32_t* hot = a.hot + (int64_t)sq * nhot;
  const uint16_t* ent = a.t.ent + ((sh * a.t.nchunk + c) * kSub) * (int64_t)kChunk;
  {
    constexpr int kHotPer = (kSub * kCentroids + kVoteThreads - 1) / kVoteThreads;  // hot entries per thread
    const int per = (nhot + blockDim.x - 1) / blockDim.x;
    uint32_t hv[kHotPer];
#pragma unroll
    for (int i = 0; i < kHotPer; ++i) {
      const int e = tid * per + i;
      hv[i] = (i < per && e < nhot) ? __ldcg(hot + e) : 0u;
    }
    cp_async_wait_all();
    __syncthreads();
    uint32_t lens[kHotPer];
    uint32_t my = 0;
#pragma unroll
    for (int i = 0; i < kHotPer; ++i) {
      const int e = tid * per + i;
      lens[i] = 0;
      if (i < per && e < nhot) {
        const int b = e / a.rho;
        const uint32_t id = hv[i] & 0xffffu;
        const uint32_t beg = offs[b * kOffStride + id];
        lens[i] = offs[b * kOffStride + id + 1] - beg;
        hbeg[e] = (uint32_t)b * kChunk + beg;
        hwt[e] = hv[i] >> 16;
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
  const uint32_t total = hpre[nhot];
  // thread t takes kWalk consecutive list entries: one search, then linear
  // steps; all kWalk loads in flight together
  constexpr int kWalk = 8;
  for (uint32_t f0 = kWalk * tid; f0 < total; f0 += kWalk * blockDim.x) {
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
      if (wt[u]) atomicAdd(&votes[key[u] >> 2], wt[u] << ((key[u] & 3) * 8));
  }
  __syncthreads();
  trace_mark(tr, kTrVote4);

  // histogram of the chunk's votes, votes out
  uint8_t* vout = a.votes + (int64_t)sq * a.t.nchunk * kChunk + base;
  uint32_t nz = 0, small = 0;
  for (int i = tid; i < kChunk / 16; i += blockDim.x) {
    const uint4 w4 = reinterpret_cast<const uint4*>(votes)[i];
    reinterpret_cast<uint4*>(vout)[i] = w4;
    const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t v = (ws[k >> 2] >> (8 * (k & 3))) & 0xffu;
      const bool in = v != 0 && 16 * i + k < len;
      if (in && v <= 4) small += 1u << (8 * (v - 1));  // per-thread counts <= 64 fit a byte
      else if (in) atomicAdd(&hist[v], 1u);
      nz += in ? 1u : 0u;
    }
  }
#pragma unroll
  for (int v = 1; v <= 4; ++v) {
    const uint32_t cnt = __reduce_add_sync(kFull, (small >> (8 * (v - 1))) & 0xffu);
    if (lane == 0 && cnt) atomicAdd(&hist[v], cnt);
  }
  uint32_t nz_total;
  block_excl_scan(nz, tmp, &nz_total);
  uint32_t* hout = a.hist + ((int64_t)sq * a.t.nchunk + c) * kMaxBins;
  for (int s = tid; s < a.nbins; s += blockDim.x) hout[s] = s == 0 ? (uint32_t)len - nz_total : hist[s];
  trace_block(a.trace, kTkVote, 3);
}

// ===========================================================================
// k_compact
// ===========================================================================
//
// The candidates are the first C keys by (votes desc, index asc): with T the
// largest vote value whose suffix count reaches C, every key above T and the
// lowest-index keys equal to T, up to C.  Each tile derives T and its own
// offsets from all chunk histograms of its query head, then writes its
// candidates' positions at their place in the ascending-position list.
struct CompactArgs {
  int nbins, nch, sink, nchunk;
  int64_t N, C, cmax;
  const uint8_t* votes;
  const uint32_t* hist;
  int32_t* cand_idx;
  uint64_t* trace;
};

// Sums of two values over the block (every thread gets both).  `red` holds
// 2 * 32 words of shared memory.
__device__ __forceinline__ void block_sum2(uint32_t& x, uint32_t& y, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  x = __reduce_add_sync(kFull, x);
  y = __reduce_add_sync(kFull, y);
  if (lane == 0) {
    red[warp] = x;
    red[32 + warp] = y;
  }
  __syncthreads();
  x = 0;
  y = 0;
  for (int w = 0; w < nw; ++w) {
    x += red[w];
    y += red[32 + w];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kCompactThreads, 2) k_compact(CompactArgs a) {
  __shared__ uint32_t tot[kMaxBins];
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t red[64];
  __shared__ int s_T;
  __shared__ int64_t s_quota;
  const int c = blockIdx.x, sq = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, a.N - base);
  const int nitems = a.nch * a.nbins;
  const uint32_t* h = a.hist + (int64_t)sq * a.nchunk * kMaxBins;
  uint64_t* tr = (c == 0 && sq == 0) ? a.trace : nullptr;
  for (int i = tid; i < kMaxBins; i += blockDim.x) tot[i] = 0;
  trace_block(a.trace, kTkCompact, 0);
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkCompact, 1);
  trace_mark(tr, kTrCompact0);

  // loads in flight together: histogram cells and this chunk's votes
  uint32_t hv[kHistRegs];
#pragma unroll
  for (int u = 0; u < kHistRegs; ++u) {
    const int i = tid + u * blockDim.x;
    hv[u] = i < nitems ? __ldcg(h + (int64_t)(i / a.nbins) * kMaxBins + i % a.nbins) : 0u;
  }
  constexpr int kPer = kChunk / kCompactThreads;  // 32 keys per thread
  const int k0 = tid * kPer;
  uint32_t vw[kPer / 4];
  {
    const uint4* vin = reinterpret_cast<const uint4*>(a.votes + (int64_t)sq * a.nchunk * kChunk + base + k0);
#pragma unroll
    for (int i = 0; i < kPer / 16; ++i) {
      const uint4 x = __ldcg(vin + i);
      vw[4 * i] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
    }
  }
  __syncthreads();
  trace_mark(tr, kTrCompact1);
#pragma unroll
  for (int u = 0; u < kHistRegs; ++u) {
    const int i = tid + u * blockDim.x;
    if (i < nitems && hv[u]) atomicAdd(&tot[i % a.nbins], hv[u]);
  }
  for (int i = tid + kHistRegs * blockDim.x; i < nitems; i += blockDim.x) {
    const uint32_t x = __ldcg(h + (int64_t)(i / a.nbins) * kMaxBins + i % a.nbins);
    if (x) atomicAdd(&tot[i % a.nbins], x);
  }
  __syncthreads();
  if (warp == 0) {
    // suffix sums from the top vote value down: lane l owns values 255-8l .. 248-8l
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += tot[255 - 8 * lane - i];
    const uint32_t inc = warp_incl_scan(part, lane);
    const uint32_t exc = inc - part;
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
  // keys above T / equal to T in the chunks before this one
  uint32_t gt_before = 0, eq_before = 0;
#pragma unroll
  for (int u = 0; u < kHistRegs; ++u) {
    const int i = tid + u * blockDim.x;
    if (i < nitems && i / a.nbins < c) {
      const int s = i % a.nbins;
      gt_before += s > T ? hv[u] : 0u;
      eq_before += s == T ? hv[u] : 0u;
    }
  }
  for (int i = tid + kHistRegs * blockDim.x; i < nitems; i += blockDim.x) {
    if (i / a.nbins < c) {
      const int s = i % a.nbins;
      const uint32_t x = __ldcg(h + (int64_t)(i / a.nbins) * kMaxBins + s);
      gt_before += s > T ? x : 0u;
      eq_before += s == T ? x : 0u;
    }
  }
  block_sum2(gt_before, eq_before, red);
  const int64_t sel_before = gt_before + min64(eq_before, quota);
  const int64_t eq_allow = max64(0, quota - (int64_t)eq_before);

  // ordered compaction: thread t owns keys [32t, 32t + 32)
  uint32_t n_eq = 0, n_gt = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t v = (vw[i >> 2] >> (8 * (i & 3))) & 0xffu;
    const bool in = k0 + i < len;
    n_eq += (in && v == (uint32_t)T) ? 1u : 0u;
    n_gt += (in && v > (uint32_t)T) ? 1u : 0u;
  }
  uint32_t dummy;
  const uint32_t eq_rank0 = block_excl_scan(n_eq, tmp, &dummy);
  const uint32_t eq_take = (uint32_t)max64(0, min64((int64_t)n_eq, eq_allow - (int64_t)eq_rank0));
  uint32_t nsel;
  uint32_t pos = block_excl_scan(n_gt + eq_take, tmp, &nsel);
  int32_t* out = a.cand_idx + (int64_t)sq * a.cmax + sel_before;
  uint32_t eq_seen = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t v = (vw[i >> 2] >> (8 * (i & 3))) & 0xffu;
    const bool in = k0 + i < len;
    bool take = in && v > (uint32_t)T;
    if (in && v == (uint32_t)T) {
      take = eq_seen < eq_take;
      ++eq_seen;
    }
    if (take) out[pos++] = (int32_t)(a.sink + base + k0 + i);
  }
  trace_mark(tr, kTrCompact2);
  trace_block(a.trace, kTkCompact, 3);
}

// ===========================================================================
// k_rerank
// ===========================================================================
//
// Estimate, float32 in this order:
//   acc = 0; for b: dot = 0; for j: dot = dot + v_{b,j} q~_{b,j};
//   acc = acc + w_b dot;   est = ||q|| acc,
// where v_{b,j} q~_{b,j} comes from a per-query table of the 16 possible
// products of each coordinate (sign bit x 8 levels), each rounded once.
// Top-k (last block of the query head): the k_eff-th best (estimate desc,
// position asc) candidate is found by a search over the 32-bit order keys of
// the estimates with block-wide counts (three probes per round), then the
// lowest positions among keys equal to it; every candidate at least as good
// is kept, listed in ascending position order.
struct RerankArgs {
  Tables t;
  RsqParams rp;
  int hq, g, sink, nblk;
  int64_t C, k, k_eff, cmax;
  const float* qt;
  const float* qnorm;
  const int32_t* cand_idx;
  float* cand_est;
  uint32_t* counter;
  int32_t* out_idx;
  float* out_score;
  uint64_t* trace;
};

__device__ __forceinline__ float rerank_record(const uint4 (&x)[8], const float* tq, float qn) {
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

__global__ void __launch_bounds__(kRerankThreads, 3) k_rerank(RerankArgs a) {
  __shared__ float tq[kDim * 16];
  const int blk = blockIdx.x, sq = blockIdx.y;
  const int seq = sq / a.hq, qh = sq - seq * a.hq, kvh = qh / a.g;
  const int64_t sh = (int64_t)seq * (a.hq / a.g) + kvh;
  const int tid = threadIdx.x;
  const int64_t r0 = (int64_t)blk * kRerankPer * kRerankThreads;
  uint64_t* tr = (blk == 0 && sq == 0) ? a.trace : nullptr;
  trace_mark(tr, kTrRerank0);
  trace_block(a.trace, kTkRerank, 0);

  // before the wait: q~ and ||q|| (written by the query preparation, three
  // kernels back) and the product table
  const float qv = __ldcg(a.qt + (int64_t)sq * kDim + (tid >> 1));
  const float qn = __ldcg(a.qnorm + sq);
  {
    const int coord = tid >> 1, nb0 = (tid & 1) * 8;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int nib = nb0 + n;
      const float l = a.rp.lev[nib & 7];
      tq[coord * 16 + nib] = __fmul_rn((nib & 8) ? -l : l, qv);
    }
  }
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkRerank, 1);
  int32_t pos[kRerankPer];
#pragma unroll
  for (int p = 0; p < kRerankPer; ++p) {
    const int64_t r = r0 + p * kRerankThreads + tid;
    pos[p] = r < a.C ? __ldcg(a.cand_idx + (int64_t)sq * a.cmax + r) : -1;
  }
  // the candidates' 128-byte records
  const uint8_t* rec = a.t.rec + sh * a.t.rcap * kRecBytes;
  uint4 x[kRerankPer][8];
#pragma unroll
  for (int p = 0; p < kRerankPer; ++p) {
    const uint4* rp4 = reinterpret_cast<const uint4*>(rec + (int64_t)max(0, pos[p] - a.sink) * kRecBytes);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[p][i] = pos[p] >= 0 ? __ldg(rp4 + i) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  trace_mark(tr, kTrRerank1);
  float* cest = a.cand_est + (int64_t)sq * a.cmax;
#pragma unroll
  for (int p = 0; p < kRerankPer; ++p) {
    const int64_t r = r0 + p * kRerankThreads + tid;
    if (pos[p] >= 0) cest[r] = rerank_record(x[p], tq, qn);
  }

  trace_mark(tr, kTrRerank2);
  trace_block(a.trace, kTkRerank, 3);
}

// ===========================================================================
// k_topk
// ===========================================================================
//
// One block of 1024 threads per (sequence, query head).  The k_eff-th best
// candidate by (estimate desc, position asc) is found by a radix select on
// the 32-bit order keys of the estimates (8 bits per pass, counted in shared
// memory), then the lowest positions among keys equal to it; every
// candidate at least as good is kept, listed in ascending position order.
// Thread t owns a contiguous slice of the candidates (in registers when the
// slice has at most kTopkRegs of them).
struct TopkArgs {
  int64_t C, k, k_eff, cmax;
  const int32_t* cand_idx;
  const float* cand_est;
  int32_t* out_idx;
  float* out_score;
  uint64_t* trace;
};

// E, I: the query head's estimates and positions (staged in shared memory,
// or the global arrays).  Counting passes use strided ownership (i = t +
// blockDim * u); the tie and output passes use contiguous slices so that the
// result comes out in ascending position order.
__device__ __forceinline__ void topk_select(const TopkArgs& a, int sq, const float* E, const int32_t* I) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t s_d, s_above;
  __shared__ int64_t s_pos;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const int64_t C = a.C, kk = a.k_eff;
  int32_t* oi = a.out_idx + (int64_t)sq * a.k;
  float* os = a.out_score ? a.out_score + (int64_t)sq * a.k : nullptr;
  uint64_t* tr = sq == 0 ? a.trace : nullptr;
  trace_mark(tr, kTrTopk1);
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)kk;
  int64_t pstar = C;
  const int64_t per = (C + nt - 1) / nt;
  const int64_t i0 = min64(C, tid * per), i1 = min64(C, i0 + per);
  if (kk < C) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < C; i += nt) {
        const uint32_t key = order_key(E[i]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      {
        // threads t < 256 own digit 255 - t: block-wide exclusive sums from the top
        const uint32_t v = tid < 256 ? hist[255 - tid] : 0u;
        const uint32_t inc = warp_incl_scan(v, lane);
        if (tid < 256 && lane == 31) tmp[warp] = inc;
        __syncthreads();
        if (tid < 256) {
          uint32_t off = 0;
          for (int w = 0; w < warp; ++w) off += tmp[w];
          const uint32_t exc = off + inc - v;
          if (exc < remaining && exc + v >= remaining) {
            s_d = 255 - tid;
            s_above = exc;
          }
        }
      }
      __syncthreads();
      prefix |= s_d << shift;
      mask |= 255u << shift;
      remaining -= s_above;
    }
    trace_mark(tr, kTrTopk2);
    // `remaining` keys equal to prefix are kept: the lowest positions
    uint32_t n_eq = 0;
    for (int64_t i = i0; i < i1; ++i) n_eq += order_key(E[i]) == prefix ? 1u : 0u;
    uint32_t tot;
    const uint32_t before = block_excl_scan(n_eq, tmp, &tot);
    if (before < remaining && before + n_eq >= remaining) {
      uint32_t seen = before;
      for (int64_t i = i0; i < i1; ++i)
        if (order_key(E[i]) == prefix && ++seen == remaining) {
          s_pos = i;
          break;
        }
    }
    __syncthreads();
    pstar = s_pos;
  }
  trace_mark(tr, kTrTopk3);
  // ordered compaction: keep (key, position) at least as good as (prefix, pstar)
  uint32_t cnt = 0;
  for (int64_t i = i0; i < i1; ++i) {
    const uint32_t key = order_key(E[i]);
    cnt += (kk >= C || key > prefix || (key == prefix && i <= pstar)) ? 1u : 0u;
  }
  uint32_t tot;
  uint32_t opos = block_excl_scan(cnt, tmp, &tot);
  for (int64_t i = i0; i < i1; ++i) {
    const float e = E[i];
    const uint32_t key = order_key(e);
    if (kk >= C || key > prefix || (key == prefix && i <= pstar)) {
      oi[opos] = I[i];
      if (os) os[opos] = e;
      ++opos;
    }
  }
  for (int64_t i = kk + tid; i < a.k; i += nt) {
    oi[i] = -1;
    if (os) os[i] = -INFINITY;
  }
  trace_mark(tr, kTrTopk4);
}

__global__ void __launch_bounds__(kTopkThreads) k_topk(TopkArgs a) {
  extern __shared__ __align__(16) uint32_t stage[];
  const int sq = blockIdx.x;
  trace_block(a.trace, kTkTopk, 0);
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkTopk, 1);
  trace_mark(sq == 0 ? a.trace : nullptr, kTrTopk0);
  const float* est = a.cand_est + (int64_t)sq * a.cmax;
  const int32_t* cid = a.cand_idx + (int64_t)sq * a.cmax;
  if (a.C <= kTopkStage) {
    // 16-byte copies, all in flight together (rows start on 16-byte boundaries)
    float* se = reinterpret_cast<float*>(stage);
    int32_t* si = reinterpret_cast<int32_t*>(stage + ((a.C + 3) / 4) * 4);
    const int nch = (int)((a.C + 3) / 4);
    for (int i = threadIdx.x; i < nch; i += blockDim.x) {
      cp_async16(se + 4 * i, est + 4 * i);
      cp_async16(si + 4 * i, cid + 4 * i);
    }
    cp_async_wait_all();
    __syncthreads();
    topk_select(a, sq, se, si);
  } else {
    topk_select(a, sq, est, cid);
  }
  trace_block(a.trace, kTkTopk, 3);
}

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

size_t vote_smem_bytes(int rho) {
  const int nhot = kSub * rho;
  return (size_t)kChunk + (size_t)kSub * kOffStride * 4 + (size_t)(3 * nhot + 1) * 4;
}

cudaError_t launch_qprep(const void* q, int dtype, const RetrieveArgs& a, const AppendFuse* ap, cudaStream_t st) {
  QprepArgs p;
  p.sm = a.sm;
  p.s = a.s;
  p.rho = a.rho;
  p.flat = a.flat;
  p.q = q;
  p.qdtype = dtype;
  p.qt = a.qt;
  p.qnorm = a.qnorm;
  p.hot = a.hot;
  p.k_new = ap ? ap->k : nullptr;
  p.v_new = ap ? ap->v : nullptr;
  p.kvdtype = ap ? ap->dtype : 0;
  p.pos = ap ? ap->pos : 0;
  p.kv = ap ? ap->kv : KvStore{};
  p.t = a.t;
  p.rp = a.rp;
  p.trace = a.trace;
  return launch_pdl(k_qprep, dim3(a.s.batch * a.s.hq), dim3(kQprepThreads), 0, st, p);
}

cudaError_t launch_vote(const RetrieveArgs& a, cudaStream_t st) {
  VoteArgs v;
  v.t = a.t;
  v.s = a.s;
  v.rho = a.rho;
  v.nbins = a.nbins;
  v.N = a.N;
  v.hot = a.hot;
  v.votes = a.votes;
  v.hist = a.hist;
  v.trace = a.trace;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_vote, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vote_smem_bytes(kCentroids));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(k_vote, dim3(a.nchunk_active, a.s.batch * a.s.hq), dim3(kVoteThreads), vote_smem_bytes(a.rho), st, v);
}

cudaError_t launch_compact(const RetrieveArgs& a, cudaStream_t st) {
  CompactArgs c;
  c.nbins = a.nbins;
  c.nch = a.nchunk_active;
  c.sink = a.s.sink;
  c.nchunk = a.t.nchunk;
  c.N = a.N;
  c.C = a.C;
  c.cmax = a.cmax;
  c.votes = a.votes;
  c.hist = a.hist;
  c.cand_idx = a.cand_idx;
  c.trace = a.trace;
  return launch_pdl(k_compact, dim3(a.nchunk_active, a.s.batch * a.s.hq), dim3(kCompactThreads), 0, st, c);
}

cudaError_t launch_rerank(const RetrieveArgs& a, cudaStream_t st) {
  RerankArgs r;
  r.t = a.t;
  r.rp = a.rp;
  r.hq = a.s.hq;
  r.g = a.s.g;
  r.sink = a.s.sink;
  r.nblk = (int)((a.C + kRerankPer * kRerankThreads - 1) / (kRerankPer * kRerankThreads));
  r.C = a.C;
  r.k = a.k;
  r.k_eff = a.k_eff;
  r.cmax = a.cmax;
  r.qt = a.qt;
  r.qnorm = a.qnorm;
  r.cand_idx = a.cand_idx;
  r.cand_est = a.cand_est;
  r.counter = a.counter_select;
  r.out_idx = a.topk_idx;
  r.out_score = a.topk_score;
  r.trace = a.trace;
  return launch_pdl(k_rerank, dim3(r.nblk, a.s.batch * a.s.hq), dim3(kRerankThreads), 0, st, r);
}

cudaError_t launch_topk(const RetrieveArgs& a, cudaStream_t st) {
  TopkArgs t;
  t.C = a.C;
  t.k = a.k;
  t.k_eff = a.k_eff;
  t.cmax = a.cmax;
  t.cand_idx = a.cand_idx;
  t.cand_est = a.cand_est;
  t.out_idx = a.topk_idx;
  t.out_score = a.topk_score;
  t.trace = a.trace;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkStage * 8);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = a.C <= kTopkStage ? (size_t)((a.C + 3) / 4) * 4 * 8 : 0;
  return launch_pdl(k_topk, dim3(a.s.batch * a.s.hq), dim3(kTopkThreads), smem, st, t);
}

}  // namespace paris
