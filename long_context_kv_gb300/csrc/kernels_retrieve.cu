// Retrieval kernels of ParisKV: (A) query preparation + collision votes +
// candidate plan, (B) candidate selection + RSQ-IP rerank + top-k.
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// Methodology 2, "Coarse candidate generation (collision-based)" and
// "Candidate reranking (RSQ-IP)", "Estimation":
//   <k, q> ~ ||q||_2 sum_b w_{i,b} <v_{i,b}, q~_b>.
//
// Both kernels run one block per tile = (chunk of kChunk Retrieval-zone
// keys, sequence x query head).  The per-query-head reductions (the
// candidate plan after A, the top-k after B) are done by the last block of
// the query head to finish, found with an atomic counter after a memory
// fence; no block ever waits for another.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kVoteThreads = 256;
constexpr int kSelThreads = 256;
constexpr int kTopBins = 2048;         // = 8 * kSelThreads
constexpr int kRankMax = 512;          // threshold-bin size resolved by pairwise ranks
constexpr int kStageMax = kChunk / 2;  // candidate keys the top-k stages in shared memory

// ===========================================================================
// (A) query preparation, votes, plan
// ===========================================================================
//
// Query preparation (every tile recomputes the rotation and the hot
// centroids of its query; tile 0 also publishes q~ and ||q||):
//   ||q|| = sqrt(sequential sum over the d inputs of q_j q_j);
//   z = fwht(D q); ||z|| likewise; q~ = z / ||z|| (0 if ||z|| = 0);
//   score of centroid c in subspace b = sequential sum over j of +-z_{b,j}
//   (minus where bit j of c is set); the top rho per subspace by
//   (score desc, id asc) get weight rho - r (rank r) or 1 (flat).
// Votes: each key of the chunk sits in exactly one bucket per subspace, so
// walking the hot buckets' lists and adding their weights gives every key
// sum_b weight_b(id_{i,b}) (one byte per key, at most 255).
// Plan (last tile of the query head): T = the largest vote value whose
// suffix count reaches C; keys above T are candidates, then keys equal to T
// in ascending index order until C.  Per chunk: candidates in earlier
// chunks, and how many keys equal to T the chunk may still take.
struct VoteArgs {
  Tables t;
  SignMask sm;
  Shape s;
  int rho, flat, nbins, nch, plan_stride;
  int64_t N, C;
  const void* q;
  int qdtype;
  float* qt;
  float* qnorm;
  uint32_t* hot;
  uint8_t* votes;
  uint32_t* hist;
  int32_t* plan;
  uint32_t* counter;
  // fused append of one decode token (k_new == nullptr: none)
  const void* k_new;
  const void* v_new;
  int kvdtype;
  int64_t pos;
  KvStore kv;
  RsqParams rp;
};

__global__ void __launch_bounds__(kVoteThreads) k_vote(VoteArgs a) {
  extern __shared__ __align__(16) uint32_t dyn[];
  const int nhot = kSub * a.rho;
  uint32_t* votes = dyn;                                                 // kChunk / 4 words
  float* sc = reinterpret_cast<float*>(votes + kChunk / 4);              // [kSub][kCentroids]
  uint32_t* hbeg = reinterpret_cast<uint32_t*>(sc + kSub * kCentroids);  // nhot
  uint32_t* hpre = hbeg + nhot;                                          // nhot + 1
  uint32_t* hwt = hpre + nhot + 1;                                       // nhot
  __shared__ float qs[kDim], zs[kDim];
  __shared__ uint32_t hist[kMaxBins];
  __shared__ uint32_t s_gt[kMaxChunks], s_eq[kMaxChunks];
  __shared__ uint32_t tmp[33];
  __shared__ float s_zn;
  __shared__ int s_last, s_T;
  __shared__ int64_t s_quota;

  const int c = blockIdx.x, sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, a.N - base);

  // -- phase 0: clear, rotate the query, fused append ------------------------
  for (int i = tid; i < kChunk / 16; i += blockDim.x) reinterpret_cast<uint4*>(votes)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kMaxBins; i += blockDim.x) hist[i] = 0;
  if (warp == 0) {
    float y[4];
    load4(a.q, a.qdtype, (int64_t)sq * kDim + 4 * lane, y);
#pragma unroll
    for (int i = 0; i < 4; ++i) qs[4 * lane + i] = y[i];
    apply_signs(y, a.sm, lane);
    fwht128_warp(y, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) zs[4 * lane + i] = y[i];
  } else if (warp == kVoteThreads / 32 - 1 && a.k_new != nullptr && c == 0 && qh % a.s.g == 0) {
    append_token_warp(a.k_new, a.v_new, a.kvdtype, a.pos, sh, lane, a.s, a.kv, a.t, a.sm, a.rp);
  }
  __syncthreads();

  // -- phase 1: norms (tile 0), centroid scores, hot centroids --------------
  if (c == 0 && tid == 32) {
    float acc = 0.f;
    for (int j = 0; j < kDim; ++j) acc = __fadd_rn(acc, __fmul_rn(qs[j], qs[j]));
    a.qnorm[sq] = __fsqrt_rn(acc);
  }
  if (c == 0 && tid == 64) {
    float acc = 0.f;
    for (int j = 0; j < kDim; ++j) acc = __fadd_rn(acc, __fmul_rn(zs[j], zs[j]));
    s_zn = __fsqrt_rn(acc);
  }
  for (int cid = tid; cid < kCentroids; cid += blockDim.x) {
#pragma unroll 4
    for (int b = 0; b < kSub; ++b) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kM; ++j) {
        const float zz = zs[b * kM + j];
        acc = __fadd_rn(acc, ((cid >> j) & 1) ? -zz : zz);
      }
      sc[b * kCentroids + cid] = acc;
    }
  }
  __syncthreads();
  if (c == 0 && tid < kDim) {
    const float zn = s_zn;
    a.qt[(int64_t)sq * kDim + tid] = zn > 0.f ? __fdiv_rn(zs[tid], zn) : 0.f;
  }
  for (int b = warp; b < kSub; b += kVoteThreads / 32) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = sc[b * kCentroids + lane + 32 * i];
    uint32_t taken = 0;
    for (int r = 0; r < a.rho; ++r) {
      float best = -FLT_MAX;
      int bid = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int id = lane + 32 * i;
        if (!((taken >> i) & 1u) && (v[i] > best || (v[i] == best && id < bid))) {
          best = v[i];
          bid = id;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(kFull, best, o);
        const int oid = __shfl_xor_sync(kFull, bid, o);
        if (ob > best || (ob == best && oid < bid)) {
          best = ob;
          bid = oid;
        }
      }
      if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
      if (lane == 0) {
        const uint32_t wgt = a.flat ? 1u : (uint32_t)(a.rho - r);
        const int e = b * a.rho + r;
        hbeg[e] = (uint32_t)bid;
        hwt[e] = wgt;
        if (c == 0) a.hot[(int64_t)sq * nhot + e] = (uint32_t)bid | (wgt << 16);
      }
    }
  }
  __syncthreads();

  // -- phase 2: walk the hot buckets' lists ---------------------------------
  const uint32_t* off = a.t.off + ((sh * a.t.nchunk + c) * kSub) * kOffStride;
  const uint16_t* ent = a.t.ent + ((sh * a.t.nchunk + c) * kSub) * (int64_t)kChunk;
  {
    const int per = (nhot + blockDim.x - 1) / blockDim.x;  // <= 16
    uint32_t lens[16];
    uint32_t my = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = tid * per + i;
      lens[i] = 0;
      if (i < per && e < nhot) {
        const int b = e / a.rho;
        const uint32_t id = hbeg[e];
        const uint32_t beg = __ldg(off + b * kOffStride + id);
        const uint32_t end = __ldg(off + b * kOffStride + id + 1);
        lens[i] = end - beg;
        hbeg[e] = (uint32_t)b * kChunk + beg;
      }
      my += lens[i];
    }
    uint32_t total;
    uint32_t run = block_excl_scan(my, tmp, &total);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = tid * per + i;
      if (i < per && e < nhot) hpre[e] = run;
      run += lens[i];
    }
    if (tid == 0) hpre[nhot] = total;
  }
  __syncthreads();
  const uint32_t total = hpre[nhot];
  for (uint32_t f0 = tid; f0 < total; f0 += 8 * blockDim.x) {
    uint32_t key[8], wt[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t f = f0 + u * blockDim.x;
      wt[u] = 0;
      key[u] = 0;
      if (f < total) {
        int lo = 0, hi = nhot - 1;  // last e with hpre[e] <= f
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (hpre[mid] <= f) lo = mid; else hi = mid - 1;
        }
        key[u] = __ldg(ent + hbeg[lo] + (f - hpre[lo]));
        wt[u] = hwt[lo];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (wt[u]) atomicAdd(&votes[key[u] >> 2], wt[u] << ((key[u] & 3) * 8));
  }
  __syncthreads();

  // -- phase 3: histogram of the chunk's votes, votes out --------------------
  uint8_t* vout = a.votes + (int64_t)sq * a.t.nchunk * kChunk + base;
  uint32_t nz = 0;
  for (int i = tid; i < kChunk / 16; i += blockDim.x) {
    const uint4 w4 = reinterpret_cast<const uint4*>(votes)[i];
    reinterpret_cast<uint4*>(vout)[i] = w4;
    const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t v = (ws[k >> 2] >> (8 * (k & 3))) & 0xffu;
      if (v && 16 * i + k < len) {
        atomicAdd(&hist[v], 1u);
        ++nz;
      }
    }
  }
  uint32_t nz_total;
  block_excl_scan(nz, tmp, &nz_total);
  uint32_t* hout = a.hist + ((int64_t)sq * a.t.nchunk + c) * kMaxBins;
  for (int s = tid; s < a.nbins; s += blockDim.x) hout[s] = s == 0 ? (uint32_t)len - nz_total : hist[s];

  // -- phase 4: the last tile of the query head writes the plan --------------
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counter[sq], 1u) == (uint32_t)(a.nch - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const uint32_t* hin = a.hist + (int64_t)sq * a.t.nchunk * kMaxBins;
  for (int s = tid; s < kMaxBins; s += blockDim.x) {
    uint32_t tot = 0;
    if (s < a.nbins) {
      for (int c0 = 0; c0 < a.nch; c0 += 8) {
        uint32_t x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = c0 + u < a.nch ? __ldcg(hin + (int64_t)(c0 + u) * kMaxBins + s) : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) tot += x[u];
      }
    }
    hist[s] = tot;
  }
  __syncthreads();
  if (warp == 0) {
    // suffix sums from the top vote value down: lane l owns values 255-8l .. 248-8l
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += hist[255 - 8 * lane - i];
    const uint32_t inc = warp_incl_scan(part, lane);
    const uint32_t exc = inc - part;
    const uint32_t C = (uint32_t)a.C;
    const int owner = __ffs(__ballot_sync(kFull, exc < C && inc >= C)) - 1;
    if (lane == (owner < 0 ? 0 : owner)) {
      uint32_t run = exc;
      int T = 255 - 8 * lane;
      for (int i = 0; i < 8; ++i) {
        const int s = 255 - 8 * lane - i;
        if (run + hist[s] >= C) {
          T = s;
          break;
        }
        run += hist[s];
      }
      s_T = owner < 0 ? 0 : T;
      s_quota = (int64_t)a.C - (owner < 0 ? 0 : run);
    }
  }
  __syncthreads();
  const int T = s_T;
  // keys above T and equal to T in every chunk: one warp per chunk
  for (int cc = warp; cc < a.nch; cc += kVoteThreads / 32) {
    uint32_t x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = T + 1 + lane + 32 * u;
      x[u] = s < a.nbins ? __ldcg(hin + (int64_t)cc * kMaxBins + s) : 0u;
    }
    uint32_t g = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) g += x[u];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(kFull, g, o);
    if (lane == 0) {
      s_gt[cc] = g;
      s_eq[cc] = __ldcg(hin + (int64_t)cc * kMaxBins + T);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int32_t* pl = a.plan + (int64_t)sq * a.plan_stride;
    pl[0] = T;
    int64_t gt_before = 0, eq_before = 0;
    const int64_t quota = s_quota;
    for (int cc = 0; cc < a.nch; ++cc) {
      pl[1 + 2 * cc] = (int32_t)(gt_before + min64(eq_before, quota));
      pl[2 + 2 * cc] = (int32_t)max64(0, quota - eq_before);
      gt_before += s_gt[cc];
      eq_before += s_eq[cc];
    }
    a.counter[sq] = 0;
  }
}

// ===========================================================================
// (B) selection, rerank, top-k
// ===========================================================================
//
// Estimate, float32 in this order:
//   acc = 0; for b: dot = 0; for j: dot = dot + v_{b,j} q~_{b,j};
//   acc = acc + w_b dot;   est = ||q|| acc,
// where v_{b,j} q~_{b,j} comes from a per-query table of the 16 possible
// products of each coordinate (sign bit x 8 levels), each rounded once.
// Top-k (last tile of the query head): the k_eff-th best (estimate desc,
// position asc) candidate is found from a 2048-bin histogram over the
// estimates' range (bins are monotone in the estimate, so only the
// threshold bin needs exact ranks) or, for a degenerate range, an 8-bit
// radix select; every candidate at least as good is kept, listed in
// ascending position order.
struct SelectArgs {
  Tables t;
  RsqParams rp;
  Shape s;
  int nch, plan_stride;
  int64_t N, C, k, k_eff, cmax;
  const float* qt;
  const float* qnorm;
  const uint8_t* votes;
  const int32_t* plan;
  int32_t* cand_idx;
  float* cand_est;
  uint32_t* minmax;  // [batch*Hq][2] order keys, reset to (max, 0) after use
  uint32_t* counter;
  int32_t* out_idx;
  float* out_score;
};

__device__ __forceinline__ float rerank_one(const uint4* rp4, const float* tq, float qn) {
  uint32_t cw[16];
  float ww[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = __ldg(rp4 + i);
    cw[4 * i] = x.x; cw[4 * i + 1] = x.y; cw[4 * i + 2] = x.z; cw[4 * i + 3] = x.w;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = __ldg(rp4 + 4 + i);
    ww[4 * i] = __uint_as_float(x.x); ww[4 * i + 1] = __uint_as_float(x.y);
    ww[4 * i + 2] = __uint_as_float(x.z); ww[4 * i + 3] = __uint_as_float(x.w);
  }
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < kSub; ++b) {
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kM; ++j) dot = __fadd_rn(dot, tq[(b * kM + j) * 16 + ((cw[b] >> (4 * j)) & 15u)]);
    acc = __fadd_rn(acc, __fmul_rn(ww[b], dot));
  }
  return __fmul_rn(qn, acc);
}

// The kk-th best (key desc, position asc) of C candidates, 1 <= kk < C, where
// key_at(i) is the order key of candidate i.  All threads get the result.
template <typename KeyAt>
__device__ void kth_best(int64_t C, int64_t kk, uint32_t kmin, uint32_t kmax, KeyAt key_at, uint32_t* bins,
                         uint32_t* list, uint32_t* tmp, uint32_t* out_key, int64_t* out_pos) {
  __shared__ uint32_t s_b, s_above, s_m, s_key;
  __shared__ int64_t s_pos;
  const int tid = threadIdx.x, nt = blockDim.x;
  const float fmin = key_to_float(kmin), fmax = key_to_float(kmax);
  const float range = fmax - fmin;
  bool linear = kmax > kmin && range > 0.f && range <= FLT_MAX;
  const float scale = linear ? (float)kTopBins / range : 0.f;
  linear = linear && scale > 0.f && scale <= FLT_MAX;
  if (linear) {
    for (int i = tid; i < kTopBins; i += nt) bins[i] = 0;
    if (tid == 0) s_m = 0;
    __syncthreads();
    for (int64_t i = tid; i < C; i += nt) {
      const float e = key_to_float(key_at(i));
      atomicAdd(&bins[min(kTopBins - 1, (int)((e - fmin) * scale))], 1u);
    }
    __syncthreads();
    // thread t owns bins 2047 - 8t .. 2040 - 8t
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += bins[kTopBins - 1 - 8 * tid - i];
    uint32_t tot;
    const uint32_t exc = block_excl_scan(part, tmp, &tot);
    if (exc < (uint32_t)kk && exc + part >= (uint32_t)kk) {
      uint32_t run = exc;
      for (int i = 0; i < 8; ++i) {
        const int bb = kTopBins - 1 - 8 * tid - i;
        if (run + bins[bb] >= (uint32_t)kk) {
          s_b = (uint32_t)bb;
          s_above = run;
          break;
        }
        run += bins[bb];
      }
    }
    __syncthreads();
    const int bstar = (int)s_b;
    for (int64_t i = tid; i < C; i += nt) {
      const float e = key_to_float(key_at(i));
      if (min(kTopBins - 1, (int)((e - fmin) * scale)) == bstar) {
        const uint32_t slot = atomicAdd(&s_m, 1u);
        if (slot < kRankMax) list[slot] = (uint32_t)i;
      }
    }
    __syncthreads();
    const uint32_t m = s_m;
    if (m <= kRankMax) {
      const uint32_t need = (uint32_t)kk - s_above;  // 1 <= need <= m
      for (uint32_t x = tid; x < m; x += nt) {
        const uint32_t pi = list[x], ki = key_at(pi);
        uint32_t rank = 0;
        for (uint32_t y = 0; y < m; ++y) {
          const uint32_t pj = list[y], kj = key_at(pj);
          rank += (kj > ki || (kj == ki && pj < pi)) ? 1u : 0u;
        }
        if (rank == need - 1) {
          s_key = ki;
          s_pos = pi;
        }
      }
      __syncthreads();
      *out_key = s_key;
      *out_pos = s_pos;
      return;
    }
  }
  // radix select of the kk-th largest key, 8 bits at a time
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)kk;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) bins[i] = 0;
    __syncthreads();
    for (int64_t i = tid; i < C; i += nt) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&bins[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {  // lane t owns digits 255 - 8t .. 248 - 8t
      uint32_t part = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) part += bins[255 - 8 * tid - i];
      const uint32_t inc = warp_incl_scan(part, tid);
      const uint32_t exc = inc - part;
      if (exc < remaining && inc >= remaining) {
        uint32_t run = exc;
        for (int i = 0; i < 8; ++i) {
          const int dg = 255 - 8 * tid - i;
          if (run + bins[dg] >= remaining) {
            s_b = (uint32_t)dg;
            s_above = run;
            break;
          }
          run += bins[dg];
        }
      }
    }
    __syncthreads();
    prefix |= s_b << shift;
    mask |= 255u << shift;
    remaining -= s_above;
    __syncthreads();
  }
  // the remaining-th lowest position among keys equal to prefix
  const int64_t per = (C + nt - 1) / nt;
  const int64_t i0 = min64(C, tid * per), i1 = min64(C, i0 + per);
  uint32_t n_eq = 0;
  for (int64_t i = i0; i < i1; ++i) n_eq += key_at(i) == prefix ? 1u : 0u;
  uint32_t tot;
  const uint32_t before = block_excl_scan(n_eq, tmp, &tot);
  if (before < remaining && before + n_eq >= remaining) {
    uint32_t seen = before;
    for (int64_t i = i0; i < i1; ++i) {
      if (key_at(i) == prefix && ++seen == remaining) {
        s_pos = i;
        break;
      }
    }
  }
  __syncthreads();
  *out_key = prefix;
  *out_pos = s_pos;
}

__global__ void __launch_bounds__(kSelThreads, 2) k_select(SelectArgs a) {
  __shared__ float tq[kDim * 16];
  __shared__ __align__(16) uint32_t keys32[kStageMax];  // u16 candidate keys, later staged order keys
  __shared__ uint32_t list[kRankMax];
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t s_min[kSelThreads / 32], s_max[kSelThreads / 32];
  __shared__ int s_last;
  uint16_t* keys = reinterpret_cast<uint16_t*>(keys32);

  const int c = blockIdx.x, sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, a.N - base);

  // -- loads: plan, this chunk's votes, q~ -> product table ------------------
  const int32_t* pl = a.plan + (int64_t)sq * a.plan_stride;
  const int T = __ldcg(pl);
  const int64_t sel_before = __ldcg(pl + 1 + 2 * c);
  const int64_t eq_allow = __ldcg(pl + 2 + 2 * c);
  constexpr int kPer = kChunk / kSelThreads;  // 64 keys per thread
  const int k0 = tid * kPer;
  const uint4* vin = reinterpret_cast<const uint4*>(a.votes + (int64_t)sq * a.t.nchunk * kChunk + base + k0);
  uint32_t vw[kPer / 4];
#pragma unroll
  for (int i = 0; i < kPer / 16; ++i) {
    const uint4 x = __ldcg(vin + i);
    vw[4 * i] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
  }
  {
    const int coord = tid >> 1, nb0 = (tid & 1) * 8;
    const float qv = __ldcg(a.qt + (int64_t)sq * kDim + coord);
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int nib = nb0 + n;
      const float l = a.rp.lev[nib & 7];
      tq[coord * 16 + nib] = __fmul_rn((nib & 8) ? -l : l, qv);
    }
  }
  const float qn = __ldcg(a.qnorm + sq);

  // -- ordered compaction of this chunk's candidates ------------------------
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
  {
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
      if (take) keys[pos++] = (uint16_t)(k0 + i);
    }
  }
  __syncthreads();

  // -- rerank: one candidate per thread, 128 bytes in flight each ----------
  int32_t* cidx = a.cand_idx + (int64_t)sq * a.cmax + sel_before;
  float* cest = a.cand_est + (int64_t)sq * a.cmax + sel_before;
  const uint8_t* rec = a.t.rec + (sh * a.t.rcap + base) * kRecBytes;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (uint32_t r = tid; r < nsel; r += blockDim.x) {
    const uint32_t key = keys[r];
    const float e = rerank_one(reinterpret_cast<const uint4*>(rec + (int64_t)key * kRecBytes), tq, qn);
    cidx[r] = (int32_t)(a.s.sink + base + key);
    cest[r] = e;
    kmin = min(kmin, order_key(e));
    kmax = max(kmax, order_key(e));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
  }
  if (lane == 0) {
    s_min[warp] = kmin;
    s_max[warp] = kmax;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kSelThreads / 32; ++w) {
      kmin = min(kmin, s_min[w]);
      kmax = max(kmax, s_max[w]);
    }
    if (nsel) {
      atomicMin(&a.minmax[2 * sq], kmin);
      atomicMax(&a.minmax[2 * sq + 1], kmax);
    }
  }

  // -- the last tile of the query head takes the top-k ----------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counter[sq], 1u) == (uint32_t)(a.nch - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t C = a.C, kk = a.k_eff;
  const float* est = a.cand_est + (int64_t)sq * a.cmax;
  const int32_t* cid = a.cand_idx + (int64_t)sq * a.cmax;
  int32_t* oi = a.out_idx + (int64_t)sq * a.k;
  float* os = a.out_score ? a.out_score + (int64_t)sq * a.k : nullptr;
  const uint32_t gmin = __ldcg(a.minmax + 2 * sq), gmax = __ldcg(a.minmax + 2 * sq + 1);
  const bool staged = C <= kStageMax;
  if (staged)
    for (int64_t i = tid; i < C; i += blockDim.x) keys32[i] = order_key(__ldcg(est + i));
  __syncthreads();
  auto key_at = [&](int64_t i) -> uint32_t { return staged ? keys32[i] : order_key(__ldcg(est + i)); };
  uint32_t kstar = 0;
  int64_t pstar = C - 1;
  if (kk < C) kth_best(C, kk, gmin, gmax, key_at, reinterpret_cast<uint32_t*>(tq), list, tmp, &kstar, &pstar);
  // ordered compaction: keep (key, position) at least as good as (kstar, pstar)
  const int64_t per = (C + blockDim.x - 1) / blockDim.x;
  const int64_t i0 = min64(C, tid * per), i1 = min64(C, i0 + per);
  uint32_t cnt = 0;
  for (int64_t i = i0; i < i1; ++i) {
    const uint32_t key = key_at(i);
    cnt += (kk >= C || key > kstar || (key == kstar && i <= pstar)) ? 1u : 0u;
  }
  uint32_t tot;
  uint32_t opos = block_excl_scan(cnt, tmp, &tot);
  for (int64_t i = i0; i < i1; ++i) {
    const uint32_t key = key_at(i);
    if (kk >= C || key > kstar || (key == kstar && i <= pstar)) {
      oi[opos] = __ldcg(cid + i);
      if (os) os[opos] = __ldcg(est + i);
      ++opos;
    }
  }
  for (int64_t i = kk + tid; i < a.k; i += blockDim.x) {
    oi[i] = -1;
    if (os) os[i] = -INFINITY;
  }
  if (tid == 0) {
    a.minmax[2 * sq] = 0xffffffffu;
    a.minmax[2 * sq + 1] = 0u;
    a.counter[sq] = 0;
  }
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
  return (size_t)kChunk + (size_t)kSub * kCentroids * 4 + (size_t)(3 * nhot + 1) * 4;
}

cudaError_t launch_vote(const void* q, int dtype, const RetrieveArgs& a, const AppendFuse* ap, cudaStream_t st) {
  VoteArgs v;
  v.t = a.t;
  v.sm = a.sm;
  v.s = a.s;
  v.rho = a.rho;
  v.flat = a.flat;
  v.nbins = a.nbins;
  v.nch = a.nchunk_active;
  v.plan_stride = a.plan_stride;
  v.N = a.N;
  v.C = a.C;
  v.q = q;
  v.qdtype = dtype;
  v.qt = a.qt;
  v.qnorm = a.qnorm;
  v.hot = a.hot;
  v.votes = a.votes;
  v.hist = a.hist;
  v.plan = a.plan;
  v.counter = a.counter_vote;
  v.k_new = ap ? ap->k : nullptr;
  v.v_new = ap ? ap->v : nullptr;
  v.kvdtype = ap ? ap->dtype : 0;
  v.pos = ap ? ap->pos : 0;
  v.kv = ap ? ap->kv : KvStore{};
  v.rp = a.rp;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_vote, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vote_smem_bytes(kCentroids));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_vote<<<dim3(a.nchunk_active, a.s.batch * a.s.hq), kVoteThreads, vote_smem_bytes(a.rho), st>>>(v);
  return cudaGetLastError();
}

cudaError_t launch_select(const RetrieveArgs& a, cudaStream_t st) {
  SelectArgs s;
  s.t = a.t;
  s.rp = a.rp;
  s.s = a.s;
  s.nch = a.nchunk_active;
  s.plan_stride = a.plan_stride;
  s.N = a.N;
  s.C = a.C;
  s.k = a.k;
  s.k_eff = a.k_eff;
  s.cmax = a.cmax;
  s.qt = a.qt;
  s.qnorm = a.qnorm;
  s.votes = a.votes;
  s.plan = a.plan;
  s.cand_idx = a.cand_idx;
  s.cand_est = a.cand_est;
  s.minmax = a.minmax;
  s.counter = a.counter_select;
  s.out_idx = a.topk_idx;
  s.out_score = a.topk_score;
  k_select<<<dim3(a.nchunk_active, a.s.batch * a.s.hq), kSelThreads, 0, st>>>(s);
  return cudaGetLastError();
}

}  // namespace paris
