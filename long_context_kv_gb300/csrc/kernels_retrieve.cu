// Retrieval kernels of ParisKV: query preparation, collision votes over the
// inverted bucket index, candidate selection fused with the RSQ-IP rerank,
// and the final top-k.
//
// ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context LLMs --
// Methodology 2, "Coarse candidate generation (collision-based)" and
// "Candidate reranking (RSQ-IP)", "Estimation":
//   <k, q> ~ ||q||_2 sum_b w_{i,b} <v_{i,b}, q~_b>.
#include <float.h>

#include "paris_device.cuh"

namespace paris {
namespace {

// ---------------------------------------------------------------------------
// Query preparation: one block of 256 threads per (sequence, query head).
//   ||q|| = sqrt(sequential sum over the d inputs of q_j q_j);
//   z = fwht(D q); ||z|| likewise; q~ = z / ||z|| (0 if ||z|| = 0);
//   score of centroid c in subspace b = sequential sum over j of +-z_{b,j}
//   (minus where bit j of c is set); the top rho per subspace by
//   (score desc, id asc) get weight rho - r (rank r) or 1 (flat).
// Outputs q~, ||q|| and the hot list: entry b * rho + r = id | weight << 16.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_qprep(const void* __restrict__ q, int dtype, SignMask sm,
                                               int rho, int flat, float* __restrict__ qt,
                                               float* __restrict__ qnorm, uint32_t* __restrict__ hot) {
  __shared__ float qs[kDim], zs[kDim];
  __shared__ float sc[kSub][kCentroids];
  __shared__ float norms[2];
  const int sq = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kDim) qs[tid] = load1(q, dtype, (int64_t)sq * kDim + tid);
  __syncthreads();
  if (warp == 0) {
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = qs[4 * lane + i];
    apply_signs(y, sm, lane);
    fwht128_warp(y, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) zs[4 * lane + i] = y[i];
  } else if (warp == 1 && lane == 0) {
    float acc = 0.f;
    for (int j = 0; j < kDim; ++j) acc = __fadd_rn(acc, __fmul_rn(qs[j], qs[j]));
    norms[0] = __fsqrt_rn(acc);
  }
  __syncthreads();
  if (tid == 32) {
    float acc = 0.f;
    for (int j = 0; j < kDim; ++j) acc = __fadd_rn(acc, __fmul_rn(zs[j], zs[j]));
    norms[1] = __fsqrt_rn(acc);
  }
  {
    const int c = tid;  // centroid id
#pragma unroll 1
    for (int b = 0; b < kSub; ++b) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kM; ++j) {
        const float zz = zs[b * kM + j];
        acc = __fadd_rn(acc, ((c >> j) & 1) ? -zz : zz);
      }
      sc[b][c] = acc;
    }
  }
  __syncthreads();
  if (tid < kDim) {
    const float zn = norms[1];
    qt[(int64_t)sq * kDim + tid] = zn > 0.f ? __fdiv_rn(zs[tid], zn) : 0.f;
  }
  if (tid == 0) qnorm[sq] = norms[0];
  uint32_t* hot_out = hot + (int64_t)sq * kSub * rho;
  for (int b = warp; b < kSub; b += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = sc[b][lane + 32 * i];
    uint32_t taken = 0;
    for (int r = 0; r < rho; ++r) {
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
      if (lane == 0) hot_out[b * rho + r] = (uint32_t)bid | ((uint32_t)(flat ? 1 : rho - r) << 16);
    }
  }
}

// ---------------------------------------------------------------------------
// Collision votes: one block per (chunk, sequence x query head).  Votes of
// the chunk's keys accumulate in shared memory (one byte per key, at most
// 255) from the bucket lists the query's hot centroids point at; each key
// sits in exactly one bucket per subspace, so its total is
// sum_b weight_b(id_{i,b}).  Writes the votes and their histogram.
// ---------------------------------------------------------------------------
constexpr int kVoteThreads = 512;

struct VoteParams {
  Tables t;
  int hq, g, rho, nbins;
  int64_t N;
  const uint32_t* hot;
  uint8_t* votes;
  uint32_t* hist;
};

__global__ void __launch_bounds__(kVoteThreads) k_vote(VoteParams p) {
  extern __shared__ uint32_t sm_dyn[];
  uint32_t* votes = sm_dyn;                      // kChunk / 4 words
  uint32_t* hbeg = votes + kChunk / 4;           // nhot
  uint32_t* hpre = hbeg + kSub * p.rho;          // nhot + 1 (prefix of list lengths)
  uint32_t* hwt = hpre + kSub * p.rho + 1;       // nhot (weight | b << 8)
  __shared__ uint32_t hist[kMaxBins];
  __shared__ uint32_t tmp[33];

  const int c = blockIdx.x;
  const int sq = blockIdx.y;
  const int seq = sq / p.hq, qh = sq - seq * p.hq, kvh = qh / p.g;
  const int64_t sh = (int64_t)seq * (p.hq / p.g) + kvh;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, p.N - base);
  const int nhot = kSub * p.rho;
  const uint32_t* off = p.t.off + ((sh * p.t.nchunk + c) * kSub) * kOffStride;
  const uint16_t* ent = p.t.ent + ((sh * p.t.nchunk + c) * kSub) * (int64_t)kChunk;
  const uint32_t* hot = p.hot + (int64_t)sq * nhot;

  for (int i = threadIdx.x; i < kChunk / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(votes)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < kMaxBins; i += blockDim.x) hist[i] = 0;
  // bucket list of every hot entry: begin and length
  uint32_t my_len = 0;
  for (int e = threadIdx.x; e < nhot; e += blockDim.x) {
    const uint32_t h = hot[e];
    const int b = e / p.rho;
    const uint32_t id = h & 0xffffu;
    const uint32_t beg = off[b * kOffStride + id];
    const uint32_t end = off[b * kOffStride + id + 1];
    hbeg[e] = (uint32_t)b * kChunk + beg;
    hwt[e] = h >> 16;
    hpre[e] = end - beg;
  }
  __syncthreads();
  // exclusive prefix of list lengths (nhot <= 4096 entries, 8 per thread)
  {
    const int per = (nhot + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * per;
    uint32_t loc[8];
    my_len = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      loc[i] = e < nhot ? hpre[e] : 0u;
      my_len += loc[i];
    }
    uint32_t total;
    uint32_t run = block_excl_scan(my_len, tmp, &total);
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < nhot) hpre[e] = run;
      run += loc[i];
    }
    if (threadIdx.x == 0) hpre[nhot] = total;
  }
  __syncthreads();
  const uint32_t total = hpre[nhot];
  // flattened walk over all hot list entries
  for (uint32_t f = threadIdx.x; f < total; f += blockDim.x) {
    int lo = 0, hi = nhot - 1;  // last e with hpre[e] <= f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (hpre[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const uint32_t key = ent[hbeg[lo] + (f - hpre[lo])];
    atomicAdd(&votes[key >> 2], hwt[lo] << ((key & 3) * 8));
  }
  __syncthreads();
  // histogram of non-zero votes; write the chunk's votes
  uint8_t* vout = p.votes + (int64_t)sq * p.t.nchunk * kChunk + base;
  uint32_t nz = 0;
  for (int wi = threadIdx.x; wi < kChunk / 4; wi += blockDim.x) {
    const uint32_t w = votes[wi];
    reinterpret_cast<uint32_t*>(vout)[wi] = w;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t v = (w >> (8 * k)) & 0xffu;
      if (v && 4 * wi + k < len) {
        atomicAdd(&hist[v], 1u);
        ++nz;
      }
    }
  }
  uint32_t nz_total;
  block_excl_scan(nz, tmp, &nz_total);
  uint32_t* hout = p.hist + ((int64_t)sq * p.t.nchunk + c) * kMaxBins;
  for (int s = threadIdx.x; s < p.nbins; s += blockDim.x)
    hout[s] = s == 0 ? (uint32_t)len - nz_total : hist[s];
}

// ---------------------------------------------------------------------------
// Candidate selection + RSQ-IP rerank: one block per (chunk, sequence x
// query head).  The candidates are the first C keys by (votes desc, index
// asc): with T the largest vote value whose suffix count reaches C, every
// key above T and the lowest-index keys equal to T, up to C.  Chunk
// histograms give each chunk its share and its output offset, so the
// candidate list comes out in ascending index order with no global sort.
// Estimate, float32 in this order:
//   acc = 0; for b: dot = 0; for j: dot = dot + v_{b,j} q~_{b,j};
//   acc = acc + w_b dot;   est = ||q|| acc,
// where v_{b,j} q~_{b,j} is read from a per-query table of the 16 possible
// products of coordinate c (sign bit x 8 levels), each rounded once.
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 512;

struct SelectParams {
  Tables t;
  RsqParams rp;
  int hq, g, nbins, sink;
  int64_t N, C;
  const float* qt;
  const float* qnorm;
  const uint8_t* votes;
  const uint32_t* hist;
  int32_t* cand_idx;
  float* cand_est;
  int64_t cmax;
};

__global__ void __launch_bounds__(kSelThreads) k_select_rerank(SelectParams p) {
  __shared__ float tq[kDim * 16];
  __shared__ uint16_t keys[kChunk];
  __shared__ uint32_t s_tot[kMaxBins], s_bef[kMaxBins];
  __shared__ uint32_t tmp[33];
  __shared__ int64_t s_info[4];

  const int c = blockIdx.x;
  const int sq = blockIdx.y;
  const int seq = sq / p.hq, qh = sq - seq * p.hq, kvh = qh / p.g;
  const int64_t sh = (int64_t)seq * (p.hq / p.g) + kvh;
  const int64_t base = (int64_t)c * kChunk;
  const int len = (int)min64(kChunk, p.N - base);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_info[0] = 0;
    s_info[1] = p.C;
  }

  // product table: tq[coord * 16 + nibble] = v(nibble) * q~_coord
  for (int i = tid; i < kDim * 16; i += blockDim.x) {
    const int coord = i >> 4, nib = i & 15;
    const float l = p.rp.lev[nib & 7];
    const float v = (nib & 8) ? -l : l;
    tq[i] = __fmul_rn(v, p.qt[(int64_t)sq * kDim + coord]);
  }
  // vote totals and totals of the chunks before this one
  const uint32_t* h = p.hist + (int64_t)sq * p.t.nchunk * kMaxBins;
  const int nch = (int)((p.N + kChunk - 1) / kChunk);
  for (int s = tid; s < kMaxBins; s += blockDim.x) {
    uint32_t tot = 0, bef = 0;
    if (s < p.nbins) {
      for (int cc = 0; cc < nch; ++cc) {
        const uint32_t x = h[(int64_t)cc * kMaxBins + s];
        tot += x;
        if (cc < c) bef += x;
      }
    }
    s_tot[s] = tot;
    s_bef[s] = bef;
  }
  __syncthreads();
  if (warp == 0) {
    // suffix sums from the top vote value down: lane l owns bins 255-8l .. 248-8l
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += s_tot[255 - 8 * lane - i];
    const uint32_t inc = warp_incl_scan(part, lane);
    const uint32_t exc = inc - part;
    // threshold T: largest value whose suffix count reaches C
    const bool here = exc < (uint32_t)p.C && inc >= (uint32_t)p.C;
    const unsigned ball = __ballot_sync(kFull, here);
    const int owner = __ffs(ball) - 1;
    if (lane == owner) {
      uint32_t run = exc;
      int T = 255 - 8 * lane;
      for (int i = 0; i < 8; ++i) {
        const int s = 255 - 8 * lane - i;
        if (run + s_tot[s] >= (uint32_t)p.C) {
          T = s;
          break;
        }
        run += s_tot[s];
      }
      s_info[0] = T;
      s_info[1] = (int64_t)p.C - run;  // keys equal to T to take
    }
  }
  __syncthreads();
  const int T = (int)max64(0, min64(kMaxBins - 1, s_info[0]));
  const int64_t quota = s_info[1];
  if (warp == 0) {
    uint32_t gt = 0;
    for (int s = T + 1 + lane; s < kMaxBins; s += 32) gt += s_bef[s];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gt += __shfl_xor_sync(kFull, gt, o);
    if (lane == 0) {
      const int64_t eq_bef = s_bef[T];
      s_info[2] = gt + min64(eq_bef, quota);  // candidates in earlier chunks
      s_info[3] = max64(0, quota - eq_bef);   // keys equal to T this chunk may take
    }
  }
  __syncthreads();
  const int64_t sel_before = s_info[2];
  const int64_t eq_allow = s_info[3];

  // ordered compaction: thread t owns keys [32t, 32t + 32)
  const uint8_t* vin = p.votes + (int64_t)sq * p.t.nchunk * kChunk + base;
  const int k0 = tid * 32;
  uint32_t vw[8];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = reinterpret_cast<const uint4*>(vin + k0)[i];
    vw[4 * i + 0] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
  }
  uint32_t n_eq = 0, n_gt = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t v = (vw[i >> 2] >> (8 * (i & 3))) & 0xffu;
    const bool in = k0 + i < len;
    n_eq += (in && v == (uint32_t)T) ? 1u : 0u;
    n_gt += (in && v > (uint32_t)T) ? 1u : 0u;
  }
  uint32_t tot_dummy;
  const uint32_t eq_rank0 = block_excl_scan(n_eq, tmp, &tot_dummy);
  const uint32_t eq_take = (uint32_t)max64(0, min64((int64_t)n_eq, eq_allow - (int64_t)eq_rank0));
  uint32_t nsel;
  const uint32_t pos0 = block_excl_scan(n_gt + eq_take, tmp, &nsel);
  {
    uint32_t pos = pos0, eq_seen = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
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

  // rerank the chunk's candidates, one thread per candidate
  const float qn = p.qnorm[sq];
  int32_t* cidx = p.cand_idx + (int64_t)sq * p.cmax + sel_before;
  float* cest = p.cand_est + (int64_t)sq * p.cmax + sel_before;
  const uint8_t* rec = p.t.rec + (sh * p.t.rcap + base) * kRecBytes;
  for (uint32_t r = tid; r < nsel; r += blockDim.x) {
    const uint32_t key = keys[r];
    const uint4* rp4 = reinterpret_cast<const uint4*>(rec + (int64_t)key * kRecBytes);
    uint32_t cw[16], ww[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = rp4[i];
      cw[4 * i] = x.x; cw[4 * i + 1] = x.y; cw[4 * i + 2] = x.z; cw[4 * i + 3] = x.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = rp4[4 + i];
      ww[4 * i] = x.x; ww[4 * i + 1] = x.y; ww[4 * i + 2] = x.z; ww[4 * i + 3] = x.w;
    }
    float dots[kSub];
#pragma unroll
    for (int b = 0; b < kSub; ++b) {
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < kM; ++j) {
        const uint32_t nib = (cw[b] >> (4 * j)) & 15u;
        dot = __fadd_rn(dot, tq[(b * kM + j) * 16 + nib]);
      }
      dots[b] = dot;
    }
    float acc = 0.f;
#pragma unroll
    for (int b = 0; b < kSub; ++b) acc = __fadd_rn(acc, __fmul_rn(__uint_as_float(ww[b]), dots[b]));
    cidx[r] = (int32_t)(p.sink + base + key);
    cest[r] = __fmul_rn(qn, acc);
  }
}

// ---------------------------------------------------------------------------
// Top-k: one block of 1024 threads per (sequence, query head).  Radix select
// (8-bit digits, most significant first) of the k-th largest order key of
// the estimates (ties among equal estimates go to the lower position), then
// an ordered compaction so the result lists positions in ascending order.
// ---------------------------------------------------------------------------
constexpr int kTopThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
  if (x == 0.f) x = 0.f;  // -0 and +0 compare equal
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkParams {
  int64_t C, k, k_eff, cmax;
  const int32_t* cand_idx;
  const float* cand_est;
  int32_t* out_idx;
  float* out_score;
};

__global__ void __launch_bounds__(kTopThreads) k_topk(TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t s_sel[2];
  const int sq = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* est = p.cand_est + (int64_t)sq * p.cmax;
  const int32_t* cid = p.cand_idx + (int64_t)sq * p.cmax;
  int32_t* oi = p.out_idx + (int64_t)sq * p.k;
  float* os = p.out_score ? p.out_score + (int64_t)sq * p.k : nullptr;
  const int64_t C = p.C;

  uint32_t kstar = 0;   // k-th largest key
  uint32_t need_eq = 0; // keys equal to kstar to keep
  if (p.k_eff < C) {
    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)p.k_eff;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      if (tid == 0) {
        s_sel[0] = 0;
        s_sel[1] = remaining;
      }
      __syncthreads();
      for (int64_t i = tid; i < C; i += blockDim.x) {
        const uint32_t key = order_key(est[i]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t part = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) part += hist[255 - 8 * lane - i];
        const uint32_t inc = warp_incl_scan(part, lane);
        const uint32_t exc = inc - part;
        const bool here = exc < remaining && inc >= remaining;
        const int owner = __ffs(__ballot_sync(kFull, here)) - 1;
        if (lane == owner) {
          uint32_t run = exc;
          int dsel = 255 - 8 * lane;
          for (int i = 0; i < 8; ++i) {
            const int dgt = 255 - 8 * lane - i;
            if (run + hist[dgt] >= remaining) {
              dsel = dgt;
              break;
            }
            run += hist[dgt];
          }
          s_sel[0] = (uint32_t)dsel;
          s_sel[1] = remaining - run;
        }
      }
      __syncthreads();
      prefix |= s_sel[0] << shift;
      mask |= 255u << shift;
      remaining = s_sel[1];
      __syncthreads();
    }
    kstar = prefix;
    need_eq = remaining;
  }
  // ordered compaction over contiguous slices
  const int64_t per = (C + blockDim.x - 1) / blockDim.x;
  const int64_t i0 = min64(C, tid * per), i1 = min64(C, i0 + per);
  const bool all = p.k_eff >= C;
  uint32_t n_eq = 0, n_gt = 0;
  if (!all) {
    for (int64_t i = i0; i < i1; ++i) {
      const uint32_t key = order_key(est[i]);
      n_gt += key > kstar;
      n_eq += key == kstar;
    }
  }
  uint32_t tot;
  const uint32_t eq_rank0 = block_excl_scan(n_eq, tmp, &tot);
  const uint32_t eq_take = (uint32_t)max64(0, min64(n_eq, (int64_t)need_eq - eq_rank0));
  const uint32_t cnt = all ? (uint32_t)(i1 - i0) : n_gt + eq_take;
  const uint32_t pos0 = block_excl_scan(cnt, tmp, &tot);
  uint32_t pos = pos0, eq_seen = 0;
  for (int64_t i = i0; i < i1; ++i) {
    const float e = est[i];
    bool take = true;
    if (!all) {
      const uint32_t key = order_key(e);
      take = key > kstar;
      if (key == kstar) {
        take = eq_seen < eq_take;
        ++eq_seen;
      }
    }
    if (take) {
      oi[pos] = cid[i];
      if (os) os[pos] = e;
      ++pos;
    }
  }
  for (int64_t i = p.k_eff + tid; i < p.k; i += blockDim.x) {
    oi[i] = -1;
    if (os) os[i] = -INFINITY;
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

cudaError_t launch_qprep(const void* q, int dtype, const RetrieveArgs& a, cudaStream_t st) {
  k_qprep<<<a.s.batch * a.s.hq, 256, 0, st>>>(q, dtype, a.sm, a.rho, a.flat, a.qt, a.qnorm, a.hot);
  return cudaGetLastError();
}

cudaError_t launch_vote(const RetrieveArgs& a, cudaStream_t st) {
  VoteParams vp;
  vp.t = a.t;
  vp.hq = a.s.hq;
  vp.g = a.s.g;
  vp.rho = a.rho;
  vp.nbins = a.nbins;
  vp.N = a.N;
  vp.hot = a.hot;
  vp.votes = a.votes;
  vp.hist = a.hist;
  const int nhot = kSub * a.rho;
  const size_t vsmem = (size_t)kChunk + (size_t)(3 * nhot + 1) * 4;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_vote, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_vote<<<dim3(a.nchunk_active, a.s.batch * a.s.hq), kVoteThreads, vsmem, st>>>(vp);
  return cudaGetLastError();
}

cudaError_t launch_select_rerank(const RetrieveArgs& a, cudaStream_t st) {
  SelectParams sp;
  sp.t = a.t;
  sp.rp = a.rp;
  sp.hq = a.s.hq;
  sp.g = a.s.g;
  sp.nbins = a.nbins;
  sp.sink = a.s.sink;
  sp.N = a.N;
  sp.C = a.C;
  sp.qt = a.qt;
  sp.qnorm = a.qnorm;
  sp.votes = a.votes;
  sp.hist = a.hist;
  sp.cand_idx = a.cand_idx;
  sp.cand_est = a.cand_est;
  sp.cmax = a.cmax;
  k_select_rerank<<<dim3(a.nchunk_active, a.s.batch * a.s.hq), kSelThreads, 0, st>>>(sp);
  return cudaGetLastError();
}

cudaError_t launch_topk(const RetrieveArgs& a, cudaStream_t st) {
  TopkParams tp;
  tp.C = a.C;
  tp.k = a.k;
  tp.k_eff = a.k_eff;
  tp.cmax = a.cmax;
  tp.cand_idx = a.cand_idx;
  tp.cand_est = a.cand_est;
  tp.out_idx = a.topk_idx;
  tp.out_score = a.topk_score;
  k_topk<<<a.s.batch * a.s.hq, kTopThreads, 0, st>>>(tp);
  return cudaGetLastError();
}

}  // namespace paris
