// C ABI of the ParisKV library (include/paris.h): context creation, zone
// bookkeeping, argument checks and kernel launches.  All arithmetic of the
// retrieval path runs in the kernels of kernels_*.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/paris.h"
#include "paris_internal.cuh"

using namespace paris;

struct paris_ctx {
  paris_config cfg;
  Shape s;
  int nbins;
  int64_t rcap, cmax;
  int nchunk, nsplit_max;
  SignMask sm;
  RsqParams rp;
  // zones
  int64_t T, N, n_local, n_buf, n_flushes;
  // storage
  KvStore kv;
  Tables t;
  void* host_store;  // pinned mapped allocation backing kv.st_k / kv.st_v (retrieval_on_host)
  float* qt;
  float* qnorm;
  uint32_t* hot;
  uint8_t* votes;
  uint32_t* hist;
  int32_t* cand_idx;
  float* cand_est;
  float* part;
  uint32_t* status;
  uint32_t* counters;  // [2][batch*Hq]: rerank blocks, attention splits finished
  float* dense_part;   // dense comparator: [batch*Hq][dense_splits_max][kPartStride]
  uint32_t* dense_counter;  // [batch*Hkv]
  int32_t* gqa_list;    // GQA-shared attention: [batch*Hkv][rcap] the union of the G top-k lists, by zone slice
  float* cent_table;    // learned centroids [Hkv][16][256][8] (used when t.cent points to it)
  int32_t* ord_idx;     // top-k by score: the decode kernel's [batch*Hq][topk] positions, ascending
  float* ord_sc;        // and their estimates, before the order kernel lists them best first
  int dense_splits_max, sm_count;
  uint64_t* trace;     // kTraceSlots phase timestamps
  bool tracing;        // PARIS_TRACE=1 in the environment at creation
  std::string err;
  // accounting
  int64_t launches[PARIS_KERNEL_COUNT];
  bool prof;
  int prof_max;
  std::vector<cudaEvent_t> prof_ev;  // 2 per timed launch
  std::vector<int> prof_slot;
};

namespace {

thread_local std::string g_create_err;

paris_status fail(paris_ctx* c, paris_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf; else g_create_err = buf;
  return st;
}

paris_status cuda_fail(paris_ctx* c, cudaError_t e, const char* what) {
  return fail(c, PARIS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define PARIS_CUDA(ctx, call)                                   \
  do {                                                          \
    cudaError_t e_ = (call);                                    \
    if (e_ != cudaSuccess) return cuda_fail((ctx), e_, #call);  \
  } while (0)

// Launch one kernel through `call`, counting it and, while profiling,
// bracketing it with events on its stream.
template <typename F>
cudaError_t launch(paris_ctx* c, int slot, cudaStream_t st, F&& call) {
  c->launches[slot] += 1;
  const bool timed = c->prof && (int)c->prof_slot.size() < c->prof_max;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (timed) {
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e != cudaSuccess) return e;
    // external records: inside a stream capture they become event-record
    // nodes of the graph, so the pair still times the kernel on replay
    e = cudaEventRecordWithFlags(e0, st, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = call();
  if (timed) {
    c->prof_ev.push_back(e0);
    c->prof_ev.push_back(e1);
    c->prof_slot.push_back(slot);
    if (e == cudaSuccess) e = cudaEventRecordWithFlags(e1, st, cudaEventRecordExternal);
  }
  return e;
}

int64_t candidate_count(int64_t n, int cand_bp, int64_t k) {
  int64_t c = (cand_bp * n + 9999) / 10000;
  if (c < std::min(k, n)) c = std::min(k, n);
  return std::min(c, n);
}

// Integral of cos^n over [0, th] by the reduction formula
//   F_n = cos^{n-1} sin / n + (n-1)/n F_{n-2},  F_0 = th, F_1 = sin th.
double cos_power_integral(int n, double th) {
  const double c = std::cos(th), s = std::sin(th);
  double f = (n % 2 == 0) ? th : s;
  for (int k = (n % 2 == 0) ? 2 : 3; k <= n; k += 2) f = std::pow(c, k - 1) * s / k + (double)(k - 1) / k * f;
  return f;
}

// Lloyd-Max levels of |x_j| for x uniform on S^{m-1}.  The density of |x_j|
// on [0, 1] is proportional to (1 - t^2)^((m-3)/2); with t = sin(th) the
// mass of a cell is the integral of cos^{m-2} and the first moment is
// (1 - t^2)^((m-1)/2) / (m - 1) evaluated at the cell ends (the common
// constant cancels in the conditional mean).  Starts from uniform levels and
// iterates "thresholds = midpoints, levels = cell means" to a fixed point.
void lloyd_max_levels(int m, double lev[8], double thr[7]) {
  const int n = 8;
  for (int t = 0; t < n; ++t) lev[t] = (t + 0.5) / n;
  for (int it = 0; it < 1000000; ++it) {
    double edges[9];
    edges[0] = 0.0;
    edges[n] = 1.0;
    for (int t = 1; t < n; ++t) edges[t] = 0.5 * (lev[t - 1] + lev[t]);
    double change = 0.0;
    for (int t = 0; t < n; ++t) {
      const double a = edges[t], b = edges[t + 1];
      const double mass = cos_power_integral(m - 2, std::asin(b)) - cos_power_integral(m - 2, std::asin(a));
      const double e = 0.5 * (m - 1);
      const double mom = (std::pow(1.0 - a * a, e) - std::pow(1.0 - b * b, e)) / (m - 1);
      const double nl = mom / mass;
      change = std::max(change, std::fabs(nl - lev[t]));
      lev[t] = nl;
    }
    if (change < 1e-15) break;
  }
  for (int t = 0; t + 1 < n; ++t) thr[t] = 0.5 * (lev[t] + lev[t + 1]);
}

void free_all(paris_ctx* c) {
  void* dev[] = {c->kv.win_k, c->kv.win_v, c->t.ids, c->t.rec, c->t.ent, c->t.off, c->qt, c->qnorm,
                 c->hot, c->votes, c->hist, c->cand_idx, c->cand_est, c->part, c->status,
                 c->counters, c->trace, c->dense_part, c->dense_counter, c->gqa_list,
                 c->cent_table, c->ord_idx, c->ord_sc};
  for (void* p : dev)
    if (p) cudaFree(p);
  if (c->host_store) {
    cudaFreeHost(c->host_store);
  } else {
    if (c->kv.st_k) cudaFree(c->kv.st_k);
    if (c->kv.st_v) cudaFree(c->kv.st_v);
  }
}

template <typename T>
paris_status dalloc(paris_ctx* c, T** p, size_t bytes, const char* what) {
  *p = nullptr;
  if (bytes == 0) bytes = 256;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    cudaGetLastError();
    return fail(c, PARIS_ENOMEM, "cudaMalloc(%s, %zu bytes): %s", what, bytes, cudaGetErrorString(e));
  }
  return PARIS_OK;
}

paris_status check_dtype(paris_ctx* c, int dtype) {
  if (dtype != PARIS_F32 && dtype != PARIS_BF16) return fail(c, PARIS_EINVAL, "dtype must be PARIS_F32 or PARIS_BF16");
  return PARIS_OK;
}

}  // namespace

namespace paris {

namespace {
constexpr int kSmemMaxDevices = 64;
std::mutex g_smem_mu;
bool g_smem_set[kSmemMaxDevices][kSmemKernelCount];
}  // namespace

cudaError_t set_smem_limit(const void* func, int bytes, SmemKernel which) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kSmemMaxDevices) return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(g_smem_mu);
  if (g_smem_set[dev][which]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_set[dev][which] = true;
  return e;
}

}  // namespace paris

namespace {

RetrieveArgs retrieve_args(paris_ctx* c, int32_t* topk_idx, float* topk_score) {
  RetrieveArgs a;
  a.s = c->s;
  a.t = c->t;
  a.sm = c->sm;
  a.rp = c->rp;
  a.rho = c->cfg.rho;
  a.flat = c->cfg.vote_weighting == PARIS_VOTE_FLAT;
  a.nbins = c->nbins;
  a.N = c->N;
  a.C = candidate_count(c->N, c->cfg.cand_bp, c->cfg.topk);
  a.k = c->cfg.topk;
  a.k_eff = std::min<int64_t>(a.k, a.C);
  a.nchunk_active = (int)((c->N + kChunk - 1) / kChunk);
  a.qt = c->qt;
  a.qnorm = c->qnorm;
  a.hot = c->hot;
  a.votes = c->votes;
  a.hist = c->hist;
  a.cand_idx = c->cand_idx;
  a.cand_est = c->cand_est;
  a.cmax = c->cmax;
  a.trace = c->tracing ? c->trace : nullptr;
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  return a;
}

AttendArgs attend_args(paris_ctx* c, const int32_t* topk_idx, void* out_bf16) {
  AttendArgs a;
  a.s = c->s;
  a.kv = c->kv;
  a.T = c->T;
  a.N = c->N;
  a.n_local_buf = c->n_local + c->n_buf;
  a.k = c->cfg.topk;
  a.k_eff = c->N > 0 ? std::min<int64_t>(a.k, candidate_count(c->N, c->cfg.cand_bp, c->cfg.topk)) : 0;
  a.topk_idx = topk_idx;
  a.part = c->part;
  a.nsplit_max = c->nsplit_max;
  a.status = c->status;
  a.counter = c->counters + (int64_t)c->s.batch * c->s.hq;
  a.trace = c->tracing ? c->trace : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out_bf16);
  return a;
}

// Advance the zone bookkeeping by one appended token; returns the number of
// tokens the append moved into the Retrieval zone (their chunks need a new
// index) and the Retrieval size before it.
int64_t zones_append(paris_ctx* c, int64_t* n_old) {
  const int64_t pos = c->T;
  c->T += 1;
  *n_old = c->N;
  if (pos < c->s.sink) return 0;
  c->n_buf += 1;
  if (c->n_buf < c->s.ubuf) return 0;
  c->n_local += c->n_buf;
  c->n_buf = 0;
  c->n_flushes += 1;
  const int64_t evict = std::max<int64_t>(0, c->n_local - c->s.local);
  c->N += evict;
  c->n_local -= evict;
  return evict;
}

// Would appending one token now move tokens into the Retrieval zone?
bool append_flushes(const paris_ctx* c) {
  if (c->T < c->s.sink) return false;
  if (c->n_buf + 1 < c->s.ubuf) return false;
  return c->n_local + c->n_buf + 1 > c->s.local;
}

// The step's own token, when the decode kernel appends it.
struct NewToken {
  const void* k;
  const void* v;
  paris_dtype dtype;
  int64_t pos;
};

// Retrieval (and, with out != nullptr, the sparse attention) of the current
// zones.  With `tok`, the zone bookkeeping already counts the token and the
// decode kernel writes it into the cache.  An empty Retrieval zone gives the
// (-1, -inf) fill; the attention then runs as its own kernel.
paris_status retrieve_launch(paris_ctx* c, const void* q, paris_dtype dtype, int32_t* topk_idx, float* topk_score,
                             int64_t* k_eff, const NewToken* tok, void* out, cudaStream_t s) {
  const int64_t nq = (int64_t)c->s.batch * c->s.hq;
  if (c->N == 0) {
    *k_eff = 0;
    if (tok) {
      const NewToken f = *tok;
      PARIS_CUDA(c, launch(c, PARIS_KERNEL_APPEND, s, [&] {
                   return launch_append(f.k, f.v, f.dtype, f.pos, c->s, c->kv, c->t, c->sm, c->rp, s);
                 }));
    }
    PARIS_CUDA(c, launch(c, PARIS_KERNEL_FILL, s,
                         [&] { return launch_fill_empty(topk_idx, topk_score, nq * c->cfg.topk, s); }));
    if (out) {
      const AttendArgs a = attend_args(c, topk_idx, out);
      PARIS_CUDA(c, launch(c, PARIS_KERNEL_ATTEND, s, [&] { return launch_attend(q, dtype, a, s); }));
    }
    return PARIS_OK;
  }
  // by score: the decode kernel writes position order to the context's
  // scratch and, at its end, lists it best first into the caller's arrays
  const bool by_score = c->cfg.topk_order == PARIS_TOPK_BY_SCORE;
  DecodeLaunch L;
  L.ra = by_score ? retrieve_args(c, c->ord_idx, c->ord_sc) : retrieve_args(c, topk_idx, topk_score);
  L.kv = c->kv;
  L.nsink = std::min<int64_t>(c->s.sink, c->T);
  L.nwin = L.nsink + c->n_local + c->n_buf;
  L.q = q;
  L.qdtype = dtype;
  L.k_new = tok ? tok->k : nullptr;
  L.v_new = tok ? tok->v : nullptr;
  L.kvdtype = tok ? tok->dtype : PARIS_BF16;
  L.new_pos = tok ? tok->pos : -1;
  L.status = c->status;
  L.out = static_cast<__nv_bfloat16*>(out);
  L.ord_idx = by_score ? topk_idx : nullptr;
  L.ord_sc = by_score ? topk_score : nullptr;
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_DECODE, s, [&] { return launch_decode(L, s); }));
  *k_eff = L.ra.k_eff;
  return PARIS_OK;
}

}  // namespace

extern "C" {

paris_status paris_rsq_levels(int m, double* levels, double* thresholds) {
  if (m < 2 || m > 64 || !levels || !thresholds) return fail(nullptr, PARIS_EINVAL, "paris_rsq_levels: bad arguments");
  lloyd_max_levels(m, levels, thresholds);
  return PARIS_OK;
}

paris_status paris_create(const paris_config* cfg, const int8_t* srht_signs, paris_ctx** out) {
  if (!out) return fail(nullptr, PARIS_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg || !srht_signs) return fail(nullptr, PARIS_EINVAL, "cfg and srht_signs must not be NULL");
  const paris_config& f = *cfg;
  if (f.head_dim != kDim || f.n_sub != kSub)
    return fail(nullptr, PARIS_EINVAL, "supported geometry: head_dim = 128, n_sub = 16 (got %d, %d)", f.head_dim, f.n_sub);
  if (f.batch < 1 || f.n_kv_heads < 1 || f.n_q_heads < f.n_kv_heads || f.n_q_heads % f.n_kv_heads)
    return fail(nullptr, PARIS_EINVAL, "batch >= 1 and n_q_heads a positive multiple of n_kv_heads required");
  if (f.vote_weighting != PARIS_VOTE_RANK && f.vote_weighting != PARIS_VOTE_FLAT)
    return fail(nullptr, PARIS_EINVAL, "unknown vote_weighting");
  const int rho_max = f.vote_weighting == PARIS_VOTE_RANK ? 15 : kCentroids;
  if (f.rho < 1 || f.rho > rho_max) return fail(nullptr, PARIS_EINVAL, "rho must be in [1, %d]", rho_max);
  if (f.sink < 0 || f.local < 0 || f.update_buf < 1 || f.topk < 1 || f.cand_bp < 1 || f.cand_bp > 10000 ||
      f.max_ctx < 0)
    return fail(nullptr, PARIS_EINVAL, "sink, local >= 0; update_buf, topk >= 1; cand_bp in [1, 10000]; max_ctx >= 0");
  if (f.topk_order != PARIS_TOPK_BY_SCORE && f.topk_order != PARIS_TOPK_BY_POSITION)
    return fail(nullptr, PARIS_EINVAL, "unknown topk_order");
  if (f.topk_order == PARIS_TOPK_BY_SCORE && f.topk > kOrderMax)
    return fail(nullptr, PARIS_EINVAL, "topk above %lld needs topk_order = PARIS_TOPK_BY_POSITION", (long long)kOrderMax);
  for (int i = 0; i < kDim; ++i)
    if (srht_signs[i] != 1 && srht_signs[i] != -1) return fail(nullptr, PARIS_EINVAL, "srht_signs[%d] is not +-1", i);

  paris_ctx* c = new (std::nothrow) paris_ctx();
  if (!c) return fail(nullptr, PARIS_ENOMEM, "host allocation failed");
  c->cfg = f;
  c->s = Shape{f.batch, f.n_kv_heads, f.n_q_heads, f.n_q_heads / f.n_kv_heads, f.sink, f.local, f.update_buf};
  c->nbins = (f.vote_weighting == PARIS_VOTE_RANK ? f.rho * kSub : kSub) + 1;
  c->rcap = std::max<int64_t>(0, (int64_t)f.max_ctx - f.sink);
  c->nchunk = (int)std::max<int64_t>(1, (c->rcap + kChunk - 1) / kChunk);
  if (c->nchunk > kMaxChunks) {
    delete c;
    return fail(nullptr, PARIS_EINVAL, "max_ctx - sink must be at most %d tokens", kMaxChunks * kChunk);
  }
  // rows of the candidate arrays start on 16-byte boundaries (staged by 16-byte copies)
  c->cmax = (std::max<int64_t>(1, candidate_count(c->rcap, f.cand_bp, f.topk)) + 3) / 4 * 4;
  c->nsplit_max = (int)((f.sink + f.local + f.update_buf + f.topk + kAttnSplit - 1) / kAttnSplit) + 1;
  if (c->nsplit_max > kMaxSplits) {
    delete c;
    return fail(nullptr, PARIS_EINVAL, "sink + local + update_buf + topk must be at most %d rows",
                (kMaxSplits - 1) * kAttnSplit);
  }
  std::memset(&c->sm, 0, sizeof c->sm);
  for (int i = 0; i < kDim; ++i)
    if (srht_signs[i] < 0) c->sm.w[i >> 5] |= 1u << (i & 31);
  double lev[8], thr[7];
  lloyd_max_levels(kM, lev, thr);
  for (int i = 0; i < 8; ++i) c->rp.lev[i] = (float)lev[i];
  for (int i = 0; i < 7; ++i) c->rp.thr[i] = (float)thr[i];
  c->rp.sqrtd = std::sqrt((float)kDim);

  const int64_t bh = (int64_t)f.batch * f.n_kv_heads;
  const int64_t bq = (int64_t)f.batch * f.n_q_heads;
  c->kv.win = f.sink + f.local + f.update_buf;
  c->kv.rcap = c->rcap;
  c->t.rcap = c->rcap;
  c->t.nchunk = c->nchunk;
  const size_t row = (size_t)kDim * sizeof(__nv_bfloat16);
  paris_status st = PARIS_OK;
#define TRY(x)                   \
  if ((st = (x)) != PARIS_OK) {  \
    g_create_err = c->err;       \
    free_all(c);                 \
    delete c;                    \
    return st;                   \
  }
  TRY(dalloc(c, &c->kv.win_k, bh * c->kv.win * row, "window K"));
  TRY(dalloc(c, &c->kv.win_v, bh * c->kv.win * row, "window V"));
  const size_t store_bytes = (size_t)bh * c->rcap * row;
  if (f.retrieval_on_host) {
    cudaError_t e = cudaHostAlloc(&c->host_store, 2 * store_bytes + 512, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      c->host_store = nullptr;
      TRY(fail(c, PARIS_ENOMEM, "cudaHostAlloc(Retrieval K/V, %zu bytes): %s", 2 * store_bytes, cudaGetErrorString(e)));
    }
    void* dptr = nullptr;
    e = cudaHostGetDevicePointer(&dptr, c->host_store, 0);
    if (e != cudaSuccess) TRY(cuda_fail(c, e, "cudaHostGetDevicePointer"));
    c->kv.st_k = static_cast<__nv_bfloat16*>(dptr);
    c->kv.st_v = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(dptr) + ((store_bytes + 255) / 256) * 256);
  } else {
    TRY(dalloc(c, &c->kv.st_k, store_bytes, "Retrieval K"));
    TRY(dalloc(c, &c->kv.st_v, store_bytes, "Retrieval V"));
  }
  TRY(dalloc(c, &c->t.ids, (size_t)bh * c->rcap * kSub, "bucket ids"));
  TRY(dalloc(c, &c->t.rec, (size_t)bh * c->rcap * kRecBytes, "codes and w"));
  // 16 spare bytes: list copies round their last 16-byte piece up
  TRY(dalloc(c, &c->t.ent, (size_t)bh * c->nchunk * kSub * kChunk * sizeof(uint16_t) + 16, "bucket lists"));
  TRY(dalloc(c, &c->t.off, (size_t)bh * c->nchunk * kSub * kOffStride * sizeof(uint32_t), "bucket offsets"));
  TRY(dalloc(c, &c->qt, (size_t)bq * kDim * sizeof(float), "q~"));
  TRY(dalloc(c, &c->qnorm, (size_t)bq * sizeof(float), "||q||"));
  TRY(dalloc(c, &c->hot, (size_t)bq * kSub * f.rho * sizeof(uint32_t), "hot centroids"));
  TRY(dalloc(c, &c->votes, (size_t)bq * c->nchunk * kChunk, "votes"));
  TRY(dalloc(c, &c->hist, (size_t)bq * c->nchunk * kMaxBins * sizeof(uint32_t), "vote histograms"));
  TRY(dalloc(c, &c->cand_idx, (size_t)bq * c->cmax * sizeof(int32_t), "candidates"));
  TRY(dalloc(c, &c->cand_est, (size_t)bq * c->cmax * sizeof(float), "candidate estimates"));
  TRY(dalloc(c, &c->part, (size_t)bq * c->nsplit_max * kPartStride * sizeof(float), "attention partials"));
  TRY(dalloc(c, &c->status, sizeof(uint32_t), "status word"));
  TRY(dalloc(c, &c->counters, (size_t)2 * bq * sizeof(uint32_t), "block counters"));
  {
    int dev = 0;
    c->sm_count = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      c->sm_count = 1;
    }
    c->dense_splits_max = std::max(1, c->sm_count);  // splits per (sequence, KV head), at most one per SM
  }
  TRY(dalloc(c, &c->dense_part, (size_t)bq * c->dense_splits_max * kPartStride * sizeof(float), "dense partials"));
  TRY(dalloc(c, &c->dense_counter, (size_t)bq * sizeof(uint32_t), "dense counters"));
  TRY(dalloc(c, &c->gqa_list, (size_t)bh * c->rcap * sizeof(int32_t), "top-k unions"));
  TRY(dalloc(c, &c->cent_table, (size_t)f.n_kv_heads * kTabPerHead * sizeof(float), "centroid table"));
  if (f.topk_order == PARIS_TOPK_BY_SCORE) {
    TRY(dalloc(c, &c->ord_idx, (size_t)bq * f.topk * sizeof(int32_t), "top-k positions before ordering"));
    TRY(dalloc(c, &c->ord_sc, (size_t)bq * f.topk * sizeof(float), "top-k estimates before ordering"));
  }
  {
    const char* env = std::getenv("PARIS_TRACE");
    c->tracing = env != nullptr && env[0] == '1';
  }
  TRY(dalloc(c, &c->trace, (c->tracing ? kTraceWords : kTraceSlots) * sizeof(uint64_t), "phase trace"));
  cudaError_t e = cudaMemset(c->status, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->counters, 0, (size_t)2 * bq * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->dense_counter, 0, (size_t)bq * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->trace, 0, (c->tracing ? kTraceWords : kTraceSlots) * sizeof(uint64_t));
  if (e != cudaSuccess) TRY(cuda_fail(c, e, "initialising the context"));
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) TRY(cuda_fail(c, e, "cudaDeviceSynchronize"));
#undef TRY
  *out = c;
  return PARIS_OK;
}

void paris_destroy(paris_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  for (cudaEvent_t e : ctx->prof_ev) cudaEventDestroy(e);
  free_all(ctx);
  delete ctx;
}

paris_status paris_encode_prefill(paris_ctx* c, const void* K, const void* V, paris_dtype dtype, int64_t T,
                                  void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (c->T != 0) return fail(c, PARIS_ESTATE, "prefill needs an empty context (T = %lld)", (long long)c->T);
  if (T < 0) return fail(c, PARIS_EINVAL, "T must be >= 0");
  if (T > c->cfg.max_ctx) return fail(c, PARIS_ECAPACITY, "T = %lld exceeds max_ctx = %d", (long long)T, c->cfg.max_ctx);
  if (T > 0 && (!K || !V)) return fail(c, PARIS_EINVAL, "K and V must not be NULL");
  const int64_t rest = std::max<int64_t>(0, T - c->s.sink);
  const int64_t n_local = std::min<int64_t>(c->s.local, rest);
  const int64_t N = rest - n_local;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T > 0)
    PARIS_CUDA(c, launch(c, PARIS_KERNEL_PLACE_KV, s, [&] { return launch_place_kv(K, V, dtype, T, N, c->s, c->kv, s); }));
  if (T > c->s.sink)
    PARIS_CUDA(c, launch(c, PARIS_KERNEL_ENCODE, s,
                         [&] { return launch_encode(K, dtype, T, c->s.sink, T, c->s, c->t, c->sm, c->rp, s); }));
  if (N > 0)
    PARIS_CUDA(c, launch(c, PARIS_KERNEL_BUILD_INDEX, s, [&] {
                 return launch_build_index(N, 0, (int)((N + kChunk - 1) / kChunk), c->s, c->t, s);
               }));
  c->T = T;
  c->N = N;
  c->n_local = n_local;
  c->n_buf = 0;
  return PARIS_OK;
}

paris_status paris_append_decode(paris_ctx* c, const void* k, const void* v, paris_dtype dtype, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!k || !v) return fail(c, PARIS_EINVAL, "k and v must not be NULL");
  if (c->T + 1 > c->cfg.max_ctx) return fail(c, PARIS_ECAPACITY, "cache is full (max_ctx = %d)", c->cfg.max_ctx);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t pos = c->T;
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_APPEND, s,
                       [&] { return launch_append(k, v, dtype, pos, c->s, c->kv, c->t, c->sm, c->rp, s); }));
  int64_t n_old;
  // flush: the buffer joins Local, Local's oldest tokens beyond L join Retrieval
  if (zones_append(c, &n_old) == 0) return PARIS_OK;
  const int64_t n_new = c->N;
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_BUILD_INDEX, s, [&] {
               return launch_build_index(n_new, (int)(n_old / kChunk), (int)((n_new + kChunk - 1) / kChunk), c->s, c->t, s);
             }));
  return PARIS_OK;
}

paris_status paris_retrieve(paris_ctx* c, const void* q, paris_dtype dtype, int32_t* topk_idx, float* topk_score,
                            int64_t* k_eff, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!q || !topk_idx || !k_eff) return fail(c, PARIS_EINVAL, "q, topk_idx and k_eff must not be NULL");
  return retrieve_launch(c, q, dtype, topk_idx, topk_score, k_eff, nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

paris_status paris_sparse_attend(paris_ctx* c, const void* q, paris_dtype dtype, const int32_t* topk_idx,
                                 void* out_bf16, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!q || !out_bf16 || (!topk_idx && c->N > 0)) return fail(c, PARIS_EINVAL, "q, topk_idx and out must not be NULL");
  const AttendArgs a = attend_args(c, topk_idx, out_bf16);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_ATTEND, s, [&] { return launch_attend(q, dtype, a, s); }));
  return PARIS_OK;
}

paris_status paris_sparse_attend_gqa(paris_ctx* c, const void* q, paris_dtype dtype, const int32_t* topk_idx,
                                     void* out_bf16, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!q || !out_bf16 || (!topk_idx && c->N > 0)) return fail(c, PARIS_EINVAL, "q, topk_idx and out must not be NULL");
  if (c->s.g > 16) return fail(c, PARIS_EINVAL, "paris_sparse_attend_gqa: at most 16 query heads per KV head");
  const int64_t k = c->cfg.topk;
  const int64_t k_eff = c->N > 0 ? std::min<int64_t>(k, candidate_count(c->N, c->cfg.cand_bp, k)) : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DenseArgs a;
  a.s = c->s;
  a.kv = c->kv;
  a.N = c->N;
  a.q = q;
  a.qdtype = dtype;
  a.qscale = 1.4426950408889634f / std::sqrt((float)kDim);
  a.part = c->dense_part;
  a.nsplit_max = c->dense_splits_max;
  a.counter = c->dense_counter;
  a.out = static_cast<__nv_bfloat16*>(out_bf16);
  a.topk = topk_idx;
  a.k = k;
  a.k_eff = k_eff;
  a.ulist = c->gqa_list;
  a.status = c->status;
  a.nsink = std::min<int64_t>(c->cfg.sink, c->T);
  a.nwin = a.nsink + c->n_local + c->n_buf;
  a.T = a.nwin + (int64_t)c->s.g * k_eff;
  a.rows_per_split = 0;
  const int nsplit = std::min(dense_union_splits(a, c->sm_count), c->dense_splits_max);
  if ((a.N + nsplit - 1) / nsplit > (int64_t)8 * 200 * 1024)
    return fail(c, PARIS_EINVAL, "paris_sparse_attend_gqa: Retrieval zone too long for %d splits", nsplit);
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_DENSE, s, [&] { return launch_dense(a, nsplit, s); }));
  return PARIS_OK;
}

paris_status paris_set_centroids(paris_ctx* c, const float* centroids, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  if (c->T > 0) return fail(c, PARIS_ESTATE, "paris_set_centroids: the cache must be empty (call it before prefill)");
  if (!centroids) {
    c->t.cent = nullptr;
    return PARIS_OK;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PARIS_CUDA(c, cudaMemcpyAsync(c->cent_table, centroids, (size_t)c->s.hkv * kTabPerHead * sizeof(float),
                                cudaMemcpyDeviceToDevice, s));
  c->t.cent = c->cent_table;
  return PARIS_OK;
}

paris_status paris_dense_attend(paris_ctx* c, const void* q, paris_dtype dtype, void* out_bf16, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!q || !out_bf16) return fail(c, PARIS_EINVAL, "q and out must not be NULL");
  if (c->s.g > 16) return fail(c, PARIS_EINVAL, "paris_dense_attend: at most 16 query heads per KV head");
  DenseArgs a;
  a.s = c->s;
  a.kv = c->kv;
  a.T = c->T;
  a.N = c->N;
  a.q = q;
  a.qdtype = dtype;
  a.qscale = 1.4426950408889634f / std::sqrt((float)kDim);
  a.part = c->dense_part;
  a.nsplit_max = c->dense_splits_max;
  a.counter = c->dense_counter;
  a.out = static_cast<__nv_bfloat16*>(out_bf16);
  a.topk = nullptr;
  a.k = a.k_eff = 0;
  a.ulist = nullptr;
  a.status = c->status;
  a.nsink = a.nwin = 0;
  int nsplit = dense_splits(a, c->sm_count);
  a.rows_per_split = dense_rows_per_split(std::max<int64_t>(1, c->T), nsplit);
  nsplit = (int)std::max<int64_t>(1, (c->T + a.rows_per_split - 1) / a.rows_per_split);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_DENSE, s, [&] { return launch_dense(a, nsplit, s); }));
  return PARIS_OK;
}

paris_status paris_decode_step(paris_ctx* c, const void* k, const void* v, paris_dtype kv_dtype, const void* q,
                               paris_dtype q_dtype, int32_t* topk_idx, float* topk_score, void* out_bf16,
                               int64_t* k_eff, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, kv_dtype);
  if (st == PARIS_OK) st = check_dtype(c, q_dtype);
  if (st != PARIS_OK) return st;
  if (!k || !v || !q || !topk_idx || !out_bf16 || !k_eff)
    return fail(c, PARIS_EINVAL, "k, v, q, topk_idx, out and k_eff must not be NULL");
  if (c->T + 1 > c->cfg.max_ctx) return fail(c, PARIS_ECAPACITY, "cache is full (max_ctx = %d)", c->cfg.max_ctx);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (append_flushes(c)) {
    // the flush re-indexes chunks the retrieval reads: append first
    st = paris_append_decode(c, k, v, kv_dtype, stream);
    if (st != PARIS_OK) return st;
    return retrieve_launch(c, q, q_dtype, topk_idx, topk_score, k_eff, nullptr, out_bf16, s);
  }
  const NewToken tok{k, v, kv_dtype, c->T};
  int64_t n_old;
  zones_append(c, &n_old);
  return retrieve_launch(c, q, q_dtype, topk_idx, topk_score, k_eff, &tok, out_bf16, s);
}

paris_status paris_get_state(const paris_ctx* c, paris_state* out) {
  if (!c || !out) return fail(nullptr, PARIS_EINVAL, "ctx and out must not be NULL");
  out->T = c->T;
  out->N = c->N;
  out->n_local = c->n_local;
  out->n_buf = c->n_buf;
  out->C = c->N > 0 ? candidate_count(c->N, c->cfg.cand_bp, c->cfg.topk) : 0;
  out->k_eff = std::min<int64_t>(c->cfg.topk, out->C);
  out->n_flushes = c->n_flushes;
  return PARIS_OK;
}

paris_status paris_check_device(paris_ctx* c) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  PARIS_CUDA(c, cudaDeviceSynchronize());
  uint32_t w = 0;
  PARIS_CUDA(c, cudaMemcpy(&w, c->status, sizeof w, cudaMemcpyDeviceToHost));
  if (w) {
    PARIS_CUDA(c, cudaMemset(c->status, 0, sizeof w));
    return fail(c, PARIS_EDEVICE, "device status word 0x%x (bit 0: token index outside the Retrieval zone)", w);
  }
  return PARIS_OK;
}

paris_status paris_debug_dump(paris_ctx* c, int what, int seq, int head, void* dst, size_t bytes) {
  if (!c || !dst) return fail(nullptr, PARIS_EINVAL, "ctx and dst must not be NULL");
  PARIS_CUDA(c, cudaDeviceSynchronize());
  const bool kv_head = what == PARIS_DUMP_IDS || what == PARIS_DUMP_CODES || what == PARIS_DUMP_W || what == PARIS_DUMP_KV;
  const int nh = kv_head ? c->s.hkv : c->s.hq;
  if (what != PARIS_DUMP_LEVELS && (seq < 0 || seq >= c->s.batch || head < 0 || head >= nh))
    return fail(c, PARIS_EINVAL, "seq/head out of range");
  const int64_t sh = (int64_t)seq * nh + head;
  const int64_t N = c->N;
  const int64_t C = N > 0 ? candidate_count(N, c->cfg.cand_bp, c->cfg.topk) : 0;
  auto need = [&](size_t n) -> paris_status {
    if (bytes < n) return fail(c, PARIS_EINVAL, "dst too small: %zu < %zu bytes", bytes, n);
    return PARIS_OK;
  };
  paris_status st;
  switch (what) {
    case PARIS_DUMP_IDS:
      if ((st = need(N * kSub)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->t.ids + sh * c->rcap * kSub, N * kSub, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_CODES:
    case PARIS_DUMP_W: {
      if ((st = need(what == PARIS_DUMP_CODES ? N * kDim / 2 : N * kSub * 4)) != PARIS_OK) return st;
      std::vector<uint8_t> rec((size_t)N * kRecBytes);
      if (N) PARIS_CUDA(c, cudaMemcpy(rec.data(), c->t.rec + sh * c->rcap * kRecBytes, rec.size(), cudaMemcpyDeviceToHost));
      uint8_t* d = static_cast<uint8_t*>(dst);
      for (int64_t i = 0; i < N; ++i) {
        if (what == PARIS_DUMP_CODES) std::memcpy(d + i * 64, rec.data() + i * kRecBytes, 64);
        else std::memcpy(d + i * 64, rec.data() + i * kRecBytes + 64, 64);
      }
      return PARIS_OK;
    }
    case PARIS_DUMP_VOTES:
      if ((st = need(N)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->votes + sh * c->nchunk * kChunk, N, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_CANDS:
      if ((st = need(C * 4)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->cand_idx + sh * c->cmax, C * 4, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_CAND_EST:
      if ((st = need(C * 4)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->cand_est + sh * c->cmax, C * 4, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_QT:
      if ((st = need(kDim * 4)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->qt + sh * kDim, kDim * 4, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_QNORM:
      if ((st = need(4)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->qnorm + sh, 4, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    case PARIS_DUMP_HOT: {
      const size_t n = (size_t)kSub * c->cfg.rho * 4;
      if ((st = need(n)) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->hot + sh * kSub * c->cfg.rho, n, cudaMemcpyDeviceToHost));
      return PARIS_OK;
    }
    case PARIS_DUMP_LEVELS: {
      if ((st = need(15 * 4)) != PARIS_OK) return st;
      float* d = static_cast<float*>(dst);
      for (int i = 0; i < 8; ++i) d[i] = c->rp.lev[i];
      for (int i = 0; i < 7; ++i) d[8 + i] = c->rp.thr[i];
      return PARIS_OK;
    }
    case PARIS_DUMP_KV: {
      const int64_t T = c->T;
      const size_t rowb = kDim * 2;
      if ((st = need(2 * T * rowb)) != PARIS_OK) return st;
      uint8_t* d = static_cast<uint8_t*>(dst);
      const int ring = c->s.local + c->s.ubuf;
      for (int kvsel = 0; kvsel < 2; ++kvsel) {
        const __nv_bfloat16* win = kvsel ? c->kv.win_v : c->kv.win_k;
        const __nv_bfloat16* sto = kvsel ? c->kv.st_v : c->kv.st_k;
        for (int64_t p = 0; p < T; ++p) {
          const __nv_bfloat16* src;
          if (p < c->s.sink) src = win + (sh * c->kv.win + p) * kDim;
          else if (p < c->s.sink + N) src = sto + (sh * c->rcap + (p - c->s.sink)) * kDim;
          else src = win + (sh * c->kv.win + c->s.sink + (p - c->s.sink) % ring) * kDim;
          PARIS_CUDA(c, cudaMemcpy(d + ((size_t)kvsel * T + p) * rowb, src, rowb, cudaMemcpyDefault));
        }
      }
      return PARIS_OK;
    }
    case PARIS_DUMP_TRACE: {
      const size_t n = (size_t)(c->tracing ? kTraceWords : kTraceSlots) * sizeof(uint64_t);
      if ((st = need(std::min(n, bytes))) != PARIS_OK) return st;
      PARIS_CUDA(c, cudaMemcpy(dst, c->trace, std::min(n, bytes), cudaMemcpyDeviceToHost));
      return PARIS_OK;
    }
    default:
      return fail(c, PARIS_EINVAL, "unknown dump %d", what);
  }
}

paris_status paris_launch_counts(const paris_ctx* c, int64_t* counts) {
  if (!c || !counts) return fail(nullptr, PARIS_EINVAL, "ctx and counts must not be NULL");
  for (int i = 0; i < PARIS_KERNEL_COUNT; ++i) counts[i] = c->launches[i];
  return PARIS_OK;
}

paris_status paris_profile_begin(paris_ctx* c, int max_launches) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  if (max_launches < 0) return fail(c, PARIS_EINVAL, "max_launches must be >= 0");
  if (c->prof) return fail(c, PARIS_ESTATE, "profiling already active");
  c->prof = true;
  c->prof_max = max_launches;
  c->prof_ev.clear();
  c->prof_slot.clear();
  c->prof_ev.reserve(2 * (size_t)max_launches);
  c->prof_slot.reserve(max_launches);
  return PARIS_OK;
}

paris_status paris_profile_end(paris_ctx* c, double* total_ms, int64_t* launches) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  if (!c->prof) return fail(c, PARIS_ESTATE, "profiling not active");
  c->prof = false;
  cudaError_t first = cudaDeviceSynchronize();
  double ms[PARIS_KERNEL_COUNT] = {0};
  int64_t n[PARIS_KERNEL_COUNT] = {0};
  for (size_t i = 0; i < c->prof_slot.size(); ++i) {
    float t = 0.f;
    cudaError_t e = cudaEventElapsedTime(&t, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]);
    if (e == cudaSuccess) {
      ms[c->prof_slot[i]] += t;
      n[c->prof_slot[i]] += 1;
    } else if (first == cudaSuccess) {
      first = e;
    }
  }
  for (cudaEvent_t e : c->prof_ev) cudaEventDestroy(e);
  c->prof_ev.clear();
  c->prof_slot.clear();
  for (int i = 0; i < PARIS_KERNEL_COUNT; ++i) {
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = n[i];
  }
  if (first != cudaSuccess) return cuda_fail(c, first, "profile events");
  return PARIS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Sparse attention without per-call scratch of the context
// ---------------------------------------------------------------------------
namespace {

// Scratch of paris_sparse_attend_noalloc: one float row of kPartStride per
// (sequence, query head, split) for the split partials, then one counter per
// (sequence, query head) for the merge.  Compiled into the library, so every
// GPU that loads it holds these ~545 KB until the process exits.
constexpr int kNoAllocPartRows = 1024;
constexpr int kNoAllocHeads = 1024;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocPartRows * kPartStride + kNoAllocHeads];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
paris_status noalloc_scratch(paris_ctx* c, float** out) {
  int dev = 0;
  PARIS_CUDA(c, cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(c, PARIS_EINVAL, "device %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetSymbolAddress(attention scratch)");
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return PARIS_OK;
}

}  // namespace

extern "C" {

paris_status paris_sparse_attend_noalloc(paris_ctx* c, const void* q, paris_dtype dtype, const int32_t* topk_idx,
                                         void* out_bf16, void* stream) {
  if (!c) return fail(nullptr, PARIS_EINVAL, "ctx is NULL");
  paris_status st = check_dtype(c, dtype);
  if (st != PARIS_OK) return st;
  if (!q || !out_bf16 || (!topk_idx && c->N > 0)) return fail(c, PARIS_EINVAL, "q, topk_idx and out must not be NULL");
  AttendArgs a = attend_args(c, topk_idx, out_bf16);
  const int nsplit = attend_splits(a);
  const int64_t bq = (int64_t)c->s.batch * c->s.hq;
  if (bq * nsplit > kNoAllocPartRows || bq > kNoAllocHeads)
    return fail(c, PARIS_EINVAL,
                "paris_sparse_attend_noalloc: batch x query heads x splits = %lld x %d exceeds its fixed scratch of "
                "%d rows (splits = ceil((sink + local + buffer + k) / %d))",
                (long long)bq, nsplit, kNoAllocPartRows, kAttnSplit);
  float* scratch = nullptr;
  st = noalloc_scratch(c, &scratch);
  if (st != PARIS_OK) return st;
  a.part = scratch;
  a.nsplit_max = nsplit;
  a.counter = reinterpret_cast<uint32_t*>(scratch + (size_t)kNoAllocPartRows * kPartStride);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the merge counters must start at zero (the partial rows are always written before they are read)
  PARIS_CUDA(c, cudaMemsetAsync(a.counter, 0, (size_t)bq * sizeof(uint32_t), s));
  PARIS_CUDA(c, launch(c, PARIS_KERNEL_ATTEND, s, [&] { return launch_attend(q, dtype, a, s); }));
  return PARIS_OK;
}

const char* paris_last_error(const paris_ctx* c) { return c ? c->err.c_str() : g_create_err.c_str(); }

}  // extern "C"
