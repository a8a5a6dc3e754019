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
// One thread-block cluster of CS <= 4 blocks (1024 threads, one per SM) per
// (sequence, query head); block r owns a contiguous range of index chunks
// of the Retrieval zone, so block order is position order.  What a block
// hands to the others it stores straight into their shared memory before a
// cluster barrier.  Five barriers separate the steps (four without attention):
//   1. each block: q~, ||q|| and the hot centroids (redundantly), the votes
//      of its chunks and their histogram, pushed to every block;
//   2. barrier; every block sums the histograms, finds the vote threshold
//      and writes its candidates (positions ascending) at their place in the
//      query head's list;
//   3. barrier; block r estimates its slice [C r / CS, C (r + 1) / CS) of
//      the list and pushes the order keys of the
//      estimates (and their range) to every block;
//   4. barrier; every block finds the k-th best key over all C (a counting
//      pass in shared memory; with far more candidates than a block holds,
//      a search the cluster shares, two more barriers), counts the entries
//      taken before its slice and writes the ones its slice takes at their
//      place in the top-k (and, for the list best first, at their rank in
//      it), and pushes their count to every block;
//   5. barrier; those rows, topped up with window rows to an even share of
//      all rows, are the block's attention rows, staged in rounds of 128
//      rows, two rounds in flight, every warp copying and scoring its own 4
//      rows of a round (no block barrier between rounds) with its own online
//      softmax; the block's partial goes to block 0;
//   6. barrier; block 0 merges the partials (where step 4 could not rank
//      the entries, the last block sorts the list best first meanwhile).
// The cluster size CS is chosen per launch from the waves of clusters the
// grid needs (decode_cluster_size).
// A decode token appended in the same step is read from the caller's k/v
// where the attention needs it, and written to the cache by one warp while
// the query is prepared (nothing in this launch reads the slots it writes).
#include <float.h>

#include <mutex>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kClusterMax = 4;
constexpr int kVoteSlots = 2;       // chunks per block whose votes stay in shared memory
constexpr int kListCap = 4032;      // candidates of the block's slice kept in shared memory
constexpr int kTile = 64;           // attention rows per pipeline stage
constexpr int kStages = 4;
constexpr int kSelCap = 16384;      // candidates whose order keys every block of the cluster holds
constexpr int kSelBins = 2048;      // 11-bit radix digits
constexpr int kBinRank = 64;        // keys left in the k-th digit that are ranked directly
constexpr int kSharedSelectMin = 24576;  // candidates past which the cluster shares the k-th key search
constexpr int kRowTab = kSelCap / 2;  // attention rows whose sources are resolved into a table
static_assert(kTile * 16 == kThreads, "16 threads per staged row");
static_assert(2 * kWarps == kTile, "two rows of a tile per warp");
static_assert(kChunk / kThreads == 16, "one 16-byte vote vector per thread and chunk");
static_assert(2 * kThreads == kSelBins, "two radix digits per thread");
static_assert(kMaxBins % 32 == 0 && kMaxBins <= kThreads, "one thread per vote value, whole warps");

// byte offsets inside the phase-shared dynamic region
constexpr int kUVotes = 0;                                    // u8 [kVoteSlots][kChunk]
constexpr int kUOffs = kUVotes + kVoteSlots * kChunk;         // u32 [kVoteSlots][kSub][kOffStride]
constexpr int kWarpBins = 64;                                 // per-warp counts of votes 8 .. 71
constexpr int kUWarpHist = kUOffs + kVoteSlots * kSub * kOffStride * 4;  // u32 [kWarps][kWarpBins]
constexpr int kUHot = kUWarpHist + kWarps * kWarpBins * 4;    // hot lists: hv[nhot], then per list
                                                              // (G x nhot) hbeg, hwt, hpre (+1), hsm
constexpr int kURecSlots = 0;                                 // 128 B per thread: a candidate record being gathered
constexpr int kUStageK = 0;                                   // bf16 [kStages][kTile][kDim], pieces permuted (spiece)
constexpr int kUStageV = kStages * kTile * kDim * 2;
constexpr int kUAttnEnd = 2 * kStages * kTile * kDim * 2;
constexpr int kUSelHist = kUStageK + kStages / 2 * kTile * kDim * 2;  // u32 [kSelBins], then u32 [kBinRank]:
                                                              // in the K rows of the second attention round
constexpr int kUSelPos = kUSelHist + (kSelBins + kBinRank) * 4;  // i32 [kListCap]: positions the block's slice takes
constexpr int kUBStart = 0;                                   // u32 [kSelBins]: keys above each linear bin
constexpr int kUBucket = kUSelPos + kListCap * 4;             // u16 [kSelCap]: the taken keys' indexes, by bin
// The k-th key search over keys that are not all in shared memory (C > kSelCap)
// shares the work across the cluster: each block's own keys, every block's
// histogram, and the keys of the k-th bin with their candidate numbers.
constexpr int kUHall = 0;                                     // u32 [kClusterMax][kSelBins]
constexpr int kUOwn = kUSelPos + kListCap * 4;                // u32 [kOwnCap]: the block's slice's order keys
constexpr int kOwnCap = (kUAttnEnd - kUOwn) / 4;
constexpr int kUBinEnt = kUAttnEnd;                           // u32 [kBinRank][2]: (key, candidate number)
constexpr int kUKeys = kUAttnEnd;                             // u32 [kSelCap]: order keys of all C estimates,
                                                              // then i64 [kRowTab]: attention row sources
constexpr int kUListPos = kUKeys + kSelCap * 4;               // i32 [kListCap]: the block's rerank slice
constexpr int kUBytes = kUListPos + kListCap * 4;
static_assert(kUHot + (5 * kSub * kCentroids + 1) * 4 + 16 <= kUBytes, "hot lists (G = 1) inside the region");
static_assert(kUWarpHist + kWarps * kWarpBins * 4 <= kUHot, "per-warp vote counts before the hot lists");
static_assert(kUHot + (9 * 1024 + 1) * 4 + 16 <= kUBytes, "hot lists (G = 2) inside the region");
static_assert(kUSelPos + kListCap * 4 <= kUStageV, "top-k tables inside the second round's K rows");
static_assert(kUBucket + kSelCap * 2 <= kUKeys && kSelCap <= 65536, "key buckets below the order keys, u16 indexes");
static_assert(kUBStart + kSelBins * 4 <= kUSelHist, "bin starts below the k-th key search's bins");
static_assert(kUHall + kClusterMax * kSelBins * 4 <= kUSelHist, "pushed histograms below the search's bins");
static_assert(kOwnCap >= 16384, "a slice of up to 16384 keys held by its block");
static_assert(kURecSlots + kThreads * kRecBytes <= kUKeys, "record slots below the order keys");

struct DecodeArgs {
  Shape s;
  Tables t;
  KvStore kv;
  SignMask sm;
  RsqParams rp;
  int rho, flat, nbins, cpb, nchunk_active;
  int64_t N, C, k, k_eff, cmax;
  int64_t nsink, nwin;  // attention window rows
  // cut points q = 0 .. kClusterMax (C q / CS, clamped at q = CS): the
  // rerank slices of the candidate list
  int64_t ccut[kClusterMax + 1];
  int64_t rcut[kClusterMax + 1];  // (nwin + k_eff) q / CS: the blocks' shares of the attention rows (the last one
                                  // smaller when it also sorts the top-k)
  uint32_t nmod;        // ring slot of the first Local token
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
  int32_t* topk_idx;    // the lists in ascending position (every block writes its slice's entries)
  float* topk_score;
  __nv_bfloat16* out;   // nullptr: no attention
  int32_t* ord_idx;     // nullptr: no reordering; else the lists best first go here
  float* ord_sc;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}

// A staged K or V row is 256 B with its 16-byte pieces permuted by row
// (piece c of row r at c ^ (r & 7)): every 32-byte sector lands whole in an
// aligned 32-byte slot, so a copy instruction is served as whole-sector
// requests (a row stride padded to 272 B splits the sectors of every other
// row and doubles the requests), and the reads below meet no bank conflict.
__device__ __forceinline__ int spiece(int row, int c) { return row * kDim + 8 * (c ^ (row & 7)); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Cluster barrier: every thread of every block of the cluster arrives; the
// writes before it (shared and global) are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The same barrier in two halves: work between them overlaps the wait.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

// Address of the same shared-memory variable in block `rank` of the cluster,
// and a 32-bit store there.  Stores to other blocks are made visible by the
// next cluster barrier.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
  return ra;
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t ra, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(ra), "r"(v) : "memory");
}

// Exclusive block scan of two unsigned values per thread at once (tmp: 66
// words of shared memory); x and y are replaced by their prefixes, tx and ty
// receive the block sums.
__device__ __forceinline__ void block_excl_scan2(uint32_t& x, uint32_t& y, uint32_t* tmp, uint32_t& tx,
                                                 uint32_t& ty) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ix = x, iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t tx = __shfl_up_sync(kFull, ix, o), ty = __shfl_up_sync(kFull, iy, o);
    if (lane >= o) {
      ix += tx;
      iy += ty;
    }
  }
  if (lane == 31) {
    tmp[warp] = ix;
    tmp[33 + warp] = iy;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t vx = tmp[lane], vy = tmp[33 + lane];
    uint32_t sx = vx, sy = vy;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t tx = __shfl_up_sync(kFull, sx, o), ty = __shfl_up_sync(kFull, sy, o);
      if (lane >= o) {
        sx += tx;
        sy += ty;
      }
    }
    tmp[lane] = sx - vx;
    tmp[33 + lane] = sy - vy;
    if (lane == 31) {
      tmp[32] = sx;
      tmp[65] = sy;
    }
  }
  __syncthreads();
  x = tmp[warp] + ix - x;
  y = tmp[33 + warp] + iy - y;
  tx = tmp[32];
  ty = tmp[65];
  __syncthreads();
}

// c[q] for a q known only at run time, by constant-index selects (a
// run-time index into a kernel parameter array would copy it to local memory).
__device__ __forceinline__ int64_t cut_at(const int64_t (&c)[kClusterMax + 1], int q) {
  int64_t v = c[0];
#pragma unroll
  for (int i = 1; i <= kClusterMax; ++i)
    if (q == i) v = c[i];
  return v;
}

// Per byte of x: 0x80 where the byte is nonzero / equals the byte of c4 /
// exceeds it (unsigned); 0 elsewhere.
__device__ __forceinline__ uint32_t bytes_nonzero(uint32_t x) {
  return (((x & 0x7f7f7f7fu) + 0x7f7f7f7fu) | x) & 0x80808080u;
}
__device__ __forceinline__ uint32_t bytes_eq(uint32_t x, uint32_t c4) { return ~bytes_nonzero(x ^ c4) & 0x80808080u; }
__device__ __forceinline__ uint32_t bytes_gt(uint32_t x, uint32_t c4) {
  // per byte (x | 0x80) - (c & 0x7f) never borrows; its high bit is [x_low7 >= c_low7]
  const uint32_t d = (x | 0x80808080u) - (c4 & 0x7f7f7f7fu);
  const uint32_t ge = ((x & ~c4) | (~(x ^ c4) & d)) & 0x80808080u;
  return ge & ~bytes_eq(x, c4);
}
// 0x80 in each of the first n (clamped to 0..4) bytes.
__device__ __forceinline__ uint32_t first_bytes(int n) {
  return n >= 4 ? 0x80808080u : n <= 0 ? 0u : (0x80808080u >> (8 * (4 - n)));
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
    // nibble j times 4 (a byte offset into its 16-entry row): even j in the
    // bytes of lo4, odd j in the bytes of hi4
    const uint32_t lo4 = (cw << 2) & 0x3c3c3c3cu, hi4 = (cw >> 2) & 0x3c3c3c3cu;
    const char* row = reinterpret_cast<const char*>(tq + b * kM * 16);
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kM; ++j) {
      const uint32_t off = __byte_perm((j & 1) ? hi4 : lo4, 0u, 0x4440u + (j >> 1));
      dot = __fadd_rn(dot, *reinterpret_cast<const float*>(row + j * 64 + off));
    }
    acc = __fadd_rn(acc, __fmul_rn(w, dot));
  }
  return __fmul_rn(qn, acc);
}

// One counting pass of the k-th key search: keys are counted by bin_of(key)
// (a bin in 0 .. kSelBins-1, or -1 for a key not in play), and the bin
// holding the `remaining`-th largest key in play is found by scanning from
// the top bin (bin order must follow key order).  `remaining` loses the keys
// of the bins above it; *held receives how many keys the bin holds; starts,
// when given, receives every bin's number of keys in the bins above it.
// key_of(i) gives the i-th of n keys.  All threads of the block call it.
template <class KeyOf, class BinOf>
__device__ __forceinline__ uint32_t count_pass(KeyOf key_of, int n, BinOf bin_of, uint32_t* hist, uint32_t* tmp,
                                               uint32_t& remaining, uint32_t* held, uint32_t* starts = nullptr) {
  __shared__ uint32_t s_bin, s_skip;
  const int tid = threadIdx.x;
  for (int i = tid; i < kSelBins; i += kThreads) hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const int bn = bin_of(key_of(i));
    if (bn >= 0) atomicAdd(&hist[bn], 1u);
  }
  __syncthreads();
  // thread t owns bins kSelBins-1-2t and kSelBins-2-2t, scanned from the top
  const uint32_t c0 = hist[kSelBins - 1 - 2 * tid], c1 = hist[kSelBins - 2 - 2 * tid];
  uint32_t tot;
  const uint32_t exc = block_excl_scan(c0 + c1, tmp, &tot);
  if (starts != nullptr) {  // every bin's number of keys in the bins above it
    starts[kSelBins - 1 - 2 * tid] = exc;
    starts[kSelBins - 2 - 2 * tid] = exc + c0;
  }
  if (exc < remaining && exc + c0 >= remaining) {
    s_bin = (uint32_t)(kSelBins - 1 - 2 * tid);
    s_skip = exc;
  } else if (exc + c0 < remaining && exc + c0 + c1 >= remaining) {
    s_bin = (uint32_t)(kSelBins - 2 - 2 * tid);
    s_skip = exc + c0;
  }
  __syncthreads();
  const uint32_t bn = s_bin;
  remaining -= s_skip;
  *held = hist[bn];
  __syncthreads();
  return bn;
}

// The `remaining`-th largest of the few keys (at most kBinRank) for which
// in_bin(key) holds: the key with fewer than `remaining` of them above it and
// at least `remaining` at or above it.  Returns it; `remaining` becomes the
// number of keys equal to it that are taken.
template <class KeyOf, class InBin>
__device__ __forceinline__ uint32_t rank_in_bin(KeyOf key_of, int n, InBin in_bin, uint32_t* bin,
                                                uint32_t& remaining) {
  __shared__ uint32_t s_nbin, s_key, s_rem;
  const int tid = threadIdx.x;
  if (tid == 0) s_nbin = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t k = key_of(i);
    if (in_bin(k)) bin[atomicAdd(&s_nbin, 1u)] = k;
  }
  __syncthreads();
  const int nbin = (int)s_nbin;
  if (tid < nbin) {
    const uint32_t mine = bin[tid];
    uint32_t above = 0, at = 0;
    for (int j = 0; j < nbin; ++j) {
      const uint32_t o = bin[j];
      above += o > mine ? 1u : 0u;
      at += o >= mine ? 1u : 0u;
    }
    if (above < remaining && at >= remaining) {  // every such thread holds the same key
      s_key = mine;
      s_rem = remaining - above;
    }
  }
  __syncthreads();
  const uint32_t key = s_key;
  remaining = s_rem;
  __syncthreads();
  return key;
}

// The k_eff-th largest of the C order keys of a query head, and how many
// keys equal to it belong to the top k_eff (*remaining_out).  kmin and kmax
// are the smallest and largest key.  First pass: kSelBins bins linear in the
// estimate between the two (a monotone map, so bin order is key order); if
// the chosen bin holds at most kBinRank keys they are ranked directly.
// Otherwise (a crowded bin, or a range the linear map cannot represent):
// 11-bit radix digits below the bits kmin and kmax share, with the same
// direct ranking once a digit is small.  key_of(i) gives key i.  All threads
// of the block call it and get the same results.  *linear_out is 1 when the
// linear bins decided it (the number of keys above each bin is then left at
// U + kUBStart), else 0.
template <class KeyOf>
__device__ __forceinline__ uint32_t select_kth(KeyOf key_of, const int64_t C, const int64_t k_eff, uint32_t kmin,
                                               uint32_t kmax, uint8_t* U, uint32_t* tmp, uint32_t* remaining_out,
                                               uint32_t* linear_out) {
  uint32_t* hist = reinterpret_cast<uint32_t*>(U + kUSelHist);
  uint32_t* bin = hist + kSelBins;
  const int n = (int)C;
  uint32_t remaining = (uint32_t)k_eff;
  *linear_out = 0u;
  if (kmin == kmax) {
    *remaining_out = remaining;
    return kmin;
  }
  const float fmin = key_to_float(kmin), fmax = key_to_float(kmax);
  const float sc = (float)kSelBins / (fmax - fmin);
  if (isfinite(sc) && sc > 0.f) {
    auto lin = [&](uint32_t k) -> int { return min(kSelBins - 1, (int)((key_to_float(k) - fmin) * sc)); };
    uint32_t held;
    const int bsel = (int)count_pass(key_of, n, lin, hist, tmp, remaining, &held,
                                     reinterpret_cast<uint32_t*>(U + kUBStart));
    if (held <= (uint32_t)kBinRank) {
      const uint32_t key = rank_in_bin(key_of, n, [&](uint32_t k) { return lin(k) == bsel; }, bin, remaining);
      *remaining_out = remaining;
      *linear_out = 1u;  // hist holds the linear bins' counts
      return key;
    }
    remaining = (uint32_t)k_eff;
  }
  const int top = 31 - __clz(kmin ^ kmax);  // highest bit where keys differ
  uint32_t mask = top == 31 ? 0u : (0xffffffffu << (top + 1));
  uint32_t prefix = kmin & mask;
  for (int hi = top; hi >= 0;) {
    const int nb = min(11, hi + 1), lo = hi + 1 - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    uint32_t held;
    const uint32_t digit = count_pass(
        key_of, n, [&](uint32_t k) { return (k & mask) == prefix ? (int)((k >> lo) & dmask) : -1; }, hist, tmp,
        remaining, &held);
    prefix |= digit << lo;
    mask |= dmask << lo;
    hi = lo - 1;
    if (hi >= 0 && held <= (uint32_t)kBinRank) {
      prefix = rank_in_bin(key_of, n, [&](uint32_t k) { return (k & mask) == prefix; }, bin, remaining);
      break;
    }
  }
  *remaining_out = remaining;
  return prefix;
}

// One query head's top-k list best first.  pos_in / sc_in: its k_eff
// entries in ascending position (global memory, written by the blocks of
// the cluster before a cluster barrier); idx_out / sc_out: k entries by
// (estimate desc, position asc), then (-1, -inf).  Estimates compare by
// order_key (monotone, -0 = +0), equal ones by slot (= position order).
// Every thread of the block calls these; they start with a barrier (the
// caller's last reads of `sm`, shared memory of kUAttnEnd bytes, are done).
//
// Up to kOrdCount entries: a counting sort.  The estimates go into nb bins
// of equal width over [min, max] (bin floor((e - min) nb / (max - min)) in
// float32, round to nearest: monotone in e), numbered from the largest
// down; a bin's start is the number of entries in the bins before it, and
// an entry's rank is its bin's start plus the entries of its bin that
// precede it, found by comparing with them.  When a bin holds more than
// kOrdBinMax entries (many equal estimates, or a few far from the rest) the
// keys are sorted instead (order_bitonic), so the comparisons stay bounded.
constexpr int kOrdCount = 4096;
constexpr uint32_t kOrdBinMax = 64;

// The bitonic sort of the 64-bit keys (~order_key << 32 | slot) at `skey`
// (n2 >= k_eff, a power of two); positions and estimates come from spos /
// ssc when given (shared memory), else from global memory again.
__device__ __forceinline__ void order_bitonic(const int32_t* pos_in, const float* sc_in, int32_t* idx_out,
                                              float* sc_out, int k, int k_eff, int n2, unsigned long long* skey,
                                              const uint32_t* key, const int32_t* spos, const float* ssc) {
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    unsigned long long v = ~0ull;  // padding sorts last
    if (i < k_eff) v = ((unsigned long long)~(key ? key[i] : order_key(__ldcg(sc_in + i))) << 32) | (uint32_t)i;
    skey[i] = v;
  }
  block_sort_pow2(skey, n2);
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    int32_t p = -1;
    float e = -INFINITY;
    if (i < k_eff) {
      const uint32_t slot = (uint32_t)skey[i];
      p = spos ? spos[slot] : __ldcg(pos_in + slot);
      e = ssc ? ssc[slot] : __ldcg(sc_in + slot);
    }
    idx_out[i] = p;
    if (sc_out) sc_out[i] = e;
  }
}

__device__ __forceinline__ void order_topk(const int32_t* pos_in, const float* sc_in, int32_t* idx_out, float* sc_out,
                                           int k, int k_eff, uint8_t* sm, uint32_t* red, uint32_t* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  int n2 = 64;
  while (n2 < k_eff) n2 <<= 1;
  __syncthreads();
  if (k_eff > kOrdCount) {
    order_bitonic(pos_in, sc_in, idx_out, sc_out, k, k_eff, n2, reinterpret_cast<unsigned long long*>(sm), nullptr,
                  nullptr, nullptr);
    return;
  }
  // [0, 64 KB): key, position, estimate and the binned slots of kOrdCount
  // entries; [64 KB, 128 KB): the bins' counts and starts (nb <= 8192)
  uint32_t* key = reinterpret_cast<uint32_t*>(sm);
  int32_t* spos = reinterpret_cast<int32_t*>(sm + 4 * kOrdCount);
  float* ssc = reinterpret_cast<float*>(sm + 8 * kOrdCount);
  uint32_t* bslot = reinterpret_cast<uint32_t*>(sm + 12 * kOrdCount);
  const int nb = n2 >= 1024 ? 2 * n2 : 2048;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(sm + 16 * kOrdCount);
  uint32_t* base = cnt + 2 * kOrdCount;
  if (tid == 0) red[64] = 0u;  // the largest bin count
  float fmin = INFINITY, fmax = -INFINITY;
  for (int i = tid; i < k_eff; i += nt) {
    const float e = __ldcg(sc_in + i);
    key[i] = order_key(e);
    spos[i] = __ldcg(pos_in + i);
    ssc[i] = e;
    fmin = fminf(fmin, e);
    fmax = fmaxf(fmax, e);
  }
  for (int b = tid; b < nb; b += nt) cnt[b] = 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    fmin = fminf(fmin, __shfl_xor_sync(kFull, fmin, o));
    fmax = fmaxf(fmax, __shfl_xor_sync(kFull, fmax, o));
  }
  if (lane == 0) {
    red[warp] = __float_as_uint(fmin);
    red[32 + warp] = __float_as_uint(fmax);
  }
  __syncthreads();
  fmin = lane < nw ? __uint_as_float(red[lane]) : INFINITY;
  fmax = lane < nw ? __uint_as_float(red[32 + lane]) : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    fmin = fminf(fmin, __shfl_xor_sync(kFull, fmin, o));
    fmax = fmaxf(fmax, __shfl_xor_sync(kFull, fmax, o));
  }
  const float width = __fsub_rn(fmax, fmin);  // +inf: every entry in one bin, then the sort
  const float scale = width > 0.f ? __fdiv_rn((float)nb, width) : 0.f;
  // bin of slot i, numbered from the largest estimate down
  auto bin_of = [&](int i) -> uint32_t {
    const float x = fminf(__fmul_rn(__fsub_rn(ssc[i], fmin), scale), (float)(nb - 1));
    return (uint32_t)(nb - 1) - (uint32_t)x;
  };
  for (int i = tid; i < k_eff; i += nt) atomicAdd(&cnt[bin_of(i)], 1u);
  __syncthreads();
  const int per = nb / nt;  // nb >= 2048 >= nt
  uint32_t sum = 0, cm = 0;
  for (int j = 0; j < per; ++j) {
    const uint32_t c = cnt[tid * per + j];
    sum += c;
    cm = max(cm, c);
  }
  atomicMax(&red[64], cm);
  uint32_t total;
  uint32_t off = block_excl_scan(sum, tmp, &total);  // its barriers also publish red[64]
  for (int j = 0; j < per; ++j) {
    base[tid * per + j] = off;
    off += cnt[tid * per + j];
  }
  cm = red[64];
  if (cm > kOrdBinMax) {  // the same in every thread; the counts and starts are read no more
    __syncthreads();
    order_bitonic(pos_in, sc_in, idx_out, sc_out, k, k_eff, n2, reinterpret_cast<unsigned long long*>(cnt), key,
                  spos, ssc);
    return;
  }
  for (int i = tid; i < k_eff; i += nt) bslot[atomicAdd(&base[bin_of(i)], 1u)] = (uint32_t)i;  // base: bin ends
  __syncthreads();
  for (int i = tid; i < k_eff; i += nt) {
    const uint32_t kk = key[i], b = bin_of(i), end = base[b];
    uint32_t rank = end - cnt[b];
    for (uint32_t m = end - cnt[b]; m < end; ++m) {
      const uint32_t s2 = bslot[m], k2 = key[s2];
      rank += (k2 > kk || (k2 == kk && s2 < (uint32_t)i)) ? 1u : 0u;
    }
    idx_out[rank] = spos[i];
    if (sc_out) sc_out[rank] = ssc[i];
  }
  for (int i = k_eff + tid; i < k; i += nt) {
    idx_out[i] = -1;
    if (sc_out) sc_out[i] = -INFINITY;
  }
}

// kTable: the query's centroid scores come from a learned-centroid table
// (a separate instantiation, so the analytic path's code is untouched).
// The k-th key search over keys that are not all in shared memory, shared
// by the cluster (see the layout above): each block loads its own slice's
// order keys (est: the slice's estimates), histograms them in the linear
// bins of select_kth and pushes the histogram to every block; all find the
// bin of the k_eff-th key the same way, each pushes its keys of that bin with
// their candidate numbers, and all rank those few.  ok = false (the same in
// every block) when the bin holds more than kBinRank keys or the range cannot
// be mapped.  Every thread of every block of the cluster calls it.
struct SharedSelect {
  uint32_t P, remaining, eq_take;
  int64_t out_off;
  bool ok;
};

__device__ __noinline__ SharedSelect shared_select(const float* est, int64_t k_eff, int64_t s_lo, uint32_t nown, int r,
                                                   int cs, const uint32_t* skey_mm, uint8_t* U, uint32_t* tmp,
                                                   uint32_t* red, uint32_t* s_sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  SharedSelect res = {0u, 0u, 0u, s_lo, false};
  uint32_t x = 0xffffffffu, y = 0u;
  for (int q = 0; q < cs; ++q) {
    x = min(x, skey_mm[2 * q]);
    y = max(y, skey_mm[2 * q + 1]);
  }
  const float fmin = key_to_float(x), fmax = key_to_float(y);
  const float sc = (float)kSelBins / (fmax - fmin);
  if (x == y || !isfinite(sc) || !(sc > 0.f)) return res;
  auto lin = [&](uint32_t k) -> int { return min(kSelBins - 1, (int)((key_to_float(k) - fmin) * sc)); };
  uint32_t* hist = reinterpret_cast<uint32_t*>(U + kUSelHist);
  uint32_t* hall2 = reinterpret_cast<uint32_t*>(U + kUHall);
  uint32_t* ownw = reinterpret_cast<uint32_t*>(U + kUOwn);
  uint32_t* ent = reinterpret_cast<uint32_t*>(U + kUBinEnt);
  for (int i = tid; i < kSelBins; i += kThreads) hist[i] = 0;
  for (uint32_t i = tid; i < nown; i += kThreads) ownw[i] = order_key(__ldcg(est + i));
  __syncthreads();
  // the slice's histogram
  for (uint32_t i = tid; i < nown; i += kThreads) atomicAdd(&hist[lin(ownw[i])], 1u);
  __syncthreads();
  for (int i = tid; i < kSelBins; i += kThreads) {
    const uint32_t v = hist[i];
    for (int q = 0; q < cs; ++q) dsmem_st_u32(dsmem_addr(hall2 + r * kSelBins + i, q), v);
  }
  cluster_sync();
  // thread t owns bins kSelBins-1-2t and kSelBins-2-2t, scanned from the top
  const int hb0 = kSelBins - 1 - 2 * tid, hb1 = kSelBins - 2 - 2 * tid;
  uint32_t c0 = 0, c1 = 0;
  for (int q = 0; q < cs; ++q) {
    c0 += hall2[q * kSelBins + hb0];
    c1 += hall2[q * kSelBins + hb1];
  }
  uint32_t tot;
  const uint32_t exc = block_excl_scan(c0 + c1, tmp, &tot);
  const uint32_t want = (uint32_t)k_eff;
  if (exc < want && exc + c0 >= want) {
    s_sel[0] = (uint32_t)hb0;
    s_sel[1] = exc;
  } else if (exc + c0 < want && exc + c0 + c1 >= want) {
    s_sel[0] = (uint32_t)hb1;
    s_sel[1] = exc + c0;
  }
  __syncthreads();
  const int bsel = (int)s_sel[0];
  const uint32_t above_all = s_sel[1];
  uint32_t held = 0, base_r = 0;
  for (int q = 0; q < cs; ++q) {
    const uint32_t c = hall2[q * kSelBins + bsel];
    held += c;
    base_r += q < r ? c : 0u;
  }
  if (held > (uint32_t)kBinRank) {  // the same in every block
    __syncthreads();  // s_sel is read above
    return res;
  }
  // keys in the bins above bsel in the blocks before this one
  uint32_t gl = 0;
  for (int q = 0; q < r; ++q) {
    if (hb0 > bsel) gl += hall2[q * kSelBins + hb0];
    if (hb1 > bsel) gl += hall2[q * kSelBins + hb1];
  }
  gl = __reduce_add_sync(kFull, gl);
  __syncthreads();  // s_sel[0..1] are read above
  if (tid == 0) s_sel[2] = 0u;
  if (lane == 0) red[warp] = gl;
  __syncthreads();
  uint32_t gt_lower = 0;
  for (int w = 0; w < kWarps; ++w) gt_lower += red[w];
  // this block's keys of bin bsel, with their candidate numbers, to every block
  for (uint32_t i = tid; i < nown; i += kThreads) {
    const uint32_t k = ownw[i];
    if (lin(k) == bsel) {
      const uint32_t slot = base_r + atomicAdd(&s_sel[2], 1u);
      for (int q = 0; q < cs; ++q) {
        dsmem_st_u32(dsmem_addr(ent + 2 * slot, q), k);
        dsmem_st_u32(dsmem_addr(ent + 2 * slot + 1, q), (uint32_t)(s_lo + i));
      }
    }
  }
  cluster_sync();
  // the (k_eff - above_all)-th largest of the bin's keys, as in select_kth
  const uint32_t rem = want - above_all;
  if (tid < (int)held) {
    const uint32_t mine = ent[2 * tid];
    uint32_t ab = 0, at = 0;
    for (uint32_t j = 0; j < held; ++j) {
      const uint32_t o = ent[2 * j];
      ab += o > mine ? 1u : 0u;
      at += o >= mine ? 1u : 0u;
    }
    if (ab < rem && at >= rem) {  // every such thread holds the same key
      s_sel[3] = mine;
      s_sel[2] = rem - ab;
    }
  }
  __syncthreads();
  res.P = s_sel[3];
  res.remaining = s_sel[2];
  // keys above P and equal to P before the slice: the lower blocks' keys in
  // higher bins, and the bin's keys with smaller candidate numbers
  uint32_t gtb = gt_lower, eqb = 0;
  for (uint32_t j = 0; j < held; ++j) {
    const uint32_t o = ent[2 * j], ci = ent[2 * j + 1];
    if ((int64_t)ci < s_lo) {
      gtb += o > res.P ? 1u : 0u;
      eqb += o == res.P ? 1u : 0u;
    }
  }
  res.out_off = gtb + min(eqb, res.remaining);
  res.eq_take = res.remaining > eqb ? res.remaining - eqb : 0u;
  res.ok = true;
  __syncthreads();  // s_sel, red and ent are read above
  return res;
}

// kTable: learned centroids (a table) instead of the analytic sign patterns.
// kShared: more candidates than kSelCap, whose k-th key search the cluster
// shares (shared_select); a separate instantiation, so the other kernels keep
// their registers.
template <bool kTable, bool kShared>
__global__ void __launch_bounds__(kThreads, 1) k_decode(DecodeArgs a) {
  __shared__ __align__(16) float qs[kDim];
  __shared__ __align__(16) float zs[kDim];
  __shared__ __align__(16) float qts[kDim];
  __shared__ float tq[kDim * 16];
  __shared__ uint32_t hist[kMaxBins];                // read by the cluster
  __shared__ uint32_t tot[kMaxBins];
  __shared__ uint32_t wcnt[7][kWarps];                       // per-warp counts of votes 1..7
  __shared__ uint32_t hall[kClusterMax][kMaxBins];           // every block's histogram, pushed by its owner
  __shared__ uint32_t skey_mm[kClusterMax][2];               // smallest and largest order key of every block
  __shared__ uint32_t staken[kClusterMax];                   // top-k entries every block's slice took
  __shared__ __align__(16) float pall[kClusterMax][kPartStride];  // attention partials, pushed to block 0
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t red[2 * kWarps + 2];
  __shared__ uint8_t rvalid[kStages][kTile];
  __shared__ float s_qn;
  __shared__ int s_T;
  __shared__ int64_t s_quota;
  __shared__ uint32_t s_sel[4];  // the shared k-th key search: bin, keys above it, bin entries, lower blocks' part
  __shared__ uint32_t s_rank;  // 1: the best-first list is placed directly (no sort)
  extern __shared__ __align__(128) uint8_t U[];  // 128-byte aligned: staged rows keep whole sectors

  const int nhot = kSub * a.rho;
  const int nlist = (nhot <= 1024 ? kVoteSlots : 1) * nhot;  // hot lists of a group of chunks
  uint32_t* hv = reinterpret_cast<uint32_t*>(U + kUHot);  // hot entries: id | weight << 16 | subspace << 24
  uint32_t* hbeg = hv + nhot;
  uint32_t* hwt = hbeg + nlist;
  uint32_t* hpre = hwt + nlist;                            // nlist + 1
  int32_t* hsm = reinterpret_cast<int32_t*>(hpre + nlist + 1);  // list entry f is lists[hsm[e] + f]
  // the group's lists, copied into shared memory when they fit
  const int lists_at = (kUHot + (nhot + 4 * nlist + 1) * 4 + 15) & ~15;
  uint16_t* lists = reinterpret_cast<uint16_t*>(U + lists_at);
  const int lists_cap = (kUBytes - lists_at) / 2;
  uint32_t* offs = reinterpret_cast<uint32_t*>(U + kUOffs);
  int32_t* lpos = reinterpret_cast<int32_t*>(U + kUListPos);
  uint16_t* stK = reinterpret_cast<uint16_t*>(U + kUStageK);
  uint16_t* stV = reinterpret_cast<uint16_t*>(U + kUStageV);

  const int r = blockIdx.x, cs = gridDim.x, sq = blockIdx.y;
  const int seq = sq / a.s.hq, qh = sq - seq * a.s.hq, kvh = qh / a.s.g;
  // the query head's list best first, sorted in the attention staging area
  auto order_tail = [&]() {
    const int64_t row = (int64_t)sq * a.k;
    order_topk(a.topk_idx + row, a.topk_score + row, a.ord_idx + row, a.ord_sc ? a.ord_sc + row : nullptr,
               (int)a.k, (int)a.k_eff, U, red, tmp);
  };
  const int64_t sh = (int64_t)seq * a.s.hkv + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c_lo = min(r * a.cpb, a.nchunk_active), c_hi = min(c_lo + a.cpb, a.nchunk_active);
  uint64_t* tr = (r == 0 && sq == 0) ? a.trace : nullptr;
  trace_block(a.trace, kTkDecode0, 0);

  // ---- before the wait: cleared counters ---------------------------------
  for (int i = tid; i < kVoteSlots * kChunk / 16; i += kThreads)
    reinterpret_cast<uint4*>(U + kUVotes)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kMaxBins; i += kThreads) hist[i] = 0;
  uint32_t* whist = reinterpret_cast<uint32_t*>(U + kUWarpHist);
  for (int i = tid; i < kWarps * kWarpBins; i += kThreads) whist[i] = 0;
  pdl_wait();
  pdl_trigger();
  trace_block(a.trace, kTkDecode0, 1);
  trace_mark(tr, kTrDecode0);

  // offset tables of chunks c .. c + n - 1 (consecutive in memory)
  auto prefetch_offsets = [&](int c, int n) {
    const uint32_t* og = a.t.off + ((sh * a.t.nchunk + c) * kSub) * kOffStride;
    for (int i = tid; i < n * kSub * kOffStride / 4; i += kThreads) cp_async16(offs + 4 * i, og + 4 * i);
  };
  if (c_lo < c_hi) prefetch_offsets(c_lo, min(nhot <= 1024 ? kVoteSlots : 1, c_hi - c_lo));

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
  if (warp == kSub) {
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
  } else if (warp == kSub + 1) {
    // the step's own token into the cache (nothing in this launch reads the
    // ring slot or table row it writes: the attention takes it from k/v)
    if (a.new_pos >= 0 && r == 0 && qh % a.s.g == 0)
      append_token_warp(a.k_new, a.v_new, a.kvdtype, a.new_pos, sh, lane, a.s, a.kv, a.t, a.sm, a.rp,
                        kTable ? a.t.cent : nullptr);
  } else if (warp < kSub) {
    const int b = warp;
    // the lane's centroids are lane + 32 i: bits 0-4 of the id are the lane's,
    // so the first five terms of the sequential sum are shared, then the
    // sums branch on bits 5, 6, 7 (the same additions in the same order)
    float zz[kM];
#pragma unroll
    for (int j = 0; j < kM; ++j) zz[j] = zs[b * kM + j];
    float a8[8];
    if constexpr (!kTable) {
      float acc5 = 0.f;
#pragma unroll
      for (int j = 0; j < 5; ++j) acc5 = __fadd_rn(acc5, ((lane >> j) & 1) ? -zz[j] : zz[j]);
      float a6[2], a7[4];
#pragma unroll
      for (int t = 0; t < 2; ++t) a6[t] = __fadd_rn(acc5, (t & 1) ? -zz[5] : zz[5]);
#pragma unroll
      for (int t = 0; t < 4; ++t) a7[t] = __fadd_rn(a6[t & 1], (t & 2) ? -zz[6] : zz[6]);
#pragma unroll
      for (int t = 0; t < 8; ++t) a8[t] = __fadd_rn(a7[t & 3], (t & 4) ? -zz[7] : zz[7]);
    } else {
      // learned centroids: score of centroid c = ((0 + z_0 c_0) + z_1 c_1) + ... + z_7 c_7
      const float* tab = a.t.cent + (int64_t)kvh * kTabPerHead + (int64_t)b * kCentroids * kM;
#pragma unroll 1
      for (int i = 0; i < 8; ++i) {
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(tab + (lane + 32 * i) * kM));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(tab + (lane + 32 * i) * kM + 4));
        float sc = __fmul_rn(zz[0], c0.x);
        sc = __fadd_rn(sc, __fmul_rn(zz[1], c0.y));
        sc = __fadd_rn(sc, __fmul_rn(zz[2], c0.z));
        sc = __fadd_rn(sc, __fmul_rn(zz[3], c0.w));
        sc = __fadd_rn(sc, __fmul_rn(zz[4], c1.x));
        sc = __fadd_rn(sc, __fmul_rn(zz[5], c1.y));
        sc = __fadd_rn(sc, __fmul_rn(zz[6], c1.z));
        sc = __fadd_rn(sc, __fmul_rn(zz[7], c1.w));
        a8[i] = sc;
      }
    }
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
  // sum_b weight_b(id_{i,b}) (one byte per key, at most 255).  The block
  // takes its chunks G at a time as one span of G x kChunk keys (G = 2, or
  // 1 when the hot lists are long).
  const int G = nhot <= 1024 ? kVoteSlots : 1;
  uint8_t* span = U + kUVotes;
  uint32_t cnt[7] = {0, 0, 0, 0, 0, 0, 0}, nz_mine = 0;  // votes 1..7 counted by bit planes
  int64_t own_len = 0;
  for (int g0 = c_lo; g0 < c_hi; g0 += G) {
    const int ng = min(G, c_hi - g0), nl = ng * nhot;
    const int64_t gbase = (int64_t)g0 * kChunk;
    const int glen = (int)min64((int64_t)ng * kChunk, a.N - gbase);
    own_len += glen;
    cp_async_wait_all();
    __syncthreads();  // the group's offsets (and, first time, the hot list) are in place
    {
      // list e2 = g * nhot + e: chunk g0 + g, hot entry e; its entries start
      // at (g * B + b) * kChunk + offset in the group's entry lists
      constexpr int kHotPer = (kSub * kCentroids + kThreads - 1) / kThreads;  // lists per thread: G nhot <= 4096
      const int per = (nl + kThreads - 1) / kThreads;
      uint32_t lens[kHotPer];
      uint32_t my = 0;
#pragma unroll
      for (int i = 0; i < kHotPer; ++i) {
        const int e2 = tid * per + i;
        lens[i] = 0;
        if (i < per && e2 < nl) {
          const int g = e2 >= nhot ? 1 : 0;
          const uint32_t h = hv[e2 - g * nhot];
          const uint32_t b = h >> 24, id = h & 0xffu;
          const uint32_t* og = offs + g * (kSub * kOffStride);
          const uint32_t beg = og[b * kOffStride + id];
          lens[i] = og[b * kOffStride + id + 1] - beg;
          hbeg[e2] = ((uint32_t)g * kSub + b) * kChunk + beg;
          hwt[e2] = ((h >> 16) & 0xffu) | ((uint32_t)g << 16);
        }
        my += lens[i];
      }
      uint32_t total;
      uint32_t run = block_excl_scan(my, tmp, &total);
#pragma unroll
      for (int i = 0; i < kHotPer; ++i) {
        const int e2 = tid * per + i;
        if (i < per && e2 < nl) hpre[e2] = run;
        run += lens[i];
      }
      if (tid == 0) hpre[nl] = total;
    }
    __syncthreads();
    if (g0 == c_lo) trace_mark(tr, kTrDecodeFine + 0);
    if (g0 + G < c_hi) prefetch_offsets(g0 + G, min(G, c_hi - g0 - G));  // offsets not read again
    const uint32_t total = hpre[nl];
    const uint16_t* ent = a.t.ent + ((sh * a.t.nchunk + g0) * kSub) * (int64_t)kChunk;
    // list e2 goes to lists[S, S + pad) with S = 8-aligned(hpre + 24 e2): its
    // aligned 16-byte pieces (the list plus up to 14 neighbouring bytes)
    const bool staged = (int64_t)total + 24 * nl + 8 <= lists_cap;  // the same in the whole block
    if (staged) {
      for (int e2 = warp; e2 < nl; e2 += kWarps) {
        const uint32_t hb = hbeg[e2], len = hpre[e2 + 1] - hpre[e2];
        const uint32_t S = (hpre[e2] + 24u * e2 + 7u) & ~7u;
        const uint32_t n16 = ((hb & 7u) + len + 7u) >> 3;
        for (uint32_t k = lane; k < n16; k += 32) cp_async16(lists + S + 8 * k, ent + (hb & ~7u) + 8 * k);
        if (lane == 0) hsm[e2] = (int32_t)(S + (hb & 7u)) - (int32_t)hpre[e2];
      }
      cp_async_wait_all();
      __syncwarp();  // a warp walks exactly the lists it staged
    }
    // warp w walks lists w, w + 32, ...; lane l takes entries l, l + 32, ...
    uint32_t* votes32 = reinterpret_cast<uint32_t*>(span);
    for (int e2 = warp; e2 < nl; e2 += kWarps) {
      const uint32_t p0 = hpre[e2], len = hpre[e2 + 1] - p0, hw = hwt[e2];
      const uint32_t wt = hw & 0xffu, koff = (hw >> 16) << 14;  // weight; the chunk's place in the span
      if (staged) {
        const uint16_t* src = lists + hsm[e2] + (int32_t)p0;
        for (uint32_t i = lane; i < len; i += 32) {
          const uint32_t key = src[i] + koff;
          atomicAdd(votes32 + (key >> 2), wt << ((key & 3) * 8));
        }
      } else {
        const uint16_t* src = ent + hbeg[e2];
        for (uint32_t i0 = 0; i0 < len; i0 += 128) {
          uint32_t kk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) kk[u] = i0 + 32 * u + lane < len ? __ldg(src + i0 + 32 * u + lane) : 0xffffffffu;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (kk[u] != 0xffffffffu) {
              const uint32_t key = kk[u] + koff;
              atomicAdd(votes32 + (key >> 2), wt << ((key & 3) * 8));
            }
        }
      }
    }
    __syncthreads();
    if (g0 == c_lo) trace_mark(tr, kTrDecodeFine + 1);
    // votes out; histogram: votes 1..7 (the bytes below 8) by bit planes,
    // larger votes one by one.  Thread t: 16 keys of each chunk of the group,
    // as 4 G words; the planes of word w sit at bits 8 j + w (byte j), so one
    // population count covers all of the thread's keys.
    uint32_t P0 = 0, P1 = 0, P2 = 0;
    for (int g = 0; g < ng; ++g) {
      const int vi = g * kThreads + tid;
      uint4* vp = reinterpret_cast<uint4*>(span) + vi;
      const uint4 w4 = *vp;
      reinterpret_cast<uint4*>(a.votes + (int64_t)sq * a.t.nchunk * kChunk + gbase)[vi] = w4;
      if (g0 + G < c_hi) *vp = make_uint4(0, 0, 0, 0);  // the span is reused by the next group
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t x = ws[k];
        const uint32_t v01 = first_bytes(glen - (16 * vi + 4 * k)) >> 7;
        uint32_t big = (bytes_nonzero(x & 0xf8f8f8f8u) >> 7) & v01;  // valid bytes >= 8
        const uint32_t lo = v01 & ~big;
        const int w = 4 * g + k;
        P0 |= (x & lo) << w;
        P1 |= ((x >> 1) & lo) << w;
        P2 |= ((x >> 2) & lo) << w;
        nz_mine += __popc(big);
        while (big) {
          const int j = (31 - __clz(big & (0u - big))) >> 3;
          big &= big - 1;
          const uint32_t v = (x >> (8 * j)) & 0xffu;
          if (v < 8 + kWarpBins) atomicAdd(&whist[warp * kWarpBins + (v - 8)], 1u);
          else atomicAdd(&hist[v], 1u);
        }
      }
    }
    cnt[0] += __popc(P0 & ~P1 & ~P2);
    cnt[1] += __popc(~P0 & P1 & ~P2);
    cnt[2] += __popc(P0 & P1 & ~P2);
    cnt[3] += __popc(~P0 & ~P1 & P2);
    cnt[4] += __popc(P0 & ~P1 & P2);
    cnt[5] += __popc(~P0 & P1 & P2);
    cnt[6] += __popc(P0 & P1 & P2);
    nz_mine += __popc(P0 | P1 | P2);
  }
  {
#pragma unroll
    for (int v = 0; v < 7; ++v) {
      const uint32_t n = __reduce_add_sync(kFull, cnt[v]);
      if (lane == 0) wcnt[v][warp] = n;
    }
    uint32_t nz_all;
    block_excl_scan(nz_mine, tmp, &nz_all);  // (its barriers also order the per-warp counts)
    if (tid < kWarpBins) {
      uint32_t n = 0;
#pragma unroll 8
      for (int w = 0; w < kWarps; ++w) n += whist[w * kWarpBins + tid];
      if (n) atomicAdd(&hist[8 + tid], n);
    } else if (tid < kWarpBins + 7) {
      // votes 1..7: one thread per value sums the warps (no other writer)
      const int v = tid - kWarpBins;
      uint32_t n = 0;
#pragma unroll 8
      for (int w = 0; w < kWarps; ++w) n += wcnt[v][w];
      hist[v + 1] = n;
    }
    if (tid == 0) hist[0] = (uint32_t)own_len - nz_all;
  }
  trace_block(a.trace, kTkDecode0, 3);
  trace_mark(tr, kTrDecode1);

  // ---- 2. candidates --------------------------------------------------------
  // The candidates are the first C keys by (votes desc, index asc): with T
  // the largest vote value whose suffix count reaches C, every key above T
  // and the lowest-index keys equal to T, up to C.
  __syncthreads();
  if (tid < kMaxBins) {
    const uint32_t mine = hist[tid];
    for (int q = 0; q < cs; ++q) dsmem_st_u32(dsmem_addr(&hall[r][tid], q), mine);
  }
  cluster_sync();
  uint32_t bef = 0;
  if (tid < kMaxBins) {
    uint32_t v[kClusterMax];
#pragma unroll
    for (int q = 0; q < kClusterMax; ++q) v[q] = q < cs ? hall[q][tid] : 0u;
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
      red[kWarps + warp] = eqb;
    }
    __syncthreads();
    gtb = 0;
    eqb = 0;
#pragma unroll
    for (int w = 0; w < kMaxBins / 32; ++w) {  // the warps holding vote values
      gtb += red[w];
      eqb += red[kWarps + w];
    }
    sel_before = gtb + min64(eqb, quota);
    eq_allow = max64(0, quota - (int64_t)eqb);
  }
  trace_mark(tr, kTrDecode2);

  // ordered compaction: thread t owns keys [16 G t, 16 G (t + 1)) of each
  // group's span, compared four at a time (bytes of a word)
  const int64_t cq = (int64_t)sq * a.cmax;
  __syncthreads();  // red is read above and scanned in below
  {
    uint32_t nsel = 0;
    const uint32_t T4 = (uint32_t)T * 0x01010101u;
    int32_t* out = a.cand_idx + cq + sel_before;
    for (int g0 = c_lo; g0 < c_hi; g0 += G) {
      const int ng = min(G, c_hi - g0);
      const int64_t gbase = (int64_t)g0 * kChunk;
      const int glen = (int)min64((int64_t)ng * kChunk, a.N - gbase);
      const int k0 = 16 * G * tid;
      const bool in_smem = g0 + G >= c_hi;  // the last group's votes are still in shared memory
      uint32_t vw[4 * kVoteSlots];
#pragma unroll
      for (int i = 0; i < kVoteSlots; ++i) {
        uint4 x = make_uint4(0, 0, 0, 0);
        if (i < G && k0 + 16 * i < glen)
          x = in_smem ? reinterpret_cast<const uint4*>(span)[G * tid + i]
                      : __ldcg(reinterpret_cast<const uint4*>(a.votes + (int64_t)sq * a.t.nchunk * kChunk + gbase) + G * tid + i);
        vw[4 * i] = x.x; vw[4 * i + 1] = x.y; vw[4 * i + 2] = x.z; vw[4 * i + 3] = x.w;
      }
      // per byte: 0x80 where the vote is above T / equal to T (keys past the span: neither)
      uint32_t gtm[4 * kVoteSlots], eqm[4 * kVoteSlots];
      uint32_t n_eq = 0, n_gt = 0;
#pragma unroll
      for (int w = 0; w < 4 * kVoteSlots; ++w) {
        const uint32_t valid = w < 4 * G ? first_bytes(glen - (k0 + 4 * w)) : 0u;
        gtm[w] = bytes_gt(vw[w], T4) & valid;
        eqm[w] = bytes_eq(vw[w], T4) & valid;
        n_gt += __popc(gtm[w]);
        n_eq += __popc(eqm[w]);
      }
      // one scan of both counts: the keys equal to T are taken in position
      // order, so those taken before this thread are min(equal before it, allowance)
      uint32_t gt_rank0 = n_gt, eq_rank0 = n_eq, gt_tot, eq_tot;
      block_excl_scan2(gt_rank0, eq_rank0, red, gt_tot, eq_tot);
      uint32_t eq_left = (uint32_t)max64(0, min64((int64_t)n_eq, eq_allow - (int64_t)eq_rank0));
      const uint32_t csel = gt_tot + (uint32_t)min64((int64_t)eq_tot, eq_allow);
      uint32_t pos = nsel + gt_rank0 + (uint32_t)min64((int64_t)eq_rank0, eq_allow);
      const int32_t pbase = (int32_t)(a.s.sink + gbase + k0);
#pragma unroll
      for (int w = 0; w < 4 * kVoteSlots; ++w) {
        uint32_t e = eqm[w];
        // the lowest-position keys equal to T, up to this thread's share
        while (__popc(e) > (int)eq_left) e &= ~(0x80000000u >> __clz(e));
        eq_left -= __popc(e);
        uint32_t m = gtm[w] | e;
        while (m) {
          const int j = (31 - __clz(m & (0u - m))) >> 3;  // lowest flagged byte
          m &= m - 1;
          const int32_t p = pbase + 4 * w + j;
          out[pos++] = p;
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
  trace_block(a.trace, kTkDecode3, 0);
  const int64_t s_lo = cut_at(a.ccut, r), s_hi = cut_at(a.ccut, r + 1);
  const uint32_t nown = (uint32_t)(s_hi - s_lo);
  const bool keys_staged = a.C <= kSelCap;  // every block holds all C order keys
  uint32_t keys_at[kClusterMax];
#pragma unroll
  for (int q = 0; q < kClusterMax; ++q) keys_at[q] = q < cs ? dsmem_addr(U + kUKeys, q) : 0u;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  {
    // Warp w takes candidates 32 w + 1024 k + lane.  Its 32 records of a
    // round are copied into the warp's own 4 KB of shared memory with each
    // copy instruction covering four whole 128-byte records (lane l: piece
    // l % 8 of record l / 8 + 4 u), then every lane estimates its own.
    const uint8_t* rec = a.t.rec + sh * a.t.rcap * kRecBytes;
    const float qn = s_qn;
    uint4* wslot = reinterpret_cast<uint4*>(U + kURecSlots) + warp * 32 * 8;
    auto cand_pos = [&](uint32_t j) { return __ldcg(a.cand_idx + cq + s_lo + j); };
    for (uint32_t c0 = 32 * warp; c0 < nown; c0 += kThreads) {
      const uint32_t i = c0 + lane;
      const int32_t pm = i < nown ? cand_pos(i) : -1;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int rc = 4 * u + (lane >> 3), piece = lane & 7;
        const int32_t p = __shfl_sync(kFull, pm, rc);
        if (p >= 0)
          cp_async16(wslot + rc * 8 + (piece ^ (rc & 7)),
                     rec + (int64_t)(p - a.s.sink) * kRecBytes + 16 * piece);
      }
      cp_async_wait_all();
      __syncwarp();
      if (pm >= 0) {
        uint4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = wslot[lane * 8 + (u ^ (lane & 7))];
        const float e = estimate(x, tq, qn);
        a.cand_est[cq + s_lo + i] = e;
        if (i < kListCap) lpos[i] = pm;
        const uint32_t key = order_key(e);
        kmn = min(kmn, key);
        kmx = max(kmx, key);
        if (keys_staged) {
#pragma unroll
          for (int q = 0; q < kClusterMax; ++q)
            if (q < cs) dsmem_st_u32(keys_at[q] + 4u * (uint32_t)(s_lo + i), key);
        }
      }
      __syncwarp();  // the slots are reused by the next round
    }
  }
  kmn = __reduce_min_sync(kFull, kmn);
  kmx = __reduce_max_sync(kFull, kmx);
  if (lane == 0) {
    red[warp] = kmn;
    red[kWarps + warp] = kmx;
  }
  __syncthreads();
  if (tid < cs) {
    // the block's smallest and largest key, to every block
    uint32_t x = 0xffffffffu, y = 0u;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) {
      x = min(x, red[w]);
      y = max(y, red[kWarps + w]);
    }
    dsmem_st_u32(dsmem_addr(&skey_mm[r][0], tid), x);
    dsmem_st_u32(dsmem_addr(&skey_mm[r][1], tid), y);
  }
  trace_block(a.trace, kTkDecode1, 1);
  trace_mark(tr, kTrDecode3);

  trace_block(a.trace, kTkDecode1, 2);
  cluster_sync();  // every estimate and order key of the cluster, and their range, is in place
  trace_block(a.trace, kTkDecode3, 1);

  // ---- 4. top-k ------------------------------------------------------------
  // The k_eff-th best candidate by (estimate desc, position asc): every
  // block finds the k_eff-th largest order key P over all C estimates and
  // how many keys equal to P are taken (the lowest positions first).  The
  // taken entries in list (position) order are the top-k.  Block r counts
  // the entries taken before its slice, so knows where its slice's taken
  // entries go, writes them, and attends over them (with its share of the
  // window rows).
  const bool select_all = a.k_eff >= a.C;  // the same in every block
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(U + kUKeys);
  auto key_of = [&](int64_t i) -> uint32_t {
    return keys_staged ? keys[i] : order_key(__ldcg(a.cand_est + cq + i));
  };
  uint32_t P = 0, remaining = 0, linear = 0;
  int64_t out_off = s_lo;  // place of the slice's first taken entry
  uint32_t eq_take = 0;    // keys equal to P that the slice takes
  // Keys not all in shared memory: each block holds its own slice's keys,
  // histograms them (the linear bins of the search below) and pushes the
  // histogram to every block; all find the bin of the k_eff-th key the same
  // way, each pushes its keys of that bin, and all rank those few.  Falls back
  // (the same in every block) to the search over every key in global memory
  // when the bin holds more than kBinRank keys or the range cannot be mapped.
  const uint32_t* own = reinterpret_cast<const uint32_t*>(U + kUOwn);
  bool shared_search = false;
  if (kShared && !select_all && !keys_staged && (a.C + cs - 1) / cs <= kOwnCap) {
    const SharedSelect ss = shared_select(a.cand_est + cq + s_lo, a.k_eff, s_lo, nown, r, cs, &skey_mm[0][0], U, tmp,
                                          red, s_sel);
    if (ss.ok) {
      P = ss.P;
      remaining = ss.remaining;
      out_off = ss.out_off;
      eq_take = ss.eq_take;
      shared_search = true;
    }
  }
  if (!select_all && !shared_search) {
    uint32_t x = 0xffffffffu, y = 0u;
#pragma unroll
    for (int q = 0; q < kClusterMax; ++q)
      if (q < cs) {
        x = min(x, skey_mm[q][0]);
        y = max(y, skey_mm[q][1]);
      }
    P = select_kth(key_of, a.C, a.k_eff, x, y, U, tmp, &remaining, &linear);
  }
  trace_block(a.trace, kTkDecode3, 2);
  if (!select_all && !shared_search) {
    uint32_t gtb = 0, eqb = 0;
    for (int64_t i = tid; i < s_lo; i += kThreads) {
      const uint32_t k = key_of(i);
      gtb += k > P ? 1u : 0u;
      eqb += k == P ? 1u : 0u;
    }
    gtb = __reduce_add_sync(kFull, gtb);
    eqb = __reduce_add_sync(kFull, eqb);
    if (lane == 0) {
      red[warp] = gtb;
      red[kWarps + warp] = eqb;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t g = __reduce_add_sync(kFull, red[lane]), e = __reduce_add_sync(kFull, red[kWarps + lane]);
      __syncwarp();
      if (lane == 0) {
        red[0] = g;
        red[kWarps] = e;
      }
    }
    __syncthreads();
    gtb = red[0];
    eqb = red[kWarps];
    out_off = gtb + min(eqb, remaining);
    eq_take = remaining > eqb ? remaining - eqb : 0u;
    __syncthreads();  // red is reused below
  }
  // The list best first, placed directly: the linear count pass of the k-th
  // key search left, for every bin (bins in key order), the number of keys
  // in the bins above it; the keys at or above the k-th (every one the list
  // takes, and all that can precede one of them) go into the shared bucket of
  // their bin, so a taken entry's place in the best-first list is its bin's
  // start plus the keys of its bucket that precede it by (key desc, position
  // asc).  It needs the linear bins and every key in shared memory, the same
  // in every block (each holds the same keys); otherwise the last block sorts.
  bool rank_mode = false;  // the same in every thread
  uint32_t* bstart = reinterpret_cast<uint32_t*>(U + kUBStart);
  uint16_t* bucket = reinterpret_cast<uint16_t*>(U + kUBucket);
  float bmin = 0.f, bsc = 0.f;
  if (a.ord_idx != nullptr && !select_all && keys_staged && linear != 0u) {
    uint32_t x = 0xffffffffu, y = 0u;
#pragma unroll
    for (int q = 0; q < kClusterMax; ++q)
      if (q < cs) {
        x = min(x, skey_mm[q][0]);
        y = max(y, skey_mm[q][1]);
      }
    bmin = key_to_float(x);  // the k-th key search's linear map
    bsc = (float)kSelBins / (key_to_float(y) - bmin);
    for (int64_t i = tid; i < a.C; i += kThreads) {
      const uint32_t k = keys[i];
      if (k >= P) bucket[atomicAdd(&bstart[min(kSelBins - 1, (int)((key_to_float(k) - bmin) * bsc))], 1u)] = (uint16_t)i;
    }
    // every bin above P's is complete, so bin b's bucket is now
    // bucket[bstart[b + 1] .. bstart[b]) (from 0 for the top bin)
    __syncthreads();
    rank_mode = true;
  }
  if (tid == 0) s_rank = rank_mode ? 1u : 0u;  // read after the barriers of the placement below
  // the slice in order: thread t owns entries [t per, t per + per) of it
  int32_t* selpos = reinterpret_cast<int32_t*>(U + kUSelPos);
  uint32_t nsel;  // entries the slice takes
  {
    const uint32_t per = (nown + kThreads - 1) / kThreads;
    const uint32_t i0 = min(nown, tid * per), i1 = min(nown, i0 + per);
    uint32_t n_gt = 0, n_eq = 0;
    for (uint32_t i = i0; i < i1; ++i) {
      const uint32_t k = kShared && shared_search ? own[i] : key_of(s_lo + i);
      n_gt += select_all || k > P ? 1u : 0u;
      n_eq += !select_all && k == P ? 1u : 0u;
    }
    uint32_t gt_b = n_gt, eq_b = n_eq, gt_tot, eq_tot;
    block_excl_scan2(gt_b, eq_b, red, gt_tot, eq_tot);
    nsel = gt_tot + min(eq_tot, eq_take);
    uint32_t j = gt_b + min(eq_b, eq_take), eq_seen = eq_b;
    for (uint32_t i = i0; i < i1; ++i) {
      const uint32_t k = kShared && shared_search ? own[i] : key_of(s_lo + i);
      bool take = select_all || k > P;
      if (!select_all && k == P) take = eq_seen++ < eq_take;
      if (take) {
        const int32_t pos = i < kListCap ? lpos[i] : __ldcg(a.cand_idx + cq + s_lo + i);
        // the estimate from its key, except for the one key +0 and -0 share
        const float e = keys_staged && k != order_key(0.f) ? key_to_float(k) : __ldcg(a.cand_est + cq + s_lo + i);
        if (out_off + j < a.k_eff) {  // always, unless the counts above disagree
          a.topk_idx[(int64_t)sq * a.k + out_off + j] = pos;
          if (a.topk_score) a.topk_score[(int64_t)sq * a.k + out_off + j] = e;
        }
        if (rank_mode) {
          const int b = min(kSelBins - 1, (int)((key_to_float(k) - bmin) * bsc));
          const uint32_t lo = b == kSelBins - 1 ? 0u : bstart[b + 1], hi = bstart[b], me = (uint32_t)(s_lo + i);
          uint32_t rk = lo;
          for (uint32_t f = lo; f < hi; ++f) {
            const uint32_t o = bucket[f], ko = keys[o];
            rk += ko > k || (ko == k && o < me) ? 1u : 0u;
          }
          if (rk < a.k_eff) {
            a.ord_idx[(int64_t)sq * a.k + rk] = pos;
            a.ord_sc[(int64_t)sq * a.k + rk] = e;
          }
        }
        if (j < kListCap) selpos[j] = pos;
        ++j;
      }
    }
    if (r == 0) {
      for (int64_t i = a.k_eff + tid; i < a.k; i += kThreads) {
        a.topk_idx[(int64_t)sq * a.k + i] = -1;
        if (a.topk_score) a.topk_score[(int64_t)sq * a.k + i] = -INFINITY;
        if (rank_mode) {
          a.ord_idx[(int64_t)sq * a.k + i] = -1;
          a.ord_sc[(int64_t)sq * a.k + i] = -INFINITY;
        }
      }
    }
  }
  trace_block(a.trace, kTkDecode3, 3);
  trace_mark(tr, kTrDecode4);

  // ---- 5. sparse attention ---------------------------------------------------
  if (a.out != nullptr) {
    // The block's rows: the entries its slice took, topped up with window rows
    // so that every block has about (nwin + k_eff) / cs rows (block q's
    // window rows follow block q - 1's).  The slices' counts go to every block.
    if (tid < cs) dsmem_st_u32(dsmem_addr(&staken[r], tid), nsel);
    cluster_sync();
    int wl = 0, wh = 0;
    if (tid == 0) {
      int wrun = 0;
      for (int q = 0; q < cs; ++q) {
        const int lo = wrun;
        const int share = (int)(cut_at(a.rcut, q + 1) - cut_at(a.rcut, q));
        wrun = q == cs - 1 ? (int)a.nwin : min((int)a.nwin, wrun + max(0, share - (int)staken[q]));
        if (q == r) {
          wl = lo;
          wh = wrun;
        }
      }
      red[0] = (uint32_t)wl;
      red[1] = (uint32_t)wh;
    }
    __syncthreads();
    wl = (int)red[0];
    wh = (int)red[1];
    const int nwb = (int)(wh - wl);
    const int nrows = nwb + (int)min64(nsel, a.k_eff - out_off);
    const int ring = a.s.local + a.s.ubuf;
    // where each row comes from: element offset into the window arrays
    // (kSrcWindow set) or the Retrieval-zone store; kSrcFresh: the step's
    // own token; -1: no row
    constexpr int64_t kSrcWindow = int64_t(1) << 62, kSrcFresh = int64_t(1) << 61;
    const uint32_t nmod = a.nmod;
    auto window_source = [&](int64_t row) -> int64_t {
      int64_t slot = row, pos = row;
      if (row >= a.nsink) {
        uint32_t x = nmod + (uint32_t)(row - a.nsink);  // < 2 ring: the window holds at most ring tokens
        if (x >= (uint32_t)ring) x -= (uint32_t)ring;
        slot = a.s.sink + x;
        pos = a.s.sink + a.N + (row - a.nsink);
      }
      if (pos == a.new_pos) return kSrcFresh;
      return kSrcWindow | ((sh * a.kv.win + slot) * kDim);
    };
    auto retrieved_source = [&](int64_t pos) -> int64_t {
      if (pos >= a.s.sink && pos < a.s.sink + a.N) return (sh * a.kv.rcap + (pos - a.s.sink)) * kDim;
      if (pos >= 0) atomicOr(a.status, kStatusBadIndex);
      return -1;
    };
    // rows past the table: resolved when they are loaded (the slice's top-k
    // entries are in global memory by then)
    auto row_source = [&](int t) -> int64_t {
      return t < nwb ? window_source(wl + t)
                     : retrieved_source(__ldcg(a.topk_idx + (int64_t)sq * a.k + out_off + (t - nwb)));
    };
    int64_t* rsrc = reinterpret_cast<int64_t*>(U + kUKeys);  // the order keys are no longer read
    __syncthreads();  // the slice's taken positions are in place; every key read is done
    for (int t = tid; t < min(nrows, kRowTab); t += kThreads) {
      const int j = t - nwb;
      rsrc[t] = t < nwb ? window_source(wl + t)
                        : retrieved_source(j < kListCap ? selpos[j]
                                                        : __ldcg(a.topk_idx + (int64_t)sq * a.k + out_off + j));
    }
    if (tid < kDim) zs[tid] = qs[tid] * a.qscale;  // scaled q for the attention
    __syncthreads();
    trace_block(a.trace, kTkDecode1, 3);
    // Rounds of kRound rows through two halves of the stage area: round
    // rd + 2 loads into the half that round rd has just used, so two rounds
    // are in flight.  Warp w copies and scores rows 4 w .. 4 w + 3 of every
    // round, so it waits for its own copies only (no block barrier between
    // rounds): 16 lanes per row copy one 16-byte piece each; 8 lanes per row
    // score it (16 dimensions each) with the warp's own online softmax; lane l
    // accumulates output dimensions 4 l .. 4 l + 3 over the warp's rows.  The
    // instantiation with the cluster-shared k-th key search keeps the block
    // barriers and copies rows (tid / 16) + 64 u (its registers spill less
    // that way, and its many-round attention of large k ran faster).
    constexpr int kRound = kStages * kTile / 2;
    static_assert(kRound == 4 * kWarps && 16 * kRound == 2 * kThreads, "4 rows per warp, 2 copied rows per thread");
    const int nrounds = (nrows + kRound - 1) / kRound;
    auto issue = [&](int rd) {
      const int half = rd & 1;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int rr = kShared ? (tid >> 4) + 64 * u : 4 * warp + 2 * u + (lane >> 4), ch = lane & 15;  // round row, piece
        const int so = (half * kRound + rr) * kDim + 8 * (ch ^ (rr & 7));  // spiece
        uint16_t* kd = stK + so;
        uint16_t* vd = stV + so;
        const int rl = rd * kRound + rr;
        int64_t src = -1;
        if (rd < nrounds && rl < nrows) src = rl < kRowTab ? rsrc[rl] : row_source(rl);
        if (src == kSrcFresh) {
          // the step's own token: from the caller's k/v, converted as the append stores it
          *reinterpret_cast<uint4*>(kd) = load8_as_bf16(a.k_new, a.kvdtype, sh * kDim + 8 * ch);
          *reinterpret_cast<uint4*>(vd) = load8_as_bf16(a.v_new, a.kvdtype, sh * kDim + 8 * ch);
        } else if (src >= 0) {
          const bool win = (src & kSrcWindow) != 0;
          const int64_t e = (src & (kSrcFresh - 1)) + 8 * ch;
          cp_async16(kd, (win ? a.kv.win_k : a.kv.st_k) + e);
          cp_async16(vd, (win ? a.kv.win_v : a.kv.st_v) + e);
        } else {
          *reinterpret_cast<uint4*>(vd) = make_uint4(0, 0, 0, 0);  // finite zeros for the V sum
        }
        if (ch == 0) rvalid[half * 2 + (rr >> 6)][rr & 63] = src != -1 ? 1 : 0;
      }
      cp_async_commit();
    };
    trace_mark(tr, kTrDecodeRound - 1);
    issue(0);
    issue(1);
    // scored row of the round; the lane takes pieces oct and oct + 8 of it
    const int hrow = 4 * warp + (lane >> 3), oct = lane & 7;
    const int kofs = spiece(hrow, oct);                                    // piece oct + 8 is 64 elements on
    const int vofs = 8 * ((lane >> 1) ^ (4 * (warp & 1))) + 4 * (lane & 1);  // row 4 warp + i: vofs ^ 8 i
    float qv[16];  // the lane's 16 dimensions of the scaled q, loaded once
#pragma unroll
    for (int i = 0; i < 16; ++i) qv[i] = zs[64 * (i >> 3) + 8 * oct + (i & 7)];
    float M = -FLT_MAX, l = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int rd = 0; rd < nrounds; ++rd) {
      const int half = rd & 1;
      cp_async_wait_group<1>();  // all but the newest group: the warp's rows of round rd have landed
      if constexpr (kShared) __syncthreads(); else __syncwarp();
      if (rd < 8) trace_mark(tr, kTrDecodeRound + 2 * rd);
      const uint16_t* kh = stK + half * kRound * kDim;
      const uint16_t* vh = stV + half * kRound * kDim;
      float s = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint4 kv8 = *reinterpret_cast<const uint4*>(kh + kofs + 64 * u);
        const float* q8 = qv + 8 * u;
        s += q8[0] * bf16_bits_to_float(kv8.x & 0xffffu) + q8[1] * __uint_as_float(kv8.x & 0xffff0000u);
        s += q8[2] * bf16_bits_to_float(kv8.y & 0xffffu) + q8[3] * __uint_as_float(kv8.y & 0xffff0000u);
        s += q8[4] * bf16_bits_to_float(kv8.z & 0xffffu) + q8[5] * __uint_as_float(kv8.z & 0xffff0000u);
        s += q8[6] * bf16_bits_to_float(kv8.w & 0xffffu) + q8[7] * __uint_as_float(kv8.w & 0xffff0000u);
      }
      s += __shfl_xor_sync(kFull, s, 1);
      s += __shfl_xor_sync(kFull, s, 2);
      s += __shfl_xor_sync(kFull, s, 4);
      const bool valid = rvalid[half * 2 + (hrow >> 6)][hrow & 63] != 0;
      if (!valid) s = -FLT_MAX;
      float mx = fmaxf(s, __shfl_xor_sync(kFull, s, 8));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
      const float Mn = fmaxf(M, mx);
      const float sc = exp2f(M - Mn);
      const float pm = valid ? exp2f(s - Mn) : 0.f;
      float ps = oct == 0 ? pm : 0.f;
      ps += __shfl_xor_sync(kFull, ps, 8);
      ps += __shfl_xor_sync(kFull, ps, 16);
      l = l * sc + ps;
#pragma unroll
      for (int k = 0; k < 4; ++k) o4[k] *= sc;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __shfl_sync(kFull, pm, 8 * i);
        const uint2 v = *reinterpret_cast<const uint2*>(vh + (4 * warp + i) * kDim + (vofs ^ (8 * i)));
        o4[0] += p * bf16_bits_to_float(v.x & 0xffffu);
        o4[1] += p * __uint_as_float(v.x & 0xffff0000u);
        o4[2] += p * bf16_bits_to_float(v.y & 0xffffu);
        o4[3] += p * __uint_as_float(v.y & 0xffff0000u);
      }
      M = Mn;
      if constexpr (kShared) __syncthreads(); else __syncwarp();  // this half's rows are refilled next
      if (rd < 8) trace_mark(tr, kTrDecodeRound + 2 * rd + 1);
      issue(rd + 2);
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
    if (warp == 0) {
      // lane w: warp w's weight exp2(m_w - max) (0 for a warp without rows)
      const float mw = wml[2 * lane], lw = wml[2 * lane + 1];
      float mx = lw > 0.f ? mw : -FLT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float f = lw > 0.f ? exp2f(mw - mx) : 0.f;
      wml[2 * lane + 1] = f;  // weights replace the sums (read below)
      float lb = lw * f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lb += __shfl_xor_sync(kFull, lb, o);
      if (lane == 0) {
        // the block's (max, sum), to block 0
        dsmem_st_u32(dsmem_addr(&pall[r][0], 0), __float_as_uint(mx));
        dsmem_st_u32(dsmem_addr(&pall[r][1], 0), __float_as_uint(lb));
      }
    }
    __syncthreads();
    if (tid < kDim) {
      float ob = 0.f;
#pragma unroll 8
      for (int w2 = 0; w2 < kWarps; ++w2) ob += wo[w2 * kDim + tid] * wml[2 * w2 + 1];
      dsmem_st_u32(dsmem_addr(&pall[r][4 + tid], 0), __float_as_uint(ob));
    }
    // every block's partial is in block 0; only block 0 reads shared memory
    // after this.  Between the halves of the barrier the last block (not
    // block 0) lists the top-k best first (every slice's entries were in
    // global memory at the barrier before the attention; its row share is
    // the smaller one), then it is done.
    if (a.ord_idx != nullptr && s_rank == 0u && r == cs - 1 && r != 0) {
      cluster_arrive();
      trace_block(a.trace, kTkDecode2, 3);
      order_tail();
      trace_block(a.trace, kTkDecode2, 2);
      cluster_wait();
      return;
    }
    cluster_sync();
    trace_mark(tr, kTrDecode5);
    if (r == 0 && tid < kDim) {
      float mm[kClusterMax], ll[kClusterMax], oo[kClusterMax];
#pragma unroll
      for (int q = 0; q < kClusterMax; ++q) {
        mm[q] = q < cs ? pall[q][0] : 0.f;
        ll[q] = q < cs ? pall[q][1] : 0.f;
        oo[q] = q < cs ? pall[q][4 + tid] : 0.f;
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
    trace_block(a.trace, kTkDecode2, 1);
  }

  // ---- 6. the list best first ------------------------------------------------
  // Without attention every slice's entries are in global memory after one
  // more barrier, and the last block sorts them; with attention a cluster
  // of one block sorts here (a larger one did inside its last barrier).
  if (a.ord_idx != nullptr && s_rank == 0u) {
    if (a.out == nullptr) cluster_sync();
    if (r == cs - 1 && (a.out == nullptr || cs == 1)) order_tail();
  }

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

// Clusters of `cs` decode blocks that fit on the device at once (per device,
// queried once; the kernel's shared-memory limit must be set before).
int active_clusters(const void* func, int cs) {
  static std::mutex mu;
  static int cache[64][kClusterMax + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev][cs] > 0) return cache[dev][cs];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kUBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cs;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    int sms = 0;
    if (dev < 0 || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = cs;
    n = sms / cs > 0 ? sms / cs : 1;
  }
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    cache[dev][cs] = n;
  }
  return n;
}

// Blocks per query head.  A head's cluster runs its phases one after
// another: more blocks per head split the gathers and the passes over keys
// but leave the phase latencies, and a grid of more clusters than fit at
// once runs in waves that pay those latencies again.  The size (at most the
// head's chunks and kClusterMax) minimises waves x per-wave time, the
// per-wave time modelled as kWaveUs + (kHeadUs + kCandUs C) / size: constants
// fitted to the kernel's times on GB300 (32 heads of a 131072-token layer
// take 49 / 71 / 118 us per step at 4 / 2 / 1 blocks per head; 256 heads of
// a 32768-token layer 175 us at 2 and 135 us at 1; 160 heads of a
// 262144-token layer 409 / 366 / 402 us at 4 / 2 / 1).
constexpr float kWaveUs = 27.f, kHeadUs = 20.f, kCandUs = 0.0104f;

int decode_cluster_size(const void* func, int nchunk_active, int64_t heads, int64_t C) {
  const int cmax = nchunk_active < kClusterMax ? nchunk_active : kClusterMax;
  int best = cmax;
  float best_t = 0.f;
  for (int cs = cmax; cs >= 1; --cs) {
    const int64_t slots = active_clusters(func, cs);
    const int64_t waves = (heads + slots - 1) / slots;
    const float t = (float)waves * (kWaveUs + (kHeadUs + kCandUs * (float)C) / (float)cs);
    if (cs == cmax || t < best_t) {
      best = cs;
      best_t = t;
    }
  }
  return best;
}

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
  // Many more candidates than every block can hold: the cluster shares the
  // k-th key search.  Its two cluster barriers and pushes cost about as much as
  // two passes over 24576 keys in global memory, so below that every block
  // still searches all keys itself (measured: 1M-token layer, C = 52403:
  // 36 -> 12 us; 256K-token layer, C = 13081 at 2 blocks per head: 9.1 -> 9.7 us).
  const bool shared = ra.C > kSharedSelectMin;
  const void* func = a.t.cent ? (shared ? (const void*)k_decode<true, true> : (const void*)k_decode<true, false>)
                              : (shared ? (const void*)k_decode<false, true> : (const void*)k_decode<false, false>);
  {
    const SmemKernel which = a.t.cent ? (shared ? kSmemDecodeTableShared : kSmemDecodeTable)
                                      : (shared ? kSmemDecodeShared : kSmemDecode);
    cudaError_t e = set_smem_limit(func, kUBytes, which);
    if (e != cudaSuccess) return e;
  }
  if (ra.nchunk_active < 1) return cudaErrorInvalidValue;
  const int cs = decode_cluster_size(func, ra.nchunk_active, (int64_t)ra.s.batch * ra.s.hq, ra.C);
  a.cpb = (ra.nchunk_active + cs - 1) / cs;
  a.N = ra.N;
  a.C = ra.C;
  a.k = ra.k;
  a.k_eff = ra.k_eff;
  a.cmax = ra.cmax;
  a.nsink = L.nsink;
  a.nwin = L.nwin;
  for (int q = 0; q <= kClusterMax; ++q) {
    const int qq = q < cs ? q : cs;
    a.ccut[q] = ra.C * qq / cs;
    a.rcut[q] = (L.nwin + ra.k_eff) * qq / cs;
  }
  {
    const int ring = ra.s.local + ra.s.ubuf;
    a.nmod = ring > 0 ? (uint32_t)(ra.N % ring) : 0u;
  }
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
  a.ord_idx = L.ord_idx;
  a.ord_sc = L.ord_sc;
  static_assert(kOrderMax * 8 <= kUAttnEnd && 32 * kOrdCount <= kUAttnEnd, "the orderings fit the staging area");
  // With the sort, the last block's share of the attention rows is cut by
  // up to two rounds of rows below what an even share needs (the sort takes
  // about as long as two rounds), as far as the other blocks' larger shares
  // still fit the rounds an even share needs: the sort then overlaps the
  // other blocks' attention.
  // (Not when every block can place its entries best first itself: keys
  // staged, k_eff < C; a crowded bin then still falls back to the sort.)
  const bool placed_directly = ra.C <= kSelCap && ra.k_eff < ra.C;
  if (L.ord_idx != nullptr && L.out != nullptr && cs > 1 && !placed_directly) {
    constexpr int64_t kRoundRows = 128;  // rows per attention round
    const int64_t total = L.nwin + ra.k_eff;
    const int64_t rounds = ((total + cs - 1) / cs + kRoundRows - 1) / kRoundRows;
    for (int64_t cut = 2; cut >= 1; --cut) {
      if (rounds - cut < 0) continue;
      const int64_t last = (rounds - cut) * kRoundRows, rest = total - last;
      if ((rest + cs - 2) / (cs - 1) <= rounds * kRoundRows) {
        for (int q = 0; q <= kClusterMax; ++q) a.rcut[q] = q < cs ? rest * q / (cs - 1) : total;
        break;
      }
    }
  }
  if (L.ord_idx != nullptr && (ra.k_eff > kOrderMax || ra.topk_score == nullptr)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, ra.s.batch * ra.s.hq);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kUBytes;
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
  if (a.t.cent) return shared ? cudaLaunchKernelEx(&cfg, k_decode<true, true>, a) : cudaLaunchKernelEx(&cfg, k_decode<true, false>, a);
  return shared ? cudaLaunchKernelEx(&cfg, k_decode<false, true>, a) : cudaLaunchKernelEx(&cfg, k_decode<false, false>, a);
}

}  // namespace paris
