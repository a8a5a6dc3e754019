// Internal declarations shared by the translation units of the ParisKV CUDA
// library.  Nothing here is part of the C ABI (include/paris.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace paris {

// Geometry the kernels are written for: d = 128 split into B = 16 subspaces
// of m = 8 coordinates, so a bucket id is one byte and the 4-bit codes of a
// subspace fill one 32-bit word.
constexpr int kDim = 128;
constexpr int kSub = 16;
constexpr int kM = 8;
constexpr int kCentroids = 1 << kM;
constexpr int kRecBytes = 128;         // 64 B packed codes + 16 x float w
constexpr int kChunk = 16384;          // keys per inverted-index chunk
constexpr int kOffStride = 264;        // 257 bucket offsets, padded
constexpr int kAttnSplit = 64;         // attention rows per partial block
constexpr int kMaxSplits = 512;        // partial blocks per query head: window + k <= 32768 rows
constexpr int kPartStride = kDim + 4;  // m, l, pad, pad, o[128]
constexpr int kMaxBins = 256;          // vote values 0..255
constexpr int kMaxChunks = 256;        // chunks per (sequence, KV head): 4M Retrieval-zone keys

// RSQ-IP magnitude levels and midpoints, rounded to float32 once, and
// float32(sqrt(d)).
struct RsqParams {
  float lev[8];
  float thr[7];
  float sqrtd;
};

// Diagonal D of the SRHT as a bit mask: bit c set means D_c = -1.
struct SignMask {
  uint32_t w[4];
};

// Device view of one context's key-side tables (per sequence and KV head).
struct Tables {
  uint8_t* ids;      // [batch][Hkv][Rcap][16]
  uint8_t* rec;      // [batch][Hkv][Rcap][128]
  uint16_t* ent;     // [batch][Hkv][nchunk][16][kChunk]
  uint32_t* off;     // [batch][Hkv][nchunk][16][kOffStride]
  int64_t rcap;      // Retrieval-zone capacity (rows)
  int nchunk;        // chunks per (sequence, KV head)
  const float* cent; // learned centroids [Hkv][16][256][8] (nullptr: the analytic sign patterns)
};
constexpr int kTabPerHead = kSub * kCentroids * kM;  // floats of one KV head's centroid table

struct KvStore {
  __nv_bfloat16* win_k;  // [batch][Hkv][win][d]: sink slots then the Local/Buffer ring
  __nv_bfloat16* win_v;
  __nv_bfloat16* st_k;   // [batch][Hkv][rcap][d] by position - S (device address; may be mapped host memory)
  __nv_bfloat16* st_v;
  int win;               // S + L + U
  int64_t rcap;
};

struct Shape {
  int batch, hkv, hq, g;
  int sink, local, ubuf;
};

// ---- cache side: prefill placement, encoding, index build, append ----------
cudaError_t launch_place_kv(const void* K, const void* V, int dtype, int64_t T, int64_t N,
                            const Shape& s, const KvStore& kv, cudaStream_t st);
cudaError_t launch_encode(const void* K, int dtype, int64_t T, int64_t pos0, int64_t pos1,
                          const Shape& s, const Tables& t, const SignMask& sm, const RsqParams& rp,
                          cudaStream_t st);
cudaError_t launch_build_index(int64_t N, int chunk0, int chunk1, const Shape& s, const Tables& t,
                               cudaStream_t st);
cudaError_t launch_append(const void* k, const void* v, int dtype, int64_t pos, const Shape& s,
                          const KvStore& kv, const Tables& t, const SignMask& sm,
                          const RsqParams& rp, cudaStream_t st);

// ---- retrieval ----------------------------------------------------------
struct RetrieveArgs {
  Shape s;
  Tables t;
  SignMask sm;
  RsqParams rp;
  int rho, flat, nbins;
  int64_t N, C, k, k_eff;
  int nchunk_active;
  // scratch
  float* qt;          // [batch*Hq][d]
  float* qnorm;       // [batch*Hq]
  uint32_t* hot;      // [batch*Hq][16*rho]
  uint8_t* votes;     // [batch*Hq][nchunk*kChunk]
  uint32_t* hist;     // [batch*Hq][nchunk][kMaxBins]
  int32_t* cand_idx;  // [batch*Hq][cmax]
  float* cand_est;
  int64_t cmax;
  uint64_t* trace;           // phase timestamps (nullptr: off)
  // outputs
  int32_t* topk_idx;  // [batch*Hq][k]
  float* topk_score;  // may be null
};

// One launch of the fused decode kernel: retrieval for every (sequence,
// query head), optionally the sparse attention (out != nullptr) and the
// append of the step's own token (k_new != nullptr; the zone bookkeeping
// already counts it).
struct DecodeLaunch {
  RetrieveArgs ra;
  KvStore kv;
  int64_t nsink, nwin;  // attention window rows: Sink, then Local + Buffer
  const void* q;
  int qdtype;
  const void* k_new;
  const void* v_new;
  int kvdtype;
  int64_t new_pos;
  uint32_t* status;
  __nv_bfloat16* out;
  // the caller's arrays for the lists best first (ord_idx nullptr: the lists
  // stay in ra.topk_idx / ra.topk_score in ascending position)
  int32_t* ord_idx;
  float* ord_sc;
};

// Launch `kern` so that it may start while the preceding kernel of the
// stream finishes (the kernel itself waits with pdl_wait before it reads
// anything that kernel writes).
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to one device, so it is set once per
// (device, kernel) pair; safe to call from several host threads.
enum SmemKernel {
  kSmemDecode = 0, kSmemDecodeTable, kSmemDecodeShared, kSmemDecodeTableShared, kSmemAttend, kSmemDense,
  kSmemKernelCount
};
cudaError_t set_smem_limit(const void* func, int bytes, SmemKernel which);

int decode_cluster_size(const void* func, int nchunk_active, int64_t heads, int64_t C);
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t st);
cudaError_t launch_fill_empty(int32_t* idx, float* score, int64_t n, cudaStream_t st);

// ---- sparse attention ---------------------------------------------------
struct AttendArgs {
  Shape s;
  KvStore kv;
  int64_t T, N, n_local_buf;  // n_local_buf = tokens in Local + Buffer
  int64_t k, k_eff;
  const int32_t* topk_idx;
  float* part;                // [batch*Hq][nsplit_max][kPartStride]
  int nsplit_max;
  uint32_t* status;
  uint32_t* counter;          // [batch*Hq] splits finished, reset by the last one
  uint64_t* trace;            // phase timestamps (nullptr: off)
  __nv_bfloat16* out;
};
int attend_splits(const AttendArgs& a);
cudaError_t launch_attend(const void* q, int dtype, const AttendArgs& a, cudaStream_t st);

// ---- dense comparator: attention over every cached token --------------------
struct DenseArgs {
  Shape s;
  KvStore kv;
  int64_t T, N;               // tokens cached, Retrieval-zone tokens
  int64_t rows_per_split;     // tokens per block (a multiple of the tile)
  const void* q;
  int qdtype;
  float qscale;               // log2(e) / sqrt(d)
  float* part;                // [batch*Hq][nsplit_max][kPartStride]
  int nsplit_max;
  uint32_t* counter;          // [batch*Hkv] splits finished, reset by the last one
  __nv_bfloat16* out;
  // union mode (GQA-shared sparse attention, topk != nullptr): block
  // (split j of J, sequence x KV head) attends over its share of the window
  // rows (nsink Sink rows, then Local and Buffer) and over the union of the
  // G query heads' top-k positions (topk [batch][Hq][k], first k_eff of
  // each) that fall in its slice of the Retrieval zone, which it builds
  // itself and stores at ulist[sh][zone offset of the slice ...];
  // topk == nullptr: every token
  const int32_t* topk;
  int64_t k, k_eff;
  int32_t* ulist;      // [batch*Hkv][rcap]
  uint32_t* status;
  int64_t nsink, nwin;
};
// Splits per (sequence, KV head) of the union mode: whole waves, and each
// slice's bitmap of the Retrieval zone inside the stage area.
int dense_union_splits(const DenseArgs& a, int sm_count);
int dense_splits(const DenseArgs& a, int sm_count);  // splits per (sequence, KV head)

// Top-k lists best first: at most kOrderMax entries per query head are
// sorted by (estimate descending, position ascending) in one block's shared
// memory at the end of the decode kernel.
constexpr int64_t kOrderMax = 16384;
int64_t dense_rows_per_split(int64_t T, int nsplit);
cudaError_t launch_dense(const DenseArgs& a, int nsplit, cudaStream_t st);

// Status word bits.
constexpr uint32_t kStatusBadIndex = 1u;

// Phase-trace slots (block (0, 0) of each kernel, and the reducing block of
// query head 0).
constexpr int kTraceSlots = 64;
constexpr int kTraceBlocks = 4096;   // per-block stamps: 4 per block and trace row
constexpr int kTraceKernels = 8;
constexpr int64_t kTraceWords = kTraceSlots + (int64_t)kTraceKernels * kTraceBlocks * 4;
// trace rows: the fused decode kernel uses four (start, after wait,
// prepared, voted | compacted, reranked, top-k out, after barrier |
// attention tiles, merged, -, end | rerank start, top-k start, k-th key
// found, output offsets known); the standalone attention one
enum TraceKernel { kTkDecode0 = 0, kTkDecode1, kTkDecode2, kTkAttend, kTkDecode3 };
enum TraceSlot {
  kTrDecode0 = 0, kTrDecode1, kTrDecode2, kTrDecode3, kTrDecode4, kTrDecode5, kTrDecode6,
  kTrDecodeFine = 8,  // 8 .. 28: steps inside the vote and top-k phases
  kTrDecodeRound = 41,  // 40: attention rounds start; 41 + 2 rd: round rd landed, + 1: computed
  kTrAttend0 = 32, kTrAttend1, kTrAttend2, kTrAttend3, kTrAttend4
};

}  // namespace paris
