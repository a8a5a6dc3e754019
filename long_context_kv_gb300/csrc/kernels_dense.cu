// Dense decode attention over every cached token (Sink, Retrieval zone,
// Local, Update Buffer): the full-attention baseline that ParisKV's decode
// throughput is measured against (ParisKV -- Experiments, "Efficiency":
// throughput over full attention; the dense path reads every K/V row once
// per step, the sparse path a few percent of them).
//
// Streaming split-K flash decoding, bound by the read of K and V (HBM, or
// C2C for a Retrieval zone in pinned host memory).  Block (split, sequence
// x KV head) reads the K and V rows of its token range once for all G query
// heads of the KV head (GQA), in tiles of 128 rows through a 3-deep ring of
// 16-byte asynchronous copies.  The G heads are the rows of bf16 mma tiles
// (m16n8k16, float32 accumulation; the query as two bf16 parts): each
// warp takes 16 rows of a tile, S = Q K^T, an online softmax per head, and
// O += P V with P rounded to bf16.  The warps merge in shared memory, the
// block writes one partial (max, sum, o) per head, and the last block of a
// (sequence, KV head) to finish merges the splits (an atomic counter after
// a memory fence; nothing waits).  The tensor pipe is a small fraction of
// the time: it only keeps the per-row instruction count low enough for the
// copies to stream at the memory's rate.
#include <float.h>

#include <algorithm>

#include "paris_device.cuh"

namespace paris {
namespace {

constexpr int kDThreads = 256;
constexpr int kDWarps = kDThreads / 32;
constexpr int kDRowsW = 16;                // rows per warp and tile: one 16-deep k step of P V
constexpr int kDTile = kDRowsW * kDWarps;  // 128 rows per tile
constexpr int kDStages = 3;
constexpr int kDStride = kDim + 8;         // bf16 per row of the staged query: 272 B, conflict-free matrix loads
constexpr int kDMaxHeads = 16;             // query heads per block: the rows of one mma tile
static_assert(kDTile * 16 == kDThreads * 8, "16-byte pieces: 8 per thread and tile for K, 8 for V");
constexpr int kDMaxSplits = 1024;  // splits per (sequence, KV head) the last block's merge tables hold

constexpr size_t kDStageBytes = (size_t)2 * kDStages * kDTile * kDim * sizeof(uint16_t);
constexpr size_t kDMergeBytes = (size_t)(3 * kDMaxHeads * kDMaxSplits + kDMaxHeads) * sizeof(float);
constexpr size_t kDenseSmem = kDStageBytes > kDMergeBytes ? kDStageBytes : kDMergeBytes;
constexpr int kDUnionRows = 1792;  // union positions of a block kept in shared memory (the rest re-read)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

// A staged K or V row is 256 B with its 16-byte pieces permuted by row
// (piece c of row r at c ^ (r & 7)): every 32-byte sector lands whole in an
// aligned 32-byte slot, so a copy instruction is served as whole-sector
// requests (a row stride padded to 272 B splits the sectors of every other
// row, doubling the requests: host-resident rows then stream at about 60 %
// of the link's rate), and each 8-row matrix load touches all 32 banks once.
__device__ __forceinline__ int dpiece(int row, int c) { return row * kDim + 8 * (c ^ (row & 7)); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Four 8x8 bf16 matrices from shared memory (lane i gives the address of
// row i % 8 of matrix i / 8), plain or transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
// d += a b: a 16x16 bf16 (rows: query heads), b 16x8 bf16, d 16x8 float32.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Block (split, sequence x KV head): the G <= 16 query heads of the KV head
// are the rows of the mma tiles (rows G .. 15 are zero).  Warp w takes rows
// 16 w .. 16 w + 15 of every 128-row tile: S = Q K^T over them (two 8-row
// n-tiles, eight 16-deep k steps), an online softmax per head, then
// O += P V (one 16-deep k step, sixteen 8-wide n-tiles of output
// dimensions).  Fragment layouts are those of mma.m16n8k16: lane l holds
// rows l / 4 and l / 4 + 8 and columns 2 (l % 4), 2 (l % 4) + 1.
__global__ void __launch_bounds__(kDThreads, 1) k_dense(DenseArgs a) {
  // The dynamic region follows the static arrays; 128-byte alignment keeps
  // every staged row's 32-byte sectors on sector boundaries (at the default
  // 16-byte alignment it started 16 bytes off one, behind 17.5 KB of static
  // arrays, and every row read from host memory cost twice its sectors).
  extern __shared__ __align__(128) uint16_t dsm[];
  uint16_t* stK = dsm;                             // [kDStages][kDTile][kDim], pieces permuted (dpiece)
  uint16_t* stV = dsm + kDStages * kDTile * kDim;
  __shared__ __align__(16) uint16_t qsh[2][kDMaxHeads][kDStride];  // the query as bf16 hi + lo
  __shared__ float wml[kDWarps][kDMaxHeads][2];
  __shared__ float fs[kDMaxHeads][kDWarps];
  __shared__ int s_last;
  pdl_wait();  // the list, its length and the cache may come from the kernel before

  const int split = blockIdx.x;
  const int sh_i = blockIdx.y;  // sequence * Hkv + KV head
  const int seq = sh_i / a.s.hkv, kvh = sh_i - seq * a.s.hkv;
  const int64_t sh = (int64_t)sh_i;
  const int G = a.s.g, qh0 = kvh * G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ring = a.s.local + a.s.ubuf;
  // Union mode: this block's share of the window rows, [w_lo, w_lo + nw),
  // then the union of the G heads' top-k positions in its slice [z_lo, z_hi)
  // of the Retrieval zone: every listed position sets its bit in a bitmap of
  // the slice (in the stage area, before any tile), the set bits are read out
  // in order (a block scan of the threads' bit counts places them) into
  // ulist, nu of them, the first kDUnionRows also into shared memory.  Rows
  // t < nw are window rows, the rest the union's positions.
  __shared__ int32_t sul[kDUnionRows];
  int64_t w_lo = 0, nw = 0, z_lo = 0;
  int32_t* ul = nullptr;
  int nu = 0;
  if (a.topk != nullptr) {
    const int J = gridDim.x;
    w_lo = a.nwin * split / J;
    nw = a.nwin * (split + 1) / J - w_lo;
    z_lo = a.N * split / J;
    const int64_t z_hi = a.N * (split + 1) / J;
    const int nwords = (int)((z_hi - z_lo + 31) / 32);
    uint32_t* bm = reinterpret_cast<uint32_t*>(dsm);
    __shared__ uint32_t utmp[33];
    for (int w = tid; w < nwords; w += kDThreads) bm[w] = 0u;
    __syncthreads();
    // the G lists' entries, eight loads in flight per thread
    const int tot = G * (int)a.k_eff;
    for (int e0 = tid; e0 < tot; e0 += 8 * kDThreads) {
      int32_t pv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kDThreads;
        pv[u] = -1;
        if (e < tot) {
          const int h = e / (int)a.k_eff, i = e - h * (int)a.k_eff;
          pv[u] = __ldcg(a.topk + ((int64_t)seq * a.s.hq + qh0 + h) * a.k + i);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int32_t p = pv[u];
        if (p >= a.s.sink && p < a.s.sink + a.N) {
          const int64_t off = p - a.s.sink;
          if (off >= z_lo && off < z_hi) atomicOr(&bm[(off - z_lo) >> 5], 1u << ((off - z_lo) & 31));
        } else if (p >= 0) {
          atomicOr(a.status, kStatusBadIndex);
        }
      }
    }
    __syncthreads();
    const int per = (nwords + kDThreads - 1) / kDThreads;
    const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
    uint32_t cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += (uint32_t)__popc(bm[w]);
    uint32_t total;
    uint32_t at = block_excl_scan(cnt, utmp, &total);
    ul = a.ulist + sh * a.kv.rcap + z_lo;
    for (int w = w0; w < w1; ++w) {
      uint32_t bits = bm[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int32_t p = (int32_t)(a.s.sink + z_lo + 32 * (int64_t)w + b);
        if (at < (uint32_t)kDUnionRows) sul[at] = p;
        else ul[at] = p;
        ++at;
      }
    }
    nu = (int)total;
    __syncthreads();  // the bitmap's stage area is free, the list is written
  }
  // rows of the block: [t0, t1) of every token (a split of rows_per_split),
  // or the block's window rows and union positions
  const int64_t t0 = a.topk ? 0 : (int64_t)split * a.rows_per_split;
  const int64_t t1 = a.topk ? nw + nu : min64(a.T, t0 + a.rows_per_split);
  const int nrows = (int)max64(0, t1 - t0);
  const int ntiles = (nrows + kDTile - 1) / kDTile;

  // where row t's K/V is: the Sink slots and the Local/Buffer ring of the
  // window arrays, or the Retrieval-zone store.  Dense: row t is token t.
  // Union mode: rows below nw are the window rows w_lo + t (Sink, then Local
  // and Buffer in position order), the rest the union's positions.
  auto row_ptrs = [&](int64_t t, const __nv_bfloat16*& kp, const __nv_bfloat16*& vp) {
    if (a.topk) {
      if (t < nw) {
        t += w_lo;
        t = t < a.nsink ? t : a.s.sink + a.N + (t - a.nsink);
      } else {
        t = t - nw < kDUnionRows ? sul[t - nw] : __ldcg(ul + (t - nw));
      }
    }
    if (t < a.s.sink || t >= a.s.sink + a.N) {
      const int64_t slot = t < a.s.sink ? t : a.s.sink + (t - a.s.sink) % ring;
      kp = a.kv.win_k + (sh * a.kv.win + slot) * kDim;
      vp = a.kv.win_v + (sh * a.kv.win + slot) * kDim;
    } else {
      kp = a.kv.st_k + (sh * a.kv.rcap + (t - a.s.sink)) * kDim;
      vp = a.kv.st_v + (sh * a.kv.rcap + (t - a.s.sink)) * kDim;
    }
  };
  // tile i into stage i % kDStages: thread t copies pieces (t % 16) of rows
  // t / 16 + 16 j, j = 0 .. 7, of K and of V
  auto issue = [&](int i) {
    if (i < ntiles) {
      const int st = i % kDStages, ch = tid & 15;
#pragma unroll
      for (int j = 0; j < kDTile * 16 / kDThreads; ++j) {
        const int rr = (tid >> 4) + 16 * j;
        const int64_t t = t0 + (int64_t)i * kDTile + rr;
        uint16_t* kd = stK + dpiece(st * kDTile + rr, ch);
        uint16_t* vd = stV + dpiece(st * kDTile + rr, ch);
        if (t < t1) {
          const __nv_bfloat16 *kp, *vp;
          row_ptrs(t, kp, vp);
          cp_async16(kd, kp + 8 * ch);
          cp_async16(vd, vp + 8 * ch);
        } else {
          // past the split: zeros, so the products read finite values
          *reinterpret_cast<uint4*>(kd) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vd) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kDStages - 1; ++i) issue(i);

  // the KV head's queries, scaled by log2(e) / sqrt(d) (softmax in base 2),
  // as the sum of two bf16 parts (hi, and the rest rounded again): the
  // scores keep about 16 significant bits of q
  for (int e = tid; e < kDMaxHeads * kDim; e += kDThreads) {
    const int h = e / kDim, d = e % kDim;
    const float v = h < G ? load1(a.q, a.qdtype, ((int64_t)seq * a.s.hq + qh0 + h) * kDim + d) * a.qscale : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    reinterpret_cast<__nv_bfloat16*>(qsh[0][h])[d] = hi;
    reinterpret_cast<__nv_bfloat16*>(qsh[1][h])[d] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
  __syncthreads();
  uint32_t qa[2][kDim / 16][4];  // A fragments of Q (hi, lo), one per 16-deep k step
#pragma unroll
  for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
    for (int ks = 0; ks < kDim / 16; ++ks)
      ldsm_x4(qa[p2][ks], &qsh[p2][(lane & 7) + ((lane >> 3) & 1) * 8][16 * ks + (lane >> 4) * 8]);

  const int hr = lane >> 2, cc = 2 * (lane & 3);  // fragment row (head hr and hr + 8), column pair
  float M[2] = {-FLT_MAX, -FLT_MAX}, l[2] = {0.f, 0.f};
  float o[kDim / 8][4];
#pragma unroll
  for (int nt = 0; nt < kDim / 8; ++nt)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[nt][k] = 0.f;

  for (int i = 0; i < ntiles; ++i) {
    cp_async_wait_group<kDStages - 2>();  // tile i has landed
    __syncthreads();                      // ... for every thread; stage (i - 1) % kDStages is free
    issue(i + kDStages - 1);
    const int st = i % kDStages;
    const uint16_t* kt = stK + (st * kDTile + kDRowsW * warp) * kDim;  // 16 rows: the permutation restarts
    const uint16_t* vt = stV + (st * kDTile + kDRowsW * warp) * kDim;
    // S = Q K^T for the warp's 16 rows: n-tile r holds rows 8 r .. 8 r + 7
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
#pragma unroll
      for (int k2 = 0; k2 < kDim / 32; ++k2) {
        // matrices: rows 8 r .. 8 r + 7, dims 32 k2 + 8 m .. + 7
        uint32_t b[4];
        ldsm_x4(b, kt + dpiece(8 * r + (lane & 7), 4 * k2 + (lane >> 3)));
        mma16816(s[r], qa[0][2 * k2], b[0], b[1]);
        mma16816(s[r], qa[1][2 * k2], b[0], b[1]);
        mma16816(s[r], qa[0][2 * k2 + 1], b[2], b[3]);
        mma16816(s[r], qa[1][2 * k2 + 1], b[2], b[3]);
      }
    }
    // online softmax per head: rows past the split score -inf
    const int64_t rbase = t0 + (int64_t)i * kDTile + kDRowsW * warp;
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (rbase + 8 * r + cc + (k & 1) >= t1) s[r][k] = -FLT_MAX;
    float sc[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // head hr (hh = 0) and hr + 8 (hh = 1)
      float mx = fmaxf(fmaxf(s[0][2 * hh], s[0][2 * hh + 1]), fmaxf(s[1][2 * hh], s[1][2 * hh + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float Mn = fmaxf(M[hh], mx);
      sc[hh] = exp2f(M[hh] - Mn);
      float ps = 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int k = 2 * hh; k < 2 * hh + 2; ++k) {
          s[r][k] = s[r][k] == -FLT_MAX ? 0.f : exp2f(s[r][k] - Mn);
          ps += s[r][k];
        }
      ps += __shfl_xor_sync(kFull, ps, 1);
      ps += __shfl_xor_sync(kFull, ps, 2);
      l[hh] = l[hh] * sc[hh] + ps;
      M[hh] = Mn;
    }
    // O = O * scale + P V: P as the A fragment of one 16-deep k step over the rows
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
    for (int n2 = 0; n2 < kDim / 16; ++n2) {
      // matrices: rows 0-7 / 8-15 of the warp's rows, dims 16 n2 .. + 7 / + 8 .. + 15
      uint32_t b[4];
      ldsm_x4_t(b, vt + dpiece((lane & 7) + 8 * ((lane >> 3) & 1), 2 * n2 + (lane >> 4)));
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float* on = o[2 * n2 + h2];
        on[0] *= sc[0];
        on[1] *= sc[0];
        on[2] *= sc[1];
        on[3] *= sc[1];
        mma16816(o[2 * n2 + h2], pa, b[2 * h2], b[2 * h2 + 1]);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // merge the warps: wo[w][head][d] in the (now idle) stage area
  float* wo = reinterpret_cast<float*>(dsm);
  static_assert((size_t)kDWarps * kDMaxHeads * kDim * sizeof(float) <= kDenseSmem, "warp partials fit the stage area");
#pragma unroll
  for (int nt = 0; nt < kDim / 8; ++nt) {
    wo[(warp * kDMaxHeads + hr) * kDim + 8 * nt + cc] = o[nt][0];
    wo[(warp * kDMaxHeads + hr) * kDim + 8 * nt + cc + 1] = o[nt][1];
    wo[(warp * kDMaxHeads + hr + 8) * kDim + 8 * nt + cc] = o[nt][2];
    wo[(warp * kDMaxHeads + hr + 8) * kDim + 8 * nt + cc + 1] = o[nt][3];
  }
  if ((lane & 3) == 0) {
    wml[warp][hr][0] = M[0];
    wml[warp][hr][1] = l[0];
    wml[warp][hr + 8][0] = M[1];
    wml[warp][hr + 8][1] = l[1];
  }
  __syncthreads();
  float* part = a.part + (((int64_t)seq * a.s.hq + qh0) * a.nsplit_max + split) * kPartStride;
  for (int h = warp; h < G; h += kDWarps) {
    // head h's weights exp2(m_w - max) over the warps (0 for a warp without rows)
    const float mw = lane < kDWarps ? wml[lane][h][0] : -FLT_MAX, lw = lane < kDWarps ? wml[lane][h][1] : 0.f;
    float mx = lw > 0.f ? mw : -FLT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    const float f = lw > 0.f ? exp2f(mw - mx) : 0.f;
    if (lane < kDWarps) fs[h][lane] = f;
    float lb = lw * f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lb += __shfl_xor_sync(kFull, lb, off);
    if (lane == 0) {
      part[(int64_t)h * a.nsplit_max * kPartStride] = mx;
      part[(int64_t)h * a.nsplit_max * kPartStride + 1] = lb;
    }
  }
  __syncthreads();
  for (int e = tid; e < G * kDim; e += kDThreads) {
    const int h = e / kDim, d = e % kDim;
    float ob = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) ob += wo[(w * kDMaxHeads + h) * kDim + d] * fs[h][w];
    part[(int64_t)h * a.nsplit_max * kPartStride + 4 + d] = ob;
  }

  // the last split of the (sequence, KV head) merges all splits
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counter[blockIdx.y], 1u) == (uint32_t)(gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // every split's (max, sum) of every head at once, then per head the
  // weights exp2(m_s - max) (0 for a split without rows), then each output
  // element's weighted sum over the splits with its loads 32 at a time; a
  // thread's first batch of its first element goes out before the weights
  const int nsplit = gridDim.x;
  float* ml = reinterpret_cast<float*>(dsm);  // [G][nsplit][2], then f [G][nsplit], then Lt [G]
  float* fw = ml + 2 * G * nsplit;
  float* lt = fw + G * nsplit;
  constexpr int kMB = 32;
  auto elem_at = [&](int e) {
    return a.part + (((int64_t)seq * a.s.hq + qh0 + e / kDim) * a.nsplit_max) * kPartStride + 4 + e % kDim;
  };
  float oo[kMB];
  if (tid < G * kDim) {
    const float* ph = elem_at(tid);
#pragma unroll
    for (int u = 0; u < kMB; ++u) oo[u] = u < nsplit ? __ldcg(ph + (int64_t)u * kPartStride) : 0.f;
  }
  for (int e = tid; e < G * nsplit; e += kDThreads) {
    const int h = e / nsplit, s0 = e - h * nsplit;
    const float* ph = a.part + (((int64_t)seq * a.s.hq + qh0 + h) * a.nsplit_max + s0) * kPartStride;
    ml[2 * e] = __ldcg(ph);
    ml[2 * e + 1] = __ldcg(ph + 1);
  }
  __syncthreads();
  for (int h = warp; h < G; h += kDWarps) {
    float Mx = -FLT_MAX;
    for (int s0 = lane; s0 < nsplit; s0 += 32)
      if (ml[2 * (h * nsplit + s0) + 1] > 0.f) Mx = fmaxf(Mx, ml[2 * (h * nsplit + s0)]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(kFull, Mx, off));
    float L = 0.f;
    for (int s0 = lane; s0 < nsplit; s0 += 32) {
      const float mm = ml[2 * (h * nsplit + s0)], ll = ml[2 * (h * nsplit + s0) + 1];
      const float f = ll > 0.f ? exp2f(mm - Mx) : 0.f;
      fw[h * nsplit + s0] = f;
      L += ll * f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    if (lane == 0) lt[h] = L;
  }
  __syncthreads();
  for (int e = tid; e < G * kDim; e += kDThreads) {
    const int h = e / kDim, d = e % kDim;
    const float* ph = elem_at(e);
    float ot = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += kMB) {
      if (s0 > 0 || e != tid) {
#pragma unroll
        for (int u = 0; u < kMB; ++u) oo[u] = s0 + u < nsplit ? __ldcg(ph + (int64_t)(s0 + u) * kPartStride) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kMB; ++u)
        if (s0 + u < nsplit) ot += oo[u] * fw[h * nsplit + s0 + u];
    }
    const float L = lt[h];
    a.out[((int64_t)seq * a.s.hq + qh0 + h) * kDim + d] = __float2bfloat16_rn(L > 0.f ? ot / L : 0.f);
  }
  if (tid == 0) a.counter[blockIdx.y] = 0;
}

}  // namespace

int dense_splits(const DenseArgs& a, int sm_count) {
  // Splits per (sequence, KV head): the fewest that fill whole waves of one
  // block per SM (every block of a split has the same rows, so a partial
  // last wave idles SMs), at least one tile per split.
  const int64_t units = (int64_t)a.s.batch * a.s.hkv;
  const int64_t most = std::max<int64_t>(1, std::min<int64_t>({(a.T + kDTile - 1) / kDTile, (int64_t)a.nsplit_max}));
  int64_t best = 1;
  double best_eff = -1.0;
  for (int64_t n = 1; n <= most; ++n) {
    const int64_t blocks = n * units;
    const int64_t waves = (blocks + sm_count - 1) / sm_count;
    // fraction of the SM slots of those waves that hold a block, counting
    // one wave as full when the grid is smaller than the GPU
    const double eff = blocks < sm_count ? (double)blocks / sm_count : (double)blocks / (waves * sm_count);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = n;
    }
    if (eff > 0.999) break;
  }
  return (int)best;
}

int dense_union_splits(const DenseArgs& a, int sm_count) {
  // rows per (sequence, KV head): the window and at most G k_eff positions;
  // each slice's bitmap (zone bits / splits) must fit the stage area
  DenseArgs r = a;
  r.T = a.nwin + (int64_t)a.s.g * a.k_eff;
  int n = dense_splits(r, sm_count);
  const int64_t min_split = (a.N + (int64_t)kDenseSmem * 8 - 1) / ((int64_t)kDenseSmem * 8);
  if (n < min_split) n = (int)min_split;
  return n;
}

int64_t dense_rows_per_split(int64_t T, int nsplit) {
  const int64_t r = (T + nsplit - 1) / nsplit;
  return (r + kDTile - 1) / kDTile * kDTile;
}

cudaError_t launch_dense(const DenseArgs& a, int nsplit, cudaStream_t st) {
  static_assert((size_t)(3 * kDMaxHeads * kDMaxSplits + kDMaxHeads) * sizeof(float) <= kDenseSmem,
                "the merge tables fit the stage area");
  if (a.s.g > kDMaxHeads || nsplit > kDMaxSplits) return cudaErrorInvalidValue;
  {
    const cudaError_t e = set_smem_limit((const void*)k_dense, (int)kDenseSmem, kSmemDense);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k_dense, dim3(nsplit, a.s.batch * a.s.hkv), dim3(kDThreads), kDenseSmem, st, a);
}

}  // namespace paris
