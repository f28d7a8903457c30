// Fused single-pass N-way reduce + broadcast with bulk copies (TMA).
//
// Same result as fused.cu, bit for bit: every element of every rank is read
// once, folded in the declared order, and the result written once to every
// rank (primer ch. 4, "Collective communication: algorithms, cost and the
// library that runs them", §4.4: each rank sends its buffer once and receives
// the sum once). What differs is how the bytes move:
//
//  - a producer warp issues, per tile, one cp.async.bulk load per rank (the
//    rank's slice of the tile, T bytes) into a ring of S shared-memory stages,
//    counted on the stage's "full" mbarrier;
//  - eight consumer warps fold the N slices from shared memory in the declared
//    order (slot p holds the rank at fold position p), write the result tile
//    to one of two output buffers, and free the stage on its "empty" mbarrier;
//  - one consumer thread issues one cp.async.bulk store per rank from the
//    output buffer.
//
// Up to S x N x T (~200 KB) of loads are in flight per SM. Measured on GB300,
// this still moves fewer bytes per SM than the register pipeline's 2 CTAs of
// batched 16-byte loads (about 24 against 45 GB/s of loads per SM under an SM
// budget; both are HBM-bound on the whole GPU), so it runs only when a plan
// asks for it (AR_KERNEL_BULK).
//
// Ragged segment heads and tails (fewer than one 16-byte vector) are folded
// element by element from global memory by the CTA that owns the segment.
//
// Every mbarrier wait is bounded (bulk.cuh); a timeout sets the library's
// device status word, raises the CTA's abort flag, and the CTA winds down
// after its outstanding copies.
#include <atomic>

#include "bulk.cuh"
#include "common.cuh"

namespace ar {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;  // + one producer warp
constexpr uint32_t kWaitPolls = 1u << 22;     // polls before a wait gives up
constexpr int kMaxStages = 8;
constexpr int kTmaMaxRanks = 24;
constexpr int kTmaSmemLimit = 227 * 1024;


// Plain (generic) loads and stores for the shared-memory side of the folds.
template <bool BF16>
struct LaneSm;
template <>
struct LaneSm<false> {
  static constexpr int W = 4;
  using raw_t = uint4;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return *reinterpret_cast<const uint4*>(base + e * 4);
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) { Lane<false, true>::widen(r, f); }
};
template <>
struct LaneSm<true> {
  static constexpr int W = 8;
  using raw_t = uint4;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return *reinterpret_cast<const uint4*>(base + e * 2);
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) { Lane<true, true>::widen(r, f); }
};

struct TmaCfg {
  int stages;
  int tile_bytes;  // per rank per stage, a multiple of 4096
};

// Same segment and fold-sequence rules as fused.cu (all-reduce only).
__device__ __forceinline__ void tma_seg_range(const FusedParams& p, int seg, int64_t& lo, int64_t& hi) {
  const int64_t L = p.count;
  if (p.order == AR_ORDER_RING) {
    lo = seg * L / p.n;
    hi = (seg + 1) * L / p.n;
  } else if (p.order == AR_ORDER_HIER) {
    const int k = seg / p.m, j = seg - (seg / p.m) * p.m;
    const int64_t sk = k * L / p.g, ek = (k + 1) * L / p.g, Lk = ek - sk;
    lo = sk + j * Lk / p.m;
    hi = sk + (j + 1) * Lk / p.m;
  } else {
    lo = 0;
    hi = L;
  }
  if (lo < p.e_lo) lo = p.e_lo;
  if (hi > p.e_hi) hi = p.e_hi;
}

__device__ __forceinline__ void tma_seq(const FusedParams& p, int seg, int pos, int& rank, uint8_t& flag) {
  const int n = p.n;
  if (p.order == AR_ORDER_HIER) {
    const int g = p.g, m = p.m;
    const int k = seg / m, j = seg - (seg / m) * m;
    const int mi = pos / g, i = pos - mi * g;
    int grp = j + mi;
    if (grp >= m) grp -= m;
    rank = grp * g + (k + 1 + i) % g;
    flag = (i == 0 ? kStart : 0) | (i == g - 1 ? kEnd : 0) | (mi == 0 ? kFirst : 0);
  } else {
    int r = pos;
    if (p.order == AR_ORDER_RING) {
      r = seg + pos;
      if (r >= n) r -= n;
    }
    rank = r;
    flag = (pos == 0 ? kStart : 0) | (pos == n - 1 ? (kEnd | kFirst) : 0);
  }
}

// ---------------------------------------------------------------------------
// Tile sources. A source walks the tiles of one CTA (t = blockIdx.x,
// blockIdx.x + gridDim.x, ...) incrementally, without divisions per tile, and
// gives each non-empty tile's element range, its segment, the input pointer
// of fold position p and the output pointer of rank r.
// ---------------------------------------------------------------------------

// Flat buffers: segments of constant order (chunks, hierarchical sub-chunks or
// the whole buffer), each with its own aligned body cut into tiles.
struct FlatSource {
  const FusedParams& p;
  int64_t tile_elems;
  int W;
  int64_t t, total;
  int seg, tt;  // current tile: segment and tile inside it
  int64_t a0, a1;
  __device__ FlatSource(const FusedParams& p_, int64_t te, int w) : p(p_), tile_elems(te), W(w) {
    total = int64_t(p.n_seg) * p.tiles_per_seg;
    t = blockIdx.x;
    seg = -1;
  }
  __device__ void body(int sg) {
    int64_t slo, shi;
    tma_seg_range(p, sg, slo, shi);
    a0 = round_up(slo, W);
    a1 = round_down(shi, W);
    if (a1 < a0) a1 = a0;
  }
  // Advance to the next non-empty tile; false when none is left.
  __device__ bool next(int& sg, int64_t& lo, int64_t& hi) {
    while (t < total) {
      if (seg < 0) {
        seg = int(t / p.tiles_per_seg);
        tt = int(t - int64_t(seg) * p.tiles_per_seg);
        body(seg);
      }
      lo = a0 + int64_t(tt) * tile_elems;
      hi = lo + tile_elems < a1 ? lo + tile_elems : a1;
      sg = seg;
      t += gridDim.x;  // step to the following tile of this CTA
      tt += gridDim.x;
      bool moved = false;
      while (tt >= p.tiles_per_seg) {
        tt -= int(p.tiles_per_seg);
        ++seg;
        moved = true;
      }
      if (moved && t < total) body(seg);
      if (hi > lo) return true;
    }
    return false;
  }
  __device__ const char* in(int sg, int pos) const {
    int rank;
    uint8_t fl;
    tma_seq(p, sg, pos, rank, fl);
    return static_cast<const char*>(p.in[rank]);
  }
  __device__ char* out(int, int r) const { return static_cast<char*>(p.out[r]); }
};

// Buckets: segments are pieces of tensors between ring-chunk boundaries of the
// packed bucket; each is folded in ring order from its chunk's rank.
struct BucketSource {
  const BucketFusedParams& p;
  int64_t tile_elems;
  int W;
  int t, total, seg;
  int64_t a0, a1;
  __device__ BucketSource(const BucketFusedParams& p_, int64_t te, int w) : p(p_), tile_elems(te), W(w) {
    total = p.tile_start[p.n_seg];
    t = blockIdx.x;
    seg = 0;
  }
  __device__ bool next(int& sg, int64_t& lo, int64_t& hi) {
    while (t < total) {
      while (p.tile_start[seg + 1] <= t) ++seg;
      const BucketSeg& b = p.seg[seg];
      a0 = round_up(b.lo, W);
      a1 = round_down(b.hi, W);
      if (a1 < a0) a1 = a0;
      lo = a0 + int64_t(t - p.tile_start[seg]) * tile_elems;
      hi = lo + tile_elems < a1 ? lo + tile_elems : a1;
      sg = seg;
      t += gridDim.x;
      if (hi > lo) return true;
    }
    return false;
  }
  __device__ const char* in(int sg, int pos) const {
    const BucketSeg& b = p.seg[sg];
    int r = b.rot + pos;
    if (r >= p.n) r -= p.n;
    return static_cast<const char*>(p.ptr[b.t * p.n + r]);
  }
  __device__ char* out(int sg, int r) const { return static_cast<char*>(p.ptr[p.seg[sg].t * p.n + r]); }
};

// Combine flags of fold position `pos` (the same for every segment): one
// sequential fold, or the hierarchical order's groups.
__device__ __forceinline__ uint8_t src_flag(const FlatSource& s, int pos, int n) {
  int rank;
  uint8_t fl;
  tma_seq(s.p, 0, pos, rank, fl);
  return fl;
}
__device__ __forceinline__ uint8_t src_flag(const BucketSource&, int pos, int n) {
  return (pos == 0 ? kStart : 0) | (pos == n - 1 ? (kEnd | kFirst) : 0);
}

// What the producer tells the consumers about the tile in a stage.
struct TileInfo {
  int64_t lo;
  int elems;  // < 0: no more tiles
  int seg;
};

// The pipeline shared by the flat and bucket kernels (see the file comment).
template <bool BF16, bool TREE, int VPT, class Src>
__device__ __forceinline__ void tma_pipeline(Src& src, int n, float scale, const TmaCfg& c, unsigned char* smem) {
  using LS = LaneSm<BF16>;
  constexpr int W = LS::W;
  constexpr int64_t ES = BF16 ? 2 : 4;
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ const char* slot[kMaxStages][kTmaMaxRanks];
  __shared__ uint8_t flag[kTmaMaxRanks];
  __shared__ TileInfo info[kMaxStages];
  __shared__ int abort_flag;

  const int S = c.stages, T = c.tile_bytes;
  unsigned char* out_buf[2] = {smem + size_t(S) * n * T, smem + size_t(S) * n * T + T};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    abort_flag = 0;
    mbar_init_fence();
  }
  for (int i = threadIdx.x; i < S * n; i += blockDim.x)
    slot[i / n][i % n] = reinterpret_cast<const char*>(smem + size_t(i) * T);
  __syncthreads();
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ---------------- producer: lane 0 issues every bulk load
    if (lane == 0) {
      int it = 0, cached = -1;
      const char* src_ptr[kTmaMaxRanks];
      int seg;
      int64_t lo, hi;
      bool more = true;
      while (!*abort) {
        more = src.next(seg, lo, hi);
        const int s = it % S;
        const uint32_t ph = uint32_t(it / S) & 1u;
        if (it >= S && !mbar_wait(&empty[s], ph ^ 1u, kWaitPolls, abort)) break;
        if (!more) {  // tell the consumers there is nothing more
          info[s].elems = -1;
          mbar_arrive(&full[s]);
          break;
        }
        if (seg != cached) {
#pragma unroll 1
          for (int pos = 0; pos < n; ++pos) src_ptr[pos] = src.in(seg, pos);
          cached = seg;
        }
        const uint32_t bytes = uint32_t((hi - lo) * ES);
        info[s].lo = lo;
        info[s].elems = int(hi - lo);
        info[s].seg = seg;
        mbar_arrive_expect_tx(&full[s], bytes * uint32_t(n));
#pragma unroll 1
        for (int pos = 0; pos < n; ++pos) bulk_load(const_cast<char*>(slot[s][pos]), src_ptr[pos] + lo * ES, bytes, &full[s]);
        ++it;
      }
      if (*abort) {
        // Let the loads already issued land before shared memory goes away:
        // the last S issued are the only ones that can be in flight (a stage
        // is refilled only after its previous load completed and was
        // consumed), and a wait on a phase that already completed returns at
        // once. A bulk load reads device memory the host validated, so it
        // completes in microseconds; each poll may suspend the thread in
        // hardware, so 2^16 polls per stage allow far longer than that.
        for (int k = it > S ? it - S : 0; k < it; ++k) {
          volatile int never = 0;
          mbar_wait(&full[k % S], uint32_t(k / S) & 1u, 1u << 16, &never);
        }
      }
    }
    return;
  }

  // ---------------- consumers
  const int tid = threadIdx.x - 32;
  if (tid < n) flag[tid] = src_flag(src, tid, n);
  named_barrier(1, kConsumers);
  for (int it = 0;; ++it) {
    const int s = it % S;
    const uint32_t ph = uint32_t(it / S) & 1u;
    mbar_wait(&full[s], ph, kWaitPolls, abort);  // a timeout raises the abort flag
    unsigned char* out = out_buf[it & 1];
    if (tid == 0) bulk_wait_read<1>();  // the stores that last read this buffer are done with it
    named_barrier(1, kConsumers);       // buffer free; every consumer sees the same abort flag
    if (*abort) break;
    const TileInfo ti = info[s];
    if (ti.elems < 0) break;
    int64_t e[VPT];
    bool ok[VPT];
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = (int64_t(q) * kConsumers + tid) * W;
      ok[q] = e[q] < ti.elems;
    }
    float acc[VPT][W];
    // shared memory answers fast: a batch of 8/VPT slots per vector is enough
    if (TREE) {
#pragma unroll
      for (int q = 0; q < VPT; ++q)
        if (ok[q]) fold_tree<LS, 4>(acc[q], slot[s], n, e[q]);
    } else {
      fold_sequence<LS, 8 / VPT, VPT>(acc, slot[s], flag, n, e, ok);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp has read the stage
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      if (!ok[q]) continue;
#pragma unroll
      for (int w = 0; w < W; ++w) acc[q][w] = fmul(acc[q][w], scale);
      *reinterpret_cast<uint4*>(out + e[q] * ES) = Lane<BF16, true>::narrow(acc[q]);
    }
    fence_proxy_async();  // make the result visible to the bulk stores
    named_barrier(1, kConsumers);
    if (tid == 0) {
      const uint32_t bytes = uint32_t(ti.elems * ES);
      for (int r = 0; r < n; ++r) bulk_store(src.out(ti.seg, r) + ti.lo * ES, out, bytes);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait_all();  // every bulk store has completed before the CTA exits
}

// Ragged heads and tails of a flat launch's segments, element by element from
// global memory, by the consumer threads of the CTA that owns the segment.
template <bool BF16, bool TREE>
__device__ __forceinline__ void flat_heads_tails(const FusedParams& p) {
  using LG = Lane<BF16, false>;
  constexpr int W = BF16 ? 8 : 4;
  const int n = p.n;
  const int tid = int(threadIdx.x) - 32;
  if (tid < 0) return;
  for (int seg = blockIdx.x; seg < p.n_seg; seg += gridDim.x) {
    int64_t slo, shi;
    tma_seg_range(p, seg, slo, shi);
    if (shi <= slo) continue;
    const int64_t a0 = round_up(slo, W);
    int64_t a1 = round_down(shi, W);
    if (a1 < a0) a1 = a0;
    const int64_t head_end = a0 < shi ? a0 : shi;
    int64_t es = -1;
    if (tid < W - 1) {
      es = slo + tid;
      if (es >= head_end) es = -1;
    } else if (tid >= 32 && tid < 32 + W - 1) {
      es = a1 + (tid - 32);
      if (es >= shi) es = -1;
    }
    if (es < 0) continue;
    float total_sum = 0.f;
    if (TREE) {  // the balanced tree over ranks in index order
      float lvl[kTreeLevels];
      for (int pos = 0; pos < n; ++pos) {
        float f[1];
        LG::widen(LG::load(static_cast<const char*>(p.in[pos]), es), f);
        float carry = f[0];
        int bits = pos;
        for (int l = 0; l < kTreeLevels; ++l) {
          if (bits & 1) {
            carry = fadd(lvl[l], carry);
            bits >>= 1;
          } else {
            lvl[l] = carry;
            break;
          }
        }
      }
      for (int l = 0; l < kTreeLevels; ++l)
        if ((1 << l) == n) total_sum = lvl[l];
    } else {
      float part = 0.f;
      for (int pos = 0; pos < n; ++pos) {
        int rank;
        uint8_t fl;
        tma_seq(p, seg, pos, rank, fl);
        float f[1];
        LG::widen(LG::load(static_cast<const char*>(p.in[rank]), es), f);
        part = (fl & kStart) ? f[0] : fadd(part, f[0]);
        if (fl & kEnd) total_sum = (fl & kFirst) ? part : fadd(total_sum, part);
      }
    }
    float v[1] = {fmul(total_sum, p.scale)};
    const typename LG::raw_t r = LG::narrow(v);
    for (int q = 0; q < n; ++q) LG::store(static_cast<char*>(p.out[q]), es, r);
  }
}

// Ragged heads and tails of a bucket launch's segments (ring order).
template <bool BF16>
__device__ __forceinline__ void bucket_heads_tails(const BucketFusedParams& p) {
  using LG = Lane<BF16, false>;
  constexpr int W = BF16 ? 8 : 4;
  const int n = p.n;
  const int tid = int(threadIdx.x) - 32;
  if (tid < 0) return;
  for (int sgi = blockIdx.x; sgi < p.n_seg; sgi += gridDim.x) {
    const BucketSeg& b = p.seg[sgi];
    const int64_t a0 = round_up(b.lo, W);
    int64_t a1 = round_down(b.hi, W);
    if (a1 < a0) a1 = a0;
    const int64_t head_end = a0 < b.hi ? a0 : b.hi;
    int64_t es = -1;
    if (tid < W - 1) {
      es = b.lo + tid;
      if (es >= head_end) es = -1;
    } else if (tid >= 32 && tid < 32 + W - 1) {
      es = a1 + (tid - 32);
      if (es >= b.hi) es = -1;
    }
    if (es < 0) continue;
    float acc = 0.f;
    for (int pos = 0; pos < n; ++pos) {
      int r = b.rot + pos;
      if (r >= n) r -= n;
      float f[1];
      LG::widen(LG::load(static_cast<const char*>(p.ptr[b.t * n + r]), es), f);
      acc = pos == 0 ? f[0] : fadd(acc, f[0]);
    }
    float v[1] = {fmul(acc, p.scale)};
    const typename LG::raw_t rr = LG::narrow(v);
    for (int q = 0; q < n; ++q) LG::store(static_cast<char*>(p.ptr[b.t * n + q]), es, rr);
  }
}

template <bool BF16, bool TREE, int VPT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    fused_tma_kernel(const __grid_constant__ FusedParams p, const __grid_constant__ TmaCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  grid_dependency_wait();  // the previous kernel's writes are visible from here on
  grid_dependents_launch();
  FlatSource src(p, c.tile_bytes / (BF16 ? 2 : 4), BF16 ? 8 : 4);
  tma_pipeline<BF16, TREE, VPT>(src, p.n, p.scale, c, smem);
  flat_heads_tails<BF16, TREE>(p);
}

template <bool BF16, int VPT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    bucket_tma_kernel(const __grid_constant__ BucketFusedParams p, const __grid_constant__ TmaCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  grid_dependency_wait();
  grid_dependents_launch();
  BucketSource src(p, c.tile_bytes / (BF16 ? 2 : 4), BF16 ? 8 : 4);
  tma_pipeline<BF16, false, VPT>(src, p.n, p.scale, c, smem);
  bucket_heads_tails<BF16>(p);
}

// ---------------------------------------------------------------------------
// All-gather with bulk copies. Every tile of the result is one rank's data
// (the owner's chunk) copied to all N ranks, so one bulk load feeds N bulk
// stores: the store traffic, N times the load traffic, goes through the bulk
// copy engine rather than through the threads' 16-byte stores. One lane runs
// the pipeline: S stages of T bytes, each loaded once, stored to the N ranks
// (the owner's own buffer is skipped when the call is in place) and refilled
// with the CTA's next tile once the stores have read it. Ragged chunk heads and
// tails (fewer than 16 bytes each) are copied element by element by the other
// lanes. Every wait is bounded as in the all-reduce pipeline.
// ---------------------------------------------------------------------------
// Shape: 3 stages of 32 KiB, 2 CTAs per SM. Measured on GB300 (16 ranks x 192
// MiB fp32, one call per timing): 0.89 of HBM against 0.86 for the register
// pipeline's all-gather; 4 x 16 KiB gave 0.87, 4 x 8 KiB with 4 CTAs 0.86,
// 2 x 32 KiB 0.90 at 16 ranks but 0.87 at 64. Refilling a stage one store
// group later (two tiles' stores in flight) measured, calls back to back,
// 0.941 -> 0.944 at 16 ranks and 0.86 -> 0.87 at 8; starting each tile's
// stores at a rank that moves with the tile (AR_AGB_ROTATE) measured the
// same as rank order, so it is off.
#ifndef AR_AGB_STAGES
#define AR_AGB_STAGES 3
#endif
#ifndef AR_AGB_TILE
#define AR_AGB_TILE 32768
#endif
#ifndef AR_AGB_CTAS
#define AR_AGB_CTAS 2
#endif
#ifndef AR_AGB_ROTATE
#define AR_AGB_ROTATE 0
#endif
constexpr int kAgbThreads = 32;
static_assert(AR_AGB_STAGES >= 1 && AR_AGB_STAGES <= kMaxStages, "stage count");
static_assert(AR_AGB_TILE % 16 == 0 && AR_AGB_TILE * AR_AGB_STAGES <= kTmaSmemLimit, "tile size");

__device__ __forceinline__ void ag_chunk(const FusedParams& p, int seg, int64_t& lo, int64_t& hi) {
  lo = seg * p.count / p.n;
  hi = (seg + 1) * p.count / p.n;
  if (lo < p.e_lo) lo = p.e_lo;
  if (hi > p.e_hi) hi = p.e_hi;
}

template <bool BF16>
__global__ void __launch_bounds__(kAgbThreads)
    allgather_bulk_kernel(const __grid_constant__ FusedParams p, const __grid_constant__ TmaCfg c) {
  using LG = Lane<BF16, false>;
  constexpr int W = BF16 ? 8 : 4;  // elements per 16 bytes
  constexpr int64_t ES = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ int abort_flag;
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;
  const int lane = threadIdx.x;

  // ragged heads and tails of the chunks this CTA owns, element by element
  for (int seg = blockIdx.x; seg < p.n_seg; seg += gridDim.x) {
    int64_t lo, hi;
    ag_chunk(p, seg, lo, hi);
    if (hi <= lo) continue;
    const int64_t a0 = round_up(lo, W);
    int64_t a1 = round_down(hi, W);
    if (a1 < a0) a1 = a0;
    const int64_t head_end = a0 < hi ? a0 : hi;
    int64_t es = -1;
    if (lane < W - 1) {
      es = lo + lane;
      if (es >= head_end) es = -1;
    } else if (lane >= 16 && lane < 16 + W - 1) {
      es = a1 + (lane - 16);
      if (es >= hi) es = -1;
    }
    if (es < 0) continue;
    const char* src = static_cast<const char*>(p.in[seg]);
    const typename LG::raw_t v = LG::load(src, es);
    for (int r = 0; r < n; ++r)
      if (p.out[r] != p.in[seg]) LG::store(static_cast<char*>(p.out[r]), es, v);
  }
  if (lane != 0) return;

  const int S = c.stages;
  const int T = c.tile_bytes;
  const int64_t te = T / ES;
  for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
  abort_flag = 0;
  mbar_init_fence();
  volatile int* abort = &abort_flag;

  // this CTA's tiles: t = blockIdx.x, + gridDim.x, ...; empty ones skipped
  const int64_t total = int64_t(p.n_seg) * p.tiles_per_seg;
  int64_t t = blockIdx.x;
  int64_t tile_lo[kMaxStages];
  int tile_elems[kMaxStages], tile_seg[kMaxStages];
  auto next = [&](int s) -> bool {
    while (t < total) {
      const int seg = int(t / p.tiles_per_seg);
      const int64_t tt = t - int64_t(seg) * p.tiles_per_seg;
      t += gridDim.x;
      int64_t lo, hi;
      ag_chunk(p, seg, lo, hi);
      const int64_t a0 = round_up(lo, W);
      const int64_t a1 = round_down(hi, W);
      const int64_t s0 = a0 + tt * te;
      const int64_t s1 = s0 + te < a1 ? s0 + te : a1;
      if (s1 > s0) {
        tile_lo[s] = s0;
        tile_elems[s] = int(s1 - s0);
        tile_seg[s] = seg;
        return true;
      }
    }
    tile_elems[s] = -1;
    return false;
  };
  auto load = [&](int s) {
    const uint32_t bytes = uint32_t(tile_elems[s] * ES);
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_load(smem + size_t(s) * T, static_cast<const char*>(p.in[tile_seg[s]]) + tile_lo[s] * ES, bytes, &full[s]);
  };

  // `live`: stages holding a tile whose stores are not issued yet; bit s of
  // `inflight`: stage s has a load issued and not yet seen complete. A
  // stage's stores are issued as soon as its load lands; the stage is
  // refilled one tile later, once those stores have read it (the store group
  // before the newest has completed its reads), so the stores of two tiles
  // are in flight at once.
  int live = 0;
  uint32_t inflight = 0;
  for (int s = 0; s < S; ++s) {
    if (next(s)) {
      load(s);
      ++live;
      inflight |= 1u << s;
    }
  }
  uint32_t parity = 0;  // bit s: the parity of stage s's next completion
  int pending = -1;     // the stage whose stores were issued last, not refilled yet
  auto refill = [&](int s) {
    if (next(s)) {
      load(s);
      ++live;
      inflight |= 1u << s;
    } else {
      tile_elems[s] = -1;
    }
  };
  for (int it = 0; live > 0 || pending >= 0;) {
    if (live == 0) {  // nothing else to store: the last stage's refill cannot wait for a later tile
      bulk_wait_read<0>();
      refill(pending);
      pending = -1;
      continue;
    }
    const int s = it++ % S;
    if (tile_elems[s] < 0 || s == pending) continue;
    if (!mbar_wait(&full[s], (parity >> s) & 1u, kWaitPolls, abort)) break;
    parity ^= 1u << s;
    inflight &= ~(1u << s);
    const uint32_t bytes = uint32_t(tile_elems[s] * ES);
    const void* stage = smem + size_t(s) * T;
    const void* owner = p.in[tile_seg[s]];
    // the N ranks in turn from a rank that moves with the tile, so that the
    // CTAs' stores spread over the destination buffers
    const int r0 = AR_AGB_ROTATE ? int(tile_lo[s] / te % n) : 0;
    for (int i = 0, r = r0; i < n; ++i, r = r + 1 < n ? r + 1 : 0)
      if (p.out[r] != owner) bulk_store(static_cast<char*>(p.out[r]) + tile_lo[s] * ES, stage, bytes);
    bulk_commit();
    --live;
    if (pending >= 0) {
      bulk_wait_read<1>();  // the stores before this tile's have read their stage
      refill(pending);
    }
    pending = s;
  }
  if (*abort) {
    // Let every load still in flight land before shared memory goes away. A
    // bulk load reads device memory the host validated, so it completes in
    // microseconds; each poll of the wait may suspend the thread in hardware,
    // so 2^16 polls per stage allow far longer than any such load takes.
    volatile int never = 0;
    for (int s = 0; s < S; ++s)
      if ((inflight >> s) & 1u) mbar_wait(&full[s], (parity >> s) & 1u, 1u << 16, &never);
  }
  bulk_wait_all();  // every store has completed before the CTA exits
}

// A kernel whose wait nothing will ever satisfy: its bounded wait must give up,
// set the status word and return.
__global__ void wait_timeout_kernel(uint32_t polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_init_fence();
  abort_flag = 0;
  mbar_wait(&bar, 0, polls, &abort_flag);
}

// Raise a kernel's dynamic shared-memory limit to `smem` bytes if it is lower.
cudaError_t allow_smem(const void* kernel, size_t smem) {
  struct Entry {
    int device;
    const void* kernel;
    size_t bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> set;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (Entry& e : set)
    if (e.device == dev && e.kernel == kernel) {
      if (e.bytes >= smem) return cudaSuccess;
      const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (err == cudaSuccess) e.bytes = smem;
      return err;
    }
  const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err == cudaSuccess) set.push_back({dev, kernel, smem});
  return err;
}

template <class P>
cudaError_t launch_tma(void (*kernel)(P, TmaCfg), const P& p, const TmaCfg& c, int64_t tiles, int n_seg, size_t smem,
                       int sm_budget, cudaStream_t stream) {
  const cudaError_t e = allow_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int use = (sm_budget > 0 && sm_budget < sms) ? sm_budget : sms;
  // every segment's heads and tails need a CTA too
  const int64_t want = tiles > n_seg ? tiles : n_seg;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(want < use ? want : use));
  cfg.blockDim = dim3(kTmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, c);
}

}  // namespace

// Stage count and tile size for N ranks: the largest tile (4, 8 or 16 KiB)
// that still leaves at least 3 stages (2 for wide N) of N slices, plus two
// output tiles, within the shared memory of one CTA. Returns false when even
// 2 stages of 4 KiB slices do not fit (N too large): the register-pipelined
// kernel runs instead.
bool tma_shape(int n, int& stages, int& tile_bytes) {
  if (n < 2 || n > kTmaMaxRanks) return false;
  const int room = kTmaSmemLimit - 4096;  // the kernel's static shared memory takes under 2 KiB
  for (int min_stages : {3, 2})
    for (int k : {4, 2, 1}) {
      const int T = 4096 * k;
      const int s = (room - 2 * T) / (n * T);
      if (s >= min_stages) {
        stages = s < kMaxStages ? s : kMaxStages;
        tile_bytes = T;
        return true;
      }
    }
  return false;
}

cudaError_t launch_fused_tma(const FusedParams& p, ar_dtype dtype, int stages, int tile_bytes, int sm_budget,
                             cudaStream_t stream) {
  const TmaCfg c{stages, tile_bytes};
  const int64_t tiles = int64_t(p.n_seg) * p.tiles_per_seg;
  const size_t smem = size_t(stages) * p.n * tile_bytes + 2 * size_t(tile_bytes);
  const int vpt = tile_bytes / 4096;
  const bool tree = p.order == AR_ORDER_TREE;
#define AR_TMA_LAUNCH(BF, TR, V) launch_tma(fused_tma_kernel<BF, TR, V>, p, c, tiles, p.n_seg, smem, sm_budget, stream)
  if (dtype == AR_BF16) {
    if (tree) return vpt == 4 ? AR_TMA_LAUNCH(true, true, 4) : vpt == 2 ? AR_TMA_LAUNCH(true, true, 2) : AR_TMA_LAUNCH(true, true, 1);
    return vpt == 4 ? AR_TMA_LAUNCH(true, false, 4) : vpt == 2 ? AR_TMA_LAUNCH(true, false, 2) : AR_TMA_LAUNCH(true, false, 1);
  }
  if (tree) return vpt == 4 ? AR_TMA_LAUNCH(false, true, 4) : vpt == 2 ? AR_TMA_LAUNCH(false, true, 2) : AR_TMA_LAUNCH(false, true, 1);
  return vpt == 4 ? AR_TMA_LAUNCH(false, false, 4) : vpt == 2 ? AR_TMA_LAUNCH(false, false, 2) : AR_TMA_LAUNCH(false, false, 1);
#undef AR_TMA_LAUNCH
}

cudaError_t launch_bucket_tma(const BucketFusedParams& p, ar_dtype dtype, int stages, int tile_bytes, int sm_budget,
                              cudaStream_t stream) {
  const TmaCfg c{stages, tile_bytes};
  const int64_t tiles = p.tile_start[p.n_seg];
  const size_t smem = size_t(stages) * p.n * tile_bytes + 2 * size_t(tile_bytes);
  const int vpt = tile_bytes / 4096;
#define AR_TMA_LAUNCH(BF, V) launch_tma(bucket_tma_kernel<BF, V>, p, c, tiles, p.n_seg, smem, sm_budget, stream)
  if (dtype == AR_BF16) return vpt == 4 ? AR_TMA_LAUNCH(true, 4) : vpt == 2 ? AR_TMA_LAUNCH(true, 2) : AR_TMA_LAUNCH(true, 1);
  return vpt == 4 ? AR_TMA_LAUNCH(false, 4) : vpt == 2 ? AR_TMA_LAUNCH(false, 2) : AR_TMA_LAUNCH(false, 1);
#undef AR_TMA_LAUNCH
}

int64_t allgather_bulk_tile_elems(ar_dtype dtype) { return AR_AGB_TILE / (dtype == AR_BF16 ? 2 : 4); }

cudaError_t launch_allgather_bulk(const FusedParams& p, ar_dtype dtype, int sm_budget, cudaStream_t stream) {
  const TmaCfg c{AR_AGB_STAGES, AR_AGB_TILE};
  const size_t smem = size_t(c.stages) * c.tile_bytes;
  void (*kernel)(FusedParams, TmaCfg) = dtype == AR_BF16 ? allgather_bulk_kernel<true> : allgather_bulk_kernel<false>;
  const cudaError_t e = allow_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int use = (sm_budget > 0 && sm_budget < sms) ? sm_budget : sms;
  const int64_t tiles = int64_t(p.n_seg) * p.tiles_per_seg;
  const int64_t want = tiles > p.n_seg ? tiles : p.n_seg;  // every chunk's head and tail needs a CTA
  const int64_t cap = int64_t(AR_AGB_CTAS) * use;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(want < cap ? want : cap));
  cfg.blockDim = dim3(kAgbThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, c);
}

cudaError_t launch_wait_timeout(uint32_t polls, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(polls);
  return cudaGetLastError();
}

namespace {

constexpr int kMaxStatusDevices = 64;
// Per device ordinal: the host-visible status word, once published.
std::atomic<unsigned int*> g_host_word[kMaxStatusDevices];
std::mutex g_host_word_mu;

}  // namespace

volatile unsigned int* host_status_word_if_ready(int device) {
  if (device < 0 || device >= kMaxStatusDevices) return nullptr;
  return g_host_word[device].load(std::memory_order_acquire);
}

cudaError_t host_status_word(int device, volatile unsigned int** word) {
  *word = host_status_word_if_ready(device);
  if (*word != nullptr) return cudaSuccess;
  if (device < 0 || device >= kMaxStatusDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_host_word_mu);
  unsigned int* h = g_host_word[device].load(std::memory_order_acquire);
  if (h == nullptr) {
    // Relaxed capture mode for this thread: the one-time set-up may run while
    // another thread captures a stream. The pointer goes to the device on a
    // private non-blocking stream, which joins no capture.
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t err = cudaThreadExchangeStreamCaptureMode(&mode);
    if (err != cudaSuccess) return err;
    void* dptr = nullptr;
    cudaStream_t s = nullptr;
    err = cudaHostAlloc(reinterpret_cast<void**>(&h), sizeof(unsigned int),
                        cudaHostAllocMapped | cudaHostAllocPortable);
    if (err == cudaSuccess) {
      *reinterpret_cast<volatile unsigned int*>(h) = 0;
      err = cudaHostGetDevicePointer(&dptr, h, 0);
    }
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (err == cudaSuccess)
      err = cudaMemcpyToSymbolAsync(g_ar_status_host, &dptr, sizeof(dptr), 0, cudaMemcpyHostToDevice, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (s != nullptr) cudaStreamDestroy(s);
    cudaThreadExchangeStreamCaptureMode(&mode);  // restore the caller's mode
    if (err != cudaSuccess) {
      if (h != nullptr) cudaFreeHost(h);
      return err;
    }
    g_host_word[device].store(h, std::memory_order_release);
  }
  *word = h;
  return cudaSuccess;
}

cudaError_t read_device_status(unsigned int* value, bool clear) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(value, g_ar_status_word, sizeof(unsigned int));
  if (err != cudaSuccess || !clear) return err;
  const unsigned int zero = 0;
  err = cudaMemcpyToSymbol(g_ar_status_word, &zero, sizeof(unsigned int));
  if (err != cudaSuccess) return err;
  int dev = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (volatile unsigned int* h = host_status_word_if_ready(dev)) *h = 0;
  return cudaSuccess;
}

}  // namespace ar
