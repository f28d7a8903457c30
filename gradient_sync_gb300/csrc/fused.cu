// Fused single-pass N-way reduce + broadcast.
//
// out[r][e] = scale * (sum over ranks of g[e]) for every rank r, in a declared
// per-element order, reading every element of every rank once and writing
// the result once to every rank: N*S bytes read and N*S written, the traffic
// of a rank that sends its buffer once and receives the sum once (primer
// ch. 4, "Collective communication: algorithms, cost and the library that
// runs them", §4.4, "In-network reduction").
//
// The orders reproduce the step-by-step schedules bit for bit (the summation
// order is part of the result; Scaling ML Systems, "Collective
// communication"): ring (primer §4.2), rank order, Rabenseifner's tree
// (primer §4.3) and the hierarchical order (primer §4.4).
//
// Layout of the work: the buffer is cut into segments in which the order is
// the same for every element (ring: the N chunks; hierarchical: the G*M
// sub-chunks; rank/tree: one segment). A segment's aligned body is cut into
// tiles of kThreads 16-byte vectors; its ragged head and tail (fewer than one
// vector each) are done element by element by the CTA that takes the
// segment's first tile. A persistent grid (a multiple of the SM count) walks
// the tiles. For each segment the CTA writes the fold sequence (input
// pointer and combine flags per position) to shared memory once; each thread
// then issues NB 16-byte loads per batch before adding, keeps the sum in
// registers and stores it to all N ranks.
#include <type_traits>

#include "common.cuh"

// Tuning knob (compile time): the minimum resident CTAs per SM that the
// register allocation must allow. Two CTAs of 256 threads per SM, each thread
// keeping about eight 16-byte loads in flight, measured best on GB300 (one
// CTA left too few warps to cover HBM latency).
#ifndef AR_FUSED_MINB
#define AR_FUSED_MINB 2
#endif

namespace ar {

namespace {

__device__ __forceinline__ void seq_position(const FusedParams& p, int seg, int pos, int& rank,
                                             uint8_t& flag) {
  const int n = p.n;
  if (p.collective == AR_ALLGATHER) {  // one position: chunk seg comes from its owner
    rank = seg;
    flag = kStart | kEnd | kFirst;
    return;
  }
  if (p.collective == AR_REDUCE_SCATTER && p.order == AR_ORDER_RING) {  // fold from rank seg+1
    int r = seg + 1 + pos;
    while (r >= n) r -= n;
    rank = r;
    flag = (pos == 0 ? kStart : 0) | (pos == n - 1 ? (kEnd | kFirst) : 0);
    return;
  }
  if (p.order == AR_ORDER_HIER) {
    const int g = p.g, m = p.m;
    const int k = seg / m, j = seg - (seg / m) * m;
    const int mi = pos / g, i = pos - mi * g;
    int grp = j + mi;
    if (grp >= m) grp -= m;
    int l = k + 1 + i;
    l %= g;
    rank = grp * g + l;
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

__device__ __forceinline__ void seg_range(const FusedParams& p, int seg, int64_t& lo, int64_t& hi) {
  const int64_t L = p.count;
  if (p.order == AR_ORDER_RING || p.collective != AR_ALLREDUCE) {  // the N chunks
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
}

// The rank a segment's fold starts from when its order is a rotation of the
// rank list (every order but the hierarchical one).
__device__ __forceinline__ int seg_rotation(const FusedParams& p, int seg) {
  if (p.collective == AR_ALLGATHER) return seg;  // one position: the chunk's owner
  if (p.order != AR_ORDER_RING) return 0;        // rank order, Rabenseifner's tree
  if (p.collective == AR_REDUCE_SCATTER) return seg + 1 < p.n ? seg + 1 : 0;
  return seg;  // ring all-reduce: chunk c from rank c
}

// How a CTA gets the fold sequence of a segment:
//  kSeqWritten: written to shared memory when the CTA moves to the segment,
//    between two barriers (the hierarchical order, whose sequence is not a
//    rotation of the rank list);
//  kSeqRotated: the ranks' input pointers are written once, twice over in
//    rank order, so a segment's sequence starts at its rotation (seg_rotation)
//    with no rewrite; the per-position flags are written once too;
//  kSeqRotatedPos: the same, with the flags taken from the position
//    (fold_single).
// Moving to another segment then costs one barrier, which keeps the warps of
// a CTA on the same tile (the stores of a tile land together); without it,
// and with the rewrite's two barriers, the kernel measured slower. At 64
// ranks x 16 MiB a ring chunk is 64 tiles, so nearly every tile of a CTA
// starts a new segment.
enum SeqMode { kSeqWritten = 0, kSeqRotated = 1, kSeqRotatedPos = 2 };

template <bool BF16, bool TREE, int MODE, int NB, int VPT>
__global__ void __launch_bounds__(kThreads, AR_FUSED_MINB) fused_flat_kernel(const __grid_constant__ FusedParams p) {
  using LV = Lane<BF16, true>;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W * VPT;
  constexpr bool kRot = MODE != kSeqWritten;
  // kSeqWritten: the segment's sequence; otherwise the ranks in order, twice
  __shared__ const char* s_seq[2 * AR_MAX_RANKS];
  __shared__ uint8_t s_flag[AR_MAX_RANKS];
  __shared__ char* s_out[AR_MAX_RANKS];
  grid_dependency_wait();  // the previous kernel on the stream has finished and its writes are visible
  grid_dependents_launch();
  const int n = p.n;
  const int nf = p.collective == AR_ALLGATHER ? 1 : n;  // ranks folded per element
  const bool owner_only = p.collective == AR_REDUCE_SCATTER;
  if (threadIdx.x < n) {
    s_out[threadIdx.x] = static_cast<char*>(p.out[threadIdx.x]);
    if (kRot) {
      s_seq[threadIdx.x] = s_seq[threadIdx.x + n] = static_cast<const char*>(p.in[threadIdx.x]);
      s_flag[threadIdx.x] = (threadIdx.x == 0 ? kStart : 0) | (threadIdx.x == nf - 1 ? (kEnd | kFirst) : 0);
    }
  }
  int cur = -1, rot = 0;
  int64_t lo = 0, hi = 0;
  const int64_t total = int64_t(p.n_seg) * p.tiles_per_seg;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int seg = int(t / p.tiles_per_seg);
    const int64_t tt = t - int64_t(seg) * p.tiles_per_seg;
    if (seg != cur) {  // uniform across the CTA
      __syncthreads();
      if (!kRot) {
        if (threadIdx.x < n) {
          int rank;
          uint8_t flag;
          seq_position(p, seg, threadIdx.x, rank, flag);
          s_seq[threadIdx.x] = static_cast<const char*>(p.in[rank]);
          s_flag[threadIdx.x] = flag;
        }
        __syncthreads();
      }
      cur = seg;
      rot = kRot ? seg_rotation(p, seg) : 0;
      seg_range(p, seg, lo, hi);
    }
    const char* const* seq = s_seq + rot;
    const int64_t clo = lo > p.e_lo ? lo : p.e_lo;
    const int64_t chi = hi < p.e_hi ? hi : p.e_hi;
    if (clo >= chi) continue;
    const int64_t a0 = round_up(clo, W);
    int64_t a1 = round_down(chi, W);
    if (a1 < a0) a1 = a0;
    int64_t e[VPT];
    bool ok[VPT];
    bool any = false;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = a0 + tt * kTile + (int64_t(q) * kThreads + threadIdx.x) * W;
      ok[q] = e[q] < a1;
      any |= ok[q];
    }
    if (any) {
      float acc[VPT][W];
      if (TREE) {
        fold_tree<LV, NB>(acc[0], seq, nf, e[0]);
      } else if (MODE == kSeqRotatedPos) {
        fold_single<LV, NB, VPT>(acc, seq, nf, e, ok);
      } else {
        fold_sequence<LV, NB, VPT>(acc, seq, s_flag, nf, e, ok);
      }
      typename LV::raw_t r[VPT];
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
#pragma unroll
        for (int w = 0; w < W; ++w) acc[q][w] = fmul(acc[q][w], p.scale);
        r[q] = LV::narrow(acc[q]);
      }
      if (owner_only) {  // reduce-scatter: only the chunk's owner receives it
#pragma unroll
        for (int q = 0; q < VPT; ++q)
          if (ok[q]) LV::store(s_out[seg], e[q], r[q]);
      } else {
#pragma unroll 2
        for (int d = 0; d < n; ++d)
#pragma unroll
          for (int q = 0; q < VPT; ++q)
            if (ok[q]) LV::store(s_out[d], e[q], r[q]);
      }
    }
    if (tt == 0) {  // ragged head [clo, min(a0, chi)) and tail [a1, chi)
      int64_t es = -1;
      const int64_t head_end = a0 < chi ? a0 : chi;
      if (threadIdx.x < W - 1) {
        es = clo + threadIdx.x;
        if (es >= head_end) es = -1;
      } else if (threadIdx.x >= 32 && threadIdx.x < 32 + W - 1) {
        es = a1 + (threadIdx.x - 32);
        if (es >= chi) es = -1;
      }
      if (es >= 0) {
        float acc[1][1];
        const int64_t es1[1] = {es};
        const bool ok1[1] = {true};
        if (TREE)
          fold_tree<LS, 8>(acc[0], seq, nf, es);
        else
          fold_sequence<LS, 8, 1>(acc, seq, s_flag, nf, es1, ok1);
        acc[0][0] = fmul(acc[0][0], p.scale);
        const typename LS::raw_t r = LS::narrow(acc[0]);
        if (owner_only)
          LS::store(s_out[seg], es, r);
        else
          for (int q = 0; q < n; ++q) LS::store(s_out[q], es, r);
      }
    }
  }
}

// Budgeted launches (a few SMs, one CTA on each): a CTA alone on an SM has
// too few loads in flight to cover HBM latency, and in the kernels above none
// are in flight while a tile's N stores issue. The deep kernels below issue
// the next tile's first batch of loads (NB ranks x VPT vectors) before this
// tile's stores, into the registers the batch has just been added from, so
// those loads' latency overlaps the stores. With NB x VPT covering all the
// ranks of a tile, a CTA always has a whole tile's loads in flight. The
// summation order per element is fold_single's: the same bits as the kernels
// above.

// Adds batch `base` (ranks base..base+NB-1 of the fold, already loaded into
// v) into the running sums.
template <class L, int NB, int VPT>
__device__ __forceinline__ void add_batch(float (&part)[VPT][L::W], const typename L::raw_t (&v)[NB][VPT],
                                          int base, int n, const bool (&ok)[VPT]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (base + b < n) {
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        if (!ok[q]) continue;
        float f[L::W];
        L::widen(v[b][q], f);
        if (base + b == 0) {
#pragma unroll
          for (int w = 0; w < L::W; ++w) part[q][w] = f[w];
        } else {
#pragma unroll
          for (int w = 0; w < L::W; ++w) part[q][w] = fadd(part[q][w], f[w]);
        }
      }
    }
  }
}

// The tree order's add of batch `base`: ranks arrive in index order and are
// combined with fold_tree's binary counter (slot l holds a finished subtree
// of 2^l ranks; before rank r arrives the occupied slots are the set bits of
// r), so a batch at a time gives fold_tree's bits.
template <class L, int NB, int kLevels>
__device__ __forceinline__ void add_batch_tree(float (&slot)[kLevels][L::W], const typename L::raw_t (&v)[NB][1],
                                               int base, int n, bool ok) {
  if (!ok) return;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (base + b < n) {
      float carry[L::W];
      L::widen(v[b][0], carry);
      int bits = base + b;
      bool placed = false;
#pragma unroll
      for (int l = 0; l < kLevels; ++l) {
        if (!placed) {
          if (bits & 1) {
#pragma unroll
            for (int w = 0; w < L::W; ++w) carry[w] = fadd(slot[l][w], carry[w]);
            bits >>= 1;
          } else {
#pragma unroll
            for (int w = 0; w < L::W; ++w) slot[l][w] = carry[w];
            placed = true;
          }
        }
      }
    }
  }
}

// The same over VPT vectors per thread (a slot set per vector).
template <class L, int NB, int VPT, int kLevels>
__device__ __forceinline__ void add_batch_tree_v(float (&slot)[VPT][kLevels][L::W], const typename L::raw_t (&v)[NB][VPT],
                                               int base, int n, const bool (&ok)[VPT]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (base + b < n) {
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        if (!ok[q]) continue;
        float carry[L::W];
        L::widen(v[b][q], carry);
        int bits = base + b;
        bool placed = false;
#pragma unroll
        for (int l = 0; l < kLevels; ++l) {
          if (!placed) {
            if (bits & 1) {
#pragma unroll
              for (int w = 0; w < L::W; ++w) carry[w] = fadd(slot[q][l][w], carry[w]);
              bits >>= 1;
            } else {
#pragma unroll
              for (int w = 0; w < L::W; ++w) slot[q][l][w] = carry[w];
              placed = true;
            }
          }
        }
      }
    }
  }
}

template <class L, int NB, int VPT>
__device__ __forceinline__ void load_batch(typename L::raw_t (&v)[NB][VPT], const char* const* seq, int base, int n,
                                           const int64_t (&e)[VPT], const bool (&ok)[VPT]) {
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int q = 0; q < VPT; ++q)
      if (base + b < n && ok[q]) v[b][q] = L::load(seq[base + b], e[q]);
}

// The element-by-element head [clo, min(a0, chi)) and tail [a1, chi) of a
// segment, done by the CTA that takes its first tile. owner >= 0: only that
// rank receives the result (the reduce-scatter). TREE: the elements fold in
// the tree order (fold_tree), else in sequence (fold_single).
template <class LS, int W, bool TREE = false>
__device__ __forceinline__ void ragged_ends(const char* const* seq, char* const* out, int n, float scale,
                                            int64_t clo, int64_t chi, int64_t a0, int64_t a1, int owner = -1) {
  int64_t es = -1;
  const int64_t head_end = a0 < chi ? a0 : chi;
  if (threadIdx.x < W - 1) {
    es = clo + threadIdx.x;
    if (es >= head_end) es = -1;
  } else if (threadIdx.x >= 32 && threadIdx.x < 32 + W - 1) {
    es = a1 + (threadIdx.x - 32);
    if (es >= chi) es = -1;
  }
  if (es >= 0) {
    float acc[1][1];
    const int64_t es1[1] = {es};
    const bool ok1[1] = {true};
    if constexpr (TREE)
      fold_tree<LS, 8>(acc[0], seq, n, es);
    else
      fold_single<LS, 8, 1>(acc, seq, n, es1, ok1);
    acc[0][0] = fmul(acc[0][0], scale);
    const typename LS::raw_t r = LS::narrow(acc[0]);
    if (owner >= 0)
      LS::store(out[owner], es, r);
    else
      for (int q = 0; q < n; ++q) LS::store(out[q], es, r);
  }
}

// Ring and rank order of the all-reduce and of the reduce-scatter (rotations
// of the rank list; the reduce-scatter stores only to the chunk's owner).
// kRegPtr: the first batch's input pointers are kept in registers, reloaded
// when the CTA moves to another segment, instead of read from the
// shared-memory table for every tile; the host sets it for fp32 when one
// batch holds every rank (at 32 SMs, 16 x 192 MiB: 0.735 of HBM against
// 0.714, 12 ranks 0.612 against 0.589, 8 ranks 0.679 against 0.647, 2 ranks
// 0.556 against 0.551), except 3-4 ranks (4 x 4 vectors: 0.664 against
// 0.682); bf16, whose sums take more registers, and 64 ranks measured about
// 1 % slower with it.
// TREE: Rabenseifner's order (rank order, combined as fold_tree does; n a
// power of two below 2^kLevels).
template <bool BF16, int NB, int VPT, bool kRegPtr, bool TREE = false, int kLevels = kTreeLevels>
__global__ void __launch_bounds__(kThreads, AR_FUSED_MINB) fused_deep_kernel(const __grid_constant__ FusedParams p) {
  using LV = Lane<BF16, true>;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W * VPT;
  __shared__ const char* s_seq[2 * AR_MAX_RANKS];  // the ranks' inputs in order, twice
  __shared__ char* s_out[AR_MAX_RANKS];
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;
  if (threadIdx.x < n) {
    s_out[threadIdx.x] = static_cast<char*>(p.out[threadIdx.x]);
    s_seq[threadIdx.x] = s_seq[threadIdx.x + n] = static_cast<const char*>(p.in[threadIdx.x]);
  }
  const int64_t total = int64_t(p.n_seg) * p.tiles_per_seg;
  int64_t t = blockIdx.x;
  if (t >= total) return;  // uniform across the CTA
  __syncthreads();

  // Where tile t lies: its segment, its index in the segment, the segment's
  // element range clipped to [e_lo, e_hi) and its aligned body [a0, a1).
  struct Where {
    int seg;
    int64_t tt, clo, chi, a0, a1;
  };
  auto locate = [&](int64_t tile) {
    Where w;
    w.seg = int(tile / p.tiles_per_seg);
    w.tt = tile - int64_t(w.seg) * p.tiles_per_seg;
    int64_t lo, hi;
    seg_range(p, w.seg, lo, hi);
    w.clo = lo > p.e_lo ? lo : p.e_lo;
    w.chi = hi < p.e_hi ? hi : p.e_hi;
    w.a0 = round_up(w.clo, W);
    w.a1 = round_down(w.chi, W);
    if (w.a1 < w.a0) w.a1 = w.a0;
    return w;
  };
  auto vectors = [&](const Where& w, int64_t (&e)[VPT], bool (&ok)[VPT]) {
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = w.a0 + w.tt * kTile + (int64_t(q) * kThreads + threadIdx.x) * W;
      ok[q] = w.clo < w.chi && e[q] < w.a1;
    }
  };

  typename LV::raw_t v[NB][VPT];
  Where c = locate(t);
  int64_t e[VPT];
  bool ok[VPT];
  vectors(c, e, ok);
  const char* p0[kRegPtr ? NB : 1];
  auto first_ptrs = [&](int seg) {
    const char* const* sq = s_seq + seg_rotation(p, seg);
#pragma unroll
    for (int b = 0; b < (kRegPtr ? NB : 1); ++b) p0[b] = b < n ? sq[b] : nullptr;
  };
  if constexpr (kRegPtr) {
    first_ptrs(c.seg);
    load_batch<LV, NB, VPT>(v, p0, 0, n, e, ok);
  } else {
    load_batch<LV, NB, VPT>(v, s_seq + seg_rotation(p, c.seg), 0, n, e, ok);
  }
  for (;;) {
    const char* const* seq = s_seq + seg_rotation(p, c.seg);
    float part[VPT][W];
    if constexpr (TREE) {
      if constexpr (VPT == 1) {
        float slot[kLevels][W];
        add_batch_tree<LV, NB, kLevels>(slot, v, 0, n, ok[0]);
#pragma unroll 1
        for (int base = NB; base < n; base += NB) {
          load_batch<LV, NB, VPT>(v, seq, base, n, e, ok);
          add_batch_tree<LV, NB, kLevels>(slot, v, base, n, ok[0]);
        }
#pragma unroll
        for (int l = 0; l < kLevels; ++l)  // n = 2^K: the whole tree sits in slot K
          if ((1 << l) == n) {
#pragma unroll
            for (int w = 0; w < W; ++w) part[0][w] = slot[l][w];
          }
      } else {
        float slot[VPT][kLevels][W];
        add_batch_tree_v<LV, NB, VPT, kLevels>(slot, v, 0, n, ok);
#pragma unroll 1
        for (int base = NB; base < n; base += NB) {
          load_batch<LV, NB, VPT>(v, seq, base, n, e, ok);
          add_batch_tree_v<LV, NB, VPT, kLevels>(slot, v, base, n, ok);
        }
#pragma unroll
        for (int l = 0; l < kLevels; ++l)
          if ((1 << l) == n) {
#pragma unroll
            for (int q = 0; q < VPT; ++q)
#pragma unroll
              for (int w = 0; w < W; ++w) part[q][w] = slot[q][l][w];
          }
      }
    } else {
      add_batch<LV, NB, VPT>(part, v, 0, n, ok);
#pragma unroll 1
      for (int base = NB; base < n; base += NB) {
        load_batch<LV, NB, VPT>(v, seq, base, n, e, ok);
        add_batch<LV, NB, VPT>(part, v, base, n, ok);
      }
    }
    typename LV::raw_t r[VPT];
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
#pragma unroll
      for (int w = 0; w < W; ++w) part[q][w] = fmul(part[q][w], p.scale);
      r[q] = LV::narrow(part[q]);
    }
    // the next tile's first batch, before this tile's stores
    const int64_t t2 = t + gridDim.x;
    Where c2 = c;
    int64_t e2[VPT];
    bool ok2[VPT];
    if (t2 < total) {
      c2 = locate(t2);
      if (c2.seg != c.seg) __syncthreads();  // keeps the warps of a CTA on one tile
      vectors(c2, e2, ok2);
      if constexpr (kRegPtr) {
        if (c2.seg != c.seg) first_ptrs(c2.seg);
        load_batch<LV, NB, VPT>(v, p0, 0, n, e2, ok2);
      } else {
        load_batch<LV, NB, VPT>(v, s_seq + seg_rotation(p, c2.seg), 0, n, e2, ok2);
      }
    }
    if (p.collective == AR_REDUCE_SCATTER) {  // uniform across the grid
#pragma unroll
      for (int q = 0; q < VPT; ++q)
        if (ok[q]) LV::store(s_out[c.seg], e[q], r[q]);
    } else {
#pragma unroll 2
      for (int d = 0; d < n; ++d)
#pragma unroll
        for (int q = 0; q < VPT; ++q)
          if (ok[q]) LV::store(s_out[d], e[q], r[q]);
    }
    if (c.tt == 0 && c.clo < c.chi)
      ragged_ends<LS, W, TREE>(seq, s_out, n, p.scale, c.clo, c.chi, c.a0, c.a1,
                         p.collective == AR_REDUCE_SCATTER ? c.seg : -1);
    if (t2 >= total) break;
    t = t2;
    c = c2;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = e2[q];
      ok[q] = ok2[q];
    }
  }
}

// The bucket kernel's deep variant (below): a segment's pointers are written
// to one of two shared-memory slots, so the next segment's can be published
// while this tile's stores still read the current ones.
template <bool BF16, bool V8, int NB, int VPT>
__global__ void __launch_bounds__(kThreads, AR_FUSED_MINB)
    fused_bucket_deep_kernel(const __grid_constant__ BucketFusedParams p) {
  using LV = typename std::conditional<V8, Lane32<BF16>, Lane<BF16, true>>::type;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W * VPT;
  __shared__ const char* s_seq[2][AR_MAX_RANKS];  // the fold's inputs from the chunk's rank
  __shared__ char* s_out[2][AR_MAX_RANKS];
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;
  const int total = p.tile_start[p.n_seg];
  int t = blockIdx.x;
  if (t >= total) return;  // uniform across the CTA
  auto publish = [&](int s, int slot) {
    if (threadIdx.x < n) {
      const BucketSeg& sg = p.seg[s];
      int r = sg.rot + threadIdx.x;
      if (r >= n) r -= n;
      s_seq[slot][threadIdx.x] = static_cast<const char*>(p.ptr[sg.t * n + r]);
      s_out[slot][threadIdx.x] = static_cast<char*>(p.ptr[sg.t * n + threadIdx.x]);
    }
  };
  struct Where {
    int64_t tt, lo, hi, a0, a1;
  };
  auto locate = [&](int s, int tile) {
    Where w;
    w.tt = tile - p.tile_start[s];
    w.lo = p.seg[s].lo;
    w.hi = p.seg[s].hi;
    w.a0 = round_up(w.lo, W);
    w.a1 = round_down(w.hi, W);
    if (w.a1 < w.a0) w.a1 = w.a0;
    return w;
  };
  auto vectors = [&](const Where& w, int64_t (&e)[VPT], bool (&ok)[VPT]) {
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = w.a0 + w.tt * kTile + (int64_t(q) * kThreads + threadIdx.x) * W;
      ok[q] = e[q] < w.a1;
    }
  };

  int s = 0;
  while (p.tile_start[s + 1] <= t) ++s;
  int slot = 0;
  publish(s, slot);
  __syncthreads();
  typename LV::raw_t v[NB][VPT];
  Where c = locate(s, t);
  int64_t e[VPT];
  bool ok[VPT];
  vectors(c, e, ok);
  load_batch<LV, NB, VPT>(v, s_seq[slot], 0, n, e, ok);
  for (;;) {
    float part[VPT][W];
    add_batch<LV, NB, VPT>(part, v, 0, n, ok);
#pragma unroll 1
    for (int base = NB; base < n; base += NB) {
      load_batch<LV, NB, VPT>(v, s_seq[slot], base, n, e, ok);
      add_batch<LV, NB, VPT>(part, v, base, n, ok);
    }
    typename LV::raw_t r[VPT];
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
#pragma unroll
      for (int w = 0; w < W; ++w) part[q][w] = fmul(part[q][w], p.scale);
      r[q] = LV::narrow(part[q]);
    }
    // the next tile's first batch, before this tile's stores
    const int t2 = t + gridDim.x;
    int s2 = s, slot2 = slot;
    Where c2 = c;
    int64_t e2[VPT];
    bool ok2[VPT];
    if (t2 < total) {
      while (p.tile_start[s2 + 1] <= t2) ++s2;
      if (s2 != s) {  // uniform across the CTA
        slot2 = slot ^ 1;
        __syncthreads();  // every warp is done with the tile before this one (the other slot)
        publish(s2, slot2);
        __syncthreads();
      }
      c2 = locate(s2, t2);
      vectors(c2, e2, ok2);
      load_batch<LV, NB, VPT>(v, s_seq[slot2], 0, n, e2, ok2);
    }
#pragma unroll 2
    for (int d = 0; d < n; ++d)
#pragma unroll
      for (int q = 0; q < VPT; ++q)
        if (ok[q]) LV::store(s_out[slot][d], e[q], r[q]);
    if (c.tt == 0) ragged_ends<LS, W>(s_seq[slot], s_out[slot], n, p.scale, c.lo, c.hi, c.a0, c.a1);
    if (t2 >= total) break;
    t = t2;
    s = s2;
    slot = slot2;
    c = c2;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = e2[q];
      ok[q] = ok2[q];
    }
  }
}

// Bucket variant: every rank's gradient tensors are read in place through a
// (tensor, rank) pointer table; segments are the pieces of the tensors cut at
// the ring's chunk boundaries over the packed bucket, so each segment is
// folded in ring order from its chunk's rank. With V8 (every tensor 32-byte
// aligned, checked by the host) vectors are 32 bytes and move as 256-bit
// accesses, with half as many ranks per load batch: the 16-layer model's 81
// bf16 buckets on 8 ranks measured 0.944 of HBM against 0.895 with 16-byte
// vectors. (The flat kernel keeps 16-byte vectors: there 32 bytes measured
// 2-4 % slower at 4 and 16 ranks.)
template <bool BF16, bool V8, int NB, int VPT>
__global__ void __launch_bounds__(kThreads, AR_FUSED_MINB)
    fused_bucket_kernel(const __grid_constant__ BucketFusedParams p) {
  using LV = typename std::conditional<V8, Lane32<BF16>, Lane<BF16, true>>::type;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W * VPT;
  __shared__ const char* s_seq[AR_MAX_RANKS];
  __shared__ uint8_t s_flag[AR_MAX_RANKS];
  __shared__ char* s_out[AR_MAX_RANKS];
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;
  int cur = -1;
  const int total = p.tile_start[p.n_seg];
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int s = 0;
    while (p.tile_start[s + 1] <= t) ++s;
    const int64_t tt = t - p.tile_start[s];
    const BucketSeg sg = p.seg[s];
    if (s != cur) {
      __syncthreads();
      cur = s;
      if (threadIdx.x < n) {
        int r = sg.rot + threadIdx.x;
        if (r >= n) r -= n;
        s_seq[threadIdx.x] = static_cast<const char*>(p.ptr[sg.t * n + r]);
        s_flag[threadIdx.x] = (threadIdx.x == 0 ? kStart : 0) | (threadIdx.x == n - 1 ? (kEnd | kFirst) : 0);
        s_out[threadIdx.x] = static_cast<char*>(p.ptr[sg.t * n + threadIdx.x]);
      }
      __syncthreads();
    }
    const int64_t a0 = round_up(sg.lo, W);
    int64_t a1 = round_down(sg.hi, W);
    if (a1 < a0) a1 = a0;
    int64_t e[VPT];
    bool ok[VPT];
    bool any = false;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      e[q] = a0 + tt * kTile + (int64_t(q) * kThreads + threadIdx.x) * W;
      ok[q] = e[q] < a1;
      any |= ok[q];
    }
    if (any) {
      float acc[VPT][W];
      fold_sequence<LV, NB, VPT>(acc, s_seq, s_flag, n, e, ok);
      typename LV::raw_t r[VPT];
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
#pragma unroll
        for (int w = 0; w < W; ++w) acc[q][w] = fmul(acc[q][w], p.scale);
        r[q] = LV::narrow(acc[q]);
      }
#pragma unroll 2
      for (int d = 0; d < n; ++d)
#pragma unroll
        for (int q = 0; q < VPT; ++q)
          if (ok[q]) LV::store(s_out[d], e[q], r[q]);
    }
    if (tt == 0) {
      int64_t es = -1;
      const int64_t head_end = a0 < sg.hi ? a0 : sg.hi;
      if (threadIdx.x < W - 1) {
        es = sg.lo + threadIdx.x;
        if (es >= head_end) es = -1;
      } else if (threadIdx.x >= 32 && threadIdx.x < 32 + W - 1) {
        es = a1 + (threadIdx.x - 32);
        if (es >= sg.hi) es = -1;
      }
      if (es >= 0) {
        float acc[1][1];
        const int64_t es1[1] = {es};
        const bool ok1[1] = {true};
        fold_sequence<LS, 8, 1>(acc, s_seq, s_flag, n, es1, ok1);
        acc[0][0] = fmul(acc[0][0], p.scale);
        const typename LS::raw_t r = LS::narrow(acc[0]);
        for (int q = 0; q < n; ++q) LS::store(s_out[q], es, r);
      }
    }
  }
}

// Launched with programmatic dependent launch: the kernel may be scheduled
// while the previous kernel on the stream drains, and waits for it
// (griddepcontrol.wait) before touching memory, so stream order holds.
template <class P>
cudaError_t launch_persistent(void (*kernel)(P), const P& p, int64_t tiles, int sm_budget, cudaStream_t stream) {
  if (tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(persistent_grid(reinterpret_cast<const void*>(kernel), tiles, sm_budget));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

// Vectors per thread: about eight 16-byte loads in flight per thread for the
// all-reduce whatever N is (N loads per vector). The reduce-scatter writes one
// vector per N loaded and needs twice that: 8 ranks x 2 vectors measured 1.02
// of HBM at 16 x 192 MiB fp32 on GB300, against 0.87 with one vector. The
// all-gather folds one rank per element and is bound by its N stores per load
// (0.85 with 4 vectors; 8 measured the same).
constexpr int kRsNB = 8, kRsVPT = 2, kAgVPT = 4;

// Budgeted deep kernels with 16-byte vectors: up to 16 loads per thread in
// one batch, a whole tile's for up to 16 ranks: 16 ranks x 1 vector from
// kDeepWideMin ranks up, 8 x 2 from 5 ranks, 4 x 4 for 3 and 4 ranks and
// 2 x 5 for 2 (bf16, whose sums take twice the registers, 4 x 3 and 2 x 4:
// more spills). At 32 SMs, 16 x 192 MiB fp32 measured 0.71 of HBM with
// 16 x 1 against 0.60 with 8 x 2; 8 x 128 MiB bf16 0.55 with 8 x 2 against
// 0.36 with 16 x 1; 10 and 12 ranks were faster with 16 x 1 too.
constexpr int kDeepWideMin = 9;
int deep_nb(int n) { return n >= kDeepWideMin ? 16 : n > 4 ? 8 : n > 2 ? 4 : 2; }
int deep_vpt(int n, bool bf16) {
  return n >= kDeepWideMin ? 1 : n > 4 ? 2 : n > 2 ? (bf16 ? 3 : 4) : (bf16 ? 4 : 5);
}
// The budgeted tree order keeps a slot per tree level and vector: one vector
// per thread (above 16 bf16 ranks the full-width tree kernel runs), 2 below 8
// fp32 ranks (wider shapes spill registers). At 32 SMs, fp32: 4 ranks 0.497
// of HBM against 0.293 with one vector, 2 ranks 0.295 against 0.164.
int tree_deep_vpt(int n, bool bf16) { return !bf16 && n < 8 ? 2 : 1; }

// `deep` (a budgeted launch, see budgeted()): the all-reduce in ring or rank
// order takes the deep kernel's shape; the hierarchical order over more than
// 4 ranks takes 2 vectors per thread with 8 ranks per batch.
int fused_vpt(int n, int order, int collective, bool bf16, bool deep) {
  if (collective == AR_ALLGATHER) return kAgVPT;
  if (order == AR_ORDER_TREE) return deep ? tree_deep_vpt(n, bf16) : 1;
  if (deep && order != AR_ORDER_HIER) return deep_vpt(n, bf16);  // all-reduce or reduce-scatter
  if (collective == AR_REDUCE_SCATTER && n > 4) return kRsVPT;
  if (deep && n > 4) return 2;
  return n <= 2 ? 4 : n <= 4 ? 2 : 1;
}

// The bucket kernel's 16-byte path: the flat all-reduce's vectors per thread.
int bucket_vpt(int n, bool bf16, bool deep) { return deep ? deep_vpt(n, bf16) : n <= 2 ? 4 : n <= 4 ? 2 : 1; }

int fused_vec_elems(ar_dtype dtype, bool v8) { return (dtype == AR_BF16 ? 8 : 4) * (v8 ? 2 : 1); }

int64_t fused_tile_elems(ar_dtype dtype, int n, int order, int collective, bool deep) {
  return int64_t(kThreads) * fused_vec_elems(dtype, false) * fused_vpt(n, order, collective, dtype == AR_BF16, deep);
}

int64_t bucket_tile_elems(ar_dtype dtype, int n, bool v8, bool deep) {
  return int64_t(kThreads) * fused_vec_elems(dtype, v8) * (v8 ? 1 : bucket_vpt(n, dtype == AR_BF16, deep));
}

// Every order but the hierarchical one (rotations of the rank list). The
// flags are taken from the position for more than 16 ranks and for the
// reduce-scatter, and read from shared memory otherwise (fold_single).
template <bool BF16>
cudaError_t launch_fused_rot(const FusedParams& p, int64_t tiles, int sm_budget, cudaStream_t stream) {
  if (p.order == AR_ORDER_TREE && p.collective != AR_ALLGATHER) {  // n is a power of two
    // budgeted: the deep kernel, 16 ranks per batch (bf16, whose wider sums
    // take twice the registers, 8, and only up to 16 ranks: 5 tree levels)
    if (budgeted(sm_budget)) {  // vectors per thread: tree_deep_vpt
      if constexpr (BF16) {
        if (p.n == 16) return launch_persistent(fused_deep_kernel<true, 8, 1, false, true, 5>, p, tiles, sm_budget, stream);
        if (p.n == 8) return launch_persistent(fused_deep_kernel<true, 8, 1, false, true, 4>, p, tiles, sm_budget, stream);
        if (p.n < 8) return launch_persistent(fused_deep_kernel<true, 4, 1, false, true, 3>, p, tiles, sm_budget, stream);
      } else {
        if (p.n >= 16) return launch_persistent(fused_deep_kernel<false, 16, 1, false, true>, p, tiles, sm_budget, stream);
        if (p.n == 8) return launch_persistent(fused_deep_kernel<false, 8, 1, false, true>, p, tiles, sm_budget, stream);
        return launch_persistent(fused_deep_kernel<false, 4, 2, false, true, 3>, p, tiles, sm_budget, stream);
      }
    }
    return launch_persistent(fused_flat_kernel<BF16, true, kSeqRotated, 8, 1>, p, tiles, sm_budget, stream);
  }
  if (budgeted(sm_budget) && p.collective != AR_ALLGATHER) {  // ring or rank order
    const bool reg = !BF16 && p.n <= deep_nb(p.n);  // one batch holds every rank
    switch (deep_nb(p.n)) {
      case 16:
        return reg ? launch_persistent(fused_deep_kernel<BF16, 16, 1, !BF16>, p, tiles, sm_budget, stream)
                   : launch_persistent(fused_deep_kernel<BF16, 16, 1, false>, p, tiles, sm_budget, stream);
      case 8: return launch_persistent(fused_deep_kernel<BF16, 8, 2, !BF16>, p, tiles, sm_budget, stream);
      case 4: return launch_persistent(fused_deep_kernel<BF16, 4, BF16 ? 3 : 4, false>, p, tiles, sm_budget, stream);
      default: return launch_persistent(fused_deep_kernel<BF16, 2, BF16 ? 4 : 5, !BF16>, p, tiles, sm_budget, stream);
    }
  }
  if (p.collective == AR_REDUCE_SCATTER && p.n > 4)
    return launch_persistent(fused_flat_kernel<BF16, false, kSeqRotatedPos, kRsNB, kRsVPT>, p, tiles, sm_budget,
                             stream);
  if (p.collective == AR_ALLGATHER)
    return launch_persistent(fused_flat_kernel<BF16, false, kSeqRotated, 1, kAgVPT>, p, tiles, sm_budget, stream);
  switch (fused_vpt(p.n, p.order, p.collective, BF16, false)) {
    case 4: return launch_persistent(fused_flat_kernel<BF16, false, kSeqRotated, 2, 4>, p, tiles, sm_budget, stream);
    case 2: return launch_persistent(fused_flat_kernel<BF16, false, kSeqRotated, 4, 2>, p, tiles, sm_budget, stream);
    default:
      return p.n > 16 ? launch_persistent(fused_flat_kernel<BF16, false, kSeqRotatedPos, 8, 1>, p, tiles, sm_budget, stream)
                      : launch_persistent(fused_flat_kernel<BF16, false, kSeqRotated, 8, 1>, p, tiles, sm_budget, stream);
  }
}

// The hierarchical order writes each segment's sequence; the other orders
// are rotations of the rank list.
template <bool BF16>
cudaError_t launch_fused_t(const FusedParams& p, int64_t tiles, int sm_budget, cudaStream_t stream) {
  if (p.order == AR_ORDER_HIER && p.collective == AR_ALLREDUCE) {  // the planner allows it for all-reduce only
    switch (fused_vpt(p.n, p.order, p.collective, BF16, budgeted(sm_budget))) {
      case 4: return launch_persistent(fused_flat_kernel<BF16, false, kSeqWritten, 2, 4>, p, tiles, sm_budget, stream);
      case 2:
        return p.n > 4 ? launch_persistent(fused_flat_kernel<BF16, false, kSeqWritten, 8, 2>, p, tiles, sm_budget, stream)
                       : launch_persistent(fused_flat_kernel<BF16, false, kSeqWritten, 4, 2>, p, tiles, sm_budget, stream);
      default: return launch_persistent(fused_flat_kernel<BF16, false, kSeqWritten, 8, 1>, p, tiles, sm_budget, stream);
    }
  }
  return launch_fused_rot<BF16>(p, tiles, sm_budget, stream);
}

cudaError_t launch_fused(const FusedParams& p, ar_dtype dtype, int sm_budget, cudaStream_t stream) {
  const int64_t tiles = int64_t(p.n_seg) * p.tiles_per_seg;
  return dtype == AR_BF16 ? launch_fused_t<true>(p, tiles, sm_budget, stream)
                          : launch_fused_t<false>(p, tiles, sm_budget, stream);
}

// 32-byte lanes (N > 4 only, one vector per thread): each load moves twice the
// bytes, so a batch holds half as many ranks (the same bytes in flight).
// Budgeted launches take the deep kernel: with 32-byte lanes 8 ranks per
// batch (bf16 and fp32 alike), with 16-byte lanes the flat kernel's shapes.
template <bool BF16>
cudaError_t launch_bucket_t(const BucketFusedParams& p, int64_t tiles, int sm_budget, bool v8, cudaStream_t stream) {
  const bool deep = budgeted(sm_budget);
  if (v8)
    return deep ? launch_persistent(fused_bucket_deep_kernel<BF16, true, 8, 1>, p, tiles, sm_budget, stream)
                : launch_persistent(fused_bucket_kernel<BF16, true, 4, 1>, p, tiles, sm_budget, stream);
  if (deep) {
    switch (deep_nb(p.n)) {
      case 16: return launch_persistent(fused_bucket_deep_kernel<BF16, false, 16, 1>, p, tiles, sm_budget, stream);
      case 8: return launch_persistent(fused_bucket_deep_kernel<BF16, false, 8, 2>, p, tiles, sm_budget, stream);
      case 4:
        return launch_persistent(fused_bucket_deep_kernel<BF16, false, 4, BF16 ? 3 : 4>, p, tiles, sm_budget, stream);
      default:
        return launch_persistent(fused_bucket_deep_kernel<BF16, false, 2, BF16 ? 4 : 5>, p, tiles, sm_budget, stream);
    }
  }
  switch (bucket_vpt(p.n, BF16, false)) {
    case 4: return launch_persistent(fused_bucket_kernel<BF16, false, 2, 4>, p, tiles, sm_budget, stream);
    case 2: return launch_persistent(fused_bucket_kernel<BF16, false, 4, 2>, p, tiles, sm_budget, stream);
    default: return launch_persistent(fused_bucket_kernel<BF16, false, 8, 1>, p, tiles, sm_budget, stream);
  }
}

cudaError_t launch_bucket_fused(const BucketFusedParams& p, ar_dtype dtype, int sm_budget, bool v8, cudaStream_t stream) {
  const int64_t tiles = p.tile_start[p.n_seg];
  return dtype == AR_BF16 ? launch_bucket_t<true>(p, tiles, sm_budget, v8, stream)
                          : launch_bucket_t<false>(p, tiles, sm_budget, v8, stream);
}

}  // namespace ar
