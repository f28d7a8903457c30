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
#include "common.cuh"

namespace ar {

namespace {

__device__ __forceinline__ void seq_position(const FusedParams& p, int seg, int pos, int& rank,
                                             uint8_t& flag) {
  const int n = p.n;
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
}

template <bool BF16, bool TREE, int NB>
__global__ void __launch_bounds__(kThreads) fused_flat_kernel(const __grid_constant__ FusedParams p) {
  using LV = Lane<BF16, true>;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W;
  __shared__ const char* s_seq[AR_MAX_RANKS];
  __shared__ uint8_t s_flag[AR_MAX_RANKS];
  __shared__ char* s_out[AR_MAX_RANKS];
  const int n = p.n;
  if (threadIdx.x < n) s_out[threadIdx.x] = static_cast<char*>(p.out[threadIdx.x]);
  int cur = -1;
  int64_t lo = 0, hi = 0;
  const int64_t total = int64_t(p.n_seg) * p.tiles_per_seg;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int seg = int(t / p.tiles_per_seg);
    const int64_t tt = t - int64_t(seg) * p.tiles_per_seg;
    if (seg != cur) {  // uniform across the CTA
      __syncthreads();
      cur = seg;
      seg_range(p, seg, lo, hi);
      if (threadIdx.x < n) {
        int rank;
        uint8_t flag;
        seq_position(p, seg, threadIdx.x, rank, flag);
        s_seq[threadIdx.x] = static_cast<const char*>(p.in[rank]);
        s_flag[threadIdx.x] = flag;
      }
      __syncthreads();
    }
    const int64_t clo = lo > p.e_lo ? lo : p.e_lo;
    const int64_t chi = hi < p.e_hi ? hi : p.e_hi;
    if (clo >= chi) continue;
    const int64_t a0 = round_up(clo, W);
    int64_t a1 = round_down(chi, W);
    if (a1 < a0) a1 = a0;
    const int64_t e = a0 + tt * kTile + int64_t(threadIdx.x) * W;
    if (e < a1) {
      float acc[W];
      if (TREE)
        fold_tree<LV, NB>(acc, s_seq, n, e);
      else
        fold_sequence<LV, NB>(acc, s_seq, s_flag, n, e);
#pragma unroll
      for (int w = 0; w < W; ++w) acc[w] = fmul(acc[w], p.scale);
      const typename LV::raw_t r = LV::narrow(acc);
#pragma unroll 4
      for (int q = 0; q < n; ++q) LV::store(s_out[q], e, r);
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
        float acc[1];
        if (TREE)
          fold_tree<LS, 8>(acc, s_seq, n, es);
        else
          fold_sequence<LS, 8>(acc, s_seq, s_flag, n, es);
        acc[0] = fmul(acc[0], p.scale);
        const typename LS::raw_t r = LS::narrow(acc);
        for (int q = 0; q < n; ++q) LS::store(s_out[q], es, r);
      }
    }
  }
}

// Bucket variant: every rank's gradient tensors are read in place through a
// (tensor, rank) pointer table; segments are the pieces of the tensors cut at
// the ring's chunk boundaries over the packed bucket, so each segment is
// folded in ring order from its chunk's rank.
template <bool BF16, int NB>
__global__ void __launch_bounds__(kThreads)
    fused_bucket_kernel(const __grid_constant__ BucketFusedParams p) {
  using LV = Lane<BF16, true>;
  using LS = Lane<BF16, false>;
  constexpr int W = LV::W;
  constexpr int64_t kTile = int64_t(kThreads) * W;
  __shared__ const char* s_seq[AR_MAX_RANKS];
  __shared__ uint8_t s_flag[AR_MAX_RANKS];
  __shared__ char* s_out[AR_MAX_RANKS];
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
    const int64_t e = a0 + tt * kTile + int64_t(threadIdx.x) * W;
    if (e < a1) {
      float acc[W];
      fold_sequence<LV, NB>(acc, s_seq, s_flag, n, e);
#pragma unroll
      for (int w = 0; w < W; ++w) acc[w] = fmul(acc[w], p.scale);
      const typename LV::raw_t r = LV::narrow(acc);
#pragma unroll 4
      for (int q = 0; q < n; ++q) LV::store(s_out[q], e, r);
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
        float acc[1];
        fold_sequence<LS, 8>(acc, s_seq, s_flag, n, es);
        acc[0] = fmul(acc[0], p.scale);
        const typename LS::raw_t r = LS::narrow(acc);
        for (int q = 0; q < n; ++q) LS::store(s_out[q], es, r);
      }
    }
  }
}

template <class P>
cudaError_t launch_persistent(void (*kernel)(P), const P& p, int64_t tiles, cudaStream_t stream) {
  if (tiles <= 0) return cudaSuccess;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kernel), tiles);
  kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int64_t fused_tile_elems(ar_dtype dtype) { return int64_t(kThreads) * (dtype == AR_BF16 ? 8 : 4); }

cudaError_t launch_fused(const FusedParams& p, ar_dtype dtype, cudaStream_t stream) {
  const int64_t tiles = int64_t(p.n_seg) * p.tiles_per_seg;
  const bool tree = p.order == AR_ORDER_TREE;
  if (dtype == AR_BF16)
    return tree ? launch_persistent(fused_flat_kernel<true, true, 8>, p, tiles, stream)
                : launch_persistent(fused_flat_kernel<true, false, 16>, p, tiles, stream);
  return tree ? launch_persistent(fused_flat_kernel<false, true, 8>, p, tiles, stream)
              : launch_persistent(fused_flat_kernel<false, false, 16>, p, tiles, stream);
}

cudaError_t launch_bucket_fused(const BucketFusedParams& p, ar_dtype dtype, cudaStream_t stream) {
  const int64_t tiles = p.tile_start[p.n_seg];
  if (dtype == AR_BF16) return launch_persistent(fused_bucket_kernel<true, 16>, p, tiles, stream);
  return launch_persistent(fused_bucket_kernel<false, 16>, p, tiles, stream);
}

}  // namespace ar
