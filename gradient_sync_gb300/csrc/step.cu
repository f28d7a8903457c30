// One dependent step of a schedule (ring, Rabenseifner or hierarchical), run
// as one kernel over all of the step's transfers at once.
//
// In a step every rank sends one piece to one peer and receives one piece
// (primer ch. 4, "Collective communication: algorithms, cost and the library
// that runs them", §4.2: in each of the 2(N-1) ring steps all N links carry
// one chunk at the same time; a step cannot start before the previous chunk
// has arrived and been added). With virtual ranks in one HBM, "rank dst
// receives [lo, hi) from rank src" is dst's kernel thread reading src's buffer
// directly: reduce-scatter adds its own copy (2 reads + 1 write per element),
// all-gather overwrites (1 read + 1 write). The kernel boundary is the step
// boundary; consecutive steps are chained with programmatic dependent launch
// so that the next step's CTAs are already resident when this one drains.
//
// Within a step no transfer writes a range another transfer reads (every
// rank receives a different piece than the one it sends), so a step is safe
// in place. An exchange (`pair`: both partners receive the same sum, as in
// recursive doubling) reads both copies of an element and writes both from
// the same thread, so it is safe in place too.
#include <atomic>

#include "common.cuh"

namespace ar {

namespace {

struct Operand {
  char* base;
  bool f32;
};

template <bool BF16>
__device__ __forceinline__ Operand operand(const StepParams& p, int space, int rank) {
  if (space == RAW) return {static_cast<char*>(p.raw[rank]), !BF16};
  if (space == RES) return {static_cast<char*>(p.res[rank]), !BF16};
  // PART: fp32 partial sums -- the output buffer itself for fp32 runs, the
  // rank's slice of the workspace for bf16 runs
  if (BF16) return {reinterpret_cast<char*>(p.ws + int64_t(rank) * p.ws_stride), true};
  return {static_cast<char*>(p.res[rank]), true};
}

// 8 elements = 32 bytes of fp32 (two 16-byte words) or 16 bytes of bf16.
struct Raw8 {
  uint4 a, b;
};

// Loads and stores: streaming (evict-first) for the add steps, whose results
// are read again only a step or more later; ordinary caching for the copy
// steps, whose chunk the next step forwards (ring all-gather: 0.82 of its
// bytes against 0.79 with streaming hints, measured on GB300 at 16 x 192 MiB).
template <bool STREAM>
__device__ __forceinline__ uint4 ld16(const uint4* q) {
  if (STREAM) return __ldcs(q);
  return *q;
}
template <bool STREAM>
__device__ __forceinline__ void st16(uint4* q, const uint4& v) {
  if (STREAM)
    __stcs(q, v);
  else
    *q = v;
}

// 256-bit accesses (ld/st.global.v8.b32, sm_100 and later) move the 8 fp32
// elements of a vector with one instruction instead of two. They need 32-byte
// aligned addresses: the host selects them (V8) only when every base pointer
// of the call is 32-byte aligned, as vectors start at multiples of 8 elements.
// Measured on GB300 at 16 x 192 MiB fp32: ring 0.918 -> 0.939, Rabenseifner
// 0.921 -> 0.957, recursive doubling 0.837 -> 0.959 of their bytes (fewer
// memory instructions: the load/store queue was the second stall after
// latency).
template <bool STREAM, bool V8>
__device__ __forceinline__ Raw8 load8(const Operand& o, int64_t e) {
  Raw8 r;
  if (o.f32) {
    if (V8) {
      const char* a = o.base + e * 4;
      if (STREAM)
        asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y), "=r"(r.b.z),
                       "=r"(r.b.w)
                     : "l"(a));
      else
        asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y), "=r"(r.b.z),
                       "=r"(r.b.w)
                     : "l"(a));
      return r;
    }
    const uint4* q = reinterpret_cast<const uint4*>(o.base + e * 4);
    r.a = ld16<STREAM>(q);
    r.b = ld16<STREAM>(q + 1);
  } else {
    r.a = ld16<STREAM>(reinterpret_cast<const uint4*>(o.base + e * 2));
    r.b = make_uint4(0, 0, 0, 0);
  }
  return r;
}

// Store the 32 bytes of an fp32 vector as they are.
template <bool STREAM, bool V8>
__device__ __forceinline__ void store_raw8(char* base, int64_t e, const Raw8& r) {
  if (V8) {
    if (STREAM)
      asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(base + e * 4), "r"(r.a.x), "r"(r.a.y),
                   "r"(r.a.z), "r"(r.a.w), "r"(r.b.x), "r"(r.b.y), "r"(r.b.z), "r"(r.b.w)
                   : "memory");
    else
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(base + e * 4), "r"(r.a.x), "r"(r.a.y),
                   "r"(r.a.z), "r"(r.a.w), "r"(r.b.x), "r"(r.b.y), "r"(r.b.z), "r"(r.b.w)
                   : "memory");
    return;
  }
  uint4* q = reinterpret_cast<uint4*>(base + e * 4);
  st16<STREAM>(q, r.a);
  st16<STREAM>(q + 1, r.b);
}

__device__ __forceinline__ void widen8(const Raw8& r, bool f32, float (&f)[8]) {
  if (f32) {
    f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y);
    f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
    f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y);
    f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
  } else {
    f[0] = bf16lo(r.a.x); f[1] = bf16hi(r.a.x); f[2] = bf16lo(r.a.y); f[3] = bf16hi(r.a.y);
    f[4] = bf16lo(r.a.z); f[5] = bf16hi(r.a.z); f[6] = bf16lo(r.a.w); f[7] = bf16hi(r.a.w);
  }
}

template <bool V8>
__device__ __forceinline__ void store8(const Operand& o, int64_t e, const float (&f)[8]) {
  if (o.f32) {
    Raw8 r;
    r.a = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    r.b = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7]));
    store_raw8<true, V8>(o.base, e, r);
  } else {
    __stcs(reinterpret_cast<uint4*>(o.base + e * 2),
           make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7])));
  }
}

__device__ __forceinline__ float load1(const Operand& o, int64_t e) {
  if (o.f32) return reinterpret_cast<const float*>(o.base)[e];
  return bf16_to_f32(reinterpret_cast<const uint16_t*>(o.base)[e]);
}

__device__ __forceinline__ void store1(const Operand& o, int64_t e, float v) {
  if (o.f32)
    reinterpret_cast<float*>(o.base)[e] = v;
  else
    reinterpret_cast<uint16_t*>(o.base)[e] = f32_to_bf16(v);
}

template <bool BF16, int OP, bool V8>
__global__ void __launch_bounds__(kThreads) step_kernel(const __grid_constant__ StepParams p) {
  constexpr bool kStream = OP != OP_COPY;
  grid_dependency_wait();
  grid_dependents_launch();
  // Tile order: transfer by transfer (tile t of the prefix sums), or dealt
  // round-robin over the transfers (tile t is tile t / n_xfer of transfer
  // t % n_xfer, skipped past that transfer's end). The double binary tree's
  // steps run faster interleaved (1.00 of their bytes against 0.95 at 16 x
  // 192 MiB on GB300); the ring, Rabenseifner and hierarchical steps run 2-4 %
  // slower interleaved, so the host picks per plan.
  int max_tiles = 0;
  if (p.interleave)
    for (int x = 0; x < p.n_xfer; ++x) max_tiles = max(max_tiles, p.tile_start[x + 1] - p.tile_start[x]);
  const int total = p.interleave ? max_tiles * p.n_xfer : p.tile_start[p.n_xfer];
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int lo_i = 0;
    int64_t tt = 0;
    if (p.interleave) {  // uniform across the grid
      lo_i = t % p.n_xfer;
      tt = t / p.n_xfer;
      if (tt >= p.tile_start[lo_i + 1] - p.tile_start[lo_i]) continue;
    } else {
      int hi_i = p.n_xfer;  // find x with tile_start[x] <= t < tile_start[x+1]
      while (hi_i - lo_i > 1) {
        const int mid = (lo_i + hi_i) >> 1;
        if (p.tile_start[mid] <= t)
          lo_i = mid;
        else
          hi_i = mid;
      }
      tt = t - p.tile_start[lo_i];
    }
    const Transfer tr = p.x[lo_i];
    const Operand X = operand<BF16>(p, tr.xs, tr.src);
    const Operand Y = operand<BF16>(p, tr.ys, tr.dst);
    const Operand D = operand<BF16>(p, tr.ds, tr.dst);
    const bool two = OP == OP_ADD && tr.src2 >= 0;  // uniform over the transfer
    // pair: an add's sum also goes to the sender's copy (an exchange); a copy
    // also writes the sender's output (the all-gather's own chunk)
    const bool pair = tr.pair != 0;
    const Operand X2 = operand<BF16>(p, tr.x2s, two ? tr.src2 : tr.dst);
    const Operand D2 = operand<BF16>(p, tr.ds, tr.src);
    const bool fin = tr.fin != 0;
    const int64_t a0 = round_up(tr.lo, kStepVec);
    int64_t a1 = round_down(tr.hi, kStepVec);
    if (a1 < a0) a1 = a0;

    int64_t e[kStepUnroll];
    Raw8 rx[kStepUnroll], ry[kStepUnroll], rz[kStepUnroll];
#pragma unroll
    for (int u = 0; u < kStepUnroll; ++u) {
      e[u] = a0 + tt * kStepTile + (int64_t(u) * kThreads + threadIdx.x) * kStepVec;
      if (e[u] < a1) {
        rx[u] = load8<kStream, V8>(X, e[u]);
        if (OP == OP_ADD) ry[u] = load8<kStream, V8>(Y, e[u]);
        if (two) rz[u] = load8<kStream, V8>(X2, e[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kStepUnroll; ++u) {
      if (e[u] < a1) {
        if (OP == OP_COPY) {  // same type on both sides: move the bytes
          if (X.f32) {
            store_raw8<kStream, V8>(D.base, e[u], rx[u]);
            if (pair) store_raw8<kStream, V8>(D2.base, e[u], rx[u]);
          } else {
            st16<kStream>(reinterpret_cast<uint4*>(D.base + e[u] * 2), rx[u].a);
            if (pair) st16<kStream>(reinterpret_cast<uint4*>(D2.base + e[u] * 2), rx[u].a);
          }
        } else {
          float f[8];
          widen8(rx[u], X.f32, f);
          if (OP == OP_ADD) {
            float g[8];
            widen8(ry[u], Y.f32, g);
#pragma unroll
            for (int w = 0; w < 8; ++w) f[w] = fadd(f[w], g[w]);
            if (two) {
              widen8(rz[u], X2.f32, g);
#pragma unroll
              for (int w = 0; w < 8; ++w) f[w] = fadd(f[w], g[w]);
            }
          }
          if (fin) {
#pragma unroll
            for (int w = 0; w < 8; ++w) f[w] = fmul(f[w], p.scale);
          }
          store8<V8>(D, e[u], f);
          if (pair) store8<V8>(D2, e[u], f);
        }
      }
    }
    if (tt == 0) {  // ragged head [lo, min(a0, hi)) and tail [a1, hi), element by element
      int64_t es = -1;
      const int64_t head_end = a0 < tr.hi ? a0 : tr.hi;
      if (threadIdx.x < kStepVec - 1) {
        es = tr.lo + threadIdx.x;
        if (es >= head_end) es = -1;
      } else if (threadIdx.x >= 32 && threadIdx.x < 32 + kStepVec - 1) {
        es = a1 + (threadIdx.x - 32);
        if (es >= tr.hi) es = -1;
      }
      if (es >= 0) {
        float v = load1(X, es);
        if (OP == OP_ADD) v = fadd(v, load1(Y, es));
        if (two) v = fadd(v, load1(X2, es));
        if (OP != OP_COPY && fin) v = fmul(v, p.scale);
        store1(D, es, v);
        if (pair) store1(D2, es, v);
      }
    }
  }
}

// ---------------------------------------------------------------- small plans
// A plan whose buffers are a few KiB spends its time on the step boundaries:
// a kernel boundary costs about 1.6 us, the data of a step a fraction of that.
// Here one CTA runs every step of the schedule, with a block barrier as the
// step boundary: a step's stores are visible to every thread of the block
// after the barrier, and no CTA waits on another. Each thread takes the
// step's elements kSmallThreads apart, finds each element's transfer by a
// binary search over the step's prefix counts, and applies exactly the step
// kernel's per-element operations (x + y, + x2, times the scale, rounded to
// the destination type), so the results are the same bits.
template <bool BF16>
__device__ __forceinline__ Operand small_operand(const SmallParams& p, int space, int rank) {
  if (space == RAW) return {static_cast<char*>(p.raw[rank]), !BF16};
  if (space == RES) return {static_cast<char*>(p.res[rank]), !BF16};
  if (BF16) return {reinterpret_cast<char*>(p.ws + int64_t(rank) * p.ws_stride), true};
  return {static_cast<char*>(p.res[rank]), true};
}

constexpr int kSmallThreads = 1024;
constexpr int kSmallBatch = 4;  // elements per thread with their loads in flight together

template <bool BF16>
__global__ void __launch_bounds__(kSmallThreads) small_steps_kernel(const __grid_constant__ SmallParams p) {
  // The transfer table in shared memory: the per-element search reads it
  // there rather than from parameter memory.
  __shared__ SmallXfer tab[kMaxSmallXfers];
  static_assert(sizeof(SmallXfer) % 4 == 0, "copied as words");
  {
    const int words = p.step_start[p.n_steps] * int(sizeof(SmallXfer) / 4);
    const uint32_t* from = reinterpret_cast<const uint32_t*>(p.x);
    uint32_t* to = reinterpret_cast<uint32_t*>(tab);
    for (int i = threadIdx.x; i < words; i += kSmallThreads) to[i] = from[i];
  }
  __syncthreads();
  grid_dependency_wait();
  grid_dependents_launch();
  for (int s = 0; s < p.n_steps; ++s) {
    const int x0 = p.step_start[s], x1 = p.step_start[s + 1];
    const int total = p.step_elems[s];
    const int op = p.step_op[s];
    for (int f0 = threadIdx.x; f0 < total; f0 += kSmallThreads * kSmallBatch) {
      int xi[kSmallBatch];
      int64_t e[kSmallBatch];
      float v[kSmallBatch];
      uint32_t bits[kSmallBatch];
#pragma unroll
      for (int u = 0; u < kSmallBatch; ++u) {
        const int f = f0 + u * kSmallThreads;
        xi[u] = -1;
        if (f >= total) continue;
        int lo = x0, hi = x1;  // the last transfer whose first flat index is <= f
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (tab[mid].flat <= f)
            lo = mid;
          else
            hi = mid;
        }
        xi[u] = lo;
        const SmallXfer& t = tab[lo];
        e[u] = int64_t(t.lo) + (f - t.flat);
        const Operand X = small_operand<BF16>(p, t.xs, t.src);
        if (op == OP_COPY) {  // same type on both sides: move the bits
          bits[u] = X.f32 ? reinterpret_cast<const uint32_t*>(X.base)[e[u]]
                          : uint32_t(reinterpret_cast<const uint16_t*>(X.base)[e[u]]);
          continue;
        }
        v[u] = load1(X, e[u]);
        if (op == OP_ADD) {
          v[u] = fadd(v[u], load1(small_operand<BF16>(p, t.ys, t.dst), e[u]));
          if (t.src2 >= 0) v[u] = fadd(v[u], load1(small_operand<BF16>(p, t.x2s, t.src2), e[u]));
        }
        if (t.fin) v[u] = fmul(v[u], p.scale);
      }
#pragma unroll
      for (int u = 0; u < kSmallBatch; ++u) {
        if (xi[u] < 0) continue;
        const SmallXfer& t = tab[xi[u]];
        const Operand D = small_operand<BF16>(p, t.ds, t.dst);
        if (op == OP_COPY) {
          if (D.f32)
            reinterpret_cast<uint32_t*>(D.base)[e[u]] = bits[u];
          else
            reinterpret_cast<uint16_t*>(D.base)[e[u]] = uint16_t(bits[u]);
          continue;
        }
        store1(D, e[u], v[u]);
        if (op == OP_ADD && t.pair) store1(small_operand<BF16>(p, t.ds, t.src), e[u], v[u]);
      }
    }
    __syncthreads();  // the step boundary
  }
}

// The same schedule on chip. A step's time above is mostly a round trip to
// the L2 (a thread reads what another thread stored a step earlier), the
// per-element search for its transfer, and the barrier. Here the CTA first
// copies every rank's input (and the output of ranks that run out of place)
// into shared memory, runs every step there with the same per-element
// operations and the same roundings (a bf16 space holds bf16 values, the
// partials fp32), and finally writes every rank's output back. The spaces
// alias as they do in memory: a rank that runs in place has one copy for its
// input and output, and fp32 partials are the output itself. The host cuts
// the transfers into pieces of at most kSmallPiece elements and resolves
// each piece's operands to shared-memory offsets; a warp takes whole pieces
// (lane l: elements l, l + 32, ...), so no element searches for its transfer
// and a piece is one table read. The CTA has one warp per piece of the
// widest step (a block barrier costs less with fewer warps).
//
// Layout of the dynamic shared memory (the host computes the same offsets):
//   [0, T)             the pieces, T = their bytes rounded up to 16
//   [T, T + 4NL)       bf16 only: the fp32 partials of the N ranks
//   then               the N ranks' inputs (NL elements of the buffers' type)
//   then               the N ranks' outputs, for the ranks out of place

__device__ __forceinline__ float smem_ld(const char* base, uint32_t off, int k, bool f32) {
  if (f32) return *reinterpret_cast<const float*>(base + off + 4 * k);
  return bf16_to_f32(*reinterpret_cast<const uint16_t*>(base + off + 2 * k));
}
__device__ __forceinline__ void smem_st(char* base, uint32_t off, int k, bool f32, float v) {
  if (f32)
    *reinterpret_cast<float*>(base + off + 4 * k) = v;
  else
    *reinterpret_cast<uint16_t*>(base + off + 2 * k) = f32_to_bf16(v);
}

// Copy `words` 4-byte words or (vec) 16-byte vectors of every rank between
// memory and shared memory, all of a thread's loads issued before its stores.
// Rank r's words are [r * words, (r + 1) * words) of the shared copy; ranks
// whose bit is set in `skip` are left out.
template <class W, bool TO_SMEM>
__device__ __forceinline__ void copy_ranks(char* const* mem, const uint64_t skip, char* smem_base, int n, int words) {
  constexpr int kU = 8;
  const int total = n * words, step = int(blockDim.x);
  for (int i0 = threadIdx.x; i0 < total; i0 += step * kU) {
    W v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * step;
      if (i >= total) continue;
      const int r = i / words;
      if ((skip >> r) & 1) continue;
      W* m = reinterpret_cast<W*>(mem[r]) + (i - r * words);
      W* sm = reinterpret_cast<W*>(smem_base) + i;
      v[u] = TO_SMEM ? *m : *sm;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * step;
      if (i >= total) continue;
      const int r = i / words;
      if ((skip >> r) & 1) continue;
      W* m = reinterpret_cast<W*>(mem[r]) + (i - r * words);
      W* sm = reinterpret_cast<W*>(smem_base) + i;
      if (TO_SMEM)
        *sm = v[u];
      else
        *m = v[u];
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kSmallThreads) small_steps_smem_kernel(const __grid_constant__ SmallParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  char* const base = reinterpret_cast<char*>(smem);
  constexpr int esz = BF16 ? 2 : 4;
  const int n = p.n_ranks, L = p.count, nt = int(blockDim.x);
  const int n_x = p.step_start[p.n_steps];
  const SmemPiece* tab = reinterpret_cast<const SmemPiece*>(smem);
  const int tab_bytes = (n_x * int(sizeof(SmemPiece)) + 15) / 16 * 16;
  char* const raw_s = base + tab_bytes + (BF16 ? n * L * 4 : 0);
  char* const res_s = raw_s + n * L * esz;
  // The table and the steps' starts and ops in shared memory: a parameter
  // read at an index that changes every step can miss the constant cache.
  __shared__ int32_t s_start[kMaxSmallSteps + 1];
  __shared__ uint8_t s_op[kMaxSmallSteps];
  {
    const int words = n_x * int(sizeof(SmemPiece) / 4);
    const uint32_t* from = reinterpret_cast<const uint32_t*>(p.px);
    uint32_t* to = reinterpret_cast<uint32_t*>(smem);
    for (int i = threadIdx.x; i < words; i += nt) to[i] = from[i];
    for (int i = threadIdx.x; i <= p.n_steps; i += nt) s_start[i] = p.step_start[i];
    for (int i = threadIdx.x; i < p.n_steps; i += nt) s_op[i] = p.step_op[i];
  }
  grid_dependency_wait();
  grid_dependents_launch();
  // every rank's input, and the current output of the ranks out of place
  // (elements a plan does not write keep their value on the way back)
  const int bytes = L * esz;  // a multiple of 4 (the host checks), of 16 with vec16
  char* const* raw = reinterpret_cast<char* const*>(p.raw);
  char* const* res = reinterpret_cast<char* const*>(p.res);
  if (p.vec16) {
    copy_ranks<uint4, true>(raw, 0, raw_s, n, bytes / 16);
    copy_ranks<uint4, true>(res, p.in_place, res_s, n, bytes / 16);
  } else {
    copy_ranks<uint32_t, true>(raw, 0, raw_s, n, bytes / 4);
    copy_ranks<uint32_t, true>(res, p.in_place, res_s, n, bytes / 4);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, warps = nt >> 5;
  constexpr int kPer = kSmallPiece / 32;  // elements per lane of a piece
  const int n_steps = p.n_steps;
  const float scale = p.scale;
  for (int s = 0; s < n_steps; ++s) {
    const int x1 = s_start[s + 1];
    const int op = s_op[s];
    for (int x = s_start[s] + warp; x < x1; x += warps) {
      const SmemPiece t = tab[x];  // the same piece for the whole warp
      const bool x32 = !BF16 || (t.flags & kPieceX32), d32 = !BF16 || (t.flags & kPieceD32);
      if (op == OP_COPY) {  // same type on both sides: move the bits
        uint32_t bits[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int k = lane + 32 * u;
          if (k < t.len)
            bits[u] = x32 ? *reinterpret_cast<const uint32_t*>(base + t.x + 4 * k)
                          : uint32_t(*reinterpret_cast<const uint16_t*>(base + t.x + 2 * k));
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int k = lane + 32 * u;
          if (k >= t.len) continue;
          if (d32)
            *reinterpret_cast<uint32_t*>(base + t.d + 4 * k) = bits[u];
          else
            *reinterpret_cast<uint16_t*>(base + t.d + 2 * k) = uint16_t(bits[u]);
        }
        continue;
      }
      const bool add = op == OP_ADD;
      const bool two = add && (t.flags & kPieceTwo), pair = add && (t.flags & kPiecePair);
      const bool fin = t.flags & kPieceFin;
      const bool y32 = !BF16 || (t.flags & kPieceY32), x2_32 = !BF16 || (t.flags & kPieceX2_32);
      float v[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int k = lane + 32 * u;
        if (k >= t.len) continue;
        v[u] = smem_ld(base, t.x, k, x32);
        if (add) {
          v[u] = fadd(v[u], smem_ld(base, t.y, k, y32));
          if (two) v[u] = fadd(v[u], smem_ld(base, t.x2, k, x2_32));
        }
        if (fin) v[u] = fmul(v[u], scale);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int k = lane + 32 * u;
        if (k >= t.len) continue;
        smem_st(base, t.d, k, d32, v[u]);
        if (pair) smem_st(base, t.d2, k, d32, v[u]);
      }
    }
    __syncthreads();  // the step boundary
  }
  // every rank's output back to memory: from its own copy for the ranks out
  // of place, from the shared input copy for the ranks in place
  const uint64_t all = n == 64 ? ~uint64_t(0) : (uint64_t(1) << n) - 1;
  if (p.vec16) {
    copy_ranks<uint4, false>(res, p.in_place, res_s, n, bytes / 16);
    copy_ranks<uint4, false>(raw, all & ~p.in_place, raw_s, n, bytes / 16);
  } else {
    copy_ranks<uint32_t, false>(res, p.in_place, res_s, n, bytes / 4);
    copy_ranks<uint32_t, false>(raw, all & ~p.in_place, raw_s, n, bytes / 4);
  }
}

template <bool BF16, bool V8>
cudaError_t launch_op(const StepParams& p, StepOp op, int tiles, bool pdl, int sm_budget, cudaStream_t stream) {
  void (*k)(StepParams) = op == OP_ADD ? step_kernel<BF16, OP_ADD, V8>
                          : op == OP_COPY ? step_kernel<BF16, OP_COPY, V8>
                                          : step_kernel<BF16, OP_FINISH, V8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(persistent_grid(reinterpret_cast<const void*>(k), tiles, sm_budget));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;  // safe either way: the kernel waits on griddepcontrol.wait first
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace

cudaError_t launch_small_steps(const SmallParams& p, ar_dtype dtype, cudaStream_t stream) {
  void (*k)(SmallParams) = dtype == AR_BF16 ? small_steps_kernel<true> : small_steps_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

cudaError_t launch_small_steps_smem(const SmallParams& p, ar_dtype dtype, cudaStream_t stream) {
  void (*k)(SmallParams) = dtype == AR_BF16 ? small_steps_smem_kernel<true> : small_steps_smem_kernel<false>;
  const int64_t tab = (int64_t(p.step_start[p.n_steps]) * int64_t(sizeof(SmemPiece)) + 15) / 16 * 16;
  const int64_t bytes = tab + small_smem_data_bytes(p.n_ranks, p.count);
  // Allow the largest table and data once per device and kernel.
  static std::atomic<uint64_t> allowed[2];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  std::atomic<uint64_t>& mask = allowed[dtype == AR_BF16 ? 1 : 0];
  if ((mask.load(std::memory_order_acquire) & bit) == 0) {
    const int most = int(int64_t(kMaxSmallXfers) * int64_t(sizeof(SmemPiece)) + kSmallSmemDataBytes);
    err = cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (err != cudaSuccess) return err;
    mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = size_t(bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

cudaError_t launch_step(const StepParams& p, ar_dtype dtype, StepOp op, int total_tiles, bool pdl,
                        int sm_budget, bool v8, cudaStream_t stream) {
  if (total_tiles <= 0) return cudaSuccess;
  if (dtype == AR_BF16)
    return v8 ? launch_op<true, true>(p, op, total_tiles, pdl, sm_budget, stream)
              : launch_op<true, false>(p, op, total_tiles, pdl, sm_budget, stream);
  return v8 ? launch_op<false, true>(p, op, total_tiles, pdl, sm_budget, stream)
            : launch_op<false, false>(p, op, total_tiles, pdl, sm_budget, stream);
}

}  // namespace ar
