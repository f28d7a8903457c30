// Blockwise INT8 gradient compression with error feedback, and the compressed
// all-reduce built on it (Scaling ML Systems, "Collective communication", the
// section on gradient compression: "Quantization: reducing precision",
// "Blockwise quantization for gradient communication", "Error feedback and
// residual accumulation").
//
// Per rank r and block k of `block` elements (the last block may be short):
//   x     = g_r + e_r                       (fp32; x = g_r without feedback)
//   s     = max|x| / 127                    (fp32 quotient)
//   q     = clamp(rint(x / s), -127, 127)   (fp32 quotient, ties to even; 0 when s == 0)
//   d     = q * s                           (fp32 product: what the receiver reconstructs)
//   e_r  <- x - d                           (the residual kept for the next step)
// and the reducer sums the N reconstructions in rank order,
//   out = round(scale * (((d_0 + d_1) + ...) + d_{N-1}))
// written to every rank. Every operation is one IEEE fp32 operation rounded
// to nearest even, never contracted, so the results are bit-identical to the
// step-by-step definition.
//
// Three kernels:
//  compress_kernel              g, e -> codes, scales, e'   (the message of every rank)
//  compressed_reduce_kernel     codes, scales -> out        (the receiving side)
//  compressed_allreduce_kernel  g, e -> e', out             (both in one pass; no message
//                                                            is materialised)
//
// Thread geometry of the block-wise kernels: a group of `lanes` threads of one
// warp covers one quantisation block; each thread holds V vectors of 4
// consecutive elements, vector v of lane l at block_base + (v * lanes + l) * 4,
// so the lanes of a group read contiguous 16-byte pieces. Blocks of up to 128
// elements take block / 4 lanes and V = 1 (several blocks per warp); larger
// blocks take the whole warp and V = block / 128. The block maximum is a
// butterfly of shuffles inside the group. The group loop is warp-uniform, so
// every lane reaches every shuffle; lanes past the last block compute on zeros
// and store nothing.
#include "common.cuh"

namespace ar {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Four consecutive elements starting at e (a multiple of 4) as fp32; elements
// at or past `lim` read as 0. A whole vector is one 16-byte (fp32) or 8-byte
// (bf16) load: the base is 16-byte aligned and e a multiple of 4.
template <bool BF16>
__device__ __forceinline__ void load4(const void* base, int64_t e, int64_t lim, float (&f)[4]) {
  if (e + 4 <= lim) {
    if constexpr (BF16) {
      const uint2 w = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e));
      f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    } else {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + e));
      f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
  } else {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      f[w] = 0.0f;
      if (e + w < lim)
        f[w] = BF16 ? bf16_to_f32(static_cast<const uint16_t*>(base)[e + w]) : static_cast<const float*>(base)[e + w];
    }
  }
}

// Store four consecutive elements at e (bf16: rounded to nearest even);
// elements at or past `count` are not written.
template <bool BF16>
__device__ __forceinline__ void store4(void* base, int64_t e, int64_t count, const float (&f)[4]) {
  if (e + 4 <= count) {
    if constexpr (BF16) {
      __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + e),
             make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3])));
    } else {
      __stcs(reinterpret_cast<float4*>(static_cast<float*>(base) + e), make_float4(f[0], f[1], f[2], f[3]));
    }
  } else {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (e + w >= count) continue;
      if (BF16)
        static_cast<uint16_t*>(base)[e + w] = f32_to_bf16(f[w]);
      else
        static_cast<float*>(base)[e + w] = f[w];
    }
  }
}

// The block's scale: the largest |x| over the group's lanes, divided by 127.
// Every lane of the warp must call this (it shuffles across the warp).
template <int V>
__device__ __forceinline__ float group_scale(const float (&x)[V][4], int lanes) {
  float m = 0.0f;
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int w = 0; w < 4; ++w) m = fmaxf(m, fabsf(x[v][w]));
  for (int o = lanes >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  return __fdiv_rn(m, 127.0f);
}

// The code of x in a block of scale s: the nearest integer to the fp32
// quotient x / s (ties to even), clamped to [-127, 127]; 0 when s is 0.
__device__ __forceinline__ int quant_code(float x, float s) {
  if (!(s > 0.0f)) return 0;
  const float t = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
  return int(t);
}

__device__ __forceinline__ uint32_t pack_codes(const int (&c)[4]) {
  return (uint32_t(c[0]) & 0xFFu) | ((uint32_t(c[1]) & 0xFFu) << 8) | ((uint32_t(c[2]) & 0xFFu) << 16) |
         ((uint32_t(c[3]) & 0xFFu) << 24);
}

__device__ __forceinline__ float code_of(uint32_t word, int j) {
  return float(static_cast<int8_t>(static_cast<uint8_t>(word >> (8 * j))));
}

struct GroupGeom {
  int lanes, sub, gpw;  // lanes per group, this lane's index in it, groups per warp
  int64_t warp, n_warps;
};

template <int V>
__device__ __forceinline__ GroupGeom group_geom(int block) {
  GroupGeom g;
  g.lanes = V > 1 ? 32 : block / 4;
  const int lane = threadIdx.x & 31;
  g.sub = lane & (g.lanes - 1);
  g.gpw = 32 / g.lanes;
  g.warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  g.n_warps = (int64_t(gridDim.x) * kThreads) >> 5;
  return g;
}

// ---------------------------------------------------------------- compress
// One group per (rank, block): codes, the block's scale and (with error
// feedback) the new residual of that rank's block.
template <bool BF16, int V, bool EF>
__global__ void __launch_bounds__(kThreads) compress_kernel(const __grid_constant__ CompressParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const GroupGeom gg = group_geom<V>(p.block);
  const int64_t total = p.n_blocks * p.n;
  for (int64_t g0 = gg.warp * gg.gpw; g0 < total; g0 += gg.n_warps * gg.gpw) {
    const int64_t gid = g0 + (threadIdx.x & 31) / gg.lanes;
    const bool live = gid < total;
    const int r = live ? int(gid / p.n_blocks) : 0;
    const int64_t k = live ? gid - int64_t(r) * p.n_blocks : 0;
    const int64_t base = k * p.block;
    const int64_t lim = live ? p.count : 0;  // lanes past the last block read nothing
    float x[V][4];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int64_t e = base + (int64_t(v) * gg.lanes + gg.sub) * 4;
      load4<BF16>(p.g[r], e, lim, x[v]);
      if (EF) {
        float ev[4];
        load4<false>(p.e[r], e, lim, ev);
#pragma unroll
        for (int w = 0; w < 4; ++w) x[v][w] = fadd(x[v][w], ev[w]);
      }
    }
    const float s = group_scale<V>(x, gg.lanes);
    if (!live) continue;
    if (gg.sub == 0) p.s[r][k] = s;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int64_t e = base + (int64_t(v) * gg.lanes + gg.sub) * 4;
      if (e >= p.count) continue;
      int c[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) c[w] = quant_code(x[v][w], s);
      int8_t* q = p.q[r];
      if (e + 4 <= p.count) {
        __stcs(reinterpret_cast<unsigned int*>(q + e), pack_codes(c));
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (e + w < p.count) q[e + w] = static_cast<int8_t>(c[w]);
      }
      if (EF) {
        float res[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) res[w] = __fsub_rn(x[v][w], fmul(float(c[w]), s));
        store4<false>(p.e[r], e, p.count, res);
      }
    }
  }
}

// ---------------------------------------------------------------- reduce
// The receiving side: each thread takes 16 consecutive elements (one 16-byte
// vector of codes per rank; a block is a multiple of 16 elements, so the 16
// share one scale), reconstructs every rank's values, sums them in rank order,
// scales once and writes the result to every rank. Loads are issued NB ranks
// at a time before any arithmetic.
template <bool BF16OUT>
__global__ void __launch_bounds__(kThreads) compressed_reduce_kernel(const __grid_constant__ CompressParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  constexpr int NB = 8;
  const int64_t n16 = (p.count + 15) >> 4;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t t = int64_t(blockIdx.x) * kThreads + threadIdx.x; t < n16; t += stride) {
    const int64_t e = t << 4;
    const int64_t kb = e / p.block;
    if (e + 16 <= p.count) {
      float acc[16];
#pragma unroll 1
      for (int r0 = 0; r0 < p.n; r0 += NB) {
        uint4 c[NB];
        float s[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (r0 + b < p.n) {
            c[b] = __ldcs(reinterpret_cast<const uint4*>(p.q[r0 + b] + e));
            s[b] = __ldg(p.s[r0 + b] + kb);
          }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (r0 + b >= p.n) continue;
          const uint32_t wd[4] = {c[b].x, c[b].y, c[b].z, c[b].w};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float d = fmul(code_of(wd[i >> 2], i & 3), s[b]);
            acc[i] = (r0 + b == 0) ? d : fadd(acc[i], d);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = fmul(acc[i], p.scale);
#pragma unroll 1
      for (int r = 0; r < p.n; ++r) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float f[4] = {acc[4 * h], acc[4 * h + 1], acc[4 * h + 2], acc[4 * h + 3]};
          store4<BF16OUT>(p.out[r], e + 4 * h, p.count, f);
        }
      }
    } else {  // the ragged end of the buffer, one element at a time
      for (int64_t x = e; x < p.count; ++x) {
        float a = 0.0f;
        for (int r = 0; r < p.n; ++r) {
          const float d = fmul(float(p.q[r][x]), p.s[r][kb]);
          a = r == 0 ? d : fadd(a, d);
        }
        a = fmul(a, p.scale);
        for (int r = 0; r < p.n; ++r) {
          if (BF16OUT)
            static_cast<uint16_t*>(p.out[r])[x] = f32_to_bf16(a);
          else
            static_cast<float*>(p.out[r])[x] = a;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- fused
// One group per block index k, over all ranks in rank order: quantise rank
// r's block, add its reconstruction to the running sum, store its residual;
// then write the scaled sum to every rank. No message leaves the registers.
// For small V the next rank's block is loaded before this rank's shuffles.
template <bool BF16, int V, bool EF>
__global__ void __launch_bounds__(kThreads) compressed_allreduce_kernel(const __grid_constant__ CompressParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  constexpr bool kPrefetch = V <= 2;
  const GroupGeom gg = group_geom<V>(p.block);
  const int64_t total = p.n_blocks;
  for (int64_t g0 = gg.warp * gg.gpw; g0 < total; g0 += gg.n_warps * gg.gpw) {
    const int64_t k = g0 + (threadIdx.x & 31) / gg.lanes;
    const bool live = k < total;
    const int64_t base = live ? k * p.block : 0;
    const int64_t lim = live ? p.count : 0;
    int64_t ev_at[V];
#pragma unroll
    for (int v = 0; v < V; ++v) ev_at[v] = base + (int64_t(v) * gg.lanes + gg.sub) * 4;
    float acc[V][4];
    float ng[V][4], ne[V][4];  // the next rank's gradient and residual (prefetch)
    if (kPrefetch) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        load4<BF16>(p.g[0], ev_at[v], lim, ng[v]);
        if (EF) load4<false>(p.e[0], ev_at[v], lim, ne[v]);
      }
    }
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) {
      float x[V][4];
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float gv[4], evv[4];
        if (kPrefetch) {
#pragma unroll
          for (int w = 0; w < 4; ++w) { gv[w] = ng[v][w]; evv[w] = EF ? ne[v][w] : 0.0f; }
        } else {
          load4<BF16>(p.g[r], ev_at[v], lim, gv);
          if (EF) load4<false>(p.e[r], ev_at[v], lim, evv);
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) x[v][w] = EF ? fadd(gv[w], evv[w]) : gv[w];
      }
      if (kPrefetch && r + 1 < p.n) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          load4<BF16>(p.g[r + 1], ev_at[v], lim, ng[v]);
          if (EF) load4<false>(p.e[r + 1], ev_at[v], lim, ne[v]);
        }
      }
      const float s = group_scale<V>(x, gg.lanes);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float res[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float d = fmul(float(quant_code(x[v][w], s)), s);
          acc[v][w] = r == 0 ? d : fadd(acc[v][w], d);
          res[w] = __fsub_rn(x[v][w], d);
        }
        if (EF && live && ev_at[v] < p.count) store4<false>(p.e[r], ev_at[v], p.count, res);
      }
    }
    if (!live) continue;
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int w = 0; w < 4; ++w) acc[v][w] = fmul(acc[v][w], p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (ev_at[v] < p.count) store4<BF16>(p.out[r], ev_at[v], p.count, acc[v]);
  }
}

using Kern = void (*)(CompressParams);

template <bool BF16, bool EF>
Kern pick_compress(int V) {
  switch (V) {
    case 1: return compress_kernel<BF16, 1, EF>;
    case 2: return compress_kernel<BF16, 2, EF>;
    case 4: return compress_kernel<BF16, 4, EF>;
    default: return compress_kernel<BF16, 8, EF>;
  }
}

template <bool BF16, bool EF>
Kern pick_fused(int V) {
  switch (V) {
    case 1: return compressed_allreduce_kernel<BF16, 1, EF>;
    case 2: return compressed_allreduce_kernel<BF16, 2, EF>;
    case 4: return compressed_allreduce_kernel<BF16, 4, EF>;
    default: return compressed_allreduce_kernel<BF16, 8, EF>;
  }
}

cudaError_t launch(Kern k, int64_t tiles, const CompressParams& p, cudaStream_t stream) {
  if (tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(persistent_grid(reinterpret_cast<const void*>(k), tiles));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

// Groups of one CTA: 8 warps, each 32 / lanes groups.
int64_t groups_per_cta(int block) {
  const int lanes = block > 128 ? 32 : block / 4;
  return int64_t(kThreads / 32) * (32 / lanes);
}

int vectors_per_lane(int block) { return block > 128 ? block / 128 : 1; }

}  // namespace

cudaError_t launch_compress(const CompressParams& p, ar_dtype dtype, cudaStream_t stream) {
  const int V = vectors_per_lane(p.block);
  const bool bf = dtype == AR_BF16;
  const Kern k = bf ? (p.ef ? pick_compress<true, true>(V) : pick_compress<true, false>(V))
                    : (p.ef ? pick_compress<false, true>(V) : pick_compress<false, false>(V));
  const int64_t per = groups_per_cta(p.block);
  return launch(k, (p.n_blocks * p.n + per - 1) / per, p, stream);
}

cudaError_t launch_compressed_reduce(const CompressParams& p, ar_dtype out_dtype, cudaStream_t stream) {
  const Kern k = out_dtype == AR_BF16 ? compressed_reduce_kernel<true> : compressed_reduce_kernel<false>;
  const int64_t n16 = (p.count + 15) / 16;
  return launch(k, (n16 + kThreads - 1) / kThreads, p, stream);
}

cudaError_t launch_compressed_allreduce(const CompressParams& p, ar_dtype dtype, cudaStream_t stream) {
  const int V = vectors_per_lane(p.block);
  const bool bf = dtype == AR_BF16;
  const Kern k = bf ? (p.ef ? pick_fused<true, true>(V) : pick_fused<true, false>(V))
                    : (p.ef ? pick_fused<false, true>(V) : pick_fused<false, false>(V));
  const int64_t per = groups_per_cta(p.block);
  return launch(k, (p.n_blocks + per - 1) / per, p, stream);
}

}  // namespace ar
