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
// Kernels:
//  compress_kernel              g, e -> codes, scales, e'   (the message of every rank)
//  compress_packed_kernel       g -> codes, scales          (the same without feedback)
//  compressed_reduce_kernel     codes, scales -> out        (the receiving side)
//  compressed_allreduce_kernel  g, e -> e', out             (both in one pass; no message
//                                                            is materialised)
//  compressed_allreduce_bf16_packed_kernel  g -> out        (the same, bf16 without feedback,
//                                                            even rank counts)
//  compressed_allreduce_bf16_kernel  g -> out               (the same, odd rank counts)
//  compressed_allreduce_warp_kernel  g, e -> e', out        (the fused pass with one block
//                                                            per warp, for blocks that
//                                                            span warps; see "one block
//                                                            per warp")
// The kernels without feedback keep the loads of the ranks ahead in flight
// (pipelined loads, below); the packed ones decide codes with fewer
// instructions (see "bf16 without feedback, packed").
//
// Tiling: a CTA of 256 threads takes a tile of 256 * E consecutive elements,
// the same tile of every rank, E per thread (thread t: elements E*t..E*t+E-1;
// E = 8: one 16-byte bf16 vector or two fp32 vectors; E = 4: one 8-byte bf16
// or one 16-byte fp32 vector), ranks in order, NB ranks' values loaded before
// any of them is used. A quantisation block (a power of two from 16 to 1024
// elements) lies inside one tile: blocks of up to 32 * E elements are covered
// by block / E lanes of one warp and their maximum is a butterfly of shuffles
// among those lanes; larger blocks span block / (32 * E) warps, which combine
// their warp maxima through shared memory after one CTA barrier.
// Loops are uniform across the CTA, so every thread reaches every shuffle and
// barrier; elements past the end of the buffer read as 0 (they do not change a
// maximum) and are never stored.
//
// The code of an element is decided without a division in the common case:
// with a normal scale s, y = RN(x * r), with r = RN(1/s), or in the lean
// variant below the hardware's approximate reciprocal (at most one ulp off,
// 2^-23 relative), lies within 2^-15 of the correctly rounded quotient
// RN(x / s): |x / s| <= 127 + 2^-16, so |y - x / s| <= 127.01 * (2^-23 +
// 2^-24) < 2^-15.4 and |RN(x / s) - x / s| <= 2^-18. When every y of a thread
// is farther than 2^-12 from a half-integer, rint(y) equals rint(RN(x / s));
// otherwise (rarely: a quotient near a tie) the thread takes the correctly
// rounded quotient __fdiv_rn(x, s) itself, so ties are decided exactly as the
// definition says.
//
// The lean variant (kLean), for the kernels bound by instruction issue (the
// two without error feedback), spends fewer instructions per block and rank
// for the same results:
//  - the block maximum is one warp reduction instead of shuffle rounds;
//  - the scale s = RN(m / 127) is computed without a division: q0 = RN(m * c)
//    with c = RN(1/127) is within an ulp of the quotient, the remainder
//    m - q0 * 127 is exact in one FMA, and a second FMA, q0 + remainder * c,
//    rounds to the correctly rounded quotient (Markstein's theorem for
//    FMA-based division with a correctly rounded reciprocal); the library's
//    self-test checks it against the IEEE division for every non-negative
//    float;
//  - the screening product uses the approximate reciprocal.
// Measured at 16 ranks x 192 MiB, block 128 (fractions of each path's bytes):
// bf16 without feedback 0.61 -> 0.68 fused and 0.62 -> 0.66 in two calls;
// the kernels with feedback and the fp32 fused pass measured the same or up
// to 12 % slower with it, so they keep the IEEE operations and the shuffles.
// Codes are kept as integer-valued floats; a zero code is +0 (as an integer
// code converted to float is).
#include "common.cuh"

namespace ar {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kThreads / 32;

// Elements per thread per rank: 4 for fp32 (one 16-byte vector), 8 for bf16
// (one 16-byte vector). Measured on GB300 with 16 ranks of 192 MiB: fp32 at 8
// per thread needs 72 registers, fits 3 CTAs per SM and stalls on memory
// latency (0.89-0.93 of HBM); at 4 per thread it reaches 0.96-0.97. bf16 at 4
// per thread moves only 8 bytes per load and reaches 0.70 against 0.80.
template <bool BF16>
__host__ __device__ constexpr int ept() { return BF16 ? 8 : 4; }
// The compressor alone (two-call path) takes 16 bf16 elements per thread (two
// 16-byte vectors): its per-block work (scale, reciprocal, shuffles) is then
// shared by twice the elements. Measured with error feedback at 16 x 96 Mi
// bf16: the two calls at 0.91 of their bytes against 0.76 with 8 per thread.
// The fused pass keeps 8 (16 measured 0.75 against 0.81).
template <bool BF16>
__host__ __device__ constexpr int compress_ept() { return BF16 ? 16 : 4; }
// The reducer reads codes, not gradients: 8 (bf16 out) or 4 (fp32 out) per thread.
template <bool BF16>
__host__ __device__ constexpr int reduce_ept() { return BF16 ? 8 : 4; }

// kEPT consecutive elements starting at e (a multiple of kEPT) as fp32;
// elements at or past `lim` read as 0. The base is 16-byte aligned, so a whole
// group is whole 16-byte fp32 vectors, or one 8- or 16-byte bf16 vector.
template <bool BF16, int kEPT>
__device__ __forceinline__ void load_group(const void* base, int64_t e, int64_t lim, float (&f)[kEPT]) {
  if (e + kEPT <= lim) {
    if constexpr (BF16 && kEPT >= 8) {
#pragma unroll
      for (int h = 0; h < kEPT / 8; ++h) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e) + h);
        const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { f[8 * h + 2 * i] = bf16lo(v[i]); f[8 * h + 2 * i + 1] = bf16hi(v[i]); }
      }
    } else if constexpr (BF16) {
      const uint2 w = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e));
      f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    } else {
      const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
#pragma unroll
      for (int i = 0; i < kEPT / 4; ++i) {
        const float4 a = __ldcs(q + i);
        f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = a.z; f[4 * i + 3] = a.w;
      }
    }
  } else {
#pragma unroll
    for (int w = 0; w < kEPT; ++w) {
      f[w] = 0.0f;
      if (e + w < lim)
        f[w] = BF16 ? bf16_to_f32(static_cast<const uint16_t*>(base)[e + w]) : static_cast<const float*>(base)[e + w];
    }
  }
}

// kEPT consecutive elements starting at e (a multiple of kEPT) as raw words
// (bf16: two values per word, low half first); elements at or past `lim`
// read as +0. Loaded by the pipelined kernels ahead of use and widened only
// when used.
template <bool BF16, int kEPT>
struct RawGroup {
  static constexpr int kWords = BF16 ? kEPT / 2 : kEPT;
  static_assert(kWords % 4 == 0, "whole 16-byte vectors");
  uint4 v[kWords / 4];
};

template <bool BF16, int kEPT>
__device__ __forceinline__ void load_raw(const void* base, int64_t e, int64_t lim, RawGroup<BF16, kEPT>& g) {
  constexpr int kVecs = RawGroup<BF16, kEPT>::kWords / 4;
  const uint4* q = reinterpret_cast<const uint4*>(static_cast<const char*>(base) + e * (BF16 ? 2 : 4));
  if (e + kEPT <= lim) {
#pragma unroll
    for (int i = 0; i < kVecs; ++i) g.v[i] = __ldcs(q + i);
    return;
  }
  uint32_t u[4 * kVecs];
#pragma unroll
  for (int i = 0; i < 4 * kVecs; ++i) u[i] = 0u;
#pragma unroll
  for (int i = 0; i < kEPT; ++i) {
    if (e + i >= lim) continue;
    if (BF16)
      u[i / 2] |= uint32_t(static_cast<const uint16_t*>(base)[e + i]) << (16 * (i & 1));
    else
      u[i] = static_cast<const uint32_t*>(base)[e + i];
  }
#pragma unroll
  for (int i = 0; i < kVecs; ++i) g.v[i] = make_uint4(u[4 * i], u[4 * i + 1], u[4 * i + 2], u[4 * i + 3]);
}

template <bool BF16, int kEPT>
__device__ __forceinline__ void widen_raw(const RawGroup<BF16, kEPT>& g, float (&f)[kEPT]) {
#pragma unroll
  for (int i = 0; i < RawGroup<BF16, kEPT>::kWords / 4; ++i) {
    const uint32_t u[4] = {g.v[i].x, g.v[i].y, g.v[i].z, g.v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (BF16) {
        f[8 * i + 2 * j] = bf16lo(u[j]);
        f[8 * i + 2 * j + 1] = bf16hi(u[j]);
      } else {
        f[4 * i + j] = __uint_as_float(u[j]);
      }
    }
  }
}

// Store kEPT consecutive elements at e (bf16: rounded to nearest even);
// elements at or past `count` are not written.
template <bool BF16, int kEPT>
__device__ __forceinline__ void store_group(void* base, int64_t e, int64_t count, const float (&f)[kEPT]) {
  if (e + kEPT <= count) {
    if constexpr (BF16 && kEPT >= 8) {
#pragma unroll
      for (int h = 0; h < kEPT / 8; ++h)
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + e) + h,
               make_uint4(pack_bf16x2(f[8 * h], f[8 * h + 1]), pack_bf16x2(f[8 * h + 2], f[8 * h + 3]),
                          pack_bf16x2(f[8 * h + 4], f[8 * h + 5]), pack_bf16x2(f[8 * h + 6], f[8 * h + 7])));
    } else if constexpr (BF16) {
      __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + e),
             make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3])));
    } else {
      float4* q = reinterpret_cast<float4*>(static_cast<float*>(base) + e);
#pragma unroll
      for (int i = 0; i < kEPT / 4; ++i) __stcs(q + i, make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]));
    }
  } else {
#pragma unroll
    for (int w = 0; w < kEPT; ++w) {
      if (e + w >= count) continue;
      if (BF16)
        static_cast<uint16_t*>(base)[e + w] = f32_to_bf16(f[w]);
      else
        static_cast<float*>(base)[e + w] = f[w];
    }
  }
}

// RN(m / 127) without a division (the lean variant; see the file comment);
// +inf and NaN pass through as the division would give them.
__device__ __forceinline__ float div127(float m) {
  constexpr float kInv127 = 1.0f / 127.0f;  // RN(1/127) = 0x1.020408p-7
  static_assert(kInv127 == 0x1.020408p-7f, "correctly rounded reciprocal of 127");
  const float q0 = __fmul_rn(m, kInv127);
  const float rem = __fmaf_rn(-q0, 127.0f, m);  // exact
  const float q1 = __fmaf_rn(rem, kInv127, q0);
  return q0 < __int_as_float(0x7f800000) ? q1 : q0;
}

// The hardware's approximate reciprocal (at most one ulp off); s is normal
// here, so neither s nor 1/s is subnormal.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Barrier over the W warps (a power of two, W <= kWarps) that hold one block:
// named barrier 1 + warp / W of W * 32 threads, the whole CTA when W = kWarps.
// The warps of other blocks in the CTA do not wait.
__device__ __forceinline__ void block_group_sync(int W) {
  if (W >= kWarps) {
    __syncthreads();
    return;
  }
  asm volatile("bar.sync %0, %1;" ::"r"(1 + (int(threadIdx.x) >> 5) / W), "r"(W * 32) : "memory");
}

// The block's scale s = max|x| / 127 for this thread's kEPT values.
// `wmax` is this call's shared-memory slot; callers alternate two slots, so
// one barrier per call suffices (a warp that writes the next call's slot has
// passed this call's barrier, after every warp finished reading the slot of
// the call before).
// The maximum over the block's lanes of one warp is a butterfly of shuffles,
// or with kLean, for blocks of 16 or 32 lanes, full-warp reductions: m is a
// non-negative float (fmaxf drops NaN), and non-negative floats order as
// their bit patterns do, so an unsigned maximum of the bits is the float
// maximum. A 16-lane block takes two reductions over the whole warp, the other
// half-warp contributing 0: a reduction whose mask differs between the lanes
// of one warp measured about one pass per distinct mask.
template <int kEPT, bool kLean = false>
__device__ __forceinline__ float block_scale(const float (&x)[kEPT], int block, float* wmax) {
  float m = 0.0f;
#pragma unroll
  for (int w = 0; w < kEPT; ++w) m = fmaxf(m, fabsf(x[w]));
  constexpr int kWarpElems = 32 * kEPT;
  const int lanes = block < kWarpElems ? block / kEPT : 32;
  if (kLean && lanes == 32) {
    m = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(m)));
  } else if (kLean && lanes == 16) {  // one full-warp reduction per half-warp (see below)
    const bool low = (threadIdx.x & 16) == 0;
    const unsigned a = __reduce_max_sync(kFull, low ? __float_as_uint(m) : 0u);
    const unsigned b = __reduce_max_sync(kFull, low ? 0u : __float_as_uint(m));
    m = __uint_as_float(low ? a : b);
  } else {
    for (int o = lanes >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  }
  if (block > kWarpElems) {
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) wmax[warp] = m;
    __syncthreads();
    const int W = block / kWarpElems;
    const int w0 = warp & ~(W - 1);
    m = wmax[w0];
    for (int i = 1; i < W; ++i) m = fmaxf(m, wmax[w0 + i]);
  }
  return kLean ? div127(m) : __fdiv_rn(m, 127.0f);
}

// The scales of the NB ranks of a load batch (the first nb of them real),
// with block_scale's arithmetic. For blocks that span warps, the warps'
// maxima of all NB ranks go to shared memory together and one barrier serves
// the batch instead of one per rank (wm: the batch's slot of NB x kWarps
// floats; callers alternate two slots, as for block_scale). kGroupSync: the
// barrier holds only the block's own warps (the fused pass, fp32 block 512:
// 0.986 of its bytes against 0.964; the compressor measured 1 % slower).
template <int kEPT, int NB, bool kGroupSync = false>
__device__ __forceinline__ void batch_scales(const float (&x)[NB][kEPT], int nb, int block, float* wm,
                                             float (&s)[NB]) {
  constexpr int kWarpElems = 32 * kEPT;
  const int lanes = block < kWarpElems ? block / kEPT : 32;
  float m[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    m[b] = 0.0f;
    if (b < nb) {
#pragma unroll
      for (int w = 0; w < kEPT; ++w) m[b] = fmaxf(m[b], fabsf(x[b][w]));
    }
    for (int o = lanes >> 1; o > 0; o >>= 1) m[b] = fmaxf(m[b], __shfl_xor_sync(kFull, m[b], o));
  }
  if (block > kWarpElems) {
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) wm[b * kWarps + warp] = m[b];
    }
    const int W = block / kWarpElems;
    if (kGroupSync)
      block_group_sync(W);
    else
      __syncthreads();
    const int w0 = warp & ~(W - 1);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      m[b] = wm[b * kWarps + w0];
      for (int i = 1; i < W; ++i) m[b] = fmaxf(m[b], wm[b * kWarps + w0 + i]);
    }
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) s[b] = __fdiv_rn(m[b], 127.0f);
}

// Element-wise fp32 arithmetic, one IEEE operation per element rounded to
// nearest even and never contracted into an FMA (the definition rounds every
// product before it is summed).
template <int n>
__device__ __forceinline__ void mul_each(float (&d)[n], const float (&a)[n], float b) {
#pragma unroll
  for (int w = 0; w < n; ++w) d[w] = __fmul_rn(a[w], b);
}
template <int n>
__device__ __forceinline__ void add_each(float (&d)[n], const float (&a)[n], const float (&b)[n]) {
#pragma unroll
  for (int w = 0; w < n; ++w) d[w] = __fadd_rn(a[w], b[w]);
}
template <int n>
__device__ __forceinline__ void sub_each(float (&d)[n], const float (&a)[n], const float (&b)[n]) {
#pragma unroll
  for (int w = 0; w < n; ++w) d[w] = __fsub_rn(a[w], b[w]);
}

// The nearest integer to y (ties to even) as a float, for |y| < 2^22, by the
// classic rounding-to-integer addition: y + 1.5 * 2^23 lands in a binade whose
// spacing is 1, so the sum is rounded to an integer (nearest, ties to even),
// and subtracting 1.5 * 2^23 back is exact. Two full-rate adds, and a zero
// result is +0 (as an integer code converted to float is), never -0.
__device__ __forceinline__ float round_int(float y) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  return __fsub_rn(__fadd_rn(y, kMagic), kMagic);
}

// The codes of this thread's values in a block of scale s, as integer-valued
// floats: the nearest integer to RN(x / s) (ties to even), clamped to
// [-127, 127]; all 0 when s is 0. See the file comment for the screening.
// Every quotient here is below 255 in magnitude (a subnormal scale loses at
// most half its value to rounding), well inside round_int's range.
template <int kEPT, bool kLean = false>
__device__ __forceinline__ void quant_group(const float (&x)[kEPT], float s, float (&c)[kEPT]) {
  if (s >= 0x1p-126f) {
    float y[kEPT], dev[kEPT];
    mul_each(y, x, kLean ? rcp_approx(s) : __frcp_rn(s));
#pragma unroll
    for (int w = 0; w < kEPT; ++w) c[w] = round_int(y[w]);
    sub_each(dev, y, c);  // exact: y and its nearest integer are within a factor of 2 (or c = 0)
    float worst = 0.0f;
#pragma unroll
    for (int w = 0; w < kEPT; ++w) worst = fmaxf(worst, fabsf(dev[w]));
    if (worst >= 0.5f - 0x1p-12f) {  // a quotient near a tie: the exact quotient decides
#pragma unroll
      for (int w = 0; w < kEPT; ++w) c[w] = round_int(__fdiv_rn(x[w], s));
    }
    // |x / s| < 127.5 for a normal s, so no clamp is needed here
  } else if (s > 0.0f) {  // a subnormal scale: exact quotients, clamped
#pragma unroll
    for (int w = 0; w < kEPT; ++w) c[w] = fminf(fmaxf(round_int(__fdiv_rn(x[w], s)), -127.0f), 127.0f);
  } else {
#pragma unroll
    for (int w = 0; w < kEPT; ++w) c[w] = 0.0f;
  }
}

// Four integer-valued codes in [-127, 127] (c[i..i+3]) as four
// two's-complement bytes of one word.
template <int kEPT>
__device__ __forceinline__ uint32_t pack_codes4(const float (&c)[kEPT], int i) {
  return (uint32_t(int(c[i])) & 0xFFu) | ((uint32_t(int(c[i + 1])) & 0xFFu) << 8) |
         ((uint32_t(int(c[i + 2])) & 0xFFu) << 16) | ((uint32_t(int(c[i + 3])) & 0xFFu) << 24);
}

// Code j (a two's-complement byte) of a word of four codes as a float, with
// full-rate integer and add instructions: flipping the sign bit gives c + 128
// in 0..255, placed as the low byte under the exponent of 2^23 it is the float
// 2^23 + 128 + c exactly, and subtracting 2^23 + 128 leaves c exactly.
__device__ __forceinline__ float code_of(uint32_t word, int j) {
  const uint32_t biased = __byte_perm(word ^ 0x80808080u, 0x4B000000u, 0x7540u | uint32_t(j));
  return __fsub_rn(__uint_as_float(biased), 8388736.0f);  // 2^23 + 128
}

// ---------------------------------------------------------------- pipelined loads
// Without error feedback a rank's slice is only 2 or 4 bytes per element, so
// a thread that loads one rank and then works on it has little in flight.
// The pipelined kernels keep the raw words of the next kAhead (tile, rank)
// pairs in flight while they work on the current one. A CTA visits the pairs
// in a fixed order: tiles blockIdx.x, + gridDim.x, ...; ranks 0..n-1 within
// each tile. Measured on GB300 at 16 ranks x 96 Mi bf16, block 128 (fused
// pass): 0.615 of its bytes with 2 ahead, 0.611 with 1, 0.595 with 3, 0.586
// with 4, against 0.54 for the load-then-quantise loop. A bulk L2 prefetch of
// the tiles ahead, one thread per CTA, reached 0.596 there and cost 7-25 % on
// the paths that already have enough in flight (fp32, error feedback), so it
// is not used.
constexpr int kAhead = 2;

// Load the gradient words of the pair k positions after (tile, r) into w
// (+0 past the last tile).
template <bool BF16, int kEPT>
__device__ __forceinline__ void fetch_ahead(const CompressParams& p, int64_t n_tiles, int64_t lane_off, int64_t tile,
                                            int r, int k, RawGroup<BF16, kEPT>& w) {
  constexpr int64_t kTileElems = int64_t(kEPT) * kThreads;
  r += k;
  while (r >= p.n) {
    r -= p.n;
    tile += gridDim.x;
  }
  if (tile < n_tiles) {
    load_raw<BF16, kEPT>(p.g[r], tile * kTileElems + lane_off, p.count, w);
  } else {
#pragma unroll
    for (int i = 0; i < RawGroup<BF16, kEPT>::kWords / 4; ++i) w.v[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------- compress
// kEPT codes at e, one byte each; codes at or past `count` are not written.
template <int kEPT>
__device__ __forceinline__ void store_codes(int8_t* q, int64_t e, int64_t count, const float (&c)[kEPT]) {
  if (e + kEPT <= count) {
    if constexpr (kEPT == 16)
      __stcs(reinterpret_cast<uint4*>(q + e), make_uint4(pack_codes4<kEPT>(c, 0), pack_codes4<kEPT>(c, 4),
                                                         pack_codes4<kEPT>(c, 8), pack_codes4<kEPT>(c, 12)));
    else if constexpr (kEPT == 8)
      __stcs(reinterpret_cast<uint2*>(q + e), make_uint2(pack_codes4<kEPT>(c, 0), pack_codes4<kEPT>(c, 4)));
    else
      __stcs(reinterpret_cast<unsigned int*>(q + e), pack_codes4<kEPT>(c, 0));
  } else {
#pragma unroll
    for (int w = 0; w < kEPT; ++w)
      if (e + w < count) q[e + w] = static_cast<int8_t>(int(c[w]));
  }
}

// Each tile of every rank: codes (kEPT bytes per thread), the scale of each block
// (written by the block's first thread) and, with error feedback, the new
// residual.
// NB: ranks per load batch (fp32: 4, 1 or 2 measured slower). kBatch (fp32
// blocks that span warps): the batch's scales from batch_scales, one barrier
// per batch; block 1024 at 16 x 192 MiB, the two calls with error feedback
// measured 0.941 of their bytes against 0.899.
template <bool BF16, bool EF, int NB, bool kBatch>
__global__ void __launch_bounds__(kThreads) compress_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kEPT = compress_ept<BF16>();
  constexpr int kTileElems = kEPT * kThreads;
  __shared__ float wmax[2][NB * kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  const int shift = __ffs(p.block) - 1;  // block is a power of two
  int phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e = tile * kTileElems + int64_t(kEPT) * threadIdx.x;
#pragma unroll 1
    for (int r0 = 0; r0 < p.n; r0 += NB) {
      const int nb = p.n - r0 < NB ? p.n - r0 : NB;  // uniform across the CTA
      float x[NB][kEPT], xe[NB][kEPT];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) continue;
        load_group<BF16, kEPT>(p.g[r0 + b], e, p.count, x[b]);
        if (EF) load_group<false, kEPT>(p.e[r0 + b], e, p.count, xe[b]);
      }
      if (EF) {
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b < nb) add_each(x[b], x[b], xe[b]);
      }
      float s[NB];
      if constexpr (kBatch) {
        batch_scales<kEPT, NB>(x, nb, p.block, wmax[phase], s);
        phase ^= 1;
      } else {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b >= nb) continue;
          s[b] = block_scale<kEPT>(x[b], p.block, wmax[phase]);
          phase ^= 1;
        }
      }
      if (e >= p.count) continue;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) continue;
        const int r = r0 + b;
        float c[kEPT];
        if ((e & (p.block - 1)) == 0) p.s[r][e >> shift] = s[b];
        quant_group<kEPT>(x[b], s[b], c);
        store_codes<kEPT>(p.q[r], e, p.count, c);
        if (EF) {
          float d[kEPT], res[kEPT];
          mul_each(d, c, s[b]);
          sub_each(res, x[b], d);
          store_group<false, kEPT>(p.e[r], e, p.count, res);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- reduce
// The receiving side: for each tile, every rank's codes (kEPT bytes per thread)
// and the scale of the thread's block are loaded NB ranks at a time, the
// reconstructions summed in rank order, scaled once, and the result written to
// every rank.
template <bool BF16OUT>
__global__ void __launch_bounds__(kThreads) compressed_reduce_kernel(const __grid_constant__ CompressParams p) {
  constexpr int NB = 8;
  constexpr int kEPT = reduce_ept<BF16OUT>();
  constexpr int kTileElems = kEPT * kThreads;
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  const int shift = __ffs(p.block) - 1;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e = tile * kTileElems + int64_t(kEPT) * threadIdx.x;
    if (e >= p.count) continue;
    const int64_t kb = e >> shift;
    const bool whole = e + kEPT <= p.count;
    float acc[kEPT];
#pragma unroll 1
    for (int r0 = 0; r0 < p.n; r0 += NB) {
      uint2 c[NB];
      float s[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (r0 + b >= p.n) continue;
        const int8_t* q = p.q[r0 + b];
        if (whole) {
          if constexpr (kEPT == 8)
            c[b] = __ldcs(reinterpret_cast<const uint2*>(q + e));
          else
            c[b] = make_uint2(__ldcs(reinterpret_cast<const unsigned int*>(q + e)), 0u);
        } else {  // the ragged end: bytes past count read as code 0 and are never stored
          uint32_t lo = 0, hi = 0;
          for (int w = 0; w < kEPT; ++w)
            if (e + w < p.count) {
              const uint32_t v = uint32_t(static_cast<uint8_t>(q[e + w]));
              if (w < 4) lo |= v << (8 * w); else hi |= v << (8 * (w - 4));
            }
          c[b] = make_uint2(lo, hi);
        }
        s[b] = __ldg(p.s[r0 + b] + kb);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (r0 + b >= p.n) continue;
        float q[kEPT], d[kEPT];
#pragma unroll
        for (int w = 0; w < kEPT; ++w) q[w] = code_of(w < 4 ? c[b].x : c[b].y, w & 3);
        mul_each(d, q, s[b]);
        if (r0 + b == 0) {
#pragma unroll
          for (int w = 0; w < kEPT; ++w) acc[w] = d[w];
        } else {
          add_each(acc, acc, d);
        }
      }
    }
    mul_each(acc, acc, p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) store_group<BF16OUT, kEPT>(p.out[r], e, p.count, acc);
  }
}

// ---------------------------------------------------------------- fused
// One rank's step of the fused pass for this thread's values x: quantise the
// block, add the reconstruction d to the running sum (acc = d for rank 0)
// and, with error feedback, return the residual x - d.
template <int kEPT, bool EF, bool kLean = false>
__device__ __forceinline__ void fold_scaled(const float (&x)[kEPT], int r, float s, float (&acc)[kEPT],
                                            float (&res)[kEPT]) {
  float c[kEPT], d[kEPT];
  quant_group<kEPT, kLean>(x, s, c);
  mul_each(d, c, s);
  if (r == 0) {
#pragma unroll
    for (int w = 0; w < kEPT; ++w) acc[w] = d[w];
  } else {
    add_each(acc, acc, d);
  }
  if (EF) sub_each(res, x, d);
}

template <int kEPT, bool EF, bool kLean = false>
__device__ __forceinline__ void fold_rank(const float (&x)[kEPT], int r, int block, float* wmax, float (&acc)[kEPT],
                                          float (&res)[kEPT]) {
  float c[kEPT], d[kEPT];
  const float s = block_scale<kEPT, kLean>(x, block, wmax);
  quant_group<kEPT, kLean>(x, s, c);
  mul_each(d, c, s);
  if (r == 0) {
#pragma unroll
    for (int w = 0; w < kEPT; ++w) acc[w] = d[w];
  } else {
    add_each(acc, acc, d);
  }
  if (EF) sub_each(res, x, d);
}

// bf16 without error feedback: 2 bytes in and 2 out per element and rank,
// with the pipelined loads above.

__global__ void __launch_bounds__(kThreads) compressed_allreduce_bf16_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kEPT = 8;
  constexpr int kTileElems = kEPT * kThreads;
  __shared__ float wmax[2][kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  const int64_t lane_off = int64_t(kEPT) * threadIdx.x;
  using Raw = RawGroup<true, kEPT>;
  auto fetch = [&](int64_t tile, int r, int k, Raw& w) { fetch_ahead<true, kEPT>(p, n_tiles, lane_off, tile, r, k, w); };
  Raw ring[kAhead];
#pragma unroll
  for (int k = 0; k < kAhead; ++k) fetch(blockIdx.x, 0, k, ring[k]);
  int phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e = tile * kTileElems + lane_off;
    float acc[kEPT];
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) {
      const Raw w = ring[0];
#pragma unroll
      for (int k = 0; k + 1 < kAhead; ++k) ring[k] = ring[k + 1];
      fetch(tile, r, kAhead, ring[kAhead - 1]);
      float x[kEPT], res[kEPT];
      widen_raw<true, kEPT>(w, x);
      fold_rank<kEPT, false, true>(x, r, p.block, wmax[phase], acc, res);
      phase ^= 1;
    }
    if (e >= p.count) continue;
    mul_each(acc, acc, p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) store_group<true, kEPT>(p.out[r], e, p.count, acc);
  }
}

// ---------------------------------------------------------------- bf16 without feedback, packed
// The kernel above spends about 30 instructions per element and rank; with 2
// bytes in and 2 out that bounds it by instruction issue (0.68 of its bytes at
// 16 ranks x 96 Mi). This variant decides the same codes with fewer:
//  - the block size is a template parameter, so the lanes of one block and
//    their reduction mask are constants;
//  - the code is RN(x * rc + 1.5 * 2^23) - 1.5 * 2^23 (rc the approximate
//    reciprocal of s): the sum lands in the binade [2^23, 2^24), whose
//    spacing is 1, so one FMA rounds the exact product x * rc to the nearest
//    integer (ties to even, 1.5 * 2^23 being even) and the subtraction is
//    exact. The screening deviation is one more FMA, RN(x * rc - c), the
//    exact product's distance from its code. With |rc - 1/s| <= 2^-23 / s,
//    |x * rc - x / s| <= 127.5 * 2^-23 < 2^-16, and RN(x / s) is within 2^-18
//    of x / s; so when every |RN(x * rc - c)| is below 1/2 - 2^-14, c is the
//    one integer within 1/2 of RN(x / s), which is the code the definition
//    takes. Otherwise the element takes the correctly rounded quotient.
//  - element pairs go through Blackwell's packed fp32x2 FMA, add and multiply
//    (one instruction for two lanes of arithmetic, each lane an IEEE fp32
//    operation rounded to nearest even). The reconstruction d = RN(c * s) is
//    a packed FMA with +0: c * s is never -0 here (c is +0 or a nonzero
//    integer, s a normal), so it equals the rounded product bit for bit, and
//    an FMA is never merged with the add that follows it;
//  - the block maximum and the screening maximum take three operands per
//    instruction;
//  - the rank loop is unrolled by two over two load buffers: each buffer is
//    refilled, two (tile, rank) pairs ahead, as soon as its words are
//    widened, so no registers are copied to keep the pipeline going.
// Ranks come in pairs, so the rank count is even; the tile of the ragged end
// is folded by the generic per-rank path above (the same bits).

// Two fp32 values as the 64-bit operand of a packed instruction (lo first).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(|a|, |b|, |c|) in one instruction.
__device__ __forceinline__ float max3abs(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Pairs of one thread's 8 elements of one rank.
struct Pairs8 {
  uint64_t v[4];
};

// Fold rank `r`'s words w (8 bf16, widened here) into the running sum.
// kFirst: acc = d (rank 0). wm: this call's shared-memory slot for blocks
// that span warps (callers alternate two slots).
template <int kBlock, bool kFirst>
__device__ __forceinline__ void lean_bf16_rank(const float (&x)[8], float* wm, Pairs8& acc) {
  constexpr int kLanes = kBlock >= 32 * 8 ? 32 : kBlock / 8;  // lanes of one block within a warp
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  constexpr float kTie = 0.5f - 0x1p-14f;
  float m = max3abs(x[0], x[1], x[2]);
  m = max3abs(m, x[3], x[4]);
  m = max3abs(m, x[5], x[6]);
  m = fmaxf(m, fabsf(x[7]));
  // The maximum over the block's lanes. m is non-negative, and non-negative
  // floats order as their bits do, so a warp reduction of the bits (unsigned
  // maximum) is the float maximum. A reduction whose mask differs between the
  // lanes of one warp ran about once per distinct mask (block 16 slower than
  // shuffles, block 128 barely faster), so only full-warp reductions are
  // used: one for blocks of 32 or more lanes, two (one per half-warp, the
  // other half contributing 0) for 16 lanes, and shuffle rounds below that.
  if constexpr (kLanes == 32) {
    m = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(m)));
  } else if constexpr (kLanes == 16) {
    const bool low = (threadIdx.x & 16) == 0;
    const unsigned a = __reduce_max_sync(kFull, low ? __float_as_uint(m) : 0u);
    const unsigned b = __reduce_max_sync(kFull, low ? 0u : __float_as_uint(m));
    m = __uint_as_float(low ? a : b);
  } else {
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  }
  if constexpr (kBlock > 32 * 8) {  // the block's own warps wait, not the CTA's (block 512: 0.965
    constexpr int W = kBlock / (32 * 8);  // of its bytes against 0.870 with a CTA barrier, 1024: 0.927
    const int warp = threadIdx.x >> 5;     // against 0.874)
    if ((threadIdx.x & 31) == 0) wm[warp] = m;
    block_group_sync(W);
    const int w0 = warp & ~(W - 1);
    m = wm[w0];
#pragma unroll
    for (int i = 1; i < W; ++i) m = fmaxf(m, wm[w0 + i]);
  }
  const float s = div127(m);
  float c[8];
  if (s >= 0x1p-126f) {
    const float rc = rcp_approx(s);
    const uint64_t RC = pk2(rc, rc), MM = pk2(kMagic, kMagic);
    float worst = 0.0f, dv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t X = pk2(x[2 * i], x[2 * i + 1]);
      const uint64_t Y = fma2(X, RC, MM);  // M + the nearest integer to x * rc
      const uint64_t C = sub2(Y, MM);      // exact
      const uint64_t D = fma2(X, RC, sub2(MM, Y));  // RN(x * rc - c)
      upk2(C, c[2 * i], c[2 * i + 1]);
      upk2(D, dv[2 * i], dv[2 * i + 1]);
      worst = max3abs(worst, dv[2 * i], dv[2 * i + 1]);
    }
    if (worst >= kTie) {  // a quotient near a tie: the correctly rounded quotient decides
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (fabsf(dv[w]) >= kTie) c[w] = round_int(__fdiv_rn(x[w], s));
    }
    // |x / s| < 127.5 for a normal s, so no clamp is needed here
  } else if (s > 0.0f) {  // a subnormal scale: exact quotients, clamped
#pragma unroll
    for (int w = 0; w < 8; ++w) c[w] = fminf(fmaxf(round_int(__fdiv_rn(x[w], s)), -127.0f), 127.0f);
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) c[w] = 0.0f;
  }
  const uint64_t S2 = pk2(s, s), Z2 = pk2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t D = fma2(pk2(c[2 * i], c[2 * i + 1]), S2, Z2);  // RN(c * s), see above
    acc.v[i] = kFirst ? D : add2(acc.v[i], D);
  }
}

__device__ __forceinline__ void widen8(const uint4& w, float (&x)[8]) {
  x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
  x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
}

template <int kLogBlock>
__global__ void __launch_bounds__(kThreads) compressed_allreduce_bf16_packed_kernel(
    const __grid_constant__ CompressParams p) {
  constexpr int kEPT = 8;
  constexpr int kTileElems = kEPT * kThreads;
  constexpr int kBlock = 1 << kLogBlock;
  __shared__ float wmax[2][kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;  // even
  const int64_t n_full = p.count / kTileElems;
  const int64_t lane_off = int64_t(kEPT) * threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * kTileElems;
  // the fetch cursor: the (tile, rank) pair the next load is for, two pairs
  // ahead of the one being folded
  int64_t f_off = int64_t(blockIdx.x) * kTileElems + lane_off;
  int f_r = 0;
  const int64_t f_end = n_full * kTileElems;
  auto fetch = [&](uint4& w) {
    if (f_off < f_end) w = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.g[f_r]) + f_off));
    if (++f_r == n) {
      f_r = 0;
      f_off += stride;
    }
  };
  uint4 X0 = make_uint4(0u, 0u, 0u, 0u), X1 = X0;
  fetch(X0);
  fetch(X1);
  int phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_full; tile += gridDim.x) {
    Pairs8 acc;
    float x[8];
    widen8(X0, x);
    fetch(X0);
    lean_bf16_rank<kBlock, true>(x, wmax[phase], acc);
    phase ^= 1;
    widen8(X1, x);
    fetch(X1);
    lean_bf16_rank<kBlock, false>(x, wmax[phase], acc);
    phase ^= 1;
#pragma unroll 1
    for (int r = 2; r < n; r += 2) {
      widen8(X0, x);
      fetch(X0);
      lean_bf16_rank<kBlock, false>(x, wmax[phase], acc);
      phase ^= 1;
      widen8(X1, x);
      fetch(X1);
      lean_bf16_rank<kBlock, false>(x, wmax[phase], acc);
      phase ^= 1;
    }
    const uint64_t SC = pk2(p.scale, p.scale);
    float a[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) upk2(mul2(acc.v[i], SC), a[2 * i], a[2 * i + 1]);
    const uint4 out = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                                 pack_bf16x2(a[6], a[7]));
    const int64_t e = tile * kTileElems + lane_off;
#pragma unroll 1
    for (int r = 0; r < n; ++r) __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out[r]) + e), out);
  }
  // the ragged end: one partial tile, folded by the last CTA with bounds
  if (blockIdx.x == gridDim.x - 1 && n_full * kTileElems < p.count) {
    const int64_t e = n_full * kTileElems + lane_off;
    float acc[kEPT];
#pragma unroll 1
    for (int r = 0; r < n; ++r) {
      float x[kEPT], res[kEPT];
      load_group<true, kEPT>(p.g[r], e, p.count, x);
      fold_rank<kEPT, false, true>(x, r, kBlock, wmax[phase], acc, res);
      phase ^= 1;
    }
    if (e < p.count) {
      mul_each(acc, acc, p.scale);
#pragma unroll 1
      for (int r = 0; r < n; ++r) store_group<true, kEPT>(p.out[r], e, p.count, acc);
    }
  }
}

// ---------------------------------------------------------------- compressor without feedback, packed
// The message of every rank (codes, one byte each, and the block scales) with
// the packed kernel's arithmetic, for either input type and any rank count:
// the sum RN(x * rc + 1.5 * 2^23) is 1.5 * 2^23 + c, whose bit pattern is
// that of 1.5 * 2^23 (low byte 0) plus c, so the code's two's-complement
// byte is the sum's low byte; four codes pack into a word with three byte
// permutes instead of four float-to-integer conversions. The (tile, rank)
// pairs of a CTA are walked with a fetch cursor two pairs ahead of the one
// being quantised, over two load buffers.

// The message of one pair: x holds the 8 values at element e of rank r.
// kGroupSync: blocks that span warps wait on a barrier of their own warps
// only (the bf16 compressor: block 1024 0.813 of its bytes against 0.797
// with a CTA barrier; fp32 measured 0.83 against 0.94 and keeps the CTA
// barrier).
template <int kLogBlock, bool kGroupSync>
__device__ __forceinline__ void packed_message(const float (&x)[8], float* wm, int8_t* q, float* sc, int64_t e) {
  constexpr int kBlock = 1 << kLogBlock;
  constexpr int kLanes = kBlock >= 32 * 8 ? 32 : kBlock / 8;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  constexpr float kTie = 0.5f - 0x1p-14f;
  float m = max3abs(x[0], x[1], x[2]);
  m = max3abs(m, x[3], x[4]);
  m = max3abs(m, x[5], x[6]);
  m = fmaxf(m, fabsf(x[7]));
  if constexpr (kLanes == 32) {  // full-warp reductions only (see the fused kernel)
    m = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(m)));
  } else if constexpr (kLanes == 16) {
    const bool low = (threadIdx.x & 16) == 0;
    const unsigned a = __reduce_max_sync(kFull, low ? __float_as_uint(m) : 0u);
    const unsigned b = __reduce_max_sync(kFull, low ? 0u : __float_as_uint(m));
    m = __uint_as_float(low ? a : b);
  } else {
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  }
  if constexpr (kBlock > 32 * 8) {
    constexpr int W = kBlock / (32 * 8);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) wm[warp] = m;
    if (kGroupSync)
      block_group_sync(W);
    else
      __syncthreads();
    const int w0 = warp & ~(W - 1);
    m = wm[w0];
#pragma unroll
    for (int i = 1; i < W; ++i) m = fmaxf(m, wm[w0 + i]);
  }
  const float s = div127(m);
  uint32_t yb[8];  // bits of 1.5 * 2^23 + code
  if (s >= 0x1p-126f) {
    const float rc = rcp_approx(s);
    const uint64_t RC = pk2(rc, rc), MM = pk2(kMagic, kMagic);
    float worst = 0.0f, dv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t X = pk2(x[2 * i], x[2 * i + 1]);
      const uint64_t Y = fma2(X, RC, MM);           // 1.5 * 2^23 + the nearest integer to x * rc
      const uint64_t D = fma2(X, RC, sub2(MM, Y));  // RN(x * rc - c)
      float ylo, yhi;
      upk2(Y, ylo, yhi);
      yb[2 * i] = __float_as_uint(ylo);
      yb[2 * i + 1] = __float_as_uint(yhi);
      upk2(D, dv[2 * i], dv[2 * i + 1]);
      worst = max3abs(worst, dv[2 * i], dv[2 * i + 1]);
    }
    if (worst >= kTie) {  // a quotient near a tie: the correctly rounded quotient decides
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (fabsf(dv[w]) >= kTie) yb[w] = __float_as_uint(__fadd_rn(round_int(__fdiv_rn(x[w], s)), kMagic));
    }
  } else if (s > 0.0f) {  // a subnormal scale: exact quotients, clamped
#pragma unroll
    for (int w = 0; w < 8; ++w)
      yb[w] = __float_as_uint(__fadd_rn(fminf(fmaxf(round_int(__fdiv_rn(x[w], s)), -127.0f), 127.0f), kMagic));
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) yb[w] = __float_as_uint(kMagic);
  }
  // low bytes of the 8 words, in element order
  const uint32_t lo = __byte_perm(__byte_perm(yb[0], yb[1], 0x0040), __byte_perm(yb[2], yb[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(yb[4], yb[5], 0x0040), __byte_perm(yb[6], yb[7], 0x0040), 0x5410);
  __stcs(reinterpret_cast<uint2*>(q + e), make_uint2(lo, hi));
  if ((e & (kBlock - 1)) == 0) sc[e >> kLogBlock] = s;
}

template <bool BF16, int kLogBlock>
__global__ void __launch_bounds__(kThreads) compress_packed_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kEPT = 8;
  constexpr int kTileElems = kEPT * kThreads;
  constexpr int kBlock = 1 << kLogBlock;
  using Raw = RawGroup<BF16, kEPT>;
  __shared__ float wmax[2][kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int n = p.n;
  const int64_t n_full = p.count / kTileElems;
  const int64_t lane_off = int64_t(kEPT) * threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * kTileElems;
  const int64_t end = n_full * kTileElems;
  // fetch and quantise cursors: element offset and rank of the next pair
  int64_t f_off = int64_t(blockIdx.x) * kTileElems + lane_off, c_off = f_off;
  int f_r = 0, c_r = 0;
  auto fetch = [&](Raw& w) {
    if (f_off < end) load_raw<BF16, kEPT>(p.g[f_r], f_off, p.count, w);
    if (++f_r == n) {
      f_r = 0;
      f_off += stride;
    }
  };
  Raw X0, X1;
#pragma unroll
  for (int i = 0; i < Raw::kWords / 4; ++i) X0.v[i] = X1.v[i] = make_uint4(0u, 0u, 0u, 0u);
  fetch(X0);
  fetch(X1);
  int phase = 0;
  auto step = [&](Raw& w) {
    float x[kEPT];
    widen_raw<BF16, kEPT>(w, x);
    fetch(w);
    packed_message<kLogBlock, BF16>(x, wmax[phase], p.q[c_r], p.s[c_r], c_off);
    phase ^= 1;
    if (++c_r == n) {
      c_r = 0;
      c_off += stride;
    }
  };
  while (c_off < end) {  // the same number of steps in every thread of the CTA
    step(X0);
    if (c_off >= end) break;
    step(X1);
  }
  // the ragged end: one partial tile, by the last CTA with bounds
  if (blockIdx.x == gridDim.x - 1 && end < p.count) {
    const int64_t e = end + lane_off;
    const int shift = kLogBlock;
#pragma unroll 1
    for (int r = 0; r < n; ++r) {
      float x[kEPT], c[kEPT];
      load_group<BF16, kEPT>(p.g[r], e, p.count, x);
      const float s = block_scale<kEPT, true>(x, kBlock, wmax[phase]);
      phase ^= 1;
      if (e >= p.count) continue;  // after the block maximum, which every thread joins
      if ((e & (kBlock - 1)) == 0) p.s[r][e >> shift] = s;
      quant_group<kEPT, true>(x, s, c);
      store_codes<kEPT>(p.q[r], e, p.count, c);
    }
  }
}

// Each tile, ranks in order: quantise rank r's block, add its reconstruction
// to the running sum and store its residual; then write the scaled sum to
// every rank. No message leaves the registers.
template <bool BF16, bool EF>
__global__ void __launch_bounds__(kThreads) compressed_allreduce_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kEPT = ept<BF16>();
  constexpr int kTileElems = kEPT * kThreads;
  // Ranks per load batch. bf16 (with error feedback here; without, the
  // pipelined kernel above runs) takes one: fewer registers, more resident
  // warps (measured at 16 x 96 Mi: 0.97 of its bytes against 0.81 with two).
  // fp32 keeps 2 / 4 (one or two measured 0-3 % slower).
  constexpr int NB = BF16 ? 1 : (EF ? 2 : 4);
  __shared__ float wmax[2][kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  int phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e = tile * kTileElems + int64_t(kEPT) * threadIdx.x;
    float acc[kEPT];
#pragma unroll 1
    for (int r0 = 0; r0 < p.n; r0 += NB) {
      float xg[NB][kEPT], xe[NB][kEPT];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (r0 + b >= p.n) continue;
        load_group<BF16, kEPT>(p.g[r0 + b], e, p.count, xg[b]);
        if (EF) load_group<false, kEPT>(p.e[r0 + b], e, p.count, xe[b]);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int r = r0 + b;
        if (r >= p.n) continue;  // uniform across the CTA
        float x[kEPT], res[kEPT];
        if (EF)
          add_each(x, xg[b], xe[b]);
        else
#pragma unroll
          for (int w = 0; w < kEPT; ++w) x[w] = xg[b][w];
        fold_rank<kEPT, EF>(x, r, p.block, wmax[phase], acc, res);
        phase ^= 1;
        if (EF && e < p.count) store_group<false, kEPT>(p.e[r], e, p.count, res);
      }
    }
    if (e >= p.count) continue;
    mul_each(acc, acc, p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) store_group<BF16, kEPT>(p.out[r], e, p.count, acc);
  }
}

// The fused pass for fp32 blocks that span warps, where a block's maximum
// needs a CTA barrier: the scales of a whole load batch of NB ranks come from
// batch_scales, one barrier per batch instead of one per rank. Per element
// the same operations in the same rank order as compressed_allreduce_kernel.
// At 16 x 192 MiB fp32, block 1024 with error feedback (4 ranks per batch):
// 0.956 of its bytes against 0.918; without it the warp kernel below runs.
template <bool BF16, bool EF, int NB>
__global__ void __launch_bounds__(kThreads) compressed_allreduce_batch_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kEPT = ept<BF16>();
  constexpr int kTileElems = kEPT * kThreads;
  __shared__ float wmax[2][NB * kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  int phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e = tile * kTileElems + int64_t(kEPT) * threadIdx.x;
    float acc[kEPT];
#pragma unroll 1
    for (int r0 = 0; r0 < p.n; r0 += NB) {
      const int nb = p.n - r0 < NB ? p.n - r0 : NB;  // uniform across the CTA
      float x[NB][kEPT], xe[NB][kEPT];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) continue;
        load_group<BF16, kEPT>(p.g[r0 + b], e, p.count, x[b]);
        if (EF) load_group<false, kEPT>(p.e[r0 + b], e, p.count, xe[b]);
      }
      if (EF) {
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b < nb) add_each(x[b], x[b], xe[b]);
      }
      float s[NB];
      batch_scales<kEPT, NB, true>(x, nb, p.block, wmax[phase], s);
      phase ^= 1;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) continue;
        float res[kEPT];
        fold_scaled<kEPT, EF>(x[b], r0 + b, s[b], acc, res);
        if (EF && e < p.count) store_group<false, kEPT>(p.e[r0 + b], e, p.count, res);
      }
    }
    if (e >= p.count) continue;
    mul_each(acc, acc, p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r) store_group<BF16, kEPT>(p.out[r], e, p.count, acc);
  }
}

// ---------------------------------------------------------------- one block per warp
// Blocks of 256 or more fp32 values (512 or more bf16) span warps in the
// kernels above, whose threads hold consecutive elements: the block maximum
// then waits on a CTA barrier. Here a warp holds whole blocks: lane l takes
// kVec vectors of kW elements, vector j at element j * 32 * kW + l * kW of
// the block (each vector load of the warp is contiguous), so the block
// maximum is one full-warp reduction and no barrier is needed. A CTA takes
// kWarps blocks per tile. Per element the same operations in the same rank
// order as the other kernels (block_scale, quant_group), so the same bits.
// NB ranks per load batch.
template <bool BF16, bool EF, int kVec, int NB>
__global__ void __launch_bounds__(kThreads, 2) compressed_allreduce_warp_kernel(const __grid_constant__ CompressParams p) {
  constexpr int kW = BF16 ? 8 : 4;
  constexpr int kBlock = 32 * kW * kVec;
  constexpr int64_t kTileElems = int64_t(kBlock) * kWarps;
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t lane_off = int64_t(threadIdx.x >> 5) * kBlock + int64_t(threadIdx.x & 31) * kW;
  const int64_t n_tiles = (p.count + kTileElems - 1) / kTileElems;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t e0 = tile * kTileElems + lane_off;  // vector j at e0 + j * 32 * kW
    float acc[kVec][kW];
#pragma unroll 1
    for (int r0 = 0; r0 < p.n; r0 += NB) {
      float x[NB][kVec][kW], xe[EF ? NB : 1][EF ? kVec : 1][kW];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (r0 + b >= p.n) continue;  // uniform across the CTA
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          load_group<BF16, kW>(p.g[r0 + b], e0 + j * 32 * kW, p.count, x[b][j]);
          if constexpr (EF) load_group<false, kW>(p.e[r0 + b], e0 + j * 32 * kW, p.count, xe[b][j]);
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int r = r0 + b;
        if (r >= p.n) continue;
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          if constexpr (EF) add_each(x[b][j], x[b][j], xe[b][j]);
#pragma unroll
          for (int w = 0; w < kW; ++w) m = fmaxf(m, fabsf(x[b][j][w]));
        }
        // m >= 0: the unsigned maximum of the bits is the float maximum
        m = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(m)));
        const float s = div127(m);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          float c[kW], d[kW];
          quant_group<kW, true>(x[b][j], s, c);
          mul_each(d, c, s);
          if (r == 0) {
#pragma unroll
            for (int w = 0; w < kW; ++w) acc[j][w] = d[w];
          } else {
            add_each(acc[j], acc[j], d);
          }
          if constexpr (EF) {
            float res[kW];
            sub_each(res, x[b][j], d);
            store_group<false, kW>(p.e[r], e0 + j * 32 * kW, p.count, res);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) mul_each(acc[j], acc[j], p.scale);
#pragma unroll 1
    for (int r = 0; r < p.n; ++r)
#pragma unroll
      for (int j = 0; j < kVec; ++j) store_group<BF16, kW>(p.out[r], e0 + j * 32 * kW, p.count, acc[j]);
  }
}

// The self-test of div127: every non-negative float bit pattern (finite,
// +inf and NaN) against the IEEE division; the mismatches are counted.
__device__ unsigned long long g_div127_mismatches;

__global__ void div127_selftest_kernel() {
  unsigned long long bad = 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < 0x80000000u; u += stride) {
    const float m = __uint_as_float(u);
    const float want = __fdiv_rn(m, 127.0f);
    const float got = div127(m);
    const bool both_nan = want != want && got != got;
    if (!both_nan && __float_as_uint(want) != __float_as_uint(got)) ++bad;
  }
  if (bad != 0) atomicAdd(&g_div127_mismatches, bad);
}

using Kern = void (*)(CompressParams);

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

int64_t n_tiles(int64_t count, int elems_per_thread) {
  const int64_t tile = int64_t(elems_per_thread) * kThreads;
  return (count + tile - 1) / tile;
}

}  // namespace

// The packed compressor for each block size, 16 (2^4) to 1024 (2^10).
template <bool BF16>
Kern packed_compress_kernel(int block) {
  switch (block) {
    case 16: return compress_packed_kernel<BF16, 4>;
    case 32: return compress_packed_kernel<BF16, 5>;
    case 64: return compress_packed_kernel<BF16, 6>;
    case 128: return compress_packed_kernel<BF16, 7>;
    case 256: return compress_packed_kernel<BF16, 8>;
    case 512: return compress_packed_kernel<BF16, 9>;
    case 1024: return compress_packed_kernel<BF16, 10>;
    default: return nullptr;
  }
}

cudaError_t launch_compress(const CompressParams& p, ar_dtype dtype, cudaStream_t stream) {
  const bool bf = dtype == AR_BF16;
  if (!p.ef) {  // the block is a power of two from 16 to 1024 (checked by the host)
    const Kern k = bf ? packed_compress_kernel<true>(p.block) : packed_compress_kernel<false>(p.block);
    if (k == nullptr) return cudaErrorInvalidValue;
    return launch(k, n_tiles(p.count, 8), p, stream);
  }
  const bool wide = p.block > 32 * compress_ept<false>();  // an fp32 block spans warps
  const Kern k = bf ? compress_kernel<true, true, 1, false>
                    : (wide ? compress_kernel<false, true, 4, true> : compress_kernel<false, true, 4, false>);
  return launch(k, n_tiles(p.count, bf ? compress_ept<true>() : compress_ept<false>()), p, stream);
}

cudaError_t launch_compressed_reduce(const CompressParams& p, ar_dtype out_dtype, cudaStream_t stream) {
  const Kern k = out_dtype == AR_BF16 ? compressed_reduce_kernel<true> : compressed_reduce_kernel<false>;
  return launch(k, n_tiles(p.count, out_dtype == AR_BF16 ? reduce_ept<true>() : reduce_ept<false>()), p, stream);
}

// The packed bf16 kernel for each block size, 16 (2^4) to 1024 (2^10).
Kern packed_bf16_kernel(int block) {
  switch (block) {
    case 16: return compressed_allreduce_bf16_packed_kernel<4>;
    case 32: return compressed_allreduce_bf16_packed_kernel<5>;
    case 64: return compressed_allreduce_bf16_packed_kernel<6>;
    case 128: return compressed_allreduce_bf16_packed_kernel<7>;
    case 256: return compressed_allreduce_bf16_packed_kernel<8>;
    case 512: return compressed_allreduce_bf16_packed_kernel<9>;
    case 1024: return compressed_allreduce_bf16_packed_kernel<10>;
    default: return nullptr;
  }
}

// The one-block-per-warp kernel where it measured faster (nullptr
// elsewhere). Gradient vectors per thread per load batch: fp32 16 (8 with
// error feedback, whose residuals are loaded too), bf16 4 with error
// feedback: every loaded value is held widened to fp32 until its rank is
// folded. At 16 x 192 MiB (fp32) or 16 x 96 Mi (bf16), fraction of its bytes
// against the kernels above: fp32 without error feedback, blocks 256 / 512 /
// 1024: 0.929 / 0.886 / 0.922 against 0.858 / 0.843 / 0.823; fp32 with it,
// block 1024: 0.977 against 0.957 (block 512 0.954 against 0.961, 256 the
// same); bf16 with it, block 512: 0.787 against 0.772 (1024: 0.66 against
// 0.77). bf16 without error feedback keeps the packed kernel (0.86 against
// 0.40 here).
template <bool BF16, bool EF>
Kern warp_block_kernel(int block) {
  if constexpr (!BF16 && !EF) {
    if (block == 256) return compressed_allreduce_warp_kernel<false, false, 2, 8>;
    if (block == 512) return compressed_allreduce_warp_kernel<false, false, 4, 4>;
    if (block == 1024) return compressed_allreduce_warp_kernel<false, false, 8, 2>;
  } else if constexpr (!BF16 && EF) {
    if (block == 1024) return compressed_allreduce_warp_kernel<false, true, 8, 1>;
  } else if constexpr (BF16 && EF) {
    if (block == 512) return compressed_allreduce_warp_kernel<true, true, 2, 2>;
  }
  return nullptr;
}

cudaError_t launch_compressed_allreduce(const CompressParams& p, ar_dtype dtype, cudaStream_t stream) {
  const bool bf = dtype == AR_BF16;
  {
    const Kern k = bf ? (p.ef ? warp_block_kernel<true, true>(p.block) : warp_block_kernel<true, false>(p.block))
                      : (p.ef ? warp_block_kernel<false, true>(p.block) : warp_block_kernel<false, false>(p.block));
    if (k != nullptr) {
      const int per_thread = p.block / 32;  // kVec vectors of kW elements
      return launch(k, n_tiles(p.count, per_thread), p, stream);
    }
  }
  if (bf && !p.ef && p.n % 2 == 0) {
    const Kern k = packed_bf16_kernel(p.block);
    if (k != nullptr) return launch(k, n_tiles(p.count, ept<true>()), p, stream);
  }
  const bool wide = p.block > 32 * ept<false>();  // an fp32 block spans warps
  Kern k = compressed_allreduce_bf16_kernel;
  if (bf && p.ef)
    k = compressed_allreduce_kernel<true, true>;
  else if (!bf)
    k = p.ef ? (wide ? compressed_allreduce_batch_kernel<false, true, 4> : compressed_allreduce_kernel<false, true>)
             : (wide ? compressed_allreduce_batch_kernel<false, false, 4> : compressed_allreduce_kernel<false, false>);
  return launch(k, n_tiles(p.count, bf ? ept<true>() : ept<false>()), p, stream);
}

cudaError_t selftest_div127(unsigned long long* mismatches) {
  const unsigned long long zero = 0;
  cudaError_t err = cudaMemcpyToSymbol(g_div127_mismatches, &zero, sizeof(zero));
  if (err != cudaSuccess) return err;
  div127_selftest_kernel<<<1216, 256>>>();
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  return cudaMemcpyFromSymbol(mismatches, g_div127_mismatches, sizeof(*mismatches));
}

}  // namespace ar
