// Device helpers shared by the all-reduce kernels: 16-byte streaming loads
// and stores, exact bf16 widening, round-to-nearest-even narrowing, and the
// per-element summation folds.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace ar {

__device__ __forceinline__ int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
__device__ __forceinline__ int64_t round_down(int64_t x, int64_t a) { return x / a * a; }

// Programmatic dependent launch: wait until the previous kernel on the stream
// has completed and its writes are visible; let the next one start launching.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// bf16 is the top half of an fp32 word: widening appends 16 zero bits (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// fp32 -> bf16, round to nearest, ties to even (the CUDA conversion intrinsic).
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return uint32_t(f32_to_bf16(lo)) | (uint32_t(f32_to_bf16(hi)) << 16);
}

// The only arithmetic of the all-reduce: IEEE fp32 add and one multiply by
// the scale, each rounded to nearest even, never contracted into an FMA.
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }

// A "lane" is what one thread moves per rank per step of the hot loop:
// a 16-byte vector (4 fp32 or 8 bf16 elements) on the aligned body of a
// range, or one element on its ragged head and tail.
template <bool BF16, bool VEC>
struct Lane;

template <>
struct Lane<false, true> {  // 4 x fp32
  static constexpr int W = 4;
  using raw_t = uint4;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return __ldcs(reinterpret_cast<const uint4*>(base + e * 4));
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  }
  static __device__ __forceinline__ raw_t narrow(const float (&f)[W]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ void store(char* base, int64_t e, const raw_t& r) {
    __stcs(reinterpret_cast<uint4*>(base + e * 4), r);
  }
};

template <>
struct Lane<true, true> {  // 8 x bf16
  static constexpr int W = 8;
  using raw_t = uint4;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return __ldcs(reinterpret_cast<const uint4*>(base + e * 2));
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) {
    f[0] = bf16lo(r.x); f[1] = bf16hi(r.x); f[2] = bf16lo(r.y); f[3] = bf16hi(r.y);
    f[4] = bf16lo(r.z); f[5] = bf16hi(r.z); f[6] = bf16lo(r.w); f[7] = bf16hi(r.w);
  }
  static __device__ __forceinline__ raw_t narrow(const float (&f)[W]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
  static __device__ __forceinline__ void store(char* base, int64_t e, const raw_t& r) {
    __stcs(reinterpret_cast<uint4*>(base + e * 2), r);
  }
};

template <>
struct Lane<false, false> {  // 1 x fp32
  static constexpr int W = 1;
  using raw_t = uint32_t;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return *reinterpret_cast<const uint32_t*>(base + e * 4);
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) { f[0] = __uint_as_float(r); }
  static __device__ __forceinline__ raw_t narrow(const float (&f)[W]) { return __float_as_uint(f[0]); }
  static __device__ __forceinline__ void store(char* base, int64_t e, const raw_t& r) {
    *reinterpret_cast<uint32_t*>(base + e * 4) = r;
  }
};

template <>
struct Lane<true, false> {  // 1 x bf16
  static constexpr int W = 1;
  using raw_t = uint16_t;
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    return *reinterpret_cast<const uint16_t*>(base + e * 2);
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) { f[0] = bf16_to_f32(r); }
  static __device__ __forceinline__ raw_t narrow(const float (&f)[W]) { return f32_to_bf16(f[0]); }
  static __device__ __forceinline__ void store(char* base, int64_t e, const raw_t& r) {
    *reinterpret_cast<uint16_t*>(base + e * 2) = r;
  }
};

// A 32-byte lane: 8 fp32 or 16 bf16 elements moved by one 256-bit access
// (ld/st.global.cs.v8.b32, sm_100 and later). Addresses must be 32-byte
// aligned: kernels use it only when the host has checked every base pointer.
template <bool BF16>
struct Lane32 {
  static constexpr int W = BF16 ? 16 : 8;
  struct raw_t {
    uint32_t w[8];
  };
  static __device__ __forceinline__ raw_t load(const char* base, int64_t e) {
    raw_t r;
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]),
                   "=r"(r.w[7])
                 : "l"(base + e * (BF16 ? 2 : 4)));
    return r;
  }
  static __device__ __forceinline__ void widen(const raw_t& r, float (&f)[W]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (BF16) {
        f[2 * i] = bf16lo(r.w[i]);
        f[2 * i + 1] = bf16hi(r.w[i]);
      } else {
        f[i] = __uint_as_float(r.w[i]);
      }
    }
  }
  static __device__ __forceinline__ raw_t narrow(const float (&f)[W]) {
    raw_t r;
#pragma unroll
    for (int i = 0; i < 8; ++i) r.w[i] = BF16 ? pack_bf16x2(f[2 * i], f[2 * i + 1]) : __float_as_uint(f[i]);
    return r;
  }
  static __device__ __forceinline__ void store(char* base, int64_t e, const raw_t& r) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(base + e * (BF16 ? 2 : 4)), "r"(r.w[0]),
                 "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]), "r"(r.w[7])
                 : "memory");
  }
};

// ---------------------------------------------------------------------------
// Summation folds over the ranks of one element position.
//
// A fold visits the ranks in a fixed sequence (the order of a schedule).
// `seq_ptr[p]` is the input pointer of the rank visited at position p and
// `seq_flag[p]` tells how position p combines:
//   kStart: begin a new group partial with this value
//   kEnd:   this value completes the group partial; fold it into the total
//   kFirst: the completed group partial is the first one (total = partial)
// A ring or rank-order fold is one group of N; the hierarchical order is M
// groups of G. Each thread folds VPT vectors at once; loads are issued NB
// ranks at a time before any add, so that NB * VPT 16-byte requests per
// thread are in flight (VPT > 1 keeps that number up when N is small).
// ---------------------------------------------------------------------------
enum : uint8_t { kStart = 1, kEnd = 2, kFirst = 4 };

template <class L, int NB, int VPT>
__device__ __forceinline__ void fold_sequence(float (&acc)[VPT][L::W], const char* const* seq_ptr,
                                              const uint8_t* seq_flag, int n, const int64_t (&e)[VPT],
                                              const bool (&ok)[VPT]) {
  float part[VPT][L::W];
#pragma unroll 1
  for (int base = 0; base < n; base += NB) {
    typename L::raw_t v[NB][VPT];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int q = 0; q < VPT; ++q)
        if (base + b < n && ok[q]) v[b][q] = L::load(seq_ptr[base + b], e[q]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (base + b < n) {
        const uint8_t fl = seq_flag[base + b];
#pragma unroll
        for (int q = 0; q < VPT; ++q) {
          if (!ok[q]) continue;
          float f[L::W];
          L::widen(v[b][q], f);
          if (fl & kStart) {
#pragma unroll
            for (int w = 0; w < L::W; ++w) part[q][w] = f[w];
          } else {
#pragma unroll
            for (int w = 0; w < L::W; ++w) part[q][w] = fadd(part[q][w], f[w]);
          }
          if (fl & kEnd) {
            if (fl & kFirst) {
#pragma unroll
              for (int w = 0; w < L::W; ++w) acc[q][w] = part[q][w];
            } else {
#pragma unroll
              for (int w = 0; w < L::W; ++w) acc[q][w] = fadd(acc[q][w], part[q][w]);
            }
          }
        }
      }
    }
  }
}

// fold_sequence for a sequence of one group (ring, rank order, the ring
// reduce-scatter, the all-gather's single owner): the start and end of the
// group are known from the position, so no flags are read. Same loads in
// flight and same additions, in the same order. Measured at 16 ranks x
// 192 MiB fp32 it ran about 0.6 % slower than reading the flags; at 64
// ranks x 16 MiB 3.5 % faster and on the reduce-scatter 2 % faster.
template <class L, int NB, int VPT>
__device__ __forceinline__ void fold_single(float (&acc)[VPT][L::W], const char* const* seq_ptr, int n,
                                            const int64_t (&e)[VPT], const bool (&ok)[VPT]) {
  float part[VPT][L::W];
#pragma unroll 1
  for (int base = 0; base < n; base += NB) {
    typename L::raw_t v[NB][VPT];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int q = 0; q < VPT; ++q)
        if (base + b < n && ok[q]) v[b][q] = L::load(seq_ptr[base + b], e[q]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (base + b < n) {
        const bool first = base + b == 0, last = base + b == n - 1;
#pragma unroll
        for (int q = 0; q < VPT; ++q) {
          if (!ok[q]) continue;
          float f[L::W];
          L::widen(v[b][q], f);
          if (first) {
#pragma unroll
            for (int w = 0; w < L::W; ++w) part[q][w] = f[w];
          } else {
#pragma unroll
            for (int w = 0; w < L::W; ++w) part[q][w] = fadd(part[q][w], f[w]);
          }
          if (last) {
#pragma unroll
            for (int w = 0; w < L::W; ++w) acc[q][w] = part[q][w];
          }
        }
      }
    }
  }
}

// Balanced binary tree over ranks 0..n-1 in index order (n a power of two):
// ((g0+g1)+(g2+g3))+... . Values are combined as they arrive with a binary
// counter: slot l holds a finished subtree of 2^l ranks; before rank p
// arrives the occupied slots are the set bits of p.
constexpr int kTreeLevels = 7;  // up to 64 ranks

template <class L, int NB>
__device__ __forceinline__ void fold_tree(float (&acc)[L::W], const char* const* seq_ptr, int n,
                                          int64_t e) {
  float slot[kTreeLevels][L::W];
#pragma unroll 1
  for (int base = 0; base < n; base += NB) {
    typename L::raw_t v[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (base + b < n) v[b] = L::load(seq_ptr[base + b], e);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (base + b < n) {
        float carry[L::W];
        L::widen(v[b], carry);
        int bits = base + b;
        bool placed = false;
#pragma unroll
        for (int l = 0; l < kTreeLevels; ++l) {
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
  // n = 2^K: the whole tree sits in slot K
#pragma unroll
  for (int l = 0; l < kTreeLevels; ++l)
    if ((1 << l) == n) {
#pragma unroll
      for (int w = 0; w < L::W; ++w) acc[w] = slot[l][w];
    }
}

// ---------------------------------------------------------------------------
// Host side: persistent grids. A kernel gets min(tiles, resident CTAs) blocks,
// where resident = CTAs per SM at kThreads threads (occupancy calculator)
// times the SM count (or the caller's SM budget, if smaller), so the grid is
// a whole number of waves over the SMs it may use. Cached per (device, kernel).
// ---------------------------------------------------------------------------
inline int persistent_grid(const void* kernel, int64_t tiles, int sm_budget = 0) {
  struct Entry {
    int device;
    const void* kernel;
    int per_sm;
    int sms;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  int per_sm = 0, sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.device == dev && e.kernel == kernel) {
        per_sm = e.per_sm;
        sms = e.sms;
      }
  }
  if (per_sm == 0) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess)
      per_sm = 1;
    if (sms <= 0) sms = 1;
    if (per_sm <= 0) per_sm = 1;
    std::lock_guard<std::mutex> lock(mu);
    cache.push_back({dev, kernel, per_sm, sms});
  }
  const int use = (sm_budget > 0 && sm_budget < sms) ? sm_budget : sms;
  const int64_t blocks = int64_t(per_sm) * use;
  return int(tiles < blocks ? tiles : blocks);
}

}  // namespace ar
