// Bucket pack and unpack for the DDP-style bucketed gradient sync (Scaling ML
// Systems, "Collective communication", section "Bucket fusion": one
// all-reduce per bucket of gradients).
//
// pack:   bucket[r][off_t + e] = fp32(tensor[r][t][e])      (bf16 widened exactly)
// unpack: tensor[r][t][e]      = round(scale * bucket[r][off_t + e])  (bf16: RNE)
//
// One launch covers every rank and every tensor of a group of the bucket's
// tensors; each thread moves 8 elements. Work is tiled per (rank, tensor) so
// that tiles never straddle two tensors.
#include "common.cuh"

namespace ar {

namespace {

template <bool BF16, bool UNPACK>
__global__ void __launch_bounds__(kThreads) pack_kernel(const __grid_constant__ PackParams p) {
  grid_dependency_wait();  // stream order with the previous kernel (see launch_pack)
  grid_dependents_launch();
  const int per_rank = p.tile_start[p.n_t];
  const int total = per_rank * p.n;
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    const int r = t / per_rank;
    const int tr = t - r * per_rank;
    int i = 0;
    while (p.tile_start[i + 1] <= tr) ++i;
    const int64_t tt = tr - p.tile_start[i];
    const int64_t cnt = p.cnt[i], off = p.off[i];
    char* tens = static_cast<char*>(p.tptr[i * p.n + r]);
    float* buck = static_cast<float*>(p.bucket[r]) + off;
    const int64_t e = tt * kPackTile + int64_t(threadIdx.x) * 8;
    if (e >= cnt) continue;
    const bool vec = (e + 8 <= cnt) && (off % 4 == 0);
    if (!UNPACK) {
      float f[8];
      if (vec) {
        if (BF16) {
          const uint4 a = __ldcs(reinterpret_cast<const uint4*>(tens + e * 2));
          f[0] = bf16lo(a.x); f[1] = bf16hi(a.x); f[2] = bf16lo(a.y); f[3] = bf16hi(a.y);
          f[4] = bf16lo(a.z); f[5] = bf16hi(a.z); f[6] = bf16lo(a.w); f[7] = bf16hi(a.w);
        } else {
          const uint4* q = reinterpret_cast<const uint4*>(tens + e * 4);
          const uint4 a = __ldcs(q), b = __ldcs(q + 1);
          f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
          f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
          f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
          f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
        }
        float4* d = reinterpret_cast<float4*>(buck + e);
        __stcs(d, make_float4(f[0], f[1], f[2], f[3]));
        __stcs(d + 1, make_float4(f[4], f[5], f[6], f[7]));
      } else {
        const int64_t end = e + 8 < cnt ? e + 8 : cnt;
        for (int64_t x = e; x < end; ++x)
          buck[x] = BF16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(tens)[x])
                         : reinterpret_cast<const float*>(tens)[x];
      }
    } else {
      if (vec) {
        const float4* s = reinterpret_cast<const float4*>(buck + e);
        const float4 a = __ldcs(s), b = __ldcs(s + 1);
        float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) f[w] = fmul(f[w], p.scale);
        if (BF16) {
          __stcs(reinterpret_cast<uint4*>(tens + e * 2),
                 make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                            pack_bf16x2(f[6], f[7])));
        } else {
          float4* d = reinterpret_cast<float4*>(tens + e * 4);
          __stcs(d, make_float4(f[0], f[1], f[2], f[3]));
          __stcs(d + 1, make_float4(f[4], f[5], f[6], f[7]));
        }
      } else {
        const int64_t end = e + 8 < cnt ? e + 8 : cnt;
        for (int64_t x = e; x < end; ++x) {
          const float v = fmul(buck[x], p.scale);
          if (BF16)
            reinterpret_cast<uint16_t*>(tens)[x] = f32_to_bf16(v);
          else
            reinterpret_cast<float*>(tens)[x] = v;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, ar_dtype dtype, bool unpack, cudaStream_t stream) {
  const int64_t tiles = int64_t(p.tile_start[p.n_t]) * p.n;
  if (tiles <= 0) return cudaSuccess;
  void (*k)(PackParams) = dtype == AR_BF16 ? (unpack ? pack_kernel<true, true> : pack_kernel<true, false>)
                                           : (unpack ? pack_kernel<false, true> : pack_kernel<false, false>);
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

}  // namespace ar
