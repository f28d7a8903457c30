// Internal declarations shared by the host planner (api.cpp) and the CUDA
// launchers (*.cu). Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/ar.h"

namespace ar {

// Where a step operand lives. RAW: the rank's input buffer (input dtype).
// PART: the rank's fp32 partial sums (fp32 runs: the output buffer itself;
// bf16 runs: the workspace). RES: the rank's output buffer (output dtype).
enum Space : uint8_t { RAW = 0, PART = 1, RES = 2 };

enum StepOp : int { OP_ADD = 0, OP_COPY = 1, OP_FINISH = 2 };

// One send/receive of a step: rank `dst` receives elements [lo, hi) from
// rank `src`. ADD: D[dst] = X[src] + Y[dst], then + X2[src2] when src2 >= 0
// (a tree node receiving from two children in one step); final: times scale,
// rounded to the output type. With `pair`, src receives the same sum in
// D[src] (an exchange: fp32 addition commutes, so both partners hold the
// same bits). COPY: D[dst] = X[src], operands of one type; with `pair`,
// also D[src] = X[src] (an out-of-place all-gather's first step writing the
// sender's own chunk to its output as it sends it). FINISH (one
// rank): RES[dst] = scale * X[src], rounded to the output type.
struct Transfer {
  int16_t src, dst, src2;
  uint8_t xs, ys, ds, x2s, fin, pair;
  int64_t lo, hi;
};

struct Step {
  StepOp op;
  std::vector<Transfer> xfers;
};

}  // namespace ar

namespace ar {

// The device a plan last ran on (-1: never), written by the executing calls
// and read by ar_plan_query, possibly from other threads. Copyable, so that
// a plan can still be copied by value.
struct DeviceTag {
  std::atomic<int> v{-1};
  DeviceTag() = default;
  DeviceTag(const DeviceTag& o) : v(o.v.load(std::memory_order_relaxed)) {}
  DeviceTag& operator=(const DeviceTag& o) {
    v.store(o.v.load(std::memory_order_relaxed), std::memory_order_relaxed);
    return *this;
  }
};

}  // namespace ar

struct ar_plan {
  ar_desc desc;
  std::vector<ar::Step> steps;  // empty for AR_FUSED
  ar_stats stats;
  int64_t ws_stride;  // fp32 elements per rank in the workspace (multiple of 64)
  bool small = false; // step plan run whole in one CTA (one launch)
  bool small_smem = false;  // ... with its buffers in shared memory
  mutable ar::DeviceTag last_device;
};

namespace ar {

constexpr int kMaxXfers = AR_MAX_RANKS;

// ---- kernel launch parameter blocks (passed by value, < 4 KB each) ----

struct StepParams {
  void* raw[AR_MAX_RANKS];
  void* res[AR_MAX_RANKS];
  float* ws;
  int64_t ws_stride;
  float scale;
  int n_xfer;
  int interleave;  // 1: tiles dealt round-robin over the transfers; 0: transfer by transfer
  Transfer x[kMaxXfers];
  int32_t tile_start[kMaxXfers + 1];  // prefix sums of tiles per transfer
};

struct FusedParams {
  const void* in[AR_MAX_RANKS];
  void* out[AR_MAX_RANKS];
  int n;            // ranks
  int collective;   // ar_collective
  int order;        // ar_order
  int g, m;         // hierarchical group size and group count
  int n_seg;        // segments of constant summation order
  int64_t count;    // elements per rank
  int64_t e_lo, e_hi;  // element range processed by this launch
  int64_t tiles_per_seg;
  float scale;
};

// The whole schedule of a small step plan in one CTA (step.cu): every step's
// transfers in one table, element ranges below 2^31.
struct SmallXfer {
  int16_t src, dst, src2;
  uint8_t xs, ys, ds, x2s, fin, pair;
  int32_t lo, len;  // element range [lo, lo + len) of the ranks' buffers
  int32_t flat;     // elements of the step's earlier transfers
};

// One piece of a step run on chip (small_steps_smem_kernel): the byte
// offsets, in the kernel's shared memory, of element `lo` of each operand,
// the element count and the operation's options. The host resolves the
// ranks, spaces and types once, so a warp reads one entry per piece.
struct SmemPiece {
  uint32_t x, y, x2, d, d2;  // sources, destination, exchange partner
  uint16_t len;              // elements, at most kSmallPiece
  uint8_t flags;             // kPiece* below
  uint8_t pad;
};
enum : uint8_t {
  kPieceX32 = 1, kPieceY32 = 2, kPieceX2_32 = 4, kPieceD32 = 8,  // operand is fp32 (else bf16)
  kPieceTwo = 16, kPiecePair = 32, kPieceFin = 64                 // second source, exchange, scale
};
static_assert(sizeof(SmemPiece) == sizeof(SmallXfer), "the two tables share storage");

constexpr int kMaxSmallXfers = 1024;
constexpr int kMaxSmallSteps = 256;
// A step plan runs in one CTA when its table fits and no step moves more
// than kSmallStepElems elements (two per thread of the CTA). Measured on
// GB300, 16 ranks, bound calls: ring at 256 / 1024 elements per rank 30.7 /
// 36.9 us against 49 us one kernel per step; Rabenseifner at 256 (2048
// elements in its first step) 12.3 us against about 15. At 4096 elements per
// step and more the one-CTA path was slower (ring at 4096 per rank: 98 us
// against about 50), so those plans keep one kernel per step.
constexpr int64_t kSmallStepElems = 2048;
// Such a plan runs on chip when its buffers fit in shared memory beside the
// transfer table: 8 bytes per element and rank (input and output copies,
// plus fp32 partials for bf16), up to this many bytes.
// On chip the table holds pieces of at most kSmallPiece elements (one warp
// each) instead of whole transfers, and the ranks' rows are copied as 4-byte
// words, so count * element size must be a multiple of 4.
constexpr int64_t kSmallSmemDataBytes = 160 * 1024;
constexpr int kSmallPiece = 128;
inline int64_t small_smem_data_bytes(int n_ranks, int64_t count) { return 8 * int64_t(n_ranks) * count; }

struct SmallParams {
  void* raw[AR_MAX_RANKS];
  void* res[AR_MAX_RANKS];
  float* ws;
  int64_t ws_stride;
  float scale;
  int n_steps;
  // On chip (small_steps_smem_kernel): the ranks' elements, and which ranks
  // run in place (bit r: res[r] is raw[r]).
  int32_t n_ranks, count;
  uint64_t in_place;
  int32_t vec16;  // every buffer 16-byte aligned and count * element size a multiple of 16
  int32_t step_start[kMaxSmallSteps + 1];  // first transfer of each step in x[]
  int32_t step_elems[kMaxSmallSteps];      // elements of each step, all transfers
  uint8_t step_op[kMaxSmallSteps];         // StepOp of each step
  union {
    SmallXfer x[kMaxSmallXfers];   // small_steps_kernel
    SmemPiece px[kMaxSmallXfers];  // small_steps_smem_kernel
  };
  int32_t threads;  // small_steps_smem_kernel: the CTA's threads (32 per piece of the widest step)
};
static_assert(sizeof(SmallParams) <= 32764, "kernel parameter limit");

constexpr int kMaxBucketPtrs = 256;  // n_ranks * tensors per launch
constexpr int kMaxBucketSegs = 96;

struct BucketSeg {
  int32_t t;      // tensor slot in the launch's pointer table
  int32_t rot;    // ring order: first rank of the fold (the chunk index)
  int64_t lo, hi; // element range inside the tensor
};

struct BucketFusedParams {
  void* ptr[kMaxBucketPtrs];  // ptr[t * n + r]: rank r's tensor t
  int n;
  int n_seg;
  float scale;
  BucketSeg seg[kMaxBucketSegs];
  int32_t tile_start[kMaxBucketSegs + 1];
};

struct PackParams {
  void* tptr[kMaxBucketPtrs];  // tptr[t * n + r]
  void* bucket[AR_MAX_RANKS];
  int n;
  int n_t;
  float scale;
  int64_t off[AR_MAX_BUCKET_TENSORS];   // packed offset of each tensor
  int64_t cnt[AR_MAX_BUCKET_TENSORS];
  int32_t tile_start[AR_MAX_BUCKET_TENSORS + 1];  // tiles per tensor (one rank)
};

// Blockwise INT8 compression (compress.cu). One parameter block serves the
// three kernels: compress (g, e -> q, s, e'), the message reducer (q, s ->
// out) and the fused single pass (g, e -> e', out).
struct CompressParams {
  const void* g[AR_MAX_RANKS];  // gradients, in the call's dtype
  float* e[AR_MAX_RANKS];       // residuals (error feedback), fp32; unused when !ef
  int8_t* q[AR_MAX_RANKS];      // codes, one byte per element
  float* s[AR_MAX_RANKS];       // scales, one fp32 per block
  void* out[AR_MAX_RANKS];      // results, in the call's output dtype
  int n;                        // ranks
  int block;                    // elements per quantisation block (power of two, 16..1024)
  int ef;                       // 1: residuals given
  int64_t count;                // elements per rank
  int64_t n_blocks;             // ceil(count / block)
  float scale;                  // multiplies the complete fp32 sum once
};

// The current device's SM count (cached per device).
inline int device_sms() {
  static std::mutex mu;
  static std::vector<std::pair<int, int>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& e : cache)
      if (e.first == dev) return e.second;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({dev, sms});
  return sms;
}

// A launch held to fewer SMs than the GPU has. Its CTAs land on different
// SMs (the scheduler spreads them), each with the whole SM's memory path to
// itself, so they run the variants that keep twice the loads in flight per
// thread: a copy kernel on 64 CTAs measured 4.0 TB/s with 8 16-byte loads in
// flight per thread and 5.1 TB/s with 16 (GB300, one CTA per SM).
inline bool budgeted(int sm_budget) { return sm_budget > 0 && sm_budget < device_sms(); }

// ---- launchers (defined in the .cu files) ----
// Tile sizes the launchers and the host planner agree on (elements).
constexpr int kThreads = 256;
constexpr int kStepVec = 8;                               // elements per vector in step kernels
constexpr int kStepUnroll = 2;
constexpr int64_t kStepTile = kThreads * kStepVec * kStepUnroll;  // 4096
constexpr int kPackTile = kThreads * 8;                   // 2048 elements

// v8: every base pointer of the call is 32-byte aligned, so the fp32 vectors
// may move as 256-bit accesses.
cudaError_t launch_step(const StepParams& p, ar_dtype dtype, StepOp op, int total_tiles, bool pdl,
                        int sm_budget, bool v8, cudaStream_t stream);
cudaError_t launch_fused(const FusedParams& p, ar_dtype dtype, int sm_budget, cudaStream_t stream);
// All steps of a small plan in one CTA, a block barrier between steps.
cudaError_t launch_small_steps(const SmallParams& p, ar_dtype dtype, cudaStream_t stream);
// The same schedule with the buffers copied to shared memory first and every
// step run there (p.n_ranks, p.count, p.in_place set; the data fit).
cudaError_t launch_small_steps_smem(const SmallParams& p, ar_dtype dtype, cudaStream_t stream);
// Register pipeline: elements per vector (v8: 32-byte vectors, bucket kernel
// only, N > 4 and every pointer 32-byte aligned) and per tile.
int fused_vec_elems(ar_dtype dtype, bool v8);
int64_t fused_tile_elems(ar_dtype dtype, int n, int order, int collective, bool deep);
int64_t bucket_tile_elems(ar_dtype dtype, int n, bool v8, bool deep);
cudaError_t launch_bucket_fused(const BucketFusedParams& p, ar_dtype dtype, int sm_budget, bool v8, cudaStream_t stream);
cudaError_t launch_pack(const PackParams& p, ar_dtype dtype, bool unpack, cudaStream_t stream);
cudaError_t read_device_status(unsigned int* value, bool clear);
// Host-visible copy of a device's status word (page-locked, mapped host
// memory that the bounded waits also set). host_status_word publishes it on
// first use (a one-time pinned host allocation, no device memory);
// host_status_word_if_ready returns it only if already published, else null,
// and makes no CUDA call.
cudaError_t host_status_word(int device, volatile unsigned int** word);
volatile unsigned int* host_status_word_if_ready(int device);
// The bulk-copy variant of the fused all-reduce (fused_tma.cu).
bool tma_shape(int n, int& stages, int& tile_bytes);
cudaError_t launch_fused_tma(const FusedParams& p, ar_dtype dtype, int stages, int tile_bytes, int sm_budget,
                             cudaStream_t stream);
cudaError_t launch_bucket_tma(const BucketFusedParams& p, ar_dtype dtype, int stages, int tile_bytes, int sm_budget,
                              cudaStream_t stream);
cudaError_t launch_wait_timeout(uint32_t polls, cudaStream_t stream);
// The all-gather with bulk copies (fused_tma.cu): tile size in elements, launch.
int64_t allgather_bulk_tile_elems(ar_dtype dtype);
cudaError_t launch_allgather_bulk(const FusedParams& p, ar_dtype dtype, int sm_budget, cudaStream_t stream);
// Blockwise INT8 compression (compress.cu).
cudaError_t launch_compress(const CompressParams& p, ar_dtype dtype, cudaStream_t stream);
cudaError_t launch_compressed_reduce(const CompressParams& p, ar_dtype out_dtype, cudaStream_t stream);
cudaError_t launch_compressed_allreduce(const CompressParams& p, ar_dtype dtype, cudaStream_t stream);
// Self-test of the division-free block scale against the IEEE division, over
// every non-negative float (synchronises the device).
cudaError_t selftest_div127(unsigned long long* mismatches);

}  // namespace ar
