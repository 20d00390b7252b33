// Stateless W-way bf16 reduce: the HBM-streaming hot kernel.
//
// arx.cu, `arx_kernel`, reduce loop: for each group of 8 elements, load the
// W partials as one 16-byte vector each, add them into 8 fp32 accumulators
// from +0 in rank order, round each to bf16 once and store one 16-byte
// vector.  Each thread reads every slot at a group before it writes that
// group, so the output may be one of the slots.
//
// GB300 design: a persistent grid-stride loop (grid = SMs x resident blocks,
// capped by the work), U independent groups per thread per iteration so that
// U*W 16-byte loads are in flight before the first add (Little's law against
// HBM3e latency), coalesced 512-byte warp accesses per slot, L1 bypassed.
// The pages' fixed grid of at most 8 blocks and 512 KB cap are dropped.
#include "arx_device.cuh"
#include "arx_internal.h"

namespace arx {
namespace {

struct VecArgs {
  const uint16_t* slot[kMaxW];  // element 0 of each slot
  uint16_t* out;
  size_t n;        // elements
  size_t head;     // scalar elements before the first 16-byte boundary
  size_t groups;   // 16-byte groups after the head
};

// Independent 16-byte groups per thread per iteration.  W*U vectors are
// loaded before the first add: 8 vectors (128 B) per thread for every W.
template <int W>
struct Unroll {
  static constexpr int U = W >= 8 ? 1 : (W >= 4 ? 2 : (W >= 2 ? 4 : 8));
};

template <int W>
__device__ __forceinline__ void scalar_element(const VecArgs& a, size_t e) {
  float acc = 0.0f;
#pragma unroll
  for (int r = 0; r < W; ++r) acc = __fadd_rn(acc, widen16(a.slot[r][e]));
  a.out[e] = round_bf16(acc);
}

template <int W, bool kAlias>
__device__ __forceinline__ uint4 load_group(const uint4* p) {
  if constexpr (kAlias) {
    return ld_stream(p);
  } else {
    return ld_stream_nc(p);
  }
}

template <int W, bool kAlias>
__global__ void __launch_bounds__(kThreads) reduce_vec_kernel(const VecArgs a) {
  constexpr int U = Unroll<W>::U;
  const uint4* src[W];
#pragma unroll
  for (int r = 0; r < W; ++r) src[r] = reinterpret_cast<const uint4*>(a.slot[r] + a.head);
  uint4* dst = reinterpret_cast<uint4*>(a.out + a.head);

  const size_t stride = size_t(gridDim.x) * kThreads;
  size_t g = size_t(blockIdx.x) * kThreads + threadIdx.x;
  const size_t G = a.groups;

  // Main loop: U groups g, g + stride, ..., all loads issued before any add.
  if (U > 1) {
    for (; g + size_t(U - 1) * stride < G; g += size_t(U) * stride) {
      uint4 v[U][W];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < W; ++r) v[u][r] = load_group<W, kAlias>(src[r] + g + u * stride);
#pragma unroll
      for (int u = 0; u < U; ++u) st_global(dst + g + u * stride, sum_vectors<W>(v[u]));
    }
  }
  for (; g < G; g += stride) {
    uint4 v[W];
#pragma unroll
    for (int r = 0; r < W; ++r) v[r] = load_group<W, kAlias>(src[r] + g);
    st_global(dst + g, sum_vectors<W>(v));
  }

  // Scalar head (before the first 16-byte boundary) and tail (after the last
  // full group): at most 7 + 7 elements, done by the last block.
  const size_t tail = a.n - a.head - 8 * G;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x < a.head + tail) {
    const size_t t = threadIdx.x;
    const size_t e = t < a.head ? t : a.head + 8 * G + (t - a.head);
    scalar_element<W>(a, e);
  }
}

// Pointers with different addresses mod 16: one element per thread per step.
template <int W>
__global__ void __launch_bounds__(kThreads) reduce_scalar_kernel(const VecArgs a) {
  const size_t stride = size_t(gridDim.x) * kThreads;
  for (size_t e = size_t(blockIdx.x) * kThreads + threadIdx.x; e < a.n; e += stride)
    scalar_element<W>(a, e);
}

constexpr int kMaxDevices = 64;

template <int W, bool kAlias>
int vec_blocks_per_sm(int dev, cudaError_t* err) {
  static int cache[kMaxDevices];  // 0 = not yet queried
  if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int b = 0;
  *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, reduce_vec_kernel<W, kAlias>, kThreads, 0);
  if (*err != cudaSuccess || b < 1) return -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = b;
  return b;
}

template <int W>
cudaError_t launch_w(const ReduceCall& c, cudaStream_t stream) {
  VecArgs a{};
  for (int r = 0; r < W; ++r) a.slot[r] = c.slot[r];
  a.out = c.out;
  a.n = c.n;

  cudaError_t err = cudaSuccess;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  const int sms = current_sm_count(&err);
  if (sms < 1) return err;

  // Vector path when all pointers share the same address mod 16.
  const uintptr_t mis = reinterpret_cast<uintptr_t>(c.out) & 15u;
  bool same = true;
  for (int r = 0; r < W; ++r) same &= (reinterpret_cast<uintptr_t>(c.slot[r]) & 15u) == mis;

  if (same) {
    size_t head = mis ? (16u - mis) / 2u : 0u;
    if (head > c.n) head = c.n;
    a.head = head;
    a.groups = (c.n - head) / 8u;
    const int per_sm = c.out_aliases_slot ? vec_blocks_per_sm<W, true>(dev, &err)
                                          : vec_blocks_per_sm<W, false>(dev, &err);
    if (per_sm < 1) return err;
    const size_t per_block = size_t(kThreads) * Unroll<W>::U;
    size_t blocks = (a.groups + per_block - 1) / per_block;
    const size_t cap = size_t(sms) * size_t(per_sm);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (c.out_aliases_slot)
      reduce_vec_kernel<W, true><<<unsigned(blocks), kThreads, 0, stream>>>(a);
    else
      reduce_vec_kernel<W, false><<<unsigned(blocks), kThreads, 0, stream>>>(a);
  } else {
    size_t blocks = (c.n + kThreads - 1) / kThreads;
    const size_t cap = size_t(sms) * 8u;
    if (blocks > cap) blocks = cap;
    reduce_scalar_kernel<W><<<unsigned(blocks), kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

int current_sm_count(cudaError_t* err) {
  static int cache[kMaxDevices];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return -1;
  if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int sms = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (*err != cudaSuccess || sms < 1) return -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = sms;
  return sms;
}

cudaError_t launch_reduce(const ReduceCall& c, cudaStream_t stream) {
  switch (c.W) {
    case 1: return launch_w<1>(c, stream);
    case 2: return launch_w<2>(c, stream);
    case 3: return launch_w<3>(c, stream);
    case 4: return launch_w<4>(c, stream);
    case 5: return launch_w<5>(c, stream);
    case 6: return launch_w<6>(c, stream);
    case 7: return launch_w<7>(c, stream);
    case 8: return launch_w<8>(c, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace arx
