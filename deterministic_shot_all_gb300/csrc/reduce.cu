// Stateless W-way bf16 reduce: the HBM-streaming hot kernel.
//
// arx.cu, `arx_kernel`, reduce loop: for each group of 8 elements, load the
// W partials as one 16-byte vector each, add them into 8 fp32 accumulators
// from +0 in rank order, round each to bf16 once and store one 16-byte
// vector.  Each thread reads every slot at a group before it writes that
// group, so the output may be one of the slots.
//
// GB300 design (the pages' fixed grid of at most 8 blocks and 512 KB cap are
// dropped):
//  * persistent grid-stride loop, grid = SMs x resident blocks (capped by the
//    work), coalesced warp accesses per slot, L1 bypassed;
//  * up to 2^22 elements per partial (latency-bound and medium messages):
//    8-byte vectors (4 elements) per slot, one per thread per iteration --
//    twice the threads of the 16-byte form at half the registers each, so
//    more loads are in flight per SM and the message spreads over more SMs;
//    128-thread blocks while 256-thread ones would leave SMs idle; for
//    W <= 4, 8/W (then 16/W) vectors per thread while that keeps the
//    message within one pass of the grid (see launch_policy);
//  * above (bandwidth-bound): 16-byte vectors, U independent groups per
//    thread per iteration, all W*U loads issued before the first add
//    (Little's law against HBM3e latency);
//  * software pipelining (kPipe): the next iteration's loads are in flight
//    while the current groups are summed and stored -- measured best at
//    every W once the body needs more than one pass of the grid;
//  * programmatic dependent launch: the kernel waits on its stream
//    predecessor (griddepcontrol.wait) before touching memory and lets its
//    successor start launching at once, which hides most of the launch gap
//    between back-to-back calls;
//  * before that wait, one thread per block issues bulk L2 prefetches of the
//    block's first chunk of every slot (device or page-locked host buffers),
//    so the next call's DRAM or link latency overlaps the current call -- a
//    prefetch consumes no data, so a predecessor that writes those partials
//    stays correct (the loads come after the wait and read through L2).  W = 8 [32, 4096]:
//    1.60 -> 1.42 us per call; W = 2 at 2^23 elements: 8.76 -> 7.66 us.
// The launch policy (threads, U, kPipe per W and size) comes from a measured
// sweep of these shapes on GB300.
#include <atomic>

#include "arx_device.cuh"
#include "arx_internal.h"

namespace arx {
namespace {

// Kernel arguments.  The 16-byte-aligned body's pointers are computed on the
// host (element `head` of each slot and of out), so the streaming loop does no
// address arithmetic on them: a form that offset the slot pointers in the
// kernel and also used them for the scalar edges after the loop took 46
// instead of 30 registers at W = 8 and ran 30 % slower.
struct VecArgs {
  const uint16_t* body_src[kMaxW];  // element `head` of each slot (16-byte aligned)
  uint16_t* body_dst;               // element `head` of out
  size_t groups;                    // 16-byte groups in the body
  const uint16_t* slot[kMaxW];      // element 0 of each slot (scalar edges)
  uint16_t* out;
  size_t n;        // elements
  size_t head;     // scalar elements before the first 16-byte boundary
  int prefetch_l2; // warm L2 with the slots before the dependency wait
#ifdef ARX_BOUNDS_CHECK
  uint32_t* bounds_counter;
#endif
};

template <int W>
__device__ __forceinline__ void scalar_element(const VecArgs& a, size_t e) {
  float acc = 0.0f;
#pragma unroll
  for (int r = 0; r < W; ++r)
    ARX_CHECKED(a.slot[r] + e, 2, a.slot[r], a.n * 2, a.bounds_counter,
                acc = __fadd_rn(acc, widen16(a.slot[r][e])));
  ARX_CHECKED(a.out + e, 2, a.out, a.n * 2, a.bounds_counter, a.out[e] = round_bf16(acc));
}

template <bool kAlias, typename V>
__device__ __forceinline__ V load_group(const V* p) {
  if constexpr (kAlias) {
    return ld_stream(p);
  } else {
    return ld_stream_nc(p);
  }
}

// Scalar head (before the first 16-byte boundary) and tail (after the last
// full 16-byte group): at most 7 + 7 elements, done by the last block.
template <int W>
__device__ __forceinline__ void head_and_tail(const VecArgs& a) {
  const size_t tail = a.n - a.head - 8 * a.groups;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x < a.head + tail) {
    const size_t t = threadIdx.x;
    const size_t e = t < a.head ? t : a.head + 8 * a.groups + (t - a.head);
    scalar_element<W>(a, e);
  }
}

template <int W, int U, bool kAlias>
__device__ __forceinline__ void load_batch(uint4 (&v)[U][W], const uint4* const (&src)[W], size_t g,
                                           size_t stride, const VecArgs& a) {
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int r = 0; r < W; ++r)
      ARX_CHECKED(src[r] + g + u * stride, 16, a.slot[r], a.n * 2, a.bounds_counter,
                  v[u][r] = load_group<kAlias>(src[r] + g + u * stride));
}

template <int W, int U>
__device__ __forceinline__ void store_batch(uint4* dst, const uint4 (&v)[U][W], size_t g, size_t stride,
                                            const VecArgs& a) {
#pragma unroll
  for (int u = 0; u < U; ++u)
    ARX_CHECKED(dst + g + u * stride, 16, a.out, a.n * 2, a.bounds_counter,
                st_global(dst + g + u * stride, sum_vectors<W>(v[u])));
}

template <int W, int T, int U, bool kPipe, bool kAlias>
__global__ void __launch_bounds__(T) reduce_vec_kernel(const VecArgs a) {
  // As in reduce_half_kernel: the block's first batch (U chunks of T groups
  // per slot) is prefetched into L2 before the dependency wait.
  if (a.prefetch_l2 && threadIdx.x == 0) {
    const size_t stride0 = size_t(gridDim.x) * T;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t first = size_t(blockIdx.x) * T + size_t(u) * stride0;
      if (first < a.groups) {
        const size_t cnt = a.groups - first < size_t(T) ? a.groups - first : size_t(T);
#pragma unroll
        for (int r = 0; r < W; ++r)
          ARX_CHECKED(a.body_src[r] + 8 * first, cnt * 16, a.slot[r], a.n * 2, a.bounds_counter,
                      prefetch_l2_bulk(a.body_src[r] + 8 * first, uint32_t(cnt * 16)));
      }
    }
  }
  dependent_launch_prologue();
  const uint4* src[W];
#pragma unroll
  for (int r = 0; r < W; ++r) src[r] = reinterpret_cast<const uint4*>(a.body_src[r]);
  uint4* dst = reinterpret_cast<uint4*>(a.body_dst);

  const size_t stride = size_t(gridDim.x) * T;
  const size_t step = size_t(U) * stride;
  size_t g = size_t(blockIdx.x) * T + threadIdx.x;
  const size_t G = a.groups;

  if constexpr (kPipe) {
    // Batch i+1's loads are issued before batch i is summed and stored.
    uint4 cur[U][W];
    bool have = g + size_t(U - 1) * stride < G;
    if (have) load_batch<W, U, kAlias>(cur, src, g, stride, a);
    while (have) {
      const size_t gn = g + step;
      const bool more = gn + size_t(U - 1) * stride < G;
      uint4 nxt[U][W];
      if (more) load_batch<W, U, kAlias>(nxt, src, gn, stride, a);
      store_batch<W, U>(dst, cur, g, stride, a);
      g = gn;
      have = more;
      if (more) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int r = 0; r < W; ++r) cur[u][r] = nxt[u][r];
      }
    }
  } else if constexpr (U > 1) {
    for (; g + size_t(U - 1) * stride < G; g += step) {
      uint4 v[U][W];
      load_batch<W, U, kAlias>(v, src, g, stride, a);
      store_batch<W, U>(dst, v, g, stride, a);
    }
  }
  // Remaining groups (fewer than U per thread).
  for (; g < G; g += stride) {
    uint4 v[W];
#pragma unroll
    for (int r = 0; r < W; ++r)
      ARX_CHECKED(src[r] + g, 16, a.slot[r], a.n * 2, a.bounds_counter, v[r] = load_group<kAlias>(src[r] + g));
    ARX_CHECKED(dst + g, 16, a.out, a.n * 2, a.bounds_counter, st_global(dst + g, sum_vectors<W>(v)));
  }

  head_and_tail<W>(a);
}

// 8-byte form: the 16-byte-aligned body as 2 * groups vectors of 4 elements,
// U vectors per slot per thread per iteration (U strides apart), all W * U
// loads issued before the first add.  U = 1 unless the body needs more than
// one pass of the grid and W <= 4; then U = 8 / W (rounded) so each thread
// keeps about 8 loads in flight (Little's law against HBM latency), used
// while one pass of that grid still covers the body; W = 2, 3 have a second
// tier twice as deep.
template <int W, int T, int U, bool kAlias>
__device__ __forceinline__ void reduce_half_body(const VecArgs& a) {
  // Before waiting for the previous kernel of the stream: ask L2 for this
  // block's first chunk (U chunks when U > 1) of every slot, so its DRAM
  // latency overlaps that kernel's tail.  Only a prefetch (no data consumed),
  // so it is safe even when the previous kernel writes these partials: the
  // loads below come after the wait and see its writes through L2.
  const size_t H = 2 * a.groups;
  const size_t stride = size_t(gridDim.x) * T;
  if (a.prefetch_l2 && threadIdx.x == 0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t first = size_t(blockIdx.x) * T + size_t(u) * stride;  // even: T is
      if (first < H) {
        const size_t cnt = (H - first < size_t(T) ? H - first : size_t(T)) & ~size_t(1);
        if (cnt)
#pragma unroll
          for (int r = 0; r < W; ++r)
            ARX_CHECKED(a.body_src[r] + 4 * first, cnt * 8, a.slot[r], a.n * 2, a.bounds_counter,
                        prefetch_l2_bulk(a.body_src[r] + 4 * first, uint32_t(cnt * 8)));
      }
    }
  }
  dependent_launch_prologue();
  const uint2* src[W];
#pragma unroll
  for (int r = 0; r < W; ++r) src[r] = reinterpret_cast<const uint2*>(a.body_src[r]);
  uint2* dst = reinterpret_cast<uint2*>(a.body_dst);
  for (size_t h = size_t(blockIdx.x) * T + threadIdx.x; h < H; h += size_t(U) * stride) {
    uint2 v[U][W];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t hu = h + size_t(u) * stride;
      if (hu < H)
#pragma unroll
        for (int r = 0; r < W; ++r)
          ARX_CHECKED(src[r] + hu, 8, a.slot[r], a.n * 2, a.bounds_counter, v[u][r] = load_group<kAlias>(src[r] + hu));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t hu = h + size_t(u) * stride;
      if (hu < H) ARX_CHECKED(dst + hu, 8, a.out, a.n * 2, a.bounds_counter, st_global(dst + hu, sum_halves<W>(v[u])));
    }
  }
  head_and_tail<W>(a);
}

template <int W, int T, int U, bool kAlias>
__global__ void __launch_bounds__(T) reduce_half_kernel(const VecArgs a) {
  reduce_half_body<W, T, U, kAlias>(a);
}

// The 16-load form (W * U = 16) under a register bound that keeps four
// blocks resident per SM (64 registers; left to itself it takes 69 and fits
// three).  A separate entry point because a minimum-blocks bound on the
// other instances changes their register allocation too.
template <int W, int T, int U, bool kAlias>
__global__ void __launch_bounds__(T, 4) reduce_half_deep_kernel(const VecArgs a) {
  reduce_half_body<W, T, U, kAlias>(a);
}

// Pointers with different addresses mod 16: one element per thread per step.
template <int W>
__global__ void __launch_bounds__(kThreads) reduce_scalar_kernel(const VecArgs a) {
  dependent_launch_prologue();
  const size_t stride = size_t(gridDim.x) * kThreads;
  for (size_t e = size_t(blockIdx.x) * kThreads + threadIdx.x; e < a.n; e += stride)
    scalar_element<W>(a, e);
}

constexpr int kMaxDevices = 64;

template <typename Kernel>
int blocks_per_sm(Kernel k, int threads, int dev, std::atomic<int>* cache, cudaError_t* err) {
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int b = 0;
  *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, threads, 0);
  if (*err != cudaSuccess || b < 1) return -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(b, std::memory_order_relaxed);
  return b;
}

// Launch with the programmatic-stream-serialisation attribute (see
// dependent_launch_prologue).
template <typename Kernel>
cudaError_t launch_dependent(Kernel k, size_t blocks, int threads, cudaStream_t stream, const VecArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(blocks), 1, 1);
  cfg.blockDim = dim3(unsigned(threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

template <int W, int T, int U, bool kPipe, bool kAlias>
cudaError_t launch_vec(const VecArgs& a, int dev, int sms, cudaStream_t stream) {
  static std::atomic<int> cache[kMaxDevices];
  cudaError_t err = cudaSuccess;
  auto k = reduce_vec_kernel<W, T, U, kPipe, kAlias>;
  const int per_sm = blocks_per_sm(k, T, dev, cache, &err);
  if (per_sm < 1) return err;
  const size_t per_block = size_t(T) * U;
  size_t blocks = (a.groups + per_block - 1) / per_block;
  const size_t cap = size_t(sms) * size_t(per_sm);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_dependent(k, blocks, T, stream, a);
}

// 8-byte vectors per slot per thread per iteration of the batched 8-byte
// form: about 8 loads in flight per thread at every W.
template <int W>
constexpr int kHalfU = W >= 5 ? 1 : W >= 3 ? 2 : W == 2 ? 4 : 8;
// A second batched tier, twice as deep, where its one-pass reach is larger
// despite the lower residency its registers allow (W = 2, 3); 0 = none.
template <int W>
constexpr int kHalfU2 = W == 2 || W == 3 ? 2 * kHalfU<W> : 0;

// Launches the 8-byte form with U vectors per slot per thread if one pass
// of its grid (SMs x resident blocks x T threads x U) covers the body --
// with 1/16 slack: a second pass for a few threads costs little, one for a
// fifth of them 10-30 % -- or always when `force`.  Sets *taken; returns
// the launch status.
template <int W, int T, int U, bool kAlias>
cudaError_t launch_half(const VecArgs& a, int dev, int sms, bool force, bool* taken,
                        cudaStream_t stream) {
  static std::atomic<int> cache[kMaxDevices];
  cudaError_t err = cudaSuccess;
  *taken = false;
  void (*k)(VecArgs) = nullptr;
  if constexpr (W * U >= 16) {
    k = reduce_half_deep_kernel<W, T, U, kAlias>;
  } else {
    k = reduce_half_kernel<W, T, U, kAlias>;
  }
  const int per_sm = blocks_per_sm(k, T, dev, cache, &err);
  if (per_sm < 1) return err;
  size_t blocks = (2 * a.groups + T - 1) / T;
  const size_t cap = size_t(sms) * size_t(per_sm);
  if (!force && blocks * 16u > cap * size_t(U) * 17u) return cudaSuccess;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  *taken = true;
  return launch_dependent(k, blocks, T, stream, a);
}

// Measured policy (launch-shape sweeps of W = 2, 4, 8 from 2^15 to 2^27
// elements per partial, and a sweep of W = 1-4 from 2^20.5 to 2^22 in
// quarter powers, on GB300, CUDA-graph replays, inputs beyond L2):
//  n <= 2^22: the 8-byte form, 128 threads per block while blocks of 256
//             would number fewer than the SMs (W = 8 at 2^12 - 2^17 elements:
//             2.6-7.3 % faster than 256; 64 threads gained less), else 256.
//             W = 5-7: one vector per slot per thread.
//             W = 8: one vector while one pass of the grid covers the body
//             (+ 1/16), else the pipelined 16-byte form below: 0.97-1.03
//             against 0.77-0.92 of the copy rate from 2^20.75 to 2^22 (a
//             second pass of the 8-byte form waits for its first loads;
//             the pipelined form keeps the next group's loads in flight).
//             At W = 5-7 it won only at some of those sizes and lost at
//             others (W = 7 at 2^20.5: 0.74 against 0.88), so they keep the
//             one-vector form.
//             W <= 4: one vector while one pass of the grid covers the
//             body, else kHalfU<W> vectors while one pass covers it, else
//             the 16-byte form below -- the batched form saves 5-20 % over
//             the 16-byte one while it makes one pass (+ 1/16), and costs
//             10-30 % once a fifth of its threads need a second (those
//             threads load again only after their first loads returned, at
//             the end of the burst).
//  above:     16-byte groups -- W <= 2: 128 threads, U = 2, pipelined;
//             W >= 3: 256 threads, U = 1, pipelined (for W >= 5 it replaced
//             U = 2 without pipelining: +3-10 % from 2^22.5 to 2^25, equal
//             at 2^26, within 0.5 % at 2^27).
constexpr size_t kHalfMaxElems = size_t(1) << 22;

template <int W, bool kAlias>
cudaError_t launch_policy(const VecArgs& a, int dev, int sms, cudaStream_t stream) {
  if (a.n <= kHalfMaxElems) {
    bool taken = false;
    cudaError_t err;
    if ((2 * a.groups + 255) / 256 < size_t(sms)) {
      // Blocks of 256 would leave SMs idle: 128-thread blocks spread the
      // message (and its L2 prefetches) over twice as many SMs.
      return launch_half<W, 128, 1, kAlias>(a, dev, sms, true, &taken, stream);
    }
    err = launch_half<W, 256, 1, kAlias>(a, dev, sms, W >= 5 && W < 8, &taken, stream);
    if (err != cudaSuccess || taken) return err;
    if constexpr (kHalfU<W> > 1) {
      err = launch_half<W, 256, kHalfU<W>, kAlias>(a, dev, sms, false, &taken, stream);
      if (err != cudaSuccess || taken) return err;
    }
    if constexpr (kHalfU2<W> > 1) {
      err = launch_half<W, 256, kHalfU2<W>, kAlias>(a, dev, sms, false, &taken, stream);
      if (err != cudaSuccess || taken) return err;
    }
  }
  if constexpr (W <= 2) {
    return launch_vec<W, 128, 2, true, kAlias>(a, dev, sms, stream);
  } else {
    return launch_vec<W, 256, 1, true, kAlias>(a, dev, sms, stream);
  }
}

template <int W>
cudaError_t launch_w(const ReduceCall& c, cudaStream_t stream) {
  VecArgs a{};
  for (int r = 0; r < W; ++r) a.slot[r] = c.slot[r];
  a.out = c.out;
  a.n = c.n;
  a.prefetch_l2 = c.prefetch_l2 ? 1 : 0;
#ifdef ARX_BOUNDS_CHECK
  a.bounds_counter = c.bounds_counter;
#endif

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
    for (int r = 0; r < W; ++r) a.body_src[r] = c.slot[r] + head;
    a.body_dst = c.out + head;
    err = c.out_aliases_slot ? launch_policy<W, true>(a, dev, sms, stream)
                             : launch_policy<W, false>(a, dev, sms, stream);
    if (err != cudaSuccess) return err;
  } else {
    size_t blocks = (c.n + kThreads - 1) / kThreads;
    const size_t cap = size_t(sms) * 8u;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_dependent(reduce_scalar_kernel<W>, blocks, kThreads, stream, a);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace

int current_sm_count(cudaError_t* err) {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return -1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (*err != cudaSuccess || sms < 1) return -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
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
