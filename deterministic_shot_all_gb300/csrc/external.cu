// External-writer form of the step: partials written into page-locked host
// memory by another agent, reduced by the GPU (see arx.h, arx_ext_*).
//
// arx.cu's design on GB10: for step seq the GPU publishes seq; a CPU proxy
// has every peer's partial written (RDMA) into pinned recv[seq & 1][rank]
// and then raises flag[rank]; the kernel's wait phase spins on those flags
// with system-scope acquire loads, and the reduce loop reads the slots with
// cache-bypassing loads, because another agent wrote them.  On one GB300 the
// writer is a host thread standing in for the proxy and the NIC: it copies
// each virtual rank's partial into the page-locked recv[seq & 1][r] and then
// release-stores flag[r] = seq; the GPU waits for every flag with bounded
// ld.acquire.sys polls, reduces over the slots with ld.global.cv, and its
// last block out stores the step's seq as `consumed` with a system-scope
// release, which tells the writer that bank seq & 1 may be written again
// (for step seq + 2).
//
// Host region (page-locked, zero-filled before the first step):
//   [0, 512)      uint32 flag[r] at byte 64 * r (one cache line each)
//   [512, 516)    uint32 consumed (last step whose slots the GPU has read)
//   [1024, ...)   bf16 recv[2][W][slot_stride]
// Device words (HBM, zero-filled): header uint32 seq (completed), err,
//   blocks (blocks out).
#include <cuda_runtime.h>

#include <chrono>
#include <cstring>
#include <thread>

#include "arx.h"
#include "arx_device.cuh"
#include "arx_internal.h"

namespace arx {
namespace {

constexpr uint32_t kExtMagic = 0x41525845u;  // "ARXE"
constexpr size_t kFlagStride = 64;            // bytes between two flags
constexpr size_t kConsumedOff = 512;
constexpr size_t kRecvOff = 1024;
constexpr size_t kWordsBytes = 256;
constexpr uint32_t kErrTimeout = 4;
constexpr uint32_t kStageExtWait = 11;        // error-word stage of the flag wait

struct ExtArgs {
  const uint32_t* flags;   // device address of flag[0] (stride kFlagStride / 4 words)
  uint32_t* consumed;      // device address of `consumed`
  const uint16_t* recv;    // device address of recv[0][0]
  uint16_t* out;
  uint32_t* words;         // seq, err, blocks
  size_t n;
  uint64_t slot_stride;    // elements
  uint64_t timeout_ns;
  int out_vec;             // out 16-byte aligned
#ifdef ARX_BOUNDS_CHECK
  uint32_t* bounds_counter;
  size_t recv_elems;
#endif
};

__device__ __forceinline__ void ext_error(uint32_t* err, uint32_t rank, uint32_t block) {
  atomicCAS(err, 0u, kErrTimeout | (kStageExtWait << 8) | ((rank & 15u) << 12) | ((block & 0xFFFFu) << 16));
}

template <int W>
__global__ void __launch_bounds__(kThreads) ext_step_kernel(const ExtArgs a) {
  const uint32_t tid = threadIdx.x;
  uint32_t* seq_done = a.words;
  uint32_t* err = a.words + 1;
  uint32_t* blocks_out = a.words + 2;
  __shared__ uint32_t s_seq;

  // Thread q < W loads flag[q] before the dependency wait (the writer, not
  // the previous kernel, stores the flags, so the wait orders nothing for
  // them): the load's host round trip overlaps the wait, and a value that
  // already covers this step skips the poll below.  The load is a
  // system-scope acquire like the poll's, so the slot reads that follow it
  // in program order (and, past the block barrier, in the other threads)
  // see the writer's data.  13.90 against 14.54 us per step with the first
  // load after the wait (W = 8 [32, 4096], writer up to two steps ahead,
  // A/B in one process, GB300).
  uint32_t flag_pre = 0;
  if (tid < uint32_t(W)) flag_pre = ld_acquire_sys(a.flags + tid * (kFlagStride / 4));

  // Wait for the previous kernel of the stream (the previous step finished
  // and stored its seq), then let the next one begin launching.
  dependent_launch_prologue();

  // 1. seq / parity: this step's number and bank.
  if (tid == 0) s_seq = ld_relaxed_gpu(seq_done) + 1u;
  __syncthreads();
  const uint32_t seq = s_seq;

  // 2. wait phase: thread q < W waits until the writer has raised flag[q] to
  // this step (or beyond: it may already have posted the next step into the
  // other bank), with system-scope acquire polls, bounded.  On expiry the
  // block records ARX_ETIMEOUT and reduces whatever the slots hold.
  if (tid < uint32_t(W) && int32_t(flag_pre - seq) < 0) {
    const uint32_t* f = a.flags + tid * (kFlagStride / 4);
    const uint64_t t0 = global_timer_ns();
    const uint64_t cap = spin_cap(a.timeout_ns);
    for (uint64_t spins = 0;; ++spins) {
      if (int32_t(ld_acquire_sys(f) - seq) >= 0) break;
      if ((spins & 15u) == 15u) {
        if (global_timer_ns() - t0 > a.timeout_ns || spins > cap) {
          ext_error(err, tid, blockIdx.x);
          break;
        }
        backoff(spins);
      }
    }
  }
  __syncthreads();

  // 3. reduce over recv[seq & 1][0..W-1] in rank order, cache-bypassing loads.
  const uint16_t* bank = a.recv + size_t(seq & 1u) * size_t(W) * a.slot_stride;
  const size_t G = a.n / 8u;
  const uint4* src[W];
#pragma unroll
  for (int q = 0; q < W; ++q) src[q] = reinterpret_cast<const uint4*>(bank + size_t(q) * a.slot_stride);
  const size_t step = size_t(gridDim.x) * kThreads;
  for (size_t g = size_t(blockIdx.x) * kThreads + tid; g < G; g += step) {
    uint4 v[W];
#pragma unroll
    for (int q = 0; q < W; ++q)
      ARX_CHECKED(src[q] + g, 16, a.recv, a.recv_elems * 2, a.bounds_counter, v[q] = ld_cv(src[q] + g));
    const uint4 o = sum_vectors<W>(v);
    if (a.out_vec) {
      ARX_CHECKED(reinterpret_cast<uint4*>(a.out) + g, 16, a.out, a.n * 2, a.bounds_counter,
                  st_global(reinterpret_cast<uint4*>(a.out) + g, o));
    } else {
      uint16_t* d = a.out + 8u * g;
      ARX_CHECKED(d, 16, a.out, a.n * 2, a.bounds_counter, {
        d[0] = uint16_t(o.x & 0xFFFFu);
        d[1] = uint16_t(o.x >> 16);
        d[2] = uint16_t(o.y & 0xFFFFu);
        d[3] = uint16_t(o.y >> 16);
        d[4] = uint16_t(o.z & 0xFFFFu);
        d[5] = uint16_t(o.z >> 16);
        d[6] = uint16_t(o.w & 0xFFFFu);
        d[7] = uint16_t(o.w >> 16);
      });
    }
  }
  if (blockIdx.x == gridDim.x - 1u && tid < a.n - 8u * G) {
    const size_t e = 8u * G + tid;
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < W; ++q)
      ARX_CHECKED(bank + size_t(q) * a.slot_stride + e, 2, a.recv, a.recv_elems * 2, a.bounds_counter,
                  acc = __fadd_rn(acc, widen16(ld_cv16(bank + size_t(q) * a.slot_stride + e))));
    ARX_CHECKED(a.out + e, 2, a.out, a.n * 2, a.bounds_counter, a.out[e] = round_bf16(acc));
  }

  // 4. exit: count blocks out (acquire-release at GPU scope: every block's
  // reads of the bank happen before the last block's count); the last block
  // stores seq as completed and, with a system-scope release, as `consumed`,
  // after which the writer may overwrite this bank for step seq + 2.
  __syncthreads();
  if (tid == 0 && atom_add_acq_rel_gpu(blocks_out, 1u) == gridDim.x - 1u) {
    *blocks_out = 0u;
    st_relaxed_gpu(seq_done, seq);
    st_release_sys(a.consumed, seq);
  }
}

template <int W>
cudaError_t launch_ext_w(const ExtArgs& a, int blocks, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, ext_step_kernel<W>, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ext(int W, const ExtArgs& a, int blocks, cudaStream_t stream) {
  switch (W) {
    case 1: return launch_ext_w<1>(a, blocks, stream);
    case 2: return launch_ext_w<2>(a, blocks, stream);
    case 3: return launch_ext_w<3>(a, blocks, stream);
    case 4: return launch_ext_w<4>(a, blocks, stream);
    case 5: return launch_ext_w<5>(a, blocks, stream);
    case 6: return launch_ext_w<6>(a, blocks, stream);
    case 7: return launch_ext_w<7>(a, blocks, stream);
    case 8: return launch_ext_w<8>(a, blocks, stream);
    default: return cudaErrorInvalidValue;
  }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t slot_stride_for(size_t max_n) { return round_up(max_n > 0 ? max_n : 1, 128); }

arx_status check_ext(const arx_ext* x) {
  if (!x || x->magic != kExtMagic) return report(ARX_ESTATE, "external-writer context not initialised");
  return ARX_OK;
}

uint8_t* host_base(const arx_ext* x) { return static_cast<uint8_t*>(x->host_region); }

uint32_t* host_flag(const arx_ext* x, int r) {
  return reinterpret_cast<uint32_t*>(host_base(x) + size_t(r) * kFlagStride);
}

uint32_t* host_consumed(const arx_ext* x) { return reinterpret_cast<uint32_t*>(host_base(x) + kConsumedOff); }

uint16_t* host_slot(const arx_ext* x, uint32_t seq, int r) {
  return reinterpret_cast<uint16_t*>(host_base(x) + kRecvOff) +
         (size_t(seq & 1u) * size_t(x->W) + size_t(r)) * x->slot_stride;
}

}  // namespace
}  // namespace arx

extern "C" {

size_t arx_ext_region_bytes(int W, size_t max_n) {
  if (W < 1 || W > ARX_MAX_W || max_n > (SIZE_MAX / 8) / (2 * ARX_MAX_W)) return 0;
  return arx::kRecvOff + 2 * size_t(W) * arx::slot_stride_for(max_n) * 2;
}

size_t arx_ext_words_bytes(void) { return arx::kWordsBytes; }

arx_status arx_ext_init(arx_ext* x, void* dev_words, size_t words_bytes, void* host_region,
                        size_t region_bytes, int W, size_t max_n, int nblocks) {
  if (!x) return arx::report(ARX_EINVAL, "null external-writer context");
  std::memset(x, 0, sizeof *x);
  if (W < 1 || W > ARX_MAX_W) return arx::report(ARX_EINVAL, "W=%d outside 1..%d", W, ARX_MAX_W);
  if (nblocks < 0) return arx::report(ARX_EINVAL, "nblocks=%d is negative", nblocks);
  if (!dev_words || (reinterpret_cast<uintptr_t>(dev_words) & 255u))
    return arx::report(ARX_EINVAL, "device words missing or not 256-byte aligned");
  if (words_bytes < arx::kWordsBytes)
    return arx::report(ARX_EINVAL, "device words %zu bytes, need %zu", words_bytes, arx::kWordsBytes);
  const size_t need = arx_ext_region_bytes(W, max_n);
  if (need == 0) return arx::report(ARX_EINVAL, "max_n=%zu too large", max_n);
  if (!host_region || (reinterpret_cast<uintptr_t>(host_region) & 255u))
    return arx::report(ARX_EINVAL, "host region missing or not 256-byte aligned");
  if (region_bytes < need) return arx::report(ARX_EINVAL, "host region %zu bytes, need %zu", region_bytes, need);
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, host_region) != cudaSuccess) {
    cudaGetLastError();
    return arx::report(ARX_EINVAL, "host region is not page-locked memory known to CUDA");
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer)
    return arx::report(ARX_EINVAL, "host region is not page-locked memory known to CUDA");
  int B = nblocks;
  if (B == 0) {
    // One 16-byte group of every rank per thread, at most one block per SM.
    cudaError_t e = cudaSuccess;
    const int sms = arx::current_sm_count(&e);
    if (sms < 1) return arx::report(ARX_ECUDA, "arx_ext_init device query: %s", cudaGetErrorString(e));
    const size_t groups = (max_n + 7) / 8;
    size_t b = (groups + arx::kThreads - 1) / arx::kThreads;
    if (b > size_t(sms)) b = size_t(sms);
    B = b < 1 ? 1 : int(b);
  }
  x->magic = arx::kExtMagic;
  x->W = W;
  x->nblocks = B;
  x->max_n = max_n;
  x->slot_stride = arx::slot_stride_for(max_n);
  x->timeout_ns = ARX_DEFAULT_TIMEOUT_NS;
  x->words = dev_words;
  x->host_region = host_region;
  x->dev_region = at.devicePointer;
  x->region_bytes = region_bytes;
  return arx::report(ARX_OK, "");
}

arx_status arx_ext_set_timeout(arx_ext* x, uint64_t ns) {
  const arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  if (ns == 0) return arx::report(ARX_EINVAL, "timeout must be > 0");
  x->timeout_ns = ns;
  return arx::report(ARX_OK, "");
}

void* arx_ext_slot(const arx_ext* x, uint32_t seq, int rank) {
  if (arx::check_ext(x) != ARX_OK || rank < 0 || rank >= x->W) return nullptr;
  return arx::host_slot(x, seq, rank);
}

arx_status arx_ext_wait_free(const arx_ext* x, uint32_t seq, uint64_t wait_ns) {
  const arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  // Bank seq & 1 was last read by step seq - 2; it is free once the GPU has
  // consumed that step (steps 1 and 2 find both banks free).
  const uint32_t need = seq - 2u;
  const uint32_t* consumed = arx::host_consumed(x);
  using clock = std::chrono::steady_clock;
  const auto t0 = clock::now();
  for (uint64_t spins = 0;; ++spins) {
    if (int32_t(__atomic_load_n(consumed, __ATOMIC_ACQUIRE) - need) >= 0) return arx::report(ARX_OK, "");
    if ((spins & 63u) == 63u) {
      const auto waited = std::chrono::duration_cast<std::chrono::nanoseconds>(clock::now() - t0).count();
      if (uint64_t(waited) >= wait_ns)
        return arx::report(ARX_ETIMEOUT, "bank of step %u still in use: the GPU has consumed step %u", seq,
                           __atomic_load_n(consumed, __ATOMIC_RELAXED));
      if (spins > 4096u) std::this_thread::yield();
    }
  }
}

arx_status arx_ext_publish(const arx_ext* x, int rank, uint32_t seq) {
  const arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  if (rank < 0 || rank >= x->W) return arx::report(ARX_EINVAL, "rank %d outside 0..%d", rank, x->W - 1);
  // Release: the slot's contents, written before, are visible to the GPU's
  // system-scope acquire of the flag.
  __atomic_store_n(arx::host_flag(x, rank), seq, __ATOMIC_RELEASE);
  return arx::report(ARX_OK, "");
}

arx_status arx_ext_publish_all(const arx_ext* x, uint32_t seq, uint64_t wait_ns) {
  const arx_status s = arx_ext_wait_free(x, seq, wait_ns);
  if (s != ARX_OK) return s;
  for (int r = 0; r < x->W; ++r) __atomic_store_n(arx::host_flag(x, r), seq, __ATOMIC_RELEASE);
  return arx::report(ARX_OK, "");
}

arx_status arx_ext_post(const arx_ext* x, int rank, uint32_t seq, const void* src, size_t n,
                        uint64_t wait_ns) {
  arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  if (rank < 0 || rank >= x->W) return arx::report(ARX_EINVAL, "rank %d outside 0..%d", rank, x->W - 1);
  if (n > x->max_n) return arx::report(ARX_EINVAL, "n=%zu exceeds max_n=%llu", n,
                                       static_cast<unsigned long long>(x->max_n));
  if (n > 0 && !src) return arx::report(ARX_EINVAL, "null source");
  s = arx_ext_wait_free(x, seq, wait_ns);
  if (s != ARX_OK) return s;
  if (n > 0) std::memcpy(arx::host_slot(x, seq, rank), src, n * 2);
  return arx_ext_publish(x, rank, seq);
}

arx_status arx_ext_step(arx_ext* x, void* out, size_t n, void* stream) {
  arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  if (x->failed_err != 0)
    return arx::report(ARX_ESTATE, "the context failed (device error word 0x%08x); arx_ext_reset it first",
                       x->failed_err);
  if (n == 0) return arx::report(ARX_OK, "");
  if (n > x->max_n) return arx::report(ARX_EINVAL, "n=%zu exceeds max_n=%llu", n,
                                       static_cast<unsigned long long>(x->max_n));
  if (!out || (reinterpret_cast<uintptr_t>(out) & 1u))
    return arx::report(ARX_EINVAL, "output missing or not 2-byte aligned");
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + n * 2;
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(x->dev_region), r1 = r0 + x->region_bytes;
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(x->words), w1 = w0 + arx::kWordsBytes;
  if (!(o1 <= r0 || r1 <= o0) || !(o1 <= w0 || w1 <= o0))
    return arx::report(ARX_EOVERLAP, "output overlaps the host region or the device words");
  uint8_t* region = static_cast<uint8_t*>(x->dev_region);
  arx::ExtArgs a{};
  a.flags = reinterpret_cast<const uint32_t*>(region);
  a.consumed = reinterpret_cast<uint32_t*>(region + arx::kConsumedOff);
  a.recv = reinterpret_cast<const uint16_t*>(region + arx::kRecvOff);
  a.out = static_cast<uint16_t*>(out);
  a.words = static_cast<uint32_t*>(x->words);
  a.n = n;
  a.slot_stride = x->slot_stride;
  a.timeout_ns = x->timeout_ns;
  a.out_vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
#ifdef ARX_BOUNDS_CHECK
  a.recv_elems = 2 * size_t(x->W) * x->slot_stride;
  cudaError_t be = cudaSuccess;
  a.bounds_counter = arx::bounds_counter(&be);
  if (!a.bounds_counter) return arx::report(ARX_ECUDA, "bounds counter lookup: %s", cudaGetErrorString(be));
#endif
  int blocks = x->nblocks;
  const size_t groups = (n + 7) / 8;
  const size_t need = (groups + arx::kThreads - 1) / arx::kThreads;
  if (size_t(blocks) > need) blocks = need < 1 ? 1 : int(need);
  const cudaError_t e = arx::launch_ext(x->W, a, blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_ext_step launch: %s", cudaGetErrorString(e));
  return arx::report(ARX_OK, "");
}

arx_status arx_ext_query(arx_ext* x, uint32_t* seq, uint32_t* dev_err, void* stream) {
  const arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t w[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(w, x->words, sizeof w, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_ext_query: %s", cudaGetErrorString(e));
  if (seq) *seq = w[0];
  if (dev_err) *dev_err = w[1];
  if ((w[1] & 0xFFu) == 0) return arx::report(ARX_OK, "");
  x->failed_err = w[1];
  return arx::report((w[1] & 0xFFu) == ARX_ETIMEOUT ? ARX_ETIMEOUT : ARX_ESTATE,
                     "device error word 0x%08x (stage %u, rank %u, block %u)", w[1], (w[1] >> 8) & 15u,
                     (w[1] >> 12) & 15u, w[1] >> 16);
}

arx_status arx_ext_reset(arx_ext* x, void* stream) {
  const arx_status s = arx::check_ext(x);
  if (s != ARX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(x->words, 0, arx::kWordsBytes, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_ext_reset: %s", cudaGetErrorString(e));
  for (int r = 0; r < x->W; ++r) __atomic_store_n(arx::host_flag(x, r), 0u, __ATOMIC_RELAXED);
  __atomic_store_n(arx::host_consumed(x), 0u, __ATOMIC_RELEASE);
  x->failed_err = 0;
  return arx::report(ARX_OK, "");
}

}  // extern "C"
