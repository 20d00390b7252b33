// Host-side interface between the C ABI layer and the kernel launchers.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "arx.h"

namespace arx {

// Argument checks shared by the C entry points (see abi.cu).
arx_status validate_io(const void* const* in, int W, const void* out, size_t n, bool* out_alias);

// Sets the calling thread's arx_last_error() text and returns `s`.
arx_status report(arx_status s, const char* fmt, ...);

// One stateless reduce: out[i] = bf16(sum_r slot[r][i]) for 0 <= i < n.
struct ReduceCall {
  const uint16_t* slot[8];
  uint16_t* out;
  size_t n;
  int W;
  bool out_aliases_slot;  // out equals one slot pointer
  bool prefetch_l2;       // the kernel may prefetch its slots into L2 before the dependency wait
#ifdef ARX_BOUNDS_CHECK
  uint32_t* bounds_counter;
#endif
};

// Enqueues the reduce on `stream`.  Picks the vector kernel when every
// pointer has the same address mod 16, else the scalar kernel.
cudaError_t launch_reduce(const ReduceCall& c, cudaStream_t stream);

// One protocol step (see arx.h, arx_step).
struct StepCall {
  const uint16_t* in[8];
  uint16_t* out;
  size_t n;
  uint8_t* ws;
  uint16_t* slots;  // slots[2][W][slot_stride] (device address; may be page-locked host memory)
  uint64_t off_epoch, off_sem, off_pad, slot_stride;
  uint64_t timeout_ns;
  int W, B;
  int fault_rank;
  int sync_mode;  // ARX_SYNC_*
  int stagger;    // K >= 2: K block groups start staging in turn (slots in host memory); else 0
  uint64_t stagger_ns;  // time between two groups' starts
#ifdef ARX_BOUNDS_CHECK
  uint32_t* bounds_counter;
#endif
};

cudaError_t launch_step(const StepCall& c, cudaStream_t stream);

// Most blocks of the step kernel for W ranks that can be resident at once on
// the current device (SMs x blocks per SM), or a negative value on error.
int step_capacity(int W, cudaError_t* err);

// Most clusters of (1, W, 1) step blocks that can be resident at once on the
// current device (the cluster-launched variants), or a negative value on error.
int step_cluster_capacity(int W, cudaError_t* err);

// SM count of the current device (cached per device ordinal).
int current_sm_count(cudaError_t* err);

#ifdef ARX_BOUNDS_CHECK
// Device address of the checking build's violation counter on the current
// device, or nullptr with *err set.
uint32_t* bounds_counter(cudaError_t* err);

// Sets call.bounds_counter, or returns ARX_ECUDA from the enclosing function.
#define ARX_SET_BOUNDS_COUNTER(call)                                              \
  do {                                                                           \
    cudaError_t e_ = cudaSuccess;                                                \
    (call).bounds_counter = ::arx::bounds_counter(&e_);                          \
    if (!(call).bounds_counter)                                                  \
      return ::arx::report(ARX_ECUDA, "bounds counter lookup: %s", cudaGetErrorString(e_)); \
  } while (0)
#else
#define ARX_SET_BOUNDS_COUNTER(call) \
  do {                               \
  } while (0)
#endif

}  // namespace arx
