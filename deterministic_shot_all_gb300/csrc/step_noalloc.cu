// Allocation-free form of the protocol step (see arx.h, arx_step_noalloc).
//
// Some callers cannot allocate device memory when they call the step: a
// serving engine that reserved nearly all of HBM for its own pool at start-up,
// a plug-in whose host framework owns every allocation, or a serving loop
// whose rules forbid allocating after start-up.  cudaMalloc/cudaFree also
// synchronise the device, which a latency-critical caller cannot afford.  For them the step's workspace lives
// in a file-scope static device array of fixed size, which every GPU that
// loads this library holds until the process exits.
//
// Limits: W <= ARX_MAX_W, n <= ARX_NOALLOC_MAX_N elements, at most
// ARX_NOALLOC_MAX_BLOCKS blocks per virtual rank.  Every call shares the
// array: each call first clears the protocol words (so it runs as a fresh
// protocol instance, seq 1) and then stages and reduces; calls that overlap
// on the GPU (different streams, or host threads without ordering) race on
// the array and must not be issued.
#include <cuda_runtime.h>

#include "arx.h"
#include "arx_internal.h"

namespace {

constexpr size_t round_up_c(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxBlocks = ARX_NOALLOC_MAX_BLOCKS;
constexpr size_t kMaxN = ARX_NOALLOC_MAX_N;
// Same layout rules as the context workspace, sized for W = ARX_MAX_W and
// kMaxBlocks blocks per virtual rank.
constexpr size_t kOffEpoch = 256;
constexpr size_t kOffSem = round_up_c(kOffEpoch + size_t(ARX_MAX_W) * kMaxBlocks * 4, 128);
constexpr size_t kOffPad = round_up_c(kOffSem + size_t(ARX_MAX_W) * kMaxBlocks * 128, 128);
constexpr size_t kOffSlots = round_up_c(kOffPad + size_t(ARX_MAX_W) * kMaxBlocks * ARX_MAX_W * 4, 256);
constexpr size_t kSlotStride = round_up_c(kMaxN, 128);
constexpr size_t kScratchBytes = kOffSlots + 2 * size_t(ARX_MAX_W) * kSlotStride * 2;

// The scratch itself.  In host code this name is only a host-side stand-in:
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch in the current device's current context.
// Looked up on every call rather than cached: a context torn down by
// cudaDeviceReset and created again reloads this library's device code at a
// new address, and a cached one would then point at freed memory.  After the
// first call in a context the lookup is a table search in the runtime.
void* scratch_address(arx_status* st) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    *st = arx::report(ARX_ECUDA, "arx_step_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    return nullptr;
  }
  *st = ARX_OK;
  return p;
}

}  // namespace

extern "C" arx_status arx_step_noalloc(const void* const* inputs, int W, void* out, size_t n,
                                       uint32_t* dev_status, void* stream) {
  if (n == 0) return arx::report(ARX_OK, "");
  if (n > kMaxN)
    return arx::report(ARX_EINVAL, "arx_step_noalloc: n=%zu exceeds the static scratch limit of %zu elements",
                       n, kMaxN);
  bool alias = false;
  arx_status st = arx::validate_io(inputs, W, out, n, &alias);
  if (st != ARX_OK) return st;
  if (reinterpret_cast<uintptr_t>(dev_status) & 3u)
    return arx::report(ARX_EINVAL, "arx_step_noalloc: dev_status not 4-byte aligned");

  uint8_t* ws = static_cast<uint8_t*>(scratch_address(&st));
  if (!ws) return st;

  cudaError_t e = cudaSuccess;
  const int sms = arx::current_sm_count(&e);
  const int cap = sms > 0 ? arx::step_capacity(W, &e) : -1;
  if (sms < 1 || cap < 1) return arx::report(ARX_ECUDA, "arx_step_noalloc: device query: %s", cudaGetErrorString(e));
  // About one block per SM over the B x W grid, at least 32 groups of 8
  // elements per reducing block, within the resident capacity and the
  // scratch's block limit.
  size_t B = size_t(sms) / size_t(W);
  const size_t by_work = ((n + 7) / 8 + size_t(W) * 32 - 1) / (size_t(W) * 32);
  if (B > by_work) B = by_work;
  if (B > size_t(cap / W)) B = size_t(cap / W);
  if (B > size_t(kMaxBlocks)) B = kMaxBlocks;
  if (B < 1) B = 1;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's words: clear them so that this call
  // starts a consistent protocol instance whatever W and B the last one used.
  e = cudaMemsetAsync(ws, 0, kOffSlots, s);
  if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_step_noalloc: clear: %s", cudaGetErrorString(e));

  arx::StepCall c{};
  for (int r = 0; r < W; ++r) c.in[r] = static_cast<const uint16_t*>(inputs[r]);
  c.out = static_cast<uint16_t*>(out);
  c.n = n;
  c.ws = ws;
  c.off_epoch = kOffEpoch;
  c.off_sem = kOffSem;
  c.off_pad = kOffPad;
  c.slots = reinterpret_cast<uint16_t*>(ws + kOffSlots);
  c.slot_stride = kSlotStride;
  c.timeout_ns = ARX_DEFAULT_TIMEOUT_NS;
  c.W = W;
  c.B = int(B);
  c.fault_rank = -1;
  ARX_SET_BOUNDS_COUNTER(c);
  e = arx::launch_step(c, s);
  if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_step_noalloc: launch: %s", cudaGetErrorString(e));
  if (dev_status) {
    // The device error word sits at byte 4 of the header.
    e = cudaMemcpyAsync(dev_status, ws + 4, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return arx::report(ARX_ECUDA, "arx_step_noalloc: status copy: %s", cudaGetErrorString(e));
  }
  return arx::report(ARX_OK, "");
}
