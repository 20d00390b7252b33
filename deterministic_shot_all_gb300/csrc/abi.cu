// C ABI of libarx: argument checks on the host, then kernel launches.
//
// Mirrors the checks of arx.cu's `arx_allreduce` (bf16, contiguous, equal
// sizes, world size bounds) as status codes instead of exceptions or exit(),
// and drops its 512 KB / multiple-of-8 limits.
#include <cuda_runtime.h>

#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <thread>

#include "arx.h"
#include "arx_internal.h"
#ifdef ARX_BOUNDS_CHECK
#include "arx_device.cuh"
#endif

namespace {

constexpr uint32_t kCtxMagic = 0x41525843u;  // "ARXC"
constexpr size_t kHeaderBytes = 256;

thread_local char g_last_error[256];

arx_status fail(arx_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

arx_status fail_cuda(cudaError_t e, const char* what) {
  return fail(ARX_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

arx_status ok() {
  g_last_error[0] = '\0';
  return ARX_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// [p, p + bytes) and [q, q + bytes): 0 disjoint, 1 identical, 2 partial overlap.
int overlap_kind(const void* p, const void* q, size_t pbytes, size_t qbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + pbytes;
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(q), b1 = b0 + qbytes;
  if (a1 <= b0 || b1 <= a0) return 0;
  if (a0 == b0 && pbytes == qbytes) return 1;
  return 2;
}

// Common checks of the W input pointers and the output.
arx_status check_io(const void* const* in, int W, const void* out, size_t n, bool* out_alias) {
  if (W < 1 || W > ARX_MAX_W) return fail(ARX_EINVAL, "W=%d outside 1..%d", W, ARX_MAX_W);
  if (!in) return fail(ARX_EINVAL, "null pointer array");
  if (!out) return fail(ARX_EINVAL, "null output pointer");
  if (reinterpret_cast<uintptr_t>(out) & 1u) return fail(ARX_EINVAL, "output not 2-byte aligned");
  if (n > (SIZE_MAX / 2) / 2) return fail(ARX_EINVAL, "n=%zu too large", n);
  const size_t bytes = n * 2;
  *out_alias = false;
  for (int r = 0; r < W; ++r) {
    if (!in[r]) return fail(ARX_EINVAL, "null input pointer %d", r);
    if (reinterpret_cast<uintptr_t>(in[r]) & 1u) return fail(ARX_EINVAL, "input %d not 2-byte aligned", r);
    const int k = overlap_kind(out, in[r], bytes, bytes);
    if (k == 2) return fail(ARX_EOVERLAP, "output partially overlaps input %d", r);
    if (k == 1) *out_alias = true;
  }
  return ARX_OK;
}

}  // namespace

#ifdef ARX_BOUNDS_CHECK
namespace {

// Accesses the checking build skipped because their address fell outside
// their buffer (one counter per device, in this library's device image).
__device__ uint32_t g_bounds_violations;

__global__ void bounds_probe_kernel(uint32_t* counter, const uint16_t* base) {
  // One address past the end of an 8-element buffer: counted, never accessed.
  ARX_CHECKED(base + 8, 2, base, 16, counter, atomicAdd(counter, uint32_t(base[8])));
}

}  // namespace
#endif

namespace arx {

#ifdef ARX_BOUNDS_CHECK
// Looked up on every call, not cached: after cudaDeviceReset the context is
// created again and the counter has a new address.
uint32_t* bounds_counter(cudaError_t* err) {
  void* q = nullptr;
  *err = cudaGetSymbolAddress(&q, g_bounds_violations);
  if (*err != cudaSuccess || !q) return nullptr;
  return static_cast<uint32_t*>(q);
}
#endif

// For entry points defined in other translation units: the same argument
// checks and per-thread error text as the entry points here.
arx_status validate_io(const void* const* in, int W, const void* out, size_t n, bool* out_alias) {
  return check_io(in, W, out, n, out_alias);
}

arx_status report(arx_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace arx

extern "C" {

const char* arx_status_string(arx_status s) {
  switch (s) {
    case ARX_OK: return "ARX_OK";
    case ARX_EINVAL: return "ARX_EINVAL: invalid argument";
    case ARX_EOVERLAP: return "ARX_EOVERLAP: output partially overlaps an input";
    case ARX_ECUDA: return "ARX_ECUDA: CUDA error";
    case ARX_ETIMEOUT: return "ARX_ETIMEOUT: a bounded device wait expired";
    case ARX_ESTATE: return "ARX_ESTATE: inconsistent protocol state";
  }
  return "ARX_?: unknown status";
}

const char* arx_last_error(void) { return g_last_error; }

arx_status arx_reduce(const void* const* slots, int W, void* out, size_t n, void* stream) {
  if (n == 0) return ok();
  bool alias = false;
  const arx_status s = check_io(slots, W, out, n, &alias);
  if (s != ARX_OK) return s;
  arx::ReduceCall c{};
  for (int r = 0; r < W; ++r) c.slot[r] = static_cast<const uint16_t*>(slots[r]);
  c.out = static_cast<uint16_t*>(out);
  c.n = n;
  c.W = W;
  c.out_aliases_slot = alias;
  c.prefetch_l2 = true;
  ARX_SET_BOUNDS_COUNTER(c);
  const cudaError_t e = arx::launch_reduce(c, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "arx_reduce launch");
  return ok();
}

size_t arx_reduce_host_staging_bytes(int W, size_t n) {
  if (W < 1 || W > ARX_MAX_W || n > (SIZE_MAX / 4) / ARX_MAX_W) return 0;
  return size_t(W) * round_up(n * 2, 256);
}

namespace {

// Device-usable address of a page-locked (pinned or registered) host buffer,
// or nullptr if `p` is pageable or unknown to CUDA.
const void* pinned_device_address(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

}  // namespace

arx_status arx_reduce_host(const void* const* host_slots, int W, void* host_out, size_t n,
                           void* dev_staging, size_t staging_bytes, void* stream) {
  if (n == 0) return ok();
  if (W < 1 || W > ARX_MAX_W) return fail(ARX_EINVAL, "W=%d outside 1..%d", W, ARX_MAX_W);
  if (!host_slots || !host_out) return fail(ARX_EINVAL, "null host pointer");
  for (int r = 0; r < W; ++r)
    if (!host_slots[r]) return fail(ARX_EINVAL, "null host slot %d", r);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Direct form: every buffer page-locked, so the kernel reads the partials
  // and writes the sum in host memory itself, over the coherent CPU-GPU link
  // (arx.cu's GB10 design: pinned host buffers are GPU buffers).
  const void* dev_slots[ARX_MAX_W];
  bool direct = true;
  for (int r = 0; r < W && direct; ++r) direct = (dev_slots[r] = pinned_device_address(host_slots[r])) != nullptr;
  void* dev_out = direct ? const_cast<void*>(pinned_device_address(host_out)) : nullptr;
  if (direct && dev_out) {
    bool alias = false;
    const arx_status s = check_io(dev_slots, W, dev_out, n, &alias);
    if (s != ARX_OK) return s;
    arx::ReduceCall c{};
    for (int r = 0; r < W; ++r) c.slot[r] = static_cast<const uint16_t*>(dev_slots[r]);
    c.out = static_cast<uint16_t*>(dev_out);
    c.n = n;
    c.W = W;
    c.out_aliases_slot = alias;
    // The L2 prefetch before the dependency wait applies to host buffers too:
    // host memory read over the link is cached in L2, so the call's first
    // link reads overlap the wait for its predecessor (11.49 against 11.67 us
    // per call at W = 8 [32, 4096], A/B in one process, GB300).  A prefetch
    // returns no data; the loads after the wait read the current contents.
    c.prefetch_l2 = true;
    ARX_SET_BOUNDS_COUNTER(c);
    const cudaError_t e = arx::launch_reduce(c, st);
    if (e != cudaSuccess) return fail_cuda(e, "arx_reduce_host launch");
    return ok();
  }

  // Staged form: one copy in per slot, the reduce in place, one copy out.
  if (!dev_staging) return fail(ARX_EINVAL, "pageable host buffers need a staging buffer");
  if (reinterpret_cast<uintptr_t>(dev_staging) & 1u) return fail(ARX_EINVAL, "staging not 2-byte aligned");
  const size_t need = arx_reduce_host_staging_bytes(W, n);
  if (need == 0 || staging_bytes < need)
    return fail(ARX_EINVAL, "staging buffer %zu bytes, need %zu", staging_bytes, need);
  const size_t stride = round_up(n * 2, 256);
  uint8_t* base = static_cast<uint8_t*>(dev_staging);
  for (int r = 0; r < W; ++r) {
    dev_slots[r] = base + size_t(r) * stride;
    const cudaError_t e = cudaMemcpyAsync(base + size_t(r) * stride, host_slots[r], n * 2,
                                          cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail_cuda(e, "arx_reduce_host copy in");
  }
  arx::ReduceCall c{};
  for (int r = 0; r < W; ++r) c.slot[r] = static_cast<const uint16_t*>(dev_slots[r]);
  c.out = reinterpret_cast<uint16_t*>(base);  // in place over staged slot 0
  c.n = n;
  c.W = W;
  c.out_aliases_slot = true;
  ARX_SET_BOUNDS_COUNTER(c);
  cudaError_t e = arx::launch_reduce(c, st);
  if (e != cudaSuccess) return fail_cuda(e, "arx_reduce_host launch");
  e = cudaMemcpyAsync(host_out, base, n * 2, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail_cuda(e, "arx_reduce_host copy out");
  return ok();
}

// ---- protocol context ----------------------------------------------------------

namespace {

struct Layout {
  size_t off_epoch, off_sem, off_pad, off_slots, slot_stride, total;
};

bool layout(int W, size_t max_n, int B, Layout* L) {
  if (W < 1 || W > ARX_MAX_W || B < 1 || B > ARX_STEP_MAX_BLOCKS) return false;
  if (max_n > (SIZE_MAX / 8) / (2 * ARX_MAX_W)) return false;
  L->off_epoch = kHeaderBytes;
  L->off_sem = round_up(L->off_epoch + size_t(W) * B * 4, 128);
  L->off_pad = round_up(L->off_sem + size_t(W) * B * 128, 128);
  L->off_slots = round_up(L->off_pad + size_t(W) * B * W * 4, 256);
  L->slot_stride = round_up(max_n > 0 ? max_n : 1, 128);  // elements; 256-byte multiple
  L->total = L->off_slots + 2 * size_t(W) * L->slot_stride * 2;
  return true;
}

int auto_blocks(int W, size_t max_n, arx_status* s) {
  cudaError_t e = cudaSuccess;
  const int sms = arx::current_sm_count(&e);
  if (sms < 1) {
    *s = fail_cuda(e, "arx_ctx_init device query");
    return -1;
  }
  const int cap = arx::step_capacity(W, &e);
  if (cap < 1) {
    *s = fail_cuda(e, "arx_ctx_init occupancy query");
    return -1;
  }
  // About one block per SM over the W*B grid for small messages; for large
  // ones about 128 groups of 8 elements staged per block (more loads in
  // flight), up to the resident capacity; at least 32 groups per reducing
  // block.  Measured on GB300 (W = 8, flag barriers): B = 16-19 best at
  // 2^17 elements, 32-38 at 2^18, the capacity (72-76) from 2^20 -- 27 %
  // faster than 19 at 2^23.
  size_t B = size_t(sms) / size_t(W);
  const size_t groups = (max_n + 7) / 8;
  const size_t by_size = groups / (size_t(W) * 128);
  if (B < by_size) B = by_size;
  const size_t by_work = (groups + size_t(W) * 32 - 1) / (size_t(W) * 32);
  if (B > by_work) B = by_work;
  if (B > size_t(cap / W)) B = size_t(cap / W);
  // The cluster-launched variants (one cluster of W blocks per chunk) run in
  // one wave only if every cluster is resident at once; clusters stay within
  // one GPU processing cluster, so that can be fewer than cap / W.
  const int ccap = arx::step_cluster_capacity(W, &e);
  if (ccap < 1) {
    *s = fail_cuda(e, "arx_ctx_init cluster occupancy query");
    return -1;
  }
  if (B > size_t(ccap)) B = size_t(ccap);
  if (B > ARX_STEP_MAX_BLOCKS) B = ARX_STEP_MAX_BLOCKS;
  // Latency-bound messages (B up to two blocks per SM over the grid), from
  // 16 up: a multiple of 8, so the cluster variant's B clusters of W blocks
  // spread evenly over the GPU's graphics processing clusters (152 SMs in 8
  // on GB300) -- W = 8 [32, 4096]: 3.56 us per step at 16 against 4.05 at
  // 19; W = 4: 3.12 at 32 against 3.42 at 38 -- the flag variants within
  // +-3 %.  At the resident capacity (bandwidth-bound) rounding down cost
  // 1.5 %, so B stays there.
  if (B >= 16 && B <= 2 * size_t(sms) / size_t(W)) B &= ~size_t(7);
  if (B < 1) B = 1;
  *s = ARX_OK;
  return int(B);
}

// Block groups of the staggered staging for slots in host memory: about
// 128 KiB of staged data per group, at most B; 0 (all at once) below two.
// Group g starts writing at T0 + g * stagger_ns, stagger_ns the time the
// GPU-to-host direction of NVLink-C2C takes to write one group's bytes at
// kHostWriteBytesPerNs.  Measured on GB300 (W = 8 [32, 4096], 16 groups of
// 128 KiB): 160 bytes/ns 18.5-18.8 us per step, 190 18.7-19.4, 220 and 250
// slower (groups crowd the link), 120 slower (the link idles between
// groups).  The link's one-way copy rate is 190-206 GB/s.
constexpr uint64_t kHostWriteBytesPerNs = 160;

int stagger_groups(int W, size_t n, int B) {
  const size_t bytes = size_t(W) * n * 2;
  size_t K = (bytes + (size_t(64) << 10)) >> 17;  // nearest multiple of 128 KiB
  if (K > size_t(B)) K = size_t(B);
  return K < 2 ? 0 : int(K);
}

uint64_t stagger_ns(int W, size_t n, int K) {
  return K < 2 ? 0 : uint64_t(size_t(W) * n * 2 / size_t(K)) / kHostWriteBytesPerNs;
}

arx_status check_ctx(const arx_ctx* ctx) {
  if (!ctx || ctx->magic != kCtxMagic) return fail(ARX_ESTATE, "context not initialised");
  return ARX_OK;
}

}  // namespace

size_t arx_ctx_workspace_bytes(int W, size_t max_n, int nblocks) {
  Layout L;
  if (!layout(W, max_n, nblocks == 0 ? ARX_STEP_MAX_BLOCKS : nblocks, &L)) return 0;
  return L.total;
}

size_t arx_ctx_words_bytes(int W, int nblocks) {
  Layout L;
  if (!layout(W, 1, nblocks == 0 ? ARX_STEP_MAX_BLOCKS : nblocks, &L)) return 0;
  return L.off_slots;
}

size_t arx_ctx_slots_bytes(int W, size_t max_n) {
  Layout L;
  if (!layout(W, max_n, 1, &L)) return 0;
  return L.total - L.off_slots;
}

namespace {

// Common part of both context initialisers: `slots` is the device address of
// the slot banks, `slots_bytes` their capacity.
arx_status init_ctx(arx_ctx* ctx, void* words, size_t words_bytes, bool one_buffer, void* slots,
                    size_t slots_bytes, int slots_where, int W, size_t max_n, int nblocks) {
  if (!ctx) return fail(ARX_EINVAL, "null ctx");
  std::memset(ctx, 0, sizeof *ctx);
  if (W < 1 || W > ARX_MAX_W) return fail(ARX_EINVAL, "W=%d outside 1..%d", W, ARX_MAX_W);
  if (nblocks < 0 || nblocks > ARX_STEP_MAX_BLOCKS)
    return fail(ARX_EINVAL, "nblocks=%d outside 0..%d", nblocks, ARX_STEP_MAX_BLOCKS);
  if (!words) return fail(ARX_EINVAL, "null workspace");
  if (reinterpret_cast<uintptr_t>(words) & 255u) return fail(ARX_EINVAL, "workspace not 256-byte aligned");
  if (!one_buffer) {
    if (!slots) return fail(ARX_EINVAL, "null slots buffer");
    if (reinterpret_cast<uintptr_t>(slots) & 255u) return fail(ARX_EINVAL, "slots not 256-byte aligned");
  }
  int B = nblocks;
  if (B == 0) {
    arx_status s = ARX_OK;
    B = auto_blocks(W, max_n, &s);
    if (B < 1) return s;
  }
  Layout L;
  if (!layout(W, max_n, B, &L)) return fail(ARX_EINVAL, "max_n=%zu too large", max_n);
  if (one_buffer) {
    if (words_bytes < L.total) return fail(ARX_EINVAL, "workspace %zu bytes, need %zu", words_bytes, L.total);
    slots = static_cast<uint8_t*>(words) + L.off_slots;
    slots_bytes = L.total - L.off_slots;
  } else {
    if (words_bytes < L.off_slots)
      return fail(ARX_EINVAL, "words buffer %zu bytes, need %zu", words_bytes, L.off_slots);
    if (slots_bytes < L.total - L.off_slots)
      return fail(ARX_EINVAL, "slots buffer %zu bytes, need %zu", slots_bytes, L.total - L.off_slots);
    if (overlap_kind(words, slots, L.off_slots, L.total - L.off_slots) != 0)
      return fail(ARX_EOVERLAP, "words and slots buffers overlap");
  }
  ctx->magic = kCtxMagic;
  ctx->slots = slots;
  ctx->slots_bytes = slots_bytes;
  ctx->slots_where = slots_where;
  ctx->W = W;
  ctx->nblocks = B;
  ctx->fault_rank = -1;
  ctx->sync_mode = ARX_SYNC_SEMAPHORE;
  ctx->max_n = max_n;
  ctx->slot_stride = L.slot_stride;
  ctx->timeout_ns = ARX_DEFAULT_TIMEOUT_NS;
  ctx->ws = words;
  ctx->ws_bytes = words_bytes;
  ctx->off_epoch = L.off_epoch;
  ctx->off_sem = L.off_sem;
  ctx->off_pad = L.off_pad;
  ctx->off_slots = L.off_slots;
  ctx->ctrl_bytes = L.off_slots;
  return ok();
}

}  // namespace

arx_status arx_ctx_init(arx_ctx* ctx, void* ws, size_t ws_bytes, int W, size_t max_n, int nblocks) {
  return init_ctx(ctx, ws, ws_bytes, true, nullptr, 0, ARX_SLOTS_DEVICE, W, max_n, nblocks);
}

arx_status arx_ctx_init_split(arx_ctx* ctx, void* words, size_t words_bytes, void* slots,
                              size_t slots_bytes, int slots_where, int W, size_t max_n, int nblocks) {
  if (slots_where == ARX_SLOTS_HOST) {
    if (!slots) return fail(ARX_EINVAL, "null slots buffer");
    const void* dev = pinned_device_address(slots);
    if (!dev) return fail(ARX_EINVAL, "host slots buffer is not page-locked memory known to CUDA");
    slots = const_cast<void*>(dev);
  } else if (slots_where != ARX_SLOTS_DEVICE) {
    return fail(ARX_EINVAL, "slots_where=%d is neither ARX_SLOTS_DEVICE nor ARX_SLOTS_HOST", slots_where);
  }
  return init_ctx(ctx, words, words_bytes, false, slots, slots_bytes, slots_where, W, max_n, nblocks);
}

arx_status arx_ctx_set_timeout(arx_ctx* ctx, uint64_t ns) {
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  if (ns == 0) return fail(ARX_EINVAL, "timeout must be > 0");
  ctx->timeout_ns = ns;
  return ok();
}

arx_status arx_ctx_set_sync(arx_ctx* ctx, int mode) {
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  if (mode != ARX_SYNC_SEMAPHORE && mode != ARX_SYNC_PAD && mode != ARX_SYNC_PAD_FENCED &&
      mode != ARX_SYNC_CLUSTER && mode != ARX_SYNC_SEMAPHORE_GLOBAL)
    return fail(ARX_EINVAL, "unknown sync mode %d", mode);
  ctx->sync_mode = mode;
  return ok();
}

arx_status arx_ctx_set_fault(arx_ctx* ctx, int rank) {
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  if (rank < -1 || rank >= ctx->W) return fail(ARX_EINVAL, "fault rank %d outside -1..%d", rank, ctx->W - 1);
  ctx->fault_rank = rank;
  return ok();
}

arx_status arx_ctx_reset(arx_ctx* ctx, void* stream) {
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  const cudaError_t e = cudaMemsetAsync(ctx->ws, 0, ctx->ctrl_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "arx_ctx_reset");
  ctx->failed_err = 0;
  return ok();
}

arx_status arx_step(const arx_ctx* ctx, const void* const* inputs, void* out, size_t n, void* stream) {
  arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  if (ctx->failed_err != 0)
    return fail(ARX_ESTATE, "the context failed (device error word 0x%08x); arx_ctx_reset it before the next step",
                ctx->failed_err);
  if (n == 0) return ok();
  if (n > ctx->max_n) return fail(ARX_EINVAL, "n=%zu exceeds the context's max_n=%llu", n,
                                  static_cast<unsigned long long>(ctx->max_n));
  if (ctx->sync_mode < ARX_SYNC_SEMAPHORE || ctx->sync_mode > ARX_SYNC_SEMAPHORE_GLOBAL)
    return fail(ARX_ESTATE, "context holds an unknown sync mode %d", ctx->sync_mode);
  if (ctx->sync_mode == ARX_SYNC_CLUSTER && ctx->fault_rank >= 0)
    return fail(ARX_EINVAL, "fault injection skips a flag signal; the cluster barrier has none to skip");
  bool alias = false;
  s = check_io(inputs, ctx->W, out, n, &alias);
  if (s != ARX_OK) return s;
  if (overlap_kind(out, ctx->ws, n * 2, ctx->ws_bytes) != 0)
    return fail(ARX_EOVERLAP, "output overlaps the workspace");
  if (overlap_kind(out, ctx->slots, n * 2, ctx->slots_bytes) != 0)
    return fail(ARX_EOVERLAP, "output overlaps the slots");
  for (int r = 0; r < ctx->W; ++r) {
    if (overlap_kind(inputs[r], ctx->ws, n * 2, ctx->ws_bytes) != 0 ||
        overlap_kind(inputs[r], ctx->slots, n * 2, ctx->slots_bytes) != 0)
      return fail(ARX_EOVERLAP, "input %d overlaps the workspace or the slots", r);
  }
  cudaError_t e = cudaSuccess;
  const int cap = arx::step_capacity(ctx->W, &e);
  if (cap < 1) return fail_cuda(e, "arx_step occupancy query");
  if (ctx->nblocks * ctx->W > cap)
    return fail(ARX_EINVAL, "grid %d x %d exceeds the %d co-resident blocks of this device",
                ctx->nblocks, ctx->W, cap);
  arx::StepCall c{};
  for (int r = 0; r < ctx->W; ++r) c.in[r] = static_cast<const uint16_t*>(inputs[r]);
  c.out = static_cast<uint16_t*>(out);
  c.n = n;
  c.ws = static_cast<uint8_t*>(ctx->ws);
  c.off_epoch = ctx->off_epoch;
  c.off_sem = ctx->off_sem;
  c.off_pad = ctx->off_pad;
  c.slots = static_cast<uint16_t*>(ctx->slots);
  c.slot_stride = ctx->slot_stride;
  c.timeout_ns = ctx->timeout_ns;
  c.W = ctx->W;
  c.B = ctx->nblocks;
  c.fault_rank = ctx->fault_rank;
  c.sync_mode = ctx->sync_mode;
  c.stagger = ctx->slots_where == ARX_SLOTS_HOST ? stagger_groups(ctx->W, n, ctx->nblocks) : 0;
  c.stagger_ns = stagger_ns(ctx->W, n, c.stagger);
  ARX_SET_BOUNDS_COUNTER(c);
  e = arx::launch_step(c, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "arx_step launch");
  return ok();
}

arx_status arx_ctx_query(arx_ctx* ctx, uint32_t* seq, uint32_t* dev_err, void* stream) {
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t words[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(words, ctx->ws, sizeof words, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e, "arx_ctx_query");
  if (seq) *seq = words[0];
  if (dev_err) *dev_err = words[1];
  const uint32_t code = words[1] & 0xFFu;
  if (code == 0) return ok();
  ctx->failed_err = words[1];
  if (code == ARX_ETIMEOUT || code == ARX_ESTATE)
    return fail(static_cast<arx_status>(code), "device error word 0x%08x (stage %u, rank %u, block %u)",
                words[1], (words[1] >> 8) & 15u, (words[1] >> 12) & 15u, words[1] >> 16);
  return fail(ARX_ESTATE, "device error word 0x%08x", words[1]);
}

arx_status arx_bounds_violations(uint32_t* count, int reset) {
#ifdef ARX_BOUNDS_CHECK
  if (!count) return fail(ARX_EINVAL, "null count");
  cudaError_t e = cudaSuccess;
  uint32_t* c = arx::bounds_counter(&e);
  if (!c) return fail_cuda(e, "bounds counter lookup");
  e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(count, c, sizeof *count, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && reset) e = cudaMemset(c, 0, sizeof *count);
  if (e != cudaSuccess) return fail_cuda(e, "arx_bounds_violations");
  return ok();
#else
  (void)count;
  (void)reset;
  return fail(ARX_EINVAL, "this library was built without bounds checks");
#endif
}

#ifdef ARX_BOUNDS_CHECK
// Checking build only (not declared in arx.h): one deliberately out-of-range
// address that the check counts and skips, so a test can see the counter
// move without any out-of-range access taking place.
arx_status arx_bounds_probe(const void* dev_buffer_16_bytes) {
  cudaError_t e = cudaSuccess;
  uint32_t* c = arx::bounds_counter(&e);
  if (!c) return fail_cuda(e, "bounds counter lookup");
  bounds_probe_kernel<<<1, 1>>>(c, static_cast<const uint16_t*>(dev_buffer_16_bytes));
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e, "arx_bounds_probe");
  return ok();
}
#endif

arx_status arx_watch_step(const arx_ctx* ctx, uint32_t target_seq, uint64_t stall_ns,
                          uint64_t poll_ns, uint64_t max_wait_ns, uint32_t* host_words,
                          void* stream, arx_watch_report* report) {
  arx_watch_report rep{};
  if (report) *report = rep;
  const arx_status s = check_ctx(ctx);
  if (s != ARX_OK) return s;
  if (!host_words) return fail(ARX_EINVAL, "null host_words");
  if (poll_ns == 0 || stall_ns == 0 || max_wait_ns == 0)
    return fail(ARX_EINVAL, "poll, stall and max-wait times must be > 0");
  using clock = std::chrono::steady_clock;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const auto t0 = clock::now();
  auto since = [](clock::time_point a) {
    return uint64_t(std::chrono::duration_cast<std::chrono::nanoseconds>(clock::now() - a).count());
  };
  bool gap = false;
  clock::time_point gap_start = t0;
  arx_status result = ARX_OK;
  for (;;) {
    // Header: seq (completed), err, blocks[2], published.
    cudaError_t e = cudaMemcpyAsync(host_words, ctx->ws, 5 * sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
      result = fail_cuda(e, "arx_watch_step header copy");
      break;
    }
    ++rep.polls;
    rep.seq = host_words[0];
    rep.dev_err = host_words[1];
    rep.published = host_words[4];
    const uint32_t code = rep.dev_err & 0xFFu;
    if (code != 0) {
      result = fail(code == ARX_ETIMEOUT ? ARX_ETIMEOUT : ARX_ESTATE,
                    "device error word 0x%08x during the step", rep.dev_err);
      break;
    }
    if (int32_t(rep.seq - target_seq) >= 0) break;  // done (unsigned wrap aware)
    if (rep.published != rep.seq) {
      if (!gap) {
        gap = true;
        gap_start = clock::now();
      }
      rep.stalled_ns = since(gap_start);
      if (rep.stalled_ns >= stall_ns) {
        result = fail(ARX_ETIMEOUT, "STALL: step %u published, completed %u, for %llu ns", rep.published,
                      rep.seq, static_cast<unsigned long long>(rep.stalled_ns));
        break;
      }
    } else {
      gap = false;
      rep.stalled_ns = 0;
    }
    if (since(t0) >= max_wait_ns) {
      result = fail(ARX_ETIMEOUT, "completed seq %u did not reach %u within %llu ns", rep.seq, target_seq,
                    static_cast<unsigned long long>(max_wait_ns));
      break;
    }
    std::this_thread::sleep_for(std::chrono::nanoseconds(poll_ns));
  }
  rep.waited_ns = since(t0);
  if (report) *report = rep;
  if (result == ARX_OK) return ok();
  return result;
}

}  // extern "C"
