// Device helpers shared by the reduce and protocol kernels (sm_103a).
//
// Arithmetic of the reduce (arx.cu, `arx_kernel`, reduce loop): each bf16 is
// widened to fp32 exactly (its 16 bits become the upper half of a binary32),
// added into an fp32 accumulator that starts at +0 in rank order with
// round-to-nearest-even adds (add.rn.f32: never contracted, never flushed --
// the build passes no fast-math and keeps -ftz=false), and rounded once to
// bf16 with cvt.rn (nearest, ties to even).
#pragma once

#include <cstddef>
#include <cstdint>

namespace arx {

constexpr int kMaxW = 8;
constexpr int kThreads = 256;

// ---- bf16 <-> fp32 ------------------------------------------------------------

// Low / high bf16 of a packed 32-bit word, widened exactly.
__device__ __forceinline__ float widen_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float widen_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float widen16(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// Two fp32 -> one word of two bf16 (lo in bits 0-15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint16_t round_bf16(float x) {
  uint16_t d;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(d) : "f"(x));
  return d;
}

// acc[0..7] += the 8 bf16 of one 16-byte vector (element k of the group in acc[k]).
__device__ __forceinline__ void accumulate8(float (&acc)[8], const uint4& v) {
  acc[0] = __fadd_rn(acc[0], widen_lo(v.x));
  acc[1] = __fadd_rn(acc[1], widen_hi(v.x));
  acc[2] = __fadd_rn(acc[2], widen_lo(v.y));
  acc[3] = __fadd_rn(acc[3], widen_hi(v.y));
  acc[4] = __fadd_rn(acc[4], widen_lo(v.z));
  acc[5] = __fadd_rn(acc[5], widen_hi(v.z));
  acc[6] = __fadd_rn(acc[6], widen_lo(v.w));
  acc[7] = __fadd_rn(acc[7], widen_hi(v.w));
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  return o;
}

// Rank-order sum of W vectors: acc from +0, slot 0 first.
template <int W>
__device__ __forceinline__ uint4 sum_vectors(const uint4 (&v)[W]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll
  for (int r = 0; r < W; ++r) accumulate8(acc, v[r]);
  return pack8(acc);
}

// The same for 8-byte vectors of 4 bf16.
__device__ __forceinline__ void accumulate4(float (&acc)[4], const uint2& v) {
  acc[0] = __fadd_rn(acc[0], widen_lo(v.x));
  acc[1] = __fadd_rn(acc[1], widen_hi(v.x));
  acc[2] = __fadd_rn(acc[2], widen_lo(v.y));
  acc[3] = __fadd_rn(acc[3], widen_hi(v.y));
}

template <int W>
__device__ __forceinline__ uint2 sum_halves(const uint2 (&v)[W]) {
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int r = 0; r < W; ++r) accumulate4(acc, v[r]);
  return make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
}

// ---- 16-byte global loads and stores --------------------------------------------

// Read-only streaming load: non-coherent path, no L1 allocation.  Only for
// data no thread of the same kernel writes.
__device__ __forceinline__ uint4 ld_stream_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Coherent streaming load (safe when the same kernel writes the location
// after reading it, e.g. in-place output), no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

// Load cached at L2 only: for data other blocks of this kernel wrote before a
// release/acquire handshake (never served from a stale L1 line).
__device__ __forceinline__ uint4 ld_cg(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t ld_cg16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_global(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 8-byte forms of the streaming loads and the store.
__device__ __forceinline__ uint2 ld_stream_nc(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_global(uint2* p, const uint2& v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---- bounds checks of the opt-in checking build -----------------------------------
//
// Built with ARX_BOUNDS_CHECK (`_build.py --bounds-check`, a separate
// library), every data access of the kernels -- partials, slots, output --
// is preceded by a check that [p, p + bytes) lies inside the buffer it
// belongs to; a failed check adds 1 to a device counter and the access is
// skipped, so a wrong index is counted instead of touching memory.  In the
// normal build ARX_CHECKED(...) is exactly the access.
#ifdef ARX_BOUNDS_CHECK
__device__ __forceinline__ bool in_range(const void* p, size_t bytes, const void* base, size_t nbytes,
                                         uint32_t* counter) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
  const bool ok = a >= b && a + bytes <= b + nbytes;
  if (!ok) atomicAdd(counter, 1u);
  return ok;
}
#define ARX_CHECKED(p, bytes, base, nbytes, counter, access)                     \
  do {                                                                          \
    if (::arx::in_range((p), (bytes), (base), (nbytes), (counter))) { access; }  \
  } while (0)
#else
#define ARX_CHECKED(p, bytes, base, nbytes, counter, access) \
  do {                                                       \
    access;                                                  \
  } while (0)
#endif

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple
// of 16).  A hint only: no data is returned and nothing is made visible.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// ---- programmatic dependent launch ------------------------------------------------

// Wait for the previous kernel of the stream (when launched as its
// programmatic dependent) before any global access, then allow the next one
// to begin launching; it waits in the same way before touching memory.
__device__ __forceinline__ void dependent_launch_prologue() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---- thread-block cluster barrier ------------------------------------------------
//
// Every thread of every block of the cluster arrives, then waits for all of
// them (hardware barrier; `.aligned`: all threads of a warp execute it
// together).  Arrive with release orders the arriving thread's earlier
// writes -- and, after a block barrier, its block's -- before the waits of
// the other blocks, which acquire them.

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- distributed shared memory (words in another block of the cluster) ---------

// Shared-window address of a __shared__ variable of this block.
__device__ __forceinline__ uint32_t shared_address(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The same variable in the block of cluster rank `rank`, as a shared::cluster
// address.
__device__ __forceinline__ uint32_t cluster_peer_address(uint32_t shared_addr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(shared_addr), "r"(rank));
  return a;
}

// Fire-and-forget adds to a word in a cluster peer's shared memory: relaxed,
// or release at cluster scope (the issuing thread's earlier writes, global
// ones included, are visible to the cluster before the add is).
__device__ __forceinline__ void red_add_relaxed_cluster(uint32_t cluster_addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" :: "r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_release_cluster(uint32_t cluster_addr, uint32_t v) {
  asm volatile("red.release.cluster.shared::cluster.add.u32 [%0], %1;" :: "r"(cluster_addr), "r"(v) : "memory");
}

// Loads of a word in this block's own shared memory that cluster peers add
// to: relaxed, or acquire at cluster scope.
__device__ __forceinline__ uint32_t ld_relaxed_cluster_shared(uint32_t shared_addr) {
  uint32_t v;
  asm volatile("ld.relaxed.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(shared_addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_cluster_shared(uint32_t shared_addr) {
  uint32_t v;
  asm volatile("ld.acquire.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(shared_addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared(uint32_t shared_addr, uint32_t v) {
  asm volatile("st.shared::cta.u32 [%0], %1;" :: "r"(shared_addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// ---- scoped atomics and loads for the protocol words (one GPU: .gpu scope) -------

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Fire-and-forget adds (no return value, so the issuing thread does not wait
// for the round trip to L2).
__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_cas_relaxed_gpu(uint32_t* p, uint32_t cmp, uint32_t val) {
  uint32_t old;
  asm volatile("atom.relaxed.gpu.global.cas.b32 %0, [%1], %2, %3;"
               : "=r"(old) : "l"(p), "r"(cmp), "r"(val) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t atom_cas_release_gpu(uint32_t* p, uint32_t cmp, uint32_t val) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.cas.b32 %0, [%1], %2, %3;"
               : "=r"(old) : "l"(p), "r"(cmp), "r"(val) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t atom_cas_acquire_gpu(uint32_t* p, uint32_t cmp, uint32_t val) {
  uint32_t old;
  asm volatile("atom.acquire.gpu.global.cas.b32 %0, [%1], %2, %3;"
               : "=r"(old) : "l"(p), "r"(cmp), "r"(val) : "memory");
  return old;
}

// ---- words and data another agent (a host thread) writes: system scope ----------

// Acquire at system scope: the writes the writer released before storing the
// word are visible to this thread's later loads.
__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Cache-bypassing loads ("fetch again"): a cached copy of a host-memory line
// is treated as stale and read anew, so data another agent rewrote is never
// served from an earlier step's line.
__device__ __forceinline__ uint4 ld_cv(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cv.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t ld_cv16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.cv.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Spin budget that ends a wait even if the global timer stood still: every
// poll is a round trip to L2 (hundreds of ns) and, after the first 1024 polls,
// also sleeps, so timeout_ns / 64 polls last longer than timeout_ns.
__device__ __forceinline__ uint64_t spin_cap(uint64_t timeout_ns) {
  return 4096u + timeout_ns / 64u;
}

__device__ __forceinline__ void backoff(uint64_t spins) {
  if (spins > 1024u) __nanosleep(128);
}

}  // namespace arx
