// One protocol step of the one-shot all-reduce, as a single kernel on one GPU.
//
// The pages run one kernel per rank on different GPUs and synchronise them
// through flags.  Here the W ranks are W virtual ranks inside one grid of
// B x W blocks: block (b, r) = (blockIdx.x, blockIdx.y) plays rank r's block b.
//
//  1. seq/parity (arx.cu, `arx_kernel`): seq = completed + 1, bank = seq & 1.
//     The per-block parity epoch (common.cuh, `PushController`, two stages)
//     must equal (seq - 1) & 1.
//  2. start barrier (common.cuh, `PullController::sync`, start stage,
//     unfenced): lane 0 of warp q < W adds 1 to Semaphore sem[q][b]; lane 0 of
//     warp r waits until flag - counter >= W; then the block synchronises.
//  3. stage: rank r's chunk b -> slots[bank][r] (stands in for the RDMA write
//     into every peer's recv[seq & 1][rank]); the last block past the copy
//     resets the first block counter and publishes seq (arx.cu "last block
//     publishes").
//  4. end barrier (`PullController::sync`, end stage, fenced): block barrier,
//     release-add 1 to sem[q][b] for every q, warp r waits with acquire until
//     flag - counter >= 2W and sets counter += 2W.
//  5. reduce: sub-range r of chunk b over slots[bank][0..W-1] in rank order.
//  6. exit: triton_barrier.py `blockwise_barrier`, Pattern 2 (relaxed):
//     thread t < W sends pad[t][b][r] 0 -> 1 and waits pad[r][b][t] 1 -> 0, so
//     the pad is all zero again; `PushController::exit` flips epoch[r][b];
//     the last block out resets the second counter and stores seq as
//     completed (arx.cu "last block out").
//
// Barrier variants (the context's sync mode), all with the same data path:
//  * Semaphore (default): steps 2 and 4 with each block's flag held for the
//    step in its shared memory.  The W blocks of chunk b are one
//    thread-block cluster.  Start stage: the W arrivals at the cluster's
//    hardware barrier are its W signals (every block's zeroed flag is in
//    place once it completes).  End stage: every block adds 1 to each peer's
//    flag through distributed shared memory, then the cluster barrier
//    (release arrival, acquire wait) orders the staged slots and the adds;
//    the owner then checks flag - counter >= 2W, bounded, which waits only
//    if a signal is missing.  The flag and counter are loaded at entry (by
//    thread 0, with seq and the epoch) and written back after that check, so
//    the words in memory follow the same arithmetic.  No add is in flight after the end barrier, so no exit
//    barrier is needed; the kernel boundary stands in for Pattern 2 (the
//    next kernel on the stream starts only after every block of this one
//    has finished reading the slots).
//  * Semaphore, global: steps 2 and 4 with the flags in the workspace (as the
//    page keeps them for peers on other GPUs), step 6 a relaxed pad barrier.
//  * Pad: every barrier is triton_barrier.py's `blockwise_barrier` on the
//    signal pad, in the page's three patterns -- Pattern 0 at the start
//    (relaxed barrier, then block sync), Pattern 1 after staging (block sync,
//    acq_rel barrier, block sync) and Pattern 2 at exit.  The Semaphores are
//    not touched.
//  * Pad, fenced: as Pad, but all three barriers use acq_rel compare-and-swaps
//    (the page's "acq_rel" sem everywhere instead of "relaxed" where its
//    patterns allow it).
//  * Cluster (no counterpart on the pages, which synchronise separate GPUs):
//    the W blocks of chunk b are launched as one thread-block cluster and
//    each barrier is its hardware barrier -- relaxed at start and exit,
//    release on arrive and acquire on wait after staging.  No flag word takes
//    part; the launch needs clusters, not cooperative co-residency.
// One pad serves all three barriers of a step: a send spins until the
// receiver has consumed the previous signal (the word is back at 0), so
// consecutive barriers pair their sends and waits in order.
//
// Every flag wait is bounded by the context's timeout (global timer plus a
// spin cap): on expiry the block records ARX_ETIMEOUT with its stage, rank
// and block in the error word and carries on, so the kernel always finishes
// and the host reads the status.  The pages' waits are unbounded; these are
// not.  The cluster barrier's wait is a hardware wait without a timeout: it
// completes because every thread of every block arrives unconditionally.
// Code in the cluster variants must never return early or arrive
// conditionally (the fault knob skips a flag add, never an arrival).
//
// Latency choices (measured on GB300, W = 8, bf16 [32, 4096]): the kernel is
// a programmatic dependent of the previous kernel on its stream (it waits for
// it before touching memory, and lets the next one launch at once); fenced
// waits poll with relaxed loads and fence once after success (the
// fence-after-read form of acquire); the exit writes the flipped epoch from
// the value read at entry and counts blocks out without fences -- seq,
// epochs and counters are read only by later kernels on the stream (ordered
// by the kernel boundary) and by the host after a synchronisation, never by
// another block of the same launch.  The pages fence there because a host
// proxy and remote GPUs observe those words while the kernel runs.  Semaphore
// signals are fire-and-forget `red` adds (their old value is never needed),
// and each block's first batch of staging loads -- reads of the caller's
// input, which no barrier guards -- is issued before the start barrier so
// that its DRAM latency overlaps the barrier.
#include <atomic>
#include <cstddef>

#include "arx_device.cuh"
#include "arx_internal.h"

namespace arx {
namespace {

// Status codes written to the device error word (same values as arx_status).
constexpr uint32_t kErrTimeout = 4;
constexpr uint32_t kErrState = 5;

enum Stage : uint32_t {
  kStartWait = 1, kEndWait = 2, kPadSend = 3, kPadWait = 4, kEpoch = 5,
  kStartPadSend = 6, kStartPadWait = 7, kEndPadSend = 8, kEndPadWait = 9, kStaggerWait = 10
};

// Barrier variants (arx.h, ARX_SYNC_*).
enum SyncMode : int {
  kSyncSemaphore = 0, kSyncPad = 1, kSyncPadFenced = 2, kSyncCluster = 3, kSyncSemaphoreGlobal = 4
};

// 16-byte vectors each thread loads before storing them while staging.
constexpr int kStageBatch = 4;

// Bytes of its input chunk a block prefetches into L2 before the dependency
// wait: its first two staging batches.  Only for messages whose W inputs
// total at most kPrefetchMaxBytes: there the step is latency-bound and the
// prefetch saved 5-11 % (W = 8 [32, 4096]: 5.63 -> 5.04 us, pad barrier);
// at 2^20 elements and above it was neutral or cost 2-4 %, competing with
// the previous step's own traffic (A/B of two builds in one process, GB300).
constexpr size_t kPrefetchBytes = 2u * kStageBatch * kThreads * 16u;
constexpr size_t kPrefetchMaxBytes = size_t(4) << 20;

struct Header {  // first bytes of the workspace (256 reserved)
  uint32_t seq;        // completed steps
  uint32_t err;        // device error word
  uint32_t blocks[2];  // blocks past staging / blocks finished
  uint32_t published;  // last staged seq
  uint32_t unused[27];
  // Byte 128: the start of the last staggered step -- its seq in the high
  // half, the low 32 bits of the global timer when its first block arrived
  // in the low half (the groups' start times count from it); zero before
  // the context's first staggered step.
  unsigned long long stagger_t0;
  uint32_t unused2[30];
};
static_assert(offsetof(Header, stagger_t0) == 128 && sizeof(Header) == 256, "header layout");

// common.cuh `Semaphore`: 128-byte aligned flag + counter; the counter is
// read and written only by the owning block.
struct alignas(128) Semaphore {
  uint32_t flag;
  uint32_t counter;
};

struct StepArgs {
  const uint16_t* in[kMaxW];
  uint16_t* out;
  size_t n;
  uint8_t* ws;
  uint16_t* slots;
  uint64_t off_epoch, off_sem, off_pad, slot_stride;
  uint64_t timeout_ns;
  int B;
  int fault_rank;
  uint32_t in_vec_mask;  // bit r: input r is 16-byte aligned
  int out_vec;           // out is 16-byte aligned
  int prefetch;          // L2 prefetch of the input chunks (small messages)
  uint32_t stagger;      // K >= 2 block groups stage in turn (staggering kernels only)
  uint64_t stagger_ns;   // time between two groups' starts
#ifdef ARX_BOUNDS_CHECK
  uint32_t* bounds_counter;
#endif
};

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code, uint32_t stage,
                                             uint32_t r, uint32_t b) {
  const uint32_t word = code | (stage << 8) | ((r & 15u) << 12) | ((b & 0xFFFFu) << 16);
  atomicCAS(err, 0u, word);
}

// Wait until flag - base >= target (unsigned), bounded.  Polls with relaxed
// loads; kFence (end stage) adds a fence after the successful poll, which
// makes it an acquire of everything released before the flag reached the
// target (the start stage is unfenced).
template <bool kFence>
__device__ bool semaphore_wait(const uint32_t* flag, uint32_t base, uint32_t target,
                               uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t cap = spin_cap(timeout_ns);
  for (uint64_t spins = 0;; ++spins) {
    const uint32_t v = ld_relaxed_gpu(flag);
    if (v - base >= target) {
      if constexpr (kFence) __threadfence();
      return true;
    }
    if ((spins & 15u) == 15u) {
      if (global_timer_ns() - t0 > timeout_ns || spins > cap) return false;
      backoff(spins);
    }
  }
}

// The same wait on a Semaphore flag in this block's own shared memory, which
// the blocks of its cluster add to: polls with relaxed cluster-scope loads;
// kAcquire (end stage) makes the successful poll an acquire at cluster scope,
// so the peers' staged writes released before their adds are visible.
template <bool kAcquire>
__device__ bool shared_semaphore_wait(uint32_t flag_addr, uint32_t base, uint32_t target,
                                      uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t cap = spin_cap(timeout_ns);
  for (uint64_t spins = 0;; ++spins) {
    const uint32_t v = kAcquire ? ld_acquire_cluster_shared(flag_addr) : ld_relaxed_cluster_shared(flag_addr);
    if (v - base >= target) return true;
    if ((spins & 15u) == 15u) {
      if (global_timer_ns() - t0 > timeout_ns || spins > cap) return false;
      backoff(spins);
    }
  }
}

// Wait until a count (zero before the step) has reached `target`, bounded.
__device__ bool count_wait(const uint32_t* count, uint32_t target, uint64_t timeout_ns) {
  return semaphore_wait<false>(count, 0u, target, timeout_ns);
}

// Compare-and-swap `from -> to` until it succeeds, bounded.
__device__ bool cas_until(uint32_t* p, uint32_t from, uint32_t to, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t cap = spin_cap(timeout_ns);
  for (uint64_t spins = 0;; ++spins) {
    if (atom_cas_relaxed_gpu(p, from, to) == from) return true;
    if ((spins & 15u) == 15u) {
      if (global_timer_ns() - t0 > timeout_ns || spins > cap) return false;
      backoff(spins);
    }
  }
}

// Compare-and-swap `from -> to` until it succeeds, bounded, with acquire or
// release semantics (the "acq_rel" sem of triton_barrier.py).
template <bool kRelease>
__device__ __forceinline__ uint32_t cas_ordered(uint32_t* p, uint32_t from, uint32_t to) {
  return kRelease ? atom_cas_release_gpu(p, from, to) : atom_cas_acquire_gpu(p, from, to);
}

template <bool kRelease>
__device__ bool cas_until_ordered(uint32_t* p, uint32_t from, uint32_t to, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t cap = spin_cap(timeout_ns);
  for (uint64_t spins = 0;; ++spins) {
    if (cas_ordered<kRelease>(p, from, to) == from) return true;
    if ((spins & 15u) == 15u) {
      if (global_timer_ns() - t0 > timeout_ns || spins > cap) return false;
      backoff(spins);
    }
  }
}

// triton_barrier.py `blockwise_barrier` for block b of virtual rank r, run by
// thread t < W: send_signal to pad[t][b][r] (0 -> 1) and wait_signal on
// pad[r][b][t] (1 -> 0), which leaves the pad all zero once every block of
// the barrier has passed.  kAcqRel: release send and acquire wait (the page's
// "acq_rel" sem; after the block barrier that precedes it, the release also
// covers the other threads' earlier writes); otherwise relaxed.  The first send and wait attempts go out
// back to back; only a failed attempt is retried, within the bound.
// `send` false skips the send (fault injection).
template <bool kAcqRel>
__device__ void pad_barrier(uint32_t* pad, uint32_t B, uint32_t W, uint32_t b, uint32_t r, uint32_t t,
                            bool send, uint64_t timeout_ns, uint32_t* err, uint32_t stage_send,
                            uint32_t stage_wait) {
  uint32_t* to = &pad[(t * B + b) * W + r];
  uint32_t* from = &pad[(r * B + b) * W + t];
  const uint32_t sent = send ? (kAcqRel ? atom_cas_release_gpu(to, 0u, 1u) : atom_cas_relaxed_gpu(to, 0u, 1u)) : 0u;
  const uint32_t got = kAcqRel ? atom_cas_acquire_gpu(from, 1u, 0u) : atom_cas_relaxed_gpu(from, 1u, 0u);
  if (send && sent != 0u) {
    const bool ok = kAcqRel ? cas_until_ordered<true>(to, 0u, 1u, timeout_ns) : cas_until(to, 0u, 1u, timeout_ns);
    if (!ok) record_error(err, kErrTimeout, stage_send, r, b);
  }
  if (got != 1u) {
    const bool ok = kAcqRel ? cas_until_ordered<false>(from, 1u, 0u, timeout_ns) : cas_until(from, 1u, 0u, timeout_ns);
    if (!ok) record_error(err, kErrTimeout, stage_wait, r, b);
  }
}

__device__ __forceinline__ size_t split_point(size_t total, uint32_t parts, uint32_t i) {
  return total / parts * i + (total % parts) * i / parts;
}

template <int W, int kSync, bool kStagger>
__global__ void __launch_bounds__(kThreads) step_kernel(const StepArgs a) {
  constexpr bool kPad = kSync == kSyncPad || kSync == kSyncPadFenced;
  constexpr bool kCluster = kSync == kSyncCluster;  // grid clusters of (1, W, 1)
  constexpr bool kDsm = kSync == kSyncSemaphore;    // clusters too; Semaphores in shared memory
  constexpr bool kSemGlobal = kSync == kSyncSemaphoreGlobal;
  constexpr bool kFencedAll = kSync == kSyncPadFenced;
  const uint32_t b = blockIdx.x, r = blockIdx.y;
  const uint32_t B = uint32_t(a.B);
  const uint32_t tid = threadIdx.x, warp = tid / 32u, lane = tid % 32u;
  Header* hdr = reinterpret_cast<Header*>(a.ws);
  uint32_t* epoch = reinterpret_cast<uint32_t*>(a.ws + a.off_epoch);
  Semaphore* sem = reinterpret_cast<Semaphore*>(a.ws + a.off_sem);
  uint32_t* pad = reinterpret_cast<uint32_t*>(a.ws + a.off_pad);
  uint16_t* slots = a.slots;
  const uint32_t total_blocks = B * uint32_t(W);

  __shared__ uint32_t s_seq;
  __shared__ uint32_t s_epoch;
  // Semaphore variant: this block's Semaphore flag (common.cuh `Semaphore`),
  // held in its shared memory for the step; the W blocks of the cluster add
  // to it through distributed shared memory.  The counter is read and
  // written only by its owner, so it stays in a register (`base`).
  __shared__ uint32_t s_sem_flag;
  __shared__ uint2 s_words;  // the block's (flag, counter) as the previous step left them
  const uint32_t flag_sh = shared_address(&s_sem_flag);
  const uint32_t owner = 32u * r;  // warp r, lane 0: the thread that waits on this block's flag

  // Chunk b (in 16-byte groups) of rank r's input.
  const size_t G = a.n / 8u;
  const size_t tail = a.n - 8u * G;
  const size_t c0 = split_point(G, B, b), c1 = split_point(G, B, b + 1u);
  const bool in_vec = (a.in_vec_mask >> r) & 1u;
  const uint4* s4 = reinterpret_cast<const uint4*>(a.in[r]);
  // Before waiting for the previous kernel of the stream, ask L2 for the
  // start of this chunk, so its DRAM latency overlaps that kernel's tail.  A
  // prefetch returns no data: inputs the previous kernel writes are still
  // read after the wait below, through L2.
  if (a.prefetch && tid == 0 && in_vec && c1 > c0) {
    const size_t bytes = (c1 - c0) * 16u < kPrefetchBytes ? (c1 - c0) * 16u : kPrefetchBytes;
    ARX_CHECKED(s4 + c0, bytes, a.in[r], a.n * 2, a.bounds_counter, prefetch_l2_bulk(s4 + c0, uint32_t(bytes)));
  }
  if constexpr (kDsm) {
    // The owner zeroes its flag (the shared word counts this step's
    // end-stage adds from zero) and its warp arrives at the start barrier
    // with release, which puts the zero in place before any peer's add can
    // reach it.  Done before the dependency wait -- shared memory and the
    // cluster barrier belong to this launch alone -- so the release, about
    // 0.3 us, overlaps that wait: 3.76 against 4.0 us per step with the
    // owner's warp arriving after its first staging loads (W = 8
    // [32, 4096], A/B in one process, GB300).
    if (tid == owner) st_shared(flag_sh, 0u);
    if (warp == r) {
      __syncwarp();  // the cluster barrier instructions are warp-aligned
      cluster_arrive_release();
    }
  }
  dependent_launch_prologue();

  // 1. seq / parity; epoch check (the words loaded back to back).  In the
  // Semaphore variant tid 0 also loads the block's Semaphore words in the
  // same round trip and hands them to the owner through shared memory: 4.0
  // against 4.2 us per step with the owner loading them itself between its
  // start arrival and wait (W = 8 [32, 4096], A/B in one process, GB300).
  if (tid == 0) {
    const uint32_t done = ld_relaxed_gpu(&hdr->seq);
    const uint32_t epoch_in = epoch[r * B + b];
    if constexpr (kDsm) s_words = *reinterpret_cast<const uint2*>(&sem[r * B + b]);
    const uint32_t seq = done + 1u;
    s_seq = seq;
    s_epoch = epoch_in;
    if (epoch_in != ((seq - 1u) & 1u)) record_error(&hdr->err, kErrState, kEpoch, r, b);
  }
  Semaphore& own = sem[r * B + b];
  uint32_t base = 0;
  uint32_t flag_in = 0;  // Semaphore variant: the flag as the previous step left it
  // Semaphore variant: the owner keeps the flag and counter of the previous
  // step in registers, so the words obey the page's arithmetic: flag -
  // counter = (flag_in + W + adds) - counter, i.e. W + adds - base with
  // base = counter - flag_in.

  // The first batch of this block's staging loads.  They read only the
  // caller's input, which no barrier guards, so they are issued before the
  // start barrier and their latency overlaps it; the slot writes still wait
  // for the barrier.
  uint4 first[kStageBatch] = {};
  if (in_vec) {
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const size_t g = c0 + tid + size_t(k) * kThreads;
      if (g < c1) ARX_CHECKED(s4 + g, 16, a.in[r], a.n * 2, a.bounds_counter, first[k] = ld_stream(s4 + g));
    }
  }

  // 2. start barrier.
  if constexpr (kDsm) {
    // PullController start stage (unfenced): its W signals are the W blocks'
    // arrivals at the cluster barrier, which every block has passed once
    // this wait returns -- counted into the flag as W at write-back.  The
    // owner's warp arrived (with release) before the dependency wait; the
    // other warps arrive relaxed here, after their first staging loads.
    __syncwarp();  // the cluster barrier instructions are warp-aligned
    if (warp != r) cluster_arrive_relaxed();
    __syncwarp();
    cluster_wait();
  } else if constexpr (kCluster) {
    // The W blocks of chunk b are one cluster: its hardware barrier, relaxed.
    cluster_arrive_relaxed();
    cluster_wait();
  } else if constexpr (kSemGlobal) {
    // PullController start stage, unfenced: no block barrier before the signal.
    if (lane == 0 && warp < uint32_t(W)) {
      red_add_relaxed_gpu(&sem[warp * B + b].flag, 1u);
      if (warp == r) {
        base = own.counter;
        if (!semaphore_wait<false>(&own.flag, base, uint32_t(W), a.timeout_ns))
          record_error(&hdr->err, kErrTimeout, kStartWait, r, b);
      }
    }
  } else {
    // Pattern 0: the barrier, then the block synchronises.
    if (tid < uint32_t(W))
      pad_barrier<kFencedAll>(pad, B, uint32_t(W), b, r, tid, true, a.timeout_ns, &hdr->err,
                              kStartPadSend, kStartPadWait);
  }
  __syncthreads();
  if constexpr (kDsm) {
    if (tid == owner) {
      flag_in = s_words.x;
      base = s_words.y - flag_in;
    }
  }
  const uint32_t seq = s_seq;
  const uint32_t par = seq & 1u;
  const size_t stride = size_t(a.slot_stride);
  uint16_t* bank = slots + size_t(par) * size_t(W) * stride;

  // Staggered staging (slots in host memory): the blocks form K groups by
  // chunk, and group g starts writing its slots at T0 + g * stagger_ns,
  // where T0 is the global timer when the step's first block got here
  // (compare-and-swapped into the header, tagged with the step's seq, so a
  // block that finds its own step's tag takes that T0 and nothing has to
  // clear the word afterwards) and stagger_ns is the time the link takes to
  // write one group's staged bytes.  So the writes to host
  // memory go out at about the link's rate, group after group, and each
  // group's reads (after its end barrier) overlap the later groups' writes
  // on the full-duplex link.  A scheduling delay only -- the barriers order
  // the data -- bounded by the context's timeout (error stage 10 if a stale
  // T0 asks for longer), and no block waits for another.  Measured (W = 8
  // [32, 4096], GB300): 18.5-18.8 us per step against 22.2 us when each
  // group waited for the previous one's count through L2 (about 1.1 us per
  // hand-off, 16 hand-offs) and 23.5 us with every group at once; 18.17
  // against 18.75 us with T0 untagged and zeroed by the last block out
  // (two fences and a store on that block's exit path).  A tag left from
  // 2^32 steps earlier would only cost one step its pacing: the start times
  // compare in 32-bit modular time, so a stale T0 reads as long past.
  // Compiled only into the kernels of host-slot steps.
  uint32_t K = 0, grp = 0;
  if constexpr (kStagger) {
    K = a.stagger;
    grp = b * K / B;
    if (tid == 0) {
      const unsigned long long now = global_timer_ns();
      const unsigned long long mine = (static_cast<unsigned long long>(seq) << 32) | (now & 0xFFFFFFFFull);
      unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(&hdr->stagger_t0);
      if (static_cast<uint32_t>(cur >> 32) != seq) {
        // Only blocks of this step write the word while it runs, so a failed
        // swap returns the start another block of this step installed.
        const unsigned long long old = atomicCAS(&hdr->stagger_t0, cur, mine);
        cur = old == cur ? mine : old;
      }
      const uint32_t t0 = static_cast<uint32_t>(cur);
      const uint32_t delay = static_cast<uint32_t>(grp * a.stagger_ns);
      for (uint64_t spins = 0; static_cast<uint32_t>(global_timer_ns()) - t0 < delay; ++spins) {
        if (global_timer_ns() - now > a.timeout_ns || spins > spin_cap(a.timeout_ns)) {
          record_error(&hdr->err, kErrTimeout, kStaggerWait, r, b);
          break;
        }
        __nanosleep(32);
      }
    }
    __syncthreads();
  }

  // 3. stage rank r's chunk b into slots[par][r].
  {
    const uint16_t* in = a.in[r];
    uint16_t* dst = bank + size_t(r) * stride;
    if (in_vec) {
      // Batches of kStageBatch vectors per thread: every load of a batch is
      // in flight before the first store.  The first batch was loaded above.
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int k = 0; k < kStageBatch; ++k) {
        const size_t g = c0 + tid + size_t(k) * kThreads;
        if (g < c1) ARX_CHECKED(d4 + g, 16, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter, st_global(d4 + g, first[k]));
      }
      for (size_t g0 = c0 + tid + size_t(kStageBatch) * kThreads; g0 < c1;
           g0 += size_t(kStageBatch) * kThreads) {
        uint4 v[kStageBatch];
#pragma unroll
        for (int k = 0; k < kStageBatch; ++k) {
          const size_t g = g0 + size_t(k) * kThreads;
          if (g < c1) ARX_CHECKED(s4 + g, 16, a.in[r], a.n * 2, a.bounds_counter, v[k] = ld_stream(s4 + g));
        }
#pragma unroll
        for (int k = 0; k < kStageBatch; ++k) {
          const size_t g = g0 + size_t(k) * kThreads;
          if (g < c1) ARX_CHECKED(d4 + g, 16, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter, st_global(d4 + g, v[k]));
        }
      }
    } else {
      for (size_t e = 8u * c0 + tid; e < 8u * c1; e += kThreads)
        ARX_CHECKED(in + e, 2, a.in[r], a.n * 2, a.bounds_counter, ARX_CHECKED(dst + e, 2, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter, dst[e] = in[e]));
    }
    if (b == B - 1u && tid < tail)
      ARX_CHECKED(in + 8u * G + tid, 2, a.in[r], a.n * 2, a.bounds_counter,
                  ARX_CHECKED(dst + 8u * G + tid, 2, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter, dst[8u * G + tid] = in[8u * G + tid]));
  }
  // 4. end barrier, fenced: every thread's staging precedes the release.
  __syncthreads();
  // The cluster-launched variants count the block past the copy between their
  // end-stage arrival and wait and look at the count's old value later, so
  // the atomic's round trip overlaps the cluster barrier (and, in the cluster
  // variant, the reduce) instead of holding warp 1 before the barrier:
  // 3.43 against 3.56 us per step in the cluster variant (W = 8 [32, 4096],
  // A/B in one process).  The Semaphore variant publishes right after the
  // cluster barrier, before its end-stage check, so a block held in that
  // check by a missing signal does not hold back `published` (the host
  // watchdog reports a step published but not done).
  uint32_t published_old = 0;
  if constexpr (kCluster) {
    // Release on arrive (after the block barrier: the whole block's staging),
    // acquire on wait; the published count runs between the two.
    cluster_arrive_release();
    if (tid == 32u) published_old = atomicAdd(&hdr->blocks[0], 1u);
    __syncwarp();
    cluster_wait();
  } else if constexpr (kPad) {
    // Pattern 1: block sync, acq_rel barrier, block sync.
    if (tid < uint32_t(W)) {
      pad_barrier<true>(pad, B, uint32_t(W), b, r, tid, int(r) != a.fault_rank, a.timeout_ns, &hdr->err,
                        kEndPadSend, kEndPadWait);
    } else if (tid == 32u) {
      // Last block past the copy publishes seq (a thread outside the barrier).
      // `published` is read only by the host watchdog, never as a guard of
      // staged data, so the count needs no fence.
      if (atomicAdd(&hdr->blocks[0], 1u) == total_blocks - 1u) {
        hdr->blocks[0] = 0u;
        st_relaxed_gpu(&hdr->published, seq);
      }
    }
  } else if constexpr (kDsm) {
    // PullController end stage: lane 0 of warp q < W adds 1 to block q's
    // flag through distributed shared memory, then every thread arrives at
    // the cluster barrier with release (after the block barrier: the whole
    // block's staging, and this block's adds, are ordered before the
    // arrival) and waits with acquire.  When the wait returns, every add of
    // the cluster has landed and every staged slot of the chunk is visible;
    // no block writes into another block's shared memory after it, so no
    // exit barrier is needed.  The owner then checks flag - counter >= 2W --
    // it passes at once unless a signal is missing (the fault knob), in
    // which case it waits, bounded, and reports ARX_ETIMEOUT -- and advances
    // the counter.  Measured (W = 8 [32, 4096], GB300, A/B of library builds
    // in one process): 4.0 us per step with this end stage before the start
    // stage's changes above, 3.56-3.60 us with them (a build without the
    // adds and the check, which cannot count a missing signal, was no
    // faster); 4.4-4.5 us with the owner polling its flag for release adds
    // and no hardware barrier after staging, 4.6 us with the adds issued
    // after the arrival (the check then waits for them, and an exit barrier
    // must keep them from landing in an exited block), 5.6 us with the flags
    // in global memory; the cluster variant, with no flag traffic at all,
    // 3.4-3.5 us.
    if (lane == 0 && warp < uint32_t(W) && int(r) != a.fault_rank)
      red_add_relaxed_cluster(cluster_peer_address(flag_sh, warp), 1u);
    __syncwarp();
    cluster_arrive_release();
    if (tid == 32u) published_old = atomicAdd(&hdr->blocks[0], 1u);
    __syncwarp();
    cluster_wait();
    if (tid == 32u && published_old == total_blocks - 1u) {
      // Last block past the copy publishes seq (only the host watchdog reads it).
      hdr->blocks[0] = 0u;
      st_relaxed_gpu(&hdr->published, seq);
    }
    if (tid == owner) {
      // flag - counter = (flag_in + W + adds) - (flag_in + base): the page's
      // unsigned test flag - counter >= 2W is adds - (base - W) >= 2W.
      if (shared_semaphore_wait<false>(flag_sh, base - uint32_t(W), 2u * uint32_t(W), a.timeout_ns)) {
        base += 2u * uint32_t(W);  // the counter after this step
      } else {
        record_error(&hdr->err, kErrTimeout, kEndWait, r, b);
      }
      // Write the step's Semaphore words back (common.cuh keeps them in
      // memory between calls): the flag with every signal of the step
      // counted (W at the start barrier, the landed end-stage adds), the
      // counter advanced by 2W after a successful end stage.  Stored here,
      // where every add has landed, so the stores overlap the reduce: 4.19
      // against 4.27 us per step storing them at the block's exit.
      own.flag = flag_in + uint32_t(W) + ld_relaxed_cluster_shared(flag_sh);
      own.counter = base + flag_in;
    }
  } else if (lane == 0 && warp < uint32_t(W)) {
    if (int(r) != a.fault_rank) {
      // Release after the block barrier: every thread's staged data is
      // ordered before the signal (the waiter acquires).  No extra fence:
      // the barrier plus the release already order the block's writes, as
      // in the pad barrier; dropping the fence here (and before the
      // `published` counts) saved 8-10 % of the step (A/B on two GPUs).
      red_add_release_gpu(&sem[warp * B + b].flag, 1u);
    }
    if (warp == r) {
      if (semaphore_wait<true>(&own.flag, base, 2u * uint32_t(W), a.timeout_ns)) {
        own.counter = base + 2u * uint32_t(W);
      } else {
        record_error(&hdr->err, kErrTimeout, kEndWait, r, b);
      }
    }
  } else if (tid == 1) {
    // Last block past the copy publishes seq.  Done by a thread that neither
    // signals nor waits, so it overlaps the barrier instead of preceding it;
    // no fence, as above (only the host watchdog reads `published`).
    if (atomicAdd(&hdr->blocks[0], 1u) == total_blocks - 1u) {
      hdr->blocks[0] = 0u;
      st_relaxed_gpu(&hdr->published, seq);
    }
  }
  __syncthreads();

  // 5. reduce sub-range r of chunk b over slots[par][0..W-1].
  {
    const size_t s0 = c0 + split_point(c1 - c0, uint32_t(W), r);
    const size_t s1 = c0 + split_point(c1 - c0, uint32_t(W), r + 1u);
    const uint4* src[W];
#pragma unroll
    for (int q = 0; q < W; ++q) src[q] = reinterpret_cast<const uint4*>(bank + size_t(q) * stride);
    for (size_t g = s0 + tid; g < s1; g += kThreads) {
      uint4 v[W];
#pragma unroll
      for (int q = 0; q < W; ++q) ARX_CHECKED(src[q] + g, 16, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter, v[q] = ld_cg(src[q] + g));
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
    if (b == B - 1u && r == uint32_t(W) - 1u && tid < tail) {
      const size_t e = 8u * G + tid;
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < W; ++q)
        ARX_CHECKED(bank + size_t(q) * stride + e, 2, a.slots, size_t(4) * W * a.slot_stride, a.bounds_counter,
                    acc = __fadd_rn(acc, widen16(ld_cg16(bank + size_t(q) * stride + e))));
      ARX_CHECKED(a.out + e, 2, a.out, a.n * 2, a.bounds_counter, a.out[e] = round_bf16(acc));
    }
  }

  // 6. exit: zero-resetting pad barrier (Pattern 2: block barrier, then the
  // barrier -- relaxed, or acq_rel in the fenced variant), then the epoch
  // flip and the block-out count.  No block of this launch reads those two
  // words (later kernels and the host see them after the kernel ends), so a
  // thread outside the barrier does them concurrently with it: pad variant
  // 6.3 -> 5.6 us per step, Semaphore variant 6.46 -> 6.01 us (W = 8
  // [32, 4096], A/B of two builds in one process, the same on two GPUs).
  __syncthreads();
  if constexpr (kCluster) cluster_arrive_relaxed();
  if ((kPad || kSemGlobal) && tid < uint32_t(W)) {
    pad_barrier<kFencedAll>(pad, B, uint32_t(W), b, r, tid, true, a.timeout_ns, &hdr->err, kPadSend,
                            kPadWait);
  } else if (tid == 32u) {
    if constexpr (kCluster) {
      // Last block past the copy publishes seq (only the host watchdog reads
      // it); its count was taken at the end barrier.
      if (published_old == total_blocks - 1u) {
        hdr->blocks[0] = 0u;
        st_relaxed_gpu(&hdr->published, seq);
      }
    }
    epoch[r * B + b] = (s_epoch + 1u) % 2u;  // PushController::exit
    if (atomicAdd(&hdr->blocks[1], 1u) == total_blocks - 1u) {  // last block out
      hdr->blocks[1] = 0u;
      st_relaxed_gpu(&hdr->seq, seq);
    }
  }
  if constexpr (kCluster) {
    // All arrivals are unconditional (no thread returns early), so the wait
    // always ends.
    __syncwarp();
    cluster_wait();
  }
}

constexpr int kMaxDevices = 64;

// Resident blocks per SM of the step kernel for W ranks: the least over the
// sync modes (with and without staggered staging), so one capacity serves
// every mode.
template <int W>
int blocks_per_sm(int dev, cudaError_t* err) {
  static std::atomic<int> cache[kMaxDevices];  // per-device results, shared by host threads
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int lo = 0;
  const void* kernels[10] = {reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphore, false>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphore, true>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncCluster, true>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncPad, false>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncPadFenced, false>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncCluster, false>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphoreGlobal, false>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphoreGlobal, true>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncPad, true>),
                             reinterpret_cast<const void*>(step_kernel<W, kSyncPadFenced, true>)};
  for (const void* k : kernels) {
    int b = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kThreads, 0);
    if (*err != cudaSuccess || b < 1) return -1;
    lo = lo == 0 || b < lo ? b : lo;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(lo, std::memory_order_relaxed);
  return lo;
}

template <int W>
cudaError_t launch_w(const StepCall& c, cudaStream_t stream) {
  StepArgs a{};
  for (int r = 0; r < W; ++r) a.in[r] = c.in[r];
  a.out = c.out;
  a.n = c.n;
  a.ws = c.ws;
  a.off_epoch = c.off_epoch;
  a.off_sem = c.off_sem;
  a.off_pad = c.off_pad;
  a.slots = c.slots;
  a.slot_stride = c.slot_stride;
#ifdef ARX_BOUNDS_CHECK
  a.bounds_counter = c.bounds_counter;
#endif
  a.timeout_ns = c.timeout_ns;
  a.B = c.B;
  a.fault_rank = c.fault_rank;
  for (int r = 0; r < W; ++r)
    if ((reinterpret_cast<uintptr_t>(c.in[r]) & 15u) == 0) a.in_vec_mask |= 1u << r;
  a.stagger = uint32_t(c.stagger < 0 ? 0 : c.stagger);
  if (a.stagger > uint32_t(c.B)) a.stagger = uint32_t(c.B);
  if (a.stagger < 2u) a.stagger = 0;
  a.stagger_ns = c.stagger_ns;
  a.prefetch = size_t(W) * c.n * 2u <= kPrefetchMaxBytes;
  a.out_vec = (reinterpret_cast<uintptr_t>(c.out) & 15u) == 0;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(c.B), unsigned(W), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // Every block of the grid waits on others: the launch must make them all
  // resident at once.  It is also a programmatic dependent of the previous
  // kernel on the stream (see dependent_launch_prologue).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t err = cudaErrorInvalidValue;
  const bool st = a.stagger >= 2u;
  // The W blocks of a chunk as one cluster of (1, W, 1), waiting only on each
  // other: clusters need not be resident together, so no cooperative launch.
  cudaLaunchAttribute cattr[2];
  cattr[0].id = cudaLaunchAttributeClusterDimension;
  cattr[0].val.clusterDim.x = 1;
  cattr[0].val.clusterDim.y = unsigned(W);
  cattr[0].val.clusterDim.z = 1;
  cattr[1] = attr[1];
  switch (c.sync_mode) {
    case kSyncSemaphore:
      // Staggered steps (slots in host memory) too: 18.4 us per step
      // against 18.9 with the Semaphores in global memory (W = 8
      // [32, 4096], A/B in one process, GB300).
      cfg.attrs = cattr;
      cfg.numAttrs = 2;
      err = st ? cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncSemaphore, true>, a)
               : cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncSemaphore, false>, a);
      break;
    case kSyncSemaphoreGlobal:
      err = st ? cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncSemaphoreGlobal, true>, a)
               : cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncSemaphoreGlobal, false>, a);
      break;
    case kSyncPad:
      err = st ? cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncPad, true>, a)
               : cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncPad, false>, a);
      break;
    case kSyncPadFenced:
      err = st ? cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncPadFenced, true>, a)
               : cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncPadFenced, false>, a);
      break;
    case kSyncCluster:
      // The staggered staging waits for no other block, so the clusters
      // need not be co-resident in this variant either.
      cfg.attrs = cattr;
      cfg.numAttrs = 2;
      err = st ? cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncCluster, true>, a)
               : cudaLaunchKernelEx(&cfg, step_kernel<W, kSyncCluster, false>, a);
      break;
    default: break;
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Clusters of (1, W, 1) blocks of the cluster-launched step kernels that can
// be resident at once on the current device: the least over those kernels.
// A cluster's blocks share one GPU processing cluster, so this can be fewer
// than the resident blocks / W (GB300: 152 SMs in 8 of them).
template <int W>
int cluster_capacity_w(cudaError_t* err) {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return -1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1, unsigned(W), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = unsigned(W);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int lo = 0;
  const void* kernels[4] = {reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphore, false>),
                            reinterpret_cast<const void*>(step_kernel<W, kSyncSemaphore, true>),
                            reinterpret_cast<const void*>(step_kernel<W, kSyncCluster, false>),
                            reinterpret_cast<const void*>(step_kernel<W, kSyncCluster, true>)};
  for (const void* k : kernels) {
    int c = 0;
    *err = cudaOccupancyMaxActiveClusters(&c, k, &cfg);
    if (*err != cudaSuccess || c < 1) return -1;
    lo = lo == 0 || c < lo ? c : lo;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(lo, std::memory_order_relaxed);
  return lo;
}

template <int W>
int capacity_w(cudaError_t* err) {
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return -1;
  const int sms = current_sm_count(err);
  if (sms < 1) return -1;
  const int per = blocks_per_sm<W>(dev, err);
  if (per < 1) return -1;
  return sms * per;
}

}  // namespace

cudaError_t launch_step(const StepCall& c, cudaStream_t stream) {
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

int step_cluster_capacity(int W, cudaError_t* err) {
  switch (W) {
    case 1: return cluster_capacity_w<1>(err);
    case 2: return cluster_capacity_w<2>(err);
    case 3: return cluster_capacity_w<3>(err);
    case 4: return cluster_capacity_w<4>(err);
    case 5: return cluster_capacity_w<5>(err);
    case 6: return cluster_capacity_w<6>(err);
    case 7: return cluster_capacity_w<7>(err);
    case 8: return cluster_capacity_w<8>(err);
    default: *err = cudaErrorInvalidValue; return -1;
  }
}

int step_capacity(int W, cudaError_t* err) {
  switch (W) {
    case 1: return capacity_w<1>(err);
    case 2: return capacity_w<2>(err);
    case 3: return capacity_w<3>(err);
    case 4: return capacity_w<4>(err);
    case 5: return capacity_w<5>(err);
    case 6: return capacity_w<6>(err);
    case 7: return capacity_w<7>(err);
    case 8: return capacity_w<8>(err);
    default: *err = cudaErrorInvalidValue; return -1;
  }
}

}  // namespace arx
