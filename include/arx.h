/*
 * arx.h -- C ABI of the deterministic W-way bf16 reduce on one GB300 (sm_103a).
 *
 * The operation is the data-parallel core of the one-shot all-reduce of
 * arx.cu ("one-shot all-reduce over RoCE for GB10, no NCCL"): the sum of W
 * bf16 partials, each element widened to fp32, accumulated from +0.0 in rank
 * order 0, 1, ..., W-1, and rounded once to bf16 (round to nearest, ties to
 * even), so that every consumer gets the same bits (arx.cu, `arx_kernel`,
 * reduce loop, "rank order: every rank gets the same bits").  On one GPU the
 * W rank partials are W slots in this GPU's HBM; there are no peers.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device (or managed) addresses of this
 *    process's current device; pointers named "host" are host addresses.
 *  - bf16 data is passed as untyped pointers to IEEE bfloat16 elements
 *    (2 bytes, little-endian), contiguous, element i at byte offset 2*i.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is enqueued on it and the call returns without waiting,
 *    except where a function says it synchronises.
 *  - The library allocates no memory and owns no caller buffer: the caller
 *    owns every byte (PyTorch tensors in the Python binding), except the one
 *    static device array behind arx_step_noalloc (below).  Nothing here takes
 *    ownership of a pointer.
 *  - Errors are returned as arx_status; nothing calls exit() or throws.
 *    Argument errors are detected on the host before anything is enqueued.
 *    arx_last_error() gives a one-line detail for the calling thread.
 *  - Enqueuing entry points (arx_reduce, arx_step) launch kernels only, so
 *    they can be captured into a CUDA graph (arx.cu: allreduce "runs on the
 *    current stream and is CUDA-graph capturable").
 */
#ifndef ARX_H_
#define ARX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Most ranks (partials) per reduce: arx.cu `kMaxWorld`, common.cuh `kMaxNumGPU`. */
#define ARX_MAX_W 8
/* Most thread blocks per virtual rank in arx_step (bounds the control words). */
#define ARX_STEP_MAX_BLOCKS 256
/* Default bound of every device-side wait of arx_step, in nanoseconds. */
#define ARX_DEFAULT_TIMEOUT_NS 1000000000ull

typedef enum arx_status {
  ARX_OK = 0,
  ARX_EINVAL = 1,    /* bad argument: W out of range, null or misaligned pointer, n too large */
  ARX_EOVERLAP = 2,  /* out partially overlaps an input (only exact aliasing is allowed) */
  ARX_ECUDA = 3,     /* a CUDA runtime call or kernel launch failed; see arx_last_error() */
  ARX_ETIMEOUT = 4,  /* a bounded device wait of arx_step expired (reported by arx_ctx_query) */
  ARX_ESTATE = 5     /* protocol words inconsistent (epoch != completed steps mod 2), or bad ctx */
} arx_status;

/* One-line name of a status code (static storage). */
const char* arx_status_string(arx_status s);

/* Detail of the last non-OK status returned to the calling thread, or "". */
const char* arx_last_error(void);

/* ---------------------------------------------------------------------------
 * Stateless reduce.
 *
 * out[i] = bf16_rne( (((+0.0f + f32(s0[i])) + f32(s1[i])) + ...) + f32(s{W-1}[i]) )
 * for 0 <= i < n, every add in fp32 round-to-nearest-even, subnormals kept
 * (arx.cu, `arx_kernel`, reduce loop).
 *
 *   slots   HOST array of W device pointers (device memory), each to n
 *           bf16 elements.  The array itself is read during the call only (it
 *           is copied into the kernel's parameters).  Slots may repeat or
 *           overlap each other.  The kernel may prefetch them into L2 before
 *           the previous kernel on the stream has finished (a hint: the data
 *           it sums are read after that kernel's writes).
 *   W       1 <= W <= ARX_MAX_W.  (The page requires W >= 2; W = 1 is the
 *           identity, except that -0 becomes +0.)
 *   out     device pointer to n bf16 elements.  It may be exactly equal to
 *           one slot pointer ("in and out may alias", arx.cu); any other
 *           overlap with a slot is ARX_EOVERLAP.
 *   n       elements per slot.  n == 0 returns ARX_OK and launches nothing
 *           (pointers are not inspected).  No upper limit besides memory.
 *   stream  cudaStream_t as void*.
 * Alignment: every pointer must be 2-byte aligned (ARX_EINVAL otherwise).
 * When all of them share the same address mod 16 the kernel streams 16-byte
 * vectors (a scalar head/tail covers the rest); otherwise a scalar kernel runs.
 * Returns ARX_ECUDA if the launch fails (the stream is left as CUDA left it).
 * ------------------------------------------------------------------------- */
arx_status arx_reduce(const void* const* slots, int W, void* out, size_t n, void* stream);

/* ---------------------------------------------------------------------------
 * Host-buffer form of arx_reduce, for callers whose partials live in host
 * memory (the end-to-end form: host partials in, host sum out, enqueued on
 * `stream`).  Same arithmetic and bits as arx_reduce.
 *
 * Direct form -- when every host buffer (all slots and host_out) is
 * page-locked (cudaHostAlloc, cudaHostRegister, torch pin_memory): the reduce
 * kernel reads the partials and writes the sum in host memory itself, over
 * GB300's coherent CPU-GPU link, as arx.cu does on GB10 ("pinned host buffers
 * are GPU buffers").  One kernel, no copies; dev_staging is not used and may
 * be NULL.  As in arx_reduce, the kernel may prefetch the partials into L2
 * before the previous kernel on the stream has finished (a hint: the data it
 * sums are read after that kernel's writes; the CPU must not write the
 * buffers while the call is in flight).
 * Staged form -- otherwise: one cudaMemcpyAsync per slot into dev_staging,
 * the reduce in place over staged slot 0, one cudaMemcpyAsync back (copies
 * from and to pageable memory synchronise with the host).
 *
 *   host_slots     HOST array of W host pointers, each to n bf16 elements.
 *   host_out       host pointer to n bf16 elements; may equal one slot
 *                  exactly (written when the stream gets there; synchronise
 *                  `stream` before reading it, and keep every buffer alive
 *                  until then).
 *   dev_staging    staged form only: device buffer of at least
 *                  arx_reduce_host_staging_bytes(W, n) bytes, owned by the
 *                  caller and overwritten.  Slot r is staged at byte offset
 *                  r * stride, stride = n*2 rounded up to 256.
 * Errors as arx_reduce; ARX_EINVAL if the staged form is needed and the
 * staging buffer is missing or too small.
 * ------------------------------------------------------------------------- */
size_t arx_reduce_host_staging_bytes(int W, size_t n);
arx_status arx_reduce_host(const void* const* host_slots, int W, void* host_out, size_t n,
                           void* dev_staging, size_t staging_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Stateful protocol step: seq/parity double-buffered slots, per-block
 * Semaphore epochs and a zero-resetting signal pad, run as one kernel.
 *
 * The pages synchronise ranks on different GPUs: arx.cu stages each partial
 * into send[seq & 1] and waits for the peers' flags; common.cuh's
 * PullController counts per-block Semaphore arrivals (start stage W, end
 * stage 2W, then counter += 2W) and PushController keeps a per-block parity
 * epoch; triton_barrier.py's blockwise_barrier leaves its signal pad all zero
 * after every synchronisation so no host-side flag is needed under CUDA graph
 * replay.  On one GPU the W ranks are W virtual ranks: the step runs a grid of
 * B x W thread blocks, block (b, r) playing rank r's block b:
 *   1. seq = completed + 1, par = seq & 1; check epoch[r][b] == (seq-1) & 1;
 *   2. start barrier (unfenced): +1 to sem[q][b] for every q, wait for W;
 *   3. stage input r's chunk b into slots[par][r]; last block publishes seq
 *      (slots in host memory: block groups start staging in turn, see
 *      arx_ctx_init_split);
 *   4. end barrier (release/acquire): +1 to sem[q][b], wait for 2W, counter += 2W;
 *   5. reduce sub-range r of chunk b over slots[par][0..W-1] into out;
 *   6. pad barrier (0->1 sends, 1->0 waits), epoch[r][b] ^= 1, last block out
 *      stores seq as completed.
 * This outline is the page's, and the ARX_SYNC_SEMAPHORE_GLOBAL variant's;
 * the other barrier variants below realise steps 2, 4 and 6 differently
 * (the default on a thread-block cluster), with the same data path.
 * The output equals arx_reduce's bit for bit.  Every flag wait is bounded by
 * the context's timeout; on expiry the block records ARX_ETIMEOUT in the
 * device error word and carries on, so the kernel always finishes (the
 * cluster barriers of ARX_SYNC_SEMAPHORE and ARX_SYNC_CLUSTER are hardware
 * waits that complete because every thread arrives unconditionally; see the
 * barrier variants below).
 *
 * Workspace: one caller-owned device buffer, ZERO-FILLED before the first
 * step (e.g. torch.zeros(uint8)), of arx_ctx_workspace_bytes(W, max_n,
 * nblocks) bytes and 256-byte aligned.  Layout (offsets in arx_ctx):
 *   [0, 256)        header, uint32: seq (completed steps), err (device error
 *                   word, 0 = none), blocks[2] (publish / exit counters),
 *                   published (last staged seq); at byte 128 a uint64,
 *                   the start of the last staggered host-slot step: its
 *                   seq in the high half, the low 32 bits of its
 *                   global-timer start in the low half (zero before the
 *                   first)
 *   off_epoch       uint32 epoch[W][B]                    (PushController)
 *   off_sem         struct { uint32 flag, counter; } sem[W][B], 128-byte
 *                   stride                                (Semaphore)
 *   off_pad         uint32 pad[W][B][W], pad[owner][b][sender]  (signal pad)
 *   off_slots       bf16 slots[2][W][slot_stride]         (parity x rank)
 * Device error word: low 8 bits an arx_status, bits 8-11 the stage that
 * failed (1 start Semaphore wait, 2 end Semaphore wait, 3 exit pad send,
 * 4 exit pad wait, 5 epoch check, 6 start pad send, 7 start pad wait, 8 end
 * pad send, 9 end pad wait, 10 staggered-staging wait), bits 12-15 the
 * virtual rank, bits 16-31 the block.
 * ------------------------------------------------------------------------- */
typedef struct arx_ctx {
  uint32_t magic;        /* set by arx_ctx_init */
  int32_t W;             /* virtual ranks, 1..ARX_MAX_W */
  int32_t nblocks;       /* B, thread blocks per virtual rank */
  int32_t fault_rank;    /* -1, or a virtual rank that skips its end-barrier signal (testing) */
  int32_t sync_mode;     /* ARX_SYNC_* (arx_ctx_set_sync); ARX_SYNC_SEMAPHORE after init */
  int32_t slots_where;   /* ARX_SLOTS_DEVICE or ARX_SLOTS_HOST */
  uint64_t max_n;        /* capacity of one slot, elements */
  uint64_t slot_stride;  /* elements from one slot to the next (multiple of 128) */
  uint64_t timeout_ns;   /* bound of every device wait */
  void* ws;              /* device workspace base */
  uint64_t ws_bytes;
  uint64_t off_epoch, off_sem, off_pad, off_slots;
  uint64_t ctrl_bytes;   /* bytes [0, ctrl_bytes) hold every protocol word */
  void* slots;           /* device address of slots[2][W][slot_stride]: ws + off_slots,
                            or the separate buffer of arx_ctx_init_split */
  uint64_t slots_bytes;
  uint32_t failed_err;   /* 0, or the nonzero device error word arx_ctx_query
                            last read: arx_step refuses to launch (ARX_ESTATE)
                            until arx_ctx_reset clears it */
  uint32_t reserved;
} arx_ctx;

/* Workspace bytes for W virtual ranks, slots of max_n elements and `nblocks`
 * blocks per rank (nblocks == 0 sizes for ARX_STEP_MAX_BLOCKS, which fits
 * any nblocks).  Returns 0 for invalid W or nblocks. */
size_t arx_ctx_workspace_bytes(int W, size_t max_n, int nblocks);

/* Fills *ctx (a host struct; no allocation, no device access unless
 * nblocks == 0).  nblocks == 0 picks B from the current device's SM count
 * and max_n.  The workspace must be zero-filled before the first step, and
 * after any step that reported an error (see arx_ctx_reset). */
arx_status arx_ctx_init(arx_ctx* ctx, void* ws, size_t ws_bytes, int W, size_t max_n,
                        int nblocks);

/* The same context with the protocol words and the slot banks in two
 * buffers, so that the slots can live in page-locked host memory -- arx.cu's
 * GB10 layout, where the send and receive slots are pinned host buffers that
 * the GPU reads and writes directly.  On GB300 the kernel then stages every
 * partial into host memory and reads the staged slots back over NVLink-C2C.
 *   words        DEVICE buffer, zero-filled, 256-byte aligned, of at least
 *                arx_ctx_words_bytes(W, nblocks) bytes: the header, epochs,
 *                Semaphores and pad (every atomic stays in device memory).
 *   slots        at least arx_ctx_slots_bytes(W, max_n) bytes, 256-byte
 *                aligned, contents irrelevant:
 *                  slots_where == ARX_SLOTS_DEVICE: a device pointer;
 *                  slots_where == ARX_SLOTS_HOST: the HOST address of
 *                  page-locked memory (cudaHostAlloc, cudaHostRegister,
 *                  torch pin_memory); the library looks up its device
 *                  address (ARX_EINVAL if it is not page-locked).
 * Everything else as arx_ctx_init; arx_ctx_reset zeroes the words only.
 * Buffers are the caller's and must outlive the context's last step.
 * With the slots in host memory a step of at least 192 KiB of partials
 * stages in turn: its blocks form groups by chunk (about 128 KiB of staged
 * data each, at most one per block), and group g starts writing its slots at
 * T0 + g * (the time the GPU-to-host link takes to write one group), T0 the
 * global timer when the step's first block arrived -- so writes to host
 * memory go out at about the link's rate and overlap the earlier groups'
 * reads on the full-duplex link.  Only the start times move; barriers and
 * result are the same, and no block waits for another to start. */
#define ARX_SLOTS_DEVICE 0
#define ARX_SLOTS_HOST 1
size_t arx_ctx_words_bytes(int W, int nblocks);
size_t arx_ctx_slots_bytes(int W, size_t max_n);
arx_status arx_ctx_init_split(arx_ctx* ctx, void* words, size_t words_bytes, void* slots,
                              size_t slots_bytes, int slots_where, int W, size_t max_n,
                              int nblocks);

/* Sets the bound of every device wait (ns > 0). */
arx_status arx_ctx_set_timeout(arx_ctx* ctx, uint64_t ns);

/* Barrier variants of the step (same data path and result; they differ in
 * which of the pages' barriers run, where their words live and in their
 * memory ordering):
 *  ARX_SYNC_SEMAPHORE   (default) common.cuh's PullController over the
 *                       Semaphores, with each Semaphore flag held for the
 *                       step in its block's shared memory: the W blocks of a
 *                       chunk are one thread-block cluster.  Start stage
 *                       (unfenced): the W blocks' arrivals at the cluster's
 *                       hardware barrier are its W signals.  End stage: each
 *                       block adds 1 to every peer's flag through distributed
 *                       shared memory, the cluster barrier (release arrival,
 *                       acquire wait) makes the staged slots and the adds
 *                       visible, and the owner checks flag - counter >= 2W,
 *                       a bounded wait that waits only when a signal is
 *                       missing (the fault knob skips one, as in the flag
 *                       modes below).  The flag and counter are loaded from
 *                       the workspace at entry and written back after that
 *                       check, so the words follow the same arithmetic as in
 *                       the global form.  The hardware barrier's waits
 *                       complete because every thread arrives
 *                       unconditionally.
 *  ARX_SYNC_SEMAPHORE_GLOBAL  the same barriers with the Semaphores in the
 *                       workspace (global memory), as the page keeps them for
 *                       peers on other GPUs: release adds and acquire polls
 *                       through L2; triton_barrier.py's blockwise_barrier,
 *                       Pattern 2, relaxed, at exit; a cooperative grid.
 *  ARX_SYNC_PAD         triton_barrier.py's blockwise_barrier on the signal
 *                       pad for all three: Pattern 0 (relaxed) at the start,
 *                       Pattern 1 (acq_rel) after staging, Pattern 2
 *                       (relaxed) at exit.  The Semaphores stay untouched.
 *  ARX_SYNC_PAD_FENCED  as ARX_SYNC_PAD with acq_rel compare-and-swaps in all
 *                       three barriers.
 *  ARX_SYNC_CLUSTER     no counterpart on the pages, which synchronise
 *                       separate GPUs: the W blocks of a chunk are one
 *                       thread-block cluster and each of the three barriers
 *                       is the cluster's hardware barrier (relaxed at start
 *                       and exit; release on arrive, acquire on wait after
 *                       staging).  Semaphores and pad are left alone; seq,
 *                       epochs and the counters advance as in the others.
 *                       The hardware barrier's wait has no timeout: it cannot
 *                       stall because every thread arrives unconditionally,
 *                       and the fault-injection knob, which would make a
 *                       block skip an arrival, is refused (ARX_EINVAL).  So
 *                       "every wait is bounded" holds in this mode only in
 *                       that sense.  Slots in host memory are staged in
 *                       turn, as in the flag modes (the fastest host-slot
 *                       step).
 * After every completed step the pad is all zero in every mode; in the pad
 * and cluster modes the Semaphore flags and counters keep their values.
 * Every mode may be selected on any context: the co-residency limit that
 * arx_step checks (B * W blocks resident at once) applies in all of them,
 * because the cooperative modes need it and a context may switch modes. */
#define ARX_SYNC_SEMAPHORE 0
#define ARX_SYNC_PAD 1
#define ARX_SYNC_PAD_FENCED 2
#define ARX_SYNC_CLUSTER 3
#define ARX_SYNC_SEMAPHORE_GLOBAL 4

/* Selects the barrier variant of later steps (ARX_EINVAL for an unknown
 * mode).  Switching between steps is allowed: every mode leaves the pad all
 * zero and reads the Semaphores only as its own barriers wrote them. */
arx_status arx_ctx_set_sync(arx_ctx* ctx, int mode);

/* Testing knob: virtual rank `rank` (0..W-1) skips its end-barrier signal, so
 * the step's waits expire and report ARX_ETIMEOUT; -1 turns it off.  No GPU
 * fault, trap or unbounded wait results. */
arx_status arx_ctx_set_fault(arx_ctx* ctx, int rank);

/* Enqueues a zero fill of the protocol words [0, ctrl_bytes) (not the slots):
 * seq, epochs, Semaphores, pad and the error word all return to zero; clears
 * ctx->failed_err, so steps may be launched again. */
arx_status arx_ctx_reset(arx_ctx* ctx, void* stream);

/* One protocol step: out = rank-order reduce of inputs[0..W-1].
 *   inputs  HOST array of ctx->W device pointers, each to n bf16 elements;
 *           none may overlap the protocol words or the slots (ARX_EOVERLAP).
 *   out     device pointer to n bf16; may equal one input exactly; must not
 *           overlap the protocol words or the slots.
 *   n       0 < n <= ctx->max_n (n == 0 returns ARX_OK, no launch).
 * Steps on one context must be serialised (one stream, or events).  Like the
 * pages' error flag checked before every launch: once arx_ctx_query has read
 * a device error (ctx->failed_err != 0), arx_step returns ARX_ESTATE without
 * launching until arx_ctx_reset. */
arx_status arx_step(const arx_ctx* ctx, const void* const* inputs, void* out, size_t n,
                    void* stream);

/* Synchronises `stream`, then reads the header: *seq = completed steps,
 * *dev_err = device error word (either pointer may be NULL).  Returns the
 * status in the error word's low 8 bits (ARX_OK when it is 0), or ARX_ECUDA.
 * A nonzero error word is also kept in ctx->failed_err (see arx_step). */
arx_status arx_ctx_query(arx_ctx* ctx, uint32_t* seq, uint32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * Bounds checks.  The library can be built a second way, with every data
 * access of its kernels (partials, slots, output) checked against the buffer
 * it belongs to (`python deterministic_shot_all_gb300/_build.py
 * --bounds-check`, which writes libarx_boundscheck.so).  A failed check is
 * counted and the access skipped.  In that build this call reads the count
 * of skipped accesses since the last reset into *count (and zeroes it if
 * reset != 0); it synchronises the device.  The normal build returns
 * ARX_EINVAL: it has no checks.
 * ------------------------------------------------------------------------- */
arx_status arx_bounds_violations(uint32_t* count, int reset);

/* ---------------------------------------------------------------------------
 * Host-side watchdog of the protocol step (arx.cu's proxy watchdog: a step
 * published but not done for too long is reported once as a stall).
 *
 * arx_watch_step polls the context's header words -- completed seq,
 * device error word, published seq -- by a small device-to-host copy on
 * `stream` every poll_ns, without synchronising the stream the steps run on
 * (pass a different, non-blocking stream).  It returns:
 *   ARX_OK        once completed seq has reached target_seq (modulo 2^32);
 *   ARX_ETIMEOUT  if a staged step stays not done (published != completed)
 *                 for stall_ns -- typically while the step kernel is still
 *                 inside its own bounded wait, so the stall is seen before
 *                 the device reports it -- or if max_wait_ns passes first;
 *   ARX_ETIMEOUT / ARX_ESTATE as soon as the device error word is set (its
 *                 low byte);
 *   ARX_EINVAL / ARX_ESTATE / ARX_ECUDA for bad arguments or a failed copy.
 *   host_words   page-locked host memory for 8 uint32 (the copy target).
 *   report       filled on return (may be NULL).
 * It blocks the calling thread: run it on a thread of your own while steps
 * are enqueued elsewhere.  It only reads; it never touches the GPU's work.
 * ------------------------------------------------------------------------- */
typedef struct arx_watch_report {
  uint32_t seq;         /* completed steps at the last poll */
  uint32_t published;   /* last staged step at the last poll */
  uint32_t dev_err;     /* device error word at the last poll */
  uint32_t polls;
  uint64_t stalled_ns;  /* how long published != completed had lasted */
  uint64_t waited_ns;   /* time spent in the call */
} arx_watch_report;

arx_status arx_watch_step(const arx_ctx* ctx, uint32_t target_seq, uint64_t stall_ns,
                          uint64_t poll_ns, uint64_t max_wait_ns, uint32_t* host_words,
                          void* stream, arx_watch_report* report);

/* ---------------------------------------------------------------------------
 * External-writer form: partials written into page-locked host memory by
 * another agent (a host thread), reduced by the GPU.
 *
 * arx.cu's GB10 design: for step seq a CPU proxy has every peer's partial
 * written into pinned recv[seq & 1][rank] and then raises flag[rank]; the
 * kernel waits for the flags with system-scope acquire loads and reads the
 * slots with cache-bypassing loads ("the NIC wrote it"), then sums them in
 * rank order (header comment, steps 1-3; `arx_kernel`, wait phase and reduce
 * loop).  On one GB300 the writer is a host thread standing in for the proxy
 * and the NIC:
 *   producer (host):  arx_ext_post(x, r, seq, src, n) for r = 0..W-1 --
 *                     waits until bank seq & 1 is free (the GPU has consumed
 *                     step seq - 2), copies src into recv[seq & 1][r], then
 *                     release-stores flag[r] = seq;
 *   consumer (GPU):   arx_ext_step(x, out, n, stream) -- step seq = completed
 *                     + 1 waits until every flag[r] has reached seq (bounded
 *                     ld.acquire.sys polls), writes out = the rank-order
 *                     reduce of recv[seq & 1][0..W-1] (ld.global.cv loads),
 *                     and its last block stores seq as completed and, with a
 *                     system-scope release, as `consumed`.
 * Steps are numbered 1, 2, 3, ... from a zero-filled (or reset) context; the
 * producer may run up to two steps ahead of the GPU (the two banks).
 *
 * Host region: page-locked host memory (cudaHostAlloc, cudaHostRegister,
 * torch pin_memory), 256-byte aligned, zero-filled before the first step, of
 * arx_ext_region_bytes(W, max_n) bytes:
 *   [0, 512)     uint32 flag[r] at byte 64 * r (written by the producer)
 *   [512, 516)   uint32 consumed (written by the GPU)
 *   [1024, ...)  bf16 recv[2][W][slot_stride], slot_stride = max_n rounded up
 *                to 128 elements; arx_ext_slot gives a slot's host address
 * Device words: a zero-filled device buffer of arx_ext_words_bytes() bytes,
 * 256-byte aligned: uint32 completed seq, device error word (stage 11: a
 * flag wait expired; rank in bits 12-15, block in bits 16-31), blocks out.
 * Both buffers are the caller's and must outlive the last step.
 * ------------------------------------------------------------------------- */
typedef struct arx_ext {
  uint32_t magic;        /* set by arx_ext_init */
  int32_t W;             /* writers (virtual ranks), 1..ARX_MAX_W */
  int32_t nblocks;       /* thread blocks of a step (at most) */
  int32_t reserved0;
  uint64_t max_n;        /* capacity of one slot, elements */
  uint64_t slot_stride;  /* elements from one slot to the next (multiple of 128) */
  uint64_t timeout_ns;   /* bound of the GPU's flag waits */
  void* words;           /* device words */
  void* host_region;     /* host address of the page-locked region */
  void* dev_region;      /* its device address */
  uint64_t region_bytes;
  uint32_t failed_err;   /* nonzero device error word read by arx_ext_query:
                            arx_ext_step refuses (ARX_ESTATE) until arx_ext_reset */
  uint32_t reserved1;
} arx_ext;

/* Bytes of the host region for W writers and slots of max_n elements (0 for
 * invalid arguments), and of the device words. */
size_t arx_ext_region_bytes(int W, size_t max_n);
size_t arx_ext_words_bytes(void);

/* Fills *x (host struct; no allocation).  dev_words: device buffer (above);
 * host_region: the HOST address of the page-locked region, whose device
 * address the library looks up (ARX_EINVAL if it is not page-locked).
 * nblocks == 0: one 16-byte group of every slot per thread, at most one block
 * per SM. */
arx_status arx_ext_init(arx_ext* x, void* dev_words, size_t words_bytes, void* host_region,
                        size_t region_bytes, int W, size_t max_n, int nblocks);

/* Bound of the GPU's flag waits (ns > 0; default ARX_DEFAULT_TIMEOUT_NS). */
arx_status arx_ext_set_timeout(arx_ext* x, uint64_t ns);

/* Producer side, host only (never enqueues GPU work; any host thread):
 *  arx_ext_wait_free  blocks until bank seq & 1 may be written for step seq
 *                     (consumed >= seq - 2), or returns ARX_ETIMEOUT after
 *                     wait_ns;
 *  arx_ext_slot       host address of recv[seq & 1][rank] (NULL for bad
 *                     arguments), for a producer that writes in place;
 *  arx_ext_publish    release-stores flag[rank] = seq: everything the calling
 *                     thread wrote before (the slot) is visible to the GPU
 *                     once it sees the flag;
 *  arx_ext_post       arx_ext_wait_free, a copy of n bf16 from src into the
 *                     slot, arx_ext_publish;
 *  arx_ext_publish_all  arx_ext_wait_free, then arx_ext_publish for every
 *                     rank: for a producer that wrote all W slots of the
 *                     step in place (through arx_ext_slot).
 * A producer must publish steps of one rank in order, each once. */
arx_status arx_ext_wait_free(const arx_ext* x, uint32_t seq, uint64_t wait_ns);
void* arx_ext_slot(const arx_ext* x, uint32_t seq, int rank);
arx_status arx_ext_publish(const arx_ext* x, int rank, uint32_t seq);
arx_status arx_ext_post(const arx_ext* x, int rank, uint32_t seq, const void* src, size_t n,
                        uint64_t wait_ns);
arx_status arx_ext_publish_all(const arx_ext* x, uint32_t seq, uint64_t wait_ns);

/* Consumer side: enqueues the next step on `stream` (graph-capturable: the
 * step number is read on the device).  out: device pointer to n bf16, not
 * overlapping the region or the words; 0 < n <= max_n (n == 0: ARX_OK, no
 * launch).  Every step of a context must use the same n as its producer
 * posted.  Steps of one context must be serialised (one stream). */
arx_status arx_ext_step(arx_ext* x, void* out, size_t n, void* stream);

/* Synchronises `stream` and reads the device words (as arx_ctx_query);
 * a nonzero error word is kept in x->failed_err. */
arx_status arx_ext_query(arx_ext* x, uint32_t* seq, uint32_t* dev_err, void* stream);

/* Zeroes the device words (enqueued on `stream`, which it then
 * synchronises) and the region's flags and `consumed`; clears failed_err.
 * Call it with no step of the context in flight and no producer running;
 * steps then start again at 1. */
arx_status arx_ext_reset(arx_ext* x, void* stream);

/* ---------------------------------------------------------------------------
 * Allocation-free protocol step.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory at the time
 * they call: a serving engine that reserved nearly all of HBM for its own pool
 * at start-up, a plug-in whose host framework owns every allocation, a
 * serving loop whose rules forbid allocating after start-up, or a
 * latency-critical path that cannot afford the device-wide synchronisation of
 * cudaMalloc/cudaFree.
 *
 * Same operation and result as arx_step, bit for bit, but the workspace is a
 * static device array inside this library (about 4 MiB: ARX_NOALLOC_MAX_N
 * elements x ARX_MAX_W ranks x 2 parity banks, plus the protocol words), held
 * by every GPU that loads the library until the process exits.  Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library routine is called.
 *
 *   inputs      HOST array of W device pointers, each to n bf16 elements.
 *   W           1..ARX_MAX_W virtual ranks.
 *   out         device pointer to n bf16; may equal one input exactly.
 *   n           0 < n <= ARX_NOALLOC_MAX_N; larger n returns ARX_EINVAL with
 *               a message naming the limit (n == 0 returns ARX_OK).
 *   dev_status  optional DEVICE pointer to one uint32, 4-byte aligned: receives
 *               the step's device error word (0 = success; layout as for
 *               arx_step) when the stream reaches it.  NULL skips it.
 *   stream      cudaStream_t as void*.
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress, with the calling thread's device current); nothing is
 * cached, so a context torn down by cudaDeviceReset and created again is
 * served at the array's new address (its contents do not survive the reset).
 * The first call in a context may load this library's device code: make it
 * before any stream capture.  Every call shares the array and
 * first clears its protocol words, so each call is a fresh protocol instance;
 * calls that overlap on the GPU (several streams, or unordered host threads)
 * race on the array and must be serialised by the caller.
 * ------------------------------------------------------------------------- */
#define ARX_NOALLOC_MAX_N 131072
#define ARX_NOALLOC_MAX_BLOCKS 32
arx_status arx_step_noalloc(const void* const* inputs, int W, void* out, size_t n,
                            uint32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ARX_H_ */
