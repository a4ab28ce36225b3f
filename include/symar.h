/*
 * symar.h -- C ABI of the symmetric-window collectives library (libsymar.so).
 *
 * One GPU holds R "rank windows" of equal layout.  A window is one device
 * allocation; rank r's part starts at base + r * stride (stride a multiple of
 * 4096 bytes), and every address the library touches is base + r*stride + off.
 * The collectives run as hand-written CUDA kernels for sm_103a; no collective
 * library, no second GPU and no host fallback are involved.
 *
 * Sources (web pages, cited by title and section):
 *  [SYMEX] "NCCL symmetric memory windows: examples 01_allreduce /
 *          02_allgather" -- allocation (ncclMemAlloc), window registration
 *          flags and 4096-byte alignment, Example 1 (AllReduce), Example 2
 *          (AllGather), the cleanup order.
 *  [GIN]   "NCCL Device API GIN reference" -- put, signals and counters
 *          (32-bit IDs, 64-bit values, counters of at most 56 bits), strong
 *          and weak signals, readSignal / waitSignal / resetSignal, the
 *          rolling comparison, the barrier's timeout overload.
 *  [LSA]   "NCCL Device API and LSA source notes" -- peer buffers reached by
 *          plain loads and stores at a mapped base plus an offset, 16-byte
 *          vector copies, alignment.
 *  [GDA]   "GPUDirect Async deep dive" -- a batch of puts closed by one
 *          signal; per-chunk counters with release/acquire flags and a
 *          sleeping acquire spin.
 *
 * Conventions
 *  - Every call returns sym_status_t (0 = SYM_OK).  Arguments are checked on
 *    the host before anything is enqueued; a failed check enqueues nothing.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; host buffers handed to
 *    sym_window_write / sym_window_read must stay valid until the stream
 *    reaches that point (pinned memory for overlap).
 *  - Sizes are bytes unless named `count` (elements).  Offsets and sizes of
 *    puts need not be multiples of 16; 16-byte multiples take the vector path.
 *  - Device-side waits are bounded (default 2 s, env SYM_TIMEOUT_NS).  A wait
 *    that runs out sets the device's status word and returns; the host sees it
 *    as SYM_ERR_TIMEOUT from sym_stream_status(); sym_last_error() then names
 *    the wait site: 1 signal wait, 2 counter wait, 3 pull-tile flag, 4 put +
 *    signal / AlltoAll receiver, 5 bulk-copy stage, 6 put + signal batch
 *    order, 7 barrier.  No call traps the GPU.
 *  - Windows are owned by the library (sym_window_alloc) or by the caller
 *    (sym_window_register).  Free a window only after every stream that used
 *    it has finished with it; windows must be freed before unloading.
 *  - Calls that touch the same window on two streams at once race, as
 *    collectives on one communicator do; order them on one stream.
 */
#ifndef SYMAR_H
#define SYMAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: sym_algo_t takes the values of the library's first published table
 * (SYM_ALGO_PUT_SIGNAL = 3; algorithms added later follow it). */
#define SYMAR_ABI_VERSION 2

typedef struct sym_window* sym_win_t;   /* opaque handle */
typedef void* sym_stream_t;             /* a cudaStream_t */

typedef enum {
    SYM_OK = 0,
    SYM_ERR_INVALID_ARG = 1,   /* a host-side argument check failed */
    SYM_ERR_OOM = 2,           /* device allocation failed */
    SYM_ERR_CUDA = 3,          /* a CUDA runtime call failed (sym_last_error()) */
    SYM_ERR_TIMEOUT = 4,       /* a bounded device wait ran out */
    SYM_ERR_UNSUPPORTED = 5,   /* valid request this build does not implement */
    SYM_ERR_DEVICE_STATUS = 6  /* a kernel reported another device-side error */
} sym_status_t;

typedef enum { SYM_F32 = 0, SYM_BF16 = 1, SYM_F16 = 2 } sym_dtype_t;
typedef enum { SYM_SUM = 0, SYM_MAX = 1, SYM_MIN = 2 } sym_op_t;

typedef enum {
    SYM_ALGO_AUTO = 0,
    SYM_ALGO_ONESHOT = 1,        /* AllReduce: every rank-slot reads all R windows, writes its own */
    SYM_ALGO_TWOSHOT = 2,        /* AllReduce: reduce-scatter by loads + all-gather by stores, 1 launch */
    SYM_ALGO_PUT_SIGNAL = 3,     /* AllGather / AlltoAll: chunked puts, one strong signal per batch,
                                    receivers wait */
    /* values added after the four above; existing values never change */
    SYM_ALGO_TWOSHOT_PULL = 4,   /* AllReduce: reduce-scatter, per-tile release flags, pull all-gather,
                                    1 launch */
    SYM_ALGO_TWOSHOT_SPLIT = 5,  /* AllReduce: reduce-scatter launch, then pull all-gather launch */
    SYM_ALGO_COPY = 6,           /* AllGather / AlltoAll: read each segment once, store it to all R
                                    ranks */
    SYM_ALGO_CE = 7              /* AllGather: copy engines, no kernel: one 1-D memcpy per (sender,
                                    destination) */
} sym_algo_t;

/* ---------------------------------------------------------------- windows */

/* Allocate R windows of bytes_per_rank each, plus nsignals signal slots and
 * ncounters counter slots per rank (64-bit, zeroed).
 * [SYMEX] allocation (ncclMemAlloc) and ncclCommWindowRegister with
 * NCCL_WIN_COLL_SYMMETRIC; the 4096-byte window alignment requirement.
 * Layout: one device allocation; rank r at base + r*stride,
 * stride = bytes_per_rank rounded up to 4096.  R in 1..64, bytes_per_rank > 0.
 * Errors: INVALID_ARG, OOM, CUDA.  On error *out is set to NULL. */
sym_status_t sym_window_alloc(int R, size_t bytes_per_rank, uint32_t nsignals,
                              uint32_t ncounters, sym_win_t* out);

/* How a window's memory was obtained (sym_window_kind). */
typedef enum {
    SYM_WINDOW_CUDA_MALLOC = 0,       /* one cudaMalloc of R*stride bytes */
    SYM_WINDOW_REGISTERED = 1,        /* caller memory (sym_window_register) */
    SYM_WINDOW_VMM_EXPORTABLE = 2,    /* VMM, one physical allocation per rank, POSIX-fd handles */
    SYM_WINDOW_VMM = 3                /* VMM, one physical allocation per rank, no exportable handle */
} sym_window_kind_t;

/* The same windows from the virtual-memory API, as [SYMEX]'s symmetric
 * allocator builds them: one physical allocation per rank (cuMemCreate,
 * with a POSIX-file-descriptor handle where the platform allows one), all
 * mapped back to back into one reserved virtual range (cuMemAddressReserve,
 * cuMemMap) with read-write access for the device (cuMemSetAccess).  The
 * layout is the one above -- rank r at base + r*stride -- with stride rounded
 * up to the allocation granularity (2 MiB on GB300), so every collective
 * works on these windows unchanged.  Falls back to one cudaMalloc, as the
 * allocator on the pages does, when the platform has no VMM support;
 * sym_window_kind() tells which.  Errors: INVALID_ARG, CUDA.  On error *out
 * is NULL. */
sym_status_t sym_window_alloc_vmm(int R, size_t bytes_per_rank, uint32_t nsignals,
                                  uint32_t ncounters, sym_win_t* out);

/* sym_window_kind_t of a window; -1 for NULL. */
int sym_window_kind(sym_win_t w);

/* Wrap caller-owned device memory (e.g. a torch tensor) as R windows at
 * base + r*stride.  base must be 256-byte aligned, stride a multiple of 4096
 * and >= bytes_per_rank.  Signal, counter and flag slots are still allocated
 * by the library.  [SYMEX] window registration; unlike NCCL, an unsupported
 * request is an error, never a silent null window.  The caller keeps
 * ownership of base and must free it after sym_window_free. */
sym_status_t sym_window_register(void* base, int R, size_t bytes_per_rank, size_t stride,
                                 uint32_t nsignals, uint32_t ncounters, sym_win_t* out);

/* Release a window (and its memory when the library owns it).  [SYMEX]
 * cleanup order: deregister before freeing.  Synchronises the device first.
 * NULL is accepted and ignored. */
sym_status_t sym_window_free(sym_win_t w);

/* Device address of rank `rank`'s part: base + rank*stride ([LSA] base plus
 * offset addressing).  Errors: INVALID_ARG. */
sym_status_t sym_window_rank_ptr(sym_win_t w, int rank, void** dptr);
size_t sym_window_stride(sym_win_t w);     /* 0 for NULL */
size_t sym_window_bytes(sym_win_t w);      /* bytes_per_rank; 0 for NULL */
int sym_window_nranks(sym_win_t w);        /* R; 0 for NULL */
int sym_window_device(sym_win_t w);        /* CUDA device ordinal; -1 for NULL */

/* Stream-ordered copies between a host (or device) buffer and rank `rank`'s
 * part at byte offset `off`.  off + bytes <= bytes_per_rank.  [SYMEX] steps
 * 4-6 (fill from the host, copy back to verify). */
sym_status_t sym_window_write(sym_win_t w, int rank, size_t off, const void* src, size_t bytes,
                              sym_stream_t stream);
sym_status_t sym_window_read(sym_win_t w, int rank, size_t off, void* dst, size_t bytes,
                             sym_stream_t stream);

/* ---------------------------------------------------------------- collectives */

/* AllReduce over the R rank windows: for every element i < count,
 *   recv_r[i] = ((send_0[i] + send_1[i]) + ...) + send_{R-1}[i]   for all r,
 * added in rank order 0..R-1 (so fp32 results are bit-exact and identical on
 * every rank).  bf16 / fp16 inputs are widened exactly, accumulated in fp32
 * and rounded to nearest-even once.  SYM_MAX / SYM_MIN fold the same values
 * with IEEE 754-2019 maximumNumber / minimumNumber (a NaN operand is ignored;
 * -0 < +0).
 * [SYMEX] Example 1: ncclAllReduce(send, recv, count, float, sum, comm,
 * stream) on symmetric windows; each element is the sum over all ranks.
 * count: elements per rank; count*sizeof(dtype) <= bytes of both windows.
 * send == recv (in place) is allowed for the two-shot algorithms, not for
 * ONESHOT.  Two different windows must not share a byte of the ranges the
 * call touches (possible with sym_window_register): INVALID_ARG, checked on
 * the host.  count == 0 is a no-op.  AUTO picks ONESHOT up to
 * SYM_ONESHOT_MAX_BYTES per rank (env, default 128 KiB), else TWOSHOT.
 * TWOSHOT_PULL enqueues a one-thread kernel that advances the recv window's
 * flag epoch on the device before the main launch, so the call can be
 * recorded into a CUDA graph and replayed; every algorithm only enqueues
 * kernels (no host synchronisation) after its first call on a device.
 * Errors: INVALID_ARG (windows of different R or device, count too large,
 * bad algo), UNSUPPORTED (op/dtype/in-place combination), CUDA. */
sym_status_t sym_allreduce(sym_win_t send, sym_win_t recv, size_t count, sym_dtype_t dtype,
                           sym_op_t op, sym_algo_t algo, sym_stream_t stream);

/* AllReduce that allocates nothing.  The pages have no counterpart: this is
 * an addition for callers that cannot call cudaMalloc -- engines that reserve
 * all device memory at start-up and forbid later allocations, plug-ins whose
 * host framework owns the device allocator, and latency-critical paths that
 * cannot afford the device-wide synchronisation cudaMalloc / cudaFree may do.
 * Every other entry point allocates (windows and their slots), so such a
 * caller passes its own buffers here instead: rank r's input is at
 * send + r*stride and its result goes to recv + r*stride (device pointers,
 * 16-byte aligned, stride a multiple of 16 and >= count*sizeof(dtype)); the
 * R input and R output ranges must not overlap.  The result is the same as
 * sym_allreduce's (rank-order fold in fp32, one rounding for bf16/fp16; any
 * op).  The kernel is the fused pull two-shot; its per-tile flags and status
 * words live in one fixed 256 KiB __device__ array inside this library, which
 * every GPU that loads the library holds until the process exits.
 * Limit: R * ceil(ceil(count*sizeof(dtype)/16/R) / 1024) <= 65536 (one flag
 * per 16 KiB tile of each rank's chunk; about 1 GiB per rank); larger
 * requests return SYM_ERR_INVALID_ARG with the reason in sym_last_error().
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls on a device share the array and it
 * keeps the last call's contents (flags carry an epoch that the host draws
 * for each call at the moment the call is made; the status words, which are
 * diagnostics no call reads back, are cleared at each call), so calls that
 * overlap on the GPU race: order them on one stream.  If a wait for another block's tile ever runs
 * out, the waiting block reduces that tile itself from the inputs, so the
 * result is still complete.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
sym_status_t sym_allreduce_noalloc(const void* send, void* recv, size_t stride, int R, size_t count,
                                   sym_dtype_t dtype, sym_op_t op, sym_stream_t stream);

/* The algorithm AUTO resolves to for this request (host only, no launch). */
sym_status_t sym_allreduce_algo(sym_win_t send, size_t count, sym_dtype_t dtype,
                                sym_algo_t* out);

/* AllGather: recv_r[q*S + i] = send_q[i] for all ranks r, q and bytes
 * i < S = sendcount*sizeof(dtype).  [SYMEX] Example 2: the receive buffer
 * holds sendcount*nranks elements and segment q holds rank q's data.
 * recv bytes_per_rank >= R*S.  send and recv must be different windows that
 * share no byte of the ranges the call touches (INVALID_ARG).
 * algo: AUTO or COPY (SM kernel: each 16 KiB segment tile is loaded once
 * into shared memory by a bulk copy and stored to the R ranks by R bulk
 * copies; env SYM_ALLGATHER_KERNEL=ldst selects a register load/store kernel
 * instead), CE ([SYMEX] Example 2's copy-engine policy, CTAPolicy ZERO: no SM
 * is used; R*R cudaMemcpyAsync copies, one per (sender, destination)
 * pair, sender-major), or PUT_SIGNAL (see sym_allgather_put_signal, with chunk_bytes
 * and chunks_per_signal; 0 selects 64 KiB and 8).  For COPY and CE the two
 * chunk arguments are ignored. */
sym_status_t sym_allgather(sym_win_t send, sym_win_t recv, size_t sendcount, sym_dtype_t dtype,
                           sym_algo_t algo, size_t chunk_bytes, uint32_t chunks_per_signal,
                           sym_stream_t stream);

/* Chunked put + signal AllGather in one launch.
 * [GIN] put with remoteAction SignalInc and localAction CounterInc; strong
 * signals; [GDA] a batch of puts closed by one signal.
 * Every sender q puts its S bytes to every peer p (p = q included, [GIN]
 * loopback) in chunks of chunk_bytes, in ascending order; after every
 * chunks_per_signal chunks of a (q, p) stream, and after its last chunk, it
 * adds 1 to signal slot q of rank p in `recv` as a strong signal: once a
 * receiver sees the value k, batches 0..k-1 from q are visible in its window.
 * Each put adds 1 to counter slot 0 of rank q in `send`.  Signal slots 0..R-1
 * of every rank of `recv` and counter slot 0 of every rank of `send` are set
 * to 0 first (stream-ordered), so afterwards signal[p][q] ==
 * ceil(ceil(S/chunk)/batch) and counter[q] == R*ceil(S/chunk).
 * Batches of different (q, p) streams run in parallel; the signals of one
 * stream are added in batch order (the put of batch k waits, bounded, until
 * the stream's signal reads k).  When S and chunk_bytes are multiples of 16
 * the bytes move by bulk copies through shared memory (TMA engine), the R
 * puts of one source range of a sender sharing one read; env
 * SYM_PUT_KERNEL=ldst selects register copies per stream, as do other sizes.
 * The same launch holds the receivers: each (p, q) waits (bounded by
 * timeout_ns, 0 = default) until its signal reaches that count.
 * If d_mismatch (device pointer to one uint64) is not NULL, receivers check
 * prefix visibility while the senders run: once signal[p][q] reads k+1 they
 * compare batch k with the source and add differing bytes to *d_mismatch
 * (expected 0).  Requires recv nsignals >= R, send ncounters >= 1.
 * If one receiver's wait runs out, the launch's other waits stop early (each
 * launch is tagged with the recv window's device epoch).  For failure tests,
 * env SYM_TEST_DROP_SIGNAL=last (or SYM_TEST_DROP_LAST_SIGNAL=1) makes the
 * (0 -> 0) stream omit its last signal, so that receiver's wait runs out
 * (site 4); SYM_TEST_DROP_SIGNAL=first makes it omit its first signal, so the
 * stream's next batch runs out waiting to signal in order (site 6).  Read once
 * per process; off by default.
 * Errors: INVALID_ARG, CUDA; a wait that runs out -> SYM_ERR_TIMEOUT from
 * sym_stream_status(). */
sym_status_t sym_allgather_put_signal(sym_win_t send, sym_win_t recv, size_t bytes_per_rank,
                                      size_t chunk_bytes, uint32_t chunks_per_signal,
                                      uint64_t* d_mismatch, uint64_t timeout_ns,
                                      sym_stream_t stream);

/* AlltoAll: recv_p[q*B + i] = send_q[p*B + i] for all ranks p, q and bytes
 * i < B = count*sizeof(dtype); both windows hold R segments of B bytes per
 * rank.  [GIN] pure-GIN AlltoAll example: every rank puts `count` elements
 * to every rank (itself included) at my_rank*count of the receiver's buffer,
 * each put incrementing one signal; the receiver waits for nRanks
 * increments.  algo COPY (or AUTO): one launch of plain segment copies.
 * algo PUT_SIGNAL: the same copies, each followed by a release increment of
 * signal slot 0 of the receiving rank (reset to 0 first, stream-ordered), and
 * receivers in the same launch wait (bounded by timeout_ns, 0 = default)
 * until it reaches R; requires recv nsignals >= 1.  send and recv must be
 * different windows that share no byte of the ranges the call touches.
 * Errors: INVALID_ARG, CUDA; a wait that runs out -> SYM_ERR_TIMEOUT from
 * sym_stream_status(). */
sym_status_t sym_alltoall(sym_win_t send, sym_win_t recv, size_t count, sym_dtype_t dtype,
                          sym_algo_t algo, uint64_t timeout_ns, sym_stream_t stream);

/* Producer + AllReduce in one launch.  Every rank r first produces its
 * contribution s_r[i] = alpha[r] * in_r[i] (one fp32 multiply, rounded to
 * nearest) into `send`; then recv_r[i] = s_0[i] + s_1[i] + ... + s_{R-1}[i]
 * (rank order, fp32) for every rank r.  [GDA] section 5.1 (fused GEMM +
 * AllReduce): producer tiles bump a per-tile counter, the R-th arrival
 * publishes the tile's flag with a release store, and the reduction of that
 * tile starts as soon as it acquires the flag, overlapping the production of
 * later tiles.  alpha: host array of R floats (copied at the call).  f32
 * only; the three windows must have the same R and share no byte of the
 * ranges the call touches.  count
 * elements per rank.  Errors: INVALID_ARG, UNSUPPORTED, CUDA; a wait that
 * runs out -> SYM_ERR_TIMEOUT from sym_stream_status(). */
sym_status_t sym_scale_allreduce(sym_win_t in, sym_win_t send, sym_win_t recv, const float* alpha,
                                 size_t count, sym_stream_t stream);

/* ---------------------------------------------------------------- one-sided */

/* put: copy `bytes` from rank src_rank's part of `src` at src_off to rank
 * `peer`'s part of `dst` at dst_off, then (signal_id != UINT32_MAX) add 1 to
 * signal slot signal_id of rank `peer` in `dst` as a strong signal, and
 * (counter_id != UINT32_MAX) add 1 to counter slot counter_id of rank
 * src_rank in `src`.  [GIN] put(team, peer, dstWnd, dstOffset, srcWnd,
 * srcOffset, bytes, remoteAction, localAction); peer may equal src_rank.
 * Ordering: the signal is made visible after every byte of this put, and
 * calls on one stream are ordered, so a signal seen by a later waiter on the
 * stream covers all earlier puts on it (the stream plays the GIN context).
 * Ranges must lie inside the windows; src and dst ranges must not overlap.
 * Errors: INVALID_ARG, CUDA. */
sym_status_t sym_put_signal(sym_win_t src, sym_win_t dst, int src_rank, int peer, size_t dst_off,
                            size_t src_off, size_t bytes, uint32_t signal_id, uint32_t counter_id,
                            sym_stream_t stream);

/* get: the one-sided read, the reverse of put.  Copies `bytes` from rank
 * `peer`'s part of `remote` at remote_off into rank `rank`'s part of `local`
 * at local_off.  [GIN] get(team, peer, remoteWnd, remoteOffset, localWnd,
 * localOffset, bytes, ...): no remote action; the page's flush() is what
 * makes the data visible to the reader, and on one GPU the stream order does
 * that.  For in-kernel consumers, counter_id != UINT32_MAX adds 1 to counter
 * slot counter_id of rank `rank` in `local` once every byte has landed
 * (UINT32_MAX = none).  peer may equal rank (loopback) when the ranges do
 * not overlap.  Ranges must lie inside the windows.  bytes == 0 with no
 * counter is a no-op.  Errors: INVALID_ARG, CUDA. */
sym_status_t sym_get(sym_win_t remote, sym_win_t local, int rank, int peer, size_t local_off,
                     size_t remote_off, size_t bytes, uint32_t counter_id, sym_stream_t stream);

/* Barrier across the R rank slots of `w` on signal slot signal_id.  [GIN]
 * ncclGinBarrierSession::sync with the strongest fence (Put | Get): every
 * rank adds 1 to that slot of every rank with a release, then waits
 * (acquire, bounded by timeout_ns, 0 = default) until its own slot has
 * received all R adds, so work enqueued after the barrier sees everything
 * every rank did before it.  Each barrier adds exactly R to every rank's
 * slot; the slot must be used by nothing else.  A barrier that runs out
 * (SYM_ERR_TIMEOUT, site 7) leaves the slots short: reset them
 * (sym_signal_reset on every rank) before the next barrier.  One cooperative
 * launch of R blocks.  Errors: INVALID_ARG, CUDA. */
sym_status_t sym_barrier(sym_win_t w, uint32_t signal_id, uint64_t timeout_ns, sym_stream_t stream);

/* Signal without data: add `value` to signal slot signal_id of rank `peer`
 * ([GIN] signal() with a SignalAdd action), with release ordering. */
sym_status_t sym_signal(sym_win_t dst, int peer, uint32_t signal_id, uint64_t value,
                        sym_stream_t stream);

/* Enqueue a bounded device wait until the low `bits` bits (1..64) of signal
 * slot signal_id of rank `rank` are rolling-greater-or-equal to `least`:
 * with m = 2^bits - 1, done when ((v & m) - least) mod 2^bits < 2^(bits-1).
 * [GIN] waitSignal(coop, signal, least, bits) and the rolling comparison.
 * Later work on `stream` starts after the wait ends.  timeout_ns 0 = default.
 * A wait that runs out sets the device status (see sym_stream_status). */
sym_status_t sym_signal_wait(sym_win_t w, int rank, uint32_t signal_id, uint64_t least, int bits,
                             uint64_t timeout_ns, sym_stream_t stream);

/* Read the low `bits` bits (1..64) of a signal after the work queued on
 * `stream` ([GIN] readSignal(signal, bits)); synchronises `stream`.  `bits`
 * and `stream` extend the first published signature (w, rank, id, out):
 * readSignal takes a width, and on one GPU the read must be ordered after the
 * stream's own puts. */
sym_status_t sym_signal_read(sym_win_t w, int rank, uint32_t signal_id, int bits, uint64_t* out,
                             sym_stream_t stream);

/* Set a signal to 0 ([GIN] resetSignal; must not race with other updates). */
sym_status_t sym_signal_reset(sym_win_t w, int rank, uint32_t signal_id, sym_stream_t stream);

/* Counters ([GIN] readCounter / waitCounter / resetCounter): the same as the
 * signal calls, on counter slots; values are read through at most 56 bits
 * (bits 1..56).  sym_counter_read takes `bits` and `stream` for the same
 * reasons as sym_signal_read. */
sym_status_t sym_counter_read(sym_win_t w, int rank, uint32_t counter_id, int bits, uint64_t* out,
                              sym_stream_t stream);
sym_status_t sym_counter_wait(sym_win_t w, int rank, uint32_t counter_id, uint64_t least, int bits,
                              uint64_t timeout_ns, sym_stream_t stream);
sym_status_t sym_counter_reset(sym_win_t w, int rank, uint32_t counter_id, sym_stream_t stream);

/* ---------------------------------------------------------------- status */

/* Synchronise `stream`, then report and clear the current device's status
 * word: SYM_ERR_TIMEOUT if a bounded device wait of this library ran out
 * since the last call, SYM_ERR_CUDA on a CUDA error, else SYM_OK.  [GIN] the
 * barrier's timeoutCycles overload (a wait that gives up instead of hanging).
 * sym_allreduce_noalloc's waits are not reported here: a gather of that entry
 * that gives up reduces its tile itself, so its result is complete anyway. */
sym_status_t sym_stream_status(sym_stream_t stream);

const char* sym_status_string(sym_status_t s);
/* Text of the last CUDA error seen by this thread ("" if none). */
const char* sym_last_error(void);
/* Number of kernels this library has launched in this process. */
uint64_t sym_launch_count(void);
int sym_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SYMAR_H */
