// Internal declarations shared by the library's translation units.
// Nothing here is part of the C ABI (include/symar.h is).
#pragma once

#include <cuda_runtime.h>
#include <atomic>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/symar.h"

namespace symar {

// ----------------------------------------------------------------- constants

constexpr int kMaxRanks = 64;
constexpr size_t kWindowAlign = 4096;        // window stride granularity
constexpr int kVecBytes = 16;                // one 128-bit access
constexpr size_t kPullTileBytes = 16384;     // pull two-shot: bytes of a chunk per flag

// Device status word bits (DevCtx::status[0]).
constexpr uint32_t kStatusTimeout = 1u;      // a bounded wait ran out
constexpr uint32_t kStatusBadArg = 2u;       // a kernel-side range check failed

// Where a wait gave up (DevCtx::status[1]); [2], [3] hold the item coordinates.
enum WaitSite : uint32_t {
    kSiteNone = 0,
    kSiteSignalWait = 1,
    kSiteCounterWait = 2,
    kSitePullFlag = 3,
    kSitePutSignalRecv = 4,
    kSiteBulkStage = 5,
    kSiteSignalChain = 6,      // a put waited for the previous batch's signal of its pair
    kSiteBarrier = 7,          // a rank waited at a barrier for the other ranks' signals
};

// Per-device context: the status block and the arrival ring used by
// multi-CTA puts (and gets) to find the last CTA.  Each launch takes the next
// of kArriveRing counters, so up to that many such launches may be in flight
// at once on a device, across all streams.
//
// status[0] bits, [1] site, [2..3] coordinates of the first wait that ran out
// (read and cleared by sym_stream_status).  A launch's other waits stop early
// through the give-up word of its window (see report_timeout).
struct DevCtx {
    int device = -1;
    int num_sms = 0;
    uint32_t* status = nullptr;   // kStatusWords words, see above
    uint32_t* arrive = nullptr;   // kArriveRing counters, zero when idle
    std::atomic<uint64_t> arrive_next{0};   // host-side ring cursor (calls from several threads)
};
constexpr int kArriveRing = 1024;
constexpr int kStatusWords = 8;

DevCtx* dev_ctx(int device);      // created on first use, lives until exit

}  // namespace symar

// The window: R equal parts of one allocation, plus per-rank slot arrays.
struct sym_window {
    int device;
    int R;
    size_t bytes;          // usable bytes per rank
    size_t stride;         // bytes between rank bases (multiple of 4096)
    char* base;            // device
    bool owns_base;
    uint32_t nsignals, ncounters;
    uint64_t* sig;         // device [R][nsignals]
    uint64_t* cnt;         // device [R][ncounters]
    uint32_t* flags;       // device [R][flag_tiles]: per-tile ready flags (epoch-tagged)
    uint32_t* arrivals;    // device [R][flag_tiles]: per-tile producer counters (zero when idle)
    uint32_t* pair_arrivals;  // device [R][R]: pieces done per (sender, receiver) (zero when idle)
    uint32_t* pair_ring;      // device [R][R][2]: pieces of a batch done, by batch parity (zero when idle)
    size_t flag_tiles;     // flag slots per rank
    uint32_t* epoch;       // device word: epoch of the last waiting launch (bumped on device)
    uint32_t* giveup;      // device word: epoch of the last launch whose wait gave up
    unsigned long long* ticket;   // device word: next work item of a flag-synchronised launch
    void* aux;             // the allocation holding sig, cnt and flags
    symar::DevCtx* ctx;
    int kind;              // SYM_WINDOW_* : how base was allocated
    unsigned long long* vmm_handles;   // VMM windows: one physical allocation per rank
};

namespace symar {

// ----------------------------------------------------------------- host utils

sym_status_t cuda_fail(cudaError_t e, const char* what);   // records the error text
void set_last_error(const char* text);                      // text for sym_last_error()
#define SYM_CUDA(call)                                                   \
    do {                                                                 \
        cudaError_t e_ = (call);                                         \
        if (e_ != cudaSuccess) return ::symar::cuda_fail(e_, #call);     \
    } while (0)

// True when a byte of some rank's range [0, a_bytes) of window `a` is also a
// byte of some rank's range [0, b_bytes) of window `b` (caller memory can make
// two windows alias; interleaved windows that share no byte are not flagged).
bool windows_overlap(const sym_window* a, size_t a_bytes, const sym_window* b, size_t b_bytes);

// Makes `w->device` current for the scope, restoring the previous device.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev);
    ~DeviceGuard();
};

void count_launch(int n = 1);          // sym_launch_count bookkeeping
bool trace_on();
uint64_t default_timeout_ns();
size_t oneshot_max_bytes();
bool twoshot_use_bulk();          // env SYM_TWOSHOT_KERNEL=bulk|ldst
bool allgather_use_bulk();        // env SYM_ALLGATHER_KERNEL=bulk (default)|ldst
bool put_use_bulk();              // env SYM_PUT_KERNEL=bulk (default)|ldst
// Fused pull two-shot kernel for `bytes` per rank: env SYM_PULL_KERNEL=ws (warp-specialised),
// items (single-role), or auto (default: ws above 256 KiB per rank).
bool pull_use_ws(size_t bytes);
// Grid waves between a tile's producing item and the items that wait for it
// (fused pull two-shot); env SYM_PULL_LAG_WAVES, default 4, 1..64.
uint32_t pull_lag_waves();
// Tile blocks between the producers and the consumers of a tile in the fused
// producer + AllReduce; env SYM_FUSED_LAG_BLOCKS, -1 when unset (then about
// one grid wave).
int64_t fused_lag_blocks();
// Fault injection for failure-detection tests: the put + signal AllGather's
// (0 -> 0) stream omits one signal, so a bounded wait runs out.  1 = its last
// signal (env SYM_TEST_DROP_SIGNAL=last, or SYM_TEST_DROP_LAST_SIGNAL=1): the
// stream's receiver waits; 2 = its first signal (SYM_TEST_DROP_SIGNAL=first):
// the stream's next batch waits to signal in order.  0 (default) = off.
// Never needs a GPU fault.
int test_drop_signal();
int occupancy(const void* kernel, int threads, size_t smem);   // blocks per SM, cached
size_t dtype_size(sym_dtype_t t);       // 0 if unknown

inline size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }

// ----------------------------------------------------------------- device utils

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_u64(uint64_t* p, uint64_t v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Strong (relaxed, gpu scope) add; preceded by a fence it forms a release pattern.
__device__ __forceinline__ void red_relaxed_add_u64(uint64_t* p, uint64_t v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Rolling "a <= b" on the low `bits` bits: (b - a) mod 2^bits < 2^(bits-1).
__device__ __forceinline__ bool rolling_le_dev(uint64_t a, uint64_t b, int bits) {
    uint64_t m = bits >= 64 ? ~0ull : ((1ull << bits) - 1ull);
    uint64_t d = (b - a) & m;
    return d < (1ull << (bits - 1));
}

// Records a timeout in the device status block (first site wins) and writes
// this launch's tag into its give-up word, so the launch's other waits stop.
// The give-up word belongs to the window the launch works on (calls on one
// window never overlap), and the tag is the window's device epoch of that
// launch, so a stale give-up never matches a later launch or a graph replay.
__device__ __forceinline__ void report_timeout(uint32_t* status, uint32_t* giveup, uint32_t tag,
                                               uint32_t site, uint32_t a, uint32_t b) {
    uint32_t prev = atomicOr(status, kStatusTimeout);
    if ((prev & kStatusTimeout) == 0) {
        status[1] = site;
        status[2] = a;
        status[3] = b;
    }
    if (giveup && tag) atomicExch(giveup, tag);
}

// Bounded spin: polls pred() with a sleeping back-off until it holds, the
// timeout elapses, an iteration cap is hit, or (giveup != null) another wait
// of the same launch has already given up.  Returns true when pred() held.
template <class Pred>
__device__ __forceinline__ bool bounded_spin(Pred pred, uint64_t timeout_ns,
                                             const uint32_t* giveup, uint32_t tag) {
    if (pred()) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t max_iters = timeout_ns / 16u + 65536u;
    unsigned sleep_ns = 32;
    for (uint64_t it = 1; it <= max_iters; ++it) {
        __nanosleep(sleep_ns);
        if (sleep_ns < 512) sleep_ns <<= 1;
        if (pred()) return true;
        if ((it & 7u) == 0u) {
            if (giveup && tag && ld_volatile_u32(giveup) == tag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
    return false;
}

// Epochs of flag-synchronised launches live on the device: a one-thread
// kernel bumps the window's epoch word in stream order before each such
// launch (never to 0, the value of fresh flags), and the launch reads it at
// start.  A launch recorded in a CUDA graph therefore gets a new epoch on
// every replay.
// The bump also zeroes the window's item ticket (if given) for the launch.
sym_status_t bump_epoch(uint32_t* epoch, cudaStream_t st, unsigned long long* ticket = nullptr);

// Work items of a persistent, flag-synchronised launch are handed out in
// index order by one atomic ticket, not by a static stride: the items in
// flight then stay a compact range (HBM pages close together, like blocks
// of a non-persistent grid), and an item that waits only ever waits for
// items handed out before it, which running blocks already hold.  s_slot is
// a __shared__ pair; every thread of the block must call this.
__device__ __forceinline__ uint64_t fetch_item(unsigned long long* ticket, unsigned long long* s_slot,
                                               int& par) {
    if (threadIdx.x == 0) s_slot[par] = atomicAdd(ticket, 1ull);
    __syncthreads();
    const uint64_t w = s_slot[par];
    par ^= 1;
    return w;
}

__device__ __forceinline__ uint32_t read_epoch(const uint32_t* epoch) {
    __shared__ uint32_t s_epoch;
    if (threadIdx.x == 0) s_epoch = ld_volatile_u32(epoch);
    __syncthreads();
    return s_epoch;
}

// ----------------------------------------------------------------- bulk async copies (TMA engine)
//
// Untiled cp.async.bulk: both addresses 16-byte aligned, size a multiple of 16.
// Loads complete on an mbarrier (transaction bytes); stores complete in bulk
// groups (commit / wait_group).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gsrc, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
        "[%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace symar
