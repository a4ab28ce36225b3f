// Internal declarations shared by the library's translation units.
// Nothing here is part of the C ABI (include/symar.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/symar.h"

namespace symar {

// ----------------------------------------------------------------- constants

constexpr int kMaxRanks = 64;
constexpr size_t kWindowAlign = 4096;        // window stride granularity
constexpr int kVecBytes = 16;                // one 128-bit access

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
};

// Per-device context: the status block and the arrival ring used by
// multi-CTA puts to find the last CTA.
struct DevCtx {
    int device = -1;
    int num_sms = 0;
    uint32_t* status = nullptr;   // [0] bits, [1] site, [2..3] coordinates
    uint32_t* arrive = nullptr;   // kArriveRing counters, zero when idle
    uint64_t arrive_next = 0;     // host-side ring cursor
};
constexpr int kArriveRing = 1024;

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
    uint32_t* flags;       // device [R][flag_tiles]: pull two-shot tile flags
    size_t flag_tiles;     // flag slots per rank
    uint32_t epoch;        // last epoch used for the flags (host)
    void* aux;             // the allocation holding sig, cnt and flags
    symar::DevCtx* ctx;
};

namespace symar {

// ----------------------------------------------------------------- host utils

sym_status_t cuda_fail(cudaError_t e, const char* what);   // records the error text
#define SYM_CUDA(call)                                                   \
    do {                                                                 \
        cudaError_t e_ = (call);                                         \
        if (e_ != cudaSuccess) return ::symar::cuda_fail(e_, #call);     \
    } while (0)

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

// Records a timeout in the device status block (first site wins).
__device__ __forceinline__ void report_timeout(uint32_t* status, uint32_t site, uint32_t a,
                                               uint32_t b) {
    uint32_t prev = atomicOr(status, kStatusTimeout);
    if ((prev & kStatusTimeout) == 0) {
        status[1] = site;
        status[2] = a;
        status[3] = b;
    }
}

// Bounded spin: polls pred() with a sleeping back-off until it holds, the
// timeout elapses, an iteration cap is hit, or another wait of this device
// has already timed out.  Returns true when pred() held.
template <class Pred>
__device__ __forceinline__ bool bounded_spin(Pred pred, uint64_t timeout_ns,
                                             const uint32_t* status) {
    if (pred()) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t max_iters = timeout_ns / 16u + 65536u;
    unsigned sleep_ns = 32;
    for (uint64_t it = 1; it <= max_iters; ++it) {
        __nanosleep(sleep_ns);
        if (sleep_ns < 512) sleep_ns <<= 1;
        if (pred()) return true;
        if ((it & 7u) == 0u) {
            if (ld_volatile_u32(status) & kStatusTimeout) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
    return false;
}

// ----------------------------------------------------------------- launchers

struct ArPlan;   // defined in allreduce.cu

}  // namespace symar
