// Symmetric windows: allocation, registration, addressing, host copies,
// per-device status, and the library's host-side bookkeeping.
//
// [SYMEX] "NCCL symmetric memory windows" guide: ncclMemAlloc and
// ncclCommWindowRegister(NCCL_WIN_COLL_SYMMETRIC) give every rank a buffer of
// the same size and layout, registration requires 4096-byte alignment, and
// windows are deregistered before their memory is freed.  Here all R ranks
// live in one allocation at base + r*stride ([LSA] "base plus offset"), so a
// peer address is pure integer arithmetic and every kernel can reach every
// rank with ordinary loads and stores.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "symar_internal.cuh"

namespace symar {

static thread_local char g_last_error[256] = "";
static std::atomic<uint64_t> g_launches{0};

sym_status_t cuda_fail(cudaError_t e, const char* what) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", what, cudaGetErrorString(e),
             cudaGetErrorName(e));
    if (trace_on()) fprintf(stderr, "[symar] CUDA error %s\n", g_last_error);
    return e == cudaErrorMemoryAllocation ? SYM_ERR_OOM : SYM_ERR_CUDA;
}

void set_last_error(const char* text) {
    snprintf(g_last_error, sizeof g_last_error, "%s", text);
}

bool windows_overlap(const sym_window* a, size_t a_bytes, const sym_window* b, size_t b_bytes) {
    if (a_bytes == 0 || b_bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a->base, b0 = (uintptr_t)b->base;
    const uintptr_t a1 = a0 + (size_t)(a->R - 1) * a->stride + a_bytes;
    const uintptr_t b1 = b0 + (size_t)(b->R - 1) * b->stride + b_bytes;
    if (a1 <= b0 || b1 <= a0) return false;          // the extents are apart
    // interleaved windows can share an extent without sharing a byte: compare
    // the R x R rank ranges one by one (R <= 64)
    for (int i = 0; i < a->R; ++i) {
        const uintptr_t s = a0 + (size_t)i * a->stride, e = s + a_bytes;
        for (int j = 0; j < b->R; ++j) {
            const uintptr_t t = b0 + (size_t)j * b->stride;
            if (s < t + b_bytes && t < e) return true;
        }
    }
    return false;
}

DeviceGuard::DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
        prev = -1;
        ok = false;
        return;
    }
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
}

DeviceGuard::~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static uint64_t env_u64(const char* name, uint64_t dflt) {
    const char* s = getenv(name);
    if (!s || !*s) return dflt;
    char* end = nullptr;
    unsigned long long v = strtoull(s, &end, 0);
    return (end && *end == 0) ? (uint64_t)v : dflt;
}

bool trace_on() {
    static const bool on = env_u64("SYM_TRACE", 0) != 0;
    return on;
}

uint64_t default_timeout_ns() {
    // bounded: at most 60 s whatever the environment says
    static const uint64_t t = [] {
        uint64_t v = env_u64("SYM_TIMEOUT_NS", 2000000000ull);
        if (v == 0) v = 2000000000ull;
        return v > 60000000000ull ? 60000000000ull : v;
    }();
    return t;
}

size_t oneshot_max_bytes() {
    // measured crossover on GB300 (R = 8, device time per call from CUDA-graph
    // replay): one-shot is faster up to 64 KiB per rank, two-shot from 256 KiB;
    // the default splits the gap (geometric mean)
    static const size_t v = (size_t)env_u64("SYM_ONESHOT_MAX_BYTES", 131072);
    return v;
}

uint32_t pull_lag_waves() {
    static const uint32_t v = [] {
        uint64_t w = env_u64("SYM_PULL_LAG_WAVES", 4);
        return (uint32_t)(w < 1 ? 1 : (w > 64 ? 64 : w));
    }();
    return v;
}

int test_drop_signal() {
    static const int v = [] {
        const char* s = getenv("SYM_TEST_DROP_SIGNAL");
        if (s && strcmp(s, "first") == 0) return 2;
        if (s && strcmp(s, "last") == 0) return 1;
        return env_u64("SYM_TEST_DROP_LAST_SIGNAL", 0) != 0 ? 1 : 0;
    }();
    return v;
}

bool twoshot_use_bulk() {
    static const bool v = [] {
        const char* s = getenv("SYM_TWOSHOT_KERNEL");
        return s && strcmp(s, "bulk") == 0;
    }();
    return v;
}

bool pull_use_ws(size_t bytes) {
    static const int mode = [] {          // 0 auto, 1 ws, 2 items
        const char* s = getenv("SYM_PULL_KERNEL");
        if (s && strcmp(s, "ws") == 0) return 1;
        if (s && strcmp(s, "items") == 0) return 2;
        return 0;
    }();
    return mode == 1 || (mode == 0 && bytes > (size_t)256 * 1024);
}

int64_t fused_lag_blocks() {
    static const int64_t v = [] {
        const uint64_t none = ~0ull;
        uint64_t b = env_u64("SYM_FUSED_LAG_BLOCKS", none);
        return b == none ? (int64_t)-1 : (int64_t)(b > 4096 ? 4096 : b);
    }();
    return v;
}

bool put_use_bulk() {
    static const bool v = [] {
        const char* s = getenv("SYM_PUT_KERNEL");
        return !(s && strcmp(s, "ldst") == 0);
    }();
    return v;
}

bool allgather_use_bulk() {
    static const bool v = [] {
        const char* s = getenv("SYM_ALLGATHER_KERNEL");
        return !(s && strcmp(s, "ldst") == 0);
    }();
    return v;
}

size_t dtype_size(sym_dtype_t t) {
    switch (t) {
        case SYM_F32: return 4;
        case SYM_BF16: return 2;
        case SYM_F16: return 2;
    }
    return 0;
}

int occupancy(const void* kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(dev, kernel);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
        n = 1;
    if (n < 1) n = 1;
    cache[key] = n;
    return n;
}

DevCtx* dev_ctx(int device) {
    static std::mutex mu;
    static std::map<int, DevCtx*> ctxs;
    std::lock_guard<std::mutex> lk(mu);
    auto it = ctxs.find(device);
    if (it != ctxs.end()) return it->second;
    DeviceGuard g(device);
    if (!g.ok) return nullptr;
    DevCtx* c = new DevCtx();
    c->device = device;
    if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        c->num_sms = 1;
    const size_t words = kStatusWords + kArriveRing;
    uint32_t* mem = nullptr;
    if (cudaMalloc(&mem, words * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(mem, 0, words * sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return nullptr;
    }
    c->status = mem;
    c->arrive = mem + kStatusWords;
    ctxs[device] = c;
    return c;
}

__global__ void k_bump_epoch(uint32_t* epoch, unsigned long long* ticket) {
    uint32_t e = *epoch + 1u;
    *epoch = e ? e : 1u;
    if (ticket) *ticket = 0ull;
}

sym_status_t bump_epoch(uint32_t* epoch, cudaStream_t st, unsigned long long* ticket) {
    k_bump_epoch<<<1, 1, 0, st>>>(epoch, ticket);
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

}  // namespace symar

using namespace symar;

// Slot arrays and flags for a window: one allocation, zeroed.
static sym_status_t alloc_aux(sym_window* w) {
    // pull two-shot: one flag per (rank-slot, tile) of a chunk
    size_t chunk_bytes = ceil_div(ceil_div(w->bytes, (size_t)kVecBytes), (size_t)w->R) * kVecBytes;
    w->flag_tiles = ceil_div(chunk_bytes, kPullTileBytes) + 1;
    size_t sig_b = sizeof(uint64_t) * (size_t)w->R * w->nsignals;
    size_t cnt_b = sizeof(uint64_t) * (size_t)w->R * w->ncounters;
    size_t flg_b = sizeof(uint32_t) * (size_t)w->R * w->flag_tiles;
    size_t pair_b = sizeof(uint32_t) * (size_t)w->R * w->R;
    size_t ring_b = 2 * pair_b;      // [R][R][2] per-stream batch arrival ring
    // the item ticket (u64) leads, so every u64 array stays 8-byte aligned
    size_t total = sizeof(uint64_t) + sig_b + cnt_b + 2 * flg_b + pair_b + ring_b + 2 * sizeof(uint32_t);
    char* p = nullptr;
    SYM_CUDA(cudaMalloc(&p, total));
    cudaError_t e = cudaMemset(p, 0, total);
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "cudaMemset(window slots)");
    }
    w->aux = p;
    w->ticket = (unsigned long long*)p;
    p += sizeof(uint64_t);
    w->sig = (uint64_t*)p;
    w->cnt = (uint64_t*)(p + sig_b);
    w->flags = (uint32_t*)(p + sig_b + cnt_b);
    w->arrivals = (uint32_t*)(p + sig_b + cnt_b + flg_b);
    w->pair_arrivals = (uint32_t*)(p + sig_b + cnt_b + 2 * flg_b);
    w->pair_ring = (uint32_t*)(p + sig_b + cnt_b + 2 * flg_b + pair_b);
    w->epoch = (uint32_t*)(p + sig_b + cnt_b + 2 * flg_b + pair_b + ring_b);
    w->giveup = w->epoch + 1;
    return SYM_OK;
}

// ----------------------------------------------------------------- VMM windows
//
// [SYMEX] memory allocation: the symmetric allocator creates physical memory
// with cuMemCreate (an exportable handle where the platform allows),
// reserves a virtual range with cuMemAddressReserve, maps the memory there
// with cuMemMap and grants access with cuMemSetAccess, and falls back to
// cudaMalloc.  Here each rank's window is its own physical allocation, mapped
// at base + r*stride of one reserved range, so the kernels' base + r*stride
// addressing is unchanged.  The driver calls are looked up through the
// runtime (cudaGetDriverEntryPointByVersion): the library does not link the
// driver library itself.
struct VmmApi {
    PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
    PFN_cuMemCreate_v10020 create = nullptr;
    PFN_cuMemRelease_v10020 release = nullptr;
    PFN_cuMemAddressReserve_v10020 reserve = nullptr;
    PFN_cuMemAddressFree_v10020 addr_free = nullptr;
    PFN_cuMemMap_v10020 map = nullptr;
    PFN_cuMemUnmap_v10020 unmap = nullptr;
    PFN_cuMemSetAccess_v10020 set_access = nullptr;
    bool ok = false;
};

static const VmmApi& vmm_api() {
    static const VmmApi api = [] {
        VmmApi a;
        auto get = [](const char* name, void** fn) {
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) ==
                       cudaSuccess &&
                   q == cudaDriverEntryPointSuccess && *fn != nullptr;
        };
        a.ok = get("cuMemGetAllocationGranularity", (void**)&a.granularity) &&
               get("cuMemCreate", (void**)&a.create) && get("cuMemRelease", (void**)&a.release) &&
               get("cuMemAddressReserve", (void**)&a.reserve) &&
               get("cuMemAddressFree", (void**)&a.addr_free) && get("cuMemMap", (void**)&a.map) &&
               get("cuMemUnmap", (void**)&a.unmap) && get("cuMemSetAccess", (void**)&a.set_access);
        return a;
    }();
    return api;
}

// Undo a (possibly partial) VMM window: unmap and release `mapped` ranks,
// then free the reserved range.
static void vmm_release(char* base, size_t stride, int R, const unsigned long long* h, int mapped) {
    const VmmApi& v = vmm_api();
    for (int r = 0; r < mapped; ++r) {
        v.unmap((CUdeviceptr)(base + (size_t)r * stride), stride);
        v.release((CUmemGenericAllocationHandle)h[r]);
    }
    if (base) v.addr_free((CUdeviceptr)base, stride * (size_t)R);
}

// R physical allocations of `stride` bytes mapped back to back; kind reports
// whether the memory carries an exportable (POSIX file descriptor) handle.
static sym_status_t vmm_alloc(int dev, int R, size_t stride, char** base_out,
                              unsigned long long** handles_out, int* kind_out) {
    const VmmApi& v = vmm_api();
    if (!v.ok) return SYM_ERR_UNSUPPORTED;
    for (int attempt = 0; attempt < 2; ++attempt) {
        CUmemAllocationProp prop = {};
        prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
        prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
        prop.location.id = dev;
        prop.requestedHandleTypes =
            attempt == 0 ? CU_MEM_HANDLE_TYPE_POSIX_FILE_DESCRIPTOR : CU_MEM_HANDLE_TYPE_NONE;
        size_t gran = 0;
        if (v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS || !gran ||
            stride % gran != 0)
            continue;
        CUdeviceptr base = 0;
        if (v.reserve(&base, stride * (size_t)R, gran, 0, 0) != CUDA_SUCCESS) continue;
        unsigned long long* h = new unsigned long long[R]();
        int mapped = 0;
        bool ok = true;
        for (int r = 0; r < R && ok; ++r) {
            CUmemGenericAllocationHandle hr = 0;
            if (v.create(&hr, stride, &prop, 0) != CUDA_SUCCESS) {
                ok = false;
                break;
            }
            if (v.map(base + (CUdeviceptr)((size_t)r * stride), stride, 0, hr, 0) != CUDA_SUCCESS) {
                v.release(hr);
                ok = false;
                break;
            }
            h[r] = (unsigned long long)hr;
            ++mapped;
        }
        if (ok) {
            CUmemAccessDesc acc = {};
            acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
            acc.location.id = dev;
            acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
            ok = v.set_access(base, stride * (size_t)R, &acc, 1) == CUDA_SUCCESS;
        }
        if (!ok) {
            vmm_release((char*)base, stride, R, h, mapped);
            delete[] h;
            continue;
        }
        *base_out = (char*)base;
        *handles_out = h;
        *kind_out = attempt == 0 ? SYM_WINDOW_VMM_EXPORTABLE : SYM_WINDOW_VMM;
        return SYM_OK;
    }
    return SYM_ERR_UNSUPPORTED;
}

static size_t vmm_granularity(int dev) {
    const VmmApi& v = vmm_api();
    if (!v.ok) return 0;
    CUmemAllocationProp prop = {};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = dev;
    size_t gran = 0;
    if (v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS) return 0;
    return gran;
}

static sym_status_t make_window(void* base, bool owns, int R, size_t bytes, size_t stride,
                                uint32_t nsig, uint32_t ncnt, sym_win_t* out, bool vmm = false) {
    int dev = 0;
    SYM_CUDA(cudaGetDevice(&dev));
    DevCtx* ctx = dev_ctx(dev);
    if (!ctx) return SYM_ERR_CUDA;
    sym_window* w = new sym_window();
    w->device = dev;
    w->R = R;
    w->bytes = bytes;
    w->stride = stride;
    w->owns_base = owns;
    w->nsignals = nsig;
    w->ncounters = ncnt;
    w->ctx = ctx;
    w->aux = nullptr;
    w->kind = owns ? SYM_WINDOW_CUDA_MALLOC : SYM_WINDOW_REGISTERED;
    w->vmm_handles = nullptr;
    if (owns && vmm) {
        // the VMM path; a platform without it falls back to cudaMalloc below
        char* p = nullptr;
        if (vmm_alloc(dev, R, stride, &p, &w->vmm_handles, &w->kind) == SYM_OK) w->base = p;
        else vmm = false;
    }
    if (owns && !vmm) {
        char* p = nullptr;
        cudaError_t e = cudaMalloc(&p, stride * (size_t)R);
        if (e != cudaSuccess) {
            delete w;
            return cuda_fail(e, "cudaMalloc(window)");
        }
        w->base = p;
        w->kind = SYM_WINDOW_CUDA_MALLOC;
    } else if (!owns) {
        w->base = (char*)base;
    }
    sym_status_t s = alloc_aux(w);
    if (s != SYM_OK) {
        if (w->vmm_handles) {
            vmm_release(w->base, w->stride, w->R, w->vmm_handles, w->R);
            delete[] w->vmm_handles;
        } else if (owns) {
            cudaFree(w->base);
        }
        delete w;
        return s;
    }
    *out = w;
    return SYM_OK;
}

extern "C" {

sym_status_t sym_window_alloc(int R, size_t bytes_per_rank, uint32_t nsignals, uint32_t ncounters,
                              sym_win_t* out) {
    if (!out) return SYM_ERR_INVALID_ARG;
    *out = nullptr;
    if (R < 1 || R > kMaxRanks || bytes_per_rank == 0) return SYM_ERR_INVALID_ARG;
    if (nsignals > (1u << 20) || ncounters > (1u << 20)) return SYM_ERR_INVALID_ARG;
    if (bytes_per_rank > ((size_t)1 << 40)) return SYM_ERR_INVALID_ARG;
    size_t stride = ceil_div(bytes_per_rank, kWindowAlign) * kWindowAlign;
    return make_window(nullptr, true, R, bytes_per_rank, stride, nsignals, ncounters, out);
}

sym_status_t sym_window_alloc_vmm(int R, size_t bytes_per_rank, uint32_t nsignals,
                                  uint32_t ncounters, sym_win_t* out) {
    if (!out) return SYM_ERR_INVALID_ARG;
    *out = nullptr;
    if (R < 1 || R > kMaxRanks || bytes_per_rank == 0) return SYM_ERR_INVALID_ARG;
    if (nsignals > (1u << 20) || ncounters > (1u << 20)) return SYM_ERR_INVALID_ARG;
    if (bytes_per_rank > ((size_t)1 << 40)) return SYM_ERR_INVALID_ARG;
    int dev = 0;
    SYM_CUDA(cudaGetDevice(&dev));
    size_t align = kWindowAlign;
    const size_t gran = vmm_granularity(dev);
    if (gran > align && gran % kWindowAlign == 0) align = gran;   // whole physical pages per rank
    const size_t stride = ceil_div(bytes_per_rank, align) * align;
    return make_window(nullptr, true, R, bytes_per_rank, stride, nsignals, ncounters, out, true);
}

int sym_window_kind(sym_win_t w) { return w ? w->kind : -1; }

sym_status_t sym_window_register(void* base, int R, size_t bytes_per_rank, size_t stride,
                                 uint32_t nsignals, uint32_t ncounters, sym_win_t* out) {
    if (!out) return SYM_ERR_INVALID_ARG;
    *out = nullptr;
    if (!base || R < 1 || R > kMaxRanks || bytes_per_rank == 0) return SYM_ERR_INVALID_ARG;
    if (((uintptr_t)base & 255u) != 0 || stride % kWindowAlign != 0 || stride < bytes_per_rank)
        return SYM_ERR_INVALID_ARG;
    if (nsignals > (1u << 20) || ncounters > (1u << 20)) return SYM_ERR_INVALID_ARG;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, base);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return SYM_ERR_INVALID_ARG;
    int dev = 0;
    SYM_CUDA(cudaGetDevice(&dev));
    if (attr.device != dev) return SYM_ERR_INVALID_ARG;
    return make_window(base, false, R, bytes_per_rank, stride, nsignals, ncounters, out);
}

sym_status_t sym_window_free(sym_win_t w) {
    if (!w) return SYM_OK;
    DeviceGuard g(w->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (w->aux) cudaFree(w->aux);
    if (w->vmm_handles) {
        vmm_release(w->base, w->stride, w->R, w->vmm_handles, w->R);
        delete[] w->vmm_handles;
    } else if (w->owns_base && w->base) {
        cudaFree(w->base);
    }
    delete w;
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize(window_free)");
    return SYM_OK;
}

sym_status_t sym_window_rank_ptr(sym_win_t w, int rank, void** dptr) {
    if (!w || !dptr || rank < 0 || rank >= w->R) return SYM_ERR_INVALID_ARG;
    *dptr = w->base + (size_t)rank * w->stride;
    return SYM_OK;
}

size_t sym_window_stride(sym_win_t w) { return w ? w->stride : 0; }
size_t sym_window_bytes(sym_win_t w) { return w ? w->bytes : 0; }
int sym_window_nranks(sym_win_t w) { return w ? w->R : 0; }
int sym_window_device(sym_win_t w) { return w ? w->device : -1; }

sym_status_t sym_window_write(sym_win_t w, int rank, size_t off, const void* src, size_t bytes,
                              sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || (!src && bytes)) return SYM_ERR_INVALID_ARG;
    if (off > w->bytes || bytes > w->bytes - off) return SYM_ERR_INVALID_ARG;
    if (bytes == 0) return SYM_OK;
    DeviceGuard g(w->device);
    SYM_CUDA(cudaMemcpyAsync(w->base + (size_t)rank * w->stride + off, src, bytes, cudaMemcpyDefault,
                             (cudaStream_t)stream));
    return SYM_OK;
}

sym_status_t sym_window_read(sym_win_t w, int rank, size_t off, void* dst, size_t bytes,
                             sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || (!dst && bytes)) return SYM_ERR_INVALID_ARG;
    if (off > w->bytes || bytes > w->bytes - off) return SYM_ERR_INVALID_ARG;
    if (bytes == 0) return SYM_OK;
    DeviceGuard g(w->device);
    SYM_CUDA(cudaMemcpyAsync(dst, w->base + (size_t)rank * w->stride + off, bytes, cudaMemcpyDefault,
                             (cudaStream_t)stream));
    return SYM_OK;
}

sym_status_t sym_stream_status(sym_stream_t stream) {
    int dev = 0;
    SYM_CUDA(cudaGetDevice(&dev));
    SYM_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    SYM_CUDA(cudaGetLastError());
    DevCtx* c = dev_ctx(dev);
    if (!c) return SYM_ERR_CUDA;
    uint32_t st[4] = {0, 0, 0, 0};
    SYM_CUDA(cudaMemcpy(st, c->status, sizeof st, cudaMemcpyDeviceToHost));
    if (st[0] == 0) return SYM_OK;
    static const char* const kSiteNames[] = {"none", "signal wait", "counter wait", "pull tile flag",
                                             "put+signal/AlltoAll receiver", "bulk-copy stage",
                                             "put+signal batch order", "barrier"};
    const char* name = st[1] < sizeof kSiteNames / sizeof kSiteNames[0] ? kSiteNames[st[1]] : "?";
    snprintf(g_last_error, sizeof g_last_error, "device status 0x%x at site %u (%s) (%u, %u)", st[0],
             st[1], name, st[2], st[3]);
    SYM_CUDA(cudaMemset(c->status, 0, sizeof st));
    if (st[0] & kStatusTimeout) return SYM_ERR_TIMEOUT;
    return SYM_ERR_DEVICE_STATUS;
}

const char* sym_status_string(sym_status_t s) {
    switch (s) {
        case SYM_OK: return "SYM_OK";
        case SYM_ERR_INVALID_ARG: return "SYM_ERR_INVALID_ARG";
        case SYM_ERR_OOM: return "SYM_ERR_OOM";
        case SYM_ERR_CUDA: return "SYM_ERR_CUDA";
        case SYM_ERR_TIMEOUT: return "SYM_ERR_TIMEOUT";
        case SYM_ERR_UNSUPPORTED: return "SYM_ERR_UNSUPPORTED";
        case SYM_ERR_DEVICE_STATUS: return "SYM_ERR_DEVICE_STATUS";
    }
    return "SYM_ERR_UNKNOWN";
}

const char* sym_last_error(void) { return g_last_error; }

uint64_t sym_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int sym_abi_version(void) { return SYMAR_ABI_VERSION; }

}  // extern "C"
