// AllReduce for callers that cannot allocate device memory.
//
// Every other entry point of this library allocates: windows, their signal,
// counter and flag slots, and the per-device status block all come from
// cudaMalloc.  Some callers cannot do that: engines that reserve all device
// memory at start-up and forbid later allocations, plug-ins whose host
// framework owns the device allocator, and latency-critical paths that cannot
// afford the device-wide synchronisation cudaMalloc / cudaFree may do.  For them,
// sym_allreduce_noalloc takes plain device pointers to the caller's own send
// and receive buffers and uses no memory besides one fixed array compiled
// into this file (g_static_scratch below): the driver creates it when it
// loads the library's device code, and it stays on every GPU that loaded the
// library until the process exits.
//
// The kernel is the fused pull two-shot of SYM_ALGO_TWOSHOT_PULL with its
// per-tile ready flags and its status words moved into that array.  One
// change makes it safe without a status read-back: a gather that gives up
// waiting for a tile's flag reduces that tile itself, straight from the
// inputs (same rank order, same rounding), so the result is complete and
// bit-identical either way; that is why send and receive buffers must not
// overlap here.
#include <mutex>

#include "allreduce_kernels.cuh"

namespace symar {

namespace {

constexpr uint32_t kStaticFlagWords = 65536;   // ready flags: R * tiles_per_chunk at most
constexpr uint32_t kStaticStatusWords = 8;     // [0] bits [1] site [2..3] where [4] launch tag
constexpr int kStaticMaxDevices = 64;

}  // namespace

// The whole scratch of sym_allreduce_noalloc: 256 KiB of flags, then status.
// Host code must not pass this name to a kernel (on the host it is only a
// stand-in); its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint32_t g_static_scratch[kStaticFlagWords + kStaticStatusWords];

// Fallback of a gather that gave up: reduce tile t of chunk q from the
// inputs and store it into slot r.
template <class T, class Op, int RB>
__device__ __forceinline__ void static_reduce_into(const ArArgs& a, uint32_t r, uint32_t q,
                                                   uint32_t t) {
    reduce_tile_into<T, Op, RB, false>(a, q, t, r);
}

// The fused pull two-shot (see k_twoshot_pull, mode 0) on the static flags.
template <class T, class Op>
__global__ void __launch_bounds__(kThreads, 2) k_twoshot_pull_static(ArArgs a) {
    constexpr int RB = 4;
    constexpr size_t TILEV = (size_t)kThreads * kPullU;
    __shared__ int s_ok[2];
    const uint32_t R = (uint32_t)a.R, T_ = a.tiles_per_chunk;
    const uint32_t RR = R * R;
    uint32_t parity = 0;
    auto tile_nonempty = [&](uint32_t q, uint32_t t) {
        const size_t c0 = (size_t)q * a.chunk_vec;
        return c0 + (size_t)t * TILEV < min(c0 + a.chunk_vec, a.nvec);
    };
    const uint64_t total = (uint64_t)(T_ + a.lag) * RR;
    for (uint64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const uint32_t b = (uint32_t)(w / RR), s = (uint32_t)(w - (uint64_t)b * RR);
        if (s < R) {
            const uint32_t q = s, t = b;
            if (t >= T_ || !tile_nonempty(q, t)) continue;
            pull_reduce_item<T, Op, RB>(a, q, t);
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                st_release_u32(a.flags + (size_t)q * a.flag_stride + t, a.epoch);
            }
        } else {
            if (b < a.lag) continue;
            const uint32_t t = b - a.lag;
            if (t >= T_) continue;
            const uint32_t g = s - R, r = g / (R - 1), j = g - r * (R - 1);
            const uint32_t q = j < r ? j : j + 1;
            if (!tile_nonempty(q, t)) continue;
            if (threadIdx.x == 0) {
                const uint32_t* f = a.flags + (size_t)q * a.flag_stride + t;
                const uint32_t ep = a.epoch;
                bool got = bounded_spin([&] { return ld_acquire_u32(f) == ep; }, a.timeout_ns,
                                        a.giveup, a.tag);
                if (!got) report_timeout(a.status, a.giveup, a.tag, kSitePullFlag, q, t);
                s_ok[parity] = got ? 1 : 0;
            }
            __syncthreads();
            const bool go = s_ok[parity] != 0;
            parity ^= 1u;
            if (go)
                pull_copy_item(a, r, q, t);
            else
                static_reduce_into<T, Op, RB>(a, r, q, t);
        }
    }
    if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
}

namespace {

struct StaticDevice {
    bool ready = false;
    uint32_t* scratch = nullptr;     // device address of g_static_scratch
    int sms = 0;
    int occ[3][3] = {};              // blocks per SM, per (dtype, op)
    uint32_t epoch = 0;
    uint32_t tag = 0;
};
StaticDevice g_static_dev[kStaticMaxDevices];
std::mutex g_static_mu;

template <class T, class Op>
void* static_kernel() {
    return (void*)k_twoshot_pull_static<T, Op>;
}

void* pick_kernel(sym_dtype_t dt, sym_op_t op) {
    const int o = (int)op;
    if (dt == SYM_F32) return o == 0 ? static_kernel<F32T, OpSum>() : o == 1 ? static_kernel<F32T, OpMax>()
                                                                                : static_kernel<F32T, OpMin>();
    if (dt == SYM_BF16) return o == 0 ? static_kernel<BF16T, OpSum>() : o == 1 ? static_kernel<BF16T, OpMax>()
                                                                                  : static_kernel<BF16T, OpMin>();
    return o == 0 ? static_kernel<F16T, OpSum>() : o == 1 ? static_kernel<F16T, OpMax>()
                                                          : static_kernel<F16T, OpMin>();
}

}  // namespace
}  // namespace symar

using namespace symar;

extern "C" sym_status_t sym_allreduce_noalloc(const void* send, void* recv, size_t stride, int R,
                                              size_t count, sym_dtype_t dtype, sym_op_t op,
                                              sym_stream_t stream) {
    const size_t es = dtype_size(dtype);
    if (!es || (int)op < SYM_SUM || (int)op > SYM_MIN) return SYM_ERR_INVALID_ARG;
    if (!send || !recv || R < 1 || R > kMaxRanks) return SYM_ERR_INVALID_ARG;
    if (count == 0) return SYM_OK;
    const size_t nbytes = count * es;
    if (count > ((size_t)1 << 40) / es || stride < nbytes || stride % kVecBytes != 0 ||
        ((uintptr_t)send | (uintptr_t)recv) % kVecBytes != 0)
        return SYM_ERR_INVALID_ARG;
    // the fallback reads the inputs after other tiles are written: no overlap
    const uintptr_t s0 = (uintptr_t)send, s1 = s0 + (size_t)(R - 1) * stride + nbytes;
    const uintptr_t r0 = (uintptr_t)recv, r1 = r0 + (size_t)(R - 1) * stride + nbytes;
    if (s0 < r1 && r0 < s1) return SYM_ERR_INVALID_ARG;

    ArArgs a{};
    a.send = (const char*)send;
    a.recv = (char*)recv;
    a.sstride = a.rstride = stride;
    a.R = R;
    a.nvec = nbytes / kVecBytes;
    a.chunk_vec = ceil_div(a.nvec, (size_t)R);
    a.tail_elem0 = a.nvec * (kVecBytes / es);
    a.tail_n = (uint32_t)(count - a.tail_elem0);
    a.tiles_per_chunk = (uint32_t)ceil_div(a.chunk_vec, (size_t)kThreads * kPullU);
    if ((size_t)R * a.tiles_per_chunk > kStaticFlagWords) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "sym_allreduce_noalloc: %d ranks x %u tiles of 16 KiB need more than the %u ready "
                 "flags of the static scratch (about 1 GiB per rank at most)",
                 R, a.tiles_per_chunk, kStaticFlagWords);
        set_last_error(msg);
        return SYM_ERR_INVALID_ARG;
    }

    int dev = 0;
    SYM_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kStaticMaxDevices) return SYM_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    void* kernel = pick_kernel(dtype, op);
    uint32_t* scratch;
    int sms, occ;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        StaticDevice& d = g_static_dev[dev];
        if (!d.ready) {            // once per device, with that device current
            void* p = nullptr;
            SYM_CUDA(cudaGetSymbolAddress(&p, g_static_scratch));
            SYM_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
            d.scratch = (uint32_t*)p;
            d.ready = true;
        }
        int& o = d.occ[(int)dtype][(int)op];
        if (o == 0) {
            SYM_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kThreads, 0));
            if (o < 1) o = 1;
        }
        if (++d.epoch == 0) {      // flags are epoch-tagged; clear them once per 2^32 calls
            SYM_CUDA(cudaMemsetAsync(d.scratch, 0, sizeof(uint32_t) * kStaticFlagWords, st));
            d.epoch = 1;
        }
        if (++d.tag == 0) d.tag = 1;
        a.epoch = d.epoch;
        a.tag = d.tag;
        scratch = d.scratch;
        sms = d.sms;
        occ = o;
    }
    // status words start at zero for every call (diagnostics only)
    SYM_CUDA(cudaMemsetAsync(scratch + kStaticFlagWords, 0, sizeof(uint32_t) * 4, st));
    a.flags = scratch;
    a.flag_stride = a.tiles_per_chunk;
    a.status = scratch + kStaticFlagWords;
    a.giveup = scratch + kStaticFlagWords + 4;
    a.timeout_ns = default_timeout_ns();
    a.mode = 0;
    const size_t slots = (size_t)R * R * a.tiles_per_chunk;
    const size_t grid = std::min(std::max(slots, (size_t)1), (size_t)occ * sms);
    a.lag = (uint32_t)(pull_lag_waves() * ceil_div(grid, (size_t)R * R)) + 1;
    void* args[] = {&a};
    // gathers wait on reductions of the same launch -> co-residency required
    SYM_CUDA(cudaLaunchCooperativeKernel(kernel, dim3((unsigned)grid), dim3(kThreads), args, 0, st));
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}
