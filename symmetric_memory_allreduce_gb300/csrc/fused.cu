// Producer + AllReduce in one persistent launch, with per-tile counter relay.
//
// [GDA] section 5.1 (mKernel's fused GEMM + AllReduce): compute tiles bump a
// per-chunk counter with atomicAdd; the tile that completes a chunk publishes
// a flag with a release store; the reducing role spins on the flag with an
// acquire load and a short sleep, then reduces.  Here the producer is one
// binary32 multiply per element (each rank's contribution
// s_r = alpha_r * a_r, written to the send window as a GEMM epilogue would),
// and the consumer is the two-shot AllReduce by loads + stores over the
// contributions.  A tile of the result is reduced as soon as the R producer
// tiles it needs are in place, while other tiles are still being produced.
#include "allreduce_kernels.cuh"

namespace symar {

struct FusedArgs {
    const char* in;
    char* send;
    char* recv;
    size_t istride, sstride, rstride;
    int R;
    size_t nvec, chunk_vec;
    uint32_t tiles_per_chunk;
    size_t tail_elem0;
    uint32_t tail_n;
    uint32_t* flags;
    uint32_t* arrivals;
    size_t flag_stride;
    const uint32_t* epoch;   // device epoch word of the recv window
    uint32_t lag;
    uint32_t* status;
    uint32_t* giveup;        // the recv window's give-up word
    unsigned long long* ticket;   // the recv window's item ticket, zeroed before the launch
    uint64_t timeout_ns;
    float alpha[kMaxRanks];
};

// The relay tile: 64 KiB of a chunk (16 vectors per thread in flight for a
// producer item); the window's flag slots, sized for 16 KiB tiles, suffice.
constexpr int kFusedU = 16;
constexpr size_t kFusedTileV = (size_t)kThreads * kFusedU;

// slot sequence in blocks of R*R + R: block b holds the producer items (r, q)
// of tile b and the consumer items q of tile b - lag.
__global__ void __launch_bounds__(kThreads, 2) k_scale_allreduce(FusedArgs a) {
    constexpr int U = kFusedU;
    constexpr size_t TILEV = kFusedTileV;
    __shared__ int s_ok[2];
    const uint32_t ep = read_epoch(a.epoch);
    const uint32_t R = (uint32_t)a.R, T_ = a.tiles_per_chunk;
    const uint32_t per_block = R * R + R;
    uint32_t parity = 0;
    const uint64_t total = (uint64_t)(T_ + a.lag) * per_block;
    __shared__ unsigned long long s_item[2];
    int ipar = 0;
    for (;;) {
        const uint64_t w = fetch_item(a.ticket, s_item, ipar);
        if (w >= total) break;
        const uint32_t b = (uint32_t)(w / per_block), s = (uint32_t)(w - (uint64_t)b * per_block);
        const bool producer = s < R * R;
        const uint32_t t = producer ? b : b - a.lag;
        if (!producer && b < a.lag) continue;
        if (t >= T_) continue;
        const uint32_t q = producer ? s % R : s - R * R;
        const size_t c0 = (size_t)q * a.chunk_vec;
        const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
        const size_t v0 = c0 + (size_t)t * TILEV;
        if (v0 >= c1) continue;
        const size_t base = v0 + threadIdx.x;          // this thread's k-th vector: base + k*kThreads
        if (producer) {
            const uint32_t r = s / R;
            const float al = a.alpha[r];
            const uint4* src = reinterpret_cast<const uint4*>(a.in + (size_t)r * a.istride);
            uint4* dst = reinterpret_cast<uint4*>(a.send + (size_t)r * a.sstride);
            uint4 v[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const size_t i = base + (size_t)k * kThreads;
                if (i < c1) v[k] = __ldcs(src + i);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const size_t i = base + (size_t)k * kThreads;
                if (i >= c1) continue;
                float f[4];
                F32T::widen(v[k], f);
#pragma unroll
                for (int e = 0; e < 4; ++e) f[e] = __fmul_rn(al, f[e]);
                __stcg(dst + i, F32T::narrow(f));
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                uint32_t* cnt = a.arrivals + (size_t)q * a.flag_stride + t;
                if (atomicAdd(cnt, 1u) == R - 1) {          // the last of the R producers
                    *cnt = 0;
                    __threadfence();
                    st_release_u32(a.flags + (size_t)q * a.flag_stride + t, ep);
                }
            }
        } else {
            if (threadIdx.x == 0) {
                const uint32_t* f = a.flags + (size_t)q * a.flag_stride + t;
                bool got = bounded_spin([&] { return ld_acquire_u32(f) == ep; }, a.timeout_ns,
                                        a.giveup, ep);
                if (!got) report_timeout(a.status, a.giveup, ep, kSitePullFlag, q, t);
                s_ok[parity] = got ? 1 : 0;
            }
            __syncthreads();
            const bool go = s_ok[parity] != 0;
            parity ^= 1u;
            if (!go) continue;
            // sub-steps of two vectors per thread, ranks folded four at a time
#pragma unroll 1
            for (int h = 0; h < U / 2; ++h) {
                const size_t hidx[2] = {base + (size_t)(2 * h) * kThreads,
                                        base + (size_t)(2 * h + 1) * kThreads};
                const bool hok[2] = {hidx[0] < c1, hidx[1] < c1};
                float acc[2][4];
                // last use of the contributions: streaming loads let their
                // lines go first, ahead of contributions still to be reduced
                reduce_vectors<F32T, OpSum, 4, 2, kLoadStream>(a.send, a.sstride, a.R, hidx, hok, acc);
                const uint4 o0 = F32T::narrow(acc[0]), o1 = F32T::narrow(acc[1]);
                for (int r = 0; r < a.R; ++r) {
                    char* dst = a.recv + (size_t)r * a.rstride;
                    if (hok[0]) store16_stream(dst + hidx[0] * kVecBytes, o0);
                    if (hok[1]) store16_stream(dst + hidx[1] * kVecBytes, o1);
                }
            }
        }
    }
    // ragged tail: this block produces and reduces it alone
    if (a.tail_n && blockIdx.x == gridDim.x - 1 && threadIdx.x < a.tail_n) {
        const size_t off = (a.tail_elem0 + threadIdx.x) * 4;
        float acc = 0.f;
        for (int r = 0; r < a.R; ++r) {
            const float v = __fmul_rn(a.alpha[r], *reinterpret_cast<const float*>(a.in + (size_t)r * a.istride + off));
            *reinterpret_cast<float*>(a.send + (size_t)r * a.sstride + off) = v;
            acc = r == 0 ? v : __fadd_rn(acc, v);
        }
        for (int r = 0; r < a.R; ++r) *reinterpret_cast<float*>(a.recv + (size_t)r * a.rstride + off) = acc;
    }
}

}  // namespace symar

using namespace symar;

extern "C" sym_status_t sym_scale_allreduce(sym_win_t in, sym_win_t send, sym_win_t recv,
                                            const float* alpha, size_t count, sym_stream_t stream) {
    if (!in || !send || !recv || !alpha) return SYM_ERR_INVALID_ARG;
    if (in->R != send->R || send->R != recv->R) return SYM_ERR_INVALID_ARG;
    if (in->device != send->device || send->device != recv->device) return SYM_ERR_INVALID_ARG;
    if (in->base == send->base || send->base == recv->base || in->base == recv->base)
        return SYM_ERR_INVALID_ARG;
    if (count > in->bytes / 4 || count > send->bytes / 4 || count > recv->bytes / 4)
        return SYM_ERR_INVALID_ARG;
    if (count == 0) return SYM_OK;
    const size_t nbytes = count * 4;
    if (windows_overlap(in, nbytes, send, nbytes) || windows_overlap(send, nbytes, recv, nbytes) ||
        windows_overlap(in, nbytes, recv, nbytes)) {
        set_last_error("sym_scale_allreduce: two of the three windows share memory");
        return SYM_ERR_INVALID_ARG;
    }
    if (nbytes / kVecBytes > ((size_t)1 << 34)) return SYM_ERR_UNSUPPORTED;
    FusedArgs a{};
    a.in = in->base;
    a.send = send->base;
    a.recv = recv->base;
    a.istride = in->stride;
    a.sstride = send->stride;
    a.rstride = recv->stride;
    a.R = recv->R;
    a.nvec = nbytes / kVecBytes;
    a.chunk_vec = ceil_div(a.nvec, (size_t)a.R);
    a.tail_elem0 = a.nvec * 4;
    a.tail_n = (uint32_t)(count - a.tail_elem0);
    a.tiles_per_chunk = (uint32_t)ceil_div(a.chunk_vec, kFusedTileV);
    if (a.tiles_per_chunk > recv->flag_tiles) return SYM_ERR_INVALID_ARG;
    for (int r = 0; r < a.R; ++r) a.alpha[r] = alpha[r];
    DeviceGuard g(recv->device);
    if (!g.ok) return SYM_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    {
        sym_status_t s = bump_epoch(recv->epoch, st, recv->ticket);
        if (s != SYM_OK) return s;
    }
    a.epoch = recv->epoch;
    a.ticket = recv->ticket;
    a.flags = recv->flags;
    a.arrivals = recv->arrivals;
    a.flag_stride = recv->flag_tiles;
    a.status = recv->ctx->status;
    a.giveup = recv->giveup;
    a.timeout_ns = default_timeout_ns();
    const int occ = occupancy((const void*)k_scale_allreduce, kThreads, 0);
    const size_t cap = (size_t)occ * recv->ctx->num_sms;
    const size_t per_block = (size_t)a.R * a.R + a.R;
    const size_t slots = per_block * a.tiles_per_chunk;
    const size_t grid = std::min(std::max(slots, (size_t)1), cap);
    // consumers trail producers by about one grid wave of items (the whole
    // tile blocks that fit in it): long enough that a consumer seldom waits
    // for producers still in flight, short enough that the contributions it
    // reads back are still in L2.  Items are handed out in index order by
    // the window's ticket, so a consumer only waits for producer items that
    // running blocks already hold.  On GB300 (R = 8: 304 blocks, 72 items a
    // tile block) 3-4 blocks measured fastest; 8 was 5 % slower.
    const int64_t lb = fused_lag_blocks();
    a.lag = lb >= 0 ? (uint32_t)lb : (uint32_t)std::max<size_t>(1, grid / per_block);
    void* args[] = {&a};
    // consumers wait on producers of the same launch -> co-residency required
    SYM_CUDA(cudaLaunchCooperativeKernel((const void*)k_scale_allreduce, dim3((unsigned)grid),
                                         dim3(kThreads), args, 0, st));
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}
