// AllReduce kernels over R rank windows carved from one GPU's HBM, templated on
// the element type and the reduction operator.  Included once per element
// type by allreduce_{f32,bf16,f16}.cu; the C ABI entry lives in allreduce.cu.
//
// What is computed ([SYMEX] "NCCL symmetric memory windows", Example 1: every
// rank calls AllReduce(send, recv, count, float, sum) and every element of
// every recv buffer is the sum over ranks):
//     recv_r[i] = op(...op(op(send_0[i], send_1[i]), send_2[i])..., send_{R-1}[i])
// for every rank r -- a left fold in rank order 0..R-1 in fp32 (IEEE
// round-to-nearest adds, no contraction, no flush-to-zero), so fp32 results
// are bit-identical on every rank and to a plain sequential sum.  bf16 and
// fp16 are widened exactly, folded in fp32 and rounded to nearest-even once.
// max / min are IEEE 754-2019 maximumNumber / minimumNumber (a NaN operand is
// ignored; -0 < +0).
//
// Data movements, all hand-written with 16-byte vector accesses:
//  * one-shot   -- every rank-slot r reads all R windows at a tile and writes
//                  only recv_r ([LSA]: a peer's buffer is read directly with
//                  loads at base + offset).  Work items are ordered tile-major,
//                  slot-minor, so the R slots of a tile run side by side and
//                  their repeated reads of the same lines are served by L2.
//  * two-shot   -- rank-slot q owns chunk q (1/R of the elements, 16-byte
//                  aligned).  Reduce-scatter: slot q loads chunk q from all R
//                  windows and reduces it.  All-gather: slot q stores the
//                  reduced chunk into every window (the store form of the
//                  all-gather), so nothing is read back.  HBM traffic is the
//                  floor for the emulation: every input read once, every
//                  output written once.  Two movers: registers (LDG/STG) or
//                  the TMA engine (bulk copies staged in shared memory).
//  * two-shot pull -- the same reduce-scatter, but the reduced chunk is only
//                  written to recv_q; slot q then publishes one flag per tile
//                  (st.release.gpu = epoch) and every other slot r waits for
//                  the flag (ld.acquire.gpu, bounded) and copies the tile from
//                  recv_q into recv_r.  This is the per-chunk completion flag
//                  plus acquire spin of [GDA] section 5.1, with the give-up
//                  timeout of [GIN]'s barrier.  A split form runs the two
//                  phases as two launches (the kernel boundary is the barrier).
#pragma once

#include <cuda_fp16.h>

#include <algorithm>
#include <cstdio>
#include <type_traits>

#include "symar_internal.cuh"

namespace symar {

constexpr int kThreads = 256;
constexpr int kPullU = 4;                                    // 16 KiB tiles
static_assert(kThreads * kPullU * kVecBytes == (int)kPullTileBytes,
              "pull tile must match the window's flag tile");

// ----------------------------------------------------------------- element traits

struct F32T {
    static constexpr int V = 4;       // elements per 16 bytes
    __device__ __forceinline__ static void widen(const uint4& x, float (&f)[4]) {
        f[0] = __uint_as_float(x.x);
        f[1] = __uint_as_float(x.y);
        f[2] = __uint_as_float(x.z);
        f[3] = __uint_as_float(x.w);
    }
    __device__ __forceinline__ static uint4 narrow(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float load1(const char* p) {
        return *reinterpret_cast<const float*>(p);
    }
    __device__ __forceinline__ static void store1(char* p, float v) {
        *reinterpret_cast<float*>(p) = v;
    }
};

// 16-bit types: element 2k is the low half of word k (little endian)
struct BF16T {
    static constexpr int V = 8;
    __device__ __forceinline__ static float up(uint32_t h) { return __uint_as_float(h << 16); }
    __device__ __forceinline__ static void widen(const uint4& x, float (&f)[8]) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 narrow(const float (&f)[8]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const char* p) {
        return up(*reinterpret_cast<const uint16_t*>(p));
    }
    __device__ __forceinline__ static void store1(char* p, float v) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        *reinterpret_cast<uint16_t*>(p) = *reinterpret_cast<uint16_t*>(&h);
    }
};

struct F16T {
    static constexpr int V = 8;
    __device__ __forceinline__ static float up(uint32_t h) {
        return __half2float(__ushort_as_half((unsigned short)h));
    }
    __device__ __forceinline__ static void widen(const uint4& x, float (&f)[8]) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = up(w[k] & 0xFFFFu);
            f[2 * k + 1] = up(w[k] >> 16);
        }
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 narrow(const float (&f)[8]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const char* p) {
        return up(*reinterpret_cast<const uint16_t*>(p));
    }
    __device__ __forceinline__ static void store1(char* p, float v) {
        *reinterpret_cast<unsigned short*>(p) = __half_as_ushort(__float2half_rn(v));
    }
};

// ----------------------------------------------------------------- reduction operators

struct OpSum {
    __device__ __forceinline__ static float apply(float a, float b) { return __fadd_rn(a, b); }
};

// maximumNumber: NaN operands ignored, -0 < +0
struct OpMax {
    __device__ __forceinline__ static float apply(float a, float b) {
        if (a != a) return b;
        if (b != b) return a;
        if (a > b) return a;
        if (b > a) return b;
        return (__float_as_uint(a) >> 31) ? b : a;
    }
};

// minimumNumber: NaN operands ignored, -0 < +0
struct OpMin {
    __device__ __forceinline__ static float apply(float a, float b) {
        if (a != a) return b;
        if (b != b) return a;
        if (a < b) return a;
        if (b < a) return b;
        return (__float_as_uint(a) >> 31) ? a : b;
    }
};

// ----------------------------------------------------------------- memory access flavours

enum LoadKind { kLoadStream = 0, kLoadKeep = 1 };

template <int K>
__device__ __forceinline__ uint4 load16(const char* p) {
    if (K == kLoadStream) return __ldcs(reinterpret_cast<const uint4*>(p));   // read once
    return __ldcg(reinterpret_cast<const uint4*>(p));                        // L2, reused
}

__device__ __forceinline__ void store16_stream(char* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ void store16_keep(char* p, uint4 v) {
    __stcg(reinterpret_cast<uint4*>(p), v);
}

// L2 eviction-priority policies (createpolicy) and the accesses that carry them
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void store16_hint(char* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// ----------------------------------------------------------------- kernel arguments

struct ArArgs {
    const char* send;
    char* recv;
    size_t sstride, rstride;
    int R;
    size_t nvec;             // whole 16-byte vectors per rank
    size_t chunk_vec;        // vectors per rank-slot chunk (two-shot)
    uint32_t tiles_per_chunk;
    uint32_t ntile;          // one-shot: tiles over nvec
    size_t tail_elem0;       // first element past the last whole vector
    uint32_t tail_n;         // elements in the ragged tail (< V)
    // pull two-shot
    uint32_t* flags;
    size_t flag_stride;
    uint32_t epoch;          // flag epoch given by the host (static-scratch variant)
    const uint32_t* epoch_ptr;   // device epoch word of the window (window variants)
    uint32_t lag;            // item blocks between a reduce and its gathers
    uint32_t group;          // fused pull: 16 KiB tiles per work item (flags stay per tile)
    int mode;                // 0 fused, 1 reduce-scatter only, 2 all-gather only
    uint32_t* status;
    uint32_t* giveup;        // give-up word of the waits (see report_timeout)
    unsigned long long* ticket;  // work tickets of the warp-specialised pull (zeroed per launch)
    uint32_t tag;            // this launch's give-up tag (static-scratch variant)
    uint64_t timeout_ns;
};

// Fold of R 16-byte vectors (rank order) at vector indices idx[k] of every
// window; loads are issued RB ranks at a time before any arithmetic, for
// memory-level parallelism.
template <class T, class Op, int RB, int U, int LK>
__device__ __forceinline__ void reduce_vectors(const char* send, size_t sstride, int R,
                                               const size_t (&idx)[U], const bool (&ok)[U],
                                               float (&acc)[U][T::V]) {
    for (int r0 = 0; r0 < R; r0 += RB) {
        uint4 buf[RB][U];
#pragma unroll
        for (int j = 0; j < RB; ++j) {
#pragma unroll
            for (int k = 0; k < U; ++k) {
                buf[j][k] = make_uint4(0, 0, 0, 0);
                if (r0 + j < R && ok[k])
                    buf[j][k] = load16<LK>(send + (size_t)(r0 + j) * sstride + idx[k] * kVecBytes);
            }
        }
#pragma unroll
        for (int j = 0; j < RB; ++j) {
            if (r0 + j < R) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    float f[T::V];
                    T::widen(buf[j][k], f);
                    if (r0 + j == 0) {
#pragma unroll
                        for (int e = 0; e < T::V; ++e) acc[k][e] = f[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < T::V; ++e) acc[k][e] = Op::apply(acc[k][e], f[e]);
                    }
                }
            }
        }
    }
}

// Ragged tail (fewer than V elements past the last whole vector): element
// e of the tail is folded by thread e and written to slots [slot_lo, slot_hi).
template <class T, class Op>
__device__ __forceinline__ void reduce_tail(const ArArgs& a, int slot_lo, int slot_hi) {
    const int e = threadIdx.x;
    if ((uint32_t)e >= a.tail_n) return;
    constexpr size_t es = 16 / T::V;
    const size_t off = (a.tail_elem0 + e) * es;
    float acc = T::load1(a.send + off);
    for (int r = 1; r < a.R; ++r) acc = Op::apply(acc, T::load1(a.send + (size_t)r * a.sstride + off));
    for (int r = slot_lo; r < slot_hi; ++r) T::store1(a.recv + (size_t)r * a.rstride + off, acc);
}

// ----------------------------------------------------------------- two-shot (store all-gather)

template <class T, class Op, int RB, int U>
__global__ void __launch_bounds__(kThreads) k_twoshot_st(ArArgs a) {
    constexpr size_t TILEV = (size_t)kThreads * U;
    const uint32_t items = (uint32_t)a.R * a.tiles_per_chunk;
    for (uint32_t w = blockIdx.x; w < items; w += gridDim.x) {
        const uint32_t q = w / a.tiles_per_chunk, t = w - q * a.tiles_per_chunk;
        const size_t c0 = (size_t)q * a.chunk_vec;
        const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
        const size_t v0 = c0 + (size_t)t * TILEV;
        if (v0 >= c1) continue;
        size_t idx[U];
        bool ok[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            idx[k] = v0 + threadIdx.x + (size_t)k * kThreads;
            ok[k] = idx[k] < c1;
        }
        float acc[U][T::V];
        reduce_vectors<T, Op, RB, U, kLoadStream>(a.send, a.sstride, a.R, idx, ok, acc);
        uint4 out[U];
#pragma unroll
        for (int k = 0; k < U; ++k) out[k] = T::narrow(acc[k]);
        // all-gather by stores: slot q writes its reduced chunk into every window
        for (int r = 0; r < a.R; ++r) {
            char* dst = a.recv + (size_t)r * a.rstride;
#pragma unroll
            for (int k = 0; k < U; ++k)
                if (ok[k]) store16_stream(dst + idx[k] * kVecBytes, out[k]);
        }
    }
    if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
}

// ----------------------------------------------------------------- two-shot, bulk-copy staging
//
// The same work items, moved by the TMA engine: one thread issues R bulk
// loads of a tile (one per window) into a shared-memory stage, completing on
// an mbarrier; all threads reduce the stage into an output tile; the same
// thread then issues R bulk stores of the output tile, one per window.  Two
// input stages and two output tiles: the loads of item i+2 and the stores of
// item i overlap the reduction of item i+1.

constexpr int kBulkStages = 2;
constexpr uint32_t kBulkInBytes = 64 * 1024;      // R tiles of one stage

__host__ __device__ constexpr uint32_t bulk_tile_bytes(int R) {
    // R tiles fit one 64 KiB stage; at most 8 KiB per tile
    return R <= 8 ? 8192u : (kBulkInBytes / (uint32_t)R) / 16u * 16u;
}

__host__ constexpr size_t bulk_smem_bytes(int R) {
    return (size_t)kBulkStages * kBulkInBytes + (size_t)kBulkStages * bulk_tile_bytes(R) + 64;
}

template <class T, class Op>
__global__ void __launch_bounds__(kThreads, 1) k_twoshot_bulk(ArArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = a.R;
    const uint32_t tile = bulk_tile_bytes(R);
    const uint32_t tilev = tile / kVecBytes;
    unsigned char* in = smem;                                        // [stage][R][tile]
    unsigned char* out = smem + kBulkStages * kBulkInBytes;          // [stage][tile]
    uint64_t* full = reinterpret_cast<uint64_t*>(out + kBulkStages * tile);
    const uint32_t items = (uint32_t)R * a.tiles_per_chunk;
    const uint32_t nmine = blockIdx.x < items ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    // item -> [v0, v1) vector range of chunk q (empty when past the data)
    auto range = [&](uint32_t i, size_t& v0, size_t& v1) {
        const uint32_t w = blockIdx.x + i * gridDim.x;
        const uint32_t q = w / a.tiles_per_chunk, t = w - q * a.tiles_per_chunk;
        const size_t c0 = (size_t)q * a.chunk_vec;
        const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
        v0 = c0 + (size_t)t * tilev;
        v1 = min(v0 + tilev, c1);
        if (v0 > v1) v1 = v0;
    };
    auto issue_loads = [&](uint32_t i, int s) {
        size_t v0, v1;
        range(i, v0, v1);
        const uint32_t bytes = (uint32_t)((v1 - v0) * kVecBytes);
        mbar_expect_tx(&full[s], bytes * (uint32_t)R);
        if (bytes == 0) return;
        for (int r = 0; r < R; ++r)
            bulk_load(in + ((size_t)s * R + r) * tile, a.send + (size_t)r * a.sstride + v0 * kVecBytes,
                      bytes, &full[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        for (uint32_t i = 0; i < (uint32_t)kBulkStages && i < nmine; ++i) issue_loads(i, (int)i);
    }
    __syncthreads();

    for (uint32_t i = 0; i < nmine; ++i) {
        const int s = (int)(i % kBulkStages);
        const uint32_t parity = (i / kBulkStages) & 1u;
        size_t v0, v1;
        range(i, v0, v1);
        const uint32_t nv = (uint32_t)(v1 - v0);
        // wait for the stage (bounded; the loads cannot fail on valid ranges)
        bool ok = true;
        for (uint32_t spins = 0; !mbar_try_wait(&full[s], parity); ++spins) {
            if (spins > (1u << 26)) {
                ok = false;
                break;
            }
        }
        if (!__syncthreads_and(ok)) {               // uniform: every thread leaves together
            if (threadIdx.x == 0) report_timeout(a.status, nullptr, 0, kSiteBulkStage, blockIdx.x, i);
            break;
        }
        const unsigned char* st = in + (size_t)s * R * tile;
        unsigned char* ot = out + (size_t)s * tile;
        for (uint32_t v = threadIdx.x; v < nv; v += kThreads) {
            float acc[T::V];
            for (int r = 0; r < R; ++r) {
                const uint4 x = *reinterpret_cast<const uint4*>(st + (size_t)r * tile + v * kVecBytes);
                float f[T::V];
                T::widen(x, f);
                if (r == 0) {
#pragma unroll
                    for (int e = 0; e < T::V; ++e) acc[e] = f[e];
                } else {
#pragma unroll
                    for (int e = 0; e < T::V; ++e) acc[e] = Op::apply(acc[e], f[e]);
                }
            }
            *reinterpret_cast<uint4*>(ot + v * kVecBytes) = T::narrow(acc);
        }
        fence_proxy_async_smem();          // generic-proxy writes -> visible to the bulk stores
        if (threadIdx.x == 0) bulk_wait_read<0>();   // previous item's stores have read their tile
        __syncthreads();
        if (threadIdx.x == 0) {
            if (nv) {
                for (int r = 0; r < R; ++r)
                    bulk_store(a.recv + (size_t)r * a.rstride + v0 * kVecBytes, ot, nv * kVecBytes);
            }
            bulk_commit();
            if (i + kBulkStages < nmine) issue_loads(i + kBulkStages, s);   // stage s is free
        }
    }
    if (threadIdx.x == 0) bulk_wait_all<0>();
    if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
}

// ----------------------------------------------------------------- one-shot

template <class T, class Op, int RB, int U>
__global__ void __launch_bounds__(kThreads) k_oneshot(ArArgs a) {
    constexpr size_t TILEV = (size_t)kThreads * U;
    const uint32_t items = (uint32_t)a.R * a.ntile;
    for (uint32_t w = blockIdx.x; w < items; w += gridDim.x) {
        const uint32_t t = w / (uint32_t)a.R, r = w - t * (uint32_t)a.R;   // slot-minor
        const size_t v0 = (size_t)t * TILEV;
        size_t idx[U];
        bool ok[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            idx[k] = v0 + threadIdx.x + (size_t)k * kThreads;
            ok[k] = idx[k] < a.nvec;
        }
        float acc[U][T::V];
        reduce_vectors<T, Op, RB, U, kLoadKeep>(a.send, a.sstride, a.R, idx, ok, acc);
        char* dst = a.recv + (size_t)r * a.rstride;
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (ok[k]) store16_stream(dst + idx[k] * kVecBytes, T::narrow(acc[k]));
    }
    if (a.tail_n && blockIdx.x == gridDim.x - 1) {
        for (int r = 0; r < a.R; ++r) reduce_tail<T, Op>(a, r, r + 1);   // each slot its own
    }
}

// ----------------------------------------------------------------- two-shot (pull all-gather)

// Reduce tile t of chunk q over all windows and store it into slot `dst_slot`
// (`keep`: leave it in L2 for the gathers that read it next).  The 16 KiB tile
// is done in kPullU / 2 sub-steps of two vectors per thread, so that the
// registers of RB-rank batches stay low enough for three CTAs per SM.
template <class T, class Op, int RB, bool keep>
__device__ __forceinline__ void reduce_tile_into(const ArArgs& a, uint32_t q, uint32_t t,
                                                 uint32_t dst_slot) {
    constexpr int U = 2;
    constexpr size_t TILEV = (size_t)kThreads * kPullU;
    const size_t c0 = (size_t)q * a.chunk_vec;
    const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
    const size_t v0 = c0 + (size_t)t * TILEV;
    char* dst = a.recv + (size_t)dst_slot * a.rstride;
#pragma unroll 1
    for (int h = 0; h < kPullU / U; ++h) {
        size_t idx[U];
        bool ok[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            idx[k] = v0 + threadIdx.x + (size_t)(h * U + k) * kThreads;
            ok[k] = idx[k] < c1;
        }
        float acc[U][T::V];
        reduce_vectors<T, Op, RB, U, keep ? kLoadStream : kLoadKeep>(a.send, a.sstride, a.R, idx,
                                                                       ok, acc);
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (!ok[k]) continue;
            if (keep)
                store16_keep(dst + idx[k] * kVecBytes, T::narrow(acc[k]));
            else
                store16_stream(dst + idx[k] * kVecBytes, T::narrow(acc[k]));
        }
    }
}

template <class T, class Op, int RB>
__device__ __forceinline__ void pull_reduce_item(const ArArgs& a, uint32_t q, uint32_t t) {
    reduce_tile_into<T, Op, RB, true>(a, q, t, q);
}

__device__ __forceinline__ void pull_copy_item(const ArArgs& a, uint32_t r, uint32_t q, uint32_t t) {
    constexpr int U = kPullU;
    constexpr size_t TILEV = (size_t)kThreads * U;
    const size_t c0 = (size_t)q * a.chunk_vec;
    const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
    const size_t v0 = c0 + (size_t)t * TILEV;
    const char* src = a.recv + (size_t)q * a.rstride;
    char* dst = a.recv + (size_t)r * a.rstride;
    uint4 v[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const size_t i = v0 + threadIdx.x + (size_t)k * kThreads;
        if (i < c1) v[k] = __ldcg(reinterpret_cast<const uint4*>(src + i * kVecBytes));
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const size_t i = v0 + threadIdx.x + (size_t)k * kThreads;
        if (i < c1) store16_stream(dst + i * kVecBytes, v[k]);
    }
}

// resident CTAs per SM the pull kernels are compiled for (register budget):
// three, except two for max/min on the 16-bit types, whose widened tiles and
// compare chains would otherwise spill
template <class T, class Op>
constexpr int pull_blocks_per_sm() {
    return (T::V == 8 && !std::is_same<Op, OpSum>::value) ? 2 : 3;
}
constexpr int kPullBlocksPerSm = 3;
constexpr uint32_t kPullGroup = 2;         // fused pull: 16 KiB tiles per work item

template <class T, class Op, int RB>
__global__ void __launch_bounds__(kThreads, pull_blocks_per_sm<T, Op>()) k_twoshot_pull(ArArgs a) {
    constexpr size_t TILEV = (size_t)kThreads * kPullU;
    const uint32_t R = (uint32_t)a.R, T_ = a.tiles_per_chunk;
    const uint32_t RR = R * R;
    auto tile_nonempty = [&](uint32_t q, uint32_t t) {
        const size_t c0 = (size_t)q * a.chunk_vec;
        return c0 + (size_t)t * TILEV < min(c0 + a.chunk_vec, a.nvec);
    };
    if (a.mode == 1) {                                   // reduce-scatter launch
        for (uint32_t w = blockIdx.x; w < R * T_; w += gridDim.x) {
            const uint32_t q = w / T_, t = w - q * T_;
            if (tile_nonempty(q, t)) pull_reduce_item<T, Op, RB>(a, q, t);
        }
        if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
        return;
    }
    if (a.mode == 2) {                                   // all-gather launch
        const uint32_t items = (R - 1) * R * T_;
        for (uint32_t w = blockIdx.x; w < items; w += gridDim.x) {
            const uint32_t qt = w / (R - 1), j = w - qt * (R - 1);
            const uint32_t q = qt / T_, t = qt - q * T_;
            const uint32_t r = j < q ? j : j + 1;
            if (tile_nonempty(q, t)) pull_copy_item(a, r, q, t);
        }
        return;
    }
    // fused: slot sequence in blocks of R*R; block b holds the reduce items of
    // tile group b and the gather items of tile group b - lag.  A group is
    // `group` consecutive 16 KiB tiles of a chunk, each with its own flag: the
    // reducer releases the group's flags together (one thread per flag), and
    // a gatherer acquires them together, so one flag round trip covers the
    // whole group.
    // static stride: an ordered ticket (as in the fused producer) measured
    // 4 % slower here, the gathers waiting on reductions still in flight
    const uint32_t ep = read_epoch(a.epoch_ptr);
    const uint32_t G = a.group, TG = (T_ + G - 1) / G;
    const uint64_t total = (uint64_t)(TG + a.lag) * RR;
    for (uint64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const uint32_t b = (uint32_t)(w / RR), s = (uint32_t)(w - (uint64_t)b * RR);
        if (s < R) {
            const uint32_t q = s, g = b;
            if (g >= TG) continue;
            for (uint32_t j = 0; j < G; ++j) {
                const uint32_t t = g * G + j;
                if (t < T_ && tile_nonempty(q, t)) pull_reduce_item<T, Op, RB>(a, q, t);
            }
            __syncthreads();
            if (threadIdx.x < G) {
                const uint32_t t = g * G + threadIdx.x;
                if (t < T_ && tile_nonempty(q, t)) {
                    __threadfence();
                    st_release_u32(a.flags + (size_t)q * a.flag_stride + t, ep);
                }
            }
        } else {
            if (b < a.lag) continue;
            const uint32_t g = b - a.lag;
            if (g >= TG) continue;
            const uint32_t gi = s - R, r = gi / (R - 1), j = gi - r * (R - 1);
            const uint32_t q = j < r ? j : j + 1;
            bool got = true;
            if (threadIdx.x < G) {
                const uint32_t t = g * G + threadIdx.x;
                if (t < T_ && tile_nonempty(q, t)) {
                    const uint32_t* f = a.flags + (size_t)q * a.flag_stride + t;
                    got = bounded_spin([&] { return ld_acquire_u32(f) == ep; }, a.timeout_ns,
                                       a.giveup, ep);
                    if (!got) report_timeout(a.status, a.giveup, ep, kSitePullFlag, q, t);
                }
            }
            if (!__syncthreads_and(got)) continue;
            for (uint32_t jj = 0; jj < G; ++jj) {
                const uint32_t t = g * G + jj;
                if (t < T_ && tile_nonempty(q, t)) pull_copy_item(a, r, q, t);
            }
        }
    }
    if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
}

// ----------------------------------------------------------------- two-shot pull, warp-specialised
//
// The same reduce-scatter / flag / pull all-gather, with the two phases run by
// different warps of every CTA so that a wait for a flag never holds up a
// reduction:
//  * 8 reducer warps take reduce items (chunk q, 16 KiB tile t), tile-major,
//    from the low half of the recv window's 64-bit ticket; they fold the R
//    windows into recv_q (left in L2), meet on a named barrier, and one thread
//    releases the tile's flag (st.release.gpu = epoch);
//  * one copy warp, driven by its first lane, takes tiles in the same order
//    from the ticket's high half, acquires each tile's flag (ld.acquire.gpu,
//    bounded) and performs the pulls recv_r[tile] = recv_q[tile] for every
//    reader r != q with the TMA engine: a bulk load into a shared-memory stage,
//    a bulk store out of it, kWsLoads loads in flight.
// Both halves of the ticket hand out work in index order, so the work in
// flight is a compact range of the windows and no CTA idles while another
// still holds a long queue.  Reducers never wait, so every flag is released as
// long as all CTAs are resident (cooperative launch); copy lanes wait only on
// flags of tiles some reducer has taken or will take.

constexpr int kWsReducers = 256;                 // 8 reducer warps (threads 0..255)
constexpr int kWsThreads = kWsReducers + 32;     // + the copy warp
// The copy lane's ring: 16 KiB shared-memory stages, kWsLoads bulk loads kept in flight.
// Measured at R = 8 x 256 MiB fp32: 3 stages / 2 loads read 12 % more DRAM than the
// compulsory bytes (the pulls fell behind the reductions and missed L2) and reached 0.86 of
// the copy bandwidth; 4 stages / 3 loads 0.95 (6 / 4 the same, at fewer CTAs per SM).
constexpr int kWsStages = 4;
constexpr int kWsLoads = kWsStages - 1;

__host__ constexpr size_t ws_smem_bytes() {
    return (size_t)kWsStages * kPullTileBytes + (size_t)kWsStages * sizeof(uint64_t);
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Generic-proxy writes made visible by an acquire -> later bulk (async-proxy) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Reduce 16 KiB tile t of chunk q into recv_q, one vector per thread and rank at a time
// (RB ranks' loads in flight), four steps of kWsReducers vectors.
template <class T, class Op, int RB>
__device__ __forceinline__ void ws_reduce_tile(const ArArgs& a, uint32_t q, uint32_t t) {
    constexpr size_t TILEV = (size_t)kWsReducers * kPullU;
    const size_t c0 = (size_t)q * a.chunk_vec;
    const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
    const size_t v0 = c0 + (size_t)t * TILEV;
    char* dst = a.recv + (size_t)q * a.rstride;
#pragma unroll 1
    for (int h = 0; h < kPullU; ++h) {
        size_t idx[1] = {v0 + threadIdx.x + (size_t)h * kWsReducers};
        bool ok[1] = {idx[0] < c1};
        if (!__any_sync(0xffffffffu, ok[0])) break;        // the rest of the tile is past the chunk
        float acc[1][T::V];
        reduce_vectors<T, Op, RB, 1, kLoadStream>(a.send, a.sstride, a.R, idx, ok, acc);
        // evict-last: the tile stays in L2 until its pulls have read it (the last reader's
        // load demotes it); without the hint 4 % of the pulls missed L2 at R = 8 x 256 MiB
        if (ok[0]) store16_hint(dst + idx[0] * kVecBytes, T::narrow(acc[0]), l2_policy_evict_last());
    }
}

// resident CTAs per SM: the copy lane's 64 KiB ring allows three, so the
// register budget is set for three (no spills for any element type)
constexpr int kWsBlocksPerSm = 3;

template <class T, class Op, int RB>
__global__ void __launch_bounds__(kWsThreads, kWsBlocksPerSm) k_twoshot_pull_ws(ArArgs a) {
    extern __shared__ __align__(128) unsigned char ws_smem[];
    __shared__ uint32_t s_item[2];
    constexpr size_t TILEV = (size_t)kWsReducers * kPullU;
    const uint32_t R = (uint32_t)a.R, T_ = a.tiles_per_chunk;
    const uint32_t items = R * T_;                              // tiles, i = t * R + q
    const uint32_t ep = read_epoch(a.epoch_ptr);                // every thread: has a barrier
    auto tile_range = [&](uint32_t i, uint32_t& q, uint32_t& t, size_t& v0, size_t& v1) {
        t = i / R;
        q = i - t * R;
        const size_t c0 = (size_t)q * a.chunk_vec;
        const size_t c1 = min(c0 + a.chunk_vec, a.nvec);
        v0 = c0 + (size_t)t * TILEV;
        v1 = min(v0 + TILEV, c1);
        if (v1 < v0) v1 = v0;
    };
    if (threadIdx.x < kWsReducers) {
        // reduce items from the ticket's low half; the next item is fetched before the
        // barrier that ends the current one (two slots: readers of one never race the writer)
        int par = 0;
        if (threadIdx.x == 0) s_item[0] = (uint32_t)atomicAdd(a.ticket, 1ull);
        named_barrier_sync(1, kWsReducers);
        uint32_t i = s_item[0];
        while (i < items) {
            uint32_t q, t;
            size_t v0, v1;
            tile_range(i, q, t, v0, v1);
            if (v0 < v1) ws_reduce_tile<T, Op, RB>(a, q, t);
            if (threadIdx.x == 0) s_item[par ^ 1] = (uint32_t)atomicAdd(a.ticket, 1ull);
            named_barrier_sync(1, kWsReducers);                 // the tile is stored
            // one release after the barrier publishes every reducer thread's stores
            if (threadIdx.x == 0 && v0 < v1) st_release_u32(a.flags + (size_t)q * a.flag_stride + t, ep);
            par ^= 1;
            i = s_item[par];
        }
        if (a.tail_n && blockIdx.x == gridDim.x - 1) reduce_tail<T, Op>(a, 0, a.R);
        return;
    }
    if (threadIdx.x != kWsReducers || R < 2) return;           // lane 0 of the copy warp drives
    uint64_t* bar = reinterpret_cast<uint64_t*>(ws_smem + (size_t)kWsStages * kPullTileBytes);
    for (int s = 0; s < kWsStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    bool alive = true;                   // false once a flag wait ran out: issue nothing more
    // the copies: for every tile taken from the ticket's high half, one per reader r != q
    uint32_t cur_i = 0, cur_j = R - 1;   // tile being split into copies, next reader index
    struct Copy {
        uint32_t q, t, r, bytes;
        size_t off;
    };
    auto next_copy = [&](Copy& c) {
        while (cur_j == R - 1) {                                // take the next non-empty tile
            cur_i = (uint32_t)(atomicAdd(a.ticket, 1ull << 32) >> 32);
            if (cur_i >= items) return false;
            uint32_t q, t;
            size_t v0, v1;
            tile_range(cur_i, q, t, v0, v1);
            if (v0 < v1) cur_j = 0;
        }
        size_t v0, v1;
        tile_range(cur_i, c.q, c.t, v0, v1);
        c.r = cur_j < c.q ? cur_j : cur_j + 1;
        c.off = v0 * kVecBytes;
        c.bytes = (uint32_t)((v1 - v0) * kVecBytes);
        if (cur_j == 0 && alive) {                              // first copy of the tile: acquire
            const uint32_t* f = a.flags + (size_t)c.q * a.flag_stride + c.t;
            alive = bounded_spin([&] { return ld_acquire_u32(f) == ep; }, a.timeout_ns, a.giveup, ep);
            if (!alive) report_timeout(a.status, a.giveup, ep, kSitePullFlag, c.q, c.t);
            fence_proxy_async_global();
        }
        ++cur_j;
        return true;
    };
    const uint64_t pol_first = l2_policy_evict_first();
    auto issue_load = [&](const Copy& c, int s) {
        const uint32_t bytes = alive ? c.bytes : 0u;
        mbar_expect_tx(&bar[s], bytes);
        if (bytes) {
            // the tile's last reader marks it evict-first: nothing reads it again
            const bool last = c.r == (c.q == R - 1 ? R - 2 : R - 1);
            if (last)
                bulk_load_hint(ws_smem + (size_t)s * kPullTileBytes,
                               a.recv + (size_t)c.q * a.rstride + c.off, bytes, &bar[s], pol_first);
            else
                bulk_load(ws_smem + (size_t)s * kPullTileBytes, a.recv + (size_t)c.q * a.rstride + c.off,
                          bytes, &bar[s]);
        }
    };
    Copy ring[kWsStages];
    uint64_t issued = 0, done = 0;
    while (issued < (uint64_t)kWsLoads && next_copy(ring[issued % kWsStages])) {
        issue_load(ring[issued % kWsStages], (int)(issued % kWsStages));
        ++issued;
    }
    while (done < issued) {
        const int s = (int)(done % kWsStages);
        const uint32_t parity = (uint32_t)((done / kWsStages) & 1u);
        uint32_t spins = 0;
        while (!mbar_try_wait(&bar[s], parity)) {
            if (++spins > (1u << 26)) {                         // a bulk load never fails; bounded anyway
                report_timeout(a.status, a.giveup, ep, kSiteBulkStage, blockIdx.x, (uint32_t)done);
                bulk_wait_all<0>();
                return;
            }
        }
        const Copy& c = ring[s];
        if (alive && c.bytes)
            bulk_store(a.recv + (size_t)c.r * a.rstride + c.off, ws_smem + (size_t)s * kPullTileBytes,
                       c.bytes);
        bulk_commit();
        ++done;
        Copy n;
        if (next_copy(n)) {
            // stage issued % stages was last read by the store of copy issued - stages,
            // committed before the one just committed
            bulk_wait_read<kWsStages - kWsLoads>();
            ring[issued % kWsStages] = n;
            issue_load(n, (int)(issued % kWsStages));
            ++issued;
        }
    }
    bulk_wait_all<0>();
}

// ----------------------------------------------------------------- host launcher


template <class T, class Op>
sym_status_t launch_algo(sym_algo_t algo, ArArgs& a, sym_win_t recv, cudaStream_t st) {
    DevCtx* ctx = recv->ctx;
    const int sms = ctx->num_sms;
    const bool wide = a.R > 4;
    // two-shot: one 16-byte vector per thread and rank in flight per item (4 KiB per rank per
    // block): as fast as two at 64 MiB+ per rank, up to 20 % faster below (more blocks)
    void (*kst)(ArArgs) = wide ? k_twoshot_st<T, Op, 8, 1> : k_twoshot_st<T, Op, 4, 1>;
    void (*kone)(ArArgs) = wide ? k_oneshot<T, Op, 8, 2> : k_oneshot<T, Op, 4, 2>;
    void (*kpull)(ArArgs) = k_twoshot_pull<T, Op, 4>;   // 4-rank batches: 3 CTAs per SM
    constexpr size_t TILEV2 = (size_t)kThreads * 2, TILEVP = (size_t)kThreads * kPullU;
    a.status = ctx->status;
    a.timeout_ns = default_timeout_ns();
    switch (algo) {
        case SYM_ALGO_ONESHOT: {
            a.ntile = (uint32_t)ceil_div(a.nvec, TILEV2);
            size_t items = (size_t)a.R * a.ntile;
            int occ = occupancy((const void*)kone, kThreads, 0);
            size_t grid = std::min(std::max(items, (size_t)1), (size_t)occ * sms);
            kone<<<(unsigned)grid, kThreads, 0, st>>>(a);
            count_launch();
            break;
        }
        case SYM_ALGO_TWOSHOT: {
            if (twoshot_use_bulk()) {
                void (*kb)(ArArgs) = k_twoshot_bulk<T, Op>;
                const size_t smem = bulk_smem_bytes(a.R);
                SYM_CUDA(cudaFuncSetAttribute((const void*)kb,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
                a.tiles_per_chunk =
                    (uint32_t)ceil_div(a.chunk_vec, (size_t)bulk_tile_bytes(a.R) / kVecBytes);
                size_t items = (size_t)a.R * a.tiles_per_chunk;
                int occ = occupancy((const void*)kb, kThreads, smem);
                size_t grid = std::min(std::max(items, (size_t)1), (size_t)occ * sms);
                kb<<<(unsigned)grid, kThreads, smem, st>>>(a);
                count_launch();
                break;
            }
            a.tiles_per_chunk = (uint32_t)ceil_div(a.chunk_vec, (size_t)kThreads);
            // One work item per block, not a persistent grid: blocks start in
            // index order as earlier ones finish, so the HBM pages in use at
            // any moment stay close together.  On GB300 this streamed 4-6 %
            // faster than the best persistent shape (one resident CTA per SM
            // walking the items).
            size_t grid = std::max((size_t)a.R * a.tiles_per_chunk, (size_t)1);
            kst<<<(unsigned)grid, kThreads, 0, st>>>(a);
            count_launch();
            break;
        }
        case SYM_ALGO_TWOSHOT_PULL:
        case SYM_ALGO_TWOSHOT_SPLIT: {
            a.tiles_per_chunk = (uint32_t)ceil_div(a.chunk_vec, TILEVP);
            if (a.tiles_per_chunk > recv->flag_tiles) return SYM_ERR_INVALID_ARG;
            a.flags = recv->flags;
            a.flag_stride = recv->flag_tiles;
            int occ = occupancy((const void*)kpull, kThreads, 0);
            size_t cap = (size_t)occ * sms;
            if (algo == SYM_ALGO_TWOSHOT_SPLIT || a.R == 1) {
                size_t rs = std::max((size_t)a.R * a.tiles_per_chunk, (size_t)1);
                // split: the reduce-scatter launch takes one item per block
                // (1.5 % faster than a persistent grid); the all-gather launch
                // keeps a persistent grid (one item per block: 10 % slower)
                a.mode = 1;
                kpull<<<(unsigned)rs, kThreads, 0, st>>>(a);
                count_launch();
                if (a.R > 1 && a.tiles_per_chunk > 0) {
                    size_t ag = (size_t)(a.R - 1) * a.R * a.tiles_per_chunk;
                    a.mode = 2;
                    kpull<<<(unsigned)std::min(ag, cap), kThreads, 0, st>>>(a);
                    count_launch();
                }
                break;
            }
            // fused: blocks wait on one another -> co-residency via a cooperative launch
            // the warp-specialised kernel above 256 KiB per rank; below, the single-role
            // kernel's register copies reach a tile sooner than a bulk load and store
            // (CUDA-graph device time per call, R = 8: 5.2 vs 8.8 us at 1 KiB, 10.8 vs
            // 12.2 us at 256 KiB, 13.3 vs 12.8 us at 1 MiB)
            const bool ws = pull_use_ws(a.nvec * kVecBytes);
            {
                // the warp-specialised kernel takes its work from the window's ticket
                sym_status_t s = bump_epoch(recv->epoch, st, ws ? recv->ticket : nullptr);
                if (s != SYM_OK) return s;
            }
            a.epoch_ptr = recv->epoch;
            a.giveup = recv->giveup;
            a.ticket = recv->ticket;
            a.mode = 0;
            if (ws) {
                void (*kws)(ArArgs) = k_twoshot_pull_ws<T, Op, 8>;
                const size_t smem = ws_smem_bytes();
                SYM_CUDA(cudaFuncSetAttribute((const void*)kws,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
                const int occ_ws = occupancy((const void*)kws, kWsThreads, smem);
                const size_t items = std::max((size_t)a.R * a.tiles_per_chunk, (size_t)1);
                const size_t grid = std::min(items, (size_t)std::max(occ_ws, 1) * sms);
                void* args[] = {&a};
                SYM_CUDA(cudaLaunchCooperativeKernel((const void*)kws, dim3((unsigned)grid),
                                                     dim3(kWsThreads), args, smem, st));
                count_launch();
                break;
            }
            // two 16 KiB tiles per item, gathers 4 grid waves behind: measured best
            // of 1/2/4/8 tiles x 2/4/8 waves (R = 8 x 256 MiB fp32: 0.721 -> 0.685 ms)
            a.group = kPullGroup;
            size_t slots = (size_t)a.R * a.R * ceil_div(a.tiles_per_chunk, (size_t)a.group);
            size_t grid = std::min(std::max(slots, (size_t)1), cap);
            a.lag = (uint32_t)(pull_lag_waves() * ceil_div(grid, (size_t)a.R * a.R)) + 1;
            void* args[] = {&a};
            SYM_CUDA(cudaLaunchCooperativeKernel((const void*)kpull, dim3((unsigned)grid),
                                                 dim3(kThreads), args, 0, st));
            count_launch();
            break;
        }
        default:
            return SYM_ERR_INVALID_ARG;
    }
    if (trace_on())
        fprintf(stderr, "[symar] allreduce algo=%d R=%d nvec=%zu tail=%u\n", (int)algo, a.R, a.nvec,
                a.tail_n);
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

template <class T>
sym_status_t launch_allreduce_typed(sym_algo_t algo, sym_op_t op, ArArgs& a, sym_win_t recv,
                                    cudaStream_t st) {
    switch (op) {
        case SYM_SUM: return launch_algo<T, OpSum>(algo, a, recv, st);
        case SYM_MAX: return launch_algo<T, OpMax>(algo, a, recv, st);
        case SYM_MIN: return launch_algo<T, OpMin>(algo, a, recv, st);
    }
    return SYM_ERR_INVALID_ARG;
}

// one per element type, each in its own translation unit
sym_status_t launch_allreduce_f32(sym_algo_t, sym_op_t, ArArgs&, sym_win_t, cudaStream_t);
sym_status_t launch_allreduce_bf16(sym_algo_t, sym_op_t, ArArgs&, sym_win_t, cudaStream_t);
sym_status_t launch_allreduce_f16(sym_algo_t, sym_op_t, ArArgs&, sym_win_t, cudaStream_t);

}  // namespace symar
