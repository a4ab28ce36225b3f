// AllGather, one-sided put with signal/counter actions, and bounded waits.
//
// [SYMEX] Example 2: recv_r holds sendcount*R elements, segment q = rank q's
// send buffer.  [GIN] put(peer, dstWnd, dstOffset, srcWnd, srcOffset, bytes,
// remoteAction = SignalInc, localAction = CounterInc); a strong signal's
// visibility implies every earlier put on the same context to the same peer
// is visible; signals and counters are 64-bit values under 32-bit IDs,
// counters read through 56 bits; waitSignal(least, bits) uses a rolling
// comparison.  [GDA] section 4: a batch of puts closed by one signal orders
// the batch without a global fence; section 5.1: completion flags use
// release stores and an acquire spin with a short sleep.
//
// On one GPU a "put to peer p" is a copy into rank p's part of the
// destination window, and remote visibility is device-scope visibility, so
// every release/acquire here is .gpu scope (sys scope would also drain the
// host path and is never needed: [GDA] section 5.2 notes its cost).
#include <cstdio>

#include "symar_internal.cuh"

namespace symar {

constexpr int kCopyThreads = 256;
constexpr int kCopyU = 4;
constexpr int kPutThreads = 512;
constexpr int kPutU = 4;

// ----------------------------------------------------------------- AllGather (copy)

struct AgArgs {
    const char* send;
    char* recv;
    size_t sstride, rstride;
    int R;
    size_t S;                 // bytes per rank segment
    size_t nvec;              // S / 16 (vector path)
    uint32_t tiles;           // tiles per segment
};

// Each item reads one tile of segment q once and stores it to all R ranks.
__global__ void __launch_bounds__(kCopyThreads) k_allgather_copy(AgArgs a) {
    constexpr size_t TILEV = (size_t)kCopyThreads * kCopyU;
    const uint32_t items = (uint32_t)a.R * a.tiles;
    for (uint32_t w = blockIdx.x; w < items; w += gridDim.x) {
        const uint32_t t = w / (uint32_t)a.R, q = w - t * (uint32_t)a.R;
        const char* src = a.send + (size_t)q * a.sstride;
        const size_t seg = (size_t)q * a.S;
        uint4 v[kCopyU];
        size_t idx[kCopyU];
#pragma unroll
        for (int k = 0; k < kCopyU; ++k) {
            idx[k] = (size_t)t * TILEV + threadIdx.x + (size_t)k * kCopyThreads;
            if (idx[k] < a.nvec) v[k] = __ldcs(reinterpret_cast<const uint4*>(src + idx[k] * 16));
        }
        for (int r = 0; r < a.R; ++r) {
            char* dst = a.recv + (size_t)r * a.rstride + seg;
#pragma unroll
            for (int k = 0; k < kCopyU; ++k)
                if (idx[k] < a.nvec) __stcs(reinterpret_cast<uint4*>(dst + idx[k] * 16), v[k]);
        }
    }
}

// AllGather staged through shared memory by the TMA engine.  One block per
// 16 KiB tile of a segment: one thread loads the tile once with a bulk copy
// (mbarrier completion) and writes it to all R ranks with R bulk stores, so
// the SM's load/store queues carry none of the R-fold stores (the register
// version stalls on them).  Blocks are not persistent: they start in index
// order (segment-major), which keeps the written HBM pages close together; on
// GB300 this measured 12 % faster than a persistent ring of stages per block.
// Needs S % 16 == 0.
constexpr uint32_t kAgTile = 16384;
constexpr int kAgThreads = 32;

__global__ void __launch_bounds__(kAgThreads) k_allgather_bulk(AgArgs a, uint32_t* status) {
    __shared__ __align__(128) unsigned char tile[kAgTile];
    __shared__ uint64_t full;
    if (threadIdx.x != 0) return;
    const uint32_t q = blockIdx.x / a.tiles, t = blockIdx.x - q * a.tiles;
    const size_t off = (size_t)t * kAgTile;
    const uint32_t bytes = (uint32_t)min((size_t)kAgTile, a.S - off);
    mbar_init(&full, 1);
    fence_mbar_init();
    mbar_expect_tx(&full, bytes);
    bulk_load(tile, a.send + (size_t)q * a.sstride + off, bytes, &full);
    uint32_t spins = 0;
    while (!mbar_try_wait(&full, 0)) {
        if (++spins > (1u << 26)) {          // bounded: a load cannot stall on valid ranges
            report_timeout(status, nullptr, 0u, kSiteBulkStage, q, t);
            // the load still targets this block's shared memory: give it the
            // same bound once more before the block exits
            for (uint32_t k = 0; k < (1u << 26) && !mbar_try_wait(&full, 0); ++k) {
            }
            return;
        }
    }
    for (int r = 0; r < a.R; ++r)
        bulk_store(a.recv + (size_t)r * a.rstride + (size_t)q * a.S + off, tile, bytes);
    bulk_commit();
    bulk_wait_read<0>();          // shared memory must outlive the stores' reads
}

// Byte-granular fallback when S is not a multiple of 16.
__global__ void k_allgather_bytes(AgArgs a) {
    const size_t total = (size_t)a.R * a.S;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t q = i / a.S, off = i - q * a.S;
        const unsigned char b = (unsigned char)a.send[q * a.sstride + off];
        for (int r = 0; r < a.R; ++r) a.recv[(size_t)r * a.rstride + q * a.S + off] = (char)b;
    }
}

// ----------------------------------------------------------------- copy helper

// Block-wide copy of [lo, hi) bytes from src to dst (same offsets).
template <int THREADS, int U>
__device__ __forceinline__ void block_copy(const char* src, char* dst, size_t lo, size_t hi,
                                           bool vec) {
    if (vec) {
        const size_t v0 = lo / 16, v1 = hi / 16;
        for (size_t base = v0; base < v1; base += (size_t)THREADS * U) {
            uint4 v[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const size_t i = base + threadIdx.x + (size_t)k * THREADS;
                if (i < v1) v[k] = __ldcs(reinterpret_cast<const uint4*>(src + i * 16));
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const size_t i = base + threadIdx.x + (size_t)k * THREADS;
                if (i < v1) __stcs(reinterpret_cast<uint4*>(dst + i * 16), v[k]);
            }
        }
    } else {
        for (size_t i = lo + threadIdx.x; i < hi; i += THREADS) dst[i] = src[i];
    }
}

// ----------------------------------------------------------------- put + signal AllGather

struct PsArgs {
    const char* send;
    char* recv;
    size_t sstride, rstride;
    int R;
    size_t S, chunk;
    uint32_t B, nchunks, nbatches;
    uint64_t* sig;            // recv window signals [R][nsig]
    uint32_t nsig;
    uint64_t* cnt;            // send window counters [R][ncnt]
    uint32_t ncnt;
    uint64_t* mismatch;       // optional prefix-visibility check
    unsigned long long* ticket;   // recv window item ticket, zeroed by the reset kernel
    uint32_t* ring;           // recv window [R][R][2] piece counters by batch parity
    // item geometry (see k_put_signal_allgather)
    uint32_t nrows;           // rows of items
    uint32_t bpr;             // batches per row (ppi == 1), else 1
    uint32_t ppi;             // items per stream in a row (pieces of one batch), 1 = whole batches
    uint32_t gchunks;         // chunks per piece when ppi > 1
    uint32_t* status;
    const uint32_t* epoch;    // recv window epoch (this launch's give-up tag)
    uint32_t* giveup;         // recv window give-up word
    uint64_t timeout_ns;
    int vec;
    int bulk;                 // puts by bulk copies (needs vec); else register copies
    int drop_signal;          // fault injection for tests: stream (0 -> 0) omits its last (1) or first (2) signal
};

__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* s_red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    uint64_t t = 0;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += s_red[i];
    __syncthreads();
    return t;
}

// Bulk copy (TMA engine) of [lo, hi) from src to ndst destinations (dst,
// dst + dst_stride, ...) by one thread, through a ring of kPsStages 16 KiB
// shared-memory stages: each tile is loaded once and stored ndst times; loads
// run kPsStages - 1 tiles ahead of the stores.  `gtile` counts the tiles this
// block has moved so far (it carries the mbarrier phases from one call to the
// next).  Returns when every store has completed, or false if a stage's load
// did not arrive within the bound.  lo, hi, src, dst and dst_stride are
// 16-byte aligned.
constexpr int kPsStages = 4;
constexpr uint32_t kPsTile = 16384;
constexpr size_t kPsSmem = (size_t)kPsStages * kPsTile + kPsStages * sizeof(uint64_t);

__device__ __forceinline__ bool bulk_copy_range(const char* src, char* dst, size_t dst_stride,
                                                uint32_t ndst, size_t lo, size_t hi,
                                                unsigned char* stage, uint64_t* full, uint32_t& gtile) {
    const uint32_t n = (uint32_t)((hi - lo + kPsTile - 1) / kPsTile);
    auto bytes_of = [&](uint32_t i) { return (uint32_t)min((size_t)kPsTile, hi - lo - (size_t)i * kPsTile); };
    auto load = [&](uint32_t i) {
        const uint32_t s = (gtile + i) % kPsStages;
        mbar_expect_tx(&full[s], bytes_of(i));
        bulk_load(stage + (size_t)s * kPsTile, src + lo + (size_t)i * kPsTile, bytes_of(i), &full[s]);
    };
    for (uint32_t i = 0; i + 1 < (uint32_t)kPsStages && i < n; ++i) load(i);
    bool ok = true;
    for (uint32_t i = 0; i < n && ok; ++i) {
        const uint32_t g = gtile + i, s = g % kPsStages;
        uint32_t spins = 0;
        while (!mbar_try_wait(&full[s], (g / kPsStages) & 1u))
            if (++spins > (1u << 26)) {                   // bounded: loads of valid ranges arrive
                ok = false;
                break;
            }
        if (!ok) break;
        for (uint32_t d = 0; d < ndst; ++d)
            bulk_store(dst + (size_t)d * dst_stride + lo + (size_t)i * kPsTile,
                       stage + (size_t)s * kPsTile, bytes_of(i));
        bulk_commit();
        const uint32_t nxt = i + kPsStages - 1;           // refills the stage of tile i-1
        if (nxt < n) {
            bulk_wait_read<1>();
            load(nxt);
        }
    }
    bulk_wait_all<0>();                                   // the stores are complete
    asm volatile("fence.proxy.async.global;" ::: "memory");   // ... and ordered before generic accesses
    gtile += n;
    return ok;
}

// Work items are handed out in index order by the window's ticket
// (fetch_item) and have a fixed size whatever the batch size: in a row of
// items, either one item puts `bpr` whole batches (small batches) or `ppi`
// items each put a piece of one batch (large batches).  With bulk copies an
// item is 128 KiB of sender q's source put to all R peers (the R puts of the
// same range share one read, as the SM AllGather does); with register copies
// it is 512 KiB of one (q -> p) stream.  With the prefix check on, each row
// ends with one check item per stream; with it off, one receiver item per
// stream follows the last row and waits for the final count.
//
// A batch's signal must follow the previous batch's signal of the same
// stream: the item that completes batch b first waits (acquire) until the
// stream's signal reads b, then adds 1 with a release, so a receiver that
// reads k sees batches 0..k-1 (each release carries the earlier ones by
// causality).  Pieces of a batch count their arrivals in a two-entry ring per
// stream, or per sender with bulk copies (by batch parity); a piece of batch b
// first waits until batch b-2 is signalled, which frees its ring entry.  Every wait is for items handed out
// earlier, which running blocks hold, so no wait depends on a block that has
// not started.
__global__ void __launch_bounds__(kPutThreads) k_put_signal_allgather(PsArgs a) {
    __shared__ unsigned long long s_item[2];
    __shared__ int s_ok[2];
    __shared__ int s_sig;             // the put item completes a batch: add its signals
    __shared__ uint64_t s_red[kPutThreads / 32];
    extern __shared__ __align__(128) unsigned char ps_stage[];   // a.bulk: kPsSmem bytes
    uint64_t* ps_full = reinterpret_cast<uint64_t*>(ps_stage + (size_t)kPsStages * kPsTile);
    uint32_t gtile = 0;
    bool copy_ok = true;
    if (a.bulk && threadIdx.x == 0) {
        for (int i = 0; i < kPsStages; ++i) mbar_init(&ps_full[i], 1);
        fence_mbar_init();
    }
    const uint32_t tag = read_epoch(a.epoch);      // bumped by the reset kernel before (syncs the block)
    const uint32_t R = (uint32_t)a.R, pairs = R * R;
    const uint64_t puts = (uint64_t)(a.bulk ? R : pairs) * a.ppi;
    const uint64_t row = puts + (a.mismatch ? pairs : 0u);
    const uint64_t total = row * a.nrows + (a.mismatch ? 0ull : (uint64_t)pairs);
    int ipar = 0, opar = 0;
    auto sig_at = [&](uint32_t p, uint32_t q) { return a.sig + (size_t)p * a.nsig + q; };
    for (;;) {
        const uint64_t w = fetch_item(a.ticket, s_item, ipar);
        if (w >= total) break;
        const uint32_t r = (uint32_t)(w / row);
        const uint64_t slot = w - (uint64_t)r * row;
        // batches [b0, b1) of this row
        const uint32_t b0 = r * a.bpr, b1 = min(b0 + a.bpr, a.nbatches);
        if (r < a.nrows && slot < puts) {
            // ---- a put item: piece j of the row for one stream (q -> p), or,
            // with bulk copies, for all R streams of sender q at once (the R
            // puts of the same source range read it once)
            uint32_t q, p0, np, j, key;
            if (a.bulk) {
                j = (uint32_t)(slot / R);
                q = (uint32_t)(slot - (uint64_t)j * R);
                p0 = 0;
                np = R;
                key = q;
            } else {
                // streams vary fastest (the items in flight cover one piece of
                // many streams), senders fastest within them (peer-major
                // measured 1-3 % faster than sender-major)
                j = (uint32_t)(slot / pairs);
                const uint32_t pr = (uint32_t)(slot - (uint64_t)j * pairs);
                p0 = pr / R;
                q = pr - p0 * R;
                np = 1;
                key = pr;
            }
            uint32_t k0, k1;                      // chunks
            if (a.ppi == 1) {
                k0 = b0 * a.B;
                k1 = min(b1 * a.B, a.nchunks);
            } else {
                k0 = min(b0 * a.B + j * a.gchunks, a.nchunks);
                k1 = min(min(k0 + a.gchunks, (b0 + 1) * a.B), a.nchunks);
            }
            const char* src = a.send + (size_t)q * a.sstride;
            char* dst = a.recv + (size_t)p0 * a.rstride + (size_t)q * a.S;
            const size_t lo = min((size_t)k0 * a.chunk, a.S), hi = min((size_t)k1 * a.chunk, a.S);
            if (a.bulk) {
                if (threadIdx.x == 0 && hi > lo)
                    copy_ok = bulk_copy_range(src, dst, a.rstride, np, lo, hi, ps_stage, ps_full, gtile);
            } else {
                block_copy<kPutThreads, kPutU>(src, dst, lo, hi, a.vec != 0);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                if (!copy_ok)      // no signal: the stream's receiver then reports as well
                    report_timeout(a.status, a.giveup, tag, kSiteBulkStage, (uint32_t)(w >> 32),
                                   (uint32_t)w);
                if (copy_ok && k1 > k0)
                    atomicAdd(reinterpret_cast<unsigned long long*>(a.cnt + (size_t)q * a.ncnt),
                              (unsigned long long)(k1 - k0) * np);      // local completion
                bool last = true, ok = copy_ok;
                if (a.ppi > 1 && ok) {
                    // free ring entry: batch b0-2 signalled (its last piece
                    // reset the entry before adding any of its signals)
                    const uint64_t need = b0 >= 2 ? b0 - 1 : 0;
                    const uint64_t* sp = sig_at(p0, q);
                    ok = need == 0 || bounded_spin([&] { return ld_acquire_u64(sp) >= need; },
                                                   a.timeout_ns, a.giveup, tag);
                    if (!ok) report_timeout(a.status, a.giveup, tag, kSiteSignalChain, p0, q);
                    if (ok) {
                        uint32_t* cnt = a.ring + ((size_t)key << 1) + (b0 & 1u);
                        last = atomicAdd(cnt, 1u) == a.ppi - 1;
                        if (last) {
                            *cnt = 0;
                            __threadfence();
                        }
                    }
                }
                s_sig = ok && last ? 1 : 0;
            }
            __syncthreads();
            if (s_sig) {
                // batch order: thread i waits (acquire) until stream (p0 + i -> q)
                // has signalled batch b0-1, then, once all have, adds that
                // stream's signals for batches b0..b1-1 after a fence (a release
                // pattern: it carries the item's bytes, ordered before the
                // barrier, and the acquired predecessor)
                bool okp = true;
                const uint32_t p = p0 + threadIdx.x;
                if (threadIdx.x < np && b0 > 0) {
                    const uint64_t* sp = sig_at(p, q);
                    const uint64_t before = b0;
                    okp = bounded_spin([&] { return ld_acquire_u64(sp) >= before; }, a.timeout_ns,
                                       a.giveup, tag);
                    if (!okp) report_timeout(a.status, a.giveup, tag, kSiteSignalChain, p, q);
                }
                if (__syncthreads_and(okp) && threadIdx.x < np) {
                    __threadfence();
                    for (uint32_t b = b0; b < b1; ++b) {
                        const bool dropped = p == 0 && q == 0 &&
                                             ((a.drop_signal == 1 && b + 1 == a.nbatches) ||
                                              (a.drop_signal == 2 && b == 0));
                        if (!dropped) red_relaxed_add_u64(sig_at(p, q), 1ull);
                    }
                }
            }
        } else if (r < a.nrows) {
            // ---- check: once the signal shows batch b1-1, batches [b0, b1) equal the source
            const uint32_t pr = (uint32_t)(slot - puts), p = pr / R, q = pr - p * R;
            if (threadIdx.x == 0) {
                const uint64_t* sp = sig_at(p, q);
                const uint64_t want = b1;
                const bool got = bounded_spin([&] { return ld_acquire_u64(sp) >= want; },
                                              a.timeout_ns, a.giveup, tag);
                if (!got) report_timeout(a.status, a.giveup, tag, kSitePutSignalRecv, p, q);
                s_ok[opar] = got ? 1 : 0;
            }
            __syncthreads();
            const bool go = s_ok[opar] != 0;
            opar ^= 1;
            if (!go) continue;
            const char* src = a.send + (size_t)q * a.sstride;
            const char* seg = a.recv + (size_t)p * a.rstride + (size_t)q * a.S;
            const size_t lo = min((size_t)b0 * a.B * a.chunk, a.S);
            const size_t hi = min((size_t)b1 * a.B * a.chunk, a.S);
            uint64_t bad = 0;
            for (size_t i = lo + threadIdx.x; i < hi; i += kPutThreads)
                bad += (__ldcg(reinterpret_cast<const unsigned char*>(seg + i)) !=
                        __ldcg(reinterpret_cast<const unsigned char*>(src + i)));
            bad = block_sum_u64(bad, s_red);
            if (threadIdx.x == 0 && bad)
                atomicAdd(reinterpret_cast<unsigned long long*>(a.mismatch), (unsigned long long)bad);
        } else {
            // ---- receiver (check off): wait for the stream's final count
            const uint32_t pr = (uint32_t)slot, p = pr / R, q = pr - p * R;
            if (threadIdx.x == 0) {
                const uint64_t* sp = sig_at(p, q);
                const uint64_t want = a.nbatches;
                if (!bounded_spin([&] { return ld_acquire_u64(sp) >= want; }, a.timeout_ns,
                                  a.giveup, tag))
                    report_timeout(a.status, a.giveup, tag, kSitePutSignalRecv, p, q);
            }
        }
    }
}

// ----------------------------------------------------------------- AlltoAll

// [GIN] pure-GIN AlltoAll: sender q puts segment p of its send buffer into
// rank p's receive buffer at segment q, with one signal increment per put;
// the receiver waits for R increments.  Here a segment is moved in `pieces`
// parts by different CTAs (enough parallelism for any R); in the put+signal
// form the CTA that completes the last part of a (q -> p) segment adds 1 to
// signal slot 0 of rank p, so each segment put still signals exactly once.
struct A2aArgs {
    const char* send;
    char* recv;
    size_t sstride, rstride;
    int R;
    size_t B;                 // bytes per segment
    size_t piece;             // bytes per part (multiple of 16 when vec)
    uint32_t pieces;          // parts per segment
    int vec;
    uint64_t* sig;            // recv window signals, slot 0 of each rank (put+signal form)
    uint32_t nsig;
    uint32_t* pair_done;      // [R][R] parts completed, zero when idle (put+signal form)
    unsigned long long* ticket;   // recv window item ticket (put+signal form)
    uint32_t* status;
    const uint32_t* epoch;    // recv window epoch (put+signal form: the give-up tag)
    uint32_t* giveup;         // recv window give-up word
    uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kPutThreads) k_alltoall(A2aArgs a) {
    const uint32_t R = (uint32_t)a.R, items = R * R * a.pieces;
    auto put_part = [&](uint32_t it, uint32_t& q, uint32_t& p) {
        const uint32_t pr = it / a.pieces, part = it - pr * a.pieces;
        q = pr / R;
        p = pr - q * R;
        const char* src = a.send + (size_t)q * a.sstride + (size_t)p * a.B;
        char* dst = a.recv + (size_t)p * a.rstride + (size_t)q * a.B;
        const size_t lo = min((size_t)part * a.piece, a.B), hi = min(lo + a.piece, a.B);
        block_copy<kPutThreads, kPutU>(src, dst, lo, hi, a.vec != 0);
    };
    if (!a.sig) {                                    // copy form: one part per block
        for (uint32_t it = blockIdx.x; it < items; it += gridDim.x) {
            uint32_t q, p;
            put_part(it, q, p);
        }
        return;
    }
    // put + signal form: parts, then one receiver item per rank, handed out in
    // index order by the window's ticket (receivers wait only on parts that
    // running blocks already hold)
    const uint32_t tag = read_epoch(a.epoch);
    __shared__ unsigned long long s_item[2];
    int ipar = 0;
    for (;;) {
        const uint64_t w = fetch_item(a.ticket, s_item, ipar);
        if (w >= (uint64_t)items + R) break;
        if (w < items) {
            uint32_t q, p;
            put_part((uint32_t)w, q, p);
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                uint32_t* done = a.pair_done + (size_t)q * R + p;
                if (atomicAdd(done, 1u) == a.pieces - 1) {     // last part of the segment
                    *done = 0;
                    __threadfence();
                    red_release_add_u64(a.sig + (size_t)p * a.nsig, 1ull);
                }
            }
        } else if (threadIdx.x == 0) {
            // receiver: rank p waits until all R senders have signalled
            const uint32_t p = (uint32_t)(w - items);
            const uint64_t* sp = a.sig + (size_t)p * a.nsig;
            if (!bounded_spin([&] { return ld_acquire_u64(sp) >= (uint64_t)R; }, a.timeout_ns,
                              a.giveup, tag))
                report_timeout(a.status, a.giveup, tag, kSitePutSignalRecv, p, 0xA2Au);
        }
    }
}

// The reset kernels run in stream order before the launch that waits; they
// also advance the receiving window's epoch, the waiting launch's give-up tag.
__device__ __forceinline__ void bump_epoch_here(uint32_t* epoch) {
    if (threadIdx.x == 0) {
        const uint32_t e = *epoch + 1u;
        *epoch = e ? e : 1u;
    }
}

__global__ void k_reset_slot0(uint64_t* sig, uint32_t nsig, int R, uint32_t* epoch,
                              unsigned long long* ticket) {
    for (int p = threadIdx.x; p < R; p += blockDim.x) sig[(size_t)p * nsig] = 0;
    if (threadIdx.x == 0) *ticket = 0ull;
    bump_epoch_here(epoch);
}

__global__ void k_reset_slots(uint64_t* sig, uint32_t nsig, uint64_t* cnt, uint32_t ncnt, int R,
                              uint32_t* epoch, unsigned long long* ticket) {
    for (int i = threadIdx.x; i < R * R; i += blockDim.x) {
        const int p = i / R, q = i - p * R;
        sig[(size_t)p * nsig + q] = 0;
    }
    for (int q = threadIdx.x; q < R; q += blockDim.x) cnt[(size_t)q * ncnt] = 0;
    if (threadIdx.x == 0) *ticket = 0ull;
    bump_epoch_here(epoch);
}

// ----------------------------------------------------------------- single put

struct PutArgs {
    const char* src;
    char* dst;
    size_t bytes;
    int vec;
    uint64_t* sig;            // nullable
    uint64_t* cnt;            // nullable
    uint32_t* arrive;         // arrival counter of this launch (zero on entry)
};

__global__ void __launch_bounds__(kPutThreads) k_put(PutArgs a) {
    // this CTA's share of the bytes, 16-byte aligned
    const size_t per = ((a.bytes + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
    const size_t lo = min((size_t)blockIdx.x * per, a.bytes), hi = min(lo + per, a.bytes);
    block_copy<kPutThreads, kPutU>(a.src, a.dst, lo, hi, a.vec != 0);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(a.arrive, 1u);
        if (prev == gridDim.x - 1) {            // last CTA: every byte is in place
            *a.arrive = 0;
            __threadfence();
            if (a.cnt) atomicAdd(reinterpret_cast<unsigned long long*>(a.cnt), 1ull);
            if (a.sig) red_release_add_u64(a.sig, 1ull);
        }
    }
}

__global__ void k_signal_add(uint64_t* sig, uint64_t value) {
    __threadfence();
    red_release_add_u64(sig, value);
}

__global__ void k_wait_slot(const uint64_t* slot, uint64_t least, int bits, uint64_t timeout_ns,
                            uint32_t* status, uint32_t site, uint32_t a, uint32_t b) {
    if (threadIdx.x != 0) return;
    bool ok = bounded_spin([&] { return rolling_le_dev(least, ld_acquire_u64(slot), bits); },
                           timeout_ns, nullptr, 0u);
    if (!ok) report_timeout(status, nullptr, 0u, site, a, b);
}

}  // namespace symar

using namespace symar;

static bool same_group(sym_win_t a, sym_win_t b) {
    return a && b && a->R == b->R && a->device == b->device;
}

static sym_status_t launch_put_signal_allgather(sym_win_t send, sym_win_t recv, size_t S,
                                                size_t chunk, uint32_t B, uint64_t* d_mismatch,
                                                uint64_t timeout_ns, cudaStream_t st) {
    const int R = send->R;
    if (recv->nsignals < (uint32_t)R || send->ncounters < 1) return SYM_ERR_INVALID_ARG;
    if (chunk == 0) chunk = 64 * 1024;
    if (B == 0) B = 8;
    const size_t nchunks = ceil_div(S, chunk);
    if (nchunks > 0xFFFFFFFFull) return SYM_ERR_INVALID_ARG;
    PsArgs a{};
    a.send = send->base;
    a.recv = recv->base;
    a.sstride = send->stride;
    a.rstride = recv->stride;
    a.R = R;
    a.S = S;
    a.chunk = chunk;
    a.B = B;
    a.nchunks = (uint32_t)nchunks;
    a.nbatches = (uint32_t)ceil_div(nchunks, (size_t)B);
    a.sig = recv->sig;
    a.nsig = recv->nsignals;
    a.cnt = send->cnt;
    a.ncnt = send->ncounters;
    a.mismatch = d_mismatch;
    a.status = recv->ctx->status;
    a.epoch = recv->epoch;
    a.giveup = recv->giveup;
    a.timeout_ns = timeout_ns ? timeout_ns : default_timeout_ns();
    if (a.timeout_ns > 60000000000ull) a.timeout_ns = 60000000000ull;
    a.vec = (S % 16 == 0 && chunk % 16 == 0) ? 1 : 0;
    a.bulk = a.vec && put_use_bulk() ? 1 : 0;
    a.drop_signal = test_drop_signal();
    a.ticket = recv->ticket;
    a.ring = recv->pair_ring;
    // per item: about 512 KiB of one stream (register copies), or 128 KiB of
    // a sender's source written to all R peers (bulk copies); whole batches
    // when a batch is at most that
    const size_t gch = std::max<size_t>(1, (a.bulk ? 128 * 1024 : 512 * 1024) / chunk);
    if (B <= gch) {
        a.bpr = (uint32_t)std::max<size_t>(1, gch / B);
        a.ppi = 1;
        a.gchunks = 0;
        a.nrows = (uint32_t)ceil_div(a.nbatches, (size_t)a.bpr);
    } else {
        a.bpr = 1;
        a.ppi = (uint32_t)ceil_div((size_t)B, gch);
        a.gchunks = (uint32_t)gch;
        a.nrows = a.nbatches;
    }
    k_reset_slots<<<1, 256, 0, st>>>(a.sig, a.nsig, a.cnt, a.ncnt, R, recv->epoch, recv->ticket);
    count_launch();
    const size_t smem = a.bulk ? kPsSmem : 0;
    if (a.bulk)
        SYM_CUDA(cudaFuncSetAttribute((const void*)k_put_signal_allgather,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPsSmem));
    int occ = 0;
    SYM_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)k_put_signal_allgather,
                                                           kPutThreads, smem));
    if (occ < 1) return SYM_ERR_UNSUPPORTED;
    const size_t cap = (size_t)occ * recv->ctx->num_sms;
    const size_t pairs = (size_t)R * R;
    const size_t items = ((a.bulk ? (size_t)R : pairs) * a.ppi + (d_mismatch ? pairs : 0)) * a.nrows +
                         (d_mismatch ? 0 : pairs);
    const size_t grid = std::max<size_t>(1, std::min(items, cap));
    void* args[] = {&a};
    // all blocks resident (cooperative launch); the ticket order alone already
    // keeps every wait on items that running blocks hold
    SYM_CUDA(cudaLaunchCooperativeKernel((const void*)k_put_signal_allgather, dim3((unsigned)grid),
                                         dim3(kPutThreads), args, smem, st));
    count_launch();
    if (trace_on())
        fprintf(stderr, "[symar] put_signal_allgather R=%d S=%zu chunk=%zu B=%u grid=%zu items=%zu\n",
                R, S, chunk, B, grid, items);
    return SYM_OK;
}

extern "C" {

sym_status_t sym_allgather(sym_win_t send, sym_win_t recv, size_t sendcount, sym_dtype_t dtype,
                           sym_algo_t algo, size_t chunk_bytes, uint32_t chunks_per_signal,
                           sym_stream_t stream) {
    if (!same_group(send, recv) || send == recv || send->base == recv->base)
        return SYM_ERR_INVALID_ARG;
    const size_t es = dtype_size(dtype);
    if (!es) return SYM_ERR_INVALID_ARG;
    if (algo != SYM_ALGO_AUTO && algo != SYM_ALGO_COPY && algo != SYM_ALGO_PUT_SIGNAL &&
        algo != SYM_ALGO_CE)
        return SYM_ERR_INVALID_ARG;
    const int R = send->R;
    if (sendcount > send->bytes / es) return SYM_ERR_INVALID_ARG;
    const size_t S = sendcount * es;
    if (S > recv->bytes / (size_t)R) return SYM_ERR_INVALID_ARG;
    if (S == 0) return SYM_OK;
    if (windows_overlap(send, S, recv, (size_t)R * S)) {
        set_last_error("sym_allgather: send and recv windows share memory");
        return SYM_ERR_INVALID_ARG;
    }
    DeviceGuard g(recv->device);
    if (!g.ok) return SYM_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    if (algo == SYM_ALGO_CE) {
        // one 1-D copy per (sender q, destination r), sender-major: the R
        // copies of a segment follow one another, so the engines read it from
        // L2 after the first.  On GB300 this ran 1.8x faster than one 2-D
        // copy per destination (rows = senders) and 1.4x faster than the
        // destination-major order.
        for (int q = 0; q < R; ++q)
            for (int r = 0; r < R; ++r)
                SYM_CUDA(cudaMemcpyAsync(recv->base + (size_t)r * recv->stride + (size_t)q * S,
                                         send->base + (size_t)q * send->stride, S,
                                         cudaMemcpyDeviceToDevice, st));
        return SYM_OK;
    }
    if (algo == SYM_ALGO_PUT_SIGNAL) {
        sym_status_t s = launch_put_signal_allgather(send, recv, S, chunk_bytes, chunks_per_signal,
                                                     nullptr, 0, st);
        if (s != SYM_OK) return s;
        SYM_CUDA(cudaGetLastError());
        return SYM_OK;
    }
    AgArgs a{};
    a.send = send->base;
    a.recv = recv->base;
    a.sstride = send->stride;
    a.rstride = recv->stride;
    a.R = R;
    a.S = S;
    const int sms = recv->ctx->num_sms;
    if (S % 16 == 0 && allgather_use_bulk()) {
        a.nvec = S / 16;
        a.tiles = (uint32_t)ceil_div(S, (size_t)kAgTile);
        const size_t items = (size_t)R * a.tiles;
        if (items > 0x7fffffffu) return SYM_ERR_UNSUPPORTED;
        k_allgather_bulk<<<(unsigned)items, kAgThreads, 0, st>>>(a, recv->ctx->status);
    } else if (S % 16 == 0) {
        a.nvec = S / 16;
        a.tiles = (uint32_t)ceil_div(a.nvec, (size_t)kCopyThreads * kCopyU);
        const size_t items = (size_t)R * a.tiles;     // one item per block (see k_allgather_bulk)
        if (items > 0x7fffffffu) return SYM_ERR_UNSUPPORTED;
        k_allgather_copy<<<(unsigned)items, kCopyThreads, 0, st>>>(a);
    } else {
        const size_t total = (size_t)R * S;
        const size_t grid = std::min(ceil_div(total, (size_t)256), (size_t)sms * 8);
        k_allgather_bytes<<<(unsigned)grid, 256, 0, st>>>(a);
    }
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_allgather_put_signal(sym_win_t send, sym_win_t recv, size_t bytes_per_rank,
                                      size_t chunk_bytes, uint32_t chunks_per_signal,
                                      uint64_t* d_mismatch, uint64_t timeout_ns,
                                      sym_stream_t stream) {
    if (!same_group(send, recv) || send == recv || send->base == recv->base)
        return SYM_ERR_INVALID_ARG;
    const int R = send->R;
    if (bytes_per_rank > send->bytes || bytes_per_rank > recv->bytes / (size_t)R)
        return SYM_ERR_INVALID_ARG;
    if (bytes_per_rank == 0) return SYM_OK;
    if (windows_overlap(send, bytes_per_rank, recv, (size_t)R * bytes_per_rank)) {
        set_last_error("sym_allgather_put_signal: send and recv windows share memory");
        return SYM_ERR_INVALID_ARG;
    }
    DeviceGuard g(recv->device);
    if (!g.ok) return SYM_ERR_CUDA;
    sym_status_t s = launch_put_signal_allgather(send, recv, bytes_per_rank, chunk_bytes,
                                                 chunks_per_signal, d_mismatch, timeout_ns,
                                                 (cudaStream_t)stream);
    if (s != SYM_OK) return s;
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_alltoall(sym_win_t send, sym_win_t recv, size_t count, sym_dtype_t dtype,
                          sym_algo_t algo, uint64_t timeout_ns, sym_stream_t stream) {
    if (!same_group(send, recv) || send == recv || send->base == recv->base)
        return SYM_ERR_INVALID_ARG;
    const size_t es = dtype_size(dtype);
    if (!es) return SYM_ERR_INVALID_ARG;
    if (algo != SYM_ALGO_AUTO && algo != SYM_ALGO_COPY && algo != SYM_ALGO_PUT_SIGNAL)
        return SYM_ERR_INVALID_ARG;
    const int R = send->R;
    if (count > send->bytes / es / (size_t)R || count > recv->bytes / es / (size_t)R)
        return SYM_ERR_INVALID_ARG;
    const bool signalled = algo == SYM_ALGO_PUT_SIGNAL;
    if (signalled && recv->nsignals < 1) return SYM_ERR_INVALID_ARG;
    if (count == 0) return SYM_OK;
    if (windows_overlap(send, (size_t)R * count * es, recv, (size_t)R * count * es)) {
        set_last_error("sym_alltoall: send and recv windows share memory");
        return SYM_ERR_INVALID_ARG;
    }
    DeviceGuard g(recv->device);
    if (!g.ok) return SYM_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    A2aArgs a{};
    a.send = send->base;
    a.recv = recv->base;
    a.sstride = send->stride;
    a.rstride = recv->stride;
    a.R = R;
    a.B = count * es;
    a.vec = a.B % 16 == 0 ? 1 : 0;
    a.status = recv->ctx->status;
    a.epoch = recv->epoch;
    a.giveup = recv->giveup;
    a.timeout_ns = timeout_ns ? std::min(timeout_ns, (uint64_t)60000000000ull) : default_timeout_ns();
    const size_t pairs = (size_t)R * R;
    // parts of about 32 KiB (one pass of block_copy) for the copy form, one
    // block each; about 128 KiB for the put + signal form, whose parts also
    // count arrivals and take a ticket (measured: 32 KiB 0.87, 64-128 KiB
    // 0.88, 256 KiB 0.85 of the copy bandwidth at R = 8 x 4 MiB segments)
    const size_t part = signalled ? (128u << 10) : (size_t)kPutThreads * kPutU * 16;
    const size_t pieces = std::max<size_t>(1, ceil_div(a.B, part));
    a.piece = ceil_div(a.B, pieces);
    if (a.vec) a.piece = ceil_div(a.piece, (size_t)16) * 16;
    a.pieces = (uint32_t)ceil_div(a.B, a.piece);
    const size_t items = pairs * a.pieces;
    if (items + R > 0x7fffffffu) return SYM_ERR_UNSUPPORTED;
    if (signalled) {
        a.sig = recv->sig;
        a.nsig = recv->nsignals;
        a.pair_done = recv->pair_arrivals;
        a.ticket = recv->ticket;
        k_reset_slot0<<<1, 64, 0, st>>>(a.sig, a.nsig, R, recv->epoch, recv->ticket);
        count_launch();
        const int occ = occupancy((const void*)k_alltoall, kPutThreads, 0);
        const size_t grid = std::min(items + R, (size_t)occ * recv->ctx->num_sms);
        void* args[] = {&a};
        // all blocks resident (cooperative launch); the ticket order alone
        // already keeps every wait on parts that running blocks hold
        SYM_CUDA(cudaLaunchCooperativeKernel((const void*)k_alltoall, dim3((unsigned)grid),
                                             dim3(kPutThreads), args, 0, st));
    } else {
        k_alltoall<<<(unsigned)items, kPutThreads, 0, st>>>(a);
    }
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_get(sym_win_t remote, sym_win_t local, int rank, int peer, size_t local_off,
                     size_t remote_off, size_t bytes, uint32_t counter_id, sym_stream_t stream) {
    if (!remote || !local || remote->device != local->device) return SYM_ERR_INVALID_ARG;
    if (rank < 0 || rank >= local->R || peer < 0 || peer >= remote->R) return SYM_ERR_INVALID_ARG;
    if (remote_off > remote->bytes || bytes > remote->bytes - remote_off) return SYM_ERR_INVALID_ARG;
    if (local_off > local->bytes || bytes > local->bytes - local_off) return SYM_ERR_INVALID_ARG;
    if (counter_id != UINT32_MAX && counter_id >= local->ncounters) return SYM_ERR_INVALID_ARG;
    const char* s = remote->base + (size_t)peer * remote->stride + remote_off;
    char* d = local->base + (size_t)rank * local->stride + local_off;
    if (bytes && s < d + bytes && d < s + bytes) return SYM_ERR_INVALID_ARG;   // overlap
    if (bytes == 0 && counter_id == UINT32_MAX) return SYM_OK;
    DeviceGuard g(local->device);
    if (!g.ok) return SYM_ERR_CUDA;
    DevCtx* ctx = local->ctx;
    // the put kernel with the roles turned round: the reader's window receives,
    // and the local action lands on the reader's counter
    PutArgs a{};
    a.src = s;
    a.dst = d;
    a.bytes = bytes;
    a.vec = ((((uintptr_t)s | (uintptr_t)d | bytes) & 15u) == 0) ? 1 : 0;
    a.sig = nullptr;
    a.cnt = counter_id != UINT32_MAX ? local->cnt + (size_t)rank * local->ncounters + counter_id
                                     : nullptr;
    a.arrive = ctx->arrive + (ctx->arrive_next.fetch_add(1, std::memory_order_relaxed) % kArriveRing);
    const size_t per_cta = 64 * 1024;
    const size_t grid = std::max((size_t)1, std::min(ceil_div(bytes, per_cta),
                                                     (size_t)ctx->num_sms * 4));
    k_put<<<(unsigned)grid, kPutThreads, 0, (cudaStream_t)stream>>>(a);
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_put_signal(sym_win_t src, sym_win_t dst, int src_rank, int peer, size_t dst_off,
                            size_t src_off, size_t bytes, uint32_t signal_id, uint32_t counter_id,
                            sym_stream_t stream) {
    if (!src || !dst || src->device != dst->device) return SYM_ERR_INVALID_ARG;
    if (src_rank < 0 || src_rank >= src->R || peer < 0 || peer >= dst->R) return SYM_ERR_INVALID_ARG;
    if (src_off > src->bytes || bytes > src->bytes - src_off) return SYM_ERR_INVALID_ARG;
    if (dst_off > dst->bytes || bytes > dst->bytes - dst_off) return SYM_ERR_INVALID_ARG;
    if (signal_id != UINT32_MAX && signal_id >= dst->nsignals) return SYM_ERR_INVALID_ARG;
    if (counter_id != UINT32_MAX && counter_id >= src->ncounters) return SYM_ERR_INVALID_ARG;
    const char* s = src->base + (size_t)src_rank * src->stride + src_off;
    char* d = dst->base + (size_t)peer * dst->stride + dst_off;
    if (bytes && s < d + bytes && d < s + bytes) return SYM_ERR_INVALID_ARG;   // overlap
    DeviceGuard g(dst->device);
    if (!g.ok) return SYM_ERR_CUDA;
    DevCtx* ctx = dst->ctx;
    PutArgs a{};
    a.src = s;
    a.dst = d;
    a.bytes = bytes;
    a.vec = ((((uintptr_t)s | (uintptr_t)d | bytes) & 15u) == 0) ? 1 : 0;
    a.sig = signal_id != UINT32_MAX ? dst->sig + (size_t)peer * dst->nsignals + signal_id : nullptr;
    a.cnt = counter_id != UINT32_MAX ? src->cnt + (size_t)src_rank * src->ncounters + counter_id
                                     : nullptr;
    a.arrive = ctx->arrive + (ctx->arrive_next.fetch_add(1, std::memory_order_relaxed) % kArriveRing);
    const size_t per_cta = 64 * 1024;
    const size_t grid = std::max((size_t)1, std::min(ceil_div(bytes, per_cta),
                                                     (size_t)ctx->num_sms * 4));
    k_put<<<(unsigned)grid, kPutThreads, 0, (cudaStream_t)stream>>>(a);
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

// [GIN] ncclGinBarrierSession::sync, signal form: one block per rank r reads
// its slot (before adding anything), adds 1 to slot `id` of every rank with a
// release, then waits (acquire, bounded) until its own slot has gained all R
// adds of this barrier.  Each barrier adds exactly R to every slot, so the
// target is the next multiple of R above the value read first.
__global__ void __launch_bounds__(kMaxRanks) k_barrier(uint64_t* sig, uint32_t nsig, uint32_t id,
                                                       int R, uint64_t timeout_ns, uint32_t* status) {
    __shared__ uint64_t s_target;
    const uint32_t r = blockIdx.x;
    uint64_t* mine = sig + (size_t)r * nsig + id;
    if (threadIdx.x == 0) s_target = (ld_acquire_u64(mine) / (uint64_t)R + 1) * (uint64_t)R;
    __syncthreads();
    if (threadIdx.x < (uint32_t)R) {
        __threadfence();
        red_release_add_u64(sig + (size_t)threadIdx.x * nsig + id, 1ull);
    }
    if (threadIdx.x == 0) {
        const uint64_t target = s_target;
        if (!bounded_spin([&] { return ld_acquire_u64(mine) >= target; }, timeout_ns, nullptr, 0u))
            report_timeout(status, nullptr, 0u, kSiteBarrier, r, id);
    }
}

sym_status_t sym_barrier(sym_win_t w, uint32_t signal_id, uint64_t timeout_ns, sym_stream_t stream) {
    if (!w || signal_id >= w->nsignals) return SYM_ERR_INVALID_ARG;
    if (timeout_ns == 0) timeout_ns = default_timeout_ns();
    if (timeout_ns > 60000000000ull) timeout_ns = 60000000000ull;
    DeviceGuard g(w->device);
    if (!g.ok) return SYM_ERR_CUDA;
    uint64_t* sig = w->sig;
    uint32_t nsig = w->nsignals, id = signal_id;
    int R = w->R;
    uint32_t* status = w->ctx->status;
    void* args[] = {&sig, &nsig, &id, &R, &timeout_ns, &status};
    // ranks wait on one another -> co-resident blocks
    SYM_CUDA(cudaLaunchCooperativeKernel((const void*)k_barrier, dim3((unsigned)R), dim3(kMaxRanks),
                                         args, 0, (cudaStream_t)stream));
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_signal(sym_win_t dst, int peer, uint32_t signal_id, uint64_t value,
                        sym_stream_t stream) {
    if (!dst || peer < 0 || peer >= dst->R || signal_id >= dst->nsignals) return SYM_ERR_INVALID_ARG;
    DeviceGuard g(dst->device);
    k_signal_add<<<1, 1, 0, (cudaStream_t)stream>>>(
        dst->sig + (size_t)peer * dst->nsignals + signal_id, value);
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

static sym_status_t wait_slot(sym_win_t w, const uint64_t* slot, uint64_t least, int bits,
                              uint64_t timeout_ns, uint32_t site, uint32_t a, uint32_t b,
                              sym_stream_t stream) {
    if (timeout_ns == 0) timeout_ns = default_timeout_ns();
    if (timeout_ns > 60000000000ull) timeout_ns = 60000000000ull;
    DeviceGuard g(w->device);
    k_wait_slot<<<1, 32, 0, (cudaStream_t)stream>>>(slot, least, bits, timeout_ns, w->ctx->status,
                                                    site, a, b);
    count_launch();
    SYM_CUDA(cudaGetLastError());
    return SYM_OK;
}

sym_status_t sym_signal_wait(sym_win_t w, int rank, uint32_t signal_id, uint64_t least, int bits,
                             uint64_t timeout_ns, sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || signal_id >= w->nsignals) return SYM_ERR_INVALID_ARG;
    if (bits < 1 || bits > 64) return SYM_ERR_INVALID_ARG;
    return wait_slot(w, w->sig + (size_t)rank * w->nsignals + signal_id, least, bits, timeout_ns,
                     kSiteSignalWait, (uint32_t)rank, signal_id, stream);
}

sym_status_t sym_counter_wait(sym_win_t w, int rank, uint32_t counter_id, uint64_t least, int bits,
                              uint64_t timeout_ns, sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || counter_id >= w->ncounters) return SYM_ERR_INVALID_ARG;
    if (bits < 1 || bits > 56) return SYM_ERR_INVALID_ARG;
    return wait_slot(w, w->cnt + (size_t)rank * w->ncounters + counter_id, least, bits, timeout_ns,
                     kSiteCounterWait, (uint32_t)rank, counter_id, stream);
}

static sym_status_t read_slot(sym_win_t w, const uint64_t* slot, int bits, uint64_t* out,
                              sym_stream_t stream) {
    DeviceGuard g(w->device);
    uint64_t v = 0;
    SYM_CUDA(cudaMemcpyAsync(&v, slot, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
    SYM_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    *out = bits >= 64 ? v : (v & ((1ull << bits) - 1ull));
    return SYM_OK;
}

sym_status_t sym_signal_read(sym_win_t w, int rank, uint32_t signal_id, int bits, uint64_t* out,
                             sym_stream_t stream) {
    if (!w || !out || rank < 0 || rank >= w->R || signal_id >= w->nsignals) return SYM_ERR_INVALID_ARG;
    if (bits < 1 || bits > 64) return SYM_ERR_INVALID_ARG;
    return read_slot(w, w->sig + (size_t)rank * w->nsignals + signal_id, bits, out, stream);
}

sym_status_t sym_counter_read(sym_win_t w, int rank, uint32_t counter_id, int bits, uint64_t* out,
                              sym_stream_t stream) {
    if (!w || !out || rank < 0 || rank >= w->R || counter_id >= w->ncounters)
        return SYM_ERR_INVALID_ARG;
    if (bits < 1 || bits > 56) return SYM_ERR_INVALID_ARG;
    return read_slot(w, w->cnt + (size_t)rank * w->ncounters + counter_id, bits, out, stream);
}

sym_status_t sym_signal_reset(sym_win_t w, int rank, uint32_t signal_id, sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || signal_id >= w->nsignals) return SYM_ERR_INVALID_ARG;
    DeviceGuard g(w->device);
    SYM_CUDA(cudaMemsetAsync(w->sig + (size_t)rank * w->nsignals + signal_id, 0, sizeof(uint64_t),
                             (cudaStream_t)stream));
    return SYM_OK;
}

sym_status_t sym_counter_reset(sym_win_t w, int rank, uint32_t counter_id, sym_stream_t stream) {
    if (!w || rank < 0 || rank >= w->R || counter_id >= w->ncounters) return SYM_ERR_INVALID_ARG;
    DeviceGuard g(w->device);
    SYM_CUDA(cudaMemsetAsync(w->cnt + (size_t)rank * w->ncounters + counter_id, 0, sizeof(uint64_t),
                             (cudaStream_t)stream));
    return SYM_OK;
}

}  // extern "C"
