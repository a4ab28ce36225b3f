/*
 * CPU oracle for symmetric-window collectives.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg may load this library.  The product path (the CUDA library under
 * symmetric_memory_allreduce_gb300/) never calls it and shares no code with it.
 *
 * Every routine is the plain definition of what the method computes, written
 * out element by element, with no blocking, fusion or reordering.  Build with
 * -O2 -ffp-contract=off -fno-fast-math so that the compiler keeps IEEE binary32
 * round-to-nearest-even adds in source order (on aarch64 GCC would otherwise be
 * allowed to contract).
 *
 * Sources (web pages; cited by title and section):
 *  [SYMEX]  "NCCL symmetric memory windows: examples 01_allreduce / 02_allgather"
 *           (docs/examples/05_symmetric_memory walkthrough), Example 1 steps 4-6
 *           and expected output; Example 2 buffers and expected output.
 *  [GIN]    "NCCL Device API GIN reference": sections "put/get", "Signals and
 *           Counters", "Signal methods", "Counter methods".
 *  [GDA]    "GPUDirect Async deep dive" (GIN paper summary, section 4: ordering
 *           of a batch of puts followed by one signal; section 5.3: batches of
 *           at most 8 commands with one signalled request per batch).
 *
 * Parity status of each function is stated in its comment.  Every function is
 * pinned by tests/test_oracle.py to facts that do not come from this file.
 * oracle_rolling_le, whose formula the page names without printing, is pinned
 * to RFC 1982 serial number arithmetic (the published definition of such a
 * comparison) and to the page's stated property (see its comment).
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>

/* ------------------------------------------------------------------------ */
/* AllReduce(sum), fp32.                                                    */
/* [SYMEX] Example 1: every rank calls AllReduce(send, recv, count, float,  */
/* sum); step 6 says each element equals the sum over all ranks.  The pages */
/* do not fix an order; this oracle adds in rank order 0..R-1, one IEEE     */
/* binary32 add at a time:                                                  */
/*     y[i] = ((x[0][i] + x[1][i]) + x[2][i]) + ... + x[R-1][i]             */
/* Every rank's recv buffer holds the same y.                               */
/* x is R rows of ldx elements (row q = rank q's send buffer).              */
/* Pins: rank-fill closed form R(R-1)/2; integer-valued data (exact in any  */
/* order); brute force vs numpy float32 scalar adds; Higham error bound.    */
/* ------------------------------------------------------------------------ */
void oracle_allreduce_sum_f32(int R, size_t n, const float* x, size_t ldx, float* y)
{
    for (size_t i = 0; i < n; ++i) {
        float acc = x[i];
        for (int q = 1; q < R; ++q) {
            acc = acc + x[(size_t)q * ldx + i];
        }
        y[i] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32.                                                           */
/* bf16 is the top half of a binary32 pattern, so widening is exact:        */
/*     bits32 = bits16 << 16.                                               */
/* Narrowing rounds to nearest, ties to even (IEEE 754 roundTiesToEven),    */
/* keeping Inf and mapping every NaN to the quiet NaN 0x7FC0.  With u the   */
/* binary32 pattern, the kept half is u >> 16 and the dropped half is       */
/* u & 0xFFFF; round up when the dropped half exceeds 0x8000, or equals it  */
/* and the kept half is odd.  Adding 0x7FFF + (kept & 1) and shifting does  */
/* exactly that, and a carry out of the mantissa correctly bumps the        */
/* exponent (up to Inf for the largest finite values).                      */
/* Pins: torch CPU conversion on stratified patterns; brute-force nearest   */
/* neighbour in exact rationals; hand tie cases.                            */
/* ------------------------------------------------------------------------ */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) {
        return (uint16_t)0x7FC0u;                /* NaN */
    }
    uint32_t kept_lsb = (u >> 16) & 1u;
    uint32_t r = u + 0x7FFFu + kept_lsb;
    return (uint16_t)(r >> 16);
}

void oracle_f32_to_bf16_array(size_t n, const float* x, uint16_t* y)
{
    for (size_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------ */
/* AllReduce(sum), bf16 inputs, fp32 accumulation, one rounding.            */
/* Each input is widened exactly, the fp32 sum is taken in rank order as in */
/* the fp32 routine, and the result is rounded to bf16 once.                */
/* Pins: numpy float32 rank-order loop + torch rounding; rank-fill.         */
/* ------------------------------------------------------------------------ */
void oracle_allreduce_sum_bf16(int R, size_t n, const uint16_t* x, size_t ldx, uint16_t* y)
{
    for (size_t i = 0; i < n; ++i) {
        float acc = oracle_bf16_to_f32(x[i]);
        for (int q = 1; q < R; ++q) {
            acc = acc + oracle_bf16_to_f32(x[(size_t)q * ldx + i]);
        }
        y[i] = oracle_f32_to_bf16_rne(acc);
    }
}

/* ------------------------------------------------------------------------ */
/* fp16 (IEEE binary16) <-> fp32.                                           */
/* Widening is exact.  Narrowing rounds to nearest, ties to even, with      */
/* gradual underflow: below 2^-14 the result is a multiple of 2^-24; values */
/* of magnitude >= 65520 (half-way between the largest half, 65504, and     */
/* 2^16) round to Inf; every NaN becomes the quiet NaN 0x7E00.              */
/* Pins: numpy's float32->float16 conversion on stratified patterns; exact  */
/* rational nearest-neighbour brute force; hand cases.                      */
/* ------------------------------------------------------------------------ */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu, u;
    if (e == 0x1Fu) {
        u = sign | 0x7F800000u | (m << 13);              /* Inf / NaN */
    } else if (e != 0) {
        u = sign | ((e + 112u) << 23) | (m << 13);       /* 112 = 127 - 15 */
    } else if (m == 0) {
        u = sign;                                         /* +-0 */
    } else {                                              /* subnormal: m * 2^-24 */
        int k = 0;
        while ((m & 0x400u) == 0) { m <<= 1; ++k; }
        u = sign | ((uint32_t)(113 - k) << 23) | ((m & 0x3FFu) << 13);
    }
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_f16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)0x7E00u;       /* NaN */
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);   /* >= 65520 or Inf */
    int e = (int)(a >> 23) - 127;
    uint32_t m = a & 0x7FFFFFu;
    if (e >= -14) {                                       /* normal half */
        uint32_t h = ((uint32_t)(e + 15) << 10) | (m >> 13);
        uint32_t rem = m & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    /* below the normal range: count units of 2^-24, round to nearest even */
    if ((a >> 23) == 0) return sign;                      /* fp32 subnormal: < 2^-126 */
    uint64_t M = (uint64_t)(m | 0x800000u);               /* value = M * 2^(e-23) */
    int s = -(e + 1);                                     /* units of 2^-24: M >> s */
    if (s >= 40) return sign;
    uint64_t q = M >> s, rem = M & (((uint64_t)1 << s) - 1), halfway = (uint64_t)1 << (s - 1);
    if (rem > halfway || (rem == halfway && (q & 1u))) q += 1u;
    return (uint16_t)(sign | (uint16_t)q);
}

void oracle_f32_to_f16_array(size_t n, const float* x, uint16_t* y)
{
    for (size_t i = 0; i < n; ++i) y[i] = oracle_f32_to_f16_rne(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Reduction operators.                                                     */
/* sum: IEEE binary32 add (round to nearest even).                          */
/* max / min: IEEE 754-2019 maximumNumber / minimumNumber -- a NaN operand  */
/* is ignored (NaN only if both are NaN), and -0 < +0.                      */
/* The reduction over ranks is always a left fold in rank order 0..R-1.     */
/* Pins: numpy fmax/fmin reductions on data without signed zeros; hand     */
/* cases for the zero signs and NaN.                                        */
/* ------------------------------------------------------------------------ */
enum { ORACLE_SUM = 0, ORACLE_MAX = 1, ORACLE_MIN = 2 };
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

static int is_nan_f(float v) { return v != v; }
static int sign_bit_f(float v) { uint32_t u; memcpy(&u, &v, sizeof u); return (int)(u >> 31); }

float oracle_apply_op(int op, float a, float b)
{
    if (op == ORACLE_SUM) return a + b;
    if (is_nan_f(a)) return b;
    if (is_nan_f(b)) return a;
    if (op == ORACLE_MAX) {
        if (a > b) return a;
        if (b > a) return b;
        return sign_bit_f(a) ? b : a;                    /* equal: prefer +0 */
    }
    if (a < b) return a;
    if (b < a) return b;
    return sign_bit_f(a) ? a : b;                        /* equal: prefer -0 */
}

static float load_as_f32(int dtype, const void* x, size_t i)
{
    if (dtype == ORACLE_F32) return ((const float*)x)[i];
    if (dtype == ORACLE_BF16) return oracle_bf16_to_f32(((const uint16_t*)x)[i]);
    return oracle_f16_to_f32(((const uint16_t*)x)[i]);
}

static void store_from_f32(int dtype, void* y, size_t i, float v)
{
    if (dtype == ORACLE_F32) ((float*)y)[i] = v;
    else if (dtype == ORACLE_BF16) ((uint16_t*)y)[i] = oracle_f32_to_bf16_rne(v);
    else ((uint16_t*)y)[i] = oracle_f32_to_f16_rne(v);
}

/* AllReduce with any supported (dtype, op): widen exactly, fold in rank     */
/* order in fp32, narrow once.  For (F32, SUM) and (BF16, SUM) this is the   */
/* same arithmetic as the dedicated routines above.                          */
void oracle_allreduce(int dtype, int op, int R, size_t n, const void* x, size_t ldx, void* y)
{
    for (size_t i = 0; i < n; ++i) {
        float acc = load_as_f32(dtype, x, i);
        for (int q = 1; q < R; ++q) {
            acc = oracle_apply_op(op, acc, load_as_f32(dtype, x, (size_t)q * ldx + i));
        }
        store_from_f32(dtype, y, i, acc);
    }
}

/* ------------------------------------------------------------------------ */
/* Producer + AllReduce.                                                    */
/* [GDA] section 5.1: compute tiles produce each rank's contribution, and   */
/* the AllReduce consumes it.  The producer here is one binary32 multiply   */
/* per element, rounded to nearest:                                         */
/*     s_r[i] = alpha_r * a_r[i]                                            */
/* and the consumer is the fp32 AllReduce in rank order:                    */
/*     y[i] = ((s_0[i] + s_1[i]) + ...) + s_{R-1}[i].                       */
/* s: R rows of lds floats (the contributions), y: n floats.                */
/* Pins: alpha = 1 gives the plain AllReduce; rank fill with alpha_r = r+1  */
/* gives the closed form sum r(r+1); numpy float32 brute force.             */
/* ------------------------------------------------------------------------ */
void oracle_scale_allreduce(int R, size_t n, const float* alpha, const float* a, size_t lda,
                            float* s, size_t lds, float* y)
{
    for (int q = 0; q < R; ++q) {
        for (size_t i = 0; i < n; ++i) {
            s[(size_t)q * lds + i] = alpha[q] * a[(size_t)q * lda + i];
        }
    }
    oracle_allreduce_sum_f32(R, n, s, lds, y);
}

/* ------------------------------------------------------------------------ */
/* Threaded drivers (timing only).  The element range is split into equal   */
/* contiguous parts, each handled by the same per-element routine above, so */
/* results are identical to the single-threaded call.                       */
/* ------------------------------------------------------------------------ */
typedef struct {
    int R, is_bf16;
    size_t lo, hi, ldx;
    const void* x;
    void* y;
} oracle_job;

static void* oracle_job_run(void* arg)
{
    oracle_job* j = (oracle_job*)arg;
    size_t n = j->hi - j->lo;
    if (j->is_bf16) {
        oracle_allreduce_sum_bf16(j->R, n, (const uint16_t*)j->x + j->lo, j->ldx,
                                  (uint16_t*)j->y + j->lo);
    } else {
        oracle_allreduce_sum_f32(j->R, n, (const float*)j->x + j->lo, j->ldx,
                                 (float*)j->y + j->lo);
    }
    return NULL;
}

/* Returns the number of threads actually used. */
int oracle_allreduce_sum_mt(int is_bf16, int R, size_t n, const void* x, size_t ldx,
                            void* y, int nthreads)
{
    enum { MAXT = 256 };
    if (nthreads < 1) nthreads = 1;
    if (nthreads > MAXT) nthreads = MAXT;
    if ((size_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
    pthread_t th[MAXT];
    oracle_job jobs[MAXT];
    size_t per = (n + (size_t)nthreads - 1) / (size_t)nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo > n) lo = n;
        if (hi > n) hi = n;
        jobs[t] = (oracle_job){R, is_bf16, lo, hi, ldx, x, y};
        if (t == 0) continue;
        if (pthread_create(&th[t], NULL, oracle_job_run, &jobs[t]) != 0) {
            oracle_job_run(&jobs[t]);           /* run inline if no thread */
            th[t] = (pthread_t)0;
        } else {
            ++started;
        }
    }
    oracle_job_run(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (th[t] != (pthread_t)0) pthread_join(th[t], NULL);
    }
    return started + 1;
}

/* ------------------------------------------------------------------------ */
/* AllGather.                                                               */
/* [SYMEX] Example 2: the recv buffer holds sendcount * nranks elements and */
/* segment q holds rank q's send buffer:                                    */
/*     recv_r[q*S + i] = send_q[i]   for every rank r, q and byte i < S.    */
/* The result does not depend on r, so one buffer of R*S bytes is produced. */
/* Pins: worked example (segment q = float(q)); numpy concatenation.        */
/* ------------------------------------------------------------------------ */
void oracle_allgather(int R, size_t S, const uint8_t* x, size_t ldx, uint8_t* y)
{
    for (int q = 0; q < R; ++q) {
        for (size_t i = 0; i < S; ++i) {
            y[(size_t)q * S + i] = x[(size_t)q * ldx + i];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* AlltoAll.                                                                */
/* [GIN] "pure GIN AlltoAll" example: every rank puts count elements to     */
/* every rank r, taking them from its send buffer at r*count and placing    */
/* them in r's receive buffer at my_rank*count; one signal increment per    */
/* arriving put, the receiver waits for nRanks of them.  In bytes, with     */
/* B = count*sizeof(T) per segment:                                         */
/*     recv_p[q*B + i] = send_q[p*B + i]   for all ranks p, q and i < B.    */
/* x: R rows of ldx bytes; y: R rows of ldy bytes.                          */
/* Pins: the page's pattern my_rank*1000 + dest_rank*100 + element_idx;     */
/* numpy transpose of the (sender, receiver) segment grid.                  */
/* ------------------------------------------------------------------------ */
void oracle_alltoall(int R, size_t B, const uint8_t* x, size_t ldx, uint8_t* y, size_t ldy)
{
    for (int p = 0; p < R; ++p) {
        for (int q = 0; q < R; ++q) {
            for (size_t i = 0; i < B; ++i) {
                y[(size_t)p * ldy + (size_t)q * B + i] = x[(size_t)q * ldx + (size_t)p * B + i];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Chunked put + signal AllGather, sequential model.                        */
/* [GIN] put: copy `bytes` from the source window at src_off to the peer's  */
/* destination window at dst_off; the peer may be the caller (loopback).    */
/* remoteAction SignalInc adds 1 to a signal on the peer; localAction       */
/* CounterInc adds 1 to a counter on the caller once the source is read.    */
/* [GDA] a batch of puts followed by one signal orders the batch.           */
/* Model: for every sender q, every peer p (p = q included) and chunk k in  */
/* ascending order, put chunk k of send_q to recv_p at q*S + k*chunk; after */
/* each put, cnt[q] += 1; after every B-th chunk of a (q, p) stream and     */
/* after its last chunk, sig[p*R + q] += 1 (signal id = sender rank).       */
/* The last chunk may be short when chunk does not divide S.                */
/* Outputs: recv (R*S bytes, identical for every p, so one buffer),         */
/* sig (R*R), cnt (R).  The caller zeroes nothing; this routine does.       */
/* Pins: closed forms sig = ceil(ceil(S/chunk)/B), cnt = R*ceil(S/chunk);   */
/* recv equals the AllGather; prefix-visibility replay below.               */
/* ------------------------------------------------------------------------ */
void oracle_put_signal_allgather(int R, size_t S, size_t chunk, size_t B,
                                 const uint8_t* x, size_t ldx,
                                 uint8_t* recv, uint64_t* sig, uint64_t* cnt)
{
    memset(sig, 0, sizeof(uint64_t) * (size_t)R * (size_t)R);
    memset(cnt, 0, sizeof(uint64_t) * (size_t)R);
    size_t nchunks = (S + chunk - 1) / chunk;
    for (int q = 0; q < R; ++q) {
        for (int p = 0; p < R; ++p) {
            size_t in_batch = 0;
            for (size_t k = 0; k < nchunks; ++k) {
                size_t off = k * chunk;
                size_t len = (off + chunk <= S) ? chunk : S - off;
                /* recv is shared by all p (the result does not depend on p);
                 * every p writes the same bytes to the same place. */
                memcpy(recv + (size_t)q * S + off, x + (size_t)q * ldx + off, len);
                cnt[q] += 1;
                in_batch += 1;
                if (in_batch == B || k + 1 == nchunks) {
                    sig[(size_t)p * R + q] += 1;
                    in_batch = 0;
                }
            }
        }
    }
}

/* Prefix visibility, the strong-signal invariant of [GIN] "Signals and      */
/* Counters" (a visible strong signal implies every earlier put on the same  */
/* context to the same peer is visible): given a snapshot of recv_p's        */
/* segment q and an observed signal value k, return the number of bytes of  */
/* batches 0..k-1 (chunks 0..k*B-1) that differ from the source.  The        */
/* expected answer for a correct implementation is 0.                        */
uint64_t oracle_prefix_mismatch(size_t S, size_t chunk, size_t B, uint64_t k,
                                const uint8_t* src_q, const uint8_t* seg)
{
    size_t covered = (size_t)k * B * chunk;
    if (covered > S) covered = S;
    uint64_t bad = 0;
    for (size_t i = 0; i < covered; ++i) bad += (src_q[i] != seg[i]);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Rolling comparison.                                                      */
/* [GIN] "Signals and Counters": signal and counter values are compared     */
/* with a rolling rule so that x <= x+1 holds even across unsigned          */
/* overflow; waitSignal(least, bits) returns once the low `bits` bits of    */
/* the value are rolling-greater-or-equal to `least`.  The page names the   */
/* routine without printing it.  Reading taken: with m = 2^bits - 1 and     */
/* d = (b - a) mod 2^bits, a <= b iff d < 2^(bits-1), i.e. b is one of the  */
/* 2^(bits-1) values a, a+1, ... (mod 2^bits).                              */
/* Pins: RFC 1982 (Serial Number Arithmetic) "less than" in its case form,  */
/* exhaustively for 1..10 bits, with the pair exactly 2^(bits-1) apart      */
/* (undefined there) read as "not reached"; the page's x <= x+1 for every   */
/* x; integer <= where nothing wraps; 56/63/64-bit edges with high bits.    */
/* ------------------------------------------------------------------------ */
int oracle_rolling_le(uint64_t a, uint64_t b, int bits)
{
    if (bits < 1) bits = 1;
    if (bits > 64) bits = 64;
    uint64_t m = (bits == 64) ? ~(uint64_t)0 : (((uint64_t)1 << bits) - 1);
    uint64_t d = (b - a) & m;
    uint64_t half = (uint64_t)1 << (bits - 1);
    return d < half;
}

/* readSignal / readCounter: the low `bits` bits of the value. */
uint64_t oracle_read_bits(uint64_t v, int bits)
{
    if (bits >= 64) return v;
    if (bits < 1) return 0;
    return v & (((uint64_t)1 << bits) - 1);
}
