/*
 * A plain C caller of libsymar.so (no Python, no CUDA headers): allocates
 * windows, fills them from host buffers, runs sym_allreduce with every
 * algorithm and sym_allgather, reads the results back and compares them byte
 * for byte with the CPU oracle (liboracle.so, test infrastructure).  The
 * stream argument is NULL (the legacy default stream), so the program needs
 * only the library's own header.  Prints "C_ABI_PARITY_OK" and exits 0 when
 * every result matches.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "symar.h"

/* the oracle's entry points (oracle/oracle.c) */
void oracle_allreduce_sum_f32(int R, size_t n, const float* x, size_t ldx, float* y);
void oracle_allgather(int R, size_t S, const uint8_t* x, size_t ldx, uint8_t* y);

#define CHECK(call)                                                                   \
    do {                                                                              \
        sym_status_t s_ = (call);                                                     \
        if (s_ != SYM_OK) {                                                           \
            fprintf(stderr, "%s -> %s (%s)\n", #call, sym_status_string(s_),          \
                    sym_last_error());                                                \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

static uint64_t g_state = 20261202u;
static uint32_t next_u32(void) {          /* xorshift64*: seeded test data only */
    g_state ^= g_state >> 12;
    g_state ^= g_state << 25;
    g_state ^= g_state >> 27;
    return (uint32_t)((g_state * 2685821657736338717ull) >> 32);
}

static int allreduce_case(int R, size_t n) {
    const size_t bytes = n * sizeof(float);
    float* x = malloc((size_t)R * bytes);
    float* want = malloc(bytes);
    float* got = malloc(bytes);
    if (!x || !want || !got) return 1;
    for (size_t i = 0; i < (size_t)R * n; ++i)
        x[i] = (float)((int32_t)(next_u32() % 2000001u) - 1000000) / 65536.0f;
    oracle_allreduce_sum_f32(R, n, x, n, want);
    sym_win_t send, recv;
    CHECK(sym_window_alloc(R, bytes, 0, 0, &send));
    CHECK(sym_window_alloc(R, bytes, 0, 0, &recv));
    for (int r = 0; r < R; ++r) CHECK(sym_window_write(send, r, 0, x + (size_t)r * n, bytes, NULL));
    const sym_algo_t algos[] = {SYM_ALGO_AUTO, SYM_ALGO_ONESHOT, SYM_ALGO_TWOSHOT, SYM_ALGO_TWOSHOT_PULL,
                                SYM_ALGO_TWOSHOT_SPLIT};
    for (size_t k = 0; k < sizeof algos / sizeof algos[0]; ++k) {
        CHECK(sym_allreduce(send, recv, n, SYM_F32, SYM_SUM, algos[k], NULL));
        CHECK(sym_stream_status(NULL));
        for (int r = 0; r < R; ++r) {
            memset(got, 0xAB, bytes);
            CHECK(sym_window_read(recv, r, 0, got, bytes, NULL));
            CHECK(sym_stream_status(NULL));
            if (memcmp(got, want, bytes) != 0) {
                fprintf(stderr, "allreduce R=%d n=%zu algo=%d rank %d differs\n", R, n, (int)algos[k], r);
                return 1;
            }
        }
    }
    CHECK(sym_window_free(send));
    CHECK(sym_window_free(recv));
    free(x);
    free(want);
    free(got);
    return 0;
}

static int allgather_case(int R, size_t S) {
    uint8_t* x = malloc((size_t)R * S);
    uint8_t* want = malloc((size_t)R * S);
    uint8_t* got = malloc((size_t)R * S);
    if (!x || !want || !got) return 1;
    for (size_t i = 0; i < (size_t)R * S; ++i) x[i] = (uint8_t)next_u32();
    oracle_allgather(R, S, x, S, want);
    sym_win_t send, recv;
    CHECK(sym_window_alloc(R, S, 0, 1, &send));
    CHECK(sym_window_alloc(R, (size_t)R * S, (uint32_t)R, 0, &recv));
    for (int r = 0; r < R; ++r) CHECK(sym_window_write(send, r, 0, x + (size_t)r * S, S, NULL));
    const sym_algo_t algos[] = {SYM_ALGO_COPY, SYM_ALGO_CE, SYM_ALGO_PUT_SIGNAL};
    for (size_t k = 0; k < sizeof algos / sizeof algos[0]; ++k) {
        CHECK(sym_allgather(send, recv, S / 4, SYM_F32, algos[k], 0, 0, NULL));
        CHECK(sym_stream_status(NULL));
        for (int r = 0; r < R; ++r) {
            CHECK(sym_window_read(recv, r, 0, got, (size_t)R * S, NULL));
            CHECK(sym_stream_status(NULL));
            if (memcmp(got, want, (size_t)R * S) != 0) {
                fprintf(stderr, "allgather R=%d S=%zu algo=%d rank %d differs\n", R, S, (int)algos[k], r);
                return 1;
            }
        }
    }
    CHECK(sym_window_free(send));
    CHECK(sym_window_free(recv));
    free(x);
    free(want);
    free(got);
    return 0;
}

int main(void) {
    if (sym_abi_version() != SYMAR_ABI_VERSION) {
        fprintf(stderr, "ABI %d, header %d\n", sym_abi_version(), SYMAR_ABI_VERSION);
        return 1;
    }
    const int ranks[] = {1, 3, 8};
    const size_t sizes[] = {1, 1000, 65539, 300007};
    for (size_t i = 0; i < 3; ++i)
        for (size_t j = 0; j < 4; ++j)
            if (allreduce_case(ranks[i], sizes[j])) return 1;
    if (allgather_case(4, 3 * 16384 + 512)) return 1;
    if (allgather_case(8, 1 << 20)) return 1;
    printf("C_ABI_PARITY_OK launches=%llu\n", (unsigned long long)sym_launch_count());
    return 0;
}
