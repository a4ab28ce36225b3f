// symar_bench: a native benchmark of the C ABI, with no Python or torch.
//
//   symar_bench [--ranks R] [--bytes B] [--algo auto|oneshot|twoshot|twoshot_pull|twoshot_split]
//               [--dtype f32|bf16|f16] [--iters N] [--warmup W] [--vmm]
//
// Allocates two windows of R x B bytes (sym_window_alloc, or sym_window_alloc_vmm with --vmm),
// fills the inputs with a fixed byte pattern from the host (sym_window_write), runs W untimed
// and N timed sym_allreduce calls on one stream, each timed with CUDA events, and prints one
// JSON line: median / p10 / p90 microseconds per call, algorithm bandwidth (B / time) and the
// compulsory-byte rate (2 R B / time).  As a sanity check it compares the results of ranks 0
// and R-1 byte for byte (every rank must hold the same reduction).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/symar.h"

namespace {

int fail(const char* what, sym_status_t s) {
    fprintf(stderr, "symar_bench: %s: %s (%s)\n", what, sym_status_string(s), sym_last_error());
    return 1;
}

bool parse_algo(const std::string& s, sym_algo_t* out) {
    static const struct { const char* name; sym_algo_t algo; } kAlgos[] = {
        {"auto", SYM_ALGO_AUTO},
        {"oneshot", SYM_ALGO_ONESHOT},
        {"twoshot", SYM_ALGO_TWOSHOT},
        {"twoshot_pull", SYM_ALGO_TWOSHOT_PULL},
        {"twoshot_split", SYM_ALGO_TWOSHOT_SPLIT},
    };
    for (const auto& a : kAlgos)
        if (s == a.name) {
            *out = a.algo;
            return true;
        }
    return false;
}

bool parse_dtype(const std::string& s, sym_dtype_t* out, size_t* size) {
    if (s == "f32") *out = SYM_F32, *size = 4;
    else if (s == "bf16") *out = SYM_BF16, *size = 2;
    else if (s == "f16") *out = SYM_F16, *size = 2;
    else return false;
    return true;
}

double pct(std::vector<float> v, double q) {
    std::sort(v.begin(), v.end());
    const double k = (v.size() - 1) * q;
    const size_t lo = (size_t)k, hi = std::min(lo + 1, v.size() - 1);
    return v[lo] + (v[hi] - v[lo]) * (k - (double)lo);
}

}  // namespace

int main(int argc, char** argv) {
    int R = 8, iters = 200, warmup = 5;
    size_t bytes = 256ull << 20;
    std::string algo_name = "twoshot", dtype_name = "f32";
    bool vmm = false;
    for (int i = 1; i < argc; ++i) {
        const std::string a = argv[i];
        auto next = [&]() -> const char* {
            if (i + 1 >= argc) {
                fprintf(stderr, "symar_bench: %s needs a value\n", a.c_str());
                exit(2);
            }
            return argv[++i];
        };
        if (a == "--ranks") R = atoi(next());
        else if (a == "--bytes") bytes = strtoull(next(), nullptr, 0);
        else if (a == "--algo") algo_name = next();
        else if (a == "--dtype") dtype_name = next();
        else if (a == "--iters") iters = atoi(next());
        else if (a == "--warmup") warmup = atoi(next());
        else if (a == "--vmm") vmm = true;
        else {
            fprintf(stderr, "usage: symar_bench [--ranks R] [--bytes B] [--algo A] [--dtype D] "
                            "[--iters N] [--warmup W] [--vmm]\n");
            return 2;
        }
    }
    sym_algo_t algo;
    sym_dtype_t dtype;
    size_t es = 0;
    if (!parse_algo(algo_name, &algo) || !parse_dtype(dtype_name, &dtype, &es) || R < 1 || iters < 1 ||
        warmup < 0 || bytes < es) {
        fprintf(stderr, "symar_bench: bad arguments\n");
        return 2;
    }
    const size_t count = bytes / es;
    bytes = count * es;

    cudaStream_t st;
    if (cudaStreamCreate(&st) != cudaSuccess) return fail("cudaStreamCreate", SYM_ERR_CUDA);
    sym_win_t send = nullptr, recv = nullptr;
    sym_status_t s = vmm ? sym_window_alloc_vmm(R, bytes, 0, 0, &send) : sym_window_alloc(R, bytes, 0, 0, &send);
    if (s != SYM_OK) return fail("window alloc (send)", s);
    s = vmm ? sym_window_alloc_vmm(R, bytes, 0, 0, &recv) : sym_window_alloc(R, bytes, 0, 0, &recv);
    if (s != SYM_OK) return fail("window alloc (recv)", s);

    // a fixed pattern of small finite values: bytes 0x3c..0x3f in the high byte of every
    // 16-bit half, so f32, bf16 and f16 inputs all stay well inside their ranges
    std::vector<uint8_t> host(bytes);
    for (int r = 0; r < R; ++r) {
        for (size_t i = 0; i < bytes; ++i) host[i] = (i & 1) ? (uint8_t)(0x3c + ((i >> 1) + r) % 4) : (uint8_t)(i * 7 + r);
        if ((s = sym_window_write(send, r, 0, host.data(), bytes, st)) != SYM_OK) return fail("window write", s);
        if (cudaStreamSynchronize(st) != cudaSuccess) return fail("sync", SYM_ERR_CUDA);
    }

    for (int i = 0; i < warmup; ++i)
        if ((s = sym_allreduce(send, recv, count, dtype, SYM_SUM, algo, st)) != SYM_OK) return fail("allreduce", s);
    if ((s = sym_stream_status(st)) != SYM_OK) return fail("warm-up", s);

    std::vector<cudaEvent_t> ev(2 * (size_t)iters);
    for (auto& e : ev) cudaEventCreate(&e);
    for (int i = 0; i < iters; ++i) {
        cudaEventRecord(ev[2 * i], st);
        if ((s = sym_allreduce(send, recv, count, dtype, SYM_SUM, algo, st)) != SYM_OK) return fail("allreduce", s);
        cudaEventRecord(ev[2 * i + 1], st);
    }
    if ((s = sym_stream_status(st)) != SYM_OK) return fail("timed calls", s);
    std::vector<float> us(iters);
    for (int i = 0; i < iters; ++i) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]);
        us[i] = ms * 1000.f;
    }

    // every rank holds the same result
    std::vector<uint8_t> r0(bytes), rl(bytes);
    if ((s = sym_window_read(recv, 0, 0, r0.data(), bytes, st)) != SYM_OK) return fail("window read", s);
    if ((s = sym_window_read(recv, R - 1, 0, rl.data(), bytes, st)) != SYM_OK) return fail("window read", s);
    cudaStreamSynchronize(st);
    const bool same = memcmp(r0.data(), rl.data(), bytes) == 0;

    sym_algo_t used = algo;
    sym_allreduce_algo(send, count, dtype, &used);
    const double med = pct(us, 0.5);
    printf("{\"tool\": \"symar_bench\", \"ranks\": %d, \"bytes_per_rank\": %zu, \"dtype\": \"%s\", "
           "\"algo\": \"%s\", \"algo_used\": %d, \"window\": \"%s\", \"iters\": %d, \"us_median\": %.3f, "
           "\"us_p10\": %.3f, \"us_p90\": %.3f, \"algbw_gbs\": %.2f, \"compulsory_gbs\": %.2f, "
           "\"ranks_agree\": %s}\n",
           R, bytes, dtype_name.c_str(), algo_name.c_str(), (int)used,
           sym_window_kind(send) >= SYM_WINDOW_VMM_EXPORTABLE ? "vmm" : "cudaMalloc", iters, med,
           pct(us, 0.1), pct(us, 0.9), bytes / (med * 1e-6) / 1e9, 2.0 * R * bytes / (med * 1e-6) / 1e9,
           same ? "true" : "false");
    for (auto& e : ev) cudaEventDestroy(e);
    sym_window_free(send);
    sym_window_free(recv);
    cudaStreamDestroy(st);
    return same ? 0 : 3;
}
