// C ABI entry of the AllReduce: argument checks, chunk plan, algorithm choice,
// and dispatch to the per-element-type launchers (allreduce_{f32,bf16,f16}.cu;
// the kernels themselves are in allreduce_kernels.cuh).
#include "allreduce_kernels.cuh"

namespace symar {

static sym_algo_t resolve_algo(sym_algo_t algo, size_t nbytes, bool in_place) {
    if (algo != SYM_ALGO_AUTO) return algo;
    if (!in_place && nbytes <= oneshot_max_bytes()) return SYM_ALGO_ONESHOT;
    return SYM_ALGO_TWOSHOT;
}

}  // namespace symar

using namespace symar;

extern "C" {

sym_status_t sym_allreduce_algo(sym_win_t send, size_t count, sym_dtype_t dtype, sym_algo_t* out) {
    if (!send || !out) return SYM_ERR_INVALID_ARG;
    size_t es = dtype_size(dtype);
    if (!es) return SYM_ERR_INVALID_ARG;
    *out = resolve_algo(SYM_ALGO_AUTO, count * es, false);
    return SYM_OK;
}

sym_status_t sym_allreduce(sym_win_t send, sym_win_t recv, size_t count, sym_dtype_t dtype,
                           sym_op_t op, sym_algo_t algo, sym_stream_t stream) {
    if (!send || !recv) return SYM_ERR_INVALID_ARG;
    if (send->R != recv->R || send->device != recv->device) return SYM_ERR_INVALID_ARG;
    const size_t es = dtype_size(dtype);
    if (!es) return SYM_ERR_INVALID_ARG;
    if ((int)op < SYM_SUM || (int)op > SYM_MIN) return SYM_ERR_INVALID_ARG;
    if (algo != SYM_ALGO_AUTO && algo != SYM_ALGO_ONESHOT && algo != SYM_ALGO_TWOSHOT &&
        algo != SYM_ALGO_TWOSHOT_PULL && algo != SYM_ALGO_TWOSHOT_SPLIT)
        return SYM_ERR_INVALID_ARG;
    if (count > send->bytes / es || count > recv->bytes / es) return SYM_ERR_INVALID_ARG;
    if (count == 0) return SYM_OK;
    const bool in_place = send->base == recv->base;
    const size_t nbytes = count * es;
    if (nbytes / kVecBytes > ((size_t)1 << 34)) return SYM_ERR_UNSUPPORTED;   // work-item indices
    algo = resolve_algo(algo, nbytes, in_place);
    if (in_place && algo == SYM_ALGO_ONESHOT) return SYM_ERR_UNSUPPORTED;
    if (in_place && send != recv) return SYM_ERR_INVALID_ARG;   // two handles, one memory
    if (!in_place && windows_overlap(send, nbytes, recv, nbytes)) {
        // partly aliased windows (caller memory): one-shot would race, and the
        // pull gathers would read inputs another slot has overwritten
        set_last_error("sym_allreduce: send and recv windows share memory without being one window");
        return SYM_ERR_INVALID_ARG;
    }

    ArArgs a{};
    a.send = send->base;
    a.recv = recv->base;
    a.sstride = send->stride;
    a.rstride = recv->stride;
    a.R = send->R;
    a.nvec = nbytes / kVecBytes;
    a.chunk_vec = ceil_div(a.nvec, (size_t)a.R);
    const size_t V = kVecBytes / es;
    a.tail_elem0 = a.nvec * V;
    a.tail_n = (uint32_t)(count - a.tail_elem0);
    DeviceGuard g(recv->device);
    if (!g.ok) return SYM_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    switch (dtype) {
        case SYM_F32: return launch_allreduce_f32(algo, op, a, recv, st);
        case SYM_BF16: return launch_allreduce_bf16(algo, op, a, recv, st);
        case SYM_F16: return launch_allreduce_f16(algo, op, a, recv, st);
    }
    return SYM_ERR_INVALID_ARG;
}

}  // extern "C"
