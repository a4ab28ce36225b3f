// AllReduce kernels instantiated for one element type (see allreduce_kernels.cuh).
#include "allreduce_kernels.cuh"

namespace symar {

sym_status_t launch_allreduce_f32(sym_algo_t algo, sym_op_t op, ArArgs& a, sym_win_t recv,
                                  cudaStream_t st) {
    return launch_allreduce_typed<F32T>(algo, op, a, recv, st);
}

}  // namespace symar
