// The Newton-Schulz launch of a step: the plain instantiation of the fused kernel
// (mb_ns_kernel.cuh), or, when a bank asks its last step's epilogue to finish the
// step (FinMode), the instantiation in mb_ns_gemm_fin.cu, which carries that code.
// The two live in separate files so that each compiles on its own and the plain
// kernel's register allocation is not shaped by code it never runs.
#include "mb_ns_kernel.cuh"

namespace mb {

cudaError_t launch_ns_fused(const NsParams& p, cudaStream_t s) {
  for (int i = 0; i < p.nbank; ++i)
    if (p.bank[i].fin != FIN_NONE) return launch_ns_fused_fin(p, s);
  return launch_ns_kernel<false>(p, s);
}

}  // namespace mb
