// The fused Newton-Schulz kernel with the last-step modes (FinMode): the last
// step's APPLY epilogue also applies the update in place (FIN_UPDATE) or sums v^2
// per row for NorMuon (FIN_ROWSQ).  Only calls that ask for them launch it.
#include "mb_ns_kernel.cuh"

namespace mb {

cudaError_t launch_ns_fused_fin(const NsParams& p, cudaStream_t s) { return launch_ns_kernel<true>(p, s); }

}  // namespace mb
