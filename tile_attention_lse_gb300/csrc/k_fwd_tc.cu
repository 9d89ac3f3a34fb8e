// tcgen05 tile-attention forward (sm_103a).  Placeholder until the tensor-core
// kernel lands: reports "not supported" so the CUDA-core kernel runs.
#include "internal.h"

namespace cpattn {

bool fwd_tc_supported(const FwdArgs&) { return false; }

cp_status launch_fwd_tc(const FwdArgs&, cudaStream_t) { return CP_ERR_UNSUPPORTED; }

bool bwd_tc_supported(const BwdArgs&) { return false; }

cp_status launch_bwd_tc(const BwdArgs&, cudaStream_t) { return CP_ERR_UNSUPPORTED; }

}  // namespace cpattn
