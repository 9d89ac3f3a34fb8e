// tcgen05 tile-attention backward (sm_103a): not built yet; the CUDA-core
// backward runs meanwhile.
#include "internal.h"

namespace cpattn {

bool bwd_tc_supported(const BwdArgs&) { return false; }

cp_status launch_bwd_tc(const BwdArgs&, cudaStream_t) { return CP_ERR_UNSUPPORTED; }

}  // namespace cpattn
