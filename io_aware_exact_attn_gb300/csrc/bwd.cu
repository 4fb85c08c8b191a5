// bwd.cu -- placeholder launchers; the backward kernels follow.
#include "internal.h"

namespace attn {

cudaError_t launch_bwd_dkdv(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const BwdParams&, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_bwd_dq(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                          const CUtensorMap&, const BwdParams&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace attn
