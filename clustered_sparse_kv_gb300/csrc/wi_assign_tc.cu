// wi_assign_tc.cu -- tensor-core (tcgen05) spherical assignment.
#include "wi_internal.h"

bool wi_assign_tc_supported(const WiGeom&) { return false; }

cudaError_t wi_launch_assign_tc(const WiGeom&, const void*, const void*, int32_t*, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
