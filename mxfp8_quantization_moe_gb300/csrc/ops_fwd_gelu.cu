// ops_fwd_gelu.cu -- instantiations of the tile kernel for the fwd op with the GEGLU
// activation
// (rowwise, colwise and both scale modes; plain or blocked scales).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_fwd_gelu, kFwd, kGelu, false)
}  // namespace mx
