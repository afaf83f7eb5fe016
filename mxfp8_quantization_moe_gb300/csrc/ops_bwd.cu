// ops_bwd.cu -- instantiations of the tile kernel for the bwd op
// (rowwise, colwise and both scale modes; plain or blocked scales).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_bwd, kBwd, kSilu, false)
}  // namespace mx
