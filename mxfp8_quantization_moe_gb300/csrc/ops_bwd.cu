// ops_bwd.cu -- instantiations of the tile kernel for the bwd op
// (rowwise, colwise and both scale modes).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_bwd, kBwd, kSilu)
}  // namespace mx
