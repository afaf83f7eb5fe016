// ops_fwd_grouped.cu -- instantiations of the tile kernel for the fwd op
// (rowwise, colwise and both scale modes) with per-group blocked scales.
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_fwd_grouped, kFwd, kSilu, true)
}  // namespace mx
