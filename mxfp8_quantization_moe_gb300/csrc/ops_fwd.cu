// ops_fwd.cu -- instantiations of the tile kernel for the fwd op
// (rowwise, colwise and both scale modes; plain or blocked scales).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_fwd, kFwd, kSilu, false)
}  // namespace mx
