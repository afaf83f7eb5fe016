// ops_quant.cu -- instantiations of the tile kernel for the quant op
// (rowwise, colwise and both scale modes; plain or blocked scales).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_quant, kQuant, kSilu, false)
}  // namespace mx
