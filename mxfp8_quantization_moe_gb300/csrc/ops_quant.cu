// ops_quant.cu -- instantiations of the tile kernel for the quant op
// (rowwise, colwise and both scale modes).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_quant, kQuant, kSilu)
}  // namespace mx
