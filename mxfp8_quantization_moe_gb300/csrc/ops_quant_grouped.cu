// ops_quant_grouped.cu -- instantiations of the tile kernel for the quant op
// (rowwise, colwise and both scale modes) with per-group blocked scales.
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_quant_grouped, kQuant, kSilu, true)
}  // namespace mx
