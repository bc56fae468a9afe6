// e4m3 CTA-pair instantiations of the fused weight-gradient kernel.
#include "forge_launch.cuh"

FORGE_DEFINE_LAUNCH_PAIR()

using namespace forge;
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_ADAMW, ST_F32, false, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_ADAMW, ST_BF16, false, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_SGDM, ST_F32, false, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_SGDM, ST_BF16, false, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_DW, ST_F32, false, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_ADAMW, ST_F32, true, false)
FORGE_INSTANTIATE_PAIR(IN_E4M3, OP_ADAMW, ST_BF16, true, false)
