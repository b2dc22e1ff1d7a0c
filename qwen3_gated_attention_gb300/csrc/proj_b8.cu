// proj_b8.cu -- 8-bit instantiations of the projection kernel.
#include "proj_inst.cuh"
GATTN_PROJ_INSTANCE(8)
