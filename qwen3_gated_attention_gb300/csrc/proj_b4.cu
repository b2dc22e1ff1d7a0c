// proj_b4.cu -- 4-bit instantiations of the projection kernel.
#include "proj_inst.cuh"
GATTN_PROJ_INSTANCE(4)
