// proj_b25.cu -- 2- and 5-bit instantiations of the projection kernel.
#include "proj_inst.cuh"
GATTN_PROJ_INSTANCE(2)
GATTN_PROJ_INSTANCE(5)
